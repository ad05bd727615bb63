// Forward pass of Flex-Flash-Attention on sm_103a.
//
// MagiAttention blog, "Flex-Flash-Attention and AttnSlice" (Figure 5: data
// loading, on-chip compute, merge of partial results) and the documentation's
// "FFA_FA4 backend" (Full blocks skip masking, Partial blocks are masked,
// Empty blocks are skipped; the lists come from the CSR metadata).
//
// One persistent CTA per SM.  A work unit is (q-tile, head pair): the two q
// heads 2p and 2p+1 share the q-tile's block list (the mask does not depend on
// the head), and share K/V tiles in shared memory when they belong to the same
// GQA group.  Units follow the plan's longest-work-first order of q-tiles,
// either all head pairs of a q-tile before the next q-tile or, with many
// q-tiles, all q-tiles of a head pair before the next pair (the host picks):
// each CTA starts with unit blockIdx.x and then pops the next unit from one
// counter whenever its producer is ready for more, so that a CTA that runs
// faster takes more units (the producer hands the unit ids to the issuer and
// the softmax warps through a shared-memory ring).
//
// Warp roles (384 threads):
//   warp 0      TMA producer: Q tiles of the unit, then the K/V tile ring
//   warp 1      UMMA issuer (one thread): S_T = Q_T K^T and O_T += P_T V
//   warps 4-7   softmax + epilogue of head tile T = 0
//   warps 8-11  softmax + epilogue of head tile T = 1
// Registers: launched at 168 a thread; warpgroup 0 drops to 136 and the two
// softmax warpgroups rise to 184, enough to hold a row's 128 scores at once.
// Each SM sub-partition runs one warp of every warpgroup, so its share,
// (136 + 184 + 184) x 32, stays inside its 16384 registers.
// TMEM (512 columns): S_0 | S_1 | O_0 | O_1.  P_T (bf16) is written over the
// first 64 columns of S_T and read by the P V MMA straight from TMEM.  While
// the tensor cores run tile 0's MMAs the other warpgroup runs tile 1's softmax
// and vice versa.
//
// Online softmax in the log2 domain: p = 2^(s * scale * log2(e) - m).  The
// running max m of a row is only raised when a block's max exceeds it by more
// than 8 (so p <= 256), which leaves O untouched on most blocks; when it is
// raised the row's O and l are rescaled in TMEM.  On head pairs that load
// their own K / V tiles, a Full block's exponentials are taken against the
// running max before its max is known, and redone in the rare case the max
// had to be raised.
#include <cuda_bf16.h>

#include "ffa_internal.h"
#include "ptx.cuh"
#include "tma.h"

namespace ffa {
namespace {

constexpr int kFwdThreads = 384;
constexpr int kMaxSlots = 10;
constexpr float kRescaleThreshold = 8.0f;
constexpr int32_t kFwdPairMajorTiles = 2048;   // q-tiles from which units go head-pair major
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

struct FwdBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done[2], o_empty[2];
  uint64_t stage[2];
  uint64_t kv_full[kMaxSlots], kv_empty[kMaxSlots];
  uint64_t final_mma;
  UnitRing ring;   // unit ids from the producer to the issuer and the 8 softmax warps
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t kFwdUnitConsumers = 1 + 8;

template <int D>
struct FwdCfg {
  static constexpr int kTile = 128 * D * 2;   // bytes of one 128-row Q, K or V tile
  static constexpr int kHalves = D / 64;      // 64-column swizzle panels per tile
  static constexpr int kSlots = D == 128 ? 5 : 10;
  // TMEM columns of S_T and O_T
  __host__ __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(t) * D; }
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(2 + kSlots) * kTile + sizeof(FwdBars);
};

struct FwdParams {
  const int32_t* full_off;
  const int32_t* full_idx;
  const int32_t* mask_off;
  const int32_t* mask_idx;
  const int32_t* order;
  const int32_t* iv_off;
  const int32_t* iv;
  float* lse;
  __nv_bfloat16* out;
  int32_t seqlen_q, hq, group, n_pairs, n_qt;
  int32_t pair_major;   // unit order: see decode_unit
  int64_t n_units;
  float scale_log2;
  uint32_t* status;
  int32_t accumulate;   // merge into the (out, lse) already in memory instead of overwriting
  const float* sink;    // per-head sink logits [hq], or null
  uint64_t* trace;      // per-CTA {start ns, end ns, units, blocks}, or null
  uint32_t* next;       // unit counter, zero at launch
};

struct Unit {
  int32_t qt, h0, g0, g1, nt, nf, fo, mo, n;
  bool shared;
};

__device__ __forceinline__ Unit decode_unit(const FwdParams& p, int64_t u) {
  Unit x;
  if (p.pair_major) {   // all q-tiles of one head pair, then the next pair
    x.qt = p.order[u % p.n_qt];
    x.h0 = 2 * static_cast<int32_t>(u / p.n_qt);
  } else {               // all head pairs of one q-tile, then the next q-tile
    x.qt = p.order[u / p.n_pairs];
    x.h0 = 2 * static_cast<int32_t>(u % p.n_pairs);
  }
  x.nt = x.h0 + 1 < p.hq ? 2 : 1;
  x.g0 = x.h0 / p.group;
  x.g1 = (x.h0 + x.nt - 1) / p.group;
  x.shared = x.g0 == x.g1;
  x.fo = p.full_off[x.qt];
  x.nf = p.full_off[x.qt + 1] - x.fo;
  x.mo = p.mask_off[x.qt];
  x.n = x.nf + p.mask_off[x.qt + 1] - x.mo;
  return x;
}

__device__ __forceinline__ int32_t block_at(const FwdParams& p, const Unit& x, int32_t j, bool& partial) {
  partial = j >= x.nf;
  return partial ? p.mask_idx[x.mo + j - x.nf] : p.full_idx[x.fo + j];
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status,
                                          uint32_t code) {
  const bool ok = mbar_wait(bar, parity, abort, status, code);
  return __all_sync(0xffffffffu, ok);
}

// Allowed columns of one row inside the 128-column block starting at c0, as a
// 128-bit mask, from the row's sorted key intervals.
__device__ __forceinline__ void row_block_mask(const int32_t* iv, int32_t e0, int32_t e1, int32_t c0,
                                               uint32_t (&m)[4]) {
  m[0] = m[1] = m[2] = m[3] = 0u;
  for (int32_t e = e0; e < e1; ++e) {
    const int32_t x0 = max(iv[2 * e] - c0, 0), x1 = min(iv[2 * e + 1] - c0, 128);
    if (x1 <= x0) continue;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int32_t a = max(x0 - 32 * w, 0), b = min(x1 - 32 * w, 32);
      if (b > a) m[w] |= (b - a == 32 ? 0xffffffffu : ((1u << (b - a)) - 1u)) << a;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    ffa_fwd_kernel(const FwdParams p, const __grid_constant__ CUtensorMap map_q,
                   const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                   const __grid_constant__ CUtensorMap map_o) {
  using C = FwdCfg<D>;
  constexpr int NS = C::kSlots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ[2] = {base, base + C::kTile};
  uint8_t* slots = base + 2 * C::kTile;
  FwdBars* bars = reinterpret_cast<FwdBars*>(slots + NS * C::kTile);
  volatile int* abort = &bars->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->q_empty[t], 1);
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 128);
      mbar_init(&bars->o_done[t], 1);
      mbar_init(&bars->o_empty[t], 128);
      mbar_init(&bars->stage[t], 128);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    mbar_init(&bars->final_mma, 1);
    unit_ring_init(bars->ring, kFwdUnitConsumers);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const uint64_t t_start = p.trace && tid == 0 ? global_timer_ns() : 0;
  uint32_t traced_units = 0, traced_blocks = 0;   // counted by the producer (thread 0)

  auto producer_role = [&]() {
    // ---------------- TMA producer ----------------
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_o);
    uint32_t kv_i = 0, q_fills[2] = {0, 0};
    bool ok = true;
    auto push = [&](const CUtensorMap* map, int32_t g, int32_t b) -> bool {
      const uint32_t s = kv_i % NS, use = kv_i / NS;
      if (!mbar_wait(&bars->kv_empty[s], (use & 1u) ^ 1u, abort, p.status, kStatusTimeoutTmaEmpty)) return false;
      mbar_arrive_expect_tx(&bars->kv_full[s], C::kTile);
#pragma unroll
      for (int hf = 0; hf < C::kHalves; ++hf)
        tma_load_3d(slots + s * C::kTile + hf * 16384, map, &bars->kv_full[s], hf * 64, g, b * 128);
      ++kv_i;
      return true;
    };
    for (uint32_t ui = 0; ok; ++ui) {
      const int64_t u = unit_take_next(p.next, ui, p.n_units);
      if (!(ok = unit_publish(bars->ring, ui, u, abort, p.status)) || u < 0) break;
      const Unit x = decode_unit(p, u);
      if (x.n == 0) continue;
      ++traced_units;
      traced_blocks += static_cast<uint32_t>(x.n);
      for (int t = 0; t < x.nt && ok; ++t) {
        ok = mbar_wait(&bars->q_empty[t], (q_fills[t] & 1u) ^ 1u, abort, p.status, kStatusTimeoutTmaEmpty);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->q_full[t], C::kTile);
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf)
          tma_load_3d(sQ[t] + hf * 16384, &map_q, &bars->q_full[t], hf * 64, x.h0 + t, x.qt * 128);
        ++q_fills[t];
      }
      bool pb;
      int32_t bprev = block_at(p, x, 0, pb);
      ok = ok && push(&map_k, x.g0, bprev);
      if (!x.shared) ok = ok && push(&map_k, x.g1, bprev);
      for (int32_t j = 1; ok && j < x.n; ++j) {
        const int32_t b = block_at(p, x, j, pb);
        ok = push(&map_v, x.g0, bprev) && push(&map_k, x.g0, b);
        if (!x.shared) ok = ok && push(&map_v, x.g1, bprev) && push(&map_k, x.g1, b);
        bprev = b;
      }
      ok = ok && push(&map_v, x.g0, bprev);
      if (!x.shared) ok = ok && push(&map_v, x.g1, bprev);
    }
    // Wait for every copy this thread issued before the CTA may exit.
    for (uint32_t s = 0; s < NS; ++s) {
      const uint32_t uses = kv_i / NS + (s < kv_i % NS ? 1u : 0u);
      if (uses) mbar_wait(&bars->kv_full[s], (uses - 1) & 1u, abort, p.status, kStatusTimeoutTmaFull);
    }
    for (int t = 0; t < 2; ++t)
      if (q_fills[t]) mbar_wait(&bars->q_full[t], (q_fills[t] - 1) & 1u, abort, p.status, kStatusTimeoutTmaFull);
  };
  auto issuer_role = [&]() {
    // ---------------- UMMA issuer ----------------
    constexpr uint32_t idesc_s = umma_idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idesc_o = umma_idesc_bf16(128, D, 0, 1);
    // descriptors of Q_T (K-major), the K slots (K-major) and V slots (MN-major)
    const uint64_t dq0 = smem_desc_sw128(smem_u32(sQ[0]), 16, 1024), dq1 = smem_desc_sw128(smem_u32(sQ[1]), 16, 1024);
    const uint64_t dk0 = smem_desc_sw128(smem_u32(slots), 16, 1024);
    const uint64_t dv0 = smem_desc_sw128(smem_u32(slots), 16384, 1024);
    uint32_t kv_i = 0, q_k[2] = {0, 0}, o_k[2] = {0, 0}, p_cnt[2] = {0, 0};
    bool ok = true;
    auto take = [&](uint32_t& s) -> bool {
      s = kv_i % NS;
      const uint32_t use = kv_i / NS;
      ++kv_i;
      if (!mbar_wait(&bars->kv_full[s], use & 1u, abort, p.status, kStatusTimeoutTmaFull)) return false;
      tc_fence_after_sync();
      return true;
    };
    auto mma_s = [&](int t, uint32_t s) {
      const uint64_t dk = desc_at(dk0, s * C::kTile), dqt = t ? dq1 : dq0;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        umma_ss(tmem + C::col_s(t), desc_at(dqt, off), desc_at(dk, off), idesc_s, kk > 0);
      }
      umma_commit(&bars->s_full[t]);
    };
    // O_T (+)= P_T V.  A Full block's P (bf16) fills S_T's columns [0, 64) in
    // key order; a Partial block's P is hi + lo, keys [32c, 32c + 32) as hi in
    // columns [32c, 32c + 16) and lo in [32c + 16, 32c + 32).
    auto mma_o = [&](int t, uint32_t s, bool acc, bool partial) {
      const uint64_t dv = desc_at(dv0, s * C::kTile);
      const uint32_t d_o = tmem + C::col_o(t), a_p = tmem + C::col_s(t);
      const uint32_t acc0 = acc ? 1u : 0u;
      // One branch per block, not per MMA: with the P column a compile-time
      // offset in each path the MMAs issue back to back (a per-MMA select
      // between the two layouts measurably slowed their issue).
      if (!partial) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) umma_ts(d_o, a_p + 8 * kk, desc_at(dv, kk * 2048), idesc_o, kk > 0 ? 1u : acc0);
      } else {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(d_o, a_p + 32 * (kk >> 1) + 8 * (kk & 1), desc_at(dv, kk * 2048), idesc_o, kk > 0 ? 1u : acc0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ts(d_o, a_p + 32 * (kk >> 1) + 8 * (kk & 1) + 16, desc_at(dv, kk * 2048), idesc_o, 1u);
      }
    };
    auto wait_p = [&](int t) -> bool {
      if (!mbar_wait(&bars->p_full[t], p_cnt[t] & 1u, abort, p.status, kStatusTimeoutSoftmax)) return false;
      ++p_cnt[t];
      tc_fence_after_sync();
      return true;
    };
    auto wait_o_empty = [&](int t) -> bool {
      if (!mbar_wait(&bars->o_empty[t], (o_k[t] & 1u) ^ 1u, abort, p.status, kStatusTimeoutSoftmax)) return false;
      tc_fence_after_sync();
      return true;
    };
    for (uint32_t ui = 0; ok; ++ui) {
      int64_t u;
      if (!(ok = unit_read(bars->ring, ui, u, abort, p.status)) || u < 0) break;
      const Unit x = decode_unit(p, u);
      if (x.n == 0) continue;
      for (int t = 0; t < x.nt && ok; ++t) {
        ok = mbar_wait(&bars->q_full[t], q_k[t] & 1u, abort, p.status, kStatusTimeoutTmaFull);
        ++q_k[t];
      }
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t sk, sv;
      // block 0: S_T = Q_T K_0^T
      if (x.shared) {
        if (!(ok = take(sk))) break;
        for (int t = 0; t < x.nt; ++t) mma_s(t, sk);
        umma_commit(&bars->kv_empty[sk]);
      } else {
        for (int t = 0; t < x.nt && ok; ++t) {
          if (!(ok = take(sk))) break;
          mma_s(t, sk);
          umma_commit(&bars->kv_empty[sk]);
        }
      }
      // blocks 1..n-1: O_T += P_T(j-1) V_(j-1), then S_T = Q_T K_j^T
      for (int32_t j = 1; ok && j < x.n; ++j) {
        const bool prev_partial = j - 1 >= x.nf;
        if (x.shared) {
          if (!(ok = take(sv) && take(sk))) break;
          for (int t = 0; t < x.nt && ok; ++t) {
            if (!(ok = wait_p(t))) break;
            if (j == 1 && !(ok = wait_o_empty(t))) break;
            mma_o(t, sv, j > 1, prev_partial);
            mma_s(t, sk);
          }
          umma_commit(&bars->kv_empty[sv]);
          umma_commit(&bars->kv_empty[sk]);
        } else {
          for (int t = 0; t < x.nt && ok; ++t) {
            if (!(ok = take(sv) && take(sk))) break;
            if (!(ok = wait_p(t))) break;
            if (j == 1 && !(ok = wait_o_empty(t))) break;
            mma_o(t, sv, j > 1, prev_partial);
            umma_commit(&bars->kv_empty[sv]);
            mma_s(t, sk);
            umma_commit(&bars->kv_empty[sk]);
          }
        }
      }
      if (!ok) break;
      // last block: O_T += P_T(n-1) V_(n-1)
      if (x.shared) {
        if (!(ok = take(sv))) break;
        for (int t = 0; t < x.nt && ok; ++t) {
          if (!(ok = wait_p(t))) break;
          if (x.n == 1 && !(ok = wait_o_empty(t))) break;
          mma_o(t, sv, x.n > 1, x.n - 1 >= x.nf);
          umma_commit(&bars->o_done[t]);
        }
        umma_commit(&bars->kv_empty[sv]);
      } else {
        for (int t = 0; t < x.nt && ok; ++t) {
          if (!(ok = take(sv))) break;
          if (!(ok = wait_p(t))) break;
          if (x.n == 1 && !(ok = wait_o_empty(t))) break;
          mma_o(t, sv, x.n > 1, x.n - 1 >= x.nf);
          umma_commit(&bars->o_done[t]);
          umma_commit(&bars->kv_empty[sv]);
        }
      }
      for (int t = 0; t < x.nt; ++t) ++o_k[t];
    }
    umma_commit(&bars->final_mma);
    mbar_wait(&bars->final_mma, 0, abort, p.status, kStatusTimeoutMma);
  };
  auto softmax_role = [&]() {
    // ---------------- softmax + epilogue ----------------
    const int t = (warp - 4) >> 2;
    const int wr = warp & 3;
    const int r = wr * 32 + lane;   // row inside the q-tile == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wr * 32) << 16);
    const uint32_t tS = lane_base + C::col_s(t), tO = lane_base + C::col_o(t);
    uint32_t s_k = 0, o_k = 0;
    bool alive = true;
    for (uint32_t ui = 0; alive; ++ui) {
      int64_t u;
      if (!(alive = unit_read_warp(bars->ring, ui, u, abort, p.status)) || u < 0) break;
      const Unit x = decode_unit(p, u);
      if (t >= x.nt) continue;
      const int32_t h = x.h0 + t;
      const int32_t row = x.qt * 128 + r;
      const bool valid = row < p.seqlen_q;
      if (x.n == 0) {
        if (valid && !p.accumulate) {
          uint4* dst = reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(row) * p.hq + h) * D);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          p.lse[static_cast<int64_t>(h) * p.seqlen_q + row] = p.sink ? p.sink[h] : -INFINITY;
        }
        continue;
      }
      const int32_t e0 = valid ? p.iv_off[row] : 0, e1 = valid ? p.iv_off[row + 1] : 0;
      float m_used = -INFINITY, l = 0.f;
      for (int32_t j = 0; j < x.n; ++j) {
        bool partial;
        const int32_t b = block_at(p, x, j, partial);
        if (!warp_wait(&bars->s_full[t], s_k & 1u, abort, p.status, kStatusTimeoutMma)) {
          alive = false;
          break;
        }
        ++s_k;
        tc_fence_after_sync();
        uint32_t m[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
        if (partial) row_block_mask(p.iv, e0, e1, b * 128, m);
        __syncwarp();
        // The row's 128 scores, read from TMEM at once: one load round trip per block.
        uint32_t v[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, v[c]);
        tmem_ld_wait_only();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_pin(v[c]);
        if (partial) {   // masked scores of a Partial block become -inf
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (!((m[c] >> i) & 1u)) v[c][i] = __float_as_uint(-INFINITY);
        }
        // The block's row max: four independent chains (one per 32-column
        // chunk), 16 deep each.
        auto block_max = [&]() -> float {
          float mxc[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) mxc[c] = fmaxf(__uint_as_float(v[c][0]), __uint_as_float(v[c][1]));
#pragma unroll
          for (int i = 2; i < 32; i += 2) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              mxc[c] = fmax3(mxc[c], __uint_as_float(v[c][i]), __uint_as_float(v[c][i + 1]));
          }
          return fmaxf(fmaxf(mxc[0], mxc[1]), fmaxf(mxc[2], mxc[3]));
        };
        float alpha = 1.f;
        bool rescale = false;
        // Raise the running max when the block's max exceeds it by more than
        // the threshold; O and l are then rescaled by alpha.
        auto raise_max = [&](float mx) {
          const float m_new = fmaxf(m_used, mx * p.scale_log2);
          if (m_new > m_used + kRescaleThreshold) {
            if (m_used != -INFINITY) {
              alpha = ex2_approx(m_used - m_new);
              rescale = true;
              l *= alpha;
            }
            m_used = m_new;
          }
        };
        // p = 2^(s * scale * log2e - m) against the running max, bf16 P into
        // TMEM, and the block's row sum.  A Full block's P goes to columns
        // [16c, 16c + 16) for chunk c; a Partial block keeps hi + lo in the
        // chunk's own 32 columns.  Every score is already in registers, so no
        // store overwrites one still to be read.
        auto exps = [&]() -> float {
          const float m_use = m_used == -INFINITY ? 0.f : m_used;
          const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2), nm2 = f2_pack(-m_use, -m_use);
          uint64_t lsum2 = f2_pack(0.f, 0.f), lsum2b = f2_pack(0.f, 0.f);   // two sum chains
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t (&cur)[32] = v[c];
            if (!partial) {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float x0, x1;
                f2_unpack(ffma2(f2_pack(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1])), c2, nm2), x0,
                          x1);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                if (i & 1) lsum2b = fadd2(lsum2b, f2_pack(p0, p1));
                else lsum2 = fadd2(lsum2, f2_pack(p0, p1));
                pk[i] = pack_bf16x2(p0, p1);
              }
              tmem_st16(tS + c * 16, pk);
            } else {
              // Rows with fewer than 128 allowed keys only meet Partial blocks,
              // where a single bf16 P would dominate the output error: keep
              // P = hi + lo, both bf16, and let the MMA issuer run P V twice.
              // (two halves of 8 pairs, to keep fewer registers live)
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int i8 = 0; i8 < 8; ++i8) {
                  const int i = 8 * hh + i8;
                  const bool k0 = (m[c] >> (2 * i)) & 1u, k1 = (m[c] >> (2 * i + 1)) & 1u;
                  float x0, x1;
                  f2_unpack(ffma2(f2_pack(__uint_as_float(cur[2 * i]), __uint_as_float(cur[2 * i + 1])), c2, nm2),
                            x0, x1);
                  const float p0 = k0 ? ex2_approx(x0) : 0.f, p1 = k1 ? ex2_approx(x1) : 0.f;
                  const uint64_t p2 = f2_pack(p0, p1);
                  lsum2 = fadd2(lsum2, p2);
                  hi[i8] = pack_bf16x2(p0, p1);
                  float r0, r1;
                  f2_unpack(
                      fsub2(p2, f2_pack(__uint_as_float(hi[i8] << 16), __uint_as_float(hi[i8] & 0xffff0000u))), r0,
                      r1);
                  lo[i8] = pack_bf16x2(r0, r1);
                }
                tmem_st8(tS + c * 32 + 8 * hh, hi);
                tmem_st8(tS + c * 32 + 16 + 8 * hh, lo);
              }
            }
          }
          float a, b2;
          f2_unpack(fadd2(lsum2, lsum2b), a, b2);
          return a + b2;
        };
        // A Full block of a unit whose two heads load their own K / V tiles,
        // once every row of the warp has a running max: the exponentials are
        // taken against it straight away, P is kept packed in registers, and
        // the block's max is taken in the same pass (four chains).  Only when
        // that max exceeds the running one by more than the threshold (rare
        // after a row's first blocks) are the scores read again from TMEM,
        // still intact since no P has been stored, and the block redone
        // against the raised max.  The max pass thus stays off the chain
        // softmax -> P V and next S -> softmax.  (When the two heads share
        // their K / V tiles, storing P chunk by chunk as it is computed was
        // measured faster than this.)
        if (!x.shared && !partial && __all_sync(0xffffffffu, m_used != -INFINITY)) {
          const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2), nm2 = f2_pack(-m_used, -m_used);
          uint64_t lsum2 = f2_pack(0.f, 0.f), lsum2b = f2_pack(0.f, 0.f);
          float mxc[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
          uint32_t pk[4][16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float s0 = __uint_as_float(v[c][2 * i]), s1 = __uint_as_float(v[c][2 * i + 1]);
              mxc[c] = fmax3(mxc[c], s0, s1);
              float x0, x1;
              f2_unpack(ffma2(f2_pack(s0, s1), c2, nm2), x0, x1);
              const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              if (i & 1) lsum2b = fadd2(lsum2b, f2_pack(p0, p1));
              else lsum2 = fadd2(lsum2, f2_pack(p0, p1));
              pk[c][i] = pack_bf16x2(p0, p1);
            }
          }
          const float mx = fmaxf(fmaxf(mxc[0], mxc[1]), fmaxf(mxc[2], mxc[3]));
          if (__any_sync(0xffffffffu, mx * p.scale_log2 > m_used + kRescaleThreshold)) {
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, v[c]);
            tmem_ld_wait_only();
#pragma unroll
            for (int c = 0; c < 4; ++c) reg_pin(v[c]);
            raise_max(mx);
            l += exps();
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_st16(tS + c * 16, pk[c]);
            float a, b2;
            f2_unpack(fadd2(lsum2, lsum2b), a, b2);
            l += a + b2;
          }
        } else {
          raise_max(block_max());
          l += exps();
        }
        if (__any_sync(0xffffffffu, rescale && j > 0)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(tO + c * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&bars->p_full[t]);
      }
      if (!alive) break;
      // epilogue: O / l -> bf16 -> swizzled staging tile (the Q buffer) -> TMA store
      if (!warp_wait(&bars->o_done[t], o_k & 1u, abort, p.status, kStatusTimeoutMma)) {
        alive = false;
        break;
      }
      tc_fence_after_sync();
      // This unit's result for the row: O / l with lse_p = ln(l) + m.  It is
      // merged with a partial (out0, lse0): in accumulate mode the one
      // already stored, with a sink the sink logit with out0 = 0:
      // lse = ln(e^lse0 + e^lse_p), out = w0 out0 + wp O / l with
      // w0 = e^(lse0 - lse) and wp = e^(lse_p - lse).
      const float lse_p = l > 0.f ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
      float inv_l = l > 0.f ? 1.f / l : 0.f, w0 = 0.f, lse_out = lse_p;
      const __nv_bfloat16* out0 = p.out + (static_cast<int64_t>(valid ? row : 0) * p.hq + h) * D;
      if (p.accumulate || p.sink) {
        const float lse0 = p.sink ? p.sink[h] : valid ? p.lse[static_cast<int64_t>(h) * p.seqlen_q + row] : -INFINITY;
        const float mx = fmaxf(lse0, lse_p);
        if (mx == -INFINITY) {
          inv_l = 0.f;
        } else {
          const float e0 = ex2_approx((lse0 - mx) * kLog2e), ep = ex2_approx((lse_p - mx) * kLog2e);
          const float sum = e0 + ep;
          w0 = p.accumulate ? e0 / sum : 0.f;   // a sink's out0 is zero
          inv_l *= ep / sum;
          lse_out = mx + __log2f(sum) * kLn2;
        }
      }
      const bool merge = w0 != 0.f;
      uint8_t* stage = sQ[t];
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(tO + c * 32, o);
        tmem_ld_wait(o);
        const int col0 = c * 32;
        uint8_t* panel = stage + (col0 >> 6) * 16384 + r * 128;
        if (merge) {   // o = w0 out0 + (wp / l) O, with inv_l already holding wp / l
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 a = reinterpret_cast<const uint4*>(out0 + col0)[q];
            const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              o[8 * q + 2 * e] = __float_as_uint(__uint_as_float(o[8 * q + 2 * e]) * inv_l +
                                                 w0 * __uint_as_float(aw[e] << 16));
              o[8 * q + 2 * e + 1] = __float_as_uint(__uint_as_float(o[8 * q + 2 * e + 1]) * inv_l +
                                                     w0 * __uint_as_float(aw[e] & 0xffff0000u));
            }
          }
        }
        const float sc = merge ? 1.f : inv_l;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * sc, __uint_as_float(o[8 * q + 1]) * sc);
          v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * sc, __uint_as_float(o[8 * q + 3]) * sc);
          v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * sc, __uint_as_float(o[8 * q + 5]) * sc);
          v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * sc, __uint_as_float(o[8 * q + 7]) * sc);
          const int chunk = ((col0 & 63) >> 3) + q;
          *reinterpret_cast<uint4*>(panel + (((chunk ^ r) & 7) << 4)) = v;
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&bars->o_empty[t]);
      fence_proxy_async_smem();
      mbar_arrive(&bars->stage[t]);
      if (valid) p.lse[static_cast<int64_t>(h) * p.seqlen_q + row] = lse_out;
      if (r == 0) {
        if (mbar_wait(&bars->stage[t], o_k & 1u, abort, p.status, kStatusTimeoutOther)) {
#pragma unroll
          for (int hf = 0; hf < C::kHalves; ++hf) tma_store_3d(&map_o, stage + hf * 16384, hf * 64, h, x.qt * 128);
          tma_store_commit();
          tma_store_wait_read_all();
          mbar_arrive(&bars->q_empty[t]);
        } else {
          alive = false;
        }
      }
      ++o_k;
      alive = __all_sync(0xffffffffu, alive);
    }
    if (r == 0) tma_store_wait_all();
  };
  // Each role runs under its warpgroup's register budget (set where it
  // dominates the role's code): 128 x 136 + 256 x 184 = 384 x 168, the
  // launch's registers.
  if (warp < 4) {
    regs_dec<136>();
    if (warp == 0 && lane == 0) producer_role();
    else if (warp == 1 && lane == 0) issuer_role();
  } else {
    regs_inc<184>();
    softmax_role();
  }
  tc_fence_before_sync();
  __syncthreads();
  if (p.trace && tid == 0) {
    uint64_t* t = p.trace + 4 * static_cast<int64_t>(blockIdx.x);
    t[0] = t_start;
    t[1] = global_timer_ns();
    t[2] = traced_units;
    t[3] = traced_blocks;
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

__global__ void fill_empty_kernel(__nv_bfloat16* out, int64_t n_out, float* lse, int64_t n_lse, const float* sink,
                                  int64_t seqlen_q) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_out || i < n_lse;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < n_out) out[i] = __float2bfloat16(0.f);
    if (i < n_lse) lse[i] = sink ? sink[i / seqlen_q] : -INFINITY;   // lse is [hq][seqlen_q]
  }
}

template <int D>
ffa_status launch_fwd(const FwdParams& prm, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                      const CUtensorMap& mo, int grid, cudaStream_t stream, KernelTimer* timer) {
  // Set on every launch: the attribute belongs to the current context's copy
  // of the kernel, so a cached flag would go stale after a device reset, and
  // the call is cheap and safe from several host threads.
  if (cudaFuncSetAttribute(ffa_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(FwdCfg<D>::kSmem)) != cudaSuccess)
    return FFA_ERR_CUDA;
  ScopedKernelTimer tk(timer, FFA_KERNEL_FWD, stream);
  ffa_fwd_kernel<D><<<grid, kFwdThreads, FwdCfg<D>::kSmem, stream>>>(prm, mq, mk, mv, mo);
  return cuda_status(cudaGetLastError());
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ffa

using namespace ffa;

namespace {
ffa_status fwd_impl(const void* q, const void* k, const void* v, int64_t seqlen_q, int64_t seqlen_k, int32_t hq,
                    int32_t hkv, int32_t d, ffa_plan_t plan, float scale, void* out, float* lse, void* stream,
                    bool accumulate, const float* sink) {
  if (!plan || !q || !k || !v || !out || !lse) return FFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return FFA_ERR_INVALID_ARG;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return FFA_ERR_INVALID_ARG;
  if (seqlen_q != plan->seqlen_q || seqlen_k != plan->seqlen_k) return FFA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FFA_ERR_UNSUPPORTED;
  if (plan->tiles.fwd_bm != 128 || plan->tiles.fwd_bn != 128) return FFA_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (seqlen_q == 0) return FFA_OK;
  if (seqlen_k == 0) {
    if (accumulate) return FFA_OK;   // nothing to merge in
    const int64_t n_out = seqlen_q * hq * d, n_lse = seqlen_q * hq;
    fill_empty_kernel<<<plan->num_sms * 4, 256, 0, st>>>(static_cast<__nv_bfloat16*>(out), n_out, lse, n_lse, sink,
                                                         seqlen_q);
    return cuda_status(cudaGetLastError());
  }
  CUtensorMap mq, mk, mv, mo;
  if (!make_tile_map(&mq, q, seqlen_q, hq, d) || !make_tile_map(&mk, k, seqlen_k, hkv, d) ||
      !make_tile_map(&mv, v, seqlen_k, hkv, d) || !make_tile_map(&mo, out, seqlen_q, hq, d))
    return FFA_ERR_CUDA;
  FwdParams prm;
  prm.full_off = plan->q2k.full_off;
  prm.full_idx = plan->q2k.full_idx;
  prm.mask_off = plan->q2k.mask_off;
  prm.mask_idx = plan->q2k.mask_idx;
  prm.order = plan->q2k.order;
  prm.iv_off = plan->q2k.iv_off;
  prm.iv = plan->q2k.iv;
  prm.lse = lse;
  prm.out = static_cast<__nv_bfloat16*>(out);
  prm.seqlen_q = static_cast<int32_t>(seqlen_q);
  prm.hq = hq;
  prm.group = hq / hkv;
  prm.n_pairs = (hq + 1) / 2;
  prm.n_qt = plan->q2k.n_rt;
  // Unit order.  Head-pair major keeps the CTAs that run at one time on one
  // head pair, and so on one pair's K / V, which cuts DRAM re-reads (128K
  // varlen: 5.3 -> 1.3 GB); it was measured faster with many q-tiles (1M
  // varlen, 8192: -3 %; 256K sink + window, 2048: -3 %) and slower with few
  // (128K varlen, 1024: +3 %; 64K varlen, 512: +9 %; 128K video, 1024: even).
  prm.pair_major = plan->q2k.n_rt >= kFwdPairMajorTiles ? 1 : 0;
  prm.n_units = static_cast<int64_t>(plan->q2k.n_rt) * prm.n_pairs;
  prm.scale_log2 = scale * kLog2e;
  prm.status = &plan->words->status;
  prm.accumulate = accumulate ? 1 : 0;
  prm.sink = sink;
  if (prm.n_units > INT32_MAX) return FFA_ERR_OVERFLOW;
  const int grid = static_cast<int>(std::min<int64_t>(prm.n_units, plan->num_sms));
  prm.trace = plan->trace.begin(FFA_KERNEL_FWD, grid);
  prm.next = &plan->words->fwd_next;
  if (cudaMemsetAsync(prm.next, 0, sizeof(uint32_t), st) != cudaSuccess) return FFA_ERR_CUDA;
  return d == 128 ? launch_fwd<128>(prm, mq, mk, mv, mo, grid, st, &plan->timer)
                  : launch_fwd<64>(prm, mq, mk, mv, mo, grid, st, &plan->timer);
}
}  // namespace

extern "C" ffa_status ffa_fwd(const void* q, const void* k, const void* v, int64_t seqlen_q, int64_t seqlen_k,
                              int32_t hq, int32_t hkv, int32_t d, ffa_plan_t plan, float scale, void* out, float* lse,
                              void* stream) {
  return fwd_impl(q, k, v, seqlen_q, seqlen_k, hq, hkv, d, plan, scale, out, lse, stream, false, nullptr);
}

extern "C" ffa_status ffa_fwd_accumulate(const void* q, const void* k, const void* v, int64_t seqlen_q,
                                         int64_t seqlen_k, int32_t hq, int32_t hkv, int32_t d, ffa_plan_t plan,
                                         float scale, void* out, float* lse, void* stream) {
  return fwd_impl(q, k, v, seqlen_q, seqlen_k, hq, hkv, d, plan, scale, out, lse, stream, true, nullptr);
}

extern "C" ffa_status ffa_fwd_sink(const void* q, const void* k, const void* v, int64_t seqlen_q, int64_t seqlen_k,
                                   int32_t hq, int32_t hkv, int32_t d, ffa_plan_t plan, float scale, const float* sink,
                                   void* out, float* lse, void* stream) {
  if (!sink) return FFA_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, seqlen_q, seqlen_k, hq, hkv, d, plan, scale, out, lse, stream, false, sink);
}
