// Backward pass of Flex-Flash-Attention on sm_103a.
//
// MagiAttention blog, "Flex-Flash-Attention and AttnSlice": FFA must support
// backward for training, and slice-parallel partial results are merged by
// atomic reduction (Figure 5 caption).  Gradients of out = softmax(scale Q
// K^T) V over the mask: with P = exp(scale S - lse) and D_i = dO_i . O_i,
//   dV = P^T dO,  dS = P o (dO V^T - D),  dK = scale dS^T Q,  dQ = scale dS K.
//
// Three kernels:
//   bwd_pre   D_i and -lse * log2(e) of every (head, query) into a padded
//             workspace (-inf for empty and padded rows, so that P = 0
//             there), and a cleared fp32 dq accumulator;
//   bwd_main  persistent; a work unit is (work item, kv head), a work item
//             being one k-tile's blocks inside one q-chunk of the k2q CSR
//             lists; it loops over those q-tiles and the q heads of the GQA
//             group, keeping dK and dV of its 128 keys in TMEM, and adds them
//             to fp32 accumulators at the end (or stores them, when the unit
//             holds every block of its k-tile);
//   bwd_dq    dq, dk, dv = bf16(accumulators).
//
// bwd_main works on transposed scores, one key per TMEM lane, in half-steps
// of 64 queries:
//   S^T = K Q^T and dP^T = V dO^T          (UMMA, smem x smem -> TMEM)
//   P^T and dS^T (bf16) over S^T's columns (queries 32h + [0, 32) in
//   columns 32h + [0, 16) and 32h + [16, 32)), dS^T also to shared memory
//   dV += P^T dO                           (UMMA, A from TMEM)
//   dK += dS^T Q                           (UMMA, A from TMEM)
//   dQ^T = K^T dS^T                        (UMMA into dP^T's columns)
// and a dq warpgroup reads dQ^T (one head-dim index per lane), stages it as
// fp32 rows in shared memory and adds it to the accumulator with TMA bulk
// reduce-adds.  Two TMEM buffers for S^T / dP^T and two dS^T buffers let the
// tensor cores work on one half-step while the softmax gradient runs on the
// other.  At the end of a unit the softmax warpgroups write dK and dV from
// TMEM straight to global memory while the next unit's tiles load.
//
// Warp roles (512 threads): warp 0 TMA producer, warps 1 and 2 UMMA issuers
// (S^T / dP^T and dV / dQ^T / dK), warps 4-11 softmax gradient + dK/dV
// epilogue (two warpgroups, each on half of a half-step's queries, so that
// twice the warps hide the latency of its dependent arithmetic), warps 12-15
// dq writer.  Registers: launched at 128 a thread and rebalanced per
// warpgroup (112 / 144 / 144 / 112).
// TMEM (512 columns): dK | dV | S^T_0 dP^T_0 | S^T_1 dP^T_1.
#include <cuda_bf16.h>

#include <cstddef>

#include "ffa_internal.h"
#include "ptx.cuh"
#include "tma.h"

namespace ffa {
namespace {

constexpr int kBwdThreads = 512;
// setmaxnreg budgets of warpgroup 0 (producer, issuers), the two softmax-
// gradient warpgroups and the dq writer: RA + 2 RS + RQ = 4 x 128.
constexpr uint32_t kRegsA = 112, kRegsS = 144, kRegsQ = 112;
static_assert(kRegsA + 2 * kRegsS + kRegsQ == 4 * 128, "register budgets must add up to the launch's");
constexpr int kD = 128;                // shared-memory tiles are sized for head dim 128
constexpr int kTile = 128 * kD * 2;   // 32 KB
constexpr float kLog2e = 1.4426950408889634f;
// TMEM columns: dK | dV | buffer 0: S^T (64) dP^T (64) | buffer 1: S^T dP^T.
// dQ^T of a half-step is written over its buffer's dP^T columns.
constexpr uint32_t kColDK = 0, kColDV = 128;
__device__ __forceinline__ uint32_t col_s(uint32_t b) { return 256u + 128u * b; }
__device__ __forceinline__ uint32_t col_dp(uint32_t b) { return 256u + 128u * b + 64u; }
constexpr int kHalf = 64;                      // queries per half-step
constexpr int kDsTile = 128 * kHalf * 2;       // dS^T of one half-step: 128 keys x 64 queries bf16
constexpr int kHalfTile = kHalf * 128 * 2;     // Q or dO rows of one half-step: 2 panels of 64 x 128 B
constexpr int kStages = 3;                     // half-step stages of Q, dO, lse, D
constexpr int kDqRows = 32;                    // queries per dq reduce-add box
constexpr int kDqStage = kDqRows * kD * 4;     // fp32 dq staging tile (16 KB)
constexpr uint32_t kDqBar = 1;                 // named barrier of the dq writer warps

// What the producer records for the consumers of a stage.
struct StageMeta {
  int32_t a, h, half, partial;
};

struct alignas(16) BwdBars {
  uint64_t kv_full, kv_empty;
  uint64_t st_full[kStages], st_empty[kStages];  // half-step stages
  uint64_t s_full[2], p_full[2], ds_empty[2];    // per TMEM / dS^T buffer
  uint64_t p_read[2];                            // dV has read P^T out of S^T's columns
  uint64_t dq_full[2], dq_empty[2];
  uint64_t acc_full, acc_empty;
  uint64_t final_a, final_b;
  UnitRing ring;   // unit ids from the producer to the two issuers, 8 softmax and 4 dq warps

  uint32_t tmem_base;
  int abort;
  StageMeta meta[kStages];
  alignas(16) float nl[kStages][kHalf];          // -lse * log2(e) of the stage's 64 queries (bulk-copy target)
  alignas(16) float dv[kStages][kHalf];          // D of the stage's 64 queries (bulk-copy target)
};
// K, V, Q[3], dO[3], dS^T[2], dq staging[2] (1024-byte aligned tiles) + barriers and per-stage rows
constexpr size_t kBwdSmem = 1024 + 2 * static_cast<size_t>(kTile) + 2 * kStages * static_cast<size_t>(kHalfTile) +
                            2 * kDsTile + 2 * kDqStage + sizeof(BwdBars);
static_assert(kBwdSmem <= 232448, "shared memory budget");

struct BwdParams {
  const int4* items;         // work items {k-tile, Full start, Partial start, #Full | #Partial << 16}
  const int32_t* full_idx;   // k2q CSR lists
  const int32_t* mask_idx;
  const int32_t* full_off;   // k2q CSR offsets (per k-tile)
  const int32_t* mask_off;
  const int32_t* kiv_off;    // per-key allowed query intervals
  const int32_t* kiv;
  const float* lse2;         // [hq][sq_pad] -lse * log2(e) (-inf: no contribution)
  const float* dvec;         // [hq][sq_pad] D_i
  float* dk_acc;             // [sk][hkv][d] fp32
  float* dv_acc;             // [sk][hkv][d] fp32
  int32_t seqlen_q, seqlen_k, sq_pad, hq, hkv, group;
  int64_t n_units;
  float scale, scale_log2;
  uint32_t* status;
  uint64_t* trace;           // per-CTA {start ns, end ns, units, blocks}, or null
  uint32_t* next;            // unit counter, zero at launch
};
constexpr uint32_t kBwdUnitConsumers = 1 + 1 + 8 + 4;

struct BUnit {
  int32_t kt, g, nf, fo, mo, nm, n;
};

// Unit u = (work item u % n_items, kv head u / n_items): every item of one kv
// head, then the next head.  A work item is one k-tile with the blocks of its
// k2q lists that fall in one q-chunk; the plan orders the items chunk by
// chunk, so that the units running at one time work on one chunk of one head
// group and share its Q / dO tiles and dq rows in L2 instead of each fetching
// them from HBM.  (Item-major order, every kv head of an item before the next
// item, spread the running units over all heads: 11 % slower on the 128K
// video workload with 8 kv heads, 6 % on the 256K sink + window one with 32.)
__device__ __forceinline__ BUnit decode(const BwdParams& p, int64_t u) {
  BUnit x;
  const int64_t n_items = p.n_units / p.hkv;
  const int4 it = __ldg(&p.items[u % n_items]);
  x.kt = it.x;
  x.g = static_cast<int32_t>(u / n_items);
  x.fo = it.y;
  x.mo = it.z;
  x.nf = it.w & 0xffff;
  x.nm = it.w >> 16;
  x.n = x.nf + x.nm;
  return x;
}

// The j-th q-tile a unit visits: its Full blocks, then its Partial blocks,
// each from the highest q-tile down.
__device__ __forceinline__ int32_t qtile_at(const BwdParams& p, const BUnit& x, int32_t j, bool& partial) {
  partial = j >= x.nf;
  return partial ? p.mask_idx[x.mo + x.nm - 1 - (j - x.nf)] : p.full_idx[x.fo + x.nf - 1 - j];
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status,
                                          uint32_t code) {
  const bool ok = mbar_wait(bar, parity, abort, status, code);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void block_mask128(const int32_t* iv, int32_t e0, int32_t e1, int32_t c0, uint32_t (&m)[4]) {
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

// Write 16 bf16 values (8 packed words) of row r, columns [col0, col0+16),
// into a [128 x 128] bf16 tile stored as two 64-column 128-byte-swizzled panels.
__device__ __forceinline__ void store_row16_sw128(uint8_t* tile, int r, int col0, const uint32_t (&w)[8]) {
  uint8_t* panel = tile + (col0 >> 6) * 16384 + r * 128;
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int chunk = ((col0 & 63) >> 3) + q;
    *reinterpret_cast<uint4*>(panel + (((chunk ^ r) & 7) << 4)) =
        make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
}

// Half-step index i of a unit -> (q-tile, head, 64-query half).  The order is
// q-tile (CSR order), then the group's heads, then the two halves.
struct HalfStep {
  int32_t a, h, half, j;
  bool partial;
};
__device__ __forceinline__ HalfStep half_step(const BwdParams& p, const BUnit& x, int32_t i) {
  HalfStep hs;
  hs.half = i & 1;
  const int32_t pair = i >> 1;
  hs.j = pair / p.group;
  hs.h = x.g * p.group + pair % p.group;
  hs.a = qtile_at(p, x, hs.j, hs.partial);
  return hs;
}

// D: head dim, 128 or 64.  With D = 64 the tiles use their first 64-column
// panel only, and the K tile's second panel holds zeros, so that dQ^T =
// K^T dS^T keeps its 128-row shape: its rows 64..127 come out zero and are
// not written back.
template <int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    ffa_bwd_main_kernel(const BwdParams p, const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_do, const __grid_constant__ CUtensorMap map_dq) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sK = base;
  uint8_t* sV = base + kTile;
  uint8_t* sQ = base + 2 * kTile;                          // kStages x kHalfTile
  uint8_t* sdO = sQ + kStages * kHalfTile;                 // kStages x kHalfTile
  uint8_t* sdS[2] = {sdO + kStages * kHalfTile, sdO + kStages * kHalfTile + kDsTile};
  float* sdq[2] = {reinterpret_cast<float*>(sdS[1] + kDsTile), reinterpret_cast<float*>(sdS[1] + kDsTile + kDqStage)};
  BwdBars* bars = reinterpret_cast<BwdBars*>(sdS[1] + kDsTile + 2 * kDqStage);
  volatile int* abort = &bars->abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->st_full[s], 1);
      mbar_init(&bars->st_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->p_full[s], 256);
      mbar_init(&bars->ds_empty[s], 1);
      mbar_init(&bars->p_read[s], 1);
      mbar_init(&bars->dq_full[s], 1);
      mbar_init(&bars->dq_empty[s], 128);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 256);
    mbar_init(&bars->final_a, 1);
    mbar_init(&bars->final_b, 1);
    unit_ring_init(bars->ring, kBwdUnitConsumers);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if constexpr (D < kD) {   // the K tile's unused panel, read as zero rows of K^T by dQ^T
    uint4* z = reinterpret_cast<uint4*>(sK + 16384);
    for (int i = tid; i < 16384 / 16; i += kBwdThreads) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  constexpr int kPanels = D / 64;   // 64-column swizzle panels per row
  const uint64_t t_start = p.trace && tid == 0 ? global_timer_ns() : 0;
  uint32_t traced_units = 0, traced_blocks = 0;   // counted by the producer (thread 0)

  auto producer_role = [&]() {
    // ---------------- TMA producer ----------------
    // Per unit: K and V of the k-tile.  Per half-step (stage ring of 3): the
    // 64 Q and dO rows, their -lse * log2(e) and D values, and a record of
    // (q-tile, head, half, partial) for the consumers.
    tma_prefetch_desc(&map_q);
    tma_prefetch_desc(&map_k);
    tma_prefetch_desc(&map_v);
    tma_prefetch_desc(&map_do);
    // A unit's first stages are loaded before its K and V: their slots free
    // up as the previous unit's last MMAs finish, while K and V wait for all
    // of them.
    uint32_t kv_k = 0, g = 0;
    bool ok = true;
    auto load_stage = [&](const BUnit& x, int32_t i) -> bool {
      const HalfStep hs = half_step(p, x, i);
      const uint32_t s = g % kStages, use = g / kStages;
      if (!mbar_wait(&bars->st_empty[s], (use & 1u) ^ 1u, abort, p.status, kStatusTimeoutTmaEmpty)) return false;
      bars->meta[s] = StageMeta{hs.a, hs.h, hs.half, hs.partial ? 1 : 0};
      mbar_arrive_expect_tx(&bars->st_full[s], 2 * kPanels * (kHalfTile / 2) + 2 * kHalf * 4);
      const int32_t q0 = hs.a * 128 + hs.half * kHalf;
      for (int hf = 0; hf < kPanels; ++hf) {
        tma_load_3d(sQ + s * kHalfTile + hf * (kHalfTile / 2), &map_q, &bars->st_full[s], hf * 64, hs.h, q0);
        tma_load_3d(sdO + s * kHalfTile + hf * (kHalfTile / 2), &map_do, &bars->st_full[s], hf * 64, hs.h, q0);
      }
      const int64_t row = static_cast<int64_t>(hs.h) * p.sq_pad + q0;
      bulk_load(bars->nl[s], p.lse2 + row, kHalf * 4, &bars->st_full[s]);
      bulk_load(bars->dv[s], p.dvec + row, kHalf * 4, &bars->st_full[s]);
      ++g;
      return true;
    };
    for (uint32_t ui = 0; ok; ++ui) {
      const int64_t u = unit_take_next(p.next, ui, p.n_units);
      if (!(ok = unit_publish(bars->ring, ui, u, abort, p.status)) || u < 0) break;
      const BUnit x = decode(p, u);
      if (x.n == 0) continue;
      ++traced_units;
      traced_blocks += static_cast<uint32_t>(x.n * p.group);
      const int32_t steps = x.n * p.group * 2;
      const int32_t pre = steps < kStages ? steps : kStages;
      int32_t i = 0;
      for (; ok && i < pre; ++i) ok = load_stage(x, i);
      if (!ok) break;
      if (!(ok = mbar_wait(&bars->kv_empty, (kv_k & 1u) ^ 1u, abort, p.status, kStatusTimeoutTmaEmpty))) break;
      mbar_arrive_expect_tx(&bars->kv_full, 2 * kPanels * 16384);
      for (int hf = 0; hf < kPanels; ++hf) {
        tma_load_3d(sK + hf * 16384, &map_k, &bars->kv_full, hf * 64, x.g, x.kt * 128);
        tma_load_3d(sV + hf * 16384, &map_v, &bars->kv_full, hf * 64, x.g, x.kt * 128);
      }
      ++kv_k;
      for (; ok && i < steps; ++i) ok = load_stage(x, i);
    }
    if (kv_k) mbar_wait(&bars->kv_full, (kv_k - 1) & 1u, abort, p.status, kStatusTimeoutTmaFull);
    for (uint32_t s = 0; s < kStages; ++s) {
      const uint32_t uses = g / kStages + (s < g % kStages ? 1u : 0u);
      if (uses) mbar_wait(&bars->st_full[s], (uses - 1) & 1u, abort, p.status, kStatusTimeoutTmaFull);
    }
  };
  auto issuer_a_role = [&]() {
    // ---------------- UMMA issuer A: S^T_b = K Q^T, dP^T_b = V dO^T ----------------
    // Two threads issue the MMAs: a tcgen05.mma issue slot left empty while
    // its thread waits on a barrier is lost to the tensor cores, so the waits
    // of one issuer run while the other issues.  Half-step g uses TMEM /
    // dS^T buffer b = g mod 2 and stage g mod 3.  S^T_b is written once dV of
    // half-step g - 2 has read P^T out of it (p_read), dP^T_b once the dq
    // writer has read dQ^T of half-step g - 2 out of it (dq_empty).
    constexpr uint32_t idesc_a = umma_idesc_bf16(128, 64, 0, 0);    // 128 keys x 64 queries
    constexpr uint32_t kPanel = kHalfTile / 2;   // 64 rows x 128 bytes
    // K, V K-major (A); stage Q / dO K-major (B)
    const uint64_t dK_k = smem_desc_sw128(smem_u32(sK), 16, 1024), dV_k = smem_desc_sw128(smem_u32(sV), 16, 1024);
    const uint64_t dQ_k0 = smem_desc_sw128(smem_u32(sQ), 16, 1024), dO_k0 = smem_desc_sw128(smem_u32(sdO), 16, 1024);
    uint32_t kv_k = 0, g = 0;
    bool ok = true;
    for (uint32_t ui = 0; ok; ++ui) {
      int64_t u;
      if (!(ok = unit_read(bars->ring, ui, u, abort, p.status)) || u < 0) break;
      const BUnit x = decode(p, u);
      if (x.n == 0) continue;
      if (!(ok = mbar_wait(&bars->kv_full, kv_k & 1u, abort, p.status, kStatusTimeoutTmaFull))) break;
      ++kv_k;
      const int32_t steps = x.n * p.group * 2;
      for (int32_t i = 0; i < steps; ++i, ++g) {
        const uint32_t b = g & 1u, s = g % kStages, prev = ((g >> 1) & 1u) ^ 1u;
        if (!(ok = mbar_wait(&bars->st_full[s], (g / kStages) & 1u, abort, p.status, kStatusTimeoutTmaFull)) ||
            !(ok = mbar_wait(&bars->p_read[b], prev, abort, p.status, kStatusTimeoutMma)))
          break;
        tc_fence_after_sync();
        const uint64_t dQ_k = desc_at(dQ_k0, s * kHalfTile), dO_k = desc_at(dO_k0, s * kHalfTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + col_s(b), desc_at(dK_k, (kk >> 2) * 16384 + (kk & 3) * 32),
                  desc_at(dQ_k, (kk >> 2) * kPanel + (kk & 3) * 32), idesc_a, kk > 0);
        if (!(ok = mbar_wait(&bars->dq_empty[b], prev, abort, p.status, kStatusTimeoutSoftmax))) break;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tmem + col_dp(b), desc_at(dV_k, (kk >> 2) * 16384 + (kk & 3) * 32),
                  desc_at(dO_k, (kk >> 2) * kPanel + (kk & 3) * 32), idesc_a, kk > 0);
        umma_commit(&bars->s_full[b]);
      }
    }
    umma_commit(&bars->final_a);
    mbar_wait(&bars->final_a, 0, abort, p.status, kStatusTimeoutMma);
  };
  auto issuer_b_role = [&]() {
    // ---------------- UMMA issuer B: dV += P^T dO, dQ^T = K^T dS^T, dK += dS^T Q ----------------
    // Per half-step, once the softmax gradient has written P^T and dS^T
    // (p_full).  Each commit marks what the next user may take over: S^T_b
    // (holding P^T and a copy of dS^T) and the stage after dV and dK
    // (p_read, st_empty), dQ^T_b and the shared-memory dS^T_b after dQ^T
    // (dq_full, ds_empty); K and V after a unit's last half-step, whose MMAs
    // follow every MMA of issuer A for that unit.
    constexpr uint32_t idesc_b = umma_idesc_bf16(128, D, 0, 1);     // dV, dK: 128 keys x D dims
    constexpr uint32_t idesc_q = umma_idesc_bf16(128, 64, 1, 1);    // dQ^T: 128 dims x 64 queries
    constexpr uint32_t kPanel = kHalfTile / 2;
    // K MN-major (A of dQ^T); stage Q / dO MN-major (B of dK / dV);
    // dS^T MN-major (B of dQ^T)
    const uint64_t dK_mn = smem_desc_sw128(smem_u32(sK), 16384, 1024);
    const uint64_t dQ_mn0 = smem_desc_sw128(smem_u32(sQ), kPanel, 1024);
    const uint64_t dO_mn0 = smem_desc_sw128(smem_u32(sdO), kPanel, 1024);
    const uint64_t dS_mn0 = smem_desc_sw128(smem_u32(sdS[0]), 16384, 1024),
                   dS_mn1 = smem_desc_sw128(smem_u32(sdS[1]), 16384, 1024);
    uint32_t kv_k = 0, g = 0;
    bool ok = true;
    for (uint32_t ui = 0; ok; ++ui) {
      int64_t u;
      if (!(ok = unit_read(bars->ring, ui, u, abort, p.status)) || u < 0) break;
      const BUnit x = decode(p, u);
      if (x.n == 0) continue;
      if (!(ok = mbar_wait(&bars->kv_full, kv_k & 1u, abort, p.status, kStatusTimeoutTmaFull)) ||
          !(ok = mbar_wait(&bars->acc_empty, (kv_k & 1u) ^ 1u, abort, p.status, kStatusTimeoutSoftmax)))
        break;
      const int32_t steps = x.n * p.group * 2;
      for (int32_t i = 0; i < steps; ++i, ++g) {
        const uint32_t b = g & 1u, s = g % kStages;
        if (!(ok = mbar_wait(&bars->p_full[b], (g >> 1) & 1u, abort, p.status, kStatusTimeoutSoftmax)) ||
            !(ok = mbar_wait(&bars->st_full[s], (g / kStages) & 1u, abort, p.status, kStatusTimeoutTmaFull)))
          break;
        tc_fence_after_sync();
        const uint64_t dQ_mn = desc_at(dQ_mn0, s * kHalfTile), dO_mn = desc_at(dO_mn0, s * kHalfTile);
        const uint64_t dS_mn = b ? dS_mn1 : dS_mn0;
        const uint32_t acc = i > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)   // dV += P^T dO   (K = 64 queries)
          umma_ts(tmem + kColDV, tmem + col_s(b) + (kk >> 1) * 32 + (kk & 1) * 8, desc_at(dO_mn, kk * 2048), idesc_b,
                  (acc | kk) ? 1u : 0u);
        // dK before dQ^T: Q is then free (st_empty) one GEMM earlier, which
        // gives the stage ring more time to refill
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)   // dK += dS^T Q, dS^T from TMEM
          umma_ts(tmem + kColDK, tmem + col_s(b) + (kk >> 1) * 32 + 16 + (kk & 1) * 8, desc_at(dQ_mn, kk * 2048),
                  idesc_b, (acc | kk) ? 1u : 0u);
        umma_commit(&bars->p_read[b]);
        umma_commit(&bars->st_empty[s]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)   // dQ^T = K^T dS^T   (K = 128 keys), into dP^T's columns
          umma_ss(tmem + col_dp(b), desc_at(dK_mn, kk * 2048), desc_at(dS_mn, kk * 2048), idesc_q, kk > 0);
        umma_commit(&bars->dq_full[b]);
        umma_commit(&bars->ds_empty[b]);
      }
      if (!ok) break;
      umma_commit(&bars->acc_full);
      umma_commit(&bars->kv_empty);   // K and V are no longer read
      ++kv_k;
    }
    umma_commit(&bars->final_b);
    mbar_wait(&bars->final_b, 0, abort, p.status, kStatusTimeoutMma);
  };
  auto softmax_role = [&]() {
    // ---------------- softmax gradient + dK/dV epilogue ----------------
    // Two warpgroups; warpgroup hs takes queries [32 hs, 32 hs + 32) of every
    // half-step and columns [64 hs, 64 hs + 64) of dK and dV at the end.
    const int hs = (warp - 4) >> 2;
    const int wr = warp & 3;
    const int r = wr * 32 + lane;   // key row inside the k-tile == TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wr * 32) << 16);
    const uint64_t c2 = f2_pack(p.scale_log2, p.scale_log2);
    uint32_t g = 0, kv_k = 0;
    bool alive = true;
    for (uint32_t ui = 0; alive; ++ui) {
      int64_t u;
      if (!(alive = unit_read_warp(bars->ring, ui, u, abort, p.status)) || u < 0) break;
      const BUnit x = decode(p, u);
      const int32_t key = x.kt * 128 + r;
      const bool valid = key < p.seqlen_k;
      if (x.n == 0) continue;
      const int32_t e0 = valid ? p.kiv_off[key] : 0, e1 = valid ? p.kiv_off[key + 1] : 0;
      const int32_t steps = x.n * p.group * 2;
      uint32_t m[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
      int32_t mask_a = -1;
      for (int32_t i = 0; i < steps; ++i, ++g) {
        const uint32_t b = g & 1u, s = g % kStages;
        if (!warp_wait(&bars->s_full[b], (g >> 1) & 1u, abort, p.status, kStatusTimeoutMma) ||
            !warp_wait(&bars->st_full[s], (g / kStages) & 1u, abort, p.status, kStatusTimeoutTmaFull) ||
            !warp_wait(&bars->ds_empty[b], ((g >> 1) & 1u) ^ 1u, abort, p.status, kStatusTimeoutMma)) {
          alive = false;
          break;
        }
        tc_fence_after_sync();
        const StageMeta mt = bars->meta[s];
        if (mt.a != mask_a) {   // the allowed-query mask of this key row over the q-tile
          mask_a = mt.a;
          m[0] = m[1] = m[2] = m[3] = 0xffffffffu;
          if (mt.partial) block_mask128(p.kiv, e0, e1, mt.a * 128, m);
          __syncwarp();
        }
        const float* nlr = bars->nl[s];
        const float* dvr = bars->dv[s];
        // This key row's 32 scores and 32 dP values of the warpgroup's
        // queries, read from TMEM at once, then 16 queries at a time.
        uint32_t sv[32], dp[32];
        tmem_ld32(lane_base + col_s(b) + 32 * hs, sv);
        tmem_ld32(lane_base + col_dp(b) + 32 * hs, dp);
        tmem_ld_wait_only();
        reg_pin(sv);
        reg_pin(dp);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int c = 2 * hs + cc;   // 16-query chunk of the half-step
          float nl[16], dq[16];
#pragma unroll
          for (int i2 = 0; i2 < 4; ++i2) {
            *reinterpret_cast<float4*>(&nl[4 * i2]) = reinterpret_cast<const float4*>(nlr + c * 16)[i2];
            *reinterpret_cast<float4*>(&dq[4 * i2]) = reinterpret_cast<const float4*>(dvr + c * 16)[i2];
          }
          const uint32_t mw = (m[2 * mt.half + hs] >> (cc * 16)) & 0xffffu;
          uint32_t pk[8], dk[8];
#pragma unroll
          for (int i2 = 0; i2 < 8; ++i2) {
            // P = 2^(s * scale * log2e - lse * log2e);  dS = P (dP - D)
            const int q = 16 * cc + 2 * i2;
            float p0, p1;
            f2_unpack(ffma2(f2_pack(__uint_as_float(sv[q]), __uint_as_float(sv[q + 1])), c2,
                            f2_pack(nl[2 * i2], nl[2 * i2 + 1])),
                      p0, p1);
            p0 = ((mw >> (2 * i2)) & 1u) ? ex2_approx(p0) : 0.f;
            p1 = ((mw >> (2 * i2 + 1)) & 1u) ? ex2_approx(p1) : 0.f;
            const uint64_t pp = f2_pack(p0, p1);
            float d0, d1;
            f2_unpack(fmul2(pp, fsub2(f2_pack(__uint_as_float(dp[q]), __uint_as_float(dp[q + 1])),
                                      f2_pack(dq[2 * i2], dq[2 * i2 + 1]))),
                      d0, d1);
            pk[i2] = pack_bf16x2(p0, p1);
            dk[i2] = pack_bf16x2(d0, d1);
          }
          // P^T and dS^T (bf16) of queries [16c, 16c + 16) into S^T's
          // columns 32 hs + [8 cc, 8 cc + 8) and 32 hs + 16 + [8 cc, 8 cc + 8):
          // inside this warpgroup's own (already read) 32 columns, never in
          // the other warpgroup's.  dS^T also goes to shared memory, as the B
          // operand of dQ^T.
          tmem_st8(lane_base + col_s(b) + 32 * hs + 8 * cc, pk);
          tmem_st8(lane_base + col_s(b) + 32 * hs + 16 + 8 * cc, dk);
          store_row16_sw128(sdS[b], r, c * 16, dk);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        fence_proxy_async_smem();
        mbar_arrive(&bars->p_full[b]);
      }
      if (!alive) break;
      // epilogue: the unit's dK * scale and dV (this thread's key row) go to
      // the fp32 accumulators straight from registers, so that K and V in
      // shared memory can already take the next unit's tiles.  When the unit
      // holds every block of its k-tile (one q-chunk covers them all, as with
      // short documents) it is the rows' only writer: plain stores into the
      // cleared accumulator replace the reduce-adds, which stall the warp.
      const bool sole = x.nf == p.full_off[x.kt + 1] - p.full_off[x.kt] &&
                        x.nm == p.mask_off[x.kt + 1] - p.mask_off[x.kt];
      if (!warp_wait(&bars->acc_full, kv_k & 1u, abort, p.status, kStatusTimeoutMma)) {
        alive = false;
        break;
      }
      tc_fence_after_sync();
      float* dk_row = p.dk_acc + (static_cast<int64_t>(valid ? key : 0) * p.hkv + x.g) * D;
      float* dv_row = p.dv_acc + (static_cast<int64_t>(valid ? key : 0) * p.hkv + x.g) * D;
      // D / 64 chunks of 32 columns per warpgroup
#pragma unroll
      for (int cc = 0; cc < kPanels; ++cc) {
        const int c = kPanels * hs + cc;
        uint32_t a32[32], b32[32];
        tmem_ld32(lane_base + kColDK + c * 32, a32);
        tmem_ld32(lane_base + kColDV + c * 32, b32);
        tmem_ld_wait(a32);
        tmem_ld_wait(b32);
        if (cc == kPanels - 1) {
          tc_fence_before_sync();
          mbar_arrive(&bars->acc_empty);
        }
        if (valid && sole) {
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            *reinterpret_cast<float4*>(dk_row + c * 32 + 4 * q4) =
                make_float4(__uint_as_float(a32[4 * q4]) * p.scale, __uint_as_float(a32[4 * q4 + 1]) * p.scale,
                            __uint_as_float(a32[4 * q4 + 2]) * p.scale, __uint_as_float(a32[4 * q4 + 3]) * p.scale);
            *reinterpret_cast<float4*>(dv_row + c * 32 + 4 * q4) =
                make_float4(__uint_as_float(b32[4 * q4]), __uint_as_float(b32[4 * q4 + 1]),
                            __uint_as_float(b32[4 * q4 + 2]), __uint_as_float(b32[4 * q4 + 3]));
          }
        } else if (valid) {
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            red_add_v4(dk_row + c * 32 + 4 * q4, __uint_as_float(a32[4 * q4]) * p.scale,
                       __uint_as_float(a32[4 * q4 + 1]) * p.scale, __uint_as_float(a32[4 * q4 + 2]) * p.scale,
                       __uint_as_float(a32[4 * q4 + 3]) * p.scale);
            red_add_v4(dv_row + c * 32 + 4 * q4, __uint_as_float(b32[4 * q4]), __uint_as_float(b32[4 * q4 + 1]),
                       __uint_as_float(b32[4 * q4 + 2]), __uint_as_float(b32[4 * q4 + 3]));
          }
        }
      }
      ++kv_k;
    }
  };
  auto dq_role = [&]() {
    // ---------------- dq writer ----------------
    // dQ^T (one head-dim index per TMEM lane) -> two fp32 staging tiles of
    // 32 queries x 128 dims -> TMA bulk reduce-add into the accumulator.
    // The four warps step together on named barrier kDqBar: each half-step
    // starts with a vote on whether every warp's (bounded) wait succeeded, so
    // that all of them leave together and no warp is left at a barrier.  A
    // staging tile is rewritten once the reduction issued two tiles earlier
    // has finished reading it.
    const int wr = warp & 3;
    const int dcol = wr * 32 + lane;   // head-dim index == TMEM lane of dQ^T
    const bool leader = dcol == 0;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wr * 32) << 16);
    if (leader) tma_prefetch_desc(&map_dq);
    uint32_t g = 0;   // half-steps
    bool alive = true;
    for (uint32_t ui = 0; alive; ++ui) {
      int64_t u = -1;
      alive = named_bar_and(kDqBar, 128, unit_read_warp(bars->ring, ui, u, abort, p.status));
      if (!alive || u < 0) break;
      const BUnit x = decode(p, u);
      if (x.n == 0) continue;
      const int32_t steps = x.n * p.group * 2;
      HalfStep nxt = half_step(p, x, 0);
      for (int32_t i = 0; i < steps; ++i, ++g) {
        const HalfStep hs = nxt;
        if (i + 1 < steps) nxt = half_step(p, x, i + 1);   // global reads overlap the wait below
        const uint32_t b = g & 1u;
        alive = named_bar_and(kDqBar, 128, warp_wait(&bars->dq_full[b], (g >> 1) & 1u, abort, p.status,
                                                        kStatusTimeoutMma));
        if (!alive) break;
        tc_fence_after_sync();
        uint32_t v[64];
        tmem_ld32(lane_base + col_dp(b) + 0, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(lane_base + col_dp(b) + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait(v);
        tc_fence_before_sync();
        mbar_arrive(&bars->dq_empty[b]);
        const int32_t q0 = hs.a * 128 + hs.half * kHalf;
#pragma unroll
        for (int part = 0; part < kHalf / kDqRows; ++part) {
          float* st = sdq[part];
          if (leader) tma_store_wait_read_1();   // the reduction two tiles back has read this buffer
          named_bar_sync(kDqBar, 128);
          if (dcol < D) {   // rows D..127 of dQ^T are the zero padding of a 64-dim K
#pragma unroll
            for (int c = 0; c < kDqRows; ++c) st[c * D + dcol] = __uint_as_float(v[part * kDqRows + c]) * p.scale;
          }
          fence_proxy_async_smem();
          named_bar_sync(kDqBar, 128);
          if (leader) {
            if (q0 + part * kDqRows < p.seqlen_q) tma_reduce_add_3d(&map_dq, st, 0, hs.h, q0 + part * kDqRows);
            tma_store_commit();   // one bulk group per tile, empty past the last query
          }
        }
      }
    }
    if (leader) tma_store_wait_all();
  };
  // Each role runs under its warpgroup's register budget, set where it
  // dominates the role's code: 128 x (RA + 2 RS + RQ) = 512 x 128, the
  // launch's registers (each SM sub-partition runs one warp of every
  // warpgroup, so its share stays inside its 16384 registers).
  if (warp < 4) {
    regs_dec<kRegsA>();
    if (warp == 0 && lane == 0) producer_role();
    else if (warp == 1 && lane == 0) issuer_a_role();
    else if (warp == 2 && lane == 0) issuer_b_role();
  } else if (warp < 12) {
    regs_inc<kRegsS>();
    softmax_role();
  } else {
    regs_dec<kRegsQ>();
    dq_role();
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

// D_i = dO_i . O_i and -lse * log2(e) per (head, query), padded to whole
// q-tiles with (-inf, 0) so that P = 0 there; the fp32 dq accumulator is
// cleared (one warp per (query, head) row of D elements, D / 32 per lane),
// and so are the fp32 dk / dv accumulators (kv4 float4 each).
template <int D>
__global__ void ffa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ dout,
                                   const float* __restrict__ lse, int32_t sq, int32_t sq_pad, int32_t hq,
                                   float* __restrict__ lse2, float* __restrict__ dvec, float* __restrict__ dq_acc,
                                   float4* __restrict__ dk_acc, float4* __restrict__ dv_acc, int64_t kv4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < kv4; i += (int64_t)gridDim.x * blockDim.x)
    dk_acc[i] = dv_acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  const int lane = threadIdx.x & 31;
  const int64_t n_rows = static_cast<int64_t>(sq_pad) * hq;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; w < n_rows;
       w += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int32_t q = static_cast<int32_t>(w / hq), h = static_cast<int32_t>(w % hq);
    float dsum = 0.f, l2 = -INFINITY;
    if (q < sq) {
      constexpr int E = D / 32;   // elements per lane: 4 or 2
      const int64_t row = (static_cast<int64_t>(q) * hq + h) * D;
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(out + row + lane * E);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(dout + row + lane * E);
      if constexpr (E == 4) {
        const uint2 o = *reinterpret_cast<const uint2*>(o2), g = *reinterpret_cast<const uint2*>(g2);
        const __nv_bfloat162* ov = reinterpret_cast<const __nv_bfloat162*>(&o);
        const __nv_bfloat162* gv = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float2 of = __bfloat1622float2(ov[i]), gf = __bfloat1622float2(gv[i]);
          dsum += of.x * gf.x + of.y * gf.y;
        }
        *reinterpret_cast<float4*>(dq_acc + row + lane * E) = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        const float2 of = __bfloat1622float2(*o2), gf = __bfloat1622float2(*g2);
        dsum += of.x * gf.x + of.y * gf.y;
        *reinterpret_cast<float2*>(dq_acc + row + lane * E) = make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int o_ = 16; o_ > 0; o_ >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o_);
      const float l = lse[static_cast<int64_t>(h) * sq + q];
      l2 = l == -INFINITY ? -INFINITY : -l * kLog2e;
    }
    if (lane == 0) {
      lse2[static_cast<int64_t>(h) * sq_pad + q] = l2;
      dvec[static_cast<int64_t>(h) * sq_pad + q] = q < sq ? dsum : 0.f;
    }
  }
}

// Gradient of the attention sink: dsink_h = -sum_i e^(sink_h - lse_i) D_i,
// the sink's softmax weight in row i times the row's D_i (the sink is one
// more logit whose value vector is zero).  One block per head; the block
// reduces the head's rows and writes the result, so no accumulator needs
// clearing and the sum does not depend on timing.
__global__ void __launch_bounds__(1024) ffa_bwd_dsink_kernel(const float* __restrict__ lse,
                                                             const float* __restrict__ dvec,
                                                             const float* __restrict__ sink, int32_t sq,
                                                             int32_t sq_pad, float* __restrict__ dsink) {
  __shared__ float part[32];
  const int h = blockIdx.x;
  const float s = sink[h];
  float acc = 0.f;
  for (int32_t i = threadIdx.x; i < sq; i += blockDim.x) {
    const float l = lse[static_cast<int64_t>(h) * sq + i];
    if (l != -INFINITY) acc += ex2_approx((s - l) * kLog2e) * dvec[static_cast<int64_t>(h) * sq_pad + i];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? part[threadIdx.x] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) dsink[h] = -v;
  }
}

// dq, dk, dv = bf16 of their fp32 accumulators (q4 float4 of dq, kv4 of dk
// and of dv).
__global__ void ffa_bwd_dq_kernel(const float4* __restrict__ dq_acc, const float4* __restrict__ dk_acc,
                                  const float4* __restrict__ dv_acc, uint2* __restrict__ dq, uint2* __restrict__ dk,
                                  uint2* __restrict__ dv, int64_t q4, int64_t kv4) {
  const int64_t n = q4 + 2 * kv4;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float4* src = i < q4 ? dq_acc + i : i < q4 + kv4 ? dk_acc + (i - q4) : dv_acc + (i - q4 - kv4);
    uint2* dst = i < q4 ? dq + i : i < q4 + kv4 ? dk + (i - q4) : dv + (i - q4 - kv4);
    const float4 v = *src;
    *dst = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace ffa

using namespace ffa;

// Workspace: dq accumulator [sq][hq][d], -lse * log2(e) and D [hq][sq_pad],
// dk and dv accumulators [sk][hkv][d], all fp32, each 256-byte aligned.
extern "C" size_t ffa_bwd_workspace_size(int64_t seqlen_q, int64_t seqlen_k, int32_t hq, int32_t hkv, int32_t d) {
  if (seqlen_q < 0 || seqlen_k < 0 || hq <= 0 || hkv <= 0 || d <= 0) return 0;
  const int64_t sq_pad = (seqlen_q + 127) / 128 * 128;
  return align256(static_cast<size_t>(seqlen_q) * hq * d * 4) + 2 * align256(static_cast<size_t>(sq_pad) * hq * 4) +
         2 * align256(static_cast<size_t>(seqlen_k) * hkv * d * 4);
}

namespace {
ffa_status bwd_impl(const void* q, const void* k, const void* v, const void* out, const float* lse, const void* dout,
                    int64_t seqlen_q, int64_t seqlen_k, int32_t hq, int32_t hkv, int32_t d, ffa_plan_t plan,
                    float scale, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, void* stream,
                    const float* sink, float* dsink) {
  if (!plan || !q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return FFA_ERR_INVALID_ARG;
  if ((sink == nullptr) != (dsink == nullptr)) return FFA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return FFA_ERR_INVALID_ARG;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return FFA_ERR_INVALID_ARG;
  if (seqlen_q != plan->seqlen_q || seqlen_k != plan->seqlen_k) return FFA_ERR_INVALID_ARG;
  if (d != 128 && d != 64) return FFA_ERR_UNSUPPORTED;
  if (plan->tiles.bwd_bm != 128 || plan->tiles.bwd_bn != 128) return FFA_ERR_UNSUPPORTED;
  if (workspace_bytes < ffa_bwd_workspace_size(seqlen_q, seqlen_k, hq, hkv, d)) return FFA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FFA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (seqlen_q == 0 || seqlen_k == 0) {
    cudaError_t e = cudaSuccess;
    if (seqlen_k > 0) {
      e = cudaMemsetAsync(dk, 0, static_cast<size_t>(seqlen_k) * hkv * d * 2, st);
      if (e == cudaSuccess) e = cudaMemsetAsync(dv, 0, static_cast<size_t>(seqlen_k) * hkv * d * 2, st);
    }
    if (seqlen_q > 0 && e == cudaSuccess) e = cudaMemsetAsync(dq, 0, static_cast<size_t>(seqlen_q) * hq * d * 2, st);
    // no row has a key, so every row's out is 0 and D_i = 0: the sink gets no gradient
    if (dsink && e == cudaSuccess) e = cudaMemsetAsync(dsink, 0, static_cast<size_t>(hq) * 4, st);
    return cuda_status(e);
  }
  const int32_t sq_pad = static_cast<int32_t>((seqlen_q + 127) / 128 * 128);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* dq_acc = reinterpret_cast<float*>(ws);
  float* lse2 = reinterpret_cast<float*>(ws + align256(static_cast<size_t>(seqlen_q) * hq * d * 4));
  float* dvec = lse2 + align256(static_cast<size_t>(sq_pad) * hq * 4) / 4;
  float* dk_acc = dvec + align256(static_cast<size_t>(sq_pad) * hq * 4) / 4;
  float* dv_acc = dk_acc + align256(static_cast<size_t>(seqlen_k) * hkv * d * 4) / 4;
  const int64_t kv4 = seqlen_k * hkv * d / 4;

  CUtensorMap mq, mk, mv, mdo, mdq;
  if (!make_tile_map(&mq, q, seqlen_q, hq, d, kHalf) || !make_tile_map(&mk, k, seqlen_k, hkv, d) ||
      !make_tile_map(&mv, v, seqlen_k, hkv, d) || !make_tile_map(&mdo, dout, seqlen_q, hq, d, kHalf) ||
      !make_f32_row_map(&mdq, dq_acc, seqlen_q, hq, d, kDqRows))
    return FFA_ERR_CUDA;

  const int sms = plan->num_sms;
  {
    const int64_t warps = static_cast<int64_t>(sq_pad) * hq;
    const int blocks = static_cast<int>(std::min<int64_t>((warps * 32 + 255) / 256, static_cast<int64_t>(sms) * 16));
    ScopedKernelTimer tk(&plan->timer, FFA_KERNEL_BWD_PRE, st);
    auto pre = d == 128 ? ffa_bwd_pre_kernel<128> : ffa_bwd_pre_kernel<64>;
    pre<<<blocks, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse,
                                static_cast<int32_t>(seqlen_q), sq_pad, hq, lse2, dvec, dq_acc,
                                reinterpret_cast<float4*>(dk_acc), reinterpret_cast<float4*>(dv_acc), kv4);
    if (sink)
      ffa_bwd_dsink_kernel<<<hq, 1024, 0, st>>>(lse, dvec, sink, static_cast<int32_t>(seqlen_q), sq_pad, dsink);
  }
  BwdParams prm;
  prm.items = plan->k2q.items;
  prm.full_idx = plan->k2q.full_idx;
  prm.mask_idx = plan->k2q.mask_idx;
  prm.full_off = plan->k2q.full_off;
  prm.mask_off = plan->k2q.mask_off;
  prm.kiv_off = plan->k2q.iv_off;
  prm.kiv = plan->k2q.iv;
  prm.lse2 = lse2;
  prm.dvec = dvec;
  prm.dk_acc = dk_acc;
  prm.dv_acc = dv_acc;
  prm.seqlen_q = static_cast<int32_t>(seqlen_q);
  prm.seqlen_k = static_cast<int32_t>(seqlen_k);
  prm.sq_pad = sq_pad;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.group = hq / hkv;
  prm.n_units = plan->k2q.n_items * hkv;
  prm.scale = scale;
  prm.scale_log2 = scale * kLog2e;
  prm.status = &plan->words->status;
  auto main_kernel = d == 128 ? ffa_bwd_main_kernel<128> : ffa_bwd_main_kernel<64>;
  // Set on every launch (per context, cheap, thread-safe; see launch_fwd).
  if (cudaFuncSetAttribute(main_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kBwdSmem)) !=
      cudaSuccess)
    return FFA_ERR_CUDA;
  if (prm.n_units > INT32_MAX) return FFA_ERR_OVERFLOW;
  const int grid = static_cast<int>(std::min<int64_t>(prm.n_units, sms));
  prm.trace = plan->trace.begin(FFA_KERNEL_BWD_MAIN, grid);
  prm.next = &plan->words->bwd_next;
  if (cudaMemsetAsync(prm.next, 0, sizeof(uint32_t), st) != cudaSuccess) return FFA_ERR_CUDA;
  if (grid > 0) {   // no units: the mask is empty and the cleared accumulators are the result
    ScopedKernelTimer tk(&plan->timer, FFA_KERNEL_BWD_MAIN, st);
    main_kernel<<<grid, kBwdThreads, kBwdSmem, st>>>(prm, mq, mk, mv, mdo, mdq);
  }
  {
    const int64_t q4 = seqlen_q * hq * d / 4;
    const int blocks =
        static_cast<int>(std::min<int64_t>((q4 + 2 * kv4 + 255) / 256, static_cast<int64_t>(sms) * 16));
    ScopedKernelTimer tk(&plan->timer, FFA_KERNEL_BWD_DQ, st);
    ffa_bwd_dq_kernel<<<blocks, 256, 0, st>>>(
        reinterpret_cast<const float4*>(dq_acc), reinterpret_cast<const float4*>(dk_acc),
        reinterpret_cast<const float4*>(dv_acc), static_cast<uint2*>(dq), static_cast<uint2*>(dk),
        static_cast<uint2*>(dv), q4, kv4);
  }
  return cuda_status(cudaGetLastError());
}
}  // namespace

extern "C" ffa_status ffa_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                              const void* dout, int64_t seqlen_q, int64_t seqlen_k, int32_t hq, int32_t hkv, int32_t d,
                              ffa_plan_t plan, float scale, void* dq, void* dk, void* dv, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, out, lse, dout, seqlen_q, seqlen_k, hq, hkv, d, plan, scale, dq, dk, dv, workspace,
                  workspace_bytes, stream, nullptr, nullptr);
}

extern "C" ffa_status ffa_bwd_sink(const void* q, const void* k, const void* v, const void* out, const float* lse,
                                   const void* dout, int64_t seqlen_q, int64_t seqlen_k, int32_t hq, int32_t hkv,
                                   int32_t d, ffa_plan_t plan, float scale, const float* sink, void* dq, void* dk,
                                   void* dv, float* dsink, void* workspace, size_t workspace_bytes, void* stream) {
  if (!sink || !dsink) return FFA_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, out, lse, dout, seqlen_q, seqlen_k, hq, hkv, d, plan, scale, dq, dk, dv, workspace,
                  workspace_bytes, stream, sink, dsink);
}

// ---------------------------------------------------------------------------
// Backward pass without device allocation: the scratch lives in a fixed
// file-scope device array.  Host code must not use the array's name as an
// address (it is a host-side stand-in): every call looks up the array's
// device address in the current context with cudaGetSymbolAddress, a host-side
// lookup once the module is loaded, so the address is never stale (after a
// device reset, or on another device).
// ---------------------------------------------------------------------------
namespace ffa {
namespace {
static __device__ __align__(256) uint8_t g_bwd_noalloc_scratch[FFA_BWD_NOALLOC_SCRATCH_BYTES];
}  // namespace
}  // namespace ffa

extern "C" ffa_status ffa_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                                      const float* lse, const void* dout, int64_t seqlen_q, int64_t seqlen_k,
                                      int32_t hq, int32_t hkv, int32_t d, ffa_plan_t plan, float scale, void* dq,
                                      void* dk, void* dv, void* stream) {
  const size_t need = ffa_bwd_workspace_size(seqlen_q, seqlen_k, hq, hkv, d);
  if (need > FFA_BWD_NOALLOC_SCRATCH_BYTES) return FFA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, ffa::g_bwd_noalloc_scratch) != cudaSuccess || !scratch) return FFA_ERR_CUDA;
  return ffa_bwd(q, k, v, out, lse, dout, seqlen_q, seqlen_k, hq, hkv, d, plan, scale, dq, dk, dv, scratch,
                 FFA_BWD_NOALLOC_SCRATCH_BYTES, stream);
}
static_assert(offsetof(ffa::BwdBars, nl) % 16 == 0 && offsetof(ffa::BwdBars, dv) % 16 == 0,
              "bulk-copy targets must be 16-byte aligned");
