// Block-mask planner: per-row allowed intervals, Full / Partial / Empty block
// classification in CSR form, and the longest-work-first tile order.
//
// MagiAttention documentation, "FFA_FA4 backend": item 1 (create_block_mask
// classifies blocks as Full, Partial or Empty, in q2k order for the forward
// and k2q order for the backward; blocks out of bounds only along q count as
// Full in the forward) and item 2 (the metadata is stored in CSR form,
// full_block_offset / mask_block_offset, holding only non-empty blocks).
// The tile order follows the greedy of the blog's "Dispatch Solver" section
// (heaviest item first to the least-loaded worker), applied to SMs.
//
// All kernels are integer-only.  One direction (q2k or k2q) is built by the
// same code: k2q runs it on the transposed band slices.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "ffa_internal.h"

namespace ffa {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kSweepThreads = 256;
constexpr int kSweepStage = 2048;   // intervals staged in shared memory per row-tile
constexpr int kSweepWin = 2048;     // column tiles counted in shared memory at a time
constexpr int kItemThreads = 256;
static_assert(kSweepWin % kSweepThreads == 0, "whole scan entries per thread");

__device__ __forceinline__ void row_interval(const BandSlice& s, int64_t row, int64_t& lo, int64_t& hi) {
  const int64_t r = row - s.r_start;
  const int64_t lc = s.c_end - s.c_start;
  int64_t a = r + s.d_lo;
  int64_t b = r + s.d_hi + 1;
  a = a < 0 ? 0 : a;
  b = b > lc ? lc : b;
  lo = s.c_start + a;
  hi = s.c_start + b;
}

// Candidate slices of every row-tile (slices whose row range meets the tile).
// One thread per (slice, row-tile) pair: slices along the grid's y, each
// slice's row tiles along x.  The order of a tile's candidates depends on the
// atomics; the per-row intervals built from them are sorted afterwards.
template <bool FILL>
__global__ void cand_kernel(const BandSlice* __restrict__ slices, int64_t n, int32_t tile_r, int32_t* cnt_or_cursor,
                            const int32_t* __restrict__ off, int32_t* __restrict__ cand) {
  for (int64_t i = blockIdx.y; i < n; i += gridDim.y) {
    const BandSlice s = slices[i];
    const int64_t t0 = s.r_start / tile_r, t1 = (s.r_end - 1) / tile_r;
    for (int64_t t = t0 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t <= t1;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
      const int32_t k = atomicAdd(&cnt_or_cursor[t], 1);
      if (FILL) cand[off[t] + k] = static_cast<int32_t>(i);
    }
  }
}

// Single-block exclusive scan of n int32 counts into out[0..n] (out[n] = total).
// The int64 total is also stored to *total (for overflow checks on the host).
__global__ void __launch_bounds__(kScanThreads) scan_kernel(const int32_t* __restrict__ in, int64_t n,
                                                            int32_t* __restrict__ out, int64_t* __restrict__ total) {
  __shared__ int64_t part[kScanThreads];
  const int64_t chunk = (n + kScanThreads - 1) / kScanThreads;
  const int64_t b = threadIdx.x * chunk;
  const int64_t e = b + chunk < n ? b + chunk : n;
  int64_t sum = 0;
  for (int64_t i = b; i < e; ++i) sum += in[i];
  part[threadIdx.x] = sum;
  __syncthreads();
  for (int ofs = 1; ofs < kScanThreads; ofs <<= 1) {
    int64_t v = threadIdx.x >= ofs ? part[threadIdx.x - ofs] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int64_t run = part[threadIdx.x] - sum;
  for (int64_t i = b; i < e; ++i) {
    out[i] = static_cast<int32_t>(run);
    run += in[i];
  }
  if (threadIdx.x == kScanThreads - 1) {
    out[n] = static_cast<int32_t>(part[kScanThreads - 1]);
    *total = part[kScanThreads - 1];
  }
}

// Exclusive scan for long inputs (the per-row interval counts), in three
// launches: each block sums its contiguous segment (int64); one block turns
// the segment sums into offsets and the int64 total; each block rescans its
// segment tile by tile (coalesced loads, warp-shuffle scans) from its
// segment's offset.  Same result as scan_kernel.
constexpr int kScanSegments = 1024;

__global__ void __launch_bounds__(kScanThreads) segment_sum_kernel(const int32_t* __restrict__ in, int64_t n,
                                                                   int64_t* __restrict__ seg_sum) {
  const int64_t seg = (n + gridDim.x - 1) / gridDim.x;
  const int64_t b = blockIdx.x * seg, e = b + seg < n ? b + seg : n;
  int64_t sum = 0;
  for (int64_t i = b + threadIdx.x; i < e; i += kScanThreads) sum += in[i];
  __shared__ int64_t part[kScanThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = sum;
  __syncthreads();
  if (threadIdx.x < 32) {
    int64_t v = part[threadIdx.x];   // kScanThreads / 32 == 32 warps
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) seg_sum[blockIdx.x] = v;
  }
}

// One block, one thread per segment: seg_off[k] = sum of segments < k,
// seg_off[n_seg] and *total = the sum of all.
__global__ void __launch_bounds__(kScanThreads) segment_offsets_kernel(const int64_t* __restrict__ seg_sum,
                                                                       int32_t n_seg, int32_t* __restrict__ seg_off,
                                                                       int64_t* __restrict__ total) {
  __shared__ int64_t part[kScanThreads];
  const int t = threadIdx.x;
  const int64_t x = t < n_seg ? seg_sum[t] : 0;
  part[t] = x;
  __syncthreads();
  for (int ofs = 1; ofs < kScanThreads; ofs <<= 1) {
    const int64_t v = t >= ofs ? part[t - ofs] : 0;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  if (t < n_seg) seg_off[t] = static_cast<int32_t>(part[t] - x);
  if (t == kScanThreads - 1) {
    seg_off[n_seg] = static_cast<int32_t>(part[t]);
    *total = part[t];
  }
}

__global__ void __launch_bounds__(kScanThreads) segment_scan_kernel(const int32_t* __restrict__ in, int64_t n,
                                                                    const int32_t* __restrict__ seg_off,
                                                                    int32_t* __restrict__ out) {
  const int64_t seg = (n + gridDim.x - 1) / gridDim.x;
  const int64_t b = blockIdx.x * seg, e = b + seg < n ? b + seg : n;
  __shared__ int32_t warp_off[kScanThreads / 32];
  __shared__ int32_t tile_sum;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int32_t carry = seg_off[blockIdx.x];
  for (int64_t base = b; base < e; base += kScanThreads) {
    const int64_t i = base + threadIdx.x;
    const int32_t x = i < e ? in[i] : 0;
    int32_t incl = x;   // inclusive scan inside the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_off[w] = incl;   // the warp's total
    __syncthreads();
    if (w == 0) {   // warp totals -> exclusive warp offsets, and the tile's total
      const int32_t t = warp_off[lane];
      int32_t ti = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, ti, o);
        if (lane >= o) ti += y;
      }
      warp_off[lane] = ti - t;
      if (lane == 31) tile_sum = ti;
    }
    __syncthreads();
    if (i < e) out[i] = carry + warp_off[w] + incl - x;
    carry += tile_sum;
    __syncthreads();   // warp_off and tile_sum are rewritten by the next tile
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) out[n] = seg_off[gridDim.x];
}

// Per-row allowed column intervals: count, then fill + sort by lo.
template <bool FILL>
__global__ void iv_kernel(const BandSlice* __restrict__ slices, const int32_t* __restrict__ cand_off,
                          const int32_t* __restrict__ cand, int64_t n_rows, int32_t tile_r, int32_t* __restrict__ cnt,
                          const int32_t* __restrict__ iv_off, int32_t* __restrict__ iv) {
  for (int64_t row = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; row < n_rows;
       row += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = row / tile_r;
    int32_t c = 0;
    int32_t* dst = FILL ? iv + 2 * static_cast<int64_t>(iv_off[row]) : nullptr;
    for (int32_t k = cand_off[t]; k < cand_off[t + 1]; ++k) {
      const BandSlice s = slices[cand[k]];
      if (row < s.r_start || row >= s.r_end) continue;
      int64_t lo, hi;
      row_interval(s, row, lo, hi);
      if (lo >= hi) continue;
      if (FILL) {
        dst[2 * c] = static_cast<int32_t>(lo);
        dst[2 * c + 1] = static_cast<int32_t>(hi);
      }
      ++c;
    }
    if (!FILL) {
      cnt[row] = c;
    } else {
      for (int32_t i = 1; i < c; ++i) {   // insertion sort by lo (a row has few intervals)
        const int32_t lo = dst[2 * i], hi = dst[2 * i + 1];
        int32_t j = i - 1;
        while (j >= 0 && dst[2 * j] > lo) {
          dst[2 * j + 2] = dst[2 * j];
          dst[2 * j + 3] = dst[2 * j + 1];
          --j;
        }
        dst[2 * j + 2] = lo;
        dst[2 * j + 3] = hi;
      }
    }
  }
}

struct SweepArgs {
  int64_t n_rows, n_cols;
  int32_t tile_r, tile_c, n_rt;
  int32_t k2q;
  const int32_t* iv_off;
  const int32_t* iv;
  // k2q only (else 0 / null): column tiles per backward q-chunk (log2), and
  // the count pass adds the (row tile, chunk) pairs with a non-empty block,
  // the backward's work items, to *items.
  int32_t chunk_log2;
  unsigned long long* items;
};
constexpr int kSweepChunks = kSweepWin >> kBwdChunkLog2;   // q-chunks in one window
static_assert(kSweepWin % (1 << kBwdChunkLog2) == 0 && kBwdChunkLog2 >= 5, "windows hold whole q-chunks");

// One block per row-tile: count the allowed elements of every column tile
// between the smallest and largest allowed column of the tile's rows,
// classify, and (FILL) write the Full and Partial lists in ascending order.
//
// The counts come from the tile's row intervals in O(#intervals + #column
// tiles): an interval [lo, hi) covers its first and last column tiles in
// part (exact overlaps, added to s_edge) and every tile strictly between them
// whole (tile_c each, added as +tile_c / -tile_c to a difference array whose
// prefix sum gives the per-tile cover).  The column range is processed in
// windows of kSweepWin tiles held in shared memory.
template <bool FILL>
__global__ void __launch_bounds__(kSweepThreads) sweep_kernel(SweepArgs a, int32_t* __restrict__ n_full,
                                                              int32_t* __restrict__ n_mask,
                                                              const int32_t* __restrict__ full_off,
                                                              const int32_t* __restrict__ mask_off,
                                                              int32_t* __restrict__ full_idx,
                                                              int32_t* __restrict__ mask_idx) {
  __shared__ int32_t s_iv[2 * kSweepStage];
  __shared__ int32_t s_cnt[kSweepWin + 1];   // difference array, then the whole-tile cover
  __shared__ int32_t s_edge[kSweepWin];      // partial covers of the intervals' end tiles
  __shared__ int32_t s_wf[kSweepThreads / 32], s_wm[kSweepThreads / 32];
  __shared__ int32_t s_lo[kSweepThreads / 32], s_hi[kSweepThreads / 32];
  __shared__ int32_t s_chunk[kSweepChunks];   // q-chunks of the window with a non-empty block
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nw = kSweepThreads / 32;
  constexpr int kPer = kSweepWin / kSweepThreads;   // scan entries per thread
  const int64_t tc = a.tile_c;
  const bool count_items = !FILL && a.items != nullptr;

  for (int32_t rt = blockIdx.x; rt < a.n_rt; rt += gridDim.x) {
    const int64_t r0 = static_cast<int64_t>(rt) * a.tile_r;
    const int64_t r1 = r0 + a.tile_r < a.n_rows ? r0 + a.tile_r : a.n_rows;
    const int32_t e0 = a.iv_off[r0], e1 = a.iv_off[r1];
    const int32_t ne = e1 - e0;
    if (ne == 0) {
      if (!FILL && tid == 0) n_full[rt] = n_mask[rt] = 0;
      continue;
    }
    const bool staged = ne <= kSweepStage;
    int32_t lo_min = INT32_MAX, hi_max = INT32_MIN;
    for (int32_t e = tid; e < ne; e += kSweepThreads) {
      const int32_t lo = a.iv[2 * (int64_t)(e0 + e)], hi = a.iv[2 * (int64_t)(e0 + e) + 1];
      lo_min = min(lo_min, lo);
      hi_max = max(hi_max, hi);
      if (staged) {
        s_iv[2 * e] = lo;
        s_iv[2 * e + 1] = hi;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo_min = min(lo_min, __shfl_xor_sync(0xffffffffu, lo_min, o));
      hi_max = max(hi_max, __shfl_xor_sync(0xffffffffu, hi_max, o));
    }
    if (lane == 0) {
      s_lo[warp] = lo_min;
      s_hi[warp] = hi_max;
    }
    __syncthreads();
    lo_min = s_lo[0];
    hi_max = s_hi[0];
    for (int w = 1; w < nw; ++w) {
      lo_min = min(lo_min, s_lo[w]);
      hi_max = max(hi_max, s_hi[w]);
    }
    const int32_t ct0 = lo_min / a.tile_c, ct1 = (hi_max - 1) / a.tile_c;
    const int64_t nr = r1 - r0;
    const bool row_oob = r0 + a.tile_r > a.n_rows;
    int32_t cur_f = FILL ? full_off[rt] : 0, cur_m = FILL ? mask_off[rt] : 0;
    int32_t tot_f = 0, tot_m = 0;
    int64_t items_rt = 0;   // thread 0: q-chunks of this row tile with a non-empty block
    // windows start on a q-chunk boundary when items are counted, so that no
    // chunk straddles two windows (the tiles before ct0 are empty)
    const int32_t wbeg = count_items ? (ct0 & ~((1 << a.chunk_log2) - 1)) : ct0;
    for (int32_t w0 = wbeg; w0 <= ct1; w0 += kSweepWin) {
      const int32_t w1 = min(ct1, w0 + kSweepWin - 1);
      const int32_t nwin = w1 - w0 + 1;
      for (int32_t i = tid; i <= nwin; i += kSweepThreads) {
        s_cnt[i] = 0;
        if (i < nwin) s_edge[i] = 0;
      }
      for (int32_t i = tid; i < kSweepChunks; i += kSweepThreads) s_chunk[i] = 0;
      __syncthreads();
      for (int32_t e = tid; e < ne; e += kSweepThreads) {
        const int64_t lo = staged ? s_iv[2 * e] : a.iv[2 * (int64_t)(e0 + e)];
        const int64_t hi = staged ? s_iv[2 * e + 1] : a.iv[2 * (int64_t)(e0 + e) + 1];
        if (hi <= lo) continue;
        const int32_t ta = static_cast<int32_t>(lo / tc), tb = static_cast<int32_t>((hi - 1) / tc);
        if (tb < w0 || ta > w1) continue;
        if (ta == tb) {
          atomicAdd(&s_edge[ta - w0], static_cast<int32_t>(hi - lo));
          continue;
        }
        if (ta >= w0) atomicAdd(&s_edge[ta - w0], static_cast<int32_t>((ta + 1) * tc - lo));
        if (tb <= w1) atomicAdd(&s_edge[tb - w0], static_cast<int32_t>(hi - tb * tc));
        const int32_t i0 = max(ta + 1, w0), i1 = min(tb - 1, w1);
        if (i0 <= i1) {
          atomicAdd(&s_cnt[i0 - w0], static_cast<int32_t>(tc));
          atomicAdd(&s_cnt[i1 - w0 + 1], -static_cast<int32_t>(tc));
        }
      }
      __syncthreads();
      {   // inclusive prefix sum of s_cnt[0, nwin): kPer consecutive entries per thread
        int32_t v[kPer];
        int32_t run = 0;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int32_t i = tid * kPer + k;
          run += i < nwin ? s_cnt[i] : 0;
          v[k] = run;
        }
        int32_t x = run;   // inclusive scan of the threads' totals
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
          if (lane >= o) x += y;
        }
        if (lane == 31) s_wf[warp] = x;
        __syncthreads();
        int32_t before = x - run;
        for (int w = 0; w < warp; ++w) before += s_wf[w];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int32_t i = tid * kPer + k;
          if (i < nwin) s_cnt[i] = v[k] + before;
        }
        __syncthreads();
      }
      for (int32_t base = w0; base <= w1; base += kSweepThreads) {
        const int32_t ct = base + tid;
        bool is_f = false, is_m = false;
        if (ct <= w1) {
          const int64_t c0 = static_cast<int64_t>(ct) * tc;
          const int64_t c1 = c0 + tc < a.n_cols ? c0 + tc : a.n_cols;
          const int64_t cnt = static_cast<int64_t>(s_cnt[ct - w0]) + s_edge[ct - w0];
          const bool col_oob = c0 + tc > a.n_cols;
          const bool full_ok = !col_oob && (!a.k2q || !row_oob);
          if (cnt > 0) {
            is_f = (cnt == nr * (c1 - c0)) && full_ok;
            is_m = !is_f;
          }
        }
        const uint32_t bf = __ballot_sync(0xffffffffu, is_f), bm = __ballot_sync(0xffffffffu, is_m);
        if (lane == 0) {
          s_wf[warp] = __popc(bf);
          s_wm[warp] = __popc(bm);
        }
        __syncthreads();
        int32_t pf = __popc(bf & ((1u << lane) - 1)), pm = __popc(bm & ((1u << lane) - 1));
        int32_t rf = 0, rm = 0;
        for (int w = 0; w < nw; ++w) {
          if (w < warp) {
            pf += s_wf[w];
            pm += s_wm[w];
          }
          rf += s_wf[w];
          rm += s_wm[w];
        }
        if (FILL) {
          if (is_f) full_idx[cur_f + pf] = ct;
          if (is_m) mask_idx[cur_m + pm] = ct;
        }
        if (count_items && (is_f || is_m)) s_chunk[(ct - w0) >> a.chunk_log2] = 1;
        cur_f += rf;
        cur_m += rm;
        tot_f += rf;
        tot_m += rm;
        __syncthreads();
      }
      if (count_items) {
        if (warp == 0) {
          int32_t c = 0;
          for (int32_t i = lane; i < kSweepChunks; i += 32) c += s_chunk[i];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
          if (lane == 0) items_rt += c;
        }
        __syncthreads();
      }
    }
    if (count_items && tid == 0 && items_rt > 0) atomicAdd(a.items, static_cast<unsigned long long>(items_rt));
    if (!FILL && tid == 0) {
      n_full[rt] = tot_f;
      n_mask[rt] = tot_m;
    }
    __syncthreads();
  }
}

__device__ __forceinline__ uint64_t lpt_key(const int32_t* full_off, const int32_t* mask_off, int32_t t) {
  const int64_t cost = static_cast<int64_t>(kCostFull) * (full_off[t + 1] - full_off[t]) +
                       static_cast<int64_t>(kCostMask) * (mask_off[t + 1] - mask_off[t]);
  const int64_t c = cost < 0x7FFFFFFF ? cost : 0x7FFFFFFF;
  return (static_cast<uint64_t>(0x7FFFFFFF - c) << 32) | static_cast<uint32_t>(t);
}

// Longest-work-first order by bitonic sort of (cost desc, index asc) keys.
// In shared memory when the padded size fits, else one launch per merge step.
__global__ void __launch_bounds__(1024) lpt_sort_smem_kernel(const int32_t* __restrict__ full_off,
                                                             const int32_t* __restrict__ mask_off, int32_t n,
                                                             int32_t n_pad, int32_t* __restrict__ order) {
  extern __shared__ uint64_t keys[];
  for (int32_t i = threadIdx.x; i < n_pad; i += blockDim.x) keys[i] = i < n ? lpt_key(full_off, mask_off, i) : ~0ull;
  __syncthreads();
  for (int32_t k = 2; k <= n_pad; k <<= 1) {
    for (int32_t j = k >> 1; j > 0; j >>= 1) {
      for (int32_t i = threadIdx.x; i < n_pad; i += blockDim.x) {
        const int32_t p = i ^ j;
        if (p > i) {
          const bool up = (i & k) == 0;
          const uint64_t x = keys[i], y = keys[p];
          if ((x > y) == up) {
            keys[i] = y;
            keys[p] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int32_t i = threadIdx.x; i < n; i += blockDim.x) order[i] = static_cast<int32_t>(keys[i] & 0xffffffffu);
}

__global__ void lpt_keys_kernel(const int32_t* __restrict__ full_off, const int32_t* __restrict__ mask_off, int32_t n,
                                int32_t n_pad, uint64_t* __restrict__ keys) {
  for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n_pad; i += gridDim.x * blockDim.x)
    keys[i] = i < n ? lpt_key(full_off, mask_off, i) : ~0ull;
}
__global__ void bitonic_step_kernel(uint64_t* __restrict__ keys, int32_t n_pad, int32_t k, int32_t j) {
  for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n_pad; i += gridDim.x * blockDim.x) {
    const int32_t p = i ^ j;
    if (p > i) {
      const bool up = (i & k) == 0;
      const uint64_t x = keys[i], y = keys[p];
      if ((x > y) == up) {
        keys[i] = y;
        keys[p] = x;
      }
    }
  }
}
__global__ void lpt_order_kernel(const uint64_t* __restrict__ keys, int32_t n, int32_t* __restrict__ order) {
  for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    order[i] = static_cast<int32_t>(keys[i] & 0xffffffffu);
}

// ---------------------------------------------------------------------------
// Backward work items.  A k-tile's k2q lists are cut into q-chunks of
// 2^log2c consecutive q-tiles; an item is one (k-tile, chunk) pair with
// blocks.  Items are ordered chunk by chunk, and inside a chunk by the
// k-tiles' longest-work-first rank, so that the items running at one time
// read the same chunk's Q / dO rows and add into the same dq rows.
// ---------------------------------------------------------------------------
// First index in the ascending list a[lo, hi) whose value is >= v.
__device__ __forceinline__ int32_t lower_bound_i32(const int32_t* a, int32_t lo, int32_t hi, int32_t v) {
  while (lo < hi) {
    const int32_t mid = lo + ((hi - lo) >> 1);
    if (a[mid] < v) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// One block per q-chunk c: walk the k-tiles in their longest-work-first
// order and take those with a block of either k2q list among the chunk's
// q-tiles [c << log2c, (c + 1) << log2c), in that order.  !FILL: count them;
// FILL: write their items {k-tile, first Full index, first Partial index,
// #Full | #Partial << 16} from the chunk's item offset.  The result is the
// items sorted by (chunk, rank), without a sort.
template <bool FILL>
__global__ void __launch_bounds__(kItemThreads) chunk_items_kernel(
    const int32_t* __restrict__ full_off, const int32_t* __restrict__ full_idx, const int32_t* __restrict__ mask_off,
    const int32_t* __restrict__ mask_idx, const int32_t* __restrict__ order, int32_t n_rt, int32_t n_chunks,
    int32_t log2c, const int32_t* __restrict__ item_off, int32_t* __restrict__ cnt, int4* __restrict__ items,
    int64_t n_items) {
  __shared__ int32_t s_w[kItemThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nw = kItemThreads / 32;
  for (int32_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
    const int32_t lo = c << log2c, hi = (c + 1) << log2c;
    int32_t cur = FILL ? item_off[c] : 0, total = 0;
    for (int32_t base = 0; base < n_rt; base += kItemThreads) {
      const int32_t r = base + tid;
      bool has = false;
      int4 it = make_int4(0, 0, 0, 0);
      if (r < n_rt) {
        const int32_t kt = order[r];
        const int32_t f0 = full_off[kt], f1 = full_off[kt + 1], m0 = mask_off[kt], m1 = mask_off[kt + 1];
        // the k-tile's q-tiles span [qmin, qmax]; search its lists only when that meets the chunk
        const int32_t qmin = min(f1 > f0 ? full_idx[f0] : INT32_MAX, m1 > m0 ? mask_idx[m0] : INT32_MAX);
        const int32_t qmax = max(f1 > f0 ? full_idx[f1 - 1] : -1, m1 > m0 ? mask_idx[m1 - 1] : -1);
        if (qmin < hi && qmax >= lo) {
          const int32_t fa = lower_bound_i32(full_idx, f0, f1, lo);
          const int32_t ma = lower_bound_i32(mask_idx, m0, m1, lo);
          has = (fa < f1 && full_idx[fa] < hi) || (ma < m1 && mask_idx[ma] < hi);
          if (FILL && has) {
            const int32_t fb = lower_bound_i32(full_idx, fa, f1, hi), mb = lower_bound_i32(mask_idx, ma, m1, hi);
            it = make_int4(kt, fa, ma, (fb - fa) | ((mb - ma) << 16));
          }
        }
      }
      const uint32_t bits = __ballot_sync(0xffffffffu, has);
      if (lane == 0) s_w[warp] = __popc(bits);
      __syncthreads();
      int32_t pos = __popc(bits & ((1u << lane) - 1u)), all = 0;
      for (int w = 0; w < nw; ++w) {
        if (w < warp) pos += s_w[w];
        all += s_w[w];
      }
      if (FILL && has && cur + pos < n_items) items[cur + pos] = it;   // n_items: the array's size
      cur += all;
      total += all;
      __syncthreads();
    }
    if (!FILL && tid == 0) cnt[c] = total;
  }
}

// ---------------------------------------------------------------------------
// Small plans in one launch.  When both sequence lengths are at most
// kSmallLen and there are at most kSmallSlices slices, one block per
// direction builds that direction's whole metadata: the per-row intervals
// (each slice's interval of every row, sorted by lo), the Full / Partial /
// Empty class of every block (by summing interval overlaps over the block's
// rows, with the same out-of-bounds rules), the CSR lists, the longest-work-
// first order and (k2q) the backward work items.  The arrays are sized from
// upper bounds, so the plan waits for nothing but the end; the totals go to
// the host through the mapped channel.  The results are the general path's
// (the tests compare both with the oracle).  A mask this small spends its
// plan time on launches and synchronizations, not on work.
// ---------------------------------------------------------------------------
constexpr int kSmallLen = 2048;
constexpr int kSmallSlices = 256;
constexpr int kSmallThreads = 1024;
constexpr int kSmallTiles = kSmallLen / 8;           // row or column tiles at the smallest tile, 8
constexpr int kSmallChunks = kSmallTiles >> kBwdChunkLog2;

struct SmallDir {
  const BandSlice* slices;   // host-mapped, n_slices
  int32_t n_slices, n_rows, n_cols, tile_r, tile_c, n_rt, n_ct, k2q, chunk_log2;
  int32_t *iv_off, *iv, *full_off, *full_idx, *mask_off, *mask_idx, *order;
  int4* items;
  int64_t* totals;   // host-mapped: [intervals, Full, Partial, items]
};
struct SmallArgs {
  SmallDir d[2];
  uint32_t* words;   // the plan's device words, cleared by block 0
  int32_t n_words;
};

// Dynamic shared memory of small_plan_kernel.
struct SmallSmem {
  int32_t row_off[kSmallLen + 1];
  int32_t nf[kSmallTiles], nm[kSmallTiles];
  int32_t foff[kSmallTiles + 1], moff[kSmallTiles + 1];
  int32_t pf[kSmallTiles][kSmallChunks + 1], pm[kSmallTiles][kSmallChunks + 1];   // chunk prefix counts
  int32_t ccnt[kSmallChunks], coff[kSmallChunks + 1];
  uint64_t keys[kSmallTiles];
  BandSlice sl[kSmallSlices];                // the slices, read once from host-mapped memory
  uint8_t cls[kSmallTiles * kSmallTiles];   // EMPTY 0, PARTIAL 1, FULL 2
};

// Exclusive scan of a[0, n) in place (a[n] = total), n <= 2 * kSmallThreads.
__device__ void small_scan(int32_t* a, int32_t n, int32_t* warp_tot) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t i0 = 2 * tid, i1 = 2 * tid + 1;
  const int32_t x0 = i0 < n ? a[i0] : 0, x1 = i1 < n ? a[i1] : 0;
  int32_t incl = x0 + x1;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int32_t t = warp_tot[lane];
    int32_t ti = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, ti, o);
      if (lane >= o) ti += y;
    }
    warp_tot[lane] = ti - t;
    if (lane == 31) warp_tot[32] = ti;
  }
  __syncthreads();
  const int32_t ex = warp_tot[warp] + incl - x0 - x1;
  if (i0 < n) a[i0] = ex;
  if (i1 < n) a[i1] = ex + x0;
  if (tid == 0) a[n] = warp_tot[32];
  __syncthreads();
}

__global__ void __launch_bounds__(kSmallThreads) small_plan_kernel(const SmallArgs args) {
  extern __shared__ uint8_t small_raw[];
  SmallSmem& sm = *reinterpret_cast<SmallSmem*>(small_raw);
  __shared__ int32_t warp_tot[33];
  const SmallDir& a = args.d[blockIdx.x];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int nwarps = kSmallThreads / 32;
  if (blockIdx.x == 0 && tid < args.n_words) args.words[tid] = 0;

  for (int32_t k = tid; k < a.n_slices; k += kSmallThreads) sm.sl[k] = a.slices[k];
  __syncthreads();
  // 1. per-row intervals: counts, offsets, then each row's intervals sorted by lo
  for (int32_t r = tid; r < a.n_rows; r += kSmallThreads) {
    int32_t c = 0;
    for (int32_t k = 0; k < a.n_slices; ++k) {
      const BandSlice bs = sm.sl[k];
      if (r < bs.r_start || r >= bs.r_end) continue;
      int64_t lo, hi;
      row_interval(bs, r, lo, hi);
      c += lo < hi ? 1 : 0;
    }
    sm.row_off[r] = c;
  }
  __syncthreads();
  small_scan(sm.row_off, a.n_rows, warp_tot);
  for (int32_t r = tid; r <= a.n_rows; r += kSmallThreads) a.iv_off[r] = sm.row_off[r];
  for (int32_t r = tid; r < a.n_rows; r += kSmallThreads) {
    int32_t* dst = a.iv + 2 * static_cast<int64_t>(sm.row_off[r]);
    int32_t c = 0;
    for (int32_t k = 0; k < a.n_slices; ++k) {
      const BandSlice bs = sm.sl[k];
      if (r < bs.r_start || r >= bs.r_end) continue;
      int64_t lo, hi;
      row_interval(bs, r, lo, hi);
      if (lo >= hi) continue;
      int32_t j = c - 1;   // insertion by lo
      while (j >= 0 && dst[2 * j] > lo) {
        dst[2 * j + 2] = dst[2 * j];
        dst[2 * j + 3] = dst[2 * j + 1];
        --j;
      }
      dst[2 * j + 2] = static_cast<int32_t>(lo);
      dst[2 * j + 3] = static_cast<int32_t>(hi);
      ++c;
    }
  }
  __syncthreads();

  // 2. the class of every block: allowed elements summed over its rows
  const int32_t n_blk = a.n_rt * a.n_ct;
  for (int32_t i = tid; i < n_blk; i += kSmallThreads) {
    const int32_t rt = i / a.n_ct, ct = i % a.n_ct;
    const int32_t r0 = rt * a.tile_r, r1 = min(a.n_rows, r0 + a.tile_r);
    const int32_t c0 = ct * a.tile_c, c1 = min(a.n_cols, c0 + a.tile_c);
    int64_t cnt = 0;
    for (int32_t r = r0; r < r1; ++r)
      for (int32_t e = sm.row_off[r]; e < sm.row_off[r + 1]; ++e) {
        const int32_t x0 = max(a.iv[2 * e], c0), x1 = min(a.iv[2 * e + 1], c1);
        cnt += x1 > x0 ? x1 - x0 : 0;
      }
    const bool row_oob = r0 + a.tile_r > a.n_rows, col_oob = c0 + a.tile_c > a.n_cols;
    const bool full_ok = !col_oob && (!a.k2q || !row_oob);
    const bool full = cnt > 0 && cnt == static_cast<int64_t>(r1 - r0) * (c1 - c0) && full_ok;
    sm.cls[i] = cnt == 0 ? 0 : (full ? 2 : 1);
  }
  __syncthreads();

  // 3. per row tile: Full / Partial counts, and (k2q) their prefix counts at chunk starts
  const int32_t csz = 1 << a.chunk_log2;
  const int32_t n_chunks = a.k2q ? (a.n_ct + csz - 1) >> a.chunk_log2 : 0;
  for (int32_t rt = warp; rt < a.n_rt; rt += nwarps) {
    int32_t f = 0, m = 0;
    for (int32_t base = 0; base < a.n_ct; base += 32) {
      const int32_t ct = base + lane;
      const uint8_t c = ct < a.n_ct ? sm.cls[rt * a.n_ct + ct] : 0;
      const uint32_t bf = __ballot_sync(0xffffffffu, c == 2), bm = __ballot_sync(0xffffffffu, c == 1);
      if (a.k2q && lane == 0 && (base & (csz - 1)) == 0) {   // chunks are multiples of 32 column tiles
        sm.pf[rt][base >> a.chunk_log2] = f;
        sm.pm[rt][base >> a.chunk_log2] = m;
      }
      f += __popc(bf);
      m += __popc(bm);
    }
    if (lane == 0) {
      sm.nf[rt] = f;
      sm.nm[rt] = m;
      if (a.k2q) {
        sm.pf[rt][n_chunks] = f;
        sm.pm[rt][n_chunks] = m;
      }
    }
  }
  __syncthreads();
  for (int32_t i = tid; i < a.n_rt; i += kSmallThreads) {
    sm.foff[i] = sm.nf[i];
    sm.moff[i] = sm.nm[i];
  }
  __syncthreads();
  small_scan(sm.foff, a.n_rt, warp_tot);
  small_scan(sm.moff, a.n_rt, warp_tot);
  for (int32_t i = tid; i <= a.n_rt; i += kSmallThreads) {
    a.full_off[i] = sm.foff[i];
    a.mask_off[i] = sm.moff[i];
  }

  // 4. the lists, ascending per row tile
  for (int32_t rt = warp; rt < a.n_rt; rt += nwarps) {
    int32_t f = sm.foff[rt], m = sm.moff[rt];
    for (int32_t base = 0; base < a.n_ct; base += 32) {
      const int32_t ct = base + lane;
      const uint8_t c = ct < a.n_ct ? sm.cls[rt * a.n_ct + ct] : 0;
      const uint32_t bf = __ballot_sync(0xffffffffu, c == 2), bm = __ballot_sync(0xffffffffu, c == 1);
      const uint32_t below = (1u << lane) - 1u;
      if (c == 2) a.full_idx[f + __popc(bf & below)] = ct;
      if (c == 1) a.mask_idx[m + __popc(bm & below)] = ct;
      f += __popc(bf);
      m += __popc(bm);
    }
  }

  // 5. longest-work-first order: bitonic sort of (cost desc, index asc) keys
  int32_t n_pad = 1;
  while (n_pad < a.n_rt) n_pad <<= 1;
  for (int32_t i = tid; i < n_pad; i += kSmallThreads) {
    if (i < a.n_rt) {
      const int64_t cost = static_cast<int64_t>(kCostFull) * sm.nf[i] + static_cast<int64_t>(kCostMask) * sm.nm[i];
      sm.keys[i] = (static_cast<uint64_t>(0x7FFFFFFF - cost) << 32) | static_cast<uint32_t>(i);
    } else {
      sm.keys[i] = ~0ull;
    }
  }
  __syncthreads();
  for (int32_t k = 2; k <= n_pad; k <<= 1)
    for (int32_t j = k >> 1; j > 0; j >>= 1) {
      for (int32_t i = tid; i < n_pad; i += kSmallThreads) {
        const int32_t q = i ^ j;
        if (q > i) {
          const bool up = (i & k) == 0;
          const uint64_t x = sm.keys[i], y = sm.keys[q];
          if ((x > y) == up) {
            sm.keys[i] = y;
            sm.keys[q] = x;
          }
        }
      }
      __syncthreads();
    }
  for (int32_t i = tid; i < a.n_rt; i += kSmallThreads) a.order[i] = static_cast<int32_t>(sm.keys[i] & 0xffffffffu);

  // 6. k2q: the backward work items, chunk by chunk, inside a chunk in the
  //    k-tiles' longest-work-first order (one warp per chunk)
  int32_t n_items = 0;
  if (a.k2q) {
    for (int32_t c = warp; c < n_chunks; c += nwarps) {
      int32_t cnt = 0;
      for (int32_t base = 0; base < a.n_rt; base += 32) {
        const int32_t r = base + lane;
        bool has = false;
        if (r < a.n_rt) {
          const int32_t kt = static_cast<int32_t>(sm.keys[r] & 0xffffffffu);
          has = sm.pf[kt][c + 1] > sm.pf[kt][c] || sm.pm[kt][c + 1] > sm.pm[kt][c];
        }
        cnt += __popc(__ballot_sync(0xffffffffu, has));
      }
      if (lane == 0) sm.ccnt[c] = cnt;
    }
    __syncthreads();
    if (tid == 0) {
      int32_t run = 0;
      for (int32_t c = 0; c < n_chunks; ++c) {
        sm.coff[c] = run;
        run += sm.ccnt[c];
      }
      sm.coff[n_chunks] = run;
    }
    __syncthreads();
    n_items = sm.coff[n_chunks];
    for (int32_t c = warp; c < n_chunks; c += nwarps) {
      int32_t pos = sm.coff[c];
      for (int32_t base = 0; base < a.n_rt; base += 32) {
        const int32_t r = base + lane;
        bool has = false;
        int4 it = make_int4(0, 0, 0, 0);
        if (r < a.n_rt) {
          const int32_t kt = static_cast<int32_t>(sm.keys[r] & 0xffffffffu);
          const int32_t nfc = sm.pf[kt][c + 1] - sm.pf[kt][c], nmc = sm.pm[kt][c + 1] - sm.pm[kt][c];
          has = nfc > 0 || nmc > 0;
          it = make_int4(kt, sm.foff[kt] + sm.pf[kt][c], sm.moff[kt] + sm.pm[kt][c], nfc | (nmc << 16));
        }
        const uint32_t b = __ballot_sync(0xffffffffu, has);
        if (has) a.items[pos + __popc(b & ((1u << lane) - 1u))] = it;
        pos += __popc(b);
      }
    }
  }
  if (tid == 0) {   // the sizes out to the host
    volatile int64_t* t = a.totals;
    t[0] = sm.row_off[a.n_rows];
    t[1] = sm.foff[a.n_rt];
    t[2] = sm.moff[a.n_rt];
    t[3] = n_items;
    __threadfence_system();
  }
}

// Small transfers between the host and a plan under construction (the band
// slices in, the list sizes out) go through one pinned, device-mapped host
// buffer per device, read and written by kernels.  A cudaMemcpyAsync of a
// few bytes would wait on the copy engines behind whatever large copies other
// streams have in flight (the next batch's inputs, the last one's results),
// and plan creation waits for its result.  Layout: words [0, 8) results,
// then the slices.  The mutex is held for a whole direction build, which is
// host-synchronous anyway.
struct HostChannel {
  std::mutex mu;
  uint8_t* host = nullptr;   // pinned and mapped
  uint8_t* dev = nullptr;    // its device address
  size_t bytes = 0;
};
HostChannel g_channel[64];
constexpr size_t kChannelResults = 128;   // bytes of result words (two directions' totals) before the slices

cudaError_t channel_reserve(HostChannel& c, size_t bytes) {
  if (c.bytes >= bytes) return cudaSuccess;
  size_t cap = c.bytes ? c.bytes : size_t{1} << 20;
  while (cap < bytes) cap <<= 1;
  if (c.host) cudaFreeHost(c.host);
  c.host = c.dev = nullptr;
  c.bytes = 0;
  void* h = nullptr;
  cudaError_t e = cudaHostAlloc(&h, cap, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) return e;
  void* d = nullptr;
  e = cudaHostGetDevicePointer(&d, h, 0);
  if (e != cudaSuccess) {
    cudaFreeHost(h);
    return e;
  }
  c.host = static_cast<uint8_t*>(h);
  c.dev = static_cast<uint8_t*>(d);
  c.bytes = cap;
  return cudaSuccess;
}

__global__ void copy_u64_kernel(const uint64_t* __restrict__ src, uint64_t* __restrict__ dst, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = src[i];
}

template <typename T>
cudaError_t dalloc(T** p, int64_t count, cudaStream_t st) {
  const size_t bytes = static_cast<size_t>(count > 0 ? count : 1) * sizeof(T);
  return cudaMallocAsync(reinterpret_cast<void**>(p), bytes, st);
}

// Exclusive scan of n counts into out[0..n] (out[n] = total) and the int64
// total: one block for short inputs, three launches over segments for long
// ones.  `launches` counts the kernels.
constexpr int64_t kLongScan = 16384;
cudaError_t scan_counts(const int32_t* in, int64_t n, int32_t* out, int64_t* total, cudaStream_t st,
                        int32_t& launches) {
  if (n <= kLongScan) {
    scan_kernel<<<1, kScanThreads, 0, st>>>(in, n, out, total);
    ++launches;
    return cudaGetLastError();
  }
  const int32_t n_seg = static_cast<int32_t>(std::min<int64_t>(kScanSegments, (n + kScanThreads - 1) / kScanThreads));
  int64_t* seg_sum = nullptr;
  int32_t* seg_off = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&seg_sum), sizeof(int64_t) * n_seg, st);
  if (e == cudaSuccess) e = cudaMallocAsync(reinterpret_cast<void**>(&seg_off), sizeof(int32_t) * (n_seg + 1), st);
  if (e == cudaSuccess) {
    segment_sum_kernel<<<n_seg, kScanThreads, 0, st>>>(in, n, seg_sum);
    segment_offsets_kernel<<<1, kScanThreads, 0, st>>>(seg_sum, n_seg, seg_off, total);
    segment_scan_kernel<<<n_seg, kScanThreads, 0, st>>>(in, n, seg_off, out);
    launches += 3;
    e = cudaGetLastError();
  }
  if (seg_sum) cudaFreeAsync(seg_sum, st);
  if (seg_off) cudaFreeAsync(seg_off, st);
  return e;
}

int grid_for(int64_t n, int threads, int num_sms) {
  const int64_t g = (n + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(num_sms) * 16;
  return static_cast<int>(std::max<int64_t>(1, std::min(g, cap)));
}

}  // namespace

cudaError_t read_device_words(const void* src, void* dst, int64_t n_words, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || n_words < 0) return cudaErrorInvalidValue;
  HostChannel& chan = g_channel[dev];
  std::lock_guard<std::mutex> lock(chan.mu);
  e = channel_reserve(chan, kChannelResults + 8 * static_cast<size_t>(n_words));
  if (e != cudaSuccess || n_words == 0) return e;
  copy_u64_kernel<<<1, 32, 0, stream>>>(static_cast<const uint64_t*>(src),
                                        reinterpret_cast<uint64_t*>(chan.dev + kChannelResults), n_words);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) std::memcpy(dst, chan.host + kChannelResults, 8 * static_cast<size_t>(n_words));
  return e;
}

#define FFA_CK(x)                                  \
  do {                                             \
    cudaError_t e_ = (x);                          \
    if (e_ != cudaSuccess) {                       \
      st = FFA_ERR_CUDA;                           \
      goto done;                                   \
    }                                              \
  } while (0)

namespace {

// Device temporaries of one direction between the two phases of a plan.
struct DirTemps {
  int32_t *cand_cnt = nullptr, *cand_off = nullptr, *cand = nullptr, *iv_cnt = nullptr;
  int32_t *nf = nullptr, *nm = nullptr, *icnt = nullptr, *ioff = nullptr;
  int64_t* totals = nullptr;   // [candidates, intervals, Full, Partial, backward items]
  uint64_t* keys = nullptr;
  SweepArgs sa{};
  void release(cudaStream_t stream) {
    void* ptrs[] = {cand_cnt, cand_off, cand, iv_cnt, nf, nm, icnt, ioff, totals, keys};
    for (void* p : ptrs)
      if (p) cudaFreeAsync(p, stream);
  }
};
constexpr int kTotals = 5;

// Phase 1 of one direction, up to the sizes: the slices in through the
// mapped channel (at byte offset slice_off), candidate slices per row tile,
// per-row intervals, the Full / Partial counts per row tile and their
// offsets, and (k2q) the number of backward work items.  The five totals go
// out to the channel at byte offset result_off; nothing waits for them here.
ffa_status dir_phase1(DirMeta& m, const BandSlice* hs, int64_t ns, cudaStream_t stream, bool k2q, int num_sms,
                      HostChannel& chan, size_t slice_off, size_t result_off, DirTemps& t) {
  ffa_status st = FFA_OK;
  int64_t n_cand = 0, iv_bound = 0, max_tiles = 1;
  for (int64_t i = 0; i < ns; ++i) {
    const int64_t tiles = (hs[i].r_end - 1) / m.tile_r - hs[i].r_start / m.tile_r + 1;
    n_cand += tiles;
    max_tiles = std::max(max_tiles, tiles);
    iv_bound += hs[i].r_end - hs[i].r_start;
  }
  if (iv_bound > INT32_MAX || n_cand > INT32_MAX) return FFA_ERR_OVERFLOW;
  m.chunk_log2 = k2q ? kBwdChunkLog2 : 0;
  m.launches = 0;

  FFA_CK(dalloc(&m.slices, ns, stream));
  if (ns > 0) {   // the slices in through the mapped buffer
    std::memcpy(chan.host + slice_off, hs, sizeof(BandSlice) * ns);
    const int64_t words = static_cast<int64_t>(sizeof(BandSlice) / 8) * ns;
    copy_u64_kernel<<<grid_for(words, 256, num_sms), 256, 0, stream>>>(
        reinterpret_cast<const uint64_t*>(chan.dev + slice_off), reinterpret_cast<uint64_t*>(m.slices), words);
    ++m.launches;
    FFA_CK(cudaGetLastError());
  }
  FFA_CK(dalloc(&t.totals, kTotals, stream));
  FFA_CK(cudaMemsetAsync(t.totals, 0, sizeof(int64_t) * kTotals, stream));
  FFA_CK(dalloc(&m.iv_off, m.n_rows + 1, stream));
  FFA_CK(dalloc(&m.full_off, m.n_rt + 1, stream));
  FFA_CK(dalloc(&m.mask_off, m.n_rt + 1, stream));
  FFA_CK(dalloc(&m.order, m.n_rt, stream));
  FFA_CK(cudaMemsetAsync(m.iv_off, 0, sizeof(int32_t) * (m.n_rows + 1), stream));
  FFA_CK(cudaMemsetAsync(m.full_off, 0, sizeof(int32_t) * (m.n_rt + 1), stream));
  FFA_CK(cudaMemsetAsync(m.mask_off, 0, sizeof(int32_t) * (m.n_rt + 1), stream));

  if (m.n_rt > 0 && m.n_rows > 0) {
    // 1. candidate slices per row-tile
    FFA_CK(dalloc(&t.cand_cnt, m.n_rt, stream));
    FFA_CK(dalloc(&t.cand_off, m.n_rt + 1, stream));
    FFA_CK(dalloc(&t.cand, n_cand, stream));
    FFA_CK(cudaMemsetAsync(t.cand_cnt, 0, sizeof(int32_t) * m.n_rt, stream));
    const dim3 cgrid(static_cast<unsigned>(std::min<int64_t>((max_tiles + 255) / 256, 64)),
                     static_cast<unsigned>(std::min<int64_t>(std::max<int64_t>(ns, 1), 65535)));
    if (ns > 0) {
      cand_kernel<false><<<cgrid, 256, 0, stream>>>(m.slices, ns, m.tile_r, t.cand_cnt, nullptr, nullptr);
      ++m.launches;
    }
    FFA_CK(scan_counts(t.cand_cnt, m.n_rt, t.cand_off, t.totals + 0, stream, m.launches));
    FFA_CK(cudaMemsetAsync(t.cand_cnt, 0, sizeof(int32_t) * m.n_rt, stream));
    if (ns > 0) {
      cand_kernel<true><<<cgrid, 256, 0, stream>>>(m.slices, ns, m.tile_r, t.cand_cnt, t.cand_off, t.cand);
      ++m.launches;
    }
    // 2. per-row intervals
    FFA_CK(dalloc(&t.iv_cnt, m.n_rows, stream));
    FFA_CK(dalloc(&m.iv, 2 * std::max<int64_t>(iv_bound, 1), stream));
    iv_kernel<false><<<grid_for(m.n_rows, 256, num_sms), 256, 0, stream>>>(m.slices, t.cand_off, t.cand, m.n_rows,
                                                                           m.tile_r, t.iv_cnt, nullptr, nullptr);
    ++m.launches;
    FFA_CK(scan_counts(t.iv_cnt, m.n_rows, m.iv_off, t.totals + 1, stream, m.launches));
    iv_kernel<true><<<grid_for(m.n_rows, 256, num_sms), 256, 0, stream>>>(m.slices, t.cand_off, t.cand, m.n_rows,
                                                                          m.tile_r, nullptr, m.iv_off, m.iv);
    ++m.launches;
    // 3. block counts per row-tile, offsets; (k2q) the work items
    t.sa = SweepArgs{m.n_rows, m.n_cols, m.tile_r,  m.tile_c,     m.n_rt,
                     k2q ? 1 : 0, m.iv_off, m.iv, m.chunk_log2,
                     k2q ? reinterpret_cast<unsigned long long*>(t.totals + 4) : nullptr};
    FFA_CK(dalloc(&t.nf, m.n_rt, stream));
    FFA_CK(dalloc(&t.nm, m.n_rt, stream));
    sweep_kernel<false><<<std::min<int64_t>(m.n_rt, num_sms * 8), kSweepThreads, 0, stream>>>(
        t.sa, t.nf, t.nm, nullptr, nullptr, nullptr, nullptr);
    ++m.launches;
    FFA_CK(scan_counts(t.nf, m.n_rt, m.full_off, t.totals + 2, stream, m.launches));
    FFA_CK(scan_counts(t.nm, m.n_rt, m.mask_off, t.totals + 3, stream, m.launches));
    FFA_CK(cudaGetLastError());
  } else {
    FFA_CK(dalloc(&m.iv, 2, stream));
  }
  // the totals out through the mapped buffer
  copy_u64_kernel<<<1, 32, 0, stream>>>(reinterpret_cast<const uint64_t*>(t.totals),
                                        reinterpret_cast<uint64_t*>(chan.dev + result_off), kTotals);
  ++m.launches;
  FFA_CK(cudaGetLastError());
done:
  return st;
}

// Phase 2 of one direction, once its totals are on the host: the CSR lists,
// the longest-work-first order and (k2q) the backward work items.
ffa_status dir_phase2(DirMeta& m, const int64_t* tot, cudaStream_t stream, bool k2q, int num_sms, DirTemps& t) {
  ffa_status st = FFA_OK;
  m.n_iv = tot[1];
  m.nnz_full = tot[2];
  m.nnz_mask = tot[3];
  m.n_items = k2q ? tot[4] : 0;
  if (m.nnz_full > INT32_MAX || m.nnz_mask > INT32_MAX || m.n_iv > INT32_MAX || m.n_items > INT32_MAX / 2)
    return FFA_ERR_OVERFLOW;
  FFA_CK(dalloc(&m.full_idx, m.nnz_full, stream));
  FFA_CK(dalloc(&m.mask_idx, m.nnz_mask, stream));
  if (k2q) {
    FFA_CK(dalloc(&m.items, m.n_items, stream));
    // an item left unwritten would be one without blocks, which every role skips
    if (m.n_items > 0) FFA_CK(cudaMemsetAsync(m.items, 0, sizeof(int4) * m.n_items, stream));
  }
  if (m.n_rt > 0 && m.n_rows > 0) {
    // 4. CSR lists
    sweep_kernel<true><<<std::min<int64_t>(m.n_rt, num_sms * 8), kSweepThreads, 0, stream>>>(
        t.sa, nullptr, nullptr, m.full_off, m.mask_off, m.full_idx, m.mask_idx);
    ++m.launches;
    // 5. longest-work-first order
    int32_t n_pad = 1;
    while (n_pad < m.n_rt) n_pad <<= 1;
    if (n_pad <= 16384) {
      const size_t smem = sizeof(uint64_t) * n_pad;
      FFA_CK(cudaFuncSetAttribute(lpt_sort_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(std::max<size_t>(smem, 48 * 1024))));
      lpt_sort_smem_kernel<<<1, 1024, smem, stream>>>(m.full_off, m.mask_off, m.n_rt, n_pad, m.order);
      ++m.launches;
    } else {
      FFA_CK(dalloc(&t.keys, n_pad, stream));
      const int g = grid_for(n_pad, 256, num_sms);
      lpt_keys_kernel<<<g, 256, 0, stream>>>(m.full_off, m.mask_off, m.n_rt, n_pad, t.keys);
      ++m.launches;
      for (int32_t k = 2; k <= n_pad; k <<= 1)
        for (int32_t j = k >> 1; j > 0; j >>= 1) {
          bitonic_step_kernel<<<g, 256, 0, stream>>>(t.keys, n_pad, k, j);
          ++m.launches;
        }
      lpt_order_kernel<<<grid_for(m.n_rt, 256, num_sms), 256, 0, stream>>>(t.keys, m.n_rt, m.order);
      ++m.launches;
    }
    FFA_CK(cudaGetLastError());
    // 6. backward work items (k2q only): per q-chunk, the k-tiles with
    //    blocks in it, in longest-work-first order; their count came with
    //    the phase-1 totals, their offsets per chunk from a count pass here
    if (k2q && m.n_items > 0) {
      const int32_t n_chunks = static_cast<int32_t>((static_cast<int64_t>(m.n_ct) + (1 << m.chunk_log2) - 1) >>
                                                    m.chunk_log2);
      FFA_CK(dalloc(&t.icnt, n_chunks, stream));
      FFA_CK(dalloc(&t.ioff, n_chunks + 1, stream));
      const int cg = static_cast<int>(std::min<int64_t>(n_chunks, static_cast<int64_t>(num_sms) * 8));
      chunk_items_kernel<false><<<cg, kItemThreads, 0, stream>>>(m.full_off, m.full_idx, m.mask_off, m.mask_idx,
                                                                 m.order, m.n_rt, n_chunks, m.chunk_log2, nullptr,
                                                                 t.icnt, nullptr, 0);
      ++m.launches;
      FFA_CK(scan_counts(t.icnt, n_chunks, t.ioff, t.totals + 0, stream, m.launches));
      chunk_items_kernel<true><<<cg, kItemThreads, 0, stream>>>(m.full_off, m.full_idx, m.mask_off, m.mask_idx,
                                                                m.order, m.n_rt, n_chunks, m.chunk_log2, t.ioff,
                                                                nullptr, m.items, m.n_items);
      ++m.launches;
      FFA_CK(cudaGetLastError());
    }
  }
done:
  return st;
}

// A small plan (both lengths <= kSmallLen, <= kSmallSlices slices) in one
// launch of small_plan_kernel: every array of both directions in one
// allocation (the plan's arena), sized from upper bounds; one wait.
ffa_status build_small(DirMeta& q, DirMeta& k, const BandSlice* band, const BandSlice* tband, int64_t ns,
                       cudaStream_t stream, HostChannel& chan, void** arena, DeviceWords** words) {
  DirMeta* dirs[2] = {&q, &k};
  const BandSlice* hs[2] = {band, tband};
  auto a256 = [](size_t x) { return (x + 255) & ~size_t(255); };
  size_t off[2][8], total = 0;
  for (int d = 0; d < 2; ++d) {
    DirMeta& m = *dirs[d];
    m.chunk_log2 = d ? kBwdChunkLog2 : 0;
    int64_t iv_bound = 0;   // one interval per (slice, row) at most
    for (int64_t i = 0; i < ns; ++i) iv_bound += std::min<int64_t>(hs[d][i].r_end, m.n_rows) - hs[d][i].r_start;
    const int64_t blk = static_cast<int64_t>(m.n_rt) * m.n_ct;
    const int64_t n_chunks = d ? (m.n_ct + (1 << m.chunk_log2) - 1) >> m.chunk_log2 : 0;
    const size_t bytes[8] = {4 * static_cast<size_t>(m.n_rows + 1), 8 * static_cast<size_t>(std::max<int64_t>(iv_bound, 1)),
                             4 * static_cast<size_t>(m.n_rt + 1),  4 * static_cast<size_t>(m.n_rt + 1),
                             4 * static_cast<size_t>(std::max<int64_t>(blk, 1)),
                             4 * static_cast<size_t>(std::max<int64_t>(blk, 1)),
                             4 * static_cast<size_t>(std::max<int32_t>(m.n_rt, 1)),
                             16 * static_cast<size_t>(std::max<int64_t>(m.n_rt * n_chunks, 1))};
    for (int j = 0; j < 8; ++j) {
      off[d][j] = total;
      total += a256(bytes[j]);
    }
  }
  const size_t words_off = total;
  total += a256(sizeof(DeviceWords));
  uint8_t* base = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&base), total, stream) != cudaSuccess) return FFA_ERR_CUDA;
  *arena = base;
  *words = reinterpret_cast<DeviceWords*>(base + words_off);
  const size_t slice_bytes = sizeof(BandSlice) * static_cast<size_t>(ns);
  SmallArgs args{};
  args.words = reinterpret_cast<uint32_t*>(*words);
  args.n_words = static_cast<int32_t>(sizeof(DeviceWords) / 4);
  for (int d = 0; d < 2; ++d) {
    DirMeta& m = *dirs[d];
    m.owns_arrays = false;
    m.slices = nullptr;
    m.iv_off = reinterpret_cast<int32_t*>(base + off[d][0]);
    m.iv = reinterpret_cast<int32_t*>(base + off[d][1]);
    m.full_off = reinterpret_cast<int32_t*>(base + off[d][2]);
    m.mask_off = reinterpret_cast<int32_t*>(base + off[d][3]);
    m.full_idx = reinterpret_cast<int32_t*>(base + off[d][4]);
    m.mask_idx = reinterpret_cast<int32_t*>(base + off[d][5]);
    m.order = reinterpret_cast<int32_t*>(base + off[d][6]);
    m.items = d ? reinterpret_cast<int4*>(base + off[d][7]) : nullptr;
    m.launches = d ? 0 : 1;
    const size_t soff = kChannelResults + d * slice_bytes;
    if (ns > 0) std::memcpy(chan.host + soff, hs[d], slice_bytes);
    SmallDir& sd = args.d[d];
    sd.slices = reinterpret_cast<const BandSlice*>(chan.dev + soff);
    sd.n_slices = static_cast<int32_t>(ns);
    sd.n_rows = static_cast<int32_t>(m.n_rows);
    sd.n_cols = static_cast<int32_t>(m.n_cols);
    sd.tile_r = m.tile_r;
    sd.tile_c = m.tile_c;
    sd.n_rt = m.n_rt;
    sd.n_ct = m.n_ct;
    sd.k2q = d;
    sd.chunk_log2 = m.chunk_log2;
    sd.iv_off = m.iv_off;
    sd.iv = m.iv;
    sd.full_off = m.full_off;
    sd.full_idx = m.full_idx;
    sd.mask_off = m.mask_off;
    sd.mask_idx = m.mask_idx;
    sd.order = m.order;
    sd.items = reinterpret_cast<int4*>(base + off[d][7]);
    sd.totals = reinterpret_cast<int64_t*>(chan.dev + 32 * d);
  }
  cudaError_t e = cudaFuncSetAttribute(small_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(SmallSmem)));
  if (e == cudaSuccess) {
    small_plan_kernel<<<2, kSmallThreads, sizeof(SmallSmem), stream>>>(args);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) {
    cudaStreamSynchronize(stream);
    return FFA_ERR_CUDA;
  }
  for (int d = 0; d < 2; ++d) {
    const volatile int64_t* t = reinterpret_cast<const volatile int64_t*>(chan.host + 32 * d);
    DirMeta& m = *dirs[d];
    m.n_iv = t[0];
    m.nnz_full = t[1];
    m.nnz_mask = t[2];
    m.n_items = d ? t[3] : 0;
  }
  return FFA_OK;
}
static_assert(sizeof(SmallSmem) <= 227 * 1024, "small-plan shared memory");

}  // namespace

ffa_status build_plan(DirMeta& q, DirMeta& k, const BandSlice* band, const BandSlice* tband, int64_t ns,
                      cudaStream_t stream, int num_sms, void** arena, DeviceWords** words) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FFA_ERR_CUDA;
  HostChannel& chan = g_channel[dev];
  std::lock_guard<std::mutex> chan_lock(chan.mu);
  const size_t slice_bytes = sizeof(BandSlice) * static_cast<size_t>(ns);
  if (channel_reserve(chan, kChannelResults + 2 * slice_bytes) != cudaSuccess) return FFA_ERR_CUDA;
  if (ns <= kSmallSlices && q.n_rows > 0 && q.n_cols > 0 && q.n_rows <= kSmallLen && q.n_cols <= kSmallLen)
    return build_small(q, k, band, tband, ns, stream, chan, arena, words);
  DirTemps tq, tk;
  ffa_status st = dir_phase1(q, band, ns, stream, false, num_sms, chan, kChannelResults, 0, tq);
  if (st == FFA_OK)
    st = dir_phase1(k, tband, ns, stream, true, num_sms, chan, kChannelResults + slice_bytes, 8 * kTotals, tk);
  if (st == FFA_OK) {   // the one wait for sizes: both directions' totals
    if (cudaStreamSynchronize(stream) != cudaSuccess) st = FFA_ERR_CUDA;
  }
  if (st == FFA_OK) {
    int64_t tot[2 * kTotals];
    std::memcpy(tot, chan.host, sizeof(tot));
    st = dir_phase2(q, tot, stream, false, num_sms, tq);
    if (st == FFA_OK) st = dir_phase2(k, tot + kTotals, stream, true, num_sms, tk);
  }
  // On an error, kernels launched above may still read or write the mapped
  // channel buffer; wait for them before the channel's lock is released.
  if (st != FFA_OK) cudaStreamSynchronize(stream);
  tq.release(stream);
  tk.release(stream);
  return st;
}

void free_direction(DirMeta& m, cudaStream_t stream) {
  void* ptrs[] = {m.slices, m.iv_off, m.iv, m.full_off, m.full_idx, m.mask_off, m.mask_idx, m.order, m.items};
  if (m.owns_arrays)   // else they live in the plan's arena
    for (void* p : ptrs)
      if (p) cudaFreeAsync(p, stream);
  m.slices = nullptr;
  m.iv_off = m.iv = m.full_off = m.full_idx = m.mask_off = m.mask_idx = m.order = nullptr;
  m.items = nullptr;
  m.n_items = 0;
}

}  // namespace ffa
