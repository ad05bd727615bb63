// Range-Gather and Range-Scatter-Reduce: local row rearrangement kernels.
//
// MagiAttention blog, group-collective section: the AlltoAll-v exchange of
// the distributed pass needs Range-Gather / Range-Scatter-Reduce pre / post
// kernels, and their device-to-device rearrangement cost is not small.  Here
// they are the local kernels on their own:
//   gather          dst = the rows of src in ranges [s_k, e_k), back to back
//                   in list order (e.g. the KV rows one peer needs);
//   scatter-reduce  dst[s_k, e_k) += the rows of a contiguous buffer, in list
//                   order; ranges may overlap and then all their rows add
//                   (e.g. partial dK / dV received from several peers).
// Both are HBM-bound.  A range is one contiguous block in both buffers, so
// the gather gives each CTA a 64 KB tile of the output, finds the range of
// the tile's first row once and copies the tile range by range with
// coalesced 16-byte loads and stores.  The scatter-reduce takes one thread per
// 16-byte chunk, which finds its range by binary search over the ranges'
// offsets in the contiguous buffer.  Tables of up to 256 ranges travel in the
// launch's parameters; longer ones are copied to the device.
#include <cuda_bf16.h>

#include <algorithm>
#include <functional>
#include <utility>
#include <vector>

#include "ffa_internal.h"
#include "ptx.cuh"

namespace ffa {
namespace {

struct RangeRec {
  int64_t buf_off;   // first row of the range in the contiguous buffer
  int64_t row;       // first row of the range in the token-major tensor
};

constexpr int kParamRanges = 256;
struct RangeTable {   // a short range table passed by value (4 KB of kernel parameters)
  RangeRec r[kParamRanges];
};
constexpr int64_t kGatherTile = 4096;   // 16-byte chunks of output per gather CTA tile (64 KB)

// Index of the range holding buffer row r: the last k with buf_off <= r
// (ranges are non-empty, so offsets strictly increase).
__device__ __forceinline__ int64_t find_range(const RangeRec* rr, int64_t n, int64_t r) {
  int64_t lo = 0, hi = n - 1;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) >> 1;
    if (rr[mid].buf_off <= r) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// rr_dev: the range table in device memory, or null when it is `tab`.
__global__ void __launch_bounds__(256) range_gather_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                           const RangeRec* __restrict__ rr_dev,
                                                           const __grid_constant__ RangeTable tab, int64_t n_ranges,
                                                           int64_t total_rows, int64_t chunks_per_row) {
  const RangeRec* rr = rr_dev ? rr_dev : tab.r;
  const int64_t n = total_rows * chunks_per_row;
  for (int64_t t0 = blockIdx.x * kGatherTile; t0 < n; t0 += static_cast<int64_t>(gridDim.x) * kGatherTile) {
    const int64_t t1 = min(t0 + kGatherTile, n);
    // the ranges covering output chunks [t0, t1), from the one holding the tile's first row
    int64_t k = find_range(rr, n_ranges, t0 / chunks_per_row);
    for (int64_t c0 = t0; c0 < t1; ++k) {
      const int64_t c1 = min(t1, (k + 1 < n_ranges ? rr[k + 1].buf_off : total_rows) * chunks_per_row);
      const int64_t shift = (rr[k].row - rr[k].buf_off) * chunks_per_row;   // output chunk i is src[i + shift]
      for (int64_t i = c0 + threadIdx.x; i < c1; i += 4 * static_cast<int64_t>(blockDim.x)) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t j = i + u * static_cast<int64_t>(blockDim.x);
          if (j < c1) v[u] = src[j + shift];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int64_t j = i + u * static_cast<int64_t>(blockDim.x);
          if (j < c1) dst[j] = v[u];
        }
      }
      c0 = c1;
    }
  }
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// BF16: 16 bytes = 8 values; ATOMIC when some destination rows are covered
// by more than one range.
template <bool BF16, bool ATOMIC>
__global__ void __launch_bounds__(256) range_scatter_reduce_kernel(const uint4* __restrict__ src, uint4* dst,
                                                                   const RangeRec* __restrict__ rr_dev,
                                                                   const __grid_constant__ RangeTable tab,
                                                                   int64_t n_ranges, int64_t total_rows,
                                                                   int64_t chunks_per_row) {
  const RangeRec* rr = rr_dev ? rr_dev : tab.r;
  const int64_t n = total_rows * chunks_per_row;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / chunks_per_row, c = i - r * chunks_per_row;
    const RangeRec x = rr[find_range(rr, n_ranges, r)];
    uint4* d = dst + (x.row + r - x.buf_off) * chunks_per_row + c;
    const uint4 v = src[i];
    if (!BF16) {
      if (ATOMIC) {
        red_add_v4(reinterpret_cast<float*>(d), __uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                   __uint_as_float(v.w));
      } else {
        const uint4 o = *d;
        *d = make_uint4(__float_as_uint(__uint_as_float(o.x) + __uint_as_float(v.x)),
                        __float_as_uint(__uint_as_float(o.y) + __uint_as_float(v.y)),
                        __float_as_uint(__uint_as_float(o.z) + __uint_as_float(v.z)),
                        __float_as_uint(__uint_as_float(o.w) + __uint_as_float(v.w)));
      }
    } else {
      const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
      if (ATOMIC) {
        __nv_bfloat162* d2 = reinterpret_cast<__nv_bfloat162*>(d);
#pragma unroll
        for (int k = 0; k < 4; ++k) atomicAdd(d2 + k, *reinterpret_cast<const __nv_bfloat162*>(&vw[k]));
      } else {
        const uint4 o = *d;
        const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = pack_bf16x2(bf_lo(ow[k]) + bf_lo(vw[k]), bf_hi(ow[k]) + bf_hi(vw[k]));
        *d = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Non-empty ranges checked against [0, rows) and laid out back to back.
ffa_status build_ranges(const int64_t* ranges, int64_t n, int64_t rows, std::vector<RangeRec>& out, int64_t& total) {
  out.clear();
  total = 0;
  for (int64_t k = 0; k < n; ++k) {
    const int64_t s = ranges[2 * k], e = ranges[2 * k + 1];
    if (s < 0 || s > e || e > rows) return FFA_ERR_INVALID_ARG;
    if (e == s) continue;
    out.push_back(RangeRec{total, s});
    total += e - s;
  }
  return FFA_OK;
}

int grid_blocks(int64_t n) { return static_cast<int>(std::min<int64_t>((n + 255) / 256, int64_t{1} << 20)); }

// Launches with the range table as a parameter when it fits, else with a
// stream-ordered device copy of it, freed after the kernel.
ffa_status launch_with_table(const std::vector<RangeRec>& rr, cudaStream_t st,
                             const std::function<void(const RangeRec*, const RangeTable&)>& launch) {
  static const RangeTable empty{};
  if (rr.size() <= static_cast<size_t>(kParamRanges)) {
    RangeTable t;
    std::copy(rr.begin(), rr.end(), t.r);
    launch(nullptr, t);
    return cuda_status(cudaGetLastError());
  }
  RangeRec* d = nullptr;
  const size_t bytes = sizeof(RangeRec) * rr.size();
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&d), bytes, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(d, rr.data(), bytes, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) {
    launch(d, empty);
    e = cudaGetLastError();
  }
  if (d) {
    const cudaError_t f = cudaFreeAsync(d, st);
    if (e == cudaSuccess) e = f;
  }
  return cuda_status(e);
}

}  // namespace
}  // namespace ffa

using namespace ffa;

extern "C" ffa_status ffa_range_gather(const void* src, int64_t src_rows, int64_t row_bytes, const int64_t* ranges,
                                       int64_t n_ranges, void* dst, void* stream) {
  if (!src || !dst || (n_ranges > 0 && !ranges) || n_ranges < 0 || src_rows < 0) return FFA_ERR_INVALID_ARG;
  if (row_bytes <= 0 || row_bytes % 16 != 0 || !aligned16(src) || !aligned16(dst)) return FFA_ERR_INVALID_ARG;
  std::vector<RangeRec> rr;
  int64_t total = 0;
  const ffa_status s = build_ranges(ranges, n_ranges, src_rows, rr, total);
  if (s != FFA_OK || total == 0) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cpr = row_bytes / 16;
  const int64_t n = static_cast<int64_t>(rr.size());
  const int g = static_cast<int>(std::min<int64_t>((total * cpr + kGatherTile - 1) / kGatherTile, int64_t{1} << 20));
  return launch_with_table(rr, st, [&](const RangeRec* d, const RangeTable& t) {
    range_gather_kernel<<<g, 256, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), d, t, n, total,
                                           cpr);
  });
}

extern "C" ffa_status ffa_range_scatter_reduce(const void* src, const int64_t* ranges, int64_t n_ranges,
                                               int64_t row_elems, int32_t dtype, void* dst, int64_t dst_rows,
                                               void* stream) {
  if (!src || !dst || (n_ranges > 0 && !ranges) || n_ranges < 0 || dst_rows < 0) return FFA_ERR_INVALID_ARG;
  if (dtype != 0 && dtype != 1) return FFA_ERR_INVALID_ARG;
  const int64_t row_bytes = row_elems * (dtype == 0 ? 4 : 2);
  if (row_elems <= 0 || row_bytes % 16 != 0 || !aligned16(src) || !aligned16(dst)) return FFA_ERR_INVALID_ARG;
  std::vector<RangeRec> rr;
  int64_t total = 0;
  const ffa_status s = build_ranges(ranges, n_ranges, dst_rows, rr, total);
  if (s != FFA_OK || total == 0) return s;
  // overlapping destination ranges need atomic adds; disjoint ones read, add and write
  std::vector<std::pair<int64_t, int64_t>> iv;
  for (int64_t k = 0; k < n_ranges; ++k)
    if (ranges[2 * k + 1] > ranges[2 * k]) iv.push_back({ranges[2 * k], ranges[2 * k + 1]});
  std::sort(iv.begin(), iv.end());
  bool overlap = false;
  for (size_t k = 1; k < iv.size(); ++k) overlap = overlap || iv[k].first < iv[k - 1].second;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t cpr = row_bytes / 16;
  const int64_t n = static_cast<int64_t>(rr.size());
  const uint4* a = static_cast<const uint4*>(src);
  uint4* b = static_cast<uint4*>(dst);
  const int g = grid_blocks(total * cpr);
  return launch_with_table(rr, st, [&](const RangeRec* d, const RangeTable& t) {
    if (dtype == 0 && overlap) range_scatter_reduce_kernel<false, true><<<g, 256, 0, st>>>(a, b, d, t, n, total, cpr);
    else if (dtype == 0) range_scatter_reduce_kernel<false, false><<<g, 256, 0, st>>>(a, b, d, t, n, total, cpr);
    else if (overlap) range_scatter_reduce_kernel<true, true><<<g, 256, 0, st>>>(a, b, d, t, n, total, cpr);
    else range_scatter_reduce_kernel<true, false><<<g, 256, 0, st>>>(a, b, d, t, n, total, cpr);
  });
}
