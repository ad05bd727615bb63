// LSE merge of two partial attention results.
//
// MagiAttention blog, "Flex-Flash-Attention and AttnSlice" (Figure 5):
// partial results over parts of the mask are merged by reduction; the
// distributed pass joins the fragments computed from local and remote KV the
// same way.  For one (query row, head) with partial results (out_a, lse_a) and
// (out_b, lse_b) over disjoint key sets:
//   lse = ln(e^lse_a + e^lse_b),
//   out = e^(lse_a - lse) out_a + e^(lse_b - lse) out_b.
// A part with lse = -inf contributes nothing (its out values are ignored,
// whatever they are); a row empty in both parts comes out as (0, -inf).
#include <cuda_bf16.h>

#include <algorithm>

#include "ffa_internal.h"
#include "ptx.cuh"

namespace ffa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// w x, or 0 where the part is empty (w = 0), so that whatever its out holds
// (NaN included) does not reach the result.
__device__ __forceinline__ float wmul(float w, float x) { return w != 0.f ? w * x : 0.f; }

// One thread per 16-byte chunk (8 values) of a row; the D / 8 threads of a
// (row, head) are adjacent lanes of one warp.  Every load is independent, so
// each thread keeps its reads in flight at once.
template <int D>
__global__ void __launch_bounds__(256) lse_combine_kernel(const uint4* out_a, const float* lse_a, const uint4* out_b,
                                                          const float* lse_b, uint4* out, float* lse, int64_t seqlen,
                                                          int32_t hq) {
  constexpr int CH = D / 8;
  const int64_t n = seqlen * hq * CH;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  // The loop runs per whole warp (its bound depends on the warp's first
  // chunk only), so that every lane reaches the __syncwarp below.
  const int lane = threadIdx.x & 31;
  for (int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + (threadIdx.x & ~31); i0 < n; i0 += stride) {
    const int64_t i = i0 + lane;
    const bool act = i < n;
    const int64_t w = (act ? i : 0) / CH;   // (row, head) pair: w = row * hq + head
    const int64_t row = w / hq;
    const int32_t h = static_cast<int32_t>(w % hq);
    const int64_t li = static_cast<int64_t>(h) * seqlen + row;
    const float la = act ? lse_a[li] : -INFINITY, lb = act ? lse_b[li] : -INFINITY;
    const uint4 va = act ? out_a[i] : uint4{}, vb = act ? out_b[i] : uint4{};
    const float mx = fmaxf(la, lb);
    float wa = 0.f, wb = 0.f, l = -INFINITY;
    if (mx != -INFINITY) {
      const float ea = ex2_approx((la - mx) * kLog2e), eb = ex2_approx((lb - mx) * kLog2e);
      const float sum = ea + eb;
      wa = ea / sum;
      wb = eb / sum;
      l = mx + __log2f(sum) * kLn2;
    }
    const uint32_t ra[4] = {va.x, va.y, va.z, va.w}, rb[4] = {vb.x, vb.y, vb.z, vb.w};
    uint32_t ro[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      ro[k] = pack_bf16x2(wmul(wa, bf16_lo(ra[k])) + wmul(wb, bf16_lo(rb[k])),
                          wmul(wa, bf16_hi(ra[k])) + wmul(wb, bf16_hi(rb[k])));
    __syncwarp();   // the row's lse has been read by all its lanes before it is overwritten (lse may alias)
    if (act) {
      out[i] = make_uint4(ro[0], ro[1], ro[2], ro[3]);
      if (i % CH == 0) lse[li] = l;
    }
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace ffa

using namespace ffa;

extern "C" ffa_status ffa_lse_combine(const void* out_a, const float* lse_a, const void* out_b, const float* lse_b,
                                      void* out, float* lse, int64_t seqlen, int32_t hq, int32_t d, void* stream) {
  if (!out_a || !lse_a || !out_b || !lse_b || !out || !lse) return FFA_ERR_INVALID_ARG;
  if (!aligned16(out_a) || !aligned16(out_b) || !aligned16(out) || !aligned16(lse_a) || !aligned16(lse_b) ||
      !aligned16(lse))
    return FFA_ERR_INVALID_ARG;
  if (seqlen < 0 || hq <= 0) return FFA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FFA_ERR_UNSUPPORTED;
  if (seqlen == 0) return FFA_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t chunks = seqlen * hq * (d / 8);
  const int blocks = static_cast<int>(std::min<int64_t>((chunks + 255) / 256, int64_t{1} << 20));
  const uint4* a = static_cast<const uint4*>(out_a);
  const uint4* b = static_cast<const uint4*>(out_b);
  uint4* o = static_cast<uint4*>(out);
  if (d == 128)
    lse_combine_kernel<128><<<blocks, 256, 0, st>>>(a, lse_a, b, lse_b, o, lse, seqlen, hq);
  else
    lse_combine_kernel<64><<<blocks, 256, 0, st>>>(a, lse_a, b, lse_b, o, lse, seqlen, hq);
  return cuda_status(cudaGetLastError());
}
