// Internal declarations shared by the host API and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>
#include <cuda_runtime.h>

#include "../../include/ffa.h"

namespace ffa {

// A slice in band form, the representation the planner works on: rows
// [r_start, r_end) x columns [c_start, c_end), local (r, c) allowed when
// d_lo <= c - r <= d_hi.  FULL / CAUSAL / INV-CAUSAL / BI-CAUSAL are the four
// combinations of {no bound, 0} below and {no bound, Lk - Lq} above.  The form
// is closed under transposition (rows <-> columns, [d_lo, d_hi] -> [-d_hi,
// -d_lo]), which gives the k2q direction from the same kernels.
struct BandSlice {
  int64_t r_start, r_end, c_start, c_end;
  int64_t d_lo, d_hi;
};
constexpr int64_t kNoBound = int64_t(1) << 40;

// One direction of block metadata (q2k: rows are queries; k2q: rows are keys).
struct DirMeta {
  int64_t n_rows = 0, n_cols = 0;
  int32_t tile_r = 0, tile_c = 0;
  int32_t n_rt = 0, n_ct = 0;
  BandSlice* slices = nullptr;   // device, n_slices
  int32_t* iv_off = nullptr;     // device, n_rows + 1: per-row interval offsets
  int32_t* iv = nullptr;         // device, 2 * n_iv: (lo, hi) column intervals
  int64_t n_iv = 0;
  int32_t* full_off = nullptr;   // device, n_rt + 1
  int32_t* full_idx = nullptr;   // device, nnz_full
  int32_t* mask_off = nullptr;   // device, n_rt + 1
  int32_t* mask_idx = nullptr;   // device, nnz_mask
  int32_t* order = nullptr;      // device, n_rt: longest-work-first tile order
  int64_t nnz_full = 0, nnz_mask = 0;
  // k2q only: backward work items, one per (k-tile, q-chunk of 2^chunk_log2
  // q-tiles) with blocks, as int4 {k-tile, first Full index, first Partial
  // index, #Full | #Partial << 16}, chunk by chunk and inside a chunk in the
  // k-tiles' longest-work-first order.
  int4* items = nullptr;
  int64_t n_items = 0;
  int32_t chunk_log2 = 0;
  int32_t launches = 0;   // kernels build_plan launched for this direction
  bool owns_arrays = true;   // false: the arrays live in the plan's arena (small plans)
};
constexpr int32_t kBwdChunkLog2 = 6;   // q-tiles per backward work item: 64

// Plan-owned device words of the persistent kernels.
struct DeviceWords {
  uint32_t status;       // kStatus* bits, OR-ed by kernels
  uint32_t fwd_next;     // the forward's unit counter (cleared before each launch)
  uint32_t bwd_next;     // the backward main kernel's unit counter (cleared before each launch)
  uint32_t pad[5];
};

// Event pairs recorded around kernel launches while timing is enabled.
struct KernelTimer {
  bool enabled = false;
  struct Rec {
    int kernel;
    cudaEvent_t start, stop;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  double total_ms[FFA_KERNEL_COUNT] = {0, 0, 0, 0};
  int64_t launches[FFA_KERNEL_COUNT] = {0, 0, 0, 0};
  cudaEvent_t take();
  void begin(int kernel, cudaStream_t s, Rec& r);
  void end(Rec& r, cudaStream_t s);
  void resolve();
  void clear();
  ~KernelTimer();
};

// Per-CTA spans of the persistent kernels' last launch, for checking how
// evenly the longest-work-first deal loads the SMs: 4 words per CTA (start
// and end %globaltimer ns, units and blocks taken), one slot per kernel.
struct CtaTrace {
  uint64_t* dev = nullptr;   // [2 kernels][capacity][4], device; null while off
  int32_t capacity = 0;
  int32_t grid[2] = {0, 0};
  // The slot of kernel FFA_KERNEL_FWD or FFA_KERNEL_BWD_MAIN for a launch of
  // `ctas` CTAs, or null when tracing is off.
  uint64_t* begin(int kernel, int ctas) {
    const int slot = kernel == FFA_KERNEL_FWD ? 0 : 1;
    if (!dev || ctas > capacity) return nullptr;
    grid[slot] = ctas;
    return dev + static_cast<int64_t>(slot) * capacity * 4;
  }
};

// RAII helper: records the start event on construction and the stop event
// on destruction when the plan's timer is enabled.
struct ScopedKernelTimer {
  KernelTimer* t;
  cudaStream_t s;
  KernelTimer::Rec r{};
  ScopedKernelTimer(KernelTimer* timer, int kernel, cudaStream_t stream) : t(timer), s(stream) {
    if (t && t->enabled) t->begin(kernel, s, r);
  }
  ~ScopedKernelTimer() {
    if (t && t->enabled) t->end(r, s);
  }
};

}  // namespace ffa

struct ffa_plan_s {
  int64_t seqlen_q = 0, seqlen_k = 0;
  ffa_tile_cfg tiles{128, 128, 128, 128};
  int64_t n_slices = 0;
  int64_t mask_area = 0;
  cudaStream_t stream = nullptr;   // creation stream (frees are ordered on it)
  ffa::DirMeta q2k, k2q;
  ffa::DeviceWords* words = nullptr;   // device
  void* arena = nullptr;               // device: every metadata array of a small plan
  int num_sms = 0;
  int device = 0;
  ffa::KernelTimer timer;
  ffa::CtaTrace trace;
};

namespace ffa {

// Relative cost of a Full and a Partial block for the longest-work-first order.
constexpr int32_t kCostFull = 4;
constexpr int32_t kCostMask = 5;

// planner.cu
// Both directions of a plan's metadata (q2k from the band slices, k2q from
// their transposes), with one host synchronization for the sizes.
// A small plan puts every array, and the plan's device words, in one
// allocation (*arena, *words set); a large one leaves both null.
ffa_status build_plan(DirMeta& q2k, DirMeta& k2q, const BandSlice* band, const BandSlice* tband, int64_t n_slices,
                      cudaStream_t stream, int num_sms, void** arena, DeviceWords** words);
void free_direction(DirMeta& m, cudaStream_t stream);

// Host helper: record a CUDA error and map it.
// Host check of a slice list (api.cu): ranges, types and disjoint coverage;
// the non-empty slices in band form and the union's mask area.
ffa_status validate_and_convert(const ffa_attn_slice* slices, int64_t n, int64_t sq, int64_t sk,
                                std::vector<BandSlice>& out, int64_t& area);
inline ffa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FFA_OK : FFA_ERR_CUDA; }

}  // namespace ffa
