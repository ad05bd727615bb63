// Host side of the C ABI: argument and slice validation, plan lifetime,
// metadata copies and the device status word.  Slices and mask semantics are
// those of the MagiAttention blog, section "Flex-Flash-Attention and
// AttnSlice"; the block metadata those of the documentation's "FFA_FA4
// backend" section.
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "ffa_internal.h"

namespace ffa {

// planner.cu: copies n_words 8-byte words of device memory to the host
// through the planner's mapped buffer (a kernel and a stream synchronization,
// no copy engine), so that a small read never waits behind other streams'
// copies.
cudaError_t read_device_words(const void* src, void* dst, int64_t n_words, cudaStream_t stream);
namespace {

constexpr int64_t kMaxSeqlen = int64_t(1) << 30;

bool pow2_in(int32_t x, int32_t lo, int32_t hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

// Allowed pairs of one slice of a given type, summed row by row.
int64_t slice_area(int64_t lq, int64_t lk, int32_t type) {
  if (lq <= 0 || lk <= 0) return 0;
  switch (type) {
    case FFA_MASK_FULL:
      return lq * lk;
    case FFA_MASK_CAUSAL:   // row r keeps min(Lk, max(0, r + Lk - Lq + 1)) keys
      return lq <= lk ? lq * (lk - lq) + lq * (lq + 1) / 2 : lk * (lk + 1) / 2;
    case FFA_MASK_INV_CAUSAL:   // row r keeps max(0, Lk - r) keys
      return lq <= lk ? lq * lk - lq * (lq - 1) / 2 : lk * (lk + 1) / 2;
    case FFA_MASK_BI_CAUSAL:   // every row keeps Lk - Lq + 1 keys, or none
      return lk >= lq ? lq * (lk - lq + 1) : 0;
    default:
      return 0;
  }
}

BandSlice to_band(const ffa_attn_slice& s) {
  BandSlice b;
  b.r_start = s.q_start;
  b.r_end = s.q_end;
  b.c_start = s.k_start;
  b.c_end = s.k_end;
  const int64_t diag = (s.k_end - s.k_start) - (s.q_end - s.q_start);
  const bool lower = s.mask_type == FFA_MASK_INV_CAUSAL || s.mask_type == FFA_MASK_BI_CAUSAL;
  const bool upper = s.mask_type == FFA_MASK_CAUSAL || s.mask_type == FFA_MASK_BI_CAUSAL;
  b.d_lo = lower ? 0 : -kNoBound;
  b.d_hi = upper ? diag : kNoBound;
  return b;
}

BandSlice transpose(const BandSlice& s) {
  BandSlice t;
  t.r_start = s.c_start;
  t.r_end = s.c_end;
  t.c_start = s.r_start;
  t.c_end = s.r_end;
  t.d_lo = s.d_hi >= kNoBound ? -kNoBound : -s.d_hi;
  t.d_hi = s.d_lo <= -kNoBound ? kNoBound : -s.d_lo;
  return t;
}

// Do two band slices allow a common (row, column)?  Over the intersection of
// their rectangles both constraints read L <= j - i <= U; an integer pair
// exists iff some row i in range leaves [max(J0, i + L), min(J1 - 1, i + U)]
// non-empty.
bool bands_overlap(const BandSlice& a, const BandSlice& b) {
  const int64_t i0 = std::max(a.r_start, b.r_start), i1 = std::min(a.r_end, b.r_end);
  const int64_t j0 = std::max(a.c_start, b.c_start), j1 = std::min(a.c_end, b.c_end);
  if (i0 >= i1 || j0 >= j1) return false;
  const int64_t la = a.d_lo <= -kNoBound ? -kNoBound : a.d_lo + a.c_start - a.r_start;
  const int64_t lb = b.d_lo <= -kNoBound ? -kNoBound : b.d_lo + b.c_start - b.r_start;
  const int64_t ua = a.d_hi >= kNoBound ? kNoBound : a.d_hi + a.c_start - a.r_start;
  const int64_t ub = b.d_hi >= kNoBound ? kNoBound : b.d_hi + b.c_start - b.r_start;
  const int64_t L = std::max(la, lb), U = std::min(ua, ub);
  if (L > U) return false;
  const int64_t lo = std::max(i0, j0 - U), hi = std::min(i1 - 1, j1 - 1 - L);
  return lo <= hi;
}

}  // namespace

ffa_status validate_and_convert(const ffa_attn_slice* slices, int64_t n, int64_t sq, int64_t sk,
                                std::vector<BandSlice>& out, int64_t& area) {
  out.clear();
  area = 0;
  for (int64_t i = 0; i < n; ++i) {
    const ffa_attn_slice& s = slices[i];
    if (s.mask_type < FFA_MASK_FULL || s.mask_type > FFA_MASK_BI_CAUSAL) return FFA_ERR_INVALID_SLICE;
    if (s.q_start < 0 || s.q_start > s.q_end || s.q_end > sq) return FFA_ERR_INVALID_SLICE;
    if (s.k_start < 0 || s.k_start > s.k_end || s.k_end > sk) return FFA_ERR_INVALID_SLICE;
    const int64_t a = slice_area(s.q_end - s.q_start, s.k_end - s.k_start, s.mask_type);
    if (a == 0) continue;   // zero-length or zero-area slices are accepted and ignored
    area += a;
    out.push_back(to_band(s));
  }
  std::vector<int64_t> idx(out.size());
  for (size_t i = 0; i < idx.size(); ++i) idx[i] = static_cast<int64_t>(i);
  std::sort(idx.begin(), idx.end(), [&](int64_t x, int64_t y) { return out[x].r_start < out[y].r_start; });
  for (size_t x = 0; x < idx.size(); ++x) {
    const BandSlice& a = out[idx[x]];
    for (size_t y = x + 1; y < idx.size() && out[idx[y]].r_start < a.r_end; ++y)
      if (bands_overlap(a, out[idx[y]])) return FFA_ERR_OVERLAPPING_COVERAGE;
  }
  return FFA_OK;
}

cudaEvent_t KernelTimer::take() {
  if (!pool.empty()) {
    cudaEvent_t e = pool.back();
    pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
void KernelTimer::begin(int kernel, cudaStream_t s, Rec& r) {
  r.kernel = kernel;
  r.start = take();
  r.stop = take();
  cudaEventRecord(r.start, s);
}
void KernelTimer::end(Rec& r, cudaStream_t s) {
  cudaEventRecord(r.stop, s);
  recs.push_back(r);
}
void KernelTimer::resolve() {
  for (Rec& r : recs) {
    float ms = 0.f;
    cudaEventSynchronize(r.stop);
    if (cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
      total_ms[r.kernel] += ms;
      launches[r.kernel] += 1;
    }
    pool.push_back(r.start);
    pool.push_back(r.stop);
  }
  recs.clear();
}
void KernelTimer::clear() {
  for (Rec& r : recs) {
    pool.push_back(r.start);
    pool.push_back(r.stop);
  }
  recs.clear();
  for (int i = 0; i < FFA_KERNEL_COUNT; ++i) {
    total_ms[i] = 0;
    launches[i] = 0;
  }
}
KernelTimer::~KernelTimer() {
  clear();
  for (cudaEvent_t e : pool) cudaEventDestroy(e);
}

}  // namespace ffa

using namespace ffa;

extern "C" {

const char* ffa_status_string(ffa_status s) {
  switch (s) {
    case FFA_OK: return "ok";
    case FFA_ERR_INVALID_ARG: return "invalid argument";
    case FFA_ERR_INVALID_SLICE: return "invalid slice";
    case FFA_ERR_OVERLAPPING_COVERAGE: return "a (query, key) pair is covered by two slices";
    case FFA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FFA_ERR_OVERFLOW: return "count exceeds the int32 index range";
    case FFA_ERR_CUDA: return "CUDA runtime error";
    case FFA_ERR_DEVICE_CHECK: return "a kernel reported a failure";
  }
  return "unknown status";
}

ffa_status ffa_plan_destroy(ffa_plan_t plan) {
  if (!plan) return FFA_OK;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(plan->device);
  free_direction(plan->q2k, plan->stream);
  free_direction(plan->k2q, plan->stream);
  if (plan->words && !plan->arena) cudaFreeAsync(plan->words, plan->stream);
  if (plan->trace.dev) cudaFreeAsync(plan->trace.dev, plan->stream);
  if (plan->arena) cudaFreeAsync(plan->arena, plan->stream);
  cudaSetDevice(prev);
  delete plan;
  return FFA_OK;
}

ffa_status ffa_plan_create(const ffa_attn_slice* slices, int64_t n_slices, int64_t seqlen_q, int64_t seqlen_k,
                           const ffa_tile_cfg* tiles, void* stream, ffa_plan_t* out_plan) {
  if (!out_plan) return FFA_ERR_INVALID_ARG;
  *out_plan = nullptr;
  if (n_slices < 0 || (n_slices > 0 && !slices)) return FFA_ERR_INVALID_ARG;
  if (seqlen_q < 0 || seqlen_k < 0) return FFA_ERR_INVALID_ARG;
  if (seqlen_q > kMaxSeqlen || seqlen_k > kMaxSeqlen) return FFA_ERR_OVERFLOW;
  ffa_tile_cfg t = tiles ? *tiles : ffa_tile_cfg{0, 0, 0, 0};
  for (int32_t* x : {&t.fwd_bm, &t.fwd_bn, &t.bwd_bm, &t.bwd_bn}) {
    if (*x == 0) *x = 128;
    if (!pow2_in(*x, 8, 1024)) return FFA_ERR_UNSUPPORTED;
  }

  std::vector<BandSlice> band;
  int64_t area = 0;
  ffa_status st = validate_and_convert(slices, n_slices, seqlen_q, seqlen_k, band, area);
  if (st != FFA_OK) return st;

  ffa_plan_s* p = new (std::nothrow) ffa_plan_s();
  if (!p) return FFA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  p->seqlen_q = seqlen_q;
  p->seqlen_k = seqlen_k;
  p->tiles = t;
  p->n_slices = static_cast<int64_t>(band.size());
  p->mask_area = area;
  p->stream = s;
  if (cudaGetDevice(&p->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
    delete p;
    return FFA_ERR_CUDA;
  }
  DirMeta& q = p->q2k;
  q.n_rows = seqlen_q;
  q.n_cols = seqlen_k;
  q.tile_r = t.fwd_bm;
  q.tile_c = t.fwd_bn;
  q.n_rt = static_cast<int32_t>((seqlen_q + t.fwd_bm - 1) / t.fwd_bm);
  q.n_ct = static_cast<int32_t>((seqlen_k + t.fwd_bn - 1) / t.fwd_bn);
  DirMeta& k = p->k2q;   // rows are keys (tiles of bwd_bn), columns queries (tiles of bwd_bm)
  k.n_rows = seqlen_k;
  k.n_cols = seqlen_q;
  k.tile_r = t.bwd_bn;
  k.tile_c = t.bwd_bm;
  k.n_rt = static_cast<int32_t>((seqlen_k + t.bwd_bn - 1) / t.bwd_bn);
  k.n_ct = static_cast<int32_t>((seqlen_q + t.bwd_bm - 1) / t.bwd_bm);
  std::vector<BandSlice> tband(band.size());
  for (size_t i = 0; i < band.size(); ++i) tband[i] = transpose(band[i]);

  st = build_plan(q, k, band.data(), tband.data(), static_cast<int64_t>(band.size()), s, p->num_sms, &p->arena,
                  &p->words);
  // a small plan's words live in its arena, cleared by its one kernel, and it has already waited
  if (st == FFA_OK && !p->words) {
    if (cudaMallocAsync(reinterpret_cast<void**>(&p->words), sizeof(DeviceWords), s) != cudaSuccess ||
        cudaMemsetAsync(p->words, 0, sizeof(DeviceWords), s) != cudaSuccess)
      st = FFA_ERR_CUDA;
    if (st == FFA_OK && cudaStreamSynchronize(s) != cudaSuccess) st = FFA_ERR_CUDA;
  }
  if (st != FFA_OK) {
    cudaStreamSynchronize(s);
    ffa_plan_destroy(p);
    cudaStreamSynchronize(s);
    return st;
  }
  *out_plan = p;
  return FFA_OK;
}

ffa_status ffa_plan_info(ffa_plan_t p, ffa_plan_info_t* out) {
  if (!p || !out) return FFA_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  out->seqlen_q = p->seqlen_q;
  out->seqlen_k = p->seqlen_k;
  out->tiles = p->tiles;
  out->m_tiles = p->q2k.n_rt;
  out->n_tiles = p->q2k.n_ct;
  out->bwd_m_tiles = p->k2q.n_ct;
  out->bwd_n_tiles = p->k2q.n_rt;
  out->n_slices = p->n_slices;
  out->mask_area = p->mask_area;
  out->q2k_full = p->q2k.nnz_full;
  out->q2k_mask = p->q2k.nnz_mask;
  out->k2q_full = p->k2q.nnz_full;
  out->k2q_mask = p->k2q.nnz_mask;
  out->row_intervals = p->q2k.n_iv;
  out->key_intervals = p->k2q.n_iv;
  out->bwd_items = p->k2q.n_items;
  int64_t bytes = sizeof(DeviceWords);
  for (const DirMeta* m : {&p->q2k, &p->k2q})
    bytes += (m->owns_arrays ? static_cast<int64_t>(sizeof(BandSlice)) * p->n_slices : 0) + 4 * (m->n_rows + 1) +
             8 * m->n_iv +
             4 * 3 * static_cast<int64_t>(m->n_rt) + 8 + 4 * (m->nnz_full + m->nnz_mask) + 16 * m->n_items;
  out->plan_bytes = bytes;
  out->bwd_chunk_tiles = 1 << p->k2q.chunk_log2;
  out->plan_launches = p->q2k.launches + p->k2q.launches;
  return FFA_OK;
}

ffa_status ffa_plan_copy_csr(ffa_plan_t p, int32_t direction, int32_t* full_off, int32_t* full_idx, int32_t* mask_off,
                             int32_t* mask_idx, int32_t* order) {
  if (!p || (direction != 0 && direction != 1)) return FFA_ERR_INVALID_ARG;
  const DirMeta& m = direction == 0 ? p->q2k : p->k2q;
  cudaStream_t s = p->stream;
  const size_t rows = static_cast<size_t>(m.n_rt);
  cudaError_t e = cudaSuccess;
  if (full_off && e == cudaSuccess)
    e = cudaMemcpyAsync(full_off, m.full_off, 4 * (rows + 1), cudaMemcpyDeviceToHost, s);
  if (mask_off && e == cudaSuccess)
    e = cudaMemcpyAsync(mask_off, m.mask_off, 4 * (rows + 1), cudaMemcpyDeviceToHost, s);
  if (full_idx && m.nnz_full > 0 && e == cudaSuccess)
    e = cudaMemcpyAsync(full_idx, m.full_idx, 4 * static_cast<size_t>(m.nnz_full), cudaMemcpyDeviceToHost, s);
  if (mask_idx && m.nnz_mask > 0 && e == cudaSuccess)
    e = cudaMemcpyAsync(mask_idx, m.mask_idx, 4 * static_cast<size_t>(m.nnz_mask), cudaMemcpyDeviceToHost, s);
  if (order && rows > 0 && e == cudaSuccess) e = cudaMemcpyAsync(order, m.order, 4 * rows, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

ffa_status ffa_plan_copy_bwd_items(ffa_plan_t p, int32_t* items) {
  if (!p || !items) return FFA_ERR_INVALID_ARG;
  cudaError_t e = cudaSuccess;
  if (p->k2q.n_items > 0)
    e = cudaMemcpyAsync(items, p->k2q.items, sizeof(int4) * static_cast<size_t>(p->k2q.n_items),
                        cudaMemcpyDeviceToHost, p->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(p->stream);
  return cuda_status(e);
}

ffa_status ffa_plan_copy_row_intervals(ffa_plan_t p, int32_t* off, int32_t* iv) {
  if (!p) return FFA_ERR_INVALID_ARG;
  cudaStream_t s = p->stream;
  cudaError_t e = cudaSuccess;
  if (off) e = cudaMemcpyAsync(off, p->q2k.iv_off, 4 * static_cast<size_t>(p->seqlen_q + 1), cudaMemcpyDeviceToHost, s);
  if (iv && p->q2k.n_iv > 0 && e == cudaSuccess)
    e = cudaMemcpyAsync(iv, p->q2k.iv, 8 * static_cast<size_t>(p->q2k.n_iv), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

ffa_status ffa_plan_enable_timing(ffa_plan_t p, int32_t enable) {
  if (!p) return FFA_ERR_INVALID_ARG;
  p->timer.clear();
  p->timer.enabled = enable != 0;
  return FFA_OK;
}

ffa_status ffa_plan_read_timing(ffa_plan_t p, double* total_ms, int64_t* launches) {
  if (!p) return FFA_ERR_INVALID_ARG;
  p->timer.resolve();
  for (int i = 0; i < FFA_KERNEL_COUNT; ++i) {
    if (total_ms) total_ms[i] = p->timer.total_ms[i];
    if (launches) launches[i] = p->timer.launches[i];
  }
  return FFA_OK;
}

ffa_status ffa_plan_enable_cta_trace(ffa_plan_t p, int32_t enable) {
  if (!p) return FFA_ERR_INVALID_ARG;
  if (enable && !p->trace.dev) {
    const size_t bytes = sizeof(uint64_t) * 2 * 4 * static_cast<size_t>(p->num_sms);
    cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&p->trace.dev), bytes, p->stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->trace.dev, 0, bytes, p->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->stream);
    if (e != cudaSuccess) return FFA_ERR_CUDA;
    p->trace.capacity = p->num_sms;
    p->trace.grid[0] = p->trace.grid[1] = 0;
  } else if (!enable && p->trace.dev) {
    cudaError_t e = cudaFreeAsync(p->trace.dev, p->stream);
    p->trace.dev = nullptr;
    p->trace.capacity = 0;
    if (e != cudaSuccess) return FFA_ERR_CUDA;
  }
  return FFA_OK;
}

ffa_status ffa_plan_read_cta_trace(ffa_plan_t p, int32_t kernel, void* stream, uint64_t* out, int32_t capacity,
                                   int32_t* n_ctas) {
  if (!p || !n_ctas || (kernel != FFA_KERNEL_FWD && kernel != FFA_KERNEL_BWD_MAIN)) return FFA_ERR_INVALID_ARG;
  const int slot = kernel == FFA_KERNEL_FWD ? 0 : 1;
  *n_ctas = p->trace.dev ? p->trace.grid[slot] : 0;
  if (*n_ctas == 0) return FFA_OK;
  if (!out || capacity < *n_ctas) return FFA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(out, p->trace.dev + static_cast<int64_t>(slot) * p->trace.capacity * 4,
                                  sizeof(uint64_t) * 4 * static_cast<size_t>(*n_ctas), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return cuda_status(e);
}

ffa_status ffa_plan_check_status(ffa_plan_t p, void* stream, uint32_t* status_out) {
  if (!p) return FFA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint64_t w64 = 0;   // the status word and the padding after it (the words are 256-byte aligned)
  cudaError_t e = read_device_words(&p->words->status, &w64, 1, s);
  const uint32_t w = static_cast<uint32_t>(w64 & 0xffffffffu);
  if (e == cudaSuccess) e = cudaMemsetAsync(&p->words->status, 0, sizeof(w), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (status_out) *status_out = w;
  if (e != cudaSuccess) return FFA_ERR_CUDA;
  return w ? FFA_ERR_DEVICE_CHECK : FFA_OK;
}

}  // extern "C"
