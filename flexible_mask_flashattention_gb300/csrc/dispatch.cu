// Dispatch solver: query chunks to context-parallel buckets by mask area.
//
// MagiAttention blog, "Dispatch Solver" (Figure 10): the sequence is cut into
// n = seqlen / chunk_size query chunks C_i, each with its mask area
// Area(C_i); the chunks go to cp_size buckets of exactly n / cp_size chunks
// each (seqlen divisible by cp_size * chunk_size), so that every rank holds
// the same number of tokens for the token-priced layers, and the largest
// bucket area is kept small.  That minimum is NP-hard; the pages' solver is a
// min-heap greedy: estimate each chunk's area, then hand the heavier chunks
// first to the bucket with the least load so far.
//
// Host code only (no CUDA calls): it plans work across ranks and runs in
// O(n log n) after the chunk areas, which come in closed form from the
// slices' band form.
#include <algorithm>
#include <cstdint>
#include <functional>
#include <numeric>
#include <queue>
#include <utility>
#include <vector>

#include "ffa_internal.h"

namespace ffa {
namespace {

// sum over r in [s, e) of max(0, alpha * r + beta), alpha in {-1, 0, 1}.
int64_t sum_positive_linear(int64_t alpha, int64_t beta, int64_t s, int64_t e) {
  if (e <= s) return 0;
  if (alpha == 0) return beta > 0 ? beta * (e - s) : 0;
  // keep the rows where alpha r + beta > 0, i.e. r > -beta (alpha = 1) or r < beta (alpha = -1)
  if (alpha > 0) s = std::max(s, -beta + 1);
  else e = std::min(e, beta);
  if (e <= s) return 0;
  const int64_t n = e - s;
  // sum of alpha r + beta over r = s .. e - 1
  return alpha * ((s + e - 1) * n / 2) + beta * n;
}

// Allowed pairs of band slice b in its rows [r0, r1) (absolute rows):
// local row r keeps the local columns c in [0, Lk) with d_lo <= c - r <= d_hi,
// i.e. max(0, min(Lk - 1, r + d_hi) - max(0, r + d_lo) + 1) of them.  The
// count is linear between the rows where the two clamps switch, so each
// piece is an arithmetic series.
int64_t band_area_in_rows(const BandSlice& b, int64_t r0, int64_t r1) {
  const int64_t s = std::max(r0, b.r_start) - b.r_start, e = std::min(r1, b.r_end) - b.r_start;
  if (e <= s) return 0;
  const int64_t lk = b.c_end - b.c_start, lq = b.r_end - b.r_start;
  // no lower bound: below every local row, so that the clamp at 0 decides
  const int64_t lo_d = b.d_lo <= -kNoBound ? -(lq + lk + 1) : b.d_lo;
  const int64_t hi_d = b.d_hi >= kNoBound ? lk : b.d_hi;     // no upper bound: the clamp at Lk - 1 decides
  // hi(r) = min(Lk - 1, r + hi_d) switches at r = Lk - 1 - hi_d; lo(r) = max(0, r + lo_d) at r = -lo_d
  int64_t cuts[4] = {s, std::clamp<int64_t>(lk - 1 - hi_d, s, e), std::clamp<int64_t>(-lo_d, s, e), e};
  std::sort(cuts + 1, cuts + 3);
  int64_t total = 0;
  for (int i = 0; i < 3; ++i) {
    const int64_t a = cuts[i], z = cuts[i + 1];
    if (z <= a) continue;
    // on [a, z) both clamps are fixed: take them at r = a (at the switch rows
    // themselves both forms agree)
    const bool hi_clamped = a + hi_d >= lk - 1, lo_clamped = a + lo_d < 0;
    const int64_t alpha = (hi_clamped ? 0 : 1) - (lo_clamped ? 0 : 1);
    const int64_t beta = (hi_clamped ? lk - 1 : hi_d) - (lo_clamped ? 0 : lo_d) + 1;
    total += sum_positive_linear(alpha, beta, a, z);
  }
  return total;
}

}  // namespace
}  // namespace ffa

using namespace ffa;

extern "C" ffa_status ffa_dispatch_solve(const ffa_attn_slice* slices, int64_t n_slices, int64_t seqlen_q,
                                         int64_t seqlen_k, int64_t chunk_size, int32_t cp_size, int64_t* chunk_area,
                                         int32_t* bucket_of_chunk, int64_t* bucket_area) {
  if (!bucket_of_chunk || (n_slices > 0 && !slices) || n_slices < 0) return FFA_ERR_INVALID_ARG;
  if (seqlen_q <= 0 || seqlen_k < 0 || chunk_size <= 0 || cp_size <= 0) return FFA_ERR_INVALID_ARG;
  if (seqlen_q % (static_cast<int64_t>(cp_size) * chunk_size) != 0) return FFA_ERR_INVALID_ARG;
  std::vector<BandSlice> bands;
  int64_t total_area = 0;
  const ffa_status st = validate_and_convert(slices, n_slices, seqlen_q, seqlen_k, bands, total_area);
  if (st != FFA_OK) return st;
  const int64_t n = seqlen_q / chunk_size;
  // 1. Area(C_i): every slice adds its allowed pairs in the chunk's rows
  std::vector<int64_t> area(static_cast<size_t>(n), 0);
  for (const BandSlice& b : bands)
    for (int64_t c = b.r_start / chunk_size; c * chunk_size < b.r_end && c < n; ++c)
      area[c] += band_area_in_rows(b, c * chunk_size, (c + 1) * chunk_size);
  // 2. the heavier chunks first (ties: lower chunk index)
  std::vector<int64_t> order(static_cast<size_t>(n));
  std::iota(order.begin(), order.end(), int64_t{0});
  std::stable_sort(order.begin(), order.end(), [&](int64_t x, int64_t y) { return area[x] > area[y]; });
  // 3. each to the least-loaded bucket that still has room (ties: lower bucket index)
  const int64_t cap = n / cp_size;
  using Entry = std::pair<int64_t, int32_t>;   // (load, bucket)
  std::priority_queue<Entry, std::vector<Entry>, std::greater<Entry>> heap;
  for (int32_t j = 0; j < cp_size; ++j) heap.push({0, j});
  std::vector<int64_t> load(static_cast<size_t>(cp_size), 0), count(static_cast<size_t>(cp_size), 0);
  for (int64_t c : order) {
    const Entry top = heap.top();
    heap.pop();
    const int32_t j = top.second;
    bucket_of_chunk[c] = j;
    load[j] += area[c];
    if (++count[j] < cap) heap.push({load[j], j});
  }
  if (chunk_area) std::copy(area.begin(), area.end(), chunk_area);
  if (bucket_area) std::copy(load.begin(), load.end(), bucket_area);
  return FFA_OK;
}
