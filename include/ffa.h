/*
 * ffa.h -- C ABI of the GB300 (sm_103a) Flex-Flash-Attention hot path.
 *
 * Fused softmax attention, forward and backward, over a mask given as a list
 * of AttnSlices (QRange, KRange, MaskType) -- MagiAttention blog, section
 * "Flex-Flash-Attention and AttnSlice", and the MagiAttention documentation,
 * "FFA_FA4 backend" items 1 (create_block_mask: Full / Partial / Empty blocks
 * in q2k and k2q order) and 2 (CSR block metadata with full_block_offset and
 * mask_block_offset).
 *
 * Conventions shared by every call:
 *  - Every call returns an ffa_status and never throws.  Arguments are checked
 *    on the host before anything is launched; a rejected call launches nothing.
 *  - Device calls are ordered on the `stream` argument (a cudaStream_t passed
 *    as void*, NULL = legacy default stream) and return before the GPU work
 *    ends, except where stated.
 *  - Tensors are dense, contiguous, packed variable-length batches of one
 *    sequence (batch 1, as in the pages' benchmark settings):
 *      q, out, dout, dq : bf16 [seqlen_q][hq][d]
 *      k, v, dk, dv     : bf16 [seqlen_k][hkv][d]
 *      lse              : fp32 [hq][seqlen_q]
 *    All device pointers must be 16-byte aligned.  The caller owns them.
 *  - Mask semantics.  For slice s with Lq = q_end - q_start and
 *    Lk = k_end - k_start, query i and key j with slice-local r = i - q_start,
 *    c = j - k_start are allowed when:
 *      FULL        always
 *      CAUSAL      c <= r + (Lk - Lq)       (diagonal through the bottom-right corner)
 *      INV_CAUSAL  c >= r                   (diagonal through the top-left corner)
 *      BI_CAUSAL   r <= c <= r + (Lk - Lq)  (both)
 *    The global mask is the union over slices.  q-ranges of different slices
 *    may overlap, but no (query, key) pair may be allowed by two slices: then
 *    the union equals the log-sum-exp merge of per-slice partial results (the
 *    pages' reduction of partial outputs, blog Figure 5).
 *  - A query row with no allowed key gets out = 0, lse = -inf, dq = 0.
 *  - GQA: q head h reads kv head h / (hq / hkv).
 *  - lse is the natural log of sum_j exp(scale * q_i . k_j) over allowed j.
 */
#ifndef FFA_GB300_H
#define FFA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FFA_OK = 0,
  FFA_ERR_INVALID_ARG = 1,          /* null / misaligned pointer, bad size, bad head counts */
  FFA_ERR_INVALID_SLICE = 2,        /* range outside [0, seqlen), start > end, unknown type */
  FFA_ERR_OVERLAPPING_COVERAGE = 3, /* some (query, key) pair is allowed by two slices */
  FFA_ERR_UNSUPPORTED = 4,          /* valid but not implemented (head dim, tile size) */
  FFA_ERR_OVERFLOW = 5,             /* a count exceeds the int32 index range */
  FFA_ERR_CUDA = 6,                 /* a CUDA runtime call failed */
  FFA_ERR_DEVICE_CHECK = 7          /* a kernel recorded a failure in the plan's status word */
} ffa_status;

typedef enum {
  FFA_MASK_FULL = 0,
  FFA_MASK_CAUSAL = 1,
  FFA_MASK_INV_CAUSAL = 2,
  FFA_MASK_BI_CAUSAL = 3
} ffa_mask_type;

/* One AttnSlice, half-open ranges [q_start, q_end) x [k_start, k_end). */
typedef struct {
  int64_t q_start, q_end, k_start, k_end;
  int32_t mask_type; /* ffa_mask_type */
  int32_t reserved;  /* set to 0 */
} ffa_attn_slice;

typedef struct ffa_plan_s* ffa_plan_t;

/* Tile sizes of a plan (documentation, "FFA_FA4 backend" item 1: the blocks
 * the mask is classified in).  Each is a power of two in [8, 1024]; 0 means
 * the default, 128.
 *   fwd_bm x fwd_bn  query rows x key columns of a block in q2k (forward) order
 *   bwd_bm x bwd_bn  query rows x key columns of a block in k2q (backward) order
 * ffa_fwd needs a 128 x 128 forward tile and ffa_bwd a 128 x 128 backward
 * tile (FFA_ERR_UNSUPPORTED otherwise); other sizes serve the metadata alone. */
typedef struct {
  int32_t fwd_bm, fwd_bn, bwd_bm, bwd_bn;
} ffa_tile_cfg;

/* Summary of a plan (host values). */
typedef struct {
  int64_t seqlen_q, seqlen_k;
  ffa_tile_cfg tiles;         /* the tile sizes used (defaults filled in) */
  int32_t m_tiles, n_tiles;   /* forward grid: ceil(seqlen_q / fwd_bm), ceil(seqlen_k / fwd_bn) */
  int32_t bwd_m_tiles, bwd_n_tiles; /* backward grid: ceil(seqlen_q / bwd_bm), ceil(seqlen_k / bwd_bn) */
  int64_t n_slices;           /* slices kept (zero-area slices are dropped) */
  int64_t mask_area;          /* allowed (query, key) pairs of the union mask */
  int64_t q2k_full, q2k_mask; /* Full / Partial blocks in q2k (forward) order */
  int64_t k2q_full, k2q_mask; /* Full / Partial blocks in k2q (backward) order */
  int64_t row_intervals;      /* allowed key intervals summed over query rows */
  int64_t key_intervals;      /* allowed query intervals summed over key rows */
  int64_t bwd_items;          /* backward work items, see ffa_plan_copy_bwd_items */
  int64_t plan_bytes;         /* device bytes of the plan's metadata (intervals, CSR lists, orders,
                                 work items, and the slices where the plan keeps them) */
  int32_t bwd_chunk_tiles;    /* q-tiles per backward q-chunk */
  int32_t plan_launches;      /* kernels ffa_plan_create launched for this plan */
} ffa_plan_info_t;

/*
 * Build the block metadata of a mask (documentation, "FFA_FA4 backend" items
 * 1-2): validates the slices on the host, then on the GPU derives every query
 * row's allowed key intervals, classifies each (q-tile, k-tile) pair as Full,
 * Partial or Empty in q2k order (a block with out-of-bounds rows only may be
 * Full; with out-of-bounds columns it is never Full) and in k2q order (any
 * out-of-bounds row or column makes it Partial), stores the non-empty blocks
 * as CSR lists with ascending indices, and orders the tiles of each direction
 * longest-work-first for the persistent kernels (the min-heap greedy of the
 * pages' dispatch solver, applied to SMs).
 *
 *  slices   host array of n_slices entries (read during the call only)
 *  tiles    host pointer to the tile sizes (read during the call only), or
 *           NULL for 128 x 128 in both directions; see ffa_tile_cfg
 *  stream   work is ordered on it, and the call returns after the plan is
 *           complete: it synchronizes the stream twice (once for the sizes
 *           of both directions' lists and of the backward work items, once
 *           at the end), or once for a small plan (both lengths at most 2048,
 *           at most 256 slices), which one kernel builds.  Its small host
 *           transfers go through a pinned, device-mapped buffer moved by
 *           kernels, so they never wait behind copies that other streams
 *           have in flight
 *  out_plan receives the handle.  The plan owns its device memory (allocated
 *           stream-ordered on `stream`) until ffa_plan_destroy.  A plan is
 *           immutable and may be shared by calls for any heads and tensors
 *           of the same sequence lengths, but by one stream at a time (the
 *           kernels record failures in the plan's status word, and timing
 *           records events in it).
 * Errors: FFA_ERR_INVALID_ARG, FFA_ERR_INVALID_SLICE,
 * FFA_ERR_OVERLAPPING_COVERAGE, FFA_ERR_UNSUPPORTED, FFA_ERR_OVERFLOW,
 * FFA_ERR_CUDA.  On error *out_plan is NULL and nothing is left allocated.
 */
ffa_status ffa_plan_create(const ffa_attn_slice* slices, int64_t n_slices, int64_t seqlen_q, int64_t seqlen_k,
                           const ffa_tile_cfg* tiles, void* stream, ffa_plan_t* out_plan);

/* Release a plan.  Work that uses it must be complete, or ordered before this
 * call on the stream the plan was created on.  NULL is accepted. */
ffa_status ffa_plan_destroy(ffa_plan_t plan);

/* Fill *out with the plan's sizes (host only, no GPU work). */
ffa_status ffa_plan_info(ffa_plan_t plan, ffa_plan_info_t* out);

/*
 * Copy one CSR direction to host arrays (synchronous; for tests and tools).
 *  direction 0 = q2k: m_tiles+1 offsets, lists of k-tiles per q-tile (forward tiles);
 *  direction 1 = k2q: bwd_n_tiles+1 offsets, lists of q-tiles per k-tile (backward tiles).
 *  full_off/mask_off receive rows+1 int32 offsets; full_idx/mask_idx receive
 *  the block indices (sizes from ffa_plan_info); order receives the `rows`
 *  tile indices in longest-work-first order.  Any pointer may be NULL to
 *  skip that array.
 */
ffa_status ffa_plan_copy_csr(ffa_plan_t plan, int32_t direction, int32_t* full_off, int32_t* full_idx,
                             int32_t* mask_off, int32_t* mask_idx, int32_t* order);

/*
 * Copy the backward work items to a host array of 4 * bwd_items int32
 * (synchronous; for tests and tools).  The k2q lists of each k-tile are cut
 * into q-chunks of bwd_chunk_tiles consecutive q-tiles; an item is one
 * (k-tile, q-chunk) pair with at least one block, stored as
 *   { k-tile, index of its first Full block in the k2q Full list,
 *     index of its first Partial block in the k2q Partial list,
 *     #Full blocks | #Partial blocks << 16 }.
 * Items are ordered by q-chunk, and inside a q-chunk by the k-tiles'
 * longest-work-first order, so that the items ffa_bwd runs at one time
 * share their query rows in L2.
 */
ffa_status ffa_plan_copy_bwd_items(ffa_plan_t plan, int32_t* items);

/* Copy the query rows' key intervals: off [seqlen_q + 1] and iv [2 * n]
 * (lo, hi) pairs, half-open, ascending within a row (synchronous). */
ffa_status ffa_plan_copy_row_intervals(ffa_plan_t plan, int32_t* off, int32_t* iv);

/*
 * Forward pass (blog Figure 5: load, on-chip compute, merge of partials):
 * out_i = sum_j softmax_j(scale * q_i . k_j) v_j over allowed j, and lse.
 * One persistent kernel, one CTA per SM: each CTA takes a first (q-tile,
 * head pair) unit and then pops the next one of the plan's longest-work-first
 * order from one counter in the plan (cleared by a 4-byte memset on `stream`
 * before the launch), streams the K/V tiles of the q2k CSR lists by TMA, runs
 * Q K^T and P V on the tensor cores with TMEM accumulators, and applies
 * per-element masking on Partial tiles only.
 *
 *  q, k, v  bf16 device tensors (layouts above); out bf16 [seqlen_q][hq][d]
 *  lse      fp32 [hq][seqlen_q]
 *  hq % hkv == 0; d in {64, 128}; the plan's forward tiles must be 128 x 128
 *  and its sequence lengths must equal seqlen_q / seqlen_k.
 * Errors: FFA_ERR_INVALID_ARG, FFA_ERR_UNSUPPORTED, FFA_ERR_CUDA.  A kernel
 * timeout (which only a broken plan can cause) is recorded in the plan's
 * status word; see ffa_plan_check_status.
 */
ffa_status ffa_fwd(const void* q, const void* k, const void* v, int64_t seqlen_q, int64_t seqlen_k, int32_t hq,
                   int32_t hkv, int32_t d, ffa_plan_t plan, float scale, void* out, float* lse, void* stream);

/*
 * Forward pass merged into a partial result already in (out, lse), by LSE
 * (blog Figure 5: partial results of parts of the mask are merged by
 * reduction; the distributed pass joins the fragments computed from local
 * and remote KV the same way).  On entry (out, lse) hold a partial result over
 * keys this plan does not allow: for rows where lse = -inf it is empty and
 * its out is not read.  On return they hold the result over the union:
 *   lse = ln(e^lse_in + e^lse_plan),
 *   out = e^(lse_in - lse) out_in + e^(lse_plan - lse) out_plan,
 * with out_plan, lse_plan what ffa_fwd would compute for this plan.  Rows the
 * plan gives no keys keep (out, lse) unchanged.  The input out is bf16, so the
 * result carries its rounding once more than ffa_fwd over the union would.
 * Arguments, layouts and errors as ffa_fwd.
 */
ffa_status ffa_fwd_accumulate(const void* q, const void* k, const void* v, int64_t seqlen_q, int64_t seqlen_k,
                              int32_t hq, int32_t hkv, int32_t d, ffa_plan_t plan, float scale, void* out, float* lse,
                              void* stream);

/*
 * Forward pass with an attention sink (the pages name a learnable attention
 * sink without defining it; this is the plain reading): every row's softmax
 * also holds one logit sink[h] of its head, whose value vector is zero:
 *   lse_i = ln(sum_j e^(scale q_i . k_j) + e^sink[h]),
 *   out_i = sum_j e^(scale q_i . k_j - lse_i) v_j.
 * A row with no allowed key gets out = 0 and lse = sink[h].
 *  sink  fp32 device array [hq] (read only), in the units of scale * q . k.
 * Other arguments, layouts and errors as ffa_fwd; a NULL sink is
 * FFA_ERR_INVALID_ARG.
 */
ffa_status ffa_fwd_sink(const void* q, const void* k, const void* v, int64_t seqlen_q, int64_t seqlen_k, int32_t hq,
                        int32_t hkv, int32_t d, ffa_plan_t plan, float scale, const float* sink, void* out, float* lse,
                        void* stream);

/*
 * LSE merge of two partial results over disjoint key sets, element by element:
 *   lse = ln(e^lse_a + e^lse_b),  out = e^(lse_a - lse) out_a + e^(lse_b - lse) out_b.
 * A part with lse = -inf contributes nothing: its out values are ignored,
 * whatever they hold; a row empty in both comes out as (0, -inf).
 *
 *  out_a, out_b, out  bf16 [seqlen][hq][d]; lse_a, lse_b, lse  fp32 [hq][seqlen]
 *  out may be out_a or out_b and lse may be lse_a or lse_b (in place); other
 *  overlaps are not allowed.  All pointers 16-byte aligned; d in {64, 128}.
 * Errors: FFA_ERR_INVALID_ARG (null / misaligned pointer, seqlen < 0,
 * hq <= 0), FFA_ERR_UNSUPPORTED (d), FFA_ERR_CUDA.
 */
ffa_status ffa_lse_combine(const void* out_a, const float* lse_a, const void* out_b, const float* lse_b, void* out,
                           float* lse, int64_t seqlen, int32_t hq, int32_t d, void* stream);

/* Bytes of device workspace ffa_bwd needs: fp32 accumulators for dq
 * [seqlen_q][hq][d], dk and dv [seqlen_k][hkv][d], and the fp32 row terms
 * (lse in log2 units and D, [hq][seqlen_q rounded up to 128]), each part
 * 256-byte aligned.  Returns 0 for negative or zero sizes. */
size_t ffa_bwd_workspace_size(int64_t seqlen_q, int64_t seqlen_k, int32_t hq, int32_t hkv, int32_t d);

/*
 * Backward pass: dq, dk, dv of sum(out * dout) for the forward above, given
 * its out and lse (the pages require FFA to support backward for training).
 * A preprocess kernel forms D_i = dout_i . out_i and clears the fp32
 * accumulators.  A persistent kernel takes (work item, kv head) units in
 * the plan's item order (see ffa_plan_copy_bwd_items), popped from a counter
 * like the forward's: for the item's k2q
 * blocks and the q heads of the GQA group it recomputes P, accumulates
 * dV = P^T dO and dK = dS^T Q in TMEM and adds them to the fp32 dk / dv
 * accumulators at the end of the unit, and adds dS K into the fp32 dq
 * accumulator with TMA bulk reduce-adds.  A last kernel converts the three
 * accumulators to bf16.
 *
 *  d          64 or 128.  For 64 the shared-memory tiles use one of their two
 *             64-column panels, and dQ^T = K^T dS^T keeps its 128-row MMA
 *             shape over a zero panel (rows 64..127 are zero and not used).
 *  workspace  device buffer of at least ffa_bwd_workspace_size() bytes,
 *             256-byte aligned, owned by the caller, contents on entry ignored
 * The plan's backward tiles must be 128 x 128.
 * Errors: as ffa_fwd, plus FFA_ERR_INVALID_ARG for a short workspace.
 */
ffa_status ffa_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                   const void* dout, int64_t seqlen_q, int64_t seqlen_k, int32_t hq, int32_t hkv, int32_t d,
                   ffa_plan_t plan, float scale, void* dq, void* dk, void* dv, void* workspace,
                   size_t workspace_bytes, void* stream);

/*
 * Backward pass of ffa_fwd_sink: dq, dk, dv as ffa_bwd, given the out and lse
 * that ffa_fwd_sink returned (they already hold the sink), plus the gradient
 * of the sink logits,
 *   dsink[h] = -sum_i e^(sink[h] - lse_i) (dout_i . out_i),
 * written (not added) to the fp32 device array dsink [hq].  One extra small
 * kernel reduces each head's rows in a fixed order.
 * Other arguments and errors as ffa_bwd; NULL sink or dsink is
 * FFA_ERR_INVALID_ARG.
 */
ffa_status ffa_bwd_sink(const void* q, const void* k, const void* v, const void* out, const float* lse,
                        const void* dout, int64_t seqlen_q, int64_t seqlen_k, int32_t hq, int32_t hkv, int32_t d,
                        ffa_plan_t plan, float scale, const float* sink, void* dq, void* dk, void* dv, float* dsink,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass for callers that cannot allocate device memory (no
 * counterpart on the pages).  Some callers may not call cudaMalloc or any
 * allocator at all, e.g. a plugin inside a runtime that owns every device
 * byte and forbids allocations after start-up, or code that must not risk
 * the device-wide synchronization an allocation can cause.  For them this
 * call computes the same dq, dk, dv as ffa_bwd but keeps its scratch memory
 * (the fp32 accumulators and the per-row D / lse terms) in one fixed array
 * inside the library, FFA_BWD_NOALLOC_SCRATCH_BYTES large, which every GPU
 * that loads the library holds until the process exits.  The caller still
 * passes all inputs and outputs.
 *
 *  - Limit: ffa_bwd_workspace_size(seqlen_q, seqlen_k, hq, hkv, d) must not
 *    exceed FFA_BWD_NOALLOC_SCRATCH_BYTES (64 MiB: e.g. seqlen_q = seqlen_k
 *    = 4096 with hq = 16, hkv = 4 at d = 128 needs 48.5 MiB); larger
 *    problems return FFA_ERR_UNSUPPORTED and launch nothing.
 *  - The array belongs to the library's module, which CUDA loads into a
 *    device's context lazily (the default since CUDA 12.2): the first call
 *    of this function, or of any backward call of the library, on a device
 *    loads it.  That load reserves the array's 64 MiB on the device and can
 *    synchronize it, so warm the call up once per device (with that device
 *    current) before relying on it not to allocate, and before any stream
 *    capture.  Every call looks up the array's device address in the
 *    current context (cudaGetSymbolAddress, a host-side lookup once the
 *    module is loaded), so a device reset does not leave a stale address.
 *  - All calls on a device share the one array: calls whose GPU work
 *    overlaps (other streams, other threads) race and give wrong results.
 *    The kernels clear what must start at zero on every call.
 *  - The call allocates nothing itself; a plan whose timing is enabled
 *    creates CUDA events, so keep timing off for such callers.
 * Other arguments and errors are those of ffa_bwd.
 */
#define FFA_BWD_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
ffa_status ffa_bwd_noalloc(const void* q, const void* k, const void* v, const void* out, const float* lse,
                           const void* dout, int64_t seqlen_q, int64_t seqlen_k, int32_t hq, int32_t hkv,
                           int32_t d, ffa_plan_t plan, float scale, void* dq, void* dk, void* dv, void* stream);

/*
 * Dispatch solver (blog "Dispatch Solver", Figure 10): assign the
 * n = seqlen_q / chunk_size query chunks of a mask to cp_size buckets (ranks
 * of a context-parallel group) of exactly n / cp_size chunks each, keeping
 * the largest bucket's mask area small, by the pages' min-heap greedy:
 * chunks by area, heaviest first (ties: lower chunk index), each to the
 * bucket with the least area so far among those with room (ties: lower
 * bucket index).  Area(C_i) = allowed (query, key) pairs of the union mask in
 * rows [i chunk_size, (i + 1) chunk_size).
 *
 * Host-only and synchronous: no GPU work, usable without a GPU.
 *  slices         host array, validated as in ffa_plan_create
 *  seqlen_q       must be a multiple of cp_size * chunk_size
 *  chunk_area     host int64 [n] (may be NULL): Area(C_i)
 *  bucket_of_chunk host int32 [n]: the bucket of chunk i
 *  bucket_area    host int64 [cp_size] (may be NULL): each bucket's area
 * Errors: FFA_ERR_INVALID_ARG (sizes, divisibility, NULL bucket_of_chunk),
 * FFA_ERR_INVALID_SLICE, FFA_ERR_OVERLAPPING_COVERAGE.
 */
ffa_status ffa_dispatch_solve(const ffa_attn_slice* slices, int64_t n_slices, int64_t seqlen_q, int64_t seqlen_k,
                              int64_t chunk_size, int32_t cp_size, int64_t* chunk_area, int32_t* bucket_of_chunk,
                              int64_t* bucket_area);

/*
 * Range-Gather and Range-Scatter-Reduce (blog, group-collective section: the
 * pre / post kernels of the AlltoAll-v exchange), as local device kernels.
 * `ranges` is a host array of n_ranges (start, end) int64 pairs, half-open,
 * read during the call; empty ranges are skipped.  Tensors are token-major:
 * row i is the bytes [i row_bytes, (i + 1) row_bytes).  Up to 256 non-empty
 * ranges travel to the kernel in its launch parameters, with no allocation;
 * a longer table is copied to the device stream-ordered (cudaMallocAsync on
 * `stream`, freed after the kernel).
 *
 * ffa_range_gather: dst = the rows of src in the ranges, back to back in
 * list order.  row_bytes a multiple of 16; src, dst 16-byte aligned and not
 * overlapping; every range inside [0, src_rows).
 */
ffa_status ffa_range_gather(const void* src, int64_t src_rows, int64_t row_bytes, const int64_t* ranges,
                            int64_t n_ranges, void* dst, void* stream);

/*
 * ffa_range_scatter_reduce: dst[start, end) += the rows of the contiguous
 * buffer src, back to back in list order.  Ranges may overlap: every row of
 * every range is added (atomically, when the host finds an overlap; by a
 * plain read-add-write otherwise).  dtype 0 = fp32, 1 = bf16 (the sum is
 * rounded to bf16 at each add); row_elems values per row, row_elems * size a
 * multiple of 16; every range inside [0, dst_rows).
 * Errors (both calls): FFA_ERR_INVALID_ARG, FFA_ERR_CUDA.
 */
ffa_status ffa_range_scatter_reduce(const void* src, const int64_t* ranges, int64_t n_ranges, int64_t row_elems,
                                    int32_t dtype, void* dst, int64_t dst_rows, void* stream);

/* Synchronize `stream`, read and clear the plan's device status word.
 * Returns FFA_ERR_DEVICE_CHECK (and the word in *status_out, if not NULL)
 * when a kernel recorded a timeout or a metadata error since the last check.
 * The word is read through the device's pinned host channel, which plan
 * creation uses too: while this call waits for `stream` (e.g. for a long
 * backward still running on it), ffa_plan_create calls for the same device
 * on other host threads wait for it. */
ffa_status ffa_plan_check_status(ffa_plan_t plan, void* stream, uint32_t* status_out);

/* Kernels whose launches a plan can time (see ffa_plan_enable_timing). */
typedef enum {
  FFA_KERNEL_FWD = 0,      /* the persistent forward kernel */
  FFA_KERNEL_BWD_PRE = 1,  /* backward preprocess: D = rowsum(dout * out), lse in log2 units, clear dq */
  FFA_KERNEL_BWD_MAIN = 2, /* the persistent dK / dV / dQ kernel */
  FFA_KERNEL_BWD_DQ = 3,   /* dq, dk, dv accumulators -> bf16 */
  FFA_KERNEL_COUNT = 4
} ffa_kernel_id;

/*
 * Per-kernel timing, for profiling and benchmarks (no counterpart on the
 * pages).  While enabled, ffa_fwd and ffa_bwd with this plan record a CUDA
 * event before and after each of their kernels on the caller's stream.
 * Enabling (or disabling) discards what was recorded.
 */
ffa_status ffa_plan_enable_timing(ffa_plan_t plan, int32_t enable);

/* Wait for the recorded events and return, per ffa_kernel_id, the summed
 * device time in milliseconds and the number of launches (arrays of
 * FFA_KERNEL_COUNT entries; either may be NULL).  Recording continues. */
ffa_status ffa_plan_read_timing(ffa_plan_t plan, double* total_ms, int64_t* launches);

/*
 * Per-CTA trace of the persistent kernels, for checking how evenly the
 * longest-work-first deal loads the SMs (no counterpart on the pages).  While
 * enabled, each launch of the forward kernel (FFA_KERNEL_FWD) and of the
 * backward main kernel (FFA_KERNEL_BWD_MAIN) with this plan writes, per CTA,
 * four uint64 words: the %globaltimer (ns) when the CTA starts its first unit
 * and when it has finished its last, the units it took and their blocks
 * (forward: key blocks of its (q-tile, head pair) units; backward: blocks
 * times the GQA group).  Enabling allocates a small device buffer
 * (synchronizing the plan's creation stream); disabling frees it.  Only one
 * launch per kernel is kept, the latest.
 */
ffa_status ffa_plan_enable_cta_trace(ffa_plan_t plan, int32_t enable);

/* Wait for `stream`, then copy the latest traced launch of `kernel`
 * (FFA_KERNEL_FWD or FFA_KERNEL_BWD_MAIN) to the host array out [capacity][4]
 * and its CTA count to *n_ctas (0 when nothing was traced). */
ffa_status ffa_plan_read_cta_trace(ffa_plan_t plan, int32_t kernel, void* stream, uint64_t* out, int32_t capacity,
                                   int32_t* n_ctas);

/*
 * Self-test of the kernels' failure path (no counterpart on the pages).  Every
 * wait in the persistent kernels is bounded: after about 2 s it records a
 * timeout bit in the plan's status word (see ffa_plan_check_status), raises
 * the CTA's abort flag so that the CTA's other waits give up as well, and
 * lets the kernel release what it holds and return, without a trap.  This
 * call launches one block of 64 threads whose waits are on barriers nothing
 * ever arrives at: thread 0 times out, the other 63 leave on the abort flag.
 * It waits for the block (about 2 s) and returns the status word it recorded
 * (*status_out: bit 4, the "other wait" timeout) and how many threads gave
 * up (*gave_up_out: 64).  The device stays usable afterwards.
 * Errors: FFA_ERR_INVALID_ARG (NULL outputs), FFA_ERR_CUDA.
 */
ffa_status ffa_selftest_bounded_wait(void* stream, uint32_t* status_out, uint32_t* gave_up_out);

/* Static string for a status code. */
const char* ffa_status_string(ffa_status status);

#ifdef __cplusplus
}
#endif

#endif /* FFA_GB300_H */
