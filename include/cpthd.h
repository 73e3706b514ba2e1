/*
 * cpthd.h -- C ABI of libcpthd: the per-rank hot path of context-parallel
 * causal attention over packed THD sequences, for NVIDIA GB300 (sm_103a).
 *
 * Operations and where they are defined:
 *  - Partition strategies: TransformerEngine PR #3221 "[PyTorch] Add
 *    no-load-balance THD all-gather CP", sections "How to use", "What
 *    changed" and "Why": DUAL_CHUNK_SWAP cuts every document into
 *    2*cp_size chunks and rank r owns chunks r and 2*cp_size-1-r (the
 *    head-tail split of torchtitan PR #2144, "Summary"); NO_LOAD_BALANCE cuts
 *    the whole physical buffer into cp_size contiguous chunks, rank-major.
 *  - Reorder: the gather behind get_batch_on_this_cp_rank (TE PR, "How to
 *    use"), dst[i] = src[idx[i]] row by row.
 *  - Attention: causal THD self-attention without a sliding window
 *    (window_size = (-1, 0), TE PR "Scope and constraints"); documents stay
 *    isolated through cu_seqlens / cu_seqlens_padded ("What changed"); one
 *    rank's query slice attends to the full K/V buffer, which is what the
 *    all-gather of K/V over cp_group hands every rank.
 *
 * THD layout: tokens of all documents are concatenated along one axis of
 * length T (no batch axis). cu_seqlens[N+1] holds prefix sums of the actual
 * document lengths L_j; cu_seqlens_padded[N+1] holds prefix sums of the
 * padded lengths P_j >= L_j and gives each document's physical start.
 * Physical slots cu_seqlens_padded[j] + L_j .. cu_seqlens_padded[j+1]-1 are
 * pad slots.
 *
 * Conventions (every entry point):
 *  - Pointers named *_dev are CUDA device pointers owned and allocated by the
 *    caller. Pointers named *_host are host pointers. The library allocates
 *    no device memory itself.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and return CPTHD_OK (0) or a negative status code.
 *    Scalar arguments are validated on the host before any launch; a call
 *    that returns an error launched nothing.
 *  - Data-dependent checks (offset arrays non-decreasing, ending at T,
 *    divisibility, index ranges) run inside the kernels. A kernel that finds
 *    a violation records it in the optional caller-owned device word pair
 *    err_dev[2] (err_dev[0] = first status code, err_dev[1] = detail: the
 *    offending document, row or index position) and never traps. Pass NULL to
 *    skip the record. The caller zeroes err_dev before the call and reads it
 *    back whenever it wants; outputs of a call that recorded an error are
 *    unspecified but every write stays inside the output buffers.
 *  - Index arrays are int32 (T < 2^31).
 */
#ifndef CPTHD_H_
#define CPTHD_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CPTHD_API __attribute__((visibility("default")))
#else
#define CPTHD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* cpthd_stream_t; /* == cudaStream_t */

typedef enum {
  CPTHD_DUAL_CHUNK_SWAP = 0,  /* default strategy */
  CPTHD_NO_LOAD_BALANCE = 1,  /* experimental strategy */
  CPTHD_PACKED_MIRRORED = 2   /* the PR's interim "packed super-sequence": the whole buffer as one
                                 sequence cut into 2*cp_size mirrored chunks */
} cpthd_strategy_t;

enum {
  CPTHD_OK = 0,
  CPTHD_ERR_INVALID_ARG = -1,   /* null pointer, negative size, rank out of range ... */
  CPTHD_ERR_NOT_DIVISIBLE = -2, /* T % cp_size (NLB) or P_j % (2*cp_size) (DCS) */
  CPTHD_ERR_UNSUPPORTED = -3,   /* head dim, head counts or alignment the kernels do not take */
  CPTHD_ERR_WORKSPACE = -4,     /* workspace missing or too small */
  CPTHD_ERR_CUDA = -5,          /* a CUDA runtime call failed */
  CPTHD_ERR_BAD_OFFSETS = -6,   /* (device) offsets not non-decreasing, not starting at 0, or not ending at T */
  CPTHD_ERR_INDEX_RANGE = -7,   /* (device) an index outside [0, rows) */
  CPTHD_ERR_PAD_LENGTH = -8,    /* (device) actual length L_j larger than padded length P_j */
  CPTHD_ERR_TIMEOUT = -9,       /* (device) a pipeline wait gave up; the kernel returned early */
  CPTHD_ERR_SCRATCH_LIMIT = -10 /* slice needs more scratch than thd_causal_attn_fwd_static_scratch holds */
};

/* Human-readable name of a status code (static storage, never NULL). */
CPTHD_API const char* cpthd_status_string(int status);

/* Tokens every rank holds: T / cp_size under every strategy (TE PR, "Scope
 * and constraints": equal local Q/K/V physical lengths).
 * Host only, launches nothing. Errors: INVALID_ARG (cp_size < 1, T < 0,
 * null output, unknown strategy), NOT_DIVISIBLE (T % cp_size != 0, or
 * T % (2*cp_size) != 0 for PACKED_MIRRORED). */
CPTHD_API int cp_local_tokens(int strategy, int64_t T, int cp_size, int64_t* t_local_host);

/* Partition index: the physical token indices a CP rank owns (TE PR,
 * "Why" and "What changed").
 *   DUAL_CHUNK_SWAP: with c_j = P_j / (2*cp_size), rank r lists, document by
 *     document in pack order, slots cup[j] + r*c_j + t (t < c_j) and then
 *     cup[j] + (2*cp_size-1-r)*c_j + t (t < c_j). The rank-local offsets are
 *     therefore cu_seqlens_padded / cp_size. Needs every P_j % (2*cp_size) == 0.
 *   NO_LOAD_BALANCE: slots rank*T/cp_size + t. Needs T % cp_size == 0.
 *   PACKED_MIRRORED (TE PR commit notes: the complete physical buffer
 *     represented as one partitioning sequence, mirrored chunks, document
 *     boundaries kept by the attention's sequence metadata): DUAL_CHUNK_SWAP
 *     applied to the single sequence [0, T). Needs T % (2*cp_size) == 0, not
 *     per-document divisibility.
 * cu_seqlens_padded_dev: int32 [num_docs+1], device, read only (NLB and
 *   PACKED_MIRRORED read it only to validate it).
 * rank: 0..cp_size-1 writes T/cp_size indices; -1 writes all ranks,
 *   rank-major, cp_size*(T/cp_size) = T indices.
 * idx_out_dev: int32, device, caller-allocated, size as above.
 * Device checks (err_dev): BAD_OFFSETS, NOT_DIVISIBLE (detail = document). */
CPTHD_API int cp_partition_index(int strategy, const int32_t* cu_seqlens_padded_dev, int num_docs, int64_t T,
                       int cp_size, int rank, int32_t* idx_out_dev, int32_t* err_dev,
                       cpthd_stream_t stream);

/* K/V restore index: after an all-gather of every rank's slice, rank-major
 * (gathered[r*T/cp_size + t] = x[index of rank r][t]), restore_idx[p] is the
 * row of the gathered buffer that holds physical slot p, so that
 * cp_reorder(gathered, restore_idx) brings K/V back to token order (TE PR,
 * Greptile summary: "stable K/V restoration"; commit notes: rank-major
 * ownership needs no KV reorder). NO_LOAD_BALANCE gives the identity.
 * restore_idx_out_dev: int32 [T], device, caller-allocated.
 * Device checks (err_dev): as cp_partition_index. */
CPTHD_API int cp_restore_index(int strategy, const int32_t* cu_seqlens_padded_dev, int num_docs, int64_t T,
                               int cp_size, int32_t* restore_idx_out_dev, int32_t* err_dev, cpthd_stream_t stream);

/* Reorder: dst[i, :] = src[idx[i], :] for i < n_rows, byte for byte, for
 * any row width (TE PR "How to use": input_ids, labels, position_ids and
 * activations of a rank's slice). 16-byte vector path when row_bytes and
 * both base pointers are 16-byte aligned, 8-byte path when they are 8-byte
 * aligned, byte path otherwise.
 * src_dev: [src_rows, row_bytes] device; idx_dev: int32 [n_rows] device;
 * dst_dev: [n_rows, row_bytes] device, must not overlap src.
 * Device checks (err_dev): INDEX_RANGE (detail = i); that row is left unwritten. */
CPTHD_API int cp_reorder(const void* src_dev, int64_t src_rows, int64_t row_bytes, const int32_t* idx_dev,
               int64_t n_rows, void* dst_dev, int32_t* err_dev, cpthd_stream_t stream);

/* Several tensors gathered by the same index list in one launch (at most 8).
 * src_dev_host / dst_dev_host / row_bytes_host: host arrays of n_tensors
 * device pointers and row widths; every tensor has src_rows rows. */
CPTHD_API int cp_reorder_multi(int n_tensors, const void* const* src_dev_host, void* const* dst_dev_host,
                     const int64_t* row_bytes_host, int64_t src_rows, const int32_t* idx_dev,
                     int64_t n_rows, int32_t* err_dev, cpthd_stream_t stream);

/* Partition and gather in one launch: the index list of `rank` under
 * `strategy` (as cp_partition_index computes it, written to idx_out_dev),
 * and every tensor of the batch gathered by it (as cp_reorder_multi), with
 * each row's physical slot computed where the row is copied. One launch
 * replaces the partition-index launch and the gather that a rank's slicing
 * (TE PR "How to use": get_batch_on_this_cp_rank over input_ids, labels,
 * position_ids) otherwise takes; results are identical to the two calls.
 * The tensors have T rows each (the physical buffer); rank must be in
 * [0, cp_size).
 * cu_seqlens_padded_dev: int32 [num_docs+1] device; idx_out_dev: int32
 * [T/cp_size] device, caller-allocated; src_dev_host / dst_dev_host /
 * row_bytes_host: host arrays of n_tensors (1..8) device pointers and row
 * widths, dst [T/cp_size, row_bytes].
 * Host checks: as cp_local_tokens, rank range, null pointers.
 * Device checks (err_dev): as cp_partition_index, and INDEX_RANGE for a
 * computed slot outside [0, T) (only with malformed offsets). */
CPTHD_API int cp_partition_reorder_multi(int strategy, const int32_t* cu_seqlens_padded_dev, int num_docs,
                                         int64_t T, int cp_size, int rank, int n_tensors,
                                         const void* const* src_dev_host, void* const* dst_dev_host,
                                         const int64_t* row_bytes_host, int32_t* idx_out_dev, int32_t* err_dev,
                                         cpthd_stream_t stream);

/* Device workspace thd_causal_attn_fwd needs for a slice of t_local rows:
 * the plan (per-row key bounds, per-tile key intervals, the schedule of the
 * attention CTAs, about 33 bytes per row) and one fp32 partial-result slot
 * per boundary between two CTAs' shares of the work and per query tile (a
 * work item that a boundary cuts runs in pieces whose partial softmax
 * results are combined; about 20 MiB at d = 128, 10 MiB at d = 64, whatever
 * t_local). d must be 64 or 128 (else CPTHD_ERR_UNSUPPORTED). Host only. */
CPTHD_API int thd_causal_attn_workspace_size(int64_t t_local, int Hq, int Hkv, int d, size_t* bytes_host);

/* Causal packed-THD attention forward for one rank's query slice.
 *   q_slice_idx_dev: int32 [t_local], the physical index of every local query
 *     row (the output of cp_partition_index for this rank; any order works,
 *     but it must come from the same strategy as the slice -- TE PR "Scope and
 *     constraints": input partitioning and attention use the same strategy).
 *   q_dev: bf16 [t_local, Hq, d]; k_dev, v_dev: bf16 [T, Hkv, d] (the full,
 *     token-ordered K/V buffer); all rows contiguous, 16-byte aligned.
 *   cu_seqlens_dev / cu_seqlens_padded_dev: int32 [num_docs+1]; padded may be
 *     NULL, meaning no padding (cu_seqlens_padded == cu_seqlens).
 *   Pair (q, k) is allowed iff both lie in the same document and
 *     pos_k <= pos_q; pad keys are never allowed (they lie beyond every real
 *     query of their document).
 *   softmax_scale <= 0 selects 1/sqrt(d).
 *   out_dev: bf16 [t_local, Hq, d], round-to-nearest-even of the fp32 result.
 *   lse_dev: fp32 [Hq, t_local], natural-log sum of exp(scale * q.k) over
 *     the allowed keys. Pad query rows get out = 0 and lse = -inf.
 *   workspace_dev: at least thd_causal_attn_workspace_size() bytes, 256-byte
 *     aligned, device; contents need no initialisation and are scratch.
 * Supported: d in {64, 128}; Hq % Hkv == 0; Hq, Hkv >= 1.
 * The result is deterministic: the same inputs on the same GPU give the
 * same bits (the pieces of a cut work item are combined in a fixed order).
 * Host errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 * Device checks (err_dev): BAD_OFFSETS, PAD_LENGTH, INDEX_RANGE, TIMEOUT. */
CPTHD_API int thd_causal_attn_fwd(const int32_t* q_slice_idx_dev, int64_t t_local, const void* q_dev,
                        const void* k_dev, const void* v_dev, int64_t T,
                        const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_padded_dev,
                        int num_docs, int Hq, int Hkv, int d, float softmax_scale, void* out_dev,
                        float* lse_dev, void* workspace_dev, size_t workspace_bytes,
                        int32_t* err_dev, cpthd_stream_t stream);

/* The forward in two parts, for callers that run several attentions over
 * the same slice (every layer of a model step shares q_slice_idx and the
 * offsets): thd_causal_attn_plan writes the plan (per-row key bounds,
 * per-group key intervals, the group order when there are more work items
 * than SMs, and every attention CTA's equal share of the work) into the
 * workspace once; thd_causal_attn_fwd_planned runs the attention kernel
 * against it as often as needed. thd_causal_attn_fwd is the two in
 * sequence. The planned call must get the same t_local, T, Hq, Hkv and the
 * workspace the plan wrote, on the same GPU (caller's contract); q, k, v, d
 * and the scale may differ between planned calls. A planned call writes only
 * the workspace's partial-result slots and its counters and flags, which it
 * returns to their initial state before it ends, so planned calls on one
 * workspace must not overlap on the GPU. thd_causal_attn_plan alone checks
 * the workspace against the plan part only (it does not know d); the
 * planned call needs the full thd_causal_attn_workspace_size().
 * Arguments, layouts, errors: as thd_causal_attn_fwd. */
CPTHD_API int thd_causal_attn_plan(const int32_t* q_slice_idx_dev, int64_t t_local, int64_t T,
                                   const int32_t* cu_seqlens_dev, const int32_t* cu_seqlens_padded_dev, int num_docs,
                                   int Hq, int Hkv, void* workspace_dev, size_t workspace_bytes, int32_t* err_dev,
                                   cpthd_stream_t stream);
CPTHD_API int thd_causal_attn_fwd_planned(int64_t t_local, const void* q_dev, const void* k_dev, const void* v_dev,
                                          int64_t T, int Hq, int Hkv, int d, float softmax_scale, void* out_dev,
                                          float* lse_dev, const void* workspace_dev, size_t workspace_bytes,
                                          int32_t* err_dev, cpthd_stream_t stream);

/* The plan of rank `rank`'s slice under `strategy` (CPTHD_DUAL_CHUNK_SWAP,
 * CPTHD_NO_LOAD_BALANCE or CPTHD_PACKED_MIRRORED), with each row's physical
 * slot computed from the partition formulas (TransformerEngine PR #3221,
 * "What changed"; as cp_partition_index) instead of read from an index
 * list: the workspace it writes equals that of thd_causal_attn_plan given
 * the list cp_partition_index returns for the same rank, so the plan can run
 * before, or beside, the partition and the gather of the slice.
 *   cu_seqlens_dev / cu_seqlens_padded_dev / num_docs: as thd_causal_attn_fwd
 *     (the padded offsets define the partition; null = unpadded);
 *   t_local = T / cp_size (cp_local_tokens); the workspace is sized for it.
 * Host checks: as cp_local_tokens (T divisible), rank in [0, cp_size), and
 * the checks of thd_causal_attn_plan. Device checks (recorded in err): the
 * offset table as in thd_causal_attn_fwd and, under DualChunkSwap, padded
 * lengths that are not multiples of 2*cp_size (CPTHD_ERR_NOT_DIVISIBLE). */
CPTHD_API int thd_causal_attn_plan_partition(int strategy, int64_t T, const int32_t* cu_seqlens_dev,
                                             const int32_t* cu_seqlens_padded_dev, int num_docs, int cp_size,
                                             int rank, int Hq, int Hkv, void* workspace_dev, size_t workspace_bytes,
                                             int32_t* err_dev, cpthd_stream_t stream);

/* Device workspace thd_causal_attn_bwd needs (per-row key bounds, per-tile key
 * intervals, lse * log2(e) and rowsum(dO * O) per row and query head, and
 * 64 bytes per row and query head of per-query MMA operands for the dK/dV
 * pass). Host only. */
CPTHD_API int thd_causal_attn_bwd_workspace_size(int64_t t_local, int Hq, int Hkv, int d, size_t* bytes_host);

/* Causal packed-THD attention backward for one rank's query slice: the
 * gradients of sum(dout * out) for the forward above, with the same slice
 * layout (TE PR: the strategy is captured for backward, so forward and
 * backward use the same token layout) and the forward's LSE.
 *   q_slice_idx_dev, q_dev, k_dev, v_dev, cu_seqlens*, num_docs, Hq, Hkv, d,
 *     softmax_scale: exactly as passed to thd_causal_attn_fwd.
 *   out_dev: bf16 [t_local, Hq, d], lse_dev: fp32 [Hq, t_local] -- the
 *     forward's outputs; dout_dev: bf16 [t_local, Hq, d].
 *   dq_dev: fp32 [t_local, Hq, d].
 *   dk_dev, dv_dev: fp32 [T, Hkv, d] for the whole K/V buffer, holding this
 *     rank's contribution (the part a reduce-scatter over CP ranks would sum);
 *     every key is written, so keys no query of the slice reaches get 0.
 *   workspace_dev: thd_causal_attn_bwd_workspace_size() bytes, 256-byte aligned.
 * Supported: d in {64, 128}; Hq % Hkv == 0; t_local <= 262,144 (2048 query
 * tiles). Host errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA. Device
 * checks (err_dev): BAD_OFFSETS, PAD_LENGTH, INDEX_RANGE, TIMEOUT. */
CPTHD_API int thd_causal_attn_bwd(const int32_t* q_slice_idx_dev, int64_t t_local, const void* q_dev,
                                  const void* k_dev, const void* v_dev, const void* out_dev, const void* dout_dev,
                                  const float* lse_dev, int64_t T, const int32_t* cu_seqlens_dev,
                                  const int32_t* cu_seqlens_padded_dev, int num_docs, int Hq, int Hkv, int d,
                                  float softmax_scale, float* dq_dev, float* dk_dev, float* dv_dev,
                                  void* workspace_dev, size_t workspace_bytes, int32_t* err_dev,
                                  cpthd_stream_t stream);

/* Same computation as thd_causal_attn_fwd for callers that cannot allocate
 * device memory (a host framework that owns all allocations, a plugin that
 * must not call cudaMalloc mid-step, a path that may never enter an
 * allocator). The pages have no counterpart: this is a deployment variant.
 * Instead of a caller workspace it uses a fixed 32 MiB device array built
 * into the library, which every GPU that loads the library holds until the
 * process exits; the call allocates nothing. That is enough for slices of at
 * least 350,000 query rows; a larger slice is rejected with
 * CPTHD_ERR_SCRATCH_LIMIT before anything is launched.
 * Every call whose stream is not capturing looks up the array's device
 * address on the current device (so a device reset, or another context
 * made current, is picked up by the next such call); a call made during a
 * stream capture reuses the address the last uncaptured call on that device
 * found, so make the first call on each device before any stream capture.
 * Host checks run in the order of thd_causal_attn_fwd (shape, head dim,
 * t_local == 0 returns CPTHD_OK), then the scratch limit.
 * All calls share the one array: calls that overlap on the GPU (different
 * streams without ordering between them) race and corrupt each other's
 * results. Nothing in the array needs clearing between calls.
 * Arguments, layouts and device checks as thd_causal_attn_fwd, without the
 * workspace pair. */
CPTHD_API int thd_causal_attn_fwd_static_scratch(const int32_t* q_slice_idx_dev, int64_t t_local,
                                                 const void* q_dev, const void* k_dev, const void* v_dev,
                                                 int64_t T, const int32_t* cu_seqlens_dev,
                                                 const int32_t* cu_seqlens_padded_dev, int num_docs, int Hq,
                                                 int Hkv, int d, float softmax_scale, void* out_dev,
                                                 float* lse_dev, int32_t* err_dev, cpthd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CPTHD_H_ */
