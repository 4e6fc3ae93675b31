/*
 * paged_attn.h -- C ABI of the GB300 (sm_103a) paged-attention library.
 *
 * One operation: exact scaled-dot-product attention of a batch of queries
 * over a paged K/V pool, as defined in "Week 3 Day 5: Paged FlashAttention"
 * (tiny-llm):
 *   - Keep the Day 4 Interface: the single model-facing call is
 *     paged_attention(query, key_pages, value_pages, block_table,
 *     context_lens, page_size, scale, mask="causal"); here mask="causal"
 *     becomes causal=1 and mask=None becomes causal=0.
 *   - Task 1: logical key position s of sequence b lives at
 *     pages[block_table[b, s / page_size], kv_head, s % page_size, :].
 *   - Task 2: key s is visible to query row l iff s <= l + context_len - L
 *     (causal), every s < context_len otherwise; the output is the softmax
 *     over the visible scores (scaled by `scale`) applied to the value rows.
 *   - GQA ("Week 2 Day 5: Fused Decode Attention", Task 1):
 *     kv_head = q_head / (H_q / H_kv).
 *
 * Layouts (row-major, contiguous, device memory unless stated):
 *   query        [B, H_q, L, D]                 bf16 or fp32
 *   key_pages    [num_pages, H_kv, page_size, D] same dtype as query
 *   value_pages  [num_pages, H_kv, page_size, D] same dtype
 *   block_table  [B, max_pages_per_seq]          int32 physical page ids
 *   context_lens [B]                             int32 keys per sequence,
 *                                                including the L new queries
 *   out          [B, H_q, L, D]                  same dtype as query
 * D must be 128.  All device pointers must be 16-byte aligned.
 * Entries block_table[b, i] with i >= ceil(context_lens[b] / page_size) are
 * never used and may hold anything (the kernels may load them, always inside
 * the [B, max_pages_per_seq] table, but no page is read through them).
 * Page slots past a sequence's context length, and pages no table entry
 * names, may hold anything, NaN and Inf included: they never reach the
 * output.  (The tensor-core schedule copies whole boxes of page rows and
 * zeroes, on chip, the value rows past the context before using them.)
 * Values inside a context are taken to be finite: a key a query row does
 * not see is multiplied by an exact 0 weight, so an Inf there would reach
 * that row as NaN.
 *
 * Variants of the same operation: pa_paged_attention_masked adds an fp32
 * additive mask [B * H_q, L, mask_S]; pa_paged_attention_varlen takes a ragged
 * batch (queries and outputs packed by token [total_q, H_q, D], offsets
 * cu_q[B + 1], each sequence its own query count).  pa_append_kv stores the
 * new tokens' K/V rows in their pages, the step before the operation.
 *
 * Ownership: the caller allocates and owns every buffer, including the
 * workspace.  The library allocates no device memory in any call.  Calls are
 * asynchronous on the given stream (cudaStream_t passed as void*, NULL = the
 * legacy default stream).
 *
 * Errors: arguments are checked on the host before anything is enqueued; a
 * failed check returns an error status and launches nothing.  The device
 * arrays block_table and context_lens are not read on the host (that would
 * need a synchronisation); instead the kernels record problems they meet in a
 * sticky 32-bit flag word at the start of the workspace (PA_FLAG_* bits) and
 * carry on without faulting.  pa_check_device_flag() reads it.
 */
#ifndef PAGED_ATTN_H
#define PAGED_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,     /* bad shape, null or misaligned pointer, bad context length */
    PA_ERR_UNSUPPORTED = 2,     /* valid but not implemented here (D != 128, ...) */
    PA_ERR_BAD_BLOCK_TABLE = 3, /* a block-table entry that is read is out of range */
    PA_ERR_WORKSPACE = 4,       /* workspace missing or smaller than pa_workspace_bytes() */
    PA_ERR_CUDA = 5,            /* a CUDA runtime call or launch failed */
    PA_ERR_DEVICE_FLAG = 6      /* the kernels recorded an error in the flag word */
} pa_status;

typedef enum { PA_BF16 = 0, PA_F32 = 1 } pa_dtype;

/* Which hand-written schedule runs.  AUTO applies the library's shape rule. */
typedef enum {
    PA_SCHED_AUTO = 0,
    PA_SCHED_DECODE = 1,  /* split-S CUDA-core page walk + combine: any L, bf16 or fp32 */
    PA_SCHED_PREFILL = 2  /* tcgen05 tensor-core tiles: bf16 only */
} pa_schedule;

/* Bits of the device flag word (workspace offset 0). */
#define PA_FLAG_BAD_PAGE 0x1u    /* a block-table entry read was outside [0, num_pages) */
#define PA_FLAG_BAD_CONTEXT 0x2u /* context_lens[b] < 1, > max_pages_per_seq*page_size,
                                    or < L under causal: that sequence's rows are 0 */
#define PA_FLAG_TIMEOUT 0x4u     /* an on-chip pipeline wait gave up (bounded spin) */

typedef struct {
    int B, H_q, H_kv, L, D, num_pages, page_size, max_pages_per_seq;
    pa_dtype dtype;
} pa_shape;

/* Bytes of workspace a call with this shape needs on the current device (the
 * largest over the schedules).  The first 4 bytes are the flag word; the
 * caller must zero the workspace once before its first use (the flag is then
 * sticky across calls until cleared; the schedules' work counters in the
 * first 256 bytes are zero again whenever a call has finished).  The rest
 * holds the decode schedule's per-split partial states (m, l, o[D] in fp32),
 * the tile plan of a ragged batch (B + 2 ints) and, last, the tile schedule's
 * per-chunk partial states when it splits the keys of few, long query tiles
 * (m, l, o[D] in fp32 per query row and chunk); it needs no initialisation.
 * Returns 0 for an invalid shape. */
size_t pa_workspace_bytes(const pa_shape* shape);

/* out = attention(query, paged K/V) for every (b, q_head, l).  `scale`
 * multiplies q.k before the softmax (1/sqrt(D) for standard attention); it
 * must be finite and >= 0 (PA_ERR_INVALID_ARG otherwise, in every entry
 * point that takes it).
 * The shape rule (measured crossover) picks the decode schedule when the rows
 * sharing one kv head (H_q/H_kv * L) are at most 4, or for fp32 and shapes the
 * tiles do not take; the tensor-core tiles otherwise, and also for at most 4
 * rows on calls with B * H_kv * capacity <= 65536 and a table capacity
 * (max_pages_per_seq * page_size) of at most 1024 keys. */
pa_status pa_paged_attention(const pa_shape* shape, const void* query, const void* key_pages,
                             const void* value_pages, const int32_t* block_table,
                             const int32_t* context_lens, float scale, int causal, void* out,
                             void* workspace, size_t workspace_bytes, void* cuda_stream);

/* Same operation with the schedule chosen by the caller (pa_schedule);
 * PA_ERR_UNSUPPORTED if that schedule cannot run this shape or dtype. */
pa_status pa_paged_attention_sched(const pa_shape* shape, const void* query,
                                   const void* key_pages, const void* value_pages,
                                   const int32_t* block_table, const int32_t* context_lens,
                                   float scale, int causal, void* out, void* workspace,
                                   size_t workspace_bytes, void* cuda_stream, int schedule);

/* pa_paged_attention_sched, plus two caller-created CUDA events
 * (cudaEvent_t passed as void*; either may be NULL) recorded on the stream
 * immediately before and after the launch of the schedule's dominant kernel:
 * the split page-walk kernel of the decode schedule, the tile kernel of the
 * prefill schedule.  cudaEventElapsedTime(before, after) then times that
 * kernel alone.  The events are only recorded, never created or destroyed. */
pa_status pa_paged_attention_profiled(const pa_shape* shape, const void* query,
                                      const void* key_pages, const void* value_pages,
                                      const int32_t* block_table, const int32_t* context_lens,
                                      float scale, int causal, void* out, void* workspace,
                                      size_t workspace_bytes, void* cuda_stream, int schedule,
                                      void* event_before, void* event_after);

/* pa_paged_attention_sched with an explicit additive mask: the pages
 * normalise explicit masks to [B * H_q, L, S] and keep the causal flag next to
 * them ("Week 2 Day 5: Fused Decode Attention", Task 1).  mask is an fp32
 * device array [B * H_q, L, mask_S] over logical key positions, 16-byte
 * aligned, mask_S a multiple of 4 and at least max_pages_per_seq * page_size;
 * mask[(b * H_q + h) * L + l][s] is added to the scaled score of key s for
 * row (b, h, l) before the softmax, and the causal rule still applies when
 * causal != 0.  -inf removes a key; a row whose every visible key is removed
 * outputs 0.  Both schedules take it; every mask element a row can see is
 * read once.  Returns PA_ERR_INVALID_ARG for a null or misaligned mask or a
 * bad mask_S, otherwise as pa_paged_attention_sched. */
pa_status pa_paged_attention_masked(const pa_shape* shape, const void* query,
                                    const void* key_pages, const void* value_pages,
                                    const int32_t* block_table, const int32_t* context_lens,
                                    float scale, int causal, const float* mask,
                                    long long mask_S, void* out, void* workspace,
                                    size_t workspace_bytes, void* cuda_stream, int schedule);

/* A ragged batch in one call: sequence b has L_b = cu_q[b + 1] - cu_q[b]
 * new query positions, the last L_b of its context_lens[b] keys, so decode
 * steps (L_b = 1), prefill chunks and continuations (L_b > 1) and sequences
 * without new tokens (L_b = 0, not read) mix in one batch.  Every row is the
 * row of a batch of that sequence alone: causal visibility s <= l +
 * context_lens[b] - L_b ("Week 3 Day 5: Paged FlashAttention", Task 2; "Day
 * 22: the fused paged-attention kernel" runs decode steps, causal prefills and
 * partial continuations as one fold).
 *
 * query, out: [total_q, H_q, D] packed by token (row (b, h, l) is token
 * cu_q[b] + l), 16-byte aligned.  cu_q: int32 device array [B + 1], cu_q[0]
 * = 0, nondecreasing, cu_q[B] = total_q.  shape->L: an upper bound on every
 * L_b; shape->B: the number of sequences.  Pool, block table and context
 * lengths as for pa_paged_attention.  workspace: pa_workspace_bytes(shape).
 *
 * PA_SCHED_AUTO sends each sequence to a schedule on the device: at most 4
 * query rows per kv head ((H_q / H_kv) * L_b <= 4) to the page walk, more to
 * the tensor-core tiles (bf16, shapes the tiles take), both launched by this
 * call, the page walk as a programmatic dependent of the tile kernel so the two
 * run side by side; a forced schedule takes every sequence.  A sequence whose offsets are
 * broken (cu_q[b] < 0, L_b < 0 or > shape->L, cu_q[b + 1] > total_q) sets
 * PA_FLAG_BAD_CONTEXT and none of its rows is written; one whose context
 * length breaks the contract sets it too and gets zero rows.  No explicit
 * mask.  Returns as pa_paged_attention_sched; PA_OK at once for total_q = 0. */
pa_status pa_paged_attention_varlen(const pa_shape* shape, const void* query,
                                    const void* key_pages, const void* value_pages,
                                    const int32_t* block_table, const int32_t* context_lens,
                                    const int32_t* cu_q, int total_q, float scale, int causal,
                                    void* out, void* workspace, size_t workspace_bytes,
                                    void* cuda_stream, int schedule);

/* Self-test of the failure path of the kernels' bounded on-chip waits (every
 * mbarrier wait gives up after 2 s instead of hanging): one warp waits, with the
 * same wait, on a barrier phase that nothing completes.  After timeout_us
 * (at most 2,000,000) the wait gives up, PA_FLAG_TIMEOUT is recorded in the
 * workspace's flag word and the kernel returns, leaving the context usable.
 * No fault, no trap.  Asynchronous on cuda_stream.  Returns PA_ERR_WORKSPACE
 * for a missing or misaligned workspace, PA_ERR_INVALID_ARG for a longer
 * timeout. */
pa_status pa_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                   unsigned timeout_us, void* cuda_stream);

/* Debug gather of "Week 3 Day 5", Task 1: writes the dense history of every
 * (b, kv_head) through the block table, k_dense/v_dense [B, H_kv, max_S, D]
 * in the pool's dtype, zeros at s >= context_lens[b].  Page translation is
 * bit-exact, so this is compared bitwise with the oracle's gather. */
pa_status pa_gather_debug(const pa_shape* shape, const void* key_pages, const void* value_pages,
                          const int32_t* block_table, const int32_t* context_lens, int max_S,
                          void* k_dense, void* v_dense, void* workspace, void* cuda_stream);

/* Stores the new tokens' keys and values in their pages: the step that fills
 * the pool before the path reads it.  The pages introduce pages and block
 * tables as the prerequisite of "Week 3 Day 5: Paged FlashAttention"
 * (Prerequisites) and give the read-side translation in its Task 1; this
 * call writes through the same translation.
 *
 * Shape fields used: B, H_kv, L (new tokens per sequence), D, num_pages,
 * page_size, max_pages_per_seq, dtype (H_q must still be a multiple of H_kv).
 * k_new, v_new: [B, H_kv, L, D] device arrays in the pool's element type,
 * 16-byte aligned.  The new tokens of sequence b are its last L logical
 * positions s = context_lens[b] - L + t (t = 0..L-1; context_lens counts
 * them, as in pa_paged_attention), and
 *   key_pages[block_table[b, s / page_size], kv_head, s % page_size, :]
 *       = k_new[b, kv_head, t, :]
 * (the same for values).  The copy is exact.  Only block-table entries of the
 * pages holding new tokens are read.  Positions of two sequences must not map
 * to the same (page, slot): the pool is written, not reduced.
 * The kernel reports in the workspace's flag word (offset 0, >= 256 bytes,
 * zeroed by the caller once): PA_FLAG_BAD_CONTEXT for a sequence with
 * context_lens[b] < L or > max_pages_per_seq * page_size (nothing of it is
 * written), PA_FLAG_BAD_PAGE for a page id outside [0, num_pages) (that token
 * is not written).  Asynchronous on cuda_stream; allocates nothing.
 * Returns PA_ERR_INVALID_ARG for null or misaligned pointers,
 * PA_ERR_UNSUPPORTED for D != 128 or more than 2^31 16-byte chunks,
 * PA_ERR_WORKSPACE for a missing workspace, PA_ERR_CUDA for launch errors. */
pa_status pa_append_kv(const pa_shape* shape, const void* k_new, const void* v_new,
                       void* key_pages, void* value_pages, const int32_t* block_table,
                       const int32_t* context_lens, void* workspace, size_t workspace_bytes,
                       void* cuda_stream);

/* Synchronises the stream, copies the flag word to *flag_out and, if clear is
 * non-zero, resets it to 0.  Returns PA_ERR_DEVICE_FLAG when any bit was set. */
pa_status pa_check_device_flag(void* workspace, uint32_t* flag_out, int clear, void* cuda_stream);

/* Host-side check of the device metadata (copies block_table and
 * context_lens to the host, synchronising the stream): PA_ERR_INVALID_ARG for
 * a context length outside [max(1, causal ? L : 1), max_pages_per_seq *
 * page_size], PA_ERR_BAD_BLOCK_TABLE for a read entry outside
 * [0, num_pages).  Meant for debugging; the fast path never calls it. */
pa_status pa_validate_metadata(const pa_shape* shape, const int32_t* block_table,
                               const int32_t* context_lens, int causal, void* cuda_stream);

/* pa_validate_metadata for a ragged batch (copies cu_q, context_lens and
 * block_table to the host, synchronising the stream): PA_ERR_INVALID_ARG for
 * cu_q[0] != 0, cu_q[B] != total_q, an L_b outside [0, shape->L], or a
 * sequence with queries whose context length is outside [max(1, causal ? L_b
 * : 1), max_pages_per_seq * page_size]; PA_ERR_BAD_BLOCK_TABLE for an entry a
 * sequence with queries reads outside [0, num_pages).  Sequences with L_b = 0
 * are not checked (they are not read).  Meant for debugging. */
pa_status pa_validate_metadata_varlen(const pa_shape* shape, const int32_t* block_table,
                                      const int32_t* context_lens, const int32_t* cu_q,
                                      int total_q, int causal, void* cuda_stream);

/* The schedule pa_paged_attention would pick for this shape (PA_SCHED_*),
 * or -1 for an invalid shape. */
int pa_choose_schedule(const pa_shape* shape);

/* Kernel launches one call of this shape and schedule enqueues on the current
 * device (the tile schedule adds a merge kernel when it splits keys), or -1
 * for an invalid shape or no device. */
int pa_launch_count(const pa_shape* shape, int schedule);

/* Decode schedule without a caller workspace, for callers that cannot
 * allocate device memory: for example a serving process whose free HBM is
 * all owned by its K/V page pool and caching allocator, or a latency-bound
 * decode loop that cannot afford the device-wide synchronisation cudaMalloc
 * and cudaFree may cause.  The pages describe no such entry point; it has no
 * counterpart there.
 *
 * Computes exactly what pa_paged_attention_sched(..., PA_SCHED_DECODE) does,
 * with its scratch in one fixed array of 8 MiB that the library keeps on
 * every device it is used on, for the life of the process.  Allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   - Every argument is checked first, as in pa_paged_attention_sched
 *     (PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED on a device other than
 *     compute capability 10.3); a rejected call enqueues nothing.
 *   - Shapes whose decode scratch (the page walk's part of
 *     pa_workspace_bytes) exceeds 8 MiB are rejected with PA_ERR_WORKSPACE
 *     before anything is enqueued.
 *   - Every call looks up the array's device address with the calling
 *     thread's device current (cheap once the library's device code is
 *     loaded there; still right after a cudaDeviceReset).  The first call on
 *     a device may load that code: make it before any stream capture.
 *   - Each call clears the array's error flag, then runs; if device_flag_out
 *     (a 4-byte aligned device pointer to one uint32, may be NULL) is given,
 *     this call's PA_FLAG_* bits are copied there on the stream after the
 *     kernels.
 *   - All calls share the array and it keeps the last call's contents; calls
 *     whose kernels overlap on the GPU (e.g. on unordered streams) race. */
pa_status pa_paged_attention_decode_noalloc(const pa_shape* shape, const void* query,
                                            const void* key_pages, const void* value_pages,
                                            const int32_t* block_table,
                                            const int32_t* context_lens, float scale, int causal,
                                            void* out, uint32_t* device_flag_out,
                                            void* cuda_stream);

const char* pa_status_str(pa_status status);

#ifdef __cplusplus
}
#endif
#endif /* PAGED_ATTN_H */
