/*
 * kda.h — C ABI of the GB300 (sm_103a) chunkwise Kimi Delta Attention forward.
 *
 * The operation.  For every packed sequence n (tokens cu_seqlens[n] ..
 * cu_seqlens[n+1]-1) and head h, with a V-first state S in R^{V x K}:
 *
 *     q^ = q / sqrt(|q|^2 + 1e-6) / sqrt(K),   k^ = k / sqrt(|k|^2 + 1e-6)
 *     g  = lower_bound * sigmoid(g_raw)          (per channel, K values)
 *     b  = sigmoid(beta_raw)                     (one value per token and head)
 *     S_t = S_{t-1} Diag(exp g_t) (I - b_t k^_t k^_t^T) + b_t v_t k^_t^T
 *     o_t = S_t q^_t
 *
 *   ROCm/aiter PR #4741 "[FlyDSL] Add gfx950 Kimi Delta Attention prefill
 *   kernel", Summary: packed varlen [1, total_tokens, H, D] inputs, raw
 *   pre-activation gate and beta, V-first recurrent state; "Optimizations
 *   Applied": q/k L2 norm, lower-bounded-sigmoid gate and beta sigmoid are part
 *   of the op, padded tokens (beta = 0, g = 0) are exact no-ops.
 *
 * Computed chunkwise on the GPU (intra-chunk tiles, UT/WY solve, serial state
 * scan with the output product fused), fp32 accumulation throughout.
 *
 * Fixed shapes: K = V = 128 (KDA_HEAD_DIM).  q, k, v and out are bf16,
 * contiguous [total_tokens][H][128]; g_raw is fp32 [total_tokens][H][128];
 * beta_raw is fp32 [total_tokens][H].  All device buffers must be 16-byte
 * aligned.
 *
 * Ownership.  The caller owns every buffer passed in.  The library never
 * allocates or frees caller memory and never repacks the pool.  It owns one
 * thing: a cache of per-bounds metadata (device buffers plus a pinned staging
 * ring), kept for the life of the process or until kda_release_cache().
 *
 * Errors.  Every entry point returns KDA_OK (0) or a negative code from checks
 * made on the host before any work is enqueued.  Nothing is checked on the
 * device in a way that synchronises: the kernels compare state indices with
 * num_slots where they use them and record a bad one in a status word that
 * kda_check_status() reads afterwards.  kda_last_error() returns a message for
 * the calling thread's last failure.
 *
 * Streams.  All work is enqueued on `stream` (a cudaStream_t).  With host
 * bounds the call makes no synchronising CUDA call; without them it makes
 * exactly one device-to-host read-back of cu_seqlens (ROCm/aiter PR #6912,
 * "Changes": with cu_seqlens_cpu the bounds are never read back; without it,
 * once per tensor).
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_HEAD_DIM 128

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

typedef struct CUstream_st* kda_stream_t; /* same handle as cudaStream_t */

enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,  /* null pointer, bad size, stride, overlap, bounds */
    KDA_ERR_UNSUPPORTED = -2,  /* dtype, alignment or lower_bound out of range */
    KDA_ERR_CAPTURE_MISS = -3, /* metadata not cached while the stream captures */
    KDA_ERR_CUDA = -4,         /* a CUDA runtime or driver call failed */
    KDA_ERR_WORKSPACE = -5     /* workspace missing or smaller than required */
};

enum kda_state_dtype {
    KDA_STATE_F32 = 0,
    KDA_STATE_BF16 = 1,
    KDA_STATE_F16 = 2
};

/*
 * Chunk size C used by the kernels (tokens per intra-chunk tile).  It changes
 * nothing but rounding; exposed for tests and sizing.
 */
KDA_API int kda_chunk_size(void);

/*
 * Bytes of workspace a call with these sizes needs.  An upper bound that
 * depends only on the totals (the number of chunks is at most
 * ceil(total_tokens / C) + num_seqs), so it can be sized before the bounds are
 * known and stays valid under graph capture.  Returns 0 for invalid sizes.
 *
 * ROCm/aiter PR #4741, "Optimizations Applied" ("Single workspace pool": the
 * per-chunk tiles come from one allocation); here the caller provides it.
 */
KDA_API size_t kda_workspace_size(int64_t total_tokens, int32_t num_seqs, int32_t num_heads);

/*
 * kda_chunk_fwd — forward with the paged state pool read and written in-kernel.
 *
 *   q, k, v          device bf16 [total_tokens][num_heads][128]
 *   g_raw            device fp32 [total_tokens][num_heads][128], raw gate
 *   beta_raw         device fp32 [total_tokens][num_heads], raw beta
 *   cu_seqlens       device int32 [num_seqs+1] sequence bounds
 *   cu_seqlens_host  host int32 [num_seqs+1] holding the same values, or NULL.
 *                    Trusted, not compared with the device copy.  Must start
 *                    at 0, not decrease and end at total_tokens.
 *   state_cache      device pool [num_slots][num_heads][128 (V)][128 (K)] of
 *                    state_dtype.  Slot s, head h, element (v, k) lives at
 *                    s * state_stride0 + h * 128 * 128 + v * 128 + k.
 *   state_stride0    elements between slots, >= num_heads * 128 * 128; the
 *                    padding is never read or written.
 *   state_indices    device int32 [num_seqs], distinct slots in [0, num_slots).
 *                    Distinctness is not checked; a slot outside the range is
 *                    neither read nor written and reported by kda_check_status.
 *   has_initial_state device uint8 [num_seqs]: 0 starts the sequence from a
 *                    zero state and never reads its slot.
 *   out              device bf16 [total_tokens][num_heads][128], fully written;
 *                    must not overlap any input or the pool.
 *   lower_bound      gate lower bound (e.g. -5); must lie in [-64, 0].
 *   workspace        device scratch of at least kda_workspace_size() bytes,
 *                    256-byte aligned; contents on entry do not matter.
 *
 * Every selected slot receives its sequence's final state, rounded to the
 * pool dtype with round-to-nearest-even, empty sequences included (their final
 * state is their initial state, zeros without one).  Unselected slots and the
 * stride padding are untouched.
 *
 * Sequences of more than 8 tokens run through the chunked kernels (intra-chunk
 * tiles, then the state scan; when the scan needs few SMs, both in one
 * cooperative launch where the scan follows the intra-chunk work chunk by
 * chunk; for at most 4 (sequence, head) pairs of long sequences, the scan in
 * segments walked in parallel and chained through the segments' transitions);
 * sequences of at most 8 tokens (decode steps, empty sequences) run token by
 * token in another kernel with the state in fp32 registers.  All compute the
 * same recurrence; only rounding differs.
 *
 * CUDA graph capture: a call on a capturing stream is captured when
 * cu_seqlens_host is given and an earlier call, finished before the capture
 * began and made on any stream, had the same bounds (their tables are then
 * cached and the graph keeps them for the life of the process).  Otherwise it
 * returns KDA_ERR_CAPTURE_MISS and enqueues nothing.  Captured calls record no
 * kernel timing.
 *
 * ROCm/aiter PR #5754, "Technical Details": state_cache fp32 V-first
 * [slots, H, V, K] with a possibly padded stride(0); int32 state_indices; bool
 * has_initial_state (false starts from zero and does not read a dirty slot);
 * out required and not aliasing v; the load/store address slot * stride(0) +
 * head * V * K; the final state goes back to the same row.  ROCm/aiter PR
 * #5249, "What": 2-byte (fp16/bf16) state storage with fp32 accumulation.
 */
KDA_API int kda_chunk_fwd(const void* q, const void* k, const void* v,
                  const float* g_raw, const float* beta_raw,
                  const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                  int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                  void* state_cache, int64_t state_stride0, int32_t num_slots,
                  const int32_t* state_indices, const uint8_t* has_initial_state,
                  void* out, float lower_bound, int state_dtype,
                  void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_fwd_raw_bf16 — kda_chunk_fwd with the raw gate and raw beta in
 * bf16 (g_raw device bf16 [total_tokens][num_heads][128], beta_raw device bf16
 * [total_tokens][num_heads], 2-byte aligned); every other argument, the
 * arithmetic (fp32 from the up-converted values) and the error codes are those
 * of kda_chunk_fwd.  Reading 2 bytes per raw value instead of 4 cuts the
 * input bytes by 258 per token-head.  The pages run the fused prep on raw-bf16
 * as well as fp32 beta (ROCm/aiter PR #4741, "Accuracy": the unit tests cover
 * raw-bf16 vs fp32 beta).
 */
KDA_API int kda_chunk_fwd_raw_bf16(const void* q, const void* k, const void* v,
                  const void* g_raw, const void* beta_raw,
                  const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                  int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                  void* state_cache, int64_t state_stride0, int32_t num_slots,
                  const int32_t* state_indices, const uint8_t* has_initial_state,
                  void* out, float lower_bound, int state_dtype,
                  void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_fwd_dense — the same forward with dense per-sequence states.
 *
 *   initial_state     device [num_seqs][num_heads][128][128] of state_dtype,
 *                     or NULL for zero initial states.
 *   has_initial_state device uint8 [num_seqs] or NULL (= all set when
 *                     initial_state is given).
 *   final_state       device [num_seqs][num_heads][128][128] of state_dtype,
 *                     fully written; must not overlap any input.
 *
 * Mutually exclusive with the pool (ROCm/aiter PR #5754, "Technical Details":
 * dense initial_state unchanged and exclusive with state_cache).  It runs the
 * very same kernels and schedule as kda_chunk_fwd with identity slot numbers,
 * so out and final states are bit-identical to a paged call whose selected
 * slots hold the same initial states (same PR, "Test Result": torch.equal on
 * output and selected rows).
 */
KDA_API int kda_chunk_fwd_dense(const void* q, const void* k, const void* v,
                        const float* g_raw, const float* beta_raw,
                        const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                        int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                        const void* initial_state, const uint8_t* has_initial_state,
                        void* final_state, int state_dtype,
                        void* out, float lower_bound,
                        void* workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_plan_chunks — host-only chunk numbering (no CUDA call; usable without a
 * GPU).  From host bounds it writes, for every chunk j in launch order,
 * chunk_seq[j] (the sequence's position in cu_seqlens) and chunk_in_seq[j]
 * (the chunk's index inside its sequence), and seq_chunk_offset[n] = number of
 * chunks of sequences before n (num_seqs+1 entries).  Empty sequences keep
 * their number and own no chunk, so the table equals
 * repeat_interleave(arange(N), chunks_per_seq) paired with per-sequence aranges
 * (ROCm/aiter PR #6912, "Changes": chunks numbered by their sequence's position
 * in cu_seqlens; "Tests": numbering matches a repeat_interleave reference when
 * empty sequences come first).
 *
 *   chunk_size   tokens per chunk (> 0)
 *   capacity     entries available in chunk_seq / chunk_in_seq
 *   n_chunks     out: number of chunks
 * Returns KDA_OK, KDA_ERR_INVALID_ARG (bad bounds) or KDA_ERR_WORKSPACE
 * (capacity too small; *n_chunks still receives the count).
 */
KDA_API int kda_plan_chunks(const int32_t* cu_seqlens_host, int32_t num_seqs, int32_t chunk_size,
                    int32_t* chunk_seq, int32_t* chunk_in_seq, int32_t* seq_chunk_offset,
                    int64_t capacity, int64_t* n_chunks);

/* Message of the calling thread's last error ("" when none). */
KDA_API const char* kda_last_error(void);

/*
 * Frees the metadata cache.  Entries that a CUDA graph capture used are kept
 * (a graph may replay them).  Safe only when no call is in flight on another
 * host thread.  Returns KDA_OK or KDA_ERR_CUDA.
 */
KDA_API int kda_release_cache(void);

/* Number of entries currently held by the metadata cache (for tests). */
KDA_API int kda_cache_entries(void);

/*
 * Per-kernel timing for measurement.  While enabled, every forward records a
 * CUDA event on its stream before the first kernel and after each kernel
 * (a few microseconds of overhead, no synchronisation).  kda_kernel_times()
 * waits for the recorded events, adds each kernel's elapsed time over the calls
 * since the last read into ms[i] (i = launch order: 0 = intra-chunk kernel,
 * 1 = state scan, 2 = the two fused in one launch, used instead of 0 and 1 when
 * the scan's walks leave enough SMs free, 3 = token-by-token kernel for short
 * sequences; a kernel a call did not launch adds nothing), stores the number of
 * calls in *calls, the number of kernels (4) in *count, and clears the record.
 * ms must hold at least 4 entries.  Mirrors the per-kernel split the pages
 * report (ROCm/aiter PR #4741, "Performance": per-kernel microseconds per
 * layer-call).  Returns KDA_OK, KDA_ERR_INVALID_ARG or KDA_ERR_CUDA.
 */
KDA_API int kda_set_kernel_timing(int enable);
KDA_API int kda_kernel_times(float* ms, int capacity, int* count, int* calls);
/* Name of kernel i in launch order, or NULL. */
KDA_API const char* kda_kernel_name(int i);

/*
 * Status word of the last call that used `workspace` (NULL: the built-in
 * scratch of kda_chunk_fwd_noalloc), read after waiting for `stream`, the stream
 * that call ran on.  *status is 0 when the call completed normally; otherwise an
 * OR of KDA_STATUS_* bits.  Synchronises the stream, so it is not for use while
 * the stream captures.  Returns KDA_OK, KDA_ERR_INVALID_ARG or KDA_ERR_CUDA.
 *
 * The pages keep synchronous state-index checks off the hot path (ROCm/aiter
 * PR #5754, review findings); here the kernels compare each sequence's slot with
 * num_slots (one comparison per CTA, no synchronisation) and skip the access of a
 * slot outside the pool, and this call reports it afterwards.
 */
enum kda_status_bits {
    KDA_STATUS_WAIT_TIMEOUT = 1, /* a bounded wait in a kernel gave up: results incomplete */
    KDA_STATUS_SMEM_ALIGN = 2,   /* shared memory not 1 KB aligned: the intra kernel did nothing */
    KDA_STATUS_BAD_SLOT = 4,     /* a state index outside [0, num_slots): that sequence's
                                    slot was neither read nor written */
    KDA_STATUS_BOUNDS_MISMATCH = 8 /* kda_chunk_fwd_noalloc only: cu_seqlens (device) and
                                      cu_seqlens_host disagree; the call computed nothing
                                      (out, the pool and every other buffer unchanged) */
};
KDA_API int kda_check_status(const void* workspace, kda_stream_t stream, int* status);

/*
 * Diagnostic of the kernels' failure path, not part of the method: enqueues on
 * `stream` one kernel in which one thread runs the bounded wait every kernel
 * uses on something that never happens (kind 0: an mbarrier phase nothing
 * arrives on; kind 1: a ready flag of the fused launch that nothing sets).
 * The wait gives up after about one second and sets KDA_STATUS_WAIT_TIMEOUT,
 * which kda_check_status(workspace, stream, ...) then reads; nothing faults or
 * hangs, and the context stays usable.  `workspace`: device memory of at least
 * 256 bytes (any kda_chunk_fwd workspace), whose first 256 bytes are cleared.
 * Returns KDA_OK, KDA_ERR_INVALID_ARG or KDA_ERR_CUDA.
 */
KDA_API int kda_debug_wait_timeout(int kind, void* workspace, kda_stream_t stream);

/*
 * Enables (default) or disables the fused intra-chunk + scan launch for the
 * calls that follow, process-wide.  Disabled, every call runs the two kernels
 * one after the other; results are bit-identical either way (same arithmetic),
 * which makes this switch a check of the fused launch's hand-offs and a way to
 * time the two schedules.  Returns KDA_OK.
 */
KDA_API int kda_set_fused_launch(int enable);

/*
 * kda_chunk_fwd_noalloc — the paged forward for callers that cannot allocate
 * device memory.  The paper has no counterpart: this entry point exists for
 * integration only.
 *
 * Who needs it: code that runs where device allocation is not allowed or not
 * available, for instance a serving runtime that owns all device memory through
 * its own fixed arena and forbids cudaMalloc after start-up, a plain-C caller
 * with no device allocator of its own, or code that must not perturb another
 * allocator's bookkeeping.  kda_chunk_fwd needs a caller-provided workspace
 * and keeps a metadata cache that allocates on a miss; this call needs
 * neither.
 *
 * It takes the arguments of kda_chunk_fwd without the workspace, and
 * cu_seqlens_host is required (its values size the launch; the chunk table
 * itself is built on the device from cu_seqlens).  cu_seqlens and
 * cu_seqlens_host must hold the same values.  The device copy is not trusted:
 * the table is built from it clamped into [0, total_tokens] and made
 * non-decreasing, with every write bounded, and its totals and a checksum are
 * compared with the host copy's; on any difference no kernel of the call
 * computes anything and kda_check_status(NULL, stream, &s) reports
 * KDA_STATUS_BOUNDS_MISMATCH (the return value stays KDA_OK: the difference
 * is found on the device, after the call has returned).  Scratch memory comes from a
 * fixed array of KDA_NOALLOC_SCRATCH_BYTES compiled into the library; every
 * GPU that loads the library holds it until process exit.  The need is the
 * workspace for the call's exact chunk count (chunks of 64 tokens of the
 * sequences longer than 8 tokens, counted from cu_seqlens_host; about 74 KB
 * per chunk and head) plus the chunk table; sizes whose need exceeds the array
 * are rejected with KDA_ERR_WORKSPACE and a message giving both numbers
 * (64 MiB holds, e.g., a 4096-token prefill at 12 heads, or thousands of
 * one-token decode sequences).
 *
 * The first call on a device looks up the array's device address (a CUDA
 * runtime query, no allocation), so make the first call on each device before
 * any stream capture.  All calls share the one array and it keeps the last
 * call's contents: calls that overlap on the GPU race and give wrong results,
 * so order them (one stream, or events).  It calls no cudaMalloc, cudaFree or
 * other allocating routine.  Results equal kda_chunk_fwd's: same kernels, same
 * chunk table.  Its arguments pass kda_chunk_fwd's host checks (activations,
 * bounds, pool, overlaps) before any CUDA call, with the same error codes.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (64ull << 20)
KDA_API int kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v,
                                  const float* g_raw, const float* beta_raw,
                                  const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                                  int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                                  void* state_cache, int64_t state_stride0, int32_t num_slots,
                                  const int32_t* state_indices, const uint8_t* has_initial_state,
                                  void* out, float lower_bound, int state_dtype,
                                  kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
