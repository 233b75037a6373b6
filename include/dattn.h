/*
 * dattn.h -- C ABI of libdattn: single-query (decode-step) scaled dot-product
 * attention against an f16 KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operation is the one defined by the two kernels of "Developing Apple
 * Metal Kernels in Rust - A Deep Dive Through Attention", section "The MSL,
 * briefly":
 *   attention_qk_f16:  score[h,pos] = (sum_i Q[h,i] * K_cache[pos,h,i]) / sqrt(head_dim),
 *                      -infinity where pos > current_pos;
 *   attention_pv_f16:  out[h,d] = sum_pos softmax(score[h,:])[pos] * V_cache[pos,h,d],
 *                      the softmax taken with the row maximum subtracted.
 * This library adds a leading batch dimension (independent sequences, one
 * current_pos each) and a fused entry point that never materialises the scores.
 *
 * Conventions shared by every entry point
 *   - f16 tensors are passed as untyped pointers to IEEE binary16 data, dense
 *     and row-major in the layouts given below, and must be 16-byte aligned
 *     (the page's allocator hands out 16-byte aligned blocks; section "Testing").
 *   - Every tensor and current_pos array is a pointer the current CUDA device
 *     can access: device memory, or page-locked host memory (cudaHostAlloc,
 *     cudaMallocHost, cudaHostRegister), which under unified addressing has the
 *     same address on the device.  The kernels read and write host memory over
 *     the CPU-GPU link (NVLink-C2C on GB300), so a decode step can take the new
 *     token's inputs from the host and return its output there without a
 *     copy-engine transfer; the KV cache belongs in device memory.  The caller
 *     owns all buffers and the stream; the library keeps no pointer after a call
 *     returns (like the page-3 C API, which wraps caller buffers and never frees
 *     them).
 *   - Calls are asynchronous: they only enqueue kernels on `stream` (NULL = the
 *     legacy default stream) and return.  The page's launcher waits after every
 *     dispatch (section "Commit, wait, and reading results back"); here the
 *     caller synchronises.  Faults during execution surface at that sync.
 *   - Arguments are validated on the host before anything is launched; on any
 *     non-zero return nothing has been written.  dattn_last_error() then gives a
 *     message for the calling thread.
 *   - current_pos is uint32 per sequence, the page's `uint` (section "The MSL,
 *     briefly").  A value >= seq_len masks nothing, exactly as the page's test
 *     `pos > current_pos` never fires then: the live length is
 *     L = min(current_pos, seq_len - 1) + 1.  The library never reads
 *     current_pos on the host.
 *   - Errors found while a kernel runs (a pipeline wait that ran out, a bad
 *     block-table entry, an append position outside the cache) cannot change a
 *     return value that was already given: the kernel records them in a device
 *     error word instead, and the outputs of the affected call are not valid.
 *     dattn_device_error() synchronises the device and reports that word; a
 *     caller that must know an output is valid checks it after the call.
 *   - The library keeps per-device state for the life of the process: kernel
 *     attributes, the address of the device error word, plans and the
 *     no-alloc scratch address.  cudaDeviceReset() (or any other teardown of the
 *     device's primary context) invalidates it; do not reset a device while the
 *     library is in use on it.
 */
#ifndef DATTN_H
#define DATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (identical to cudaStream_t / CUstream). */
typedef struct CUstream_st *dattn_stream_t;

/* Status codes returned by every int-returning entry point. */
enum dattn_status {
    DATTN_OK = 0,
    DATTN_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, bad count    */
    DATTN_ERR_UNSUPPORTED = -2, /* head_dim not a multiple of 8 or above 256       */
    DATTN_ERR_MISALIGNED = -3,  /* a tensor pointer is not 16-byte aligned          */
    DATTN_ERR_WORKSPACE = -4,   /* workspace missing, misaligned or too small       */
    DATTN_ERR_CUDA = -5,        /* a CUDA runtime call or kernel launch failed      */
    DATTN_ERR_TIMEOUT = -6,     /* a kernel gave up waiting on its own pipeline     */
    DATTN_ERR_BAD_PAGE = -7,    /* a live position's block-table entry was invalid  */
    DATTN_ERR_BAD_POSITION = -8 /* an append position was outside the cache         */
};

/* Library version: major*10000 + minor*100 + patch. */
int dattn_version(void);

/* Static string naming a status code. */
const char *dattn_status_string(int status);

/* Message describing the last non-OK return on the calling thread ("" if none). */
const char *dattn_last_error(void);

/*
 * Execution plan of the fused decode for a shape on the current device.
 * Filled by dattn_decode_plan(); informational.
 *
 * Two plans exist.  The split plan ("stream-K"): the live positions of the
 * whole batch, flattened over (sequence, head group, position), are cut into
 * `partitions` equal ranges, one per CTA, so every CTA streams the same number
 * of KV bytes whatever the mix of sequence lengths; a sequence whose positions
 * span several ranges is finished by a merge kernel.  The cluster plan (a
 * single sequence, dense or paged cache, library-chosen partitions): one
 * thread-block cluster of `cluster_size` CTAs per (sequence, head group); the
 * CTAs of a cluster split the live positions (at page boundaries for a paged
 * cache) and merge their partial softmax states through distributed shared
 * memory, so one launch writes `out` and no workspace is used.
 */
typedef struct dattn_plan {
    int partitions;      /* CTAs of the decode grid (equal ranges of positions)  */
    int heads_per_cta;   /* heads one CTA streams per position                   */
    int head_groups;     /* ceil(n_heads / heads_per_cta)                        */
    int stage_positions; /* positions per shared-memory pipeline stage           */
    int stages;          /* pipeline depth                                       */
    int threads_per_cta;
    int smem_bytes;      /* dynamic shared memory per CTA                        */
    int ctas_per_sm;     /* resident CTAs per SM at that shared-memory size      */
    int sm_count;
    size_t workspace_bytes;
    int cluster_size;    /* > 0: cluster plan, CTAs per cluster (no workspace,   */
                         /* no merge kernel); 0: stream-K over the batch          */
} dattn_plan;

/*
 * Plan the fused decode for (batch, n_heads, head_dim, seq_len) on the current
 * device.  num_partitions = 0 lets the library choose (every resident CTA slot
 * of the GPU, fewer when the batch's capacity is small); a positive value
 * forces that many partitions (clamped to 65535).
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA (device query failed).
 */
int dattn_decode_plan(int batch, int n_heads, int head_dim, int seq_len, int num_partitions,
                      dattn_plan *plan);

/*
 * The plan of dattn_decode_paged_f16 for (batch, n_heads, head_dim) over a pool
 * of num_pages pages of page_size positions with max_pages table entries per
 * sequence (seq_len = page_size * max_pages).  Same fields as dattn_decode_plan.
 * Errors: as dattn_decode_plan, plus INVALID_ARG for non-positive page_size,
 * max_pages or num_pages and UNSUPPORTED when page_size * max_pages >= 2^31.
 */
int dattn_decode_paged_plan(int batch, int n_heads, int head_dim, int page_size, int max_pages,
                            long long num_pages, int num_partitions, dattn_plan *plan);

/*
 * Workspace that dattn_decode_f16_ex and dattn_decode_paged_f16 need for this
 * shape and num_partitions on the current device, in bytes: the larger of the
 * two calls' needs (0 when the split plan has a single partition; the cluster
 * plan of a dense cache needs none, dattn_decode_plan() reports the dense
 * call's own figure).  It holds the batch's live-length prefix sums and one
 * fp32 partial softmax state (m, l, acc[head_dim]) per head for each
 * (partition, head group) piece; it is scratch, rewritten by every call.
 * Errors: as dattn_decode_plan, plus INVALID_ARG for a null `bytes`.
 */
int dattn_decode_workspace_bytes(int batch, int n_heads, int head_dim, int seq_len,
                                 int num_partitions, size_t *bytes);

/*
 * Fused decode attention with a caller-provided workspace.
 *
 *   Q            [batch, n_heads, head_dim]            f16, device
 *   K_cache      [batch, seq_len, n_heads, head_dim]   f16, device
 *   V_cache      [batch, seq_len, n_heads, head_dim]   f16, device
 *   out          [batch, n_heads, head_dim]            f16, device (written)
 *   current_pos  [batch]                               uint32, device
 *   workspace       device scratch, 16-byte aligned, >= dattn_decode_workspace_bytes
 *                   (may be NULL when that is 0)
 *   num_partitions  0 = library choice, > 0 forces the number of partitions
 *
 * For each sequence b and head h, with L = min(current_pos[b], seq_len-1) + 1:
 *   out[b,h,:] = sum_{p<L} softmax_p(Q[b,h,:].K[b,p,h,:] / sqrt(head_dim)) V[b,p,h,:]
 * computed with fp32 accumulation and an online (running max/sum) softmax, then
 * rounded to f16 (round to nearest even).  Positions p >= L never enter the
 * computation, whatever their contents (NaN included): the page's -infinity
 * score gives them weight exactly zero.  (Their memory may still be touched:
 * the L2 prefetch described under dattn_decode_paged_f16 works on ranges
 * planned for full caches, and a paged cache's last live page is copied
 * whole.)  The live positions are divided among CTAs (see dattn_plan); the
 * partial softmax states of a sequence that spans several CTAs are merged
 * (log-sum-exp merge) by a second kernel, or, in the cluster plan, through
 * distributed shared memory within the same launch.  Everything is enqueued on
 * `stream`.
 *
 * Concurrent calls on different streams need different workspaces.
 * A return of DATTN_OK means the kernels were enqueued.  The output is valid
 * once the stream has reached them and dattn_device_error() reports DATTN_OK:
 * a CTA whose bounded pipeline wait ran out (after one second) leaves its part
 * of `out` unwritten and records DATTN_ERR_TIMEOUT in the device error word.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA.
 */
int dattn_decode_f16_ex(const void *Q, const void *K_cache, const void *V_cache, void *out,
                        int batch, int n_heads, int head_dim, int seq_len,
                        const uint32_t *current_pos, void *workspace, size_t workspace_bytes,
                        int num_partitions, dattn_stream_t stream);

/*
 * Fused decode attention with the library's own workspace: same operation and
 * arguments as dattn_decode_f16_ex with num_partitions = 0.  The workspace is owned
 * by the library, one per (device, stream), grown on demand with cudaMalloc
 * (serialised by a mutex) and kept until process exit; a call that has to grow
 * it synchronises the device first.  Make the first call for the largest shape
 * outside any CUDA graph capture: a call that would have to grow the workspace
 * while its stream is being captured returns DATTN_ERR_WORKSPACE and leaves the
 * capture intact.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA.
 */
int dattn_decode_f16(const void *Q, const void *K_cache, const void *V_cache, void *out,
                     int batch, int n_heads, int head_dim, int seq_len,
                     const uint32_t *current_pos, dattn_stream_t stream);

/*
 * Fused decode attention over a paged KV cache (the "direct page reads" form of
 * decode attention in "Tutorial 16: Writing Custom Metal Kernels", section 7,
 * for a cache held in fixed-size pages as the page-1 engine's paged block
 * allocator does).  Same operation and output as dattn_decode_f16_ex; only the
 * addressing of K and V differs (and, for a single sequence, possibly the plan:
 * dattn_decode_paged_plan() reports it; where both calls take the same plan
 * the rounding is the same too):
 *
 *   K_pages, V_pages  [num_pages, page_size, n_heads, head_dim]   f16, device
 *   block_table       [batch, max_pages]                          int32, device
 *   K[b, p, h, :] = K_pages[block_table[b, p / page_size], p % page_size, h, :]
 *
 * Each sequence's capacity is seq_len = page_size * max_pages (< 2^31).
 * Pages may be shared between sequences.  Entries for pages past a sequence's
 * live length have no effect: K and V are never read through them, and they
 * raise no error.  (The kernel may read a few entries, live or not, as L2
 * prefetch hints before the kernel before it on `stream` has finished; such a
 * hint is bounds-checked and changes no result.)  A live entry outside
 * [0, num_pages) is not dereferenced: page 0 is read instead, the output of
 * that call is wrong, and dattn_device_error() reports DATTN_ERR_BAD_PAGE.
 * The workspace is the one of dattn_decode_workspace_bytes(batch, n_heads,
 * head_dim, page_size * max_pages, num_partitions).
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA.
 */
int dattn_decode_paged_f16(const void *Q, const void *K_pages, const void *V_pages, void *out,
                           int batch, int n_heads, int head_dim, int page_size, int max_pages,
                           long long num_pages, const int32_t *block_table,
                           const uint32_t *current_pos, void *workspace, size_t workspace_bytes,
                           int num_partitions, dattn_stream_t stream);

/*
 * The page's first dispatch, attention_qk_f16, batched ("The MSL, briefly"):
 *   scores[b,h,p] = half( (fp32 sum over i in index order of Q[b,h,i]*K[b,p,h,i],
 *                          each product and each sum rounded to fp32)
 *                         * (1.0f / sqrtf(head_dim)) )        for p <= current_pos[b]
 *   scores[b,h,p] = -infinity                                 for p >  current_pos[b]
 *   scores  [batch, n_heads, seq_len] f16, device (written)
 * Kept for cross-checking the fused path against the page's two-dispatch form.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, CUDA.
 */
int dattn_qk_f16(const void *Q, const void *K_cache, void *scores, int batch, int n_heads,
                 int head_dim, int seq_len, const uint32_t *current_pos,
                 dattn_stream_t stream);

/*
 * The page's second dispatch, attention_pv_f16, batched: per (b,h), fp32 max of
 * the scores row, fp32 sum of expf(score - max), then
 *   out[b,h,d] = half( sum over all seq_len positions p of
 *                      (expf(score[b,h,p] - max) / sum) * V[b,p,h,d] ).
 * Masking is carried by -infinity scores (weight 0); as on the page every
 * position is multiplied in, so a NaN in V at a zero-weight position propagates.
 *   scores [batch, n_heads, seq_len] f16, device;  out [batch, n_heads, head_dim]
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, CUDA.
 */
int dattn_pv_f16(const void *scores, const void *V_cache, void *out, int batch, int n_heads,
                 int head_dim, int seq_len, dattn_stream_t stream);

/* Size of the static scratch array used by dattn_decode_f16_noalloc. */
#define DATTN_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * Fused decode attention that allocates nothing.  The paper has no counterpart
 * to this entry point; it exists for callers that cannot call cudaMalloc at
 * decode time (a runtime that owns all device memory through its own pool, or
 * code that runs where an allocation is forbidden or would synchronise).
 *
 * Same operation and arguments as dattn_decode_f16 (library-chosen partition
 * count).  Instead of a workspace it uses a static device array of
 * DATTN_NOALLOC_SCRATCH_BYTES (32 MiB) that belongs to the library image: every
 * GPU on which the library's code is loaded holds that array until the process
 * exits.  Shapes whose partial softmax states need more than that are rejected
 * with DATTN_ERR_WORKSPACE before anything is launched; dattn_decode_f16_ex
 * with a caller workspace handles them.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with the device current); make that first call
 * before any stream capture.  All calls share the one array and it keeps the
 * previous call's contents (nothing in it needs to start at zero): calls whose
 * executions overlap on the GPU (different streams, or without ordering
 * between them) race on the scratch and give wrong results.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA.
 */
int dattn_decode_f16_noalloc(const void *Q, const void *K_cache, const void *V_cache,
                             void *out, int batch, int n_heads, int head_dim, int seq_len,
                             const uint32_t *current_pos, dattn_stream_t stream);

/*
 * The step before decode attention: rotary position embedding of the new
 * token's query and key fused with appending the key and value to the cache
 * ("Tutorial 16: Writing Custom Metal Kernels", section 5: FastRoPE splits each
 * vector into pairs and rotates every pair by a position-dependent angle, with
 * one position offset per batch entry).  For sequence b the new token sits at
 * position p = current_pos[b]; for pair i < rope_dims/2,
 *   theta_i = rope_base^(-2 i / rope_dims),  a = p * theta_i  (in fp64),
 *   pair (i, i + rope_dims/2), or (2i, 2i+1) when `traditional` is non-zero,
 *   (u, w) -> (u cos a - w sin a, u sin a + w cos a)  (fp32, rounded to f16);
 *   channels from rope_dims on are copied.
 * Writes q_out[b,h,:] = rope(q_new[b,h,:]) (q_out may be q_new),
 *        K_cache[b,p,h,:] = rope(k_new[b,h,:]),  V_cache[b,p,h,:] = v_new[b,h,:].
 *   q_new, k_new, v_new, q_out  [batch, n_heads, head_dim] f16, device
 *   K_cache, V_cache            [batch, seq_len, n_heads, head_dim] f16, device
 * A position p >= seq_len is not written; dattn_device_error() then reports
 * DATTN_ERR_BAD_POSITION.  Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, CUDA.
 */
int dattn_rope_append_f16(const void *q_new, const void *k_new, const void *v_new, void *q_out,
                          void *K_cache, void *V_cache, int batch, int n_heads, int head_dim,
                          int seq_len, int rope_dims, double rope_base, int traditional,
                          const uint32_t *current_pos, dattn_stream_t stream);

/*
 * The same over a paged cache (see dattn_decode_paged_f16): the key and value
 * go to page block_table[b, p / page_size], row p % page_size.  An invalid
 * page is not written and reported as DATTN_ERR_BAD_PAGE.
 */
int dattn_rope_append_paged_f16(const void *q_new, const void *k_new, const void *v_new,
                                void *q_out, void *K_pages, void *V_pages, int batch,
                                int n_heads, int head_dim, int page_size, int max_pages,
                                long long num_pages, const int32_t *block_table, int rope_dims,
                                double rope_base, int traditional, const uint32_t *current_pos,
                                dattn_stream_t stream);

/*
 * Row softmax over the last dimension, f32: the fm_softmax operation of the C
 * API in Foundry's docs/metal.md ("Custom Compute Kernels"), i.e. the
 * max-subtracted softmax of the decode path's reduction on its own:
 *   out[r, c] = exp(x[r, c] - max_c x[r, c]) / sum_c exp(x[r, c] - max_c x[r, c])
 *   x, out  [rows, cols] f32, device, row-major, 4-byte aligned (out may equal x)
 * computed in fp32: expf for rows up to 16384 columns; longer rows whose width
 * is a multiple of 4 and whose pointers are 16-byte aligned use exp2 of the
 * log2(e)-scaled difference formed by one fused multiply-add (relative error
 * about 1e-6).  -infinity entries get weight 0; a row with a NaN, or with every
 * entry -infinity, comes out NaN, as the definition gives.
 * Errors: INVALID_ARG, MISALIGNED, UNSUPPORTED, CUDA.
 */
int dattn_softmax_f32(const float *x, float *out, long long rows, int cols,
                      dattn_stream_t stream);

/*
 * Submission batching: the analogue of the fm_batch_begin / fm_batch_end pair
 * of the C API in Foundry's docs/metal.md (section "Command Batching"), which
 * accumulates operations into one GPU submission.  Here the calls issued on a
 * stream between dattn_batch_begin and dattn_batch_end are recorded (CUDA
 * stream capture, thread-local mode) instead of run; dattn_batch_end turns
 * them into a replayable batch and dattn_batch_launch submits all of them at
 * once on any stream, as often as wanted.  A replay reads the buffers the
 * recorded calls were given, with their contents at replay time: to decode a
 * new token, write the new Q / cache rows / current_pos into the same buffers
 * and launch again.
 *
 * Calls that may be recorded: dattn_decode_f16_ex, dattn_decode_paged_f16,
 * dattn_decode_f16_noalloc after its first call on the device, dattn_qk_f16,
 * dattn_pv_f16, dattn_rope_append_f16, dattn_rope_append_paged_f16,
 * dattn_softmax_f32, and dattn_decode_f16 once its workspace is large enough
 * (a recorded call must not allocate).  Copies the caller issues on the same
 * stream meanwhile (cudaMemcpyAsync from pinned host memory, for example) are
 * recorded too.  The shape's plan is made when a call is
 * recorded; make one ordinary call per shape first if its set-up should not
 * happen during recording.  `stream` must be a created stream, not NULL.
 * Errors: INVALID_ARG, CUDA (for example a recorded call that synchronised).
 */
typedef struct dattn_batch dattn_batch;
int dattn_batch_begin(dattn_stream_t stream);
int dattn_batch_end(dattn_stream_t stream, dattn_batch **batch);
int dattn_batch_launch(const dattn_batch *batch, dattn_stream_t stream);
/* Number of GPU operations recorded in a batch (-1 for NULL). */
long long dattn_batch_nodes(const dattn_batch *batch);
int dattn_batch_destroy(dattn_batch *batch);

/*
 * Device-side error word of the current device.  Every wait inside the fused
 * kernel's shared-memory pipeline is bounded (about one second); a wait that
 * runs out records a code here, abandons its CTA's output and returns instead
 * of hanging the GPU.  The paged decode records invalid block-table entries
 * here too.  This call synchronises the device and returns DATTN_OK if no
 * kernel has recorded anything since the last clear, DATTN_ERR_TIMEOUT if a
 * wait ran out, DATTN_ERR_BAD_PAGE if a block-table entry was invalid,
 * DATTN_ERR_BAD_POSITION if an append position was outside the cache; it
 * resets the word when `clear` is non-zero.
 * Errors: TIMEOUT, BAD_PAGE, BAD_POSITION, CUDA.
 */
int dattn_device_error(int clear);

/*
 * Self-test of the failure detection above (no counterpart on the pages).
 * Enqueues on `stream` one CTA that waits, with the same bounded wait the
 * decode kernel uses, on an mbarrier nothing ever arrives on.  After about one
 * second the wait runs out, the CTA records a code in the device error word and
 * returns; no fault, trap or hang is involved and the context stays usable.  A
 * following dattn_device_error() then returns DATTN_ERR_TIMEOUT.
 * Errors: CUDA.
 */
int dattn_selftest_wait_timeout(dattn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DATTN_H */
