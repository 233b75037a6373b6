// dattn_internal.h -- kernel argument blocks and launchers shared between the
// C-ABI layer (dattn_api.cpp) and the CUDA translation units.  Host-side types.
#pragma once

#include <cuda.h>  // CUtensorMap (a plain struct; the driver library is not linked)
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace dattn {

// Threads of a decode CTA with `nwc` consumer warps: one more warp issues the
// bulk copies.  Eight consumer warps run two CTAs per SM, sixteen run one.
__host__ __device__ constexpr int decode_threads(int nwc) { return (nwc + 1) * 32; }
__host__ __device__ constexpr int decode_min_blocks(int nwc) { return nwc <= 8 ? 2 : 1; }

// Error codes a kernel records in the device error word.
constexpr unsigned kErrConsumerWait = 1u;
constexpr unsigned kErrProducerWait = 2u;
constexpr unsigned kErrDrainWait = 4u;
constexpr unsigned kErrSelftestWait = 8u;
constexpr unsigned kErrPageIndex = 16u;  // a block-table entry outside [0, num_pages)
constexpr unsigned kErrAppendPosition = 32u;  // an append position outside the cache

// Time limit of every pipeline wait in the library's kernels.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // one second

// Arguments of the stream-K decode kernel.
//
// Units are (sequence b, head group g), u = b * head_groups + g, each holding
// the L_b live positions of heads [g*heads_per_cta, min(H, (g+1)*heads_per_cta)).
// Their positions, flattened unit after unit (W in total), are cut into
// `partitions` equal ranges, one per CTA (see streamk.h).  A CTA writes the
// f16 output of every unit it covers entirely and a partial softmax state for
// the others.
struct DecodeArgs {
    // Cluster mode (cluster > 0) with a head group smaller than H: tiled tensor
    // maps of K and V as [rows, H, D] (innermost D), box {D, HG, box_pos}: for a
    // dense cache the B*S positions and one full stage of a head group, for a
    // paged cache the num_pages*page_size rows of the pool and one page.
    CUtensorMap tmap_k, tmap_v;
    const void *Q;            // f16 [B,H,D]
    const void *K;            // f16 [B,S,H,D]
    const void *V;            // f16 [B,S,H,D]
    void *out;                // f16 [B,H,D]
    const uint32_t *cur_pos;  // [B]
    long long *ws_prefix;     // [B+1] live positions before each sequence (written by CTA 0)
    float *ws_acc;            // [(G+U), HG, D] unnormalised partial outputs
    float2 *ws_ml;            // [(G+U), HG]    partial (running max, log2 units; sum)
    unsigned *err;            // device error word
    // Paged cache (block_table != nullptr): K and V are pages
    // [num_pages, page_size, H, D] and position p of sequence b lives in page
    // block_table[b * max_pages + p / page_size], row p % page_size.  S is then
    // page_size * max_pages.
    const int *block_table;
    long long num_pages;
    int page_size, max_pages;
    int B, H, D, S;
    int heads_per_cta;  // HG
    int head_groups;    // NHG
    int phases;         // PHI: lane groups sharing one head interleave positions
    int stage_pos;      // P: positions per pipeline stage (a multiple of PHI)
    int stages;         // NST: pipeline depth
    int partitions;     // G: CTAs
    int active_warps;   // consumer warps holding at least one (head, phase) slot
    int merge_offset;   // byte offset of the phase-merge area in dynamic smem
    int bar_offset;     // byte offset of the mbarriers in dynamic smem
    float qscale;       // log2(e) / sqrt(D), applied to each dot product
    // Positions of its first stages each CTA prefetches into L2 before waiting
    // on the kernel before it (0 = none).
    int prefetch_positions;
    // Cluster mode: 0 = stream-K over the batch (above).  C > 0: the grid is
    // head_groups * B clusters of C CTAs; cluster u takes unit u = (b, g) whole,
    // CTA r of it the positions [r L_b / C, (r+1) L_b / C) of that unit, and
    // the C partial states are merged through distributed shared memory into
    // `out`.  No workspace and no second kernel.
    int cluster;
    int use_tmap;      // full stages (pages) of a head group are copied as tensor boxes
    int box_pos;       // positions of a tensor box: a stage (dense) or a page (paged)
    int prefetch_lanes;  // paged cache: lanes of warp 0 that read the prefetch window's pages (1..32)
    // Cluster mode: byte offset of this CTA's record [HG][D + 2] of its
    // partial state (m, l, acc) per head, read by the cluster's other CTAs.
    int rec_offset;
};

// Arguments of the combine kernel (log-sum-exp merge of the pieces of a unit).
struct CombineArgs {
    const float *ws_acc;
    const float2 *ws_ml;
    const long long *ws_prefix;
    const uint32_t *cur_pos;
    void *out;
    int B, H, D, S;
    int heads_per_cta;
    int head_groups;
    int partitions;
    int chunk;     // channels per combine CTA (a multiple of 8)
    int inflight;  // piece loads per thread per round: 2, 4 or 8
};

// Compile-time shape of one decode-kernel instance.
struct DecodeVariant {
    int bdx;   // lanes per KV row: 1, 2, 4, 8 (chunks = 1) or 8, 16 (chunks = 2)
    int ch;    // 8-element chunks per lane: 1 or 2
    int kmax;  // (head, phase) slots per lane group: 1..2 (1 when ch = 2)
    int nwc;   // consumer warps: 8 or 16
};

// Launch the decode kernel.  smem = dynamic shared memory bytes.
cudaError_t launch_decode(const DecodeArgs &a, DecodeVariant v, int smem, cudaStream_t stream);
// Resident CTAs per SM for a variant at a given dynamic shared memory size.
cudaError_t decode_occupancy(DecodeVariant v, int smem, int *ctas_per_sm);
// Clusters of `cluster` CTAs of a variant that can be resident at once.
cudaError_t decode_max_clusters(DecodeVariant v, int smem, int cluster, bool paged, int *clusters);
// Raise the dynamic shared memory limit of every variant (once per device).
cudaError_t decode_configure_smem(int max_smem);
// Launch the combine kernel with programmatic dependent launch on `stream`.
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t stream);
// Device error word of the current device.
cudaError_t device_error_word(unsigned **ptr);

// Record `message` as the calling thread's dattn_last_error() text and return
// `status` (for entry points defined outside dattn_api.cpp).
int set_last_error(int status, const char *message);

// Failure-detection self-test: one CTA waits (bounded) on an mbarrier that
// nothing arrives on and records kErrSelftestWait in `err` when the wait runs out.
cudaError_t launch_wait_timeout_selftest(unsigned *err, cudaStream_t stream);

// Arguments of the fused rotary-embedding + KV-append kernel (passed by value;
// the frequency table travels in the kernel's parameter space).
constexpr int kRopeMaxPairs = 256;  // rope_dims / 2 for head_dim up to 512
struct RopeAppendArgs {
    // theta_i / (2 pi) as a binary fraction in units of 2^-64, theta_i =
    // rope_base^(-2 i / rope_dims)
    unsigned long long turn_frac[kRopeMaxPairs];
    const void *q_new, *k_new, *v_new;  // f16 [B,H,D]
    void *q_out;                        // f16 [B,H,D] (may be q_new)
    void *K, *V;                        // cache: [B,S,H,D] or pages [num_pages,page_size,H,D]
    const int *block_table;             // nullptr: dense cache
    long long num_pages;
    int page_size, max_pages;
    const uint32_t *cur_pos;            // [B] position of the new token
    unsigned *err;
    int B, H, D, S;
    int rope_dims;
    int traditional;
    int heads_per_cta;
};
cudaError_t launch_rope_append(const RopeAppendArgs &a, cudaStream_t stream);

// Row softmax over the last dimension of a f32 [rows, cols] matrix.
cudaError_t launch_softmax(const float *x, float *out, long long rows, int cols,
                           unsigned *err, cudaStream_t stream);

// Page-faithful split calls.
cudaError_t launch_qk(const void *Q, const void *K, void *scores, int B, int H, int D, int S,
                      const uint32_t *cur_pos, cudaStream_t stream);
cudaError_t launch_pv(const void *scores, const void *V, void *out, int B, int H, int D,
                      int S, cudaStream_t stream);

}  // namespace dattn
