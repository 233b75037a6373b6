// dattn_internal.h -- kernel argument blocks and launchers shared between the
// C-ABI layer (dattn_api.cpp) and the CUDA translation units.  Host-side types.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace dattn {

// Consumer warps per CTA of the fused split-K kernel; one more warp issues the
// bulk copies.
constexpr int kConsumerWarps = 8;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;

// Error codes a kernel records in the device error word.
constexpr unsigned kErrConsumerWait = 1u;
constexpr unsigned kErrProducerWait = 2u;
constexpr unsigned kErrDrainWait = 4u;

// Arguments of the fused split-K decode kernel.
//
// Grid: one CTA per (sequence b, head group g, split j), flattened as
// ((b * head_groups + g) * num_splits + j).  The CTA owns heads
// [g*heads_per_cta, min(H, (g+1)*heads_per_cta)) and positions
// [j*split_len, min((j+1)*split_len, L_b)).
struct DecodeArgs {
    const void *Q;            // f16 [B,H,D]
    const void *K;            // f16 [B,S,H,D]
    const void *V;            // f16 [B,S,H,D]
    void *out;                // f16 [B,H,D]
    const uint32_t *cur_pos;  // [B]
    float *ws_acc;            // [B,H,NS,D] unnormalised partial outputs
    float2 *ws_ml;            // [B,H,NS]   partial (running max in log2 units, sum)
    unsigned *err;            // device error word
    int B, H, D, S;
    int heads_per_cta;  // HG
    int head_groups;    // NHG
    int phases;         // PHI: lane groups sharing one head interleave positions
    int stage_pos;      // P: positions per pipeline stage (a multiple of PHI)
    int stages;         // NST: pipeline depth
    int num_splits;     // NS
    int split_len;      // positions per split
    int bar_offset;     // byte offset of the mbarriers in dynamic shared memory
    float qscale;       // log2(e) / sqrt(D), folded into q
};

// Arguments of the combine kernel (log-sum-exp merge of the splits).
struct CombineArgs {
    const float *ws_acc;
    const float2 *ws_ml;
    const uint32_t *cur_pos;
    void *out;
    int B, H, D, S;
    int num_splits;
    int split_len;
};

// Compile-time shape of one fused-kernel instance: lanes per KV row (head_dim/8
// rounded up to a power of two) and the number of (head, phase) slots each lane
// group keeps in registers.
struct DecodeVariant {
    int bdx;   // 1, 2, 4, 8, 16, 32
    int kmax;  // 1..4
};

// Launch the fused split-K kernel.  smem = dynamic shared memory bytes.
cudaError_t launch_decode_splitk(const DecodeArgs &a, DecodeVariant v, long long ctas,
                                 int smem, cudaStream_t stream);
// Resident CTAs per SM for a variant at a given dynamic shared memory size.
cudaError_t decode_occupancy(DecodeVariant v, int smem, int *ctas_per_sm);
// Raise the dynamic shared memory limit of every variant (once per device).
cudaError_t decode_configure_smem(int max_smem);
// Dynamic shared memory bytes the combine kernel needs.
size_t combine_smem_bytes(int num_splits, int D);
// Raise the combine kernel's dynamic shared memory limit (once per device).
cudaError_t combine_configure_smem(int max_smem);
// Launch the combine kernel with programmatic dependent launch on `stream`.
cudaError_t launch_combine(const CombineArgs &a, cudaStream_t stream);
// Device error word of the current device.
cudaError_t device_error_word(unsigned **ptr);

// Record `message` as the calling thread's dattn_last_error() text and return
// `status` (for entry points defined outside dattn_api.cpp).
int set_last_error(int status, const char *message);

// Page-faithful split calls.
cudaError_t launch_qk(const void *Q, const void *K, void *scores, int B, int H, int D, int S,
                      const uint32_t *cur_pos, cudaStream_t stream);
cudaError_t launch_pv(const void *scores, const void *V, void *out, int B, int H, int D,
                      int S, cudaStream_t stream);

}  // namespace dattn
