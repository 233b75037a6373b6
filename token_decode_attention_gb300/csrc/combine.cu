// combine.cu -- merge of the split-K partial softmax states into the f16 output.
//
// Each position range j of a sequence leaves (m_j, l_j, acc_j[D]) with
//   m_j = max score of the range (log2 units), l_j = sum 2^(s - m_j),
//   acc_j = sum 2^(s - m_j) V.
// The exact softmax-weighted sum over the whole live range is
//   out = sum_j 2^(m_j - M) acc_j / sum_j 2^(m_j - M) l_j,   M = max_j m_j,
// the log-sum-exp merge of a max-subtracted softmax (exact in real arithmetic).
// Ranges at or past the live length were never written and are not read; a
// sequence whose live length fits one range already has its output written by
// the split-K kernel and is skipped here.
//
// One CTA per (sequence, head).  Launched with programmatic dependent launch:
// the CTAs may start while the split-K kernel drains, and wait for its memory
// with griddepcontrol.wait before reading the workspace.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "dattn_internal.h"
#include "ptx.cuh"

namespace dattn {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
    pdl_wait_primary();
    extern __shared__ __align__(16) float csm[];
    float *red = csm;                        // [kCombineWarps]
    float *part = csm + 32;                  // [kCombineWarps][D]
    float *wts = part + kCombineWarps * a.D; // [num_splits]

    const long long bh = blockIdx.x;
    const long long b = bh / a.H;
    const uint32_t cp = a.cur_pos[b];
    const int L = cp >= static_cast<uint32_t>(a.S - 1) ? a.S : static_cast<int>(cp) + 1;
    const int nsl = (L + a.split_len - 1) / a.split_len;
    if (nsl <= 1) return;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float2 *ml = a.ws_ml + bh * a.num_splits;

    float M = -INFINITY;
    for (int j = tid; j < nsl; j += kCombineThreads) M = fmaxf(M, ml[j].x);
    M = warp_max(M);
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
    for (int w = 1; w < kCombineWarps; ++w) M = fmaxf(M, red[w]);
    __syncthreads();

    float lsum = 0.f;
    for (int j = tid; j < nsl; j += kCombineThreads) {
        const float2 v = ml[j];
        const float w = exp2f(v.x - M);
        wts[j] = w;
        lsum = fmaf(w, v.y, lsum);
    }
    lsum = warp_sum(lsum);
    if (lane == 0) red[warp] = lsum;
    __syncthreads();
    lsum = 0.f;
    for (int w = 0; w < kCombineWarps; ++w) lsum += red[w];

    // Weighted sum of the partial accumulators: warp w takes ranges j = w mod 8,
    // each lane four consecutive channels (two chunks when D > 128).
    const int D = a.D;
    const int D4 = D / 4;
    const float *accb = a.ws_acc + bh * a.num_splits * D;
    float4 s0 = make_float4(0.f, 0.f, 0.f, 0.f), s1 = s0;
    for (int j = warp; j < nsl; j += kCombineWarps) {
        const float w = wts[j];
        const float4 *row = reinterpret_cast<const float4 *>(accb + static_cast<size_t>(j) * D);
        if (lane < D4) {
            const float4 v = row[lane];
            s0.x = fmaf(w, v.x, s0.x); s0.y = fmaf(w, v.y, s0.y);
            s0.z = fmaf(w, v.z, s0.z); s0.w = fmaf(w, v.w, s0.w);
        }
        if (lane + 32 < D4) {
            const float4 v = row[lane + 32];
            s1.x = fmaf(w, v.x, s1.x); s1.y = fmaf(w, v.y, s1.y);
            s1.z = fmaf(w, v.z, s1.z); s1.w = fmaf(w, v.w, s1.w);
        }
    }
    if (lane < D4) reinterpret_cast<float4 *>(part + warp * D)[lane] = s0;
    if (lane + 32 < D4) reinterpret_cast<float4 *>(part + warp * D)[lane + 32] = s1;
    __syncthreads();
    for (int d = tid; d < D; d += kCombineThreads) {
        float num = 0.f;
        for (int w = 0; w < kCombineWarps; ++w) num += part[w * D + d];
        reinterpret_cast<__half *>(a.out)[bh * D + d] = __float2half_rn(num / lsum);
    }
}

}  // namespace

size_t combine_smem_bytes(int num_splits, int D) {
    return sizeof(float) * (32 + static_cast<size_t>(kCombineWarps) * D + num_splits);
}

cudaError_t combine_configure_smem(int max_smem) {
    return cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                max_smem);
}

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t stream) {
    const long long blocks = static_cast<long long>(a.B) * a.H;
    if (blocks <= 0 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = combine_smem_bytes(a.num_splits, a.D);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

}  // namespace dattn
