// split_calls.cu -- the page's two-dispatch form of decode attention, batched,
// at the page's own precision.  Cross-check entry points, not the hot path.
//
// "Developing Apple Metal Kernels in Rust - A Deep Dive Through Attention",
// section "The MSL, briefly":
//   attention_qk_f16: fp32 dot of Q and K in index order, times 1/sqrt(head_dim)
//                     (fp32), -infinity where pos > current_pos, stored as half.
//   attention_pv_f16: fp32 max and sum of exp over the half scores of a row,
//                     then out[d] = half(sum_i exp(s_i - max)/sum * V[i,h,d]).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "dattn_internal.h"

namespace dattn {
namespace {

// One thread per (b, h, pos).  Products and sums are rounded separately
// (__fmul_rn / __fadd_rn, never contracted to an FMA) so the result is the
// page's sequential fp32 arithmetic, bit for bit.
__global__ void __launch_bounds__(256) qk_kernel(const __half *__restrict__ Q,
                                                 const __half *__restrict__ K,
                                                 __half *__restrict__ scores, int B, int H,
                                                 int D, int S,
                                                 const uint32_t *__restrict__ cur_pos) {
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long total = static_cast<long long>(B) * H * S;
    if (idx >= total) return;
    const int p = static_cast<int>(idx % S);
    const long long bh = idx / S;
    const int h = static_cast<int>(bh % H);
    const long long b = bh / H;
    if (static_cast<uint32_t>(p) > cur_pos[b]) {
        scores[idx] = __float2half_rn(-INFINITY);
        return;
    }
    const float scale = 1.0f / sqrtf(static_cast<float>(D));
    const __half *q = Q + bh * D;
    const __half *k = K + ((b * S + p) * H + h) * static_cast<long long>(D);
    float score = 0.0f;
    for (int i = 0; i < D; i += 8) {
        const uint4 qa = *reinterpret_cast<const uint4 *>(q + i);
        const uint4 ka = *reinterpret_cast<const uint4 *>(k + i);
        const __half2 *q2 = reinterpret_cast<const __half2 *>(&qa);
        const __half2 *k2 = reinterpret_cast<const __half2 *>(&ka);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 qf = __half22float2(q2[e]);
            const float2 kf = __half22float2(k2[e]);
            score = __fadd_rn(score, __fmul_rn(qf.x, kf.x));
            score = __fadd_rn(score, __fmul_rn(qf.y, kf.y));
        }
    }
    score = __fmul_rn(score, scale);
    scores[idx] = __float2half_rn(score);
}

constexpr int kPvThreads = 256;
constexpr int kPvChunk = 2048;  // weights staged in shared memory per pass

__device__ __forceinline__ float block_reduce(float v, float *red, bool is_max) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float u = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, u) : v + u;
    }
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
    for (int w = 1; w < kPvThreads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    __syncthreads();
    return r;
}

// One CTA per (b, h).  The weight w_i = expf(s_i - max) / sum is computed once
// per position (the page recomputes it for every output channel; the value is
// the same) and applied to V in position order for each channel.
__global__ void __launch_bounds__(kPvThreads) pv_kernel(const __half *__restrict__ scores,
                                                        const __half *__restrict__ V,
                                                        __half *__restrict__ out, int H, int D,
                                                        int S) {
    __shared__ float red[kPvThreads / 32];
    __shared__ float wch[kPvChunk];
    const long long bh = blockIdx.x;
    const long long b = bh / H;
    const int h = static_cast<int>(bh % H);
    const __half *row = scores + bh * S;

    float mx = -INFINITY;
    for (int i = threadIdx.x; i < S; i += kPvThreads) mx = fmaxf(mx, __half2float(row[i]));
    mx = block_reduce(mx, red, true);
    float sum = 0.f;
    for (int i = threadIdx.x; i < S; i += kPvThreads) sum += expf(__half2float(row[i]) - mx);
    sum = block_reduce(sum, red, false);

    float acc = 0.f;
    const int d = threadIdx.x;
    for (int c0 = 0; c0 < S; c0 += kPvChunk) {
        const int n = min(kPvChunk, S - c0);
        for (int i = threadIdx.x; i < n; i += kPvThreads)
            wch[i] = expf(__half2float(row[c0 + i]) - mx) / sum;
        __syncthreads();
        if (d < D) {
            for (int i = 0; i < n; ++i) {
                const long long p = c0 + i;
                acc = fmaf(wch[i], __half2float(V[((b * S + p) * H + h) * D + d]), acc);
            }
        }
        __syncthreads();
    }
    if (d < D) out[bh * D + d] = __float2half_rn(acc);
}

}  // namespace

cudaError_t launch_qk(const void *Q, const void *K, void *scores, int B, int H, int D, int S,
                      const uint32_t *cur_pos, cudaStream_t stream) {
    const long long total = static_cast<long long>(B) * H * S;
    const long long blocks = (total + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    const __half *q = static_cast<const __half *>(Q);
    const __half *k = static_cast<const __half *>(K);
    __half *sc = static_cast<__half *>(scores);
    void *args[] = {&q, &k, &sc, &B, &H, &D, &S, const_cast<const uint32_t **>(&cur_pos)};
    return cudaLaunchKernel(reinterpret_cast<const void *>(qk_kernel),
                            dim3(static_cast<unsigned>(blocks)), dim3(256), args, 0, stream);
}

cudaError_t launch_pv(const void *scores, const void *V, void *out, int B, int H, int D, int S,
                      cudaStream_t stream) {
    const long long blocks = static_cast<long long>(B) * H;
    if (blocks > 0x7fffffffLL || D > kPvThreads) return cudaErrorInvalidValue;
    const __half *sc = static_cast<const __half *>(scores);
    const __half *v = static_cast<const __half *>(V);
    __half *o = static_cast<__half *>(out);
    void *args[] = {&sc, &v, &o, &H, &D, &S};
    return cudaLaunchKernel(reinterpret_cast<const void *>(pv_kernel),
                            dim3(static_cast<unsigned>(blocks)), dim3(kPvThreads), args, 0, stream);
}

}  // namespace dattn
