// softmax.cu -- standalone row softmax over the last dimension (f32), the
// fm_softmax operation of Foundry's docs/metal.md ("Custom Compute Kernels",
// softmax_row: one threadgroup per row), re-done for sm_103a:
//   out[r, c] = exp(x[r, c] - max_c x[r, c]) / sum_c exp(x[r, c] - max_c x[r, c]).
// It is the max-subtracted softmax of the decode path (running max, sum of
// exponentials) exposed on its own.  HBM-bound: 8 bytes per element when a row
// fits in registers, 12 when it is read twice.
//
//   short rows (cols <= 1024): one warp per row, the row kept in registers
//     (32 values per lane), warp-shuffle max and sum: one read, one write;
//   long rows: one CTA per row, a pass computing the running (max, sum) per
//     thread merged across the block, then a pass writing the output.
#include <cuda_runtime.h>

#include <cmath>

#include "dattn_internal.h"

namespace dattn {
namespace {

constexpr int kWarpRowMax = 1024;     // columns handled by one warp from registers
constexpr int kPerLane = kWarpRowMax / 32;
constexpr int kRowThreads = 256;

__device__ __forceinline__ void merge(float &m, float &l, float m2, float l2) {
    // fold (m2, l2) into (m, l): l = sum exp(x - m) over both parts
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) return;  // both parts empty so far
    l = l * expf(m - M) + l2 * expf(m2 - M);
    m = M;
}

__global__ void __launch_bounds__(256) softmax_warp_rows(const float *__restrict__ x,
                                                         float *__restrict__ out, long long rows,
                                                         int cols) {
    const int lane = threadIdx.x & 31;
    const long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (r >= rows) return;
    const float *xr = x + r * cols;
    float v[kPerLane];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int c = lane + 32 * i;
        v[i] = c < cols ? xr[c] : -INFINITY;
        m = fmaxf(m, v[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float l = 0.f;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        v[i] = expf(v[i] - m);  // -inf - m = -inf -> 0 for the padding
        l += v[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    const float inv = 1.f / l;
    float *orow = out + r * cols;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int c = lane + 32 * i;
        if (c < cols) orow[c] = v[i] * inv;
    }
}

__global__ void __launch_bounds__(kRowThreads) softmax_block_rows(const float *__restrict__ x,
                                                                  float *__restrict__ out,
                                                                  int cols, bool vec4) {
    __shared__ float sm_m[kRowThreads / 32], sm_l[kRowThreads / 32];
    __shared__ int sm_nan[kRowThreads / 32];
    const long long r = blockIdx.x;
    const float *xr = x + r * cols;
    float *orow = out + r * cols;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float m = -INFINITY, l = 0.f;
    bool nan = false;
    if (vec4) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xr);
        for (int c = tid; c < cols / 4; c += kRowThreads) {
            const float4 t = x4[c];
            nan |= isnan(t.x) || isnan(t.y) || isnan(t.z) || isnan(t.w);
            const float mx = fmaxf(fmaxf(t.x, t.y), fmaxf(t.z, t.w));
            const float M = fmaxf(m, mx);
            if (M != -INFINITY) {
                l = l * expf(m - M) + expf(t.x - M) + expf(t.y - M) + expf(t.z - M) +
                    expf(t.w - M);
                m = M;
            }
        }
    } else {
        for (int c = tid; c < cols; c += kRowThreads) {
            const float t = xr[c];
            nan |= isnan(t);
            const float M = fmaxf(m, t);
            if (M != -INFINITY) {
                l = l * expf(m - M) + expf(t - M);
                m = M;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
        merge(m, l, m2, l2);
    }
    const bool warp_nan = __any_sync(0xffffffffu, nan);
    if (lane == 0) {
        sm_m[warp] = m;
        sm_l[warp] = l;
        sm_nan[warp] = warp_nan;
    }
    __syncthreads();
    m = sm_m[0];
    l = sm_l[0];
    bool row_nan = sm_nan[0];
#pragma unroll
    for (int w = 1; w < kRowThreads / 32; ++w) {
        merge(m, l, sm_m[w], sm_l[w]);
        row_nan |= sm_nan[w] != 0;
    }
    // a NaN anywhere in the row makes the whole row NaN, as the definition
    // does; an all -infinity row leaves m = -inf and gives NaN below as well
    if (row_nan) l = NAN;
    const float inv = 1.f / l;
    if (vec4) {
        const float4 *x4 = reinterpret_cast<const float4 *>(xr);
        float4 *o4 = reinterpret_cast<float4 *>(orow);
        for (int c = tid; c < cols / 4; c += kRowThreads) {
            const float4 t = x4[c];
            o4[c] = make_float4(expf(t.x - m) * inv, expf(t.y - m) * inv, expf(t.z - m) * inv,
                                expf(t.w - m) * inv);
        }
    } else {
        for (int c = tid; c < cols; c += kRowThreads) orow[c] = expf(xr[c] - m) * inv;
    }
}

}  // namespace

cudaError_t launch_softmax(const float *x, float *out, long long rows, int cols,
                           cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaErrorInvalidValue;
    if (cols <= kWarpRowMax) {
        const long long blocks = (rows + 7) / 8;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
        void *args[] = {&x, &out, &rows, &cols};
        return cudaLaunchKernel(reinterpret_cast<const void *>(softmax_warp_rows),
                                dim3(static_cast<unsigned>(blocks)), dim3(256), args, 0, stream);
    }
    if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
    bool vec4 = (cols % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) &&
                ((reinterpret_cast<uintptr_t>(out) & 15u) == 0);
    void *args[] = {&x, &out, &cols, &vec4};
    return cudaLaunchKernel(reinterpret_cast<const void *>(softmax_block_rows),
                            dim3(static_cast<unsigned>(rows)), dim3(kRowThreads), args, 0, stream);
}

}  // namespace dattn
