// combine.cu -- merge of the stream-K partial softmax states into f16 output.
//
// A unit (sequence b, head group g) whose live positions span several
// partitions c_first..c_last was processed in pieces; each piece j left
//   m_j = max score (log2 units), l_j = sum 2^(s - m_j), acc_j = sum 2^(s - m_j) V
// per head in workspace slot piece_slot(j, u) (see streamk.h).  The exact
// softmax-weighted sum over the unit's whole live range is
//   out = sum_j 2^(m_j - M) acc_j / sum_j 2^(m_j - M) l_j,   M = max_j m_j,
// the log-sum-exp merge of a max-subtracted softmax (exact in real arithmetic).
// Units held by a single partition already have their output written by the
// decode kernel and are skipped.
//
// Grid: one CTA per (sequence, head, chunk of 32 channels), so even a single
// long sequence spreads its merge over H * D/32 CTAs; inside a CTA, threads
// take (piece, float4) pairs and keep several loads in flight.  Launched with
// programmatic dependent launch: it may start while the decode kernel drains
// and waits on griddepcontrol.wait before touching the workspace.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "dattn_internal.h"
#include "ptx.cuh"
#include "streamk.h"

namespace dattn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 32;  // channels per CTA

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineArgs a) {
    __shared__ float red[kWarps];
    __shared__ float4 part[kThreads];

    const int nchunks = (a.D + kChunk - 1) / kChunk;
    const long long idx = blockIdx.x;
    const int chunk = static_cast<int>(idx % nchunks);
    const long long bh = idx / nchunks;
    const int h = static_cast<int>(bh % a.H);
    const long long b = bh / a.H;
    const int g = h / a.heads_per_cta;
    const int hl = h - g * a.heads_per_cta;
    const long long u = b * a.head_groups + g;

    const uint32_t cp = __ldg(a.cur_pos + b);
    const long long Lb = cp >= static_cast<uint32_t>(a.S - 1) ? a.S : static_cast<long long>(cp) + 1;

    pdl_wait_primary();  // the decode kernel's workspace writes are visible after this
    const long long nhg = a.head_groups;
    const long long W = nhg * a.ws_prefix[a.B];
    const long long Pu = nhg * a.ws_prefix[b] + g * Lb;
    const long long c_first = range_owner(Pu, W, a.partitions);
    const long long c_last = range_owner(Pu + Lb - 1, W, a.partitions);
    if (c_first == c_last) return;  // written whole by the decode kernel
    const int npieces = static_cast<int>(c_last - c_first + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const size_t hg_stride = a.heads_per_cta;
    auto ml_of = [&](int j) -> float2 {
        return a.ws_ml[static_cast<size_t>(piece_slot(c_first + j, u)) * hg_stride + hl];
    };

    float M = -INFINITY;
    for (int j = tid; j < npieces; j += kThreads) M = fmaxf(M, ml_of(j).x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) M = fmaxf(M, red[w]);
    __syncthreads();

    float lsum = 0.f;
    for (int j = tid; j < npieces; j += kThreads) {
        const float2 v = ml_of(j);
        lsum = fmaf(fast_exp2(v.x - M), v.y, lsum);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    if (lane == 0) red[warp] = lsum;
    __syncthreads();
    lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) lsum += red[w];

    // weighted sum of the partial accumulators for this chunk of channels
    const int c0 = chunk * kChunk;
    const int width = min(kChunk, a.D - c0);  // a multiple of 8
    const int f4 = width / 4;                 // float4 per piece row
    const int nsub = kThreads / f4;           // pieces in flight per pass
    const int sub = tid / f4, f = tid - sub * f4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (sub < nsub) {
        int j = sub;
        for (; j + 3 * nsub < npieces; j += 4 * nsub) {
            float4 v[4];
            float w[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int jj = j + r * nsub;
                const size_t row = static_cast<size_t>(piece_slot(c_first + jj, u)) * hg_stride + hl;
                v[r] = *reinterpret_cast<const float4 *>(a.ws_acc + row * a.D + c0 + f * 4);
                w[r] = fast_exp2(a.ws_ml[row].x - M);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                acc.x = fmaf(w[r], v[r].x, acc.x);
                acc.y = fmaf(w[r], v[r].y, acc.y);
                acc.z = fmaf(w[r], v[r].z, acc.z);
                acc.w = fmaf(w[r], v[r].w, acc.w);
            }
        }
        for (; j < npieces; j += nsub) {
            const size_t row = static_cast<size_t>(piece_slot(c_first + j, u)) * hg_stride + hl;
            const float4 v = *reinterpret_cast<const float4 *>(a.ws_acc + row * a.D + c0 + f * 4);
            const float w = fast_exp2(a.ws_ml[row].x - M);
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
    }
    part[tid] = acc;
    __syncthreads();
    if (tid < f4) {
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < nsub; ++r) {
            const float4 v = part[r * f4 + tid];
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        const float inv = 1.f / lsum;
        __half2 lo = __floats2half2_rn(s.x * inv, s.y * inv);
        __half2 hi = __floats2half2_rn(s.z * inv, s.w * inv);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t *>(&lo);
        packed.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(reinterpret_cast<__half *>(a.out) + bh * a.D + c0 + tid * 4) =
            packed;
    }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t stream) {
    const long long blocks = static_cast<long long>(a.B) * a.H * ((a.D + kChunk - 1) / kChunk);
    if (blocks <= 0 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

}  // namespace dattn
