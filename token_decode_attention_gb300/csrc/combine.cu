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
// Grid: one CTA per (sequence, head, chunk of channels).  The host picks the
// chunk width from the expected number of pieces per unit: whole heads when
// units have few pieces (many sequences), narrow chunks when one sequence is
// spread over every partition, so each thread folds only a few pieces.  Each
// thread folds its pieces online (running max, rescaled sum and accumulator)
// after issuing their loads together; the per-thread states are folded once
// more through shared memory.  Launched with
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

constexpr int kThreads = 128;
constexpr int kInlinePrefix = 4096;  // batches summed from current_pos in the combine

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Fold one state (m, l, acc) into a running state, rescaling whichever of the
// two has the smaller maximum.
__device__ __forceinline__ void fold(float &M, float &L, float4 &A, float m, float l, float4 a) {
    if (l <= 0.f) return;
    if (m > M) {
        const float s = fast_exp2(M - m);  // 0 when M is -inf
        L *= s;
        A.x *= s;
        A.y *= s;
        A.z *= s;
        A.w *= s;
        M = m;
    }
    const float w = fast_exp2(m - M);
    L = fmaf(w, l, L);
    A.x = fmaf(w, a.x, A.x);
    A.y = fmaf(w, a.y, A.y);
    A.z = fmaf(w, a.z, A.z);
    A.w = fmaf(w, a.w, A.w);
}

__device__ __forceinline__ long long live_len(const uint32_t *cp, long long b, int S) {
    const uint32_t c = __ldg(cp + b);
    return c >= static_cast<uint32_t>(S - 1) ? S : static_cast<long long>(c) + 1;
}

__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineArgs a) {
    __shared__ float sm_m[kThreads], sm_l[kThreads];
    __shared__ float4 sm_a[kThreads];
    __shared__ long long sm_pre[kThreads / 32][2];

    const int nchunks = (a.D + a.chunk - 1) / a.chunk;
    const long long idx = blockIdx.x;
    const int chunk = static_cast<int>(idx % nchunks);
    const long long bh = idx / nchunks;
    const int h = static_cast<int>(bh % a.H);
    const long long b = bh / a.H;
    const int g = h / a.heads_per_cta;
    const int hl = h - g * a.heads_per_cta;
    const long long u = b * a.head_groups + g;

    const int tid = threadIdx.x;
    const long long Lb = live_len(a.cur_pos, b, a.S);
    // Live positions before sequence b and in total.  For batches of up to
    // kInlinePrefix sequences they are summed here from current_pos (an input,
    // readable before the decode kernel finishes); larger batches read the
    // prefix sums the decode kernel wrote.
    long long before = 0, total = 0;
    if (a.B <= kInlinePrefix) {
        for (int i = tid; i < a.B; i += kThreads) {
            const long long L = live_len(a.cur_pos, i, a.S);
            total += L;
            if (i < b) before += L;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            before += __shfl_xor_sync(0xffffffffu, before, o);
            total += __shfl_xor_sync(0xffffffffu, total, o);
        }
        if ((tid & 31) == 0) {
            sm_pre[tid >> 5][0] = before;
            sm_pre[tid >> 5][1] = total;
        }
        __syncthreads();
        before = total = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
            before += sm_pre[w][0];
            total += sm_pre[w][1];
        }
    }

    pdl_wait_primary();  // the decode kernel's workspace writes are visible after this
    // the next kernel on the stream may start its launch now; one launched with
    // programmatic dependent launch waits for this grid to complete before it
    // reads anything
    pdl_launch_dependents();
    if (a.B > kInlinePrefix) {
        before = a.ws_prefix[b];
        total = a.ws_prefix[a.B];
    }
    const long long nhg = a.head_groups;
    const long long W = nhg * total;
    const long long Pu = nhg * before + g * Lb;
    const long long c_first = range_owner(Pu, W, a.partitions);
    const long long c_last = range_owner(Pu + Lb - 1, W, a.partitions);
    if (c_first == c_last) return;  // written whole by the decode kernel
    const int npieces = static_cast<int>(c_last - c_first + 1);

    const int c0 = chunk * a.chunk;
    const int width = min(a.chunk, a.D - c0);  // a multiple of 8
    const int f4 = width / 4;                  // float4 per piece row
    const int nsub = kThreads / f4;            // pieces in flight
    const int sub = tid / f4, f = tid - sub * f4;
    const size_t hgs = a.heads_per_cta;

    float M = -INFINITY, L = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    if (sub < nsub) {
        // issue the loads of up to eight pieces before folding any of them
        for (int j0 = sub; j0 < npieces; j0 += 8 * nsub) {
            float2 ml[8];
            float4 v[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int j = j0 + r * nsub;
                ml[r] = make_float2(-INFINITY, 0.f);
                v[r] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (j < npieces) {
                    const size_t row = static_cast<size_t>(piece_slot(c_first + j, u)) * hgs + hl;
                    ml[r] = a.ws_ml[row];
                    v[r] = *reinterpret_cast<const float4 *>(a.ws_acc + row * a.D + c0 + f * 4);
                }
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) fold(M, L, A, ml[r].x, ml[r].y, v[r]);
        }
    }
    sm_m[tid] = M;
    sm_l[tid] = L;
    sm_a[tid] = A;
    __syncthreads();
    // Two-level fold over the pieces-in-flight index, for each float4 lane:
    // groups of eight subs, then the (at most eight) group results.  Each
    // level-1 thread reads only its own group and writes the group's first
    // entry, so the level needs no barrier inside it.
    const int ngroups = (nsub + 7) / 8;
    if (tid < ngroups * f4) {
        const int q = tid / f4, fq = tid - q * f4;
        const int s_end = min(nsub, q * 8 + 8);
        const int t0 = q * 8 * f4 + fq;
        float m2 = sm_m[t0], l2 = sm_l[t0];
        float4 a2 = sm_a[t0];
        for (int s2 = q * 8 + 1; s2 < s_end; ++s2) {
            const int o = s2 * f4 + fq;
            fold(m2, l2, a2, sm_m[o], sm_l[o], sm_a[o]);
        }
        sm_m[t0] = m2;
        sm_l[t0] = l2;
        sm_a[t0] = a2;
    }
    __syncthreads();
    if (tid < f4) {
        float m2 = sm_m[tid], l2 = sm_l[tid];
        float4 A2 = sm_a[tid];
        for (int q = 1; q < ngroups; ++q) {
            const int o = q * 8 * f4 + tid;
            fold(m2, l2, A2, sm_m[o], sm_l[o], sm_a[o]);
        }
        const float inv = 1.f / l2;
        __half2 lo = __floats2half2_rn(A2.x * inv, A2.y * inv);
        __half2 hi = __floats2half2_rn(A2.z * inv, A2.w * inv);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t *>(&lo);
        packed.y = *reinterpret_cast<uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(reinterpret_cast<__half *>(a.out) + bh * a.D + c0 + tid * 4) =
            packed;
    }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs &a, cudaStream_t stream) {
    if (a.chunk <= 0 || a.chunk % 8 != 0) return cudaErrorInvalidValue;
    const long long blocks = static_cast<long long>(a.B) * a.H * ((a.D + a.chunk - 1) / a.chunk);
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
