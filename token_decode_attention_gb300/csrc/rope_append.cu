// rope_append.cu -- the step before decode attention: rotary position
// embedding of the new token's q and k ("Tutorial 16: Writing Custom Metal
// Kernels", section 5, FastRoPE: pairs rotated by a position-dependent angle,
// one position offset per batch entry) fused with appending the rotated k and
// the new v to the KV cache at that position.
//
// For sequence b, head h and position p = current_pos[b]:
//   theta_i = base^(-2 i / rope_dims) (fp64, on the host), a_i = p * theta_i
//   reduced modulo 2 pi exactly in fixed point (positions up to 2^31 would
//   leave an fp32 product p * theta_i with no correct digits),
//   pairs (i, i + rope_dims/2), or (2i, 2i + 1) when `traditional`,
//   (u, w) -> (u cos a - w sin a, u sin a + w cos a) in fp32, rounded to f16;
//   channels from rope_dims on are copied.  q_out gets the rotated q; the cache
//   rows K[b, p, h, :] and V[b, p, h, :] (dense, or through the block table)
//   get the rotated k and the new v.  A position outside the cache, or a page
//   outside the pool, is not written: the device error word records it.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "dattn_internal.h"
#include "ptx.cuh"

namespace dattn {
namespace {

constexpr int kThreads = 128;

// cos/sin of p * theta_i from the turn fraction f_i = theta_i / (2 pi) held as
// a 64-bit binary fraction.  p * f_i mod 1 is an exact wrapping integer
// product (the angle reduced modulo 2 pi with no rounding, whatever the size
// of p); its top 32 bits, as a signed fraction of a half turn, go to
// sincospif.  Angle error: 2^-24 pi from the float conversion, ~1.5e-9 rad
// from the dropped low bits.
__device__ __forceinline__ void angle_sincos(uint32_t p, unsigned long long f, float *c,
                                             float *s) {
    const unsigned long long turns = static_cast<unsigned long long>(p) * f;  // mod 2^64
    const int half_turns = static_cast<int>(static_cast<unsigned>(turns >> 32));
    sincospif(static_cast<float>(half_turns) * 0x1p-31f, s, c);
}

template <int VP>  // pairs per work item: 4 when rope_dims % 8 == 0, else 1
struct Pairs {
    float u[VP], w[VP];
};

template <int VP>
__device__ __forceinline__ void load_pairs(const __half *x, int i0, int i1, bool trad,
                                           Pairs<VP> &v) {
    if constexpr (VP == 4) {
        if (trad) {  // 8 consecutive halves: (u0 w0 u1 w1 ...)
            const uint4 raw = *reinterpret_cast<const uint4 *>(x + i0);
            const __half2 *h2 = reinterpret_cast<const __half2 *>(&raw);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __half22float2(h2[e]);
                v.u[e] = f.x;
                v.w[e] = f.y;
            }
        } else {  // 4 consecutive u, 4 consecutive w
            const uint2 ru = *reinterpret_cast<const uint2 *>(x + i0);
            const uint2 rw = *reinterpret_cast<const uint2 *>(x + i1);
            const __half2 *hu = reinterpret_cast<const __half2 *>(&ru);
            const __half2 *hw = reinterpret_cast<const __half2 *>(&rw);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float2 fu = __half22float2(hu[e]), fw = __half22float2(hw[e]);
                v.u[2 * e] = fu.x;
                v.u[2 * e + 1] = fu.y;
                v.w[2 * e] = fw.x;
                v.w[2 * e + 1] = fw.y;
            }
        }
    } else {
        v.u[0] = __half2float(x[i0]);
        v.w[0] = __half2float(x[i1]);
    }
}

template <int VP>
__device__ __forceinline__ void store_rotated(__half *x, int i0, int i1, bool trad,
                                              const Pairs<VP> &v, const float *c,
                                              const float *s) {
    __half ru[VP], rw[VP];
#pragma unroll
    for (int e = 0; e < VP; ++e) {
        ru[e] = __float2half_rn(v.u[e] * c[e] - v.w[e] * s[e]);
        rw[e] = __float2half_rn(v.u[e] * s[e] + v.w[e] * c[e]);
    }
    if constexpr (VP == 4) {
        if (trad) {
            uint4 raw;
            __half2 *h2 = reinterpret_cast<__half2 *>(&raw);
#pragma unroll
            for (int e = 0; e < 4; ++e) h2[e] = __halves2half2(ru[e], rw[e]);
            *reinterpret_cast<uint4 *>(x + i0) = raw;
        } else {
            uint2 a, b;
            __half2 *ha = reinterpret_cast<__half2 *>(&a);
            __half2 *hb = reinterpret_cast<__half2 *>(&b);
            ha[0] = __halves2half2(ru[0], ru[1]);
            ha[1] = __halves2half2(ru[2], ru[3]);
            hb[0] = __halves2half2(rw[0], rw[1]);
            hb[1] = __halves2half2(rw[2], rw[3]);
            *reinterpret_cast<uint2 *>(x + i0) = a;
            *reinterpret_cast<uint2 *>(x + i1) = b;
        }
    } else {
        x[i0] = ru[0];
        x[i1] = rw[0];
    }
}

// CTA (b, chunk of heads_per_cta heads).  The angles depend on (b, i) only:
// each CTA builds its cos/sin table once in shared memory and every head of
// the chunk rotates with it.
template <int VP>
__global__ void __launch_bounds__(kThreads) rope_append_kernel(const RopeAppendArgs a) {
    __shared__ float cos_t[kRopeMaxPairs], sin_t[kRopeMaxPairs];
    // Programmatic dependent launch on both sides: the kernel after this one
    // (the decode) may start launching at once, since it reads nothing before
    // waiting for this grid to complete; and this one reads nothing before the
    // kernel before it has completed.
    pdl_launch_dependents();
    pdl_wait_primary();
    const int hpc = a.heads_per_cta;
    const int chunks = (a.H + hpc - 1) / hpc;
    const long long b = blockIdx.x / chunks;
    const int h0 = static_cast<int>(blockIdx.x - b * chunks) * hpc;
    const int nh = min(hpc, a.H - h0);
    const int D = a.D, half = a.rope_dims / 2;
    const bool trad = a.traditional != 0;
    const uint32_t p = __ldg(a.cur_pos + b);

    for (int i = threadIdx.x; i < half; i += kThreads)
        angle_sincos(p, a.turn_frac[i], &cos_t[i], &sin_t[i]);

    // first cache row (b, p, h0), or none when the position or its page is invalid
    long long row0 = -1;
    if (p < static_cast<uint32_t>(a.S)) {
        if (a.block_table == nullptr) {
            row0 = (b * a.S + p) * a.H + h0;
        } else {
            const long long page = __ldg(a.block_table + b * a.max_pages + p / a.page_size);
            if (page >= 0 && page < a.num_pages)
                row0 = (page * a.page_size + p % a.page_size) * a.H + h0;
            else if (threadIdx.x == 0)
                atomicOr(a.err, kErrPageIndex);
        }
    } else if (threadIdx.x == 0) {
        atomicOr(a.err, kErrAppendPosition);
    }
    __syncthreads();

    const long long in0 = (b * a.H + h0) * static_cast<long long>(D);
    const __half *qi = reinterpret_cast<const __half *>(a.q_new) + in0;
    const __half *ki = reinterpret_cast<const __half *>(a.k_new) + in0;
    __half *qo = reinterpret_cast<__half *>(a.q_out) + in0;
    __half *ko = row0 >= 0 ? reinterpret_cast<__half *>(a.K) + row0 * D : nullptr;

    // work item (head j, pairs i .. i+VP-1); consecutive threads on consecutive
    // items.  A thread reads all of its pairs before writing them and no other
    // thread touches them, so q_out may alias q_new.
    const int per_head = half / VP;
    for (int t = threadIdx.x; t < nh * per_head; t += kThreads) {
        const int j = t / per_head;
        const int i = (t - j * per_head) * VP;
        const int i0 = j * D + (trad ? 2 * i : i);
        const int i1 = trad ? i0 + 1 : i0 + half;
        float c[VP], s[VP];
#pragma unroll
        for (int e = 0; e < VP; ++e) {
            c[e] = cos_t[i + e];
            s[e] = sin_t[i + e];
        }
        Pairs<VP> q, k;
        load_pairs<VP>(qi, i0, i1, trad, q);
        load_pairs<VP>(ki, i0, i1, trad, k);
        store_rotated<VP>(qo, i0, i1, trad, q, c, s);
        if (ko != nullptr) store_rotated<VP>(ko, i0, i1, trad, k, c, s);
    }
    // channels from rope_dims on pass through
    const int rest = D - a.rope_dims;
    if (VP == 4) {  // rope_dims % 8 == 0: whole 16-byte vectors
        const int rv = rest / 8;
        for (int t = threadIdx.x; t < nh * rv; t += kThreads) {
            const int j = t / rv;
            const int d = j * D + a.rope_dims + (t - j * rv) * 8;
            const uint4 qd = *reinterpret_cast<const uint4 *>(qi + d);
            const uint4 kd = *reinterpret_cast<const uint4 *>(ki + d);
            *reinterpret_cast<uint4 *>(qo + d) = qd;
            if (ko != nullptr) *reinterpret_cast<uint4 *>(ko + d) = kd;
        }
    } else {
        for (int t = threadIdx.x; t < nh * rest; t += kThreads) {
            const int j = t / rest;
            const int d = j * D + a.rope_dims + (t - j * rest);
            const __half qd = qi[d], kd = ki[d];
            qo[d] = qd;
            if (ko != nullptr) ko[d] = kd;
        }
    }
    // the value row: nh * D contiguous halves, 16-byte vectors (D % 8 == 0)
    if (row0 >= 0) {
        const uint4 *vi =
            reinterpret_cast<const uint4 *>(reinterpret_cast<const __half *>(a.v_new) + in0);
        uint4 *vo = reinterpret_cast<uint4 *>(reinterpret_cast<__half *>(a.V) + row0 * D);
        for (int t = threadIdx.x; t < nh * D / 8; t += kThreads) vo[t] = vi[t];
    }
}

}  // namespace

cudaError_t launch_rope_append(const RopeAppendArgs &a, cudaStream_t stream) {
    if (a.heads_per_cta <= 0 || a.rope_dims / 2 > kRopeMaxPairs || a.D % 8 != 0 ||
        a.rope_dims % 2 != 0)
        return cudaErrorInvalidValue;
    const long long chunks = (a.H + a.heads_per_cta - 1) / a.heads_per_cta;
    const long long blocks = static_cast<long long>(a.B) * chunks;
    if (blocks <= 0 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    void *args[] = {const_cast<RopeAppendArgs *>(&a)};
    const void *fn = a.rope_dims % 8 == 0 ? reinterpret_cast<const void *>(rope_append_kernel<4>)
                                          : reinterpret_cast<const void *>(rope_append_kernel<1>);
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
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace dattn
