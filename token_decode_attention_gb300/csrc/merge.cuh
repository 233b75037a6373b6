// merge.cuh -- log-sum-exp merge of the pieces of one (sequence, head, chunk
// of channels), the work of one combine CTA.
//
// Piece j of a unit left, per head, m_j = max score (log2 units),
// l_j = sum 2^(s - m_j) and acc_j = sum 2^(s - m_j) V in workspace slot
// piece_slot(c_first + j, u).  The exact softmax-weighted sum over the unit's
// whole live range is
//   out = sum_j 2^(m_j - M) acc_j / sum_j 2^(m_j - M) l_j,   M = max_j m_j.
// NT threads share one task: thread (sub, f) takes pieces sub, sub + nsub, ...
// of float4 column f, INFLIGHT of them per round with their loads issued
// together; a round is absorbed with one rescale (its maximum first, then
// independent weights).  The per-thread states are then merged across subs:
// by an xor-shuffle butterfly inside each warp and one fold of the warps'
// results when the column count divides 32, otherwise in two levels through
// shared memory (groups of eight subs, then the group results).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "streamk.h"

namespace dattn {
namespace merge {

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Fold one state (m, l, acc) into a running state, rescaling whichever of the
// two has the smaller maximum.  Empty states (l <= 0) change nothing.
__device__ __forceinline__ void fold(float &M, float &L, float4 &A, float m, float l, float4 a) {
    if (l <= 0.f) return;
    if (m > M) {
        const float s = ex2(M - m);  // 0 when M is -inf
        L *= s;
        A.x *= s;
        A.y *= s;
        A.z *= s;
        A.w *= s;
        M = m;
    }
    const float w = ex2(m - M);
    L = fmaf(w, l, L);
    A.x = fmaf(w, a.x, A.x);
    A.y = fmaf(w, a.y, A.y);
    A.z = fmaf(w, a.z, A.z);
    A.w = fmaf(w, a.w, A.w);
}

// Merge state (m, l, a) into (M, L, A) symmetrically: both are rescaled to
// the larger maximum.  Empty states (m = -inf, l = 0) contribute nothing.
__device__ __forceinline__ void merge2(float &M, float &L, float4 &A, float m, float l, float4 a) {
    const float nm = fmaxf(M, m);
    if (nm == -INFINITY) return;  // both empty
    const float s1 = ex2(M - nm), s2 = ex2(m - nm);  // ex2(-inf) = 0
    L = fmaf(L, s1, l * s2);
    A.x = fmaf(A.x, s1, a.x * s2);
    A.y = fmaf(A.y, s1, a.y * s2);
    A.z = fmaf(A.z, s1, a.z * s2);
    A.w = fmaf(A.w, s1, a.w * s2);
    M = nm;
}

// Absorb a round of N loaded pieces (empty ones have l = 0) into the running
// state: the round's maximum first, then one rescale of the state and
// independent weights 2^(m_r - M).
template <int N>
__device__ __forceinline__ void absorb(float &M, float &L, float4 &A, const float2 *ml,
                                       const float4 *v) {
    float mr = -INFINITY;
#pragma unroll
    for (int r = 0; r < N; ++r)
        if (ml[r].y > 0.f) mr = fmaxf(mr, ml[r].x);
    if (mr == -INFINITY) return;  // nothing in this round
    const float nm = fmaxf(M, mr);
    const float s = ex2(M - nm);  // 0 while the state is empty
    L *= s;
    A.x *= s;
    A.y *= s;
    A.z *= s;
    A.w *= s;
#pragma unroll
    for (int r = 0; r < N; ++r) {
        const float w = ml[r].y > 0.f ? ex2(ml[r].x - nm) : 0.f;
        L = fmaf(w, ml[r].y, L);
        A.x = fmaf(w, v[r].x, A.x);
        A.y = fmaf(w, v[r].y, A.y);
        A.z = fmaf(w, v[r].z, A.z);
        A.w = fmaf(w, v[r].w, A.w);
    }
    M = nm;
}

__device__ __forceinline__ void store_normalised(void *out, long long bh, int D, int col,
                                                 float l, float4 A) {
    const float inv = 1.f / l;
    __half2 lo = __floats2half2_rn(A.x * inv, A.y * inv);
    __half2 hi = __floats2half2_rn(A.z * inv, A.w * inv);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t *>(&lo);
    packed.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(reinterpret_cast<__half *>(out) + bh * D + col) = packed;
}

__device__ __forceinline__ long long live_len(const uint32_t *cp, long long b, int S) {
    const uint32_t c = __ldg(cp + b);
    return c >= static_cast<uint32_t>(S - 1) ? S : static_cast<long long>(c) + 1;
}

// One merge task: head hl of unit u (output row bh = b * H + h), channels
// [c0, c0 + width) with width a multiple of 8, over partitions c_first ..
// c_first + npieces - 1 (npieces >= 2) of the W flattened positions cut into G
// ranges.  When W < G some ranges are empty and may lie between the unit's
// first and last partition: those partitions hold no piece (their slots were
// not written by this launch) and are skipped.  `sync` is a barrier of the NT
// threads; it is called the same number of times by all of them.  Shared
// buffers hold NT entries each.
template <int NT, int INFLIGHT, typename Sync>
__device__ __forceinline__ void merge_task(const float *ws_acc, const float2 *ws_ml, void *out,
                                           int D, int heads_per_cta, long long bh, int c0,
                                           int width, long long u, int hl, long long c_first,
                                           int npieces, long long W, long long G, int tid,
                                           float *sm_m, float *sm_l, float4 *sm_a, Sync sync) {
    const int f4 = width / 4;       // float4 per piece row
    const int nsub = NT / f4;       // pieces in flight
    const int sub = tid / f4, f = tid - sub * f4;
    const size_t hgs = static_cast<size_t>(heads_per_cta);

    float M = -INFINITY, L = 0.f;
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    if (sub < nsub) {
        for (int j0 = sub; j0 < npieces; j0 += INFLIGHT * nsub) {
            float2 ml[INFLIGHT];
            float4 v[INFLIGHT];
#pragma unroll
            for (int r = 0; r < INFLIGHT; ++r) {
                const int j = j0 + r * nsub;
                ml[r] = make_float2(-INFINITY, 0.f);
                v[r] = make_float4(0.f, 0.f, 0.f, 0.f);
                const long long c = c_first + j;
                // every range holds at least one position when W >= G
                if (j < npieces && (W >= G || range_begin(c + 1, W, G) > range_begin(c, W, G))) {
                    const size_t row = static_cast<size_t>(piece_slot(c, u)) * hgs + hl;
                    // through L2 (the states were written by the decode kernel's CTAs)
                    ml[r] = __ldcg(ws_ml + row);
                    v[r] = __ldcg(reinterpret_cast<const float4 *>(ws_acc + row * D + c0 + f * 4));
                }
            }
            absorb<INFLIGHT>(M, L, A, ml, v);
        }
    }
    if ((f4 & (f4 - 1)) == 0 && f4 <= 32) {
        // nsub * f4 == NT: every thread holds a sub.  The subs of column f in
        // one warp sit at lanes f, f + f4, ...: fold them with xor shuffles.
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            if (o < f4) break;
            const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
            const float l2 = __shfl_xor_sync(0xffffffffu, L, o);
            float4 a2;
            a2.x = __shfl_xor_sync(0xffffffffu, A.x, o);
            a2.y = __shfl_xor_sync(0xffffffffu, A.y, o);
            a2.z = __shfl_xor_sync(0xffffffffu, A.z, o);
            a2.w = __shfl_xor_sync(0xffffffffu, A.w, o);
            merge2(M, L, A, m2, l2, a2);
        }
        const int warp = tid >> 5, lane = tid & 31;
        if (lane < f4) {
            sm_m[warp * f4 + lane] = M;
            sm_l[warp * f4 + lane] = L;
            sm_a[warp * f4 + lane] = A;
        }
        sync();
        if (tid < f4) {
            float m2 = sm_m[tid], l2 = sm_l[tid];
            float4 a2 = sm_a[tid];
#pragma unroll
            for (int w = 1; w < NT / 32; ++w)
                merge2(m2, l2, a2, sm_m[w * f4 + tid], sm_l[w * f4 + tid], sm_a[w * f4 + tid]);
            store_normalised(out, bh, D, c0 + tid * 4, l2, a2);
        }
        return;
    }
    sm_m[tid] = M;
    sm_l[tid] = L;
    sm_a[tid] = A;
    sync();
    // Level 1: each thread folds one group of eight subs into the group's first
    // entry; it reads only its own group, so the level needs no barrier inside.
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
    sync();
    // Level 2: the group results, then normalise and store f16.
    if (tid < f4) {
        float m2 = sm_m[tid], l2 = sm_l[tid];
        float4 A2 = sm_a[tid];
        for (int q = 1; q < ngroups; ++q) {
            const int o = q * 8 * f4 + tid;
            fold(m2, l2, A2, sm_m[o], sm_l[o], sm_a[o]);
        }
        store_normalised(out, bh, D, c0 + tid * 4, l2, A2);
    }
}

}  // namespace merge
}  // namespace dattn
