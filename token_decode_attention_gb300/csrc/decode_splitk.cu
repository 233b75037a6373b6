// decode_splitk.cu -- fused split-K ("flash-decoding") decode attention for
// sm_103a.
//
// Computes, per sequence b and head h, the masked softmax attention of the
// kernels attention_qk_f16 and attention_pv_f16 of "Developing Apple Metal
// Kernels in Rust - A Deep Dive Through Attention" (section "The MSL, briefly")
// in one pass over the live KV rows, without materialising scores:
//   s_p  = (Q[b,h,:] . K[b,p,h,:]) / sqrt(D)         p < L_b = min(cp_b, S-1)+1
//   out  = sum_p exp(s_p - max s) V[b,p,h,:] / sum_p exp(s_p - max s)
//
// Design (GB300):
//   * One CTA per (sequence, head group, position range).  For a run of
//     positions, the K rows of all heads of a sequence are one contiguous span
//     of HBM (layout [B,S,H,D]); a producer warp streams that span, and the
//     matching V span, into a multi-stage shared-memory ring with bulk
//     asynchronous copies (cp.async.bulk on the TMA engine) that complete on
//     mbarriers.  Positions past L_b are never read: the page's -infinity mask
//     becomes a loop bound.
//   * Eight consumer warps split each KV row of D halves across D/8 lanes
//     (16-byte shared-memory loads), reduce the dot product with xor shuffles,
//     and keep an online softmax (running max m, running sum l, unnormalised
//     accumulator acc) per (head, phase) slot in registers, in fp32.  Scores are
//     kept in log2 units (q is pre-scaled by log2(e)/sqrt(D)) so exp2 is used.
//   * The CTA writes either the final f16 output (when its range is the only
//     live one of the sequence) or its partial state (m, l, acc) to the
//     workspace for the combine kernel.
//   * Every mbarrier wait is bounded; a wait that runs out records an error in
//     the device error word and the CTA returns after draining its copies.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "dattn_internal.h"
#include "ptx.cuh"

namespace dattn {

__device__ unsigned g_device_error = 0;

namespace {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second per wait

__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t polls = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++polls & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

__device__ __forceinline__ void unpack8(const uint4 r, float f[8]) {
    const __half2 *h = reinterpret_cast<const __half2 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __half22float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

template <int BDX, int KMAX>
__global__ void __launch_bounds__(kDecodeThreads, 2) decode_splitk_kernel(const DecodeArgs a) {
    constexpr int BDY = 32 / BDX;              // lane groups per warp
    constexpr int NLG = kConsumerWarps * BDY;  // lane groups per CTA
    extern __shared__ __align__(128) unsigned char smem[];

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    long long cta = blockIdx.x;
    const int split = static_cast<int>(cta % a.num_splits);
    cta /= a.num_splits;
    const int g = static_cast<int>(cta % a.head_groups);
    const long long b = cta / a.head_groups;
    const int h0 = g * a.heads_per_cta;
    const int hg = min(a.heads_per_cta, a.H - h0);
    const int D = a.D;

    const uint32_t cp = __ldg(a.cur_pos + b);
    const int L = cp >= static_cast<uint32_t>(a.S - 1) ? a.S : static_cast<int>(cp) + 1;
    const int p_begin = split * a.split_len;

    // The combine kernel may begin launching; it waits for this grid to finish.
    pdl_launch_dependents();
    if (p_begin >= L) return;  // range entirely masked: nothing to read or write

    const int p_end = min(p_begin + a.split_len, L);
    const int n_pos = p_end - p_begin;
    const int n_stages = (n_pos + a.stage_pos - 1) / a.stage_pos;
    const bool only_split = L <= a.split_len;

    const size_t buf_elems = static_cast<size_t>(a.stage_pos) * a.heads_per_cta * D;
    __half *ring = reinterpret_cast<__half *>(smem);
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + a.bar_offset);
    uint64_t *empty_bar = full_bar + a.stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty_bar + a.stages);

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer warp: bulk copies of K and V spans ----------------
        const uint64_t policy = l2_evict_first_policy();
        const size_t pos_stride = static_cast<size_t>(a.H) * D;  // halves between positions
        const size_t seq_base = (static_cast<size_t>(b) * a.S * a.H + h0) * D;
        const __half *Kb = reinterpret_cast<const __half *>(a.K) + seq_base;
        const __half *Vb = reinterpret_cast<const __half *>(a.V) + seq_base;
        const uint32_t row_bytes = static_cast<uint32_t>(hg) * D * 2;
        const bool contiguous = (hg == a.H);
        int issued = 0;
        for (int st = 0; st < n_stages; ++st) {
            const int slot = st % a.stages;
            int go = 1;
            if (lane == 0) {
                if (st >= a.stages &&
                    !wait_bounded(&empty_bar[slot], ((st / a.stages) - 1) & 1)) {
                    atomicOr(a.err, kErrProducerWait);
                    *abort_flag = 1;
                    go = 0;
                }
                if (*abort_flag) go = 0;
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            if (!go) break;
            const int p0 = p_begin + st * a.stage_pos;
            const int np = min(a.stage_pos, p_end - p0);
            __half *dK = ring + static_cast<size_t>(slot) * 2 * buf_elems;
            __half *dV = dK + buf_elems;
            const __half *sK = Kb + static_cast<size_t>(p0) * pos_stride;
            const __half *sV = Vb + static_cast<size_t>(p0) * pos_stride;
            if (lane == 0) mbar_arrive_expect_tx(&full_bar[slot], 2u * np * row_bytes);
            __syncwarp();
            if (contiguous) {
                if (lane == 0) {
                    bulk_g2s(dK, sK, np * row_bytes, &full_bar[slot], policy);
                    bulk_g2s(dV, sV, np * row_bytes, &full_bar[slot], policy);
                }
            } else {
                for (int j = lane; j < np; j += 32) {
                    bulk_g2s(dK + static_cast<size_t>(j) * hg * D, sK + j * pos_stride,
                             row_bytes, &full_bar[slot], policy);
                    bulk_g2s(dV + static_cast<size_t>(j) * hg * D, sV + j * pos_stride,
                             row_bytes, &full_bar[slot], policy);
                }
            }
            ++issued;
        }
        // Drain: no copy may still be landing in shared memory when the CTA exits.
        if (lane == 0) {
            for (int st = max(0, issued - a.stages); st < issued; ++st) {
                if (!wait_bounded(&full_bar[st % a.stages], (st / a.stages) & 1))
                    atomicOr(a.err, kErrDrainWait);
            }
        }
        return;
    }

    // ---------------- consumer warps ----------------
    const int lig = lane % BDX;              // lane within its group
    const int lg = warp * BDY + lane / BDX;  // lane group id in the CTA
    const bool lane_on = lig * 8 < D;        // head_dim may not fill the group
    const __half *Qb =
        reinterpret_cast<const __half *>(a.Q) + (static_cast<size_t>(b) * a.H + h0) * D;

    int hl[KMAX], ph[KMAX];
    bool sv[KMAX];
    float q[KMAX][8], acc[KMAX][8], m[KMAX], l[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        const int s = lg + k * NLG;  // slot = phase * heads_per_cta + head
        ph[k] = s / a.heads_per_cta;
        hl[k] = s - ph[k] * a.heads_per_cta;
        sv[k] = ph[k] < a.phases && hl[k] < hg;
        m[k] = -INFINITY;
        l[k] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            acc[k][i] = 0.f;
            q[k][i] = 0.f;
        }
        if (sv[k] && lane_on) {
            float f[8];
            unpack8(ldg_nc_v4(Qb + static_cast<size_t>(hl[k]) * D + lig * 8), f);
#pragma unroll
            for (int i = 0; i < 8; ++i) q[k][i] = f[i] * a.qscale;
        }
    }

    const int iters = a.stage_pos / a.phases;
    for (int st = 0; st < n_stages; ++st) {
        const int slot = st % a.stages;
        if (!wait_bounded(&full_bar[slot], (st / a.stages) & 1)) {
            if (lane == 0) atomicOr(a.err, kErrConsumerWait);
            *abort_flag = 1;
            break;
        }
        const int np = min(a.stage_pos, n_pos - st * a.stage_pos);
        const __half *sK = ring + static_cast<size_t>(slot) * 2 * buf_elems;
        const __half *sV = sK + buf_elems;
        for (int t = 0; t < iters; ++t) {
            float s[KMAX];
            uint4 vr[KMAX];
            bool valid[KMAX];
#pragma unroll
            for (int k = 0; k < KMAX; ++k) {
                const int j = ph[k] + t * a.phases;
                valid[k] = sv[k] && j < np;
                s[k] = 0.f;
                vr[k] = make_uint4(0u, 0u, 0u, 0u);
                if (valid[k] && lane_on) {
                    const size_t off = (static_cast<size_t>(j) * hg + hl[k]) * D + lig * 8;
                    const uint4 kr = *reinterpret_cast<const uint4 *>(sK + off);
                    vr[k] = *reinterpret_cast<const uint4 *>(sV + off);
                    float f[8];
                    unpack8(kr, f);
                    float d0 = 0.f, d1 = 0.f;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        d0 = fmaf(q[k][2 * i], f[2 * i], d0);
                        d1 = fmaf(q[k][2 * i + 1], f[2 * i + 1], d1);
                    }
                    s[k] = d0 + d1;
                }
            }
#pragma unroll
            for (int off = BDX / 2; off > 0; off >>= 1) {
#pragma unroll
                for (int k = 0; k < KMAX; ++k) s[k] += __shfl_xor_sync(0xffffffffu, s[k], off);
            }
#pragma unroll
            for (int k = 0; k < KMAX; ++k) {
                if (valid[k]) {
                    const float mn = fmaxf(m[k], s[k]);
                    const float alpha = exp2f(m[k] - mn);
                    const float p = exp2f(s[k] - mn);
                    m[k] = mn;
                    l[k] = fmaf(l[k], alpha, p);
                    float f[8];
                    unpack8(vr[k], f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[k][i] = fmaf(acc[k][i], alpha, p * f[i]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }

    // ---------------- epilogue: merge phases, write output or partial ----------------
    constexpr uint32_t kConsumerThreads = kConsumerWarps * 32;
    named_barrier_sync(1, kConsumerThreads);  // every consumer is done with the ring
    if (*abort_flag) return;
    float *mbuf = reinterpret_cast<float *>(smem);
    const int rec = D + 2;  // per slot: m, l, acc[D]
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        if (sv[k]) {
            float *r = mbuf + static_cast<size_t>(lg + k * NLG) * rec;
            if (lig == 0) {
                r[0] = m[k];
                r[1] = l[k];
            }
            if (lane_on) {
#pragma unroll
                for (int i = 0; i < 8; ++i) r[2 + lig * 8 + i] = acc[k][i];
            }
        }
    }
    named_barrier_sync(1, kConsumerThreads);

    for (int idx = threadIdx.x; idx < hg * D; idx += kConsumerThreads) {
        const int h = idx / D;
        const int d = idx - h * D;
        float M = -INFINITY;
        for (int f = 0; f < a.phases; ++f) {
            const float *r = mbuf + static_cast<size_t>(f * a.heads_per_cta + h) * rec;
            if (r[1] > 0.f) M = fmaxf(M, r[0]);
        }
        float lsum = 0.f, num = 0.f;
        for (int f = 0; f < a.phases; ++f) {
            const float *r = mbuf + static_cast<size_t>(f * a.heads_per_cta + h) * rec;
            if (r[1] > 0.f) {
                const float w = exp2f(r[0] - M);
                lsum = fmaf(w, r[1], lsum);
                num = fmaf(w, r[2 + d], num);
            }
        }
        const size_t bh = static_cast<size_t>(b) * a.H + h0 + h;
        if (only_split) {
            reinterpret_cast<__half *>(a.out)[bh * D + d] = __float2half_rn(num / lsum);
        } else {
            const size_t sidx = bh * a.num_splits + split;
            a.ws_acc[sidx * D + d] = num;
            if (d == 0) a.ws_ml[sidx] = make_float2(M, lsum);
        }
    }
}

template <int BDX>
const void *pick_kmax(int kmax) {
    switch (kmax) {
        case 1: return reinterpret_cast<const void *>(decode_splitk_kernel<BDX, 1>);
        case 2: return reinterpret_cast<const void *>(decode_splitk_kernel<BDX, 2>);
        case 3: return reinterpret_cast<const void *>(decode_splitk_kernel<BDX, 3>);
        case 4: return reinterpret_cast<const void *>(decode_splitk_kernel<BDX, 4>);
        default: return nullptr;
    }
}

const void *variant_fn(DecodeVariant v) {
    switch (v.bdx) {
        case 1: return pick_kmax<1>(v.kmax);
        case 2: return pick_kmax<2>(v.kmax);
        case 4: return pick_kmax<4>(v.kmax);
        case 8: return pick_kmax<8>(v.kmax);
        case 16: return pick_kmax<16>(v.kmax);
        case 32: return pick_kmax<32>(v.kmax);
        default: return nullptr;
    }
}

}  // namespace

cudaError_t launch_decode_splitk(const DecodeArgs &a, DecodeVariant v, long long ctas, int smem,
                                 cudaStream_t stream) {
    const void *fn = variant_fn(v);
    if (fn == nullptr || ctas <= 0 || ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    void *args[] = {const_cast<DecodeArgs *>(&a)};
    return cudaLaunchKernel(fn, dim3(static_cast<unsigned>(ctas)), dim3(kDecodeThreads), args,
                            static_cast<size_t>(smem), stream);
}

cudaError_t decode_occupancy(DecodeVariant v, int smem, int *ctas_per_sm) {
    const void *fn = variant_fn(v);
    if (fn == nullptr) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, fn, kDecodeThreads,
                                                         static_cast<size_t>(smem));
}

cudaError_t decode_configure_smem(int max_smem) {
    static const int bdxs[] = {1, 2, 4, 8, 16, 32};
    for (int bdx : bdxs) {
        for (int kmax = 1; kmax <= 4; ++kmax) {
            const cudaError_t e = cudaFuncSetAttribute(
                variant_fn({bdx, kmax}), cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

cudaError_t device_error_word(unsigned **ptr) {
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_device_error);
}

}  // namespace dattn
