// softmax.cu -- standalone row softmax over the last dimension (f32), the
// fm_softmax operation of Foundry's docs/metal.md ("Custom Compute Kernels",
// softmax_row: one threadgroup per row), re-done for sm_103a:
//   out[r, c] = exp(x[r, c] - max_c x[r, c]) / sum_c exp(x[r, c] - max_c x[r, c]).
// It is the max-subtracted softmax of the decode path (running max, sum of
// exponentials) exposed on its own.  HBM-bound: 8 bytes per element when a row
// stays on chip, 12 when it is read twice.
//
//   short rows (cols <= 1024): one warp per row, the row kept in registers
//     (32 values per lane), warp-shuffle max and sum: one read, one write;
//   rows up to 16384: one CTA of 256 or 512 threads per row, the row kept in
//     registers (up to 32 values per thread), block max and sum through
//     shared memory: one read, one write;
//   longer rows up to 256 KB (cols % 4 == 0, 16-byte aligned): one or two
//     persistent CTAs per SM walk the rows; the first pass loads a row with an
//     evict-last L2 policy and computes the running (max, sum) with exp2, the
//     second re-reads it from L2 and writes the output with streaming stores;
//   aligned rows above 256 KB: a thread-block cluster per row holds the row
//     in its CTAs' shared memory (bulk copies), merges the slices' (max, sum)
//     through distributed shared memory and writes the output: one read, one
//     write (rows too long for any cluster take the L2 path);
//   otherwise: one CTA per row, a pass computing the running (max, sum) per
//     thread merged across the block, then a pass writing the output.
#include <cuda_runtime.h>

#include <cmath>
#include <algorithm>
#include <map>
#include <mutex>
#include <utility>

#include "dattn_internal.h"
#include "ptx.cuh"

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

constexpr int kRegRowMax = 32 * kRowThreads;  // columns a CTA holds in registers

// max (IS_MAX) or sum of one value per thread over the CTA; every thread gets it
template <bool IS_MAX, int NT = kRowThreads>
__device__ __forceinline__ float block_all_reduce(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float u = __shfl_xor_sync(0xffffffffu, v, o);
        v = IS_MAX ? fmaxf(v, u) : v + u;
    }
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    v = red[0];
#pragma unroll
    for (int w = 1; w < NT / 32; ++w) v = IS_MAX ? fmaxf(v, red[w]) : v + red[w];
    return v;
}

// One CTA of NT threads per row, the row in registers: NV slots per thread, a
// slot being a float4 (VEC, cols % 4 == 0) or a float.  Slot k of thread t
// covers element (or float4) t + k * NT, so each load instruction is coalesced.
// Padding is -infinity, which exponentiates to 0.  A NaN anywhere, or a row
// of -infinity only (max - max = NaN), propagates through the sum to the
// whole row, as the definition does.
template <int NV, bool VEC, int NT = kRowThreads>
__global__ void __launch_bounds__(NT) softmax_reg_rows(const float *__restrict__ x,
                                                       float *__restrict__ out, int cols) {
    __shared__ float red_m[NT / 32], red_l[NT / 32];
    constexpr int W = VEC ? 4 : 1;
    const long long r = blockIdx.x;
    const int n = VEC ? cols / 4 : cols;
    float v[NV][W];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = threadIdx.x + k * NT;
        if constexpr (VEC) {
            float4 t = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            if (c < n) t = __ldcs(reinterpret_cast<const float4 *>(x + r * cols) + c);
            v[k][0] = t.x;
            v[k][1] = t.y;
            v[k][2] = t.z;
            v[k][3] = t.w;
        } else {
            v[k][0] = c < n ? __ldcs(x + r * cols + c) : -INFINITY;
        }
    }
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int e = 0; e < W; ++e) m = fmaxf(m, v[k][e]);
    m = block_all_reduce<true, NT>(m, red_m);
    float l = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int e = 0; e < W; ++e) {
            v[k][e] = expf(v[k][e] - m);
            l += v[k][e];
        }
    l = block_all_reduce<false, NT>(l, red_l);
    const float inv = 1.f / l;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = threadIdx.x + k * NT;
        if (c < n) {
            if constexpr (VEC)
                __stcs(reinterpret_cast<float4 *>(out + r * cols) + c,
                       make_float4(v[k][0] * inv, v[k][1] * inv, v[k][2] * inv, v[k][3] * inv));
            else
                __stcs(out + r * cols + c, v[k][0] * inv);
        }
    }
}

// ---- long rows, persistent: one CTA per SM walks the rows, and the second
// pass finds the row in L2 ----
constexpr int kL2Threads = 1024;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// merge() for states whose sums are 2^(x log2(e) - S(m)), S(m) = m log2(e)
__device__ __forceinline__ void merge2(float &m, float &l, float m2, float l2) {
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) return;
    const float sM = __fmul_rn(M, kLog2e);
    l = l * ex2(__fmul_rn(m, kLog2e) - sM) + l2 * ex2(__fmul_rn(m2, kLog2e) - sM);
    m = M;
}

// A row is read twice, but by at most one CTA per SM at a time, so the rows in
// flight (SMs x row bytes) stay within L2: the first pass loads with an
// evict-last policy and computes the running (max, sum of exp); the second
// pass re-reads the row (evict-first), normalises and writes with streaming
// stores.  One HBM read and one write per element when the rows in flight fit
// L2.
template <int NT>
__global__ void __launch_bounds__(NT, kL2Threads / NT) softmax_l2_rows(const float *__restrict__ x,
                                                                        float *__restrict__ out,
                                                                        long long rows, int cols) {
    __shared__ float sm_m[NT / 32], sm_l[NT / 32];
    __shared__ int sm_nan[NT / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n4 = cols / 4;
    // float4 loads in flight per thread: 6 fit the 512-thread instance's 64
    // registers; the 1024-thread one spills beyond 4
    constexpr int U = NT <= 512 ? 6 : 4;
    const uint64_t keep = l2_evict_last_policy();
    const uint64_t drop = l2_evict_first_policy();
    for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
        const float4 *x4 = reinterpret_cast<const float4 *>(x + r * cols);
        float m = -INFINITY, l = 0.f;
        bool nan = false;
        for (int c = tid; c < n4; c += NT * U) {
            float4 t[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int ck = c + k * NT;
                t[k] = ck < n4 ? ld_f4_hint(x4 + ck, keep)
                               : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                // m is kept in x units and S(m) = m log2(e) rounded once; a term is
                // 2^(x log2(e) - S(m)) with the difference formed by one fused
                // multiply-add, so S(m)'s rounding is common to every term and
                // cancels in the normalisation.  Rescale only when m rises.
                nan |= isnan(t[k].x) || isnan(t[k].y) || isnan(t[k].z) || isnan(t[k].w);
                const float M = fmaxf(m, fmaxf(fmaxf(t[k].x, t[k].y), fmaxf(t[k].z, t[k].w)));
                if (M != -INFINITY) {
                    const float sM = __fmul_rn(M, kLog2e);
                    if (M > m) {
                        l *= ex2(__fmul_rn(m, kLog2e) - sM);  // 0 while m is -inf
                        m = M;
                    }
                    l += ex2(fmaf(t[k].x, kLog2e, -sM)) + ex2(fmaf(t[k].y, kLog2e, -sM)) +
                         ex2(fmaf(t[k].z, kLog2e, -sM)) + ex2(fmaf(t[k].w, kLog2e, -sM));
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
            merge2(m, l, m2, l2);
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
        for (int w = 1; w < NT / 32; ++w) {
            merge2(m, l, sm_m[w], sm_l[w]);
            row_nan |= sm_nan[w] != 0;
        }
        __syncthreads();  // the shared states are read before the next row writes them
        // a NaN anywhere, or a row of -infinity only, gives a NaN row
        if (row_nan) l = NAN;
        const float inv = 1.f / l;
        const float sm = __fmul_rn(m, kLog2e);
        float4 *o4 = reinterpret_cast<float4 *>(out + r * cols);
        for (int c = tid; c < n4; c += NT * U) {
            float4 t[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int ck = c + k * NT;
                if (ck < n4) t[k] = ld_f4_hint(x4 + ck, drop);
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int ck = c + k * NT;
                if (ck < n4)
                    __stcs(o4 + ck, make_float4(ex2(fmaf(t[k].x, kLog2e, -sm)) * inv,
                                                ex2(fmaf(t[k].y, kLog2e, -sm)) * inv,
                                                ex2(fmaf(t[k].z, kLog2e, -sm)) * inv,
                                                ex2(fmaf(t[k].w, kLog2e, -sm)) * inv));
            }
        }
    }
}

// Rows too long for the persistent CTAs to keep in L2 between their two passes
// (above 256 KB a row, 152 rows in flight overflow L2 and part of the second
// pass comes from HBM again): a thread-block cluster of C CTAs per row, each
// CTA holding its slice of the row in shared memory.  The slice is loaded by
// bulk asynchronous copies (TMA engine) into one of `nbuf` buffers, so later
// rows' slices can land while this one is finished (with one buffer, the
// other CTA on the SM does that).  Pass one computes the
// slice's (max, sum of exp2); the C states are merged through distributed
// shared memory behind one cluster barrier per row; pass two reads the slice
// from shared memory and writes the output with streaming stores.  One HBM
// read and one write per element, whatever the number of rows in flight.
// Clusters walk the rows persistently (cluster q takes rows q, q + nq, ...).
template <int NT, int MINB>
__global__ void __launch_bounds__(NT, MINB) softmax_cluster_rows(const float *__restrict__ x,
                                                                 float *__restrict__ out,
                                                                 long long rows, int cols,
                                                                 int slice_cap, int nbuf,
                                                                 unsigned *err) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float sm_m[NT / 32], sm_l[NT / 32];
    __shared__ int sm_nan[NT / 32];
    __shared__ float s_M, s_L;
    __shared__ float2 s_xch[2];  // this CTA's (max, sum) of the rows of each parity
    __shared__ alignas(8) uint64_t s_bar[4];
    float4 *const buf = reinterpret_cast<float4 *>(smem);  // [nbuf][slice_cap], nbuf <= 4
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned C = cluster_nctarank();
    const unsigned rank = cluster_ctarank();
    const long long q = blockIdx.x / C, nq = gridDim.x / C;
    const int n4 = cols / 4;
    const int f0 = static_cast<int>(static_cast<long long>(rank) * n4 / C);
    const int nf = static_cast<int>(static_cast<long long>(rank + 1) * n4 / C) - f0;  // <= slice_cap
    if (tid == 0) {
        for (int k = 0; k < nbuf; ++k) mbar_init(&s_bar[k], 1);
        fence_barrier_init();
    }
    __syncthreads();
    const uint64_t once = l2_evict_first_policy();
    // thread 0: copy this CTA's slice of `row` into buffer b (16-byte aligned:
    // cols % 4 == 0 and x is 16-byte aligned)
    auto issue = [&](long long row, int b) {
        const char *src = reinterpret_cast<const char *>(x + row * cols) + static_cast<size_t>(f0) * 16;
        char *dst = reinterpret_cast<char *>(buf + static_cast<size_t>(b) * slice_cap);
        const uint32_t bytes = static_cast<uint32_t>(nf) * 16u;
        mbar_arrive_expect_tx(&s_bar[b], bytes);
        for (uint32_t o = 0; o < bytes; o += 32768u)
            bulk_g2s(dst + o, src + o, bytes - o < 32768u ? bytes - o : 32768u, &s_bar[b], once);
    };
    bool ok = true;  // false once a wait ran out: no more copies are issued
    // this CTA's rows in order: row q + it * nq goes to buffer it % nbuf, as
    // that buffer's (it / nbuf)-th fill
    int issued = 0, waited = 0;
    for (int k = 0; k < nbuf && q + k * nq < rows; ++k) {
        if (tid == 0) issue(q + k * nq, k);
        ++issued;
    }
    int it = 0;
    for (long long row = q; row < rows; row += nq, ++it) {
        const int b = it % nbuf;
        const int xs = it & 1;  // exchange slot: rows alternate
        const float4 *s4 = buf + static_cast<size_t>(b) * slice_cap;
        if (ok) {
            const bool done = mbar_wait_bounded(&s_bar[b], (it / nbuf) & 1, kWaitLimitNs);
            if (!__syncthreads_and(done)) {
                if (tid == 0) atomicOr(err, kErrConsumerWait);
                ok = false;
            } else {
                ++waited;
            }
        }
        // pass one: this slice's running (max, sum of 2^(x log2 e - S(max)))
        float m = -INFINITY, l = 0.f;
        bool nan = false;
        for (int i = tid; i < nf; i += NT) {
            const float4 t = s4[i];
            nan |= isnan(t.x) || isnan(t.y) || isnan(t.z) || isnan(t.w);
            const float M = fmaxf(m, fmaxf(fmaxf(t.x, t.y), fmaxf(t.z, t.w)));
            if (M != -INFINITY) {
                const float sM = __fmul_rn(M, kLog2e);
                if (M > m) {
                    l *= ex2(__fmul_rn(m, kLog2e) - sM);  // 0 while m is -inf
                    m = M;
                }
                l += ex2(fmaf(t.x, kLog2e, -sM)) + ex2(fmaf(t.y, kLog2e, -sM)) +
                     ex2(fmaf(t.z, kLog2e, -sM)) + ex2(fmaf(t.w, kLog2e, -sM));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
            merge2(m, l, m2, l2);
        }
        const bool warp_nan = __any_sync(0xffffffffu, nan);
        if (lane == 0) {
            sm_m[warp] = m;
            sm_l[warp] = l;
            sm_nan[warp] = warp_nan;
        }
        __syncthreads();
        if (tid == 0) {
            float M = sm_m[0], L = sm_l[0];
            bool any_nan = sm_nan[0] != 0;
            for (int w = 1; w < NT / 32; ++w) {
                merge2(M, L, sm_m[w], sm_l[w]);
                any_nan |= sm_nan[w] != 0;
            }
            s_xch[xs] = make_float2(M, any_nan ? NAN : L);  // a NaN sum marks a NaN
        }
        // every CTA's state of this row is visible to the cluster after this
        cluster_sync_all();
        if (warp == 0) {
            float2 v = make_float2(-INFINITY, 0.f);
            if (lane < static_cast<int>(C)) v = ld_shared_cluster_f2(cluster_map_shared(smem_addr(&s_xch[xs]), lane));
            const bool row_nan = __any_sync(0xffffffffu, isnan(v.y));
            float M = v.x, L = isnan(v.y) ? 0.f : v.y;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, M, o);
                const float l2 = __shfl_xor_sync(0xffffffffu, L, o);
                merge2(M, L, m2, l2);
            }
            if (lane == 0) {
                s_M = M;
                s_L = row_nan ? NAN : L;  // a NaN anywhere, or only -inf (0 / 0), gives a NaN row
            }
        }
        __syncthreads();
        const float inv = 1.f / s_L;
        const float sm = __fmul_rn(s_M, kLog2e);
        float4 *o4 = reinterpret_cast<float4 *>(out + row * cols) + f0;
        for (int i = tid; i < nf; i += NT) {
            const float4 t = s4[i];
            __stcs(o4 + i, make_float4(ex2(fmaf(t.x, kLog2e, -sm)) * inv,
                                       ex2(fmaf(t.y, kLog2e, -sm)) * inv,
                                       ex2(fmaf(t.z, kLog2e, -sm)) * inv,
                                       ex2(fmaf(t.w, kLog2e, -sm)) * inv));
        }
        __syncthreads();  // every thread is done with buffer b
        if (ok && row + static_cast<long long>(nbuf) * nq < rows) {
            if (tid == 0) issue(row + static_cast<long long>(nbuf) * nq, b);
            ++issued;
        }
    }
    // no copy may still be landing when the CTA exits (only after a wait ran out)
    if (tid == 0) {
        for (int k = waited; k < issued; ++k)
            if (!mbar_wait_bounded(&s_bar[k % nbuf], (k / nbuf) & 1, kWaitLimitNs)) atomicOr(err, kErrDrainWait);
    }
    // no CTA leaves while another may still read its (max, sum)
    cluster_sync_all();
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

#ifndef DATTN_SOFTMAX_CLUSTER_MIN_COLS
#define DATTN_SOFTMAX_CLUSTER_MIN_COLS (64 * 1024 + 1)  // rows above 256 KB
#endif
// Measured at 128256 and 262144 columns: one slice buffer per CTA and two
// CTAs per SM (the other CTA's row hides each load) beat two or more buffers
// with one, three or four CTAs per SM.
#ifndef DATTN_SOFTMAX_CLUSTER_BUFFERS
#define DATTN_SOFTMAX_CLUSTER_BUFFERS 1  // slices in flight per CTA (1 to 4)
#endif
#ifndef DATTN_SOFTMAX_CLUSTER_CTAS_PER_SM
#define DATTN_SOFTMAX_CLUSTER_CTAS_PER_SM 2  // 1: 512 threads per CTA; more: 256
#endif
constexpr int kClusterRowThreads = DATTN_SOFTMAX_CLUSTER_CTAS_PER_SM == 1 ? 512 : 256;
constexpr int kClusterRowMinBlocks = DATTN_SOFTMAX_CLUSTER_CTAS_PER_SM;
constexpr int kClusterRowBuffers = DATTN_SOFTMAX_CLUSTER_BUFFERS;
static_assert(kClusterRowBuffers >= 1 && kClusterRowBuffers <= 4, "1 to 4 slice buffers");

// Launch configuration of softmax_cluster_rows for a row length: the smallest
// cluster whose slices, double-buffered, fit the shared memory of one CTA, and
// as many clusters as are resident at once (cached per device and length).
struct ClusterRowsConfig {
    int cluster = 0, slice_cap = 0, clusters = 0;
    size_t smem = 0;
};

cudaError_t cluster_rows_config(int cols, ClusterRowsConfig *cfg_out) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, ClusterRowsConfig> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({dev, cols});
    if (it != cache.end()) {
        *cfg_out = it->second;
        return cudaSuccess;
    }
    int max_smem = 0;
    e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    const void *fn = reinterpret_cast<const void *>(softmax_cluster_rows<kClusterRowThreads, kClusterRowMinBlocks>);
    cudaFuncAttributes attr{};
    e = cudaFuncGetAttributes(&attr, fn);
    if (e != cudaSuccess) return e;
    const int dyn_max = max_smem - static_cast<int>(attr.sharedSizeBytes);
    // shared memory per CTA when kClusterRowMinBlocks CTAs share an SM
    const int per_sm = (max_smem + 1024) / kClusterRowMinBlocks - 1024 -
                       static_cast<int>(attr.sharedSizeBytes);
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn_max);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    ClusterRowsConfig best;
    const int n4 = cols / 4;
    for (int c = 2; c <= 16; ++c) {
        const int cap = (n4 + c - 1) / c;
        const size_t smem = static_cast<size_t>(cap) * 16 * kClusterRowBuffers;
        if (smem > static_cast<size_t>(std::min(dyn_max, per_sm))) continue;
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(static_cast<unsigned>(c));
        lc.blockDim = dim3(kClusterRowThreads);
        lc.dynamicSmemBytes = smem;
        cudaLaunchAttribute la[1];
        la[0].id = cudaLaunchAttributeClusterDimension;
        la[0].val.clusterDim.x = static_cast<unsigned>(c);
        la[0].val.clusterDim.y = 1;
        la[0].val.clusterDim.z = 1;
        lc.attrs = la;
        lc.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, fn, &lc) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (n < 1) continue;
        best.cluster = c;
        best.slice_cap = cap;
        best.clusters = n;
        best.smem = smem;
        break;  // the smallest cluster that fits
    }
    cache[{dev, cols}] = best;
    *cfg_out = best;
    return cudaSuccess;
}

cudaError_t launch_softmax(const float *x, float *out, long long rows, int cols,
                           unsigned *err, cudaStream_t stream) {
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
#ifndef DATTN_SOFTMAX_REG_MAX
#define DATTN_SOFTMAX_REG_MAX (2 * kRegRowMax)  // widest row held in registers (<= 32768)
#endif
    if (vec4 && cols > kRegRowMax && cols <= DATTN_SOFTMAX_REG_MAX) {
        // 512 or 1024 threads of 8 float4 each: the row still in registers
        void *args[] = {&x, &out, &cols};
        const void *fn = cols <= 2 * kRegRowMax
                             ? reinterpret_cast<const void *>(softmax_reg_rows<8, true, 512>)
                             : reinterpret_cast<const void *>(softmax_reg_rows<8, true, 1024>);
        return cudaLaunchKernel(fn, dim3(static_cast<unsigned>(rows)),
                                dim3(cols <= 2 * kRegRowMax ? 512 : 1024), args, 0, stream);
    }
    if (cols <= kRegRowMax) {
        // smallest register footprint that holds the row
        const int per_thread = (cols + kRowThreads - 1) / kRowThreads;  // 5 .. 32 floats
        const void *fn;
        if (vec4) {
            fn = per_thread <= 8    ? reinterpret_cast<const void *>(softmax_reg_rows<2, true>)
                 : per_thread <= 16 ? reinterpret_cast<const void *>(softmax_reg_rows<4, true>)
                                    : reinterpret_cast<const void *>(softmax_reg_rows<8, true>);
        } else {
            fn = per_thread <= 8    ? reinterpret_cast<const void *>(softmax_reg_rows<8, false>)
                 : per_thread <= 16 ? reinterpret_cast<const void *>(softmax_reg_rows<16, false>)
                                    : reinterpret_cast<const void *>(softmax_reg_rows<32, false>);
        }
        void *args[] = {&x, &out, &cols};
        return cudaLaunchKernel(fn, dim3(static_cast<unsigned>(rows)), dim3(kRowThreads), args, 0,
                                stream);
    }
    if (vec4 && cols >= DATTN_SOFTMAX_CLUSTER_MIN_COLS) {
        // rows above 256 KB: a cluster per row, the row held in shared memory
        ClusterRowsConfig cc;
        cudaError_t e = cluster_rows_config(cols, &cc);
        if (e != cudaSuccess) return e;
        if (cc.cluster > 0) {
            const long long clusters = rows < cc.clusters ? rows : cc.clusters;
            cudaLaunchConfig_t lc = {};
            lc.gridDim = dim3(static_cast<unsigned>(clusters * cc.cluster));
            lc.blockDim = dim3(kClusterRowThreads);
            lc.dynamicSmemBytes = cc.smem;
            lc.stream = stream;
            cudaLaunchAttribute la[1];
            la[0].id = cudaLaunchAttributeClusterDimension;
            la[0].val.clusterDim.x = static_cast<unsigned>(cc.cluster);
            la[0].val.clusterDim.y = 1;
            la[0].val.clusterDim.z = 1;
            lc.attrs = la;
            lc.numAttrs = 1;
            return cudaLaunchKernelEx(&lc, softmax_cluster_rows<kClusterRowThreads, kClusterRowMinBlocks>,
                                      x, out, rows, cols, cc.slice_cap, kClusterRowBuffers, err);
        }
    }
    if (vec4) {
        // long aligned rows: one or two persistent CTAs per SM walk the rows
        int sms = 0, dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        // two CTAs of 512 threads per SM while two rows per SM still fit L2,
        // else one of 1024
        const bool two = static_cast<long long>(cols) * 4 <= 256 * 1024;
        const long long slots = static_cast<long long>(sms) * (two ? 2 : 1);
        const long long grid = rows < slots ? rows : slots;
        void *args[] = {&x, &out, &rows, &cols};
        return cudaLaunchKernel(two ? reinterpret_cast<const void *>(softmax_l2_rows<512>)
                                    : reinterpret_cast<const void *>(softmax_l2_rows<1024>),
                                dim3(static_cast<unsigned>(grid)), dim3(two ? 512 : 1024), args,
                                0, stream);
    }
    void *args[] = {&x, &out, &cols, &vec4};
    return cudaLaunchKernel(reinterpret_cast<const void *>(softmax_block_rows),
                            dim3(static_cast<unsigned>(rows)), dim3(kRowThreads), args, 0, stream);
}

}  // namespace dattn
