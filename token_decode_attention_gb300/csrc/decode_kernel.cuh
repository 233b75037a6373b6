// decode_kernel.cuh -- the fused decode-attention kernel template for sm_103a,
// instantiated for the split plan (dense and paged caches) in decode_streamk.cu
// and for the cluster plan in decode_cluster.cu (dense caches) and
// decode_cluster_paged.cu (paged caches): translation units built in parallel,
// each instance holding only its own mode's code, which keeps the
// latency-bound launches of every mode lean.
// (Separate dense and paged instances of the split plan were measured too:
// the dense one ran long 1.3 % slower, so the split plan keeps one.)
//
// Computes, per sequence b and head h, the masked softmax attention of the
// kernels attention_qk_f16 and attention_pv_f16 of "Developing Apple Metal
// Kernels in Rust - A Deep Dive Through Attention" (section "The MSL, briefly")
// in one pass over the live KV rows, without materialising scores:
//   s_p  = (Q[b,h,:] . K[b,p,h,:]) / sqrt(D)         p < L_b = min(cp_b, S-1)+1
//   out  = sum_p exp(s_p - max s) V[b,p,h,:] / sum_p exp(s_p - max s)
//
// Work split (stream-K, see streamk.h): the live positions of the whole batch,
// flattened over (sequence, head group, position), are cut into G equal
// ranges, one per CTA, and the grid is sized to the resident CTA slots of the
// GPU.  Every CTA streams the same number of bytes whatever the mix of
// sequence lengths, and there is no wave tail.  A range covers one or more
// "pieces" (a run of positions of one unit); a CTA writes the f16 output of a
// unit it covers whole and the partial softmax state (m, l, acc) of the others
// for combine.cu.  Positions past L_b belong to no range: the page's -infinity
// mask is a loop bound and masked rows never enter the computation.
//
// Cluster plan (the cluster instances; one sequence, dense or paged cache):
// the grid is B * NHG thread-block clusters of C CTAs.  Cluster u takes unit u
// whole and CTA r of it the positions [r L_b / C, (r+1) L_b / C) (cut at page
// boundaries for a paged cache); a head group smaller than H is copied as 3D
// tensor boxes {D, HG, P} per stage (a dense cache; a partial stage takes the
// box that ends where the range ends) or {D, HG, page_size} per page (a paged
// cache).  Each CTA leaves its partial state in a shared-memory record, and
// the cluster's CTAs merge the C records through distributed shared memory,
// each finishing an equal share of the unit's outputs: no workspace and no
// second kernel.
//
// Per CTA:
//   * launched with programmatic dependent launch, it initialises its barriers
//     and prefetches the first stages of its likely range into L2 before
//     waiting on the kernel before it;
//   * a producer warp streams, for each piece, stages of P positions: for the
//     layout [B,S,H,D] the K rows of all heads of a run of positions are one
//     contiguous span of HBM, moved by one bulk asynchronous copy
//     (cp.async.bulk on the TMA engine, L2 evict-first) into a multi-stage
//     shared-memory ring completing on mbarriers (V likewise);
//   * eight (or sixteen) consumer warps read each KV row with D/(8*CH) lanes, CH 16-byte
//     shared loads per lane laid out so a lane group reads 128 contiguous
//     bytes per load.  The QK product uses the raw f16 query and f16 keys with
//     fp32 accumulation (products of two halves are exact in fp32); the dot is
//     reduced with xor shuffles and scaled by log2(e)/sqrt(D).  Each lane group
//     keeps an online softmax per (head, phase) slot in fp32 registers: the
//     running max is only raised (and the state rescaled) when a new score
//     exceeds it; PV accumulates with packed fp32x2 FMAs.  Groups of positions
//     that lie wholly inside a stage run a body without per-position tests.
//   * every mbarrier wait is bounded; a wait that runs out records an error in
//     the device error word and the CTA returns after draining its copies.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <type_traits>

#include "dattn_internal.h"
#include "ptx.cuh"
#include "streamk.h"

namespace dattn {
namespace {


constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxCluster = 16;  // CTAs per cluster in cluster mode (non-portable above 8)

__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity) {
    return mbar_wait_bounded(bar, parity, kWaitLimitNs);
}

__device__ __forceinline__ int live_len(const uint32_t *cp, long long b, int S) {
    const uint32_t c = __ldg(cp + b);
    return c >= static_cast<uint32_t>(S - 1) ? S : static_cast<int>(c) + 1;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// d0 += q0*k0 + q2*k2 + q4*k4 + q6*k6 ; d1 += q1*k1 + q3*k3 + q5*k5 + q7*k7
// with f16 inputs and fp32 accumulation (each product is exact in fp32).
__device__ __forceinline__ void dot8(const uint4 q, const uint4 k, float &d0, float &d1) {
    asm("{\n\t.reg .f16 qa, qb, ka, kb;\n\t"
        "mov.b32 {qa, qb}, %2;\n\tmov.b32 {ka, kb}, %6;\n\t"
        "fma.rn.f32.f16 %0, qa, ka, %0;\n\tfma.rn.f32.f16 %1, qb, kb, %1;\n\t"
        "mov.b32 {qa, qb}, %3;\n\tmov.b32 {ka, kb}, %7;\n\t"
        "fma.rn.f32.f16 %0, qa, ka, %0;\n\tfma.rn.f32.f16 %1, qb, kb, %1;\n\t"
        "mov.b32 {qa, qb}, %4;\n\tmov.b32 {ka, kb}, %8;\n\t"
        "fma.rn.f32.f16 %0, qa, ka, %0;\n\tfma.rn.f32.f16 %1, qb, kb, %1;\n\t"
        "mov.b32 {qa, qb}, %5;\n\tmov.b32 {ka, kb}, %9;\n\t"
        "fma.rn.f32.f16 %0, qa, ka, %0;\n\tfma.rn.f32.f16 %1, qb, kb, %1;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "r"(q.x), "r"(q.y), "r"(q.z), "r"(q.w), "r"(k.x), "r"(k.y), "r"(k.z), "r"(k.w));
}

// acc[0..7] += p * v[0..7]: v converted from f16, packed fp32x2 FMAs.
__device__ __forceinline__ void axpy8(float *acc, float p, const uint4 v) {
    asm("{\n\t.reg .f16 va, vb;\n\t.reg .f32 fa, fb;\n\t.reg .b64 x, c, pp;\n\t"
        "mov.b64 pp, {%8, %8};\n\t"
        "mov.b32 {va, vb}, %9;\n\tcvt.f32.f16 fa, va;\n\tcvt.f32.f16 fb, vb;\n\t"
        "mov.b64 x, {fa, fb};\n\tmov.b64 c, {%0, %1};\n\tfma.rn.f32x2 c, x, pp, c;\n\t"
        "mov.b64 {%0, %1}, c;\n\t"
        "mov.b32 {va, vb}, %10;\n\tcvt.f32.f16 fa, va;\n\tcvt.f32.f16 fb, vb;\n\t"
        "mov.b64 x, {fa, fb};\n\tmov.b64 c, {%2, %3};\n\tfma.rn.f32x2 c, x, pp, c;\n\t"
        "mov.b64 {%2, %3}, c;\n\t"
        "mov.b32 {va, vb}, %11;\n\tcvt.f32.f16 fa, va;\n\tcvt.f32.f16 fb, vb;\n\t"
        "mov.b64 x, {fa, fb};\n\tmov.b64 c, {%4, %5};\n\tfma.rn.f32x2 c, x, pp, c;\n\t"
        "mov.b64 {%4, %5}, c;\n\t"
        "mov.b32 {va, vb}, %12;\n\tcvt.f32.f16 fa, va;\n\tcvt.f32.f16 fb, vb;\n\t"
        "mov.b64 x, {fa, fb};\n\tmov.b64 c, {%6, %7};\n\tfma.rn.f32x2 c, x, pp, c;\n\t"
        "mov.b64 {%6, %7}, c;\n\t}"
        : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3]), "+f"(acc[4]), "+f"(acc[5]),
          "+f"(acc[6]), "+f"(acc[7])
        : "f"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

__device__ __forceinline__ uint4 pack8_f16(const float *x, float s) {
    uint4 r;
    __half2 h;
    h = __floats2half2_rn(x[0] * s, x[1] * s);
    r.x = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2half2_rn(x[2] * s, x[3] * s);
    r.y = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2half2_rn(x[4] * s, x[5] * s);
    r.z = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2half2_rn(x[6] * s, x[7] * s);
    r.w = *reinterpret_cast<uint32_t *>(&h);
    return r;
}

// Walks the pieces of one CTA's range in flattened order (identically in the
// producer and the consumers).
struct Walker {
    long long x, x1;   // next flattened position, end of the range
    long long base;    // flattened position where sequence b starts
    long long b;       // current sequence
    int Lb;            // its live length
    // current piece
    int g, off, len;
    long long u;
};

template <bool CLUSTER>
__device__ __forceinline__ bool next_piece(Walker &w, const DecodeArgs &a) {
    if (w.x >= w.x1) return false;
    const long long nhg = a.head_groups;
    // a cluster-plan range lies inside one unit: no later sequence to move to
    while (!CLUSTER && w.x >= w.base + nhg * w.Lb) {
        w.base += nhg * w.Lb;
        ++w.b;
        w.Lb = live_len(a.cur_pos, w.b, a.S);
    }
    // rel < head_groups * seq_len < 2^31 (checked by the host): 32-bit division
    const unsigned rel = static_cast<unsigned>(w.x - w.base);
    w.g = static_cast<int>(rel / static_cast<unsigned>(w.Lb));
    w.off = static_cast<int>(rel - static_cast<unsigned>(w.g) * static_cast<unsigned>(w.Lb));
    const long long rest = w.x1 - w.x;
    w.len = static_cast<int>(rest < w.Lb - w.off ? rest : w.Lb - w.off);
    w.u = w.b * nhg + w.g;
    w.x += w.len;
    return true;
}

// Instance modes: the split plan (dense and paged caches), the cluster plan
// over a dense cache, the cluster plan over a paged cache.  Each instance
// holds only its mode's code: on latency-bound launches the unused code of
// another mode measured up to 1.8 us per call.
constexpr int kModeSplit = 0, kModeCluster = 1, kModeClusterPaged = 2;

template <int BDX, int CH, int KMAX, int NWC, int MODE>
__global__ void __launch_bounds__(decode_threads(NWC), decode_min_blocks(NWC))
    decode_streamk_kernel(const __grid_constant__ DecodeArgs a) {
    constexpr bool CLUSTER = MODE != kModeSplit;
    constexpr bool PAGED_OK = MODE != kModeCluster;  // the dense cluster instances have no paging
    constexpr int NPOS = 2;              // positions per (head, phase) slot in a consumer group
    constexpr int BDY = 32 / BDX;        // lane groups per warp
    constexpr int NLG = NWC * BDY;       // lane groups per CTA
    constexpr int kThreads = decode_threads(NWC);
    constexpr int kWarps = NWC + 1;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ long long s_warp_sum[kWarps];
    __shared__ long long s_b0, s_base0;
    __shared__ int s_L0;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int D = a.D;

    uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + a.bar_offset);
    uint64_t *empty_bar = full_bar + a.stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty_bar + a.stages);

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.stages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], a.active_warps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();  // barrier initialisation visible to every warp
    // Launched with programmatic dependent launch: up to here only shared memory
    // is touched, so this CTA may already be resident while the kernel before it
    // on the stream finishes.  Everything after the wait sees that kernel's writes
    // (current_pos, Q, the cache).
    //
    // Before waiting, the CTA prefetches into L2 the first positions of the
    // range this CTA would own if every sequence were full (the range depends on
    // current_pos, which may not be final yet).  Kernel parameters alone give
    // that range; a prefetch only warms L2, the point of coherence, so the
    // reads after the wait still see the final data.  Exact when the caches are
    // full; elsewhere some of it is read by other CTAs, the rest is wasted
    // bandwidth.  The cluster plan (one sequence) takes the range from
    // current_pos read before the wait instead, as a hint: exact unless the
    // kernel before this one changes current_pos.
    //
    // A paged cache finds its pages through the block table, which the previous
    // kernel may still be writing: the entries read here are only used to pick
    // what to prefetch, each checked to lie inside the page pool, and are read
    // again after the wait for the copies.  A stale entry wastes a prefetch.
    //
    // Thread 0 issues a dense cache's prefetches.  For a paged cache whose
    // window spans several pages the first prefetch_lanes lanes of warp 0 do,
    // one lane per page, so that the block-table reads go out together: one
    // thread reading the entries one after another (a dependent load per page)
    // kept warp 0, and with it the CTA's consumers, ~17 us late on a window of
    // 24 pages.
    const bool paged_pf = PAGED_OK && a.block_table != nullptr;
    if (a.prefetch_positions > 0 && threadIdx.x < (paged_pf ? a.prefetch_lanes : 1)) {
        const long long S = a.S, nhg = a.head_groups;
        // capacity (every sequence full): the host keeps c * Wc in 64 bits
        const long long Wc = static_cast<long long>(a.B) * nhg * S;
        long long x, x_lim;
        if constexpr (CLUSTER) {
            // CTA r of cluster u: the range it will own if current_pos is
            // final already, [r L / C, (r+1) L / C) of unit u.  current_pos is
            // read here as a hint only, through L2 (no L1 line is left behind
            // for the read after the wait).
            const long long u = blockIdx.x / a.cluster;
            const long long r = blockIdx.x - u * a.cluster;
            const uint32_t cph = __ldcg(a.cur_pos + u / nhg);
            const long long Lh = cph >= static_cast<uint32_t>(S - 1) ? S : static_cast<long long>(cph) + 1;
            long long r0 = r * Lh / a.cluster, r1 = (r + 1) * Lh / a.cluster;
            if constexpr (MODE == kModeClusterPaged) {  // whole pages, as below
                const long long pages = (Lh + a.page_size - 1) / a.page_size;
                r0 = r * pages / a.cluster * a.page_size;
                r1 = r + 1 == a.cluster ? Lh : (r + 1) * pages / a.cluster * a.page_size;
            }
            x = u * S + r0;
            x_lim = u * S + r1;
        } else {
            x = static_cast<long long>(blockIdx.x) * Wc / a.partitions;
            x_lim = static_cast<long long>(blockIdx.x + 1) * Wc / a.partitions;
        }
        const long long x_end = min(x + a.prefetch_positions, x_lim);
        const size_t row = static_cast<size_t>(a.H) * a.D;  // halves per position
        // n positions of heads [h0, h0 + hg) from row first_pos of the cache (or pool)
        auto prefetch_run = [&](long long first_pos, long long n, int h0, int hg) {
            const __half *k0 = reinterpret_cast<const __half *>(a.K) + static_cast<size_t>(first_pos) * row;
            const __half *v0 = reinterpret_cast<const __half *>(a.V) + static_cast<size_t>(first_pos) * row;
            if (hg == a.H) {  // all heads: the run is one span
                const uint32_t bytes = static_cast<uint32_t>(n * row * 2);
                bulk_prefetch_l2(k0, bytes);
                bulk_prefetch_l2(v0, bytes);
            } else if (CLUSTER && a.use_tmap) {  // a head group: whole tensor boxes
                for (long long j = 0; j + a.box_pos <= n; j += a.box_pos) {
                    const int row0 = static_cast<int>(first_pos + j);
                    tensor3d_prefetch_l2(&a.tmap_k, 0, h0, row0);
                    tensor3d_prefetch_l2(&a.tmap_v, 0, h0, row0);
                }
            } else {  // a head group: one span per position
                const uint32_t bytes = static_cast<uint32_t>(hg) * a.D * 2;
                for (long long j = 0; j < n; ++j) {
                    const size_t o = static_cast<size_t>(j) * row + static_cast<size_t>(h0) * a.D;
                    bulk_prefetch_l2(k0 + o, bytes);
                    bulk_prefetch_l2(v0 + o, bytes);
                }
            }
        };
        while (x < x_end) {
            const long long u = x / S;  // unit (b, g)
            const long long off = x - u * S;
            const long long b = u / nhg;
            const int h0 = static_cast<int>(u - b * nhg) * a.heads_per_cta;
            const int hg = min(a.heads_per_cta, a.H - h0);
            const long long n = min(S - off, x_end - x);
            if (paged_pf) {
                // the unit's pages overlapping [off, off + n): lane l takes
                // pages p_first + l, + prefetch_lanes, ... (x and n are the same
                // in every lane)
                const long long ps = a.page_size;
                const long long p_first = off / ps, p_end = (off + n - 1) / ps + 1;
                for (long long pidx = p_first + lane; pidx < p_end; pidx += a.prefetch_lanes) {
                    // through L2 only (no L1 line is left behind for the reads after the wait)
                    const long long page = __ldcg(a.block_table + b * a.max_pages + pidx);
                    if (page >= 0 && page < a.num_pages) {
                        const long long lo = max(off, pidx * ps), hi = min(off + n, (pidx + 1) * ps);
                        prefetch_run(page * ps + (lo - pidx * ps), hi - lo, h0, hg);
                    }
                }
            } else {
                prefetch_run(b * S + off, n, h0, hg);  // dense: row index in [B*S]
            }
            x += n;
        }
    }
    pdl_wait_primary();

    // ---- the CTA's range: scan of the live lengths over the batch ----
    // W = head_groups * sum_b L_b flattened positions cut into G ranges; this
    // CTA owns [x0, x1), which starts in sequence b0 (at flattened position
    // base0, live length L0).
    const long long nhg = a.head_groups;
    const unsigned G = static_cast<unsigned>(a.partitions);
    long long W, x0, x1, b0 = 0, base0 = 0;
    int L0 = 0;
    // range_begin_split needs W / G; a 32-bit division when W fits
    auto cut = [&](long long total) {
        W = total * nhg;
        const long long wq = W < 0x100000000LL ? static_cast<long long>(static_cast<unsigned>(W) / G) : W / G;
        const unsigned wr = static_cast<unsigned>(W - wq * G);
        x0 = range_begin_split(blockIdx.x, wq, wr, G);
        x1 = range_begin_split(blockIdx.x + 1, wq, wr, G);
    };
    if constexpr (CLUSTER) {
        // Cluster mode: CTA r of cluster u takes the positions
        // [r L_b / C, (r+1) L_b / C) of unit u = (b, g), numbered from the
        // start of sequence b; no scan over the batch.
        const long long u = blockIdx.x / a.cluster;
        const long long r = blockIdx.x - u * a.cluster;
        b0 = u / nhg;
        L0 = live_len(a.cur_pos, b0, a.S);
        const long long g = u - b0 * nhg;
        long long r0 = r * L0 / a.cluster, r1 = (r + 1) * L0 / a.cluster;
        if constexpr (MODE == kModeClusterPaged) {
            // the unit's pages dealt out evenly (a CTA takes the floor or the
            // ceiling of pages / C), so every range starts on a page, and every
            // stage is whole pages (one tensor box each) but for the unit's last
            const long long pages = (L0 + a.page_size - 1) / a.page_size;
            r0 = r * pages / a.cluster * a.page_size;
            r1 = r + 1 == a.cluster ? L0 : (r + 1) * pages / a.cluster * a.page_size;
        }
        x0 = g * L0 + r0;
        x1 = g * L0 + r1;
        base0 = 0;
    } else if (a.B <= 32) {
        // Lane b holds sequence b: every warp scans the batch on its own, with
        // no shared memory and no CTA barrier.
        const long long Lb = lane < a.B ? live_len(a.cur_pos, lane, a.S) : 0;
        long long incl = Lb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        cut(__shfl_sync(kFull, incl, 31));
        // the first sequence whose positions end past x0
        const unsigned past = __ballot_sync(kFull, lane < a.B && x0 < nhg * incl);
        if (past != 0u) {
            const int first = __ffs(past) - 1;
            L0 = static_cast<int>(__shfl_sync(kFull, Lb, first));
            base0 = nhg * (__shfl_sync(kFull, incl, first) - L0);
            b0 = first;
        }
        if (blockIdx.x == 0 && warp == 0 && a.ws_prefix != nullptr) {
            if (lane < a.B) a.ws_prefix[lane] = incl - Lb;
            if (lane == a.B - 1) a.ws_prefix[a.B] = incl;
        }
    } else {
        // block scan: thread t sums sequences [bb, be)
        const long long per = (a.B + kThreads - 1) / kThreads;
        const long long bb = min(static_cast<long long>(threadIdx.x) * per, static_cast<long long>(a.B));
        const long long be = min(bb + per, static_cast<long long>(a.B));
        long long sum = 0;
        for (long long b = bb; b < be; ++b) sum += live_len(a.cur_pos, b, a.S);
        long long incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_warp_sum[warp] = incl;
        __syncthreads();
        long long before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const long long v = s_warp_sum[w];
            if (w < warp) before += v;
            total += v;
        }
        const long long excl = before + incl - sum;
        cut(total);
        if (x0 < x1 && nhg * excl <= x0 && x0 < nhg * (excl + sum)) {
            long long run = excl;
            for (long long b = bb; b < be; ++b) {
                const int L = live_len(a.cur_pos, b, a.S);
                if (x0 < nhg * (run + L)) {
                    s_b0 = b;
                    s_base0 = nhg * run;
                    s_L0 = L;
                    break;
                }
                run += L;
            }
        }
        if (blockIdx.x == 0 && a.ws_prefix != nullptr) {
            long long run = excl;
            for (long long b = bb; b < be; ++b) {
                a.ws_prefix[b] = run;
                run += live_len(a.cur_pos, b, a.S);
            }
            if (threadIdx.x == 0) a.ws_prefix[a.B] = total;
        }
        __syncthreads();
        b0 = s_b0;
        base0 = s_base0;
        L0 = s_L0;
    }
    // The combine kernel may begin launching; it waits for this grid to finish.
    pdl_launch_dependents();

    // Cluster mode.  Each CTA writes its partial state (m, l, acc) per head to
    // a record [HG][D + 2] in its own shared memory (a CTA without positions
    // writes empty ones).  After a cluster barrier the C CTAs share the
    // unit's E = HG x D outputs, CTA r finishing [r E / C, (r+1) E / C): it
    // reads the C records of each output through distributed shared memory
    // (all loads of an output issued together) and merges them.  A second,
    // relaxed barrier keeps every record alive until all reads are done.
    // (Pushing the records into the finishers' shared memory instead, with
    // remote stores and a single barrier, measured slower.)
    float *const lrec = reinterpret_cast<float *>(smem + a.rec_offset);
    // every thread of every CTA of the cluster calls this once, after its record
    auto cluster_tail = [&]() {
        cluster_sync_all();  // every record of the cluster is complete
        const int C = a.cluster;
        const long long u = blockIdx.x / C;
        const int r = static_cast<int>(blockIdx.x - u * C);
        const long long b = u / nhg;
        const int h0 = static_cast<int>(u - b * nhg) * a.heads_per_cta;
        // 32-bit share arithmetic: E = HG * D <= 12288 (the plan keeps a position's
        // K+V rows of a group within 48 KB) and C <= 16
        const int E = a.heads_per_cta * D;
        const int e1 = (r + 1) * E / C;
        const uint32_t rec0 = smem_addr(lrec);
        for (int e = r * E / C + threadIdx.x; e < e1; e += blockDim.x) {
            const int h = e / D;
            const int d = e - h * D;
            const uint32_t hrec = rec0 + static_cast<uint32_t>(h * (D + 2)) * 4u;
            float mj[kMaxCluster], lj[kMaxCluster], nj[kMaxCluster];
#pragma unroll
            for (int j = 0; j < kMaxCluster; ++j) {
                mj[j] = -INFINITY;
                lj[j] = 0.f;
                nj[j] = 0.f;
                if (j < C) {
                    const uint32_t rr = cluster_map_shared(hrec, j);
                    mj[j] = ld_shared_cluster_f32(rr);
                    lj[j] = ld_shared_cluster_f32(rr + 4u);
                    nj[j] = ld_shared_cluster_f32(rr + 8u + 4u * d);
                }
            }
            float M = -INFINITY;
#pragma unroll
            for (int j = 0; j < kMaxCluster; ++j)
                if (lj[j] > 0.f) M = fmaxf(M, mj[j]);
            float L = 0.f, N = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxCluster; ++j) {
                if (lj[j] > 0.f) {  // an empty record holds no acc
                    const float w = fast_exp2(mj[j] - M);
                    L = fmaf(w, lj[j], L);
                    N = fmaf(w, nj[j], N);
                }
            }
            reinterpret_cast<__half *>(a.out)[(static_cast<size_t>(b) * a.H + h0) * D + e] =
                __float2half_rn(N / L);
        }
        // the loads above have returned (their values were used): a relaxed
        // arrive is enough to keep every record alive until then
        cluster_arrive_relaxed();
        cluster_wait();
    };

    if (x0 >= x1) {  // empty range (fewer live positions than CTAs)
        if constexpr (CLUSTER) {  // an empty record for every head
            for (int h = threadIdx.x; h < a.heads_per_cta; h += blockDim.x) {
                lrec[h * (D + 2)] = -INFINITY;
                lrec[h * (D + 2) + 1] = 0.f;
            }
            cluster_tail();
        }
        return;
    }
    // consumer warps whose lane groups hold no (head, phase) slot have nothing to do
    if (warp < NWC && warp >= a.active_warps) {
        if constexpr (CLUSTER) cluster_tail();
        return;
    }

    Walker walk;
    walk.x = x0;
    walk.x1 = x1;
    walk.b = b0;
    walk.base = base0;
    walk.Lb = L0;

    __half *ring = reinterpret_cast<__half *>(smem);
    const size_t buf_elems = static_cast<size_t>(a.stage_pos) * a.heads_per_cta * D;

    if (warp == NWC) {
        // ---------------- producer warp ----------------
        const uint64_t policy = l2_evict_first_policy();
        const size_t pos_stride = static_cast<size_t>(a.H) * D;  // halves between positions
        const bool paged = PAGED_OK && a.block_table != nullptr;
        // tensor boxes need a 128-byte aligned destination; otherwise the
        // per-position copies below serve (same data, more copies)
        const bool tmap_ok = CLUSTER && a.use_tmap && (smem_addr(smem) & 127u) == 0;
        int st = 0, issued = 0;
        bool go = true;
        while (go && next_piece<CLUSTER>(walk, a)) {
            const int h0 = walk.g * a.heads_per_cta;
            const int hg = min(a.heads_per_cta, a.H - h0);
            const size_t seq_base = (static_cast<size_t>(walk.b) * a.S * a.H + h0) * D;
            const __half *Kb = reinterpret_cast<const __half *>(a.K) + seq_base;
            const __half *Vb = reinterpret_cast<const __half *>(a.V) + seq_base;
            const uint32_t row_bytes = static_cast<uint32_t>(hg) * D * 2;
            const bool contiguous = (hg == a.H);
            // paged cache: lane i holds block_table[b][page_first + i]
            const int *bt = paged ? a.block_table + walk.b * a.max_pages : nullptr;
            int page_first = -1, page_lane = 0;
            for (int p = 0; p < walk.len; p += a.stage_pos, ++st) {
                const int slot = st % a.stages;
                int ok = 1;
                if (lane == 0) {
                    if (st >= a.stages &&
                        !wait_bounded(&empty_bar[slot], ((st / a.stages) - 1) & 1)) {
                        atomicOr(a.err, kErrProducerWait);
                        *abort_flag = 1;
                        ok = 0;
                    }
                    if (*abort_flag) ok = 0;
                }
                ok = __shfl_sync(kFull, ok, 0);
                if (!ok) {
                    go = false;
                    break;
                }
                const int np = min(a.stage_pos, walk.len - p);
                const int pos0 = walk.off + p;
                __half *dK = ring + static_cast<size_t>(slot) * 2 * buf_elems;
                __half *dV = dK + buf_elems;
                // rows the stage's copies write: with tensor boxes a partial
                // stage still lands whole boxes (a full stage of a dense cache,
                // whole pages of a paged one)
                int tx_rows = np;
                if (tmap_ok && !contiguous)
                    tx_rows = paged ? (np + a.page_size - 1) / a.page_size * a.page_size : a.stage_pos;
                if (lane == 0) mbar_arrive_expect_tx(&full_bar[slot], 2u * tx_rows * row_bytes);
                __syncwarp();
                if (!paged) {
                    const __half *sK = Kb + static_cast<size_t>(pos0) * pos_stride;
                    const __half *sV = Vb + static_cast<size_t>(pos0) * pos_stride;
                    if (contiguous) {
                        if (lane == 0) {
                            bulk_g2s(dK, sK, np * row_bytes, &full_bar[slot], policy);
                            bulk_g2s(dV, sV, np * row_bytes, &full_bar[slot], policy);
                        }
                    } else if (tmap_ok) {
                        // a stage of the head group: one tensor box each
                        // ({D, HG, P} at row b*S + pos0; the host checked that
                        // B*S fits the 32-bit coordinate).  A partial stage
                        // (the range's last) takes the box that ends where the
                        // range ends: its first P - np rows are rows this CTA
                        // read just before (L2 hits), or the fill value where
                        // the coordinate is negative, and the consumers start
                        // at row P - np.
                        if (lane == 0) {
                            const int row0 = static_cast<int>(walk.b * a.S + pos0 + np - a.stage_pos);
                            tensor3d_g2s(dK, &a.tmap_k, 0, h0, row0, &full_bar[slot], policy);
                            tensor3d_g2s(dV, &a.tmap_v, 0, h0, row0, &full_bar[slot], policy);
                        }
                    } else {
                        for (int j = lane; j < np; j += 32) {
                            bulk_g2s(dK + static_cast<size_t>(j) * hg * D, sK + j * pos_stride,
                                     row_bytes, &full_bar[slot], policy);
                            bulk_g2s(dV + static_cast<size_t>(j) * hg * D, sV + j * pos_stride,
                                     row_bytes, &full_bar[slot], policy);
                        }
                    }
                } else {
                    // paged: lane l takes page pa + l (+ 32, ...) of the stage's
                    // pages pa..pb, so the pages' address arithmetic and copies
                    // go out side by side
                    const int pa = pos0 / a.page_size, pb = (pos0 + np - 1) / a.page_size;
                    for (int q0 = pa; q0 <= pb; q0 += 32) {
                        if (page_first < 0 || q0 < page_first || min(q0 + 31, pb) >= page_first + 32) {
                            page_first = q0;
                            // coherent load: the table may have been written by the
                            // kernel before this one, after the pre-wait prefetch read it
                            page_lane = (q0 + lane < a.max_pages) ? __ldcg(bt + q0 + lane) : 0;
                        }
                        const int qi = q0 + lane;
                        long long page = __shfl_sync(kFull, page_lane, (qi - page_first) & 31);
                        if (qi <= pb) {
                            if (page < 0 || page >= a.num_pages) {  // never read outside the pages
                                atomicOr(a.err, kErrPageIndex);
                                page = 0;
                            }
                            const int lo = max(pos0, qi * a.page_size);
                            const int run = min(pos0 + np, (qi + 1) * a.page_size) - lo;
                            __half *tK = dK + static_cast<size_t>(lo - pos0) * hg * D;
                            __half *tV = dV + static_cast<size_t>(lo - pos0) * hg * D;
                            if (tmap_ok && !contiguous) {
                                // a page of the head group: one tensor box each
                                // ({D, HG, page_size} at row page * page_size of
                                // the pool).  Stages start on a page, so every run
                                // is a page's first rows; the box of the unit's
                                // last, partial page also lands the page's rows
                                // past the live length, which the consumers never
                                // read.
                                const int row0 = static_cast<int>(page * a.page_size);
                                tensor3d_g2s(tK, &a.tmap_k, 0, h0, row0, &full_bar[slot], policy);
                                tensor3d_g2s(tV, &a.tmap_v, 0, h0, row0, &full_bar[slot], policy);
                            } else {
                                const size_t src = (static_cast<size_t>(page) * a.page_size + lo - qi * a.page_size) *
                                                       pos_stride + static_cast<size_t>(h0) * D;
                                const __half *sK = reinterpret_cast<const __half *>(a.K) + src;
                                const __half *sV = reinterpret_cast<const __half *>(a.V) + src;
                                if (contiguous) {  // the run is one span
                                    bulk_g2s(tK, sK, run * row_bytes, &full_bar[slot], policy);
                                    bulk_g2s(tV, sV, run * row_bytes, &full_bar[slot], policy);
                                } else {  // a head group: one copy per position
                                    for (int r = 0; r < run; ++r) {
                                        bulk_g2s(tK + static_cast<size_t>(r) * hg * D, sK + r * pos_stride,
                                                 row_bytes, &full_bar[slot], policy);
                                        bulk_g2s(tV + static_cast<size_t>(r) * hg * D, sV + r * pos_stride,
                                                 row_bytes, &full_bar[slot], policy);
                                    }
                                }
                            }
                        }
                    }
                }
                ++issued;
            }
        }
        // Drain: no copy may still be landing in shared memory when the CTA exits.
        if (lane == 0) {
            for (int s = max(0, issued - a.stages); s < issued; ++s) {
                if (!wait_bounded(&full_bar[s % a.stages], (s / a.stages) & 1))
                    atomicOr(a.err, kErrDrainWait);
            }
        }
        if constexpr (CLUSTER) cluster_tail();
        return;
    }

    // ---------------- consumer warps ----------------
    const int lig = lane % BDX;              // lane within its group
    const int lg = warp * BDY + lane / BDX;  // lane group id in the CTA
    const int nchunk = D >> 3;               // 8-element chunks per row
    bool con[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i) con[i] = lig + BDX * i < nchunk;
    const bool all_con = BDX * CH == nchunk;  // every lane owns all its chunks

    int hl[KMAX], ph[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
        const int s = lg + k * NLG;  // slot = phase * heads_per_cta + head
        ph[k] = s / a.heads_per_cta;
        hl[k] = s - ph[k] * a.heads_per_cta;
    }
    const int iters = a.stage_pos / a.phases;
    const uint32_t consumer_threads = static_cast<uint32_t>(a.active_warps) * 32;
    float *mbuf = reinterpret_cast<float *>(smem + a.merge_offset);
    const int rec = D + 2;
    // the producer copies a dense cache's head-group stages as tensor boxes
    // (partial ones ending at the buffer's last row) under this condition
    const bool tail_box_cta = MODE == kModeCluster && a.use_tmap && (smem_addr(smem) & 127u) == 0;
    int st = 0;
    // ok turns false (for the whole warp) once a pipeline wait has run out.  The
    // warp then skips waits, compute and writes, but keeps walking the pieces
    // and joining the consumers' named barriers, so no other warp can be left
    // waiting on it.
    bool ok = true;

    while (next_piece<CLUSTER>(walk, a)) {
        const int h0 = walk.g * a.heads_per_cta;
        const int hg = min(a.heads_per_cta, a.H - h0);
        // a unit this CTA covers whole gets its f16 output here (in cluster mode
        // every output goes through the cluster merge)
        const bool final_piece = !CLUSTER && walk.off == 0 && walk.len == walk.Lb;
        const int pstride = a.phases * hg * D;  // halves between a slot's consecutive positions
        const long long slot_id = piece_slot(blockIdx.x, walk.u);
        const __half *Qb =
            reinterpret_cast<const __half *>(a.Q) + (static_cast<size_t>(walk.b) * a.H + h0) * D;

        bool sv[KMAX];
        int kofs[KMAX];  // halves from a stage's first row to the slot's first row
        uint4 q[KMAX][CH];
        float acc[KMAX][CH * 8], m[KMAX], l[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
            sv[k] = ph[k] < a.phases && hl[k] < hg;
            kofs[k] = sv[k] ? (ph[k] * hg + hl[k]) * D : 0;
            m[k] = -INFINITY;
            l[k] = 0.f;
#pragma unroll
            for (int i = 0; i < CH * 8; ++i) acc[k][i] = 0.f;
#pragma unroll
            for (int i = 0; i < CH; ++i) {
                q[k][i] = make_uint4(0u, 0u, 0u, 0u);
                if (sv[k] && con[i])
                    q[k][i] = ldg_nc_v4(Qb + static_cast<size_t>(hl[k]) * D + (lig + BDX * i) * 8);
            }
        }

        for (int p = 0; p < walk.len; p += a.stage_pos, ++st) {
            const int slot = st % a.stages;
            if (ok) {
                const bool done = wait_bounded(&full_bar[slot], (st / a.stages) & 1);
                if (!__all_sync(kFull, done)) {
                    if (lane == 0) atomicOr(a.err, kErrConsumerWait);
                    *abort_flag = 1;
                    ok = false;
                }
            }
            if (!ok) continue;
            const int np = min(a.stage_pos, walk.len - p);
            // a partial stage of a dense cache copied as a tensor box ends at the
            // buffer's last row (see the producer)
            const int row_skip = tail_box_cta && hg < a.H && np < a.stage_pos ? a.stage_pos - np : 0;
            const __half *sK = ring + static_cast<size_t>(slot) * 2 * buf_elems +
                               static_cast<size_t>(row_skip) * hg * D;
            const __half *sV = sK + buf_elems;
            // One group: NPOS positions of each (head, phase) slot, whose dot
            // products, shuffles and exponentials are independent, so their
            // latencies overlap.  CHK = false is the path of a full group (every
            // position of it inside the stage, every chunk of the row owned):
            // no per-position tests.  A lane group without a slot still runs it,
            // on rows of the stage (kofs = 0), and its state is never written.
            auto group = [&](const int t, auto checked) {
                constexpr bool CHK = decltype(checked)::value;
                float s[KMAX][NPOS];
                bool vv[KMAX][NPOS];
                int rr[KMAX][NPOS];
#pragma unroll
                for (int k = 0; k < KMAX; ++k) {
                    float a_[NPOS], b_[NPOS];
#pragma unroll
                    for (int n = 0; n < NPOS; ++n) {
                        vv[k][n] = !CHK || (sv[k] && (t + n < iters) && ph[k] + (t + n) * a.phases < np);
                        rr[k][n] = kofs[k] + (t + n) * pstride;
                        a_[n] = 0.f;
                        b_[n] = 0.f;
                    }
#pragma unroll
                    for (int i = 0; i < CH; ++i) {
                        if (!CHK || con[i]) {
                            const int c8 = (lig + BDX * i) * 8;
#pragma unroll
                            for (int n = 0; n < NPOS; ++n)
                                if (vv[k][n])
                                    dot8(q[k][i], *reinterpret_cast<const uint4 *>(sK + rr[k][n] + c8),
                                         a_[n], b_[n]);
                        }
                    }
#pragma unroll
                    for (int n = 0; n < NPOS; ++n) s[k][n] = a_[n] + b_[n];
                }
#pragma unroll
                for (int o = BDX / 2; o > 0; o >>= 1) {
#pragma unroll
                    for (int k = 0; k < KMAX; ++k)
#pragma unroll
                        for (int n = 0; n < NPOS; ++n) s[k][n] += __shfl_xor_sync(kFull, s[k][n], o);
                }
#pragma unroll
                for (int k = 0; k < KMAX; ++k) {
                    if (CHK && !vv[k][0]) continue;  // a later position valid implies the first
                    float sc[NPOS];
                    float mx = -INFINITY;
#pragma unroll
                    for (int n = 0; n < NPOS; ++n) {
                        sc[n] = vv[k][n] ? s[k][n] * a.qscale : -INFINITY;
                        mx = fmaxf(mx, sc[n]);
                    }
                    if (mx > m[k]) {  // new running max: rescale the state
                        const float alpha = fast_exp2(m[k] - mx);
                        l[k] *= alpha;
#pragma unroll
                        for (int i = 0; i < CH * 8; ++i) acc[k][i] *= alpha;
                        m[k] = mx;
                    }
                    float pw[NPOS];
#pragma unroll
                    for (int n = 0; n < NPOS; ++n) {
                        pw[n] = vv[k][n] ? fast_exp2(sc[n] - m[k]) : 0.f;
                        l[k] += pw[n];
                    }
#pragma unroll
                    for (int i = 0; i < CH; ++i) {
                        if (!CHK || con[i]) {
                            const int c8 = (lig + BDX * i) * 8;
#pragma unroll
                            for (int n = 0; n < NPOS; ++n)
                                if (vv[k][n])
                                    axpy8(&acc[k][i * 8], pw[n],
                                          *reinterpret_cast<const uint4 *>(sV + rr[k][n] + c8));
                        }
                    }
                }
            };
            int t = 0;
            // (t + NPOS) * phases <= np puts every slot's positions of the group
            // inside the stage (ph < phases), and t + NPOS <= iters
            if (all_con)
                for (; (t + NPOS) * a.phases <= np; t += NPOS) group(t, std::false_type{});
            for (; t < iters; t += NPOS) group(t, std::true_type{});
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[slot]);
        }
        const bool write = ok && !*abort_flag;

        // ---------------- piece epilogue ----------------
        const size_t bh0 = static_cast<size_t>(walk.b) * a.H + h0;
        if (a.phases == 1) {
            // each slot is the only holder of its head: write from registers
#pragma unroll
            for (int k = 0; k < KMAX; ++k) {
                if (!sv[k] || !write) continue;
                if (final_piece) {
                    const float inv = 1.f / l[k];
#pragma unroll
                    for (int i = 0; i < CH; ++i) {
                        if (con[i]) {
                            const int c8 = (lig + BDX * i) * 8;
                            *reinterpret_cast<uint4 *>(reinterpret_cast<__half *>(a.out) +
                                                       (bh0 + hl[k]) * D + c8) =
                                pack8_f16(&acc[k][i * 8], inv);
                        }
                    }
                } else if constexpr (CLUSTER) {  // the local record of the head
                    float *rec = lrec + hl[k] * (D + 2);
                    if (lig == 0) {
                        rec[0] = m[k];
                        rec[1] = l[k];
                    }
#pragma unroll
                    for (int i = 0; i < CH; ++i) {
                        if (con[i]) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) rec[2 + (lig + BDX * i) * 8 + e] = acc[k][i * 8 + e];
                        }
                    }
                } else {
                    const size_t row = static_cast<size_t>(slot_id) * a.heads_per_cta + hl[k];
#pragma unroll
                    for (int i = 0; i < CH; ++i) {
                        if (con[i]) {
                            float4 *dst = reinterpret_cast<float4 *>(a.ws_acc + row * D +
                                                                     (lig + BDX * i) * 8);
                            dst[0] = make_float4(acc[k][i * 8 + 0], acc[k][i * 8 + 1],
                                                 acc[k][i * 8 + 2], acc[k][i * 8 + 3]);
                            dst[1] = make_float4(acc[k][i * 8 + 4], acc[k][i * 8 + 5],
                                                 acc[k][i * 8 + 6], acc[k][i * 8 + 7]);
                        }
                    }
                    if (lig == 0) a.ws_ml[row] = make_float2(m[k], l[k]);
                }
            }
        } else {
            // Several lane groups share a head.  In the cluster plan, when the
            // heads per CTA are a power of two below the lane groups per warp,
            // the lane groups of one warp that hold the same head (lane offsets
            // that are multiples of HG * BDX) first merge their states with xor
            // shuffles, and only the first HG lane groups of the warp keep a
            // state: phases f = 0, fstep, 2 fstep, ...  Then the kept states are
            // merged in shared memory.  (The split plan's instances leave the
            // shuffle step out: its code alone, never run on the latency-bound
            // split shapes, measured 0.55 us slower on a 7b call.)
            const int hgc = a.heads_per_cta;
            const bool wmerge = CLUSTER && BDY > 1 && hgc < BDY && (hgc & (hgc - 1)) == 0;
            const int fstep = wmerge ? BDY / hgc : 1;
            if (wmerge) {
#pragma unroll
                for (int k = 0; k < KMAX; ++k) {
                    if (!sv[k] || !write) {  // an empty state takes part in the exchange
                        m[k] = -INFINITY;
                        l[k] = 0.f;
                    }
                    for (int t = hgc; t < BDY; t <<= 1) {
                        const int o = t * BDX;
                        const float m2 = __shfl_xor_sync(kFull, m[k], o);
                        const float l2 = __shfl_xor_sync(kFull, l[k], o);
                        const float nm = fmaxf(m[k], m2);
                        const float s1 = nm == -INFINITY ? 0.f : fast_exp2(m[k] - nm);
                        const float s2 = nm == -INFINITY ? 0.f : fast_exp2(m2 - nm);
                        l[k] = fmaf(l[k], s1, l2 * s2);
#pragma unroll
                        for (int i = 0; i < CH * 8; ++i) {
                            const float a2 = __shfl_xor_sync(kFull, acc[k][i], o);
                            acc[k][i] = fmaf(acc[k][i], s1, a2 * s2);
                        }
                        m[k] = nm;
                    }
                }
            }
            const bool keeper = !wmerge || (lane / BDX) < hgc;
#pragma unroll
            for (int k = 0; k < KMAX; ++k) {
                if (!sv[k] || !write || !keeper) continue;
                float *r = mbuf + static_cast<size_t>(lg + k * NLG) * rec;
                if (lig == 0) {
                    r[0] = m[k];
                    r[1] = l[k];
                }
#pragma unroll
                for (int i = 0; i < CH; ++i) {
                    if (con[i]) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) r[2 + (lig + BDX * i) * 8 + e] = acc[k][i * 8 + e];
                    }
                }
            }
            named_barrier_sync(1, consumer_threads);
            const bool all_write = !*abort_flag;  // same for every consumer after the barrier
            for (int idx = threadIdx.x; all_write && idx < hg * D; idx += consumer_threads) {
                const int h = idx / D;
                const int d = idx - h * D;
                float M = -INFINITY;
                for (int f = 0; f < a.phases; f += fstep) {
                    const float *r = mbuf + static_cast<size_t>(f * a.heads_per_cta + h) * rec;
                    if (r[1] > 0.f) M = fmaxf(M, r[0]);
                }
                float lsum = 0.f, num = 0.f;
                for (int f = 0; f < a.phases; f += fstep) {
                    const float *r = mbuf + static_cast<size_t>(f * a.heads_per_cta + h) * rec;
                    if (r[1] > 0.f) {
                        const float w = fast_exp2(r[0] - M);
                        lsum = fmaf(w, r[1], lsum);
                        num = fmaf(w, r[2 + d], num);
                    }
                }
                if (final_piece) {
                    reinterpret_cast<__half *>(a.out)[(bh0 + h) * D + d] = __float2half_rn(num / lsum);
                } else if constexpr (CLUSTER) {  // the local record
                    float *rec = lrec + h * (D + 2);
                    rec[2 + d] = num;
                    if (d == 0) {
                        rec[0] = M;
                        rec[1] = lsum;
                    }
                } else {
                    const size_t row = static_cast<size_t>(slot_id) * a.heads_per_cta + h;
                    a.ws_acc[row * D + d] = num;
                    if (d == 0) a.ws_ml[row] = make_float2(M, lsum);
                }
            }
            named_barrier_sync(1, consumer_threads);
        }
    }
    if constexpr (CLUSTER) cluster_tail();
}

// Instances: lanes per row x chunks per lane x slots per lane group x consumer
// warps.  Eight consumer warps (two CTAs per SM) up to one slot of two chunks
// or two slots of one chunk per lane group; sixteen consumer warps (one CTA per
// SM, the same warps per SM) when a CTA must hold more heads.
template <int BDX, int CH, int NWC, int MODE>
const void *pick_kmax(int kmax) {
    switch (kmax) {
        case 1: return reinterpret_cast<const void *>(decode_streamk_kernel<BDX, CH, 1, NWC, MODE>);
        case 2:
            if constexpr (CH == 1)
                return reinterpret_cast<const void *>(decode_streamk_kernel<BDX, CH, 2, NWC, MODE>);
            return nullptr;
        default: return nullptr;
    }
}

template <int NWC, int MODE>
const void *pick_shape(int bdx, int ch, int kmax) {
    if (ch == 1) {
        switch (bdx) {
            case 1: return pick_kmax<1, 1, NWC, MODE>(kmax);
            case 2: return pick_kmax<2, 1, NWC, MODE>(kmax);
            case 4: return pick_kmax<4, 1, NWC, MODE>(kmax);
            case 8: return pick_kmax<8, 1, NWC, MODE>(kmax);
            default: return nullptr;
        }
    }
    if (ch == 2) {
        switch (bdx) {
            case 8: return pick_kmax<8, 2, NWC, MODE>(kmax);
            case 16: return pick_kmax<16, 2, NWC, MODE>(kmax);
            default: return nullptr;
        }
    }
    return nullptr;
}

// The instances of one mode.
template <int MODE>
const void *variant_fn_of(DecodeVariant v) {
    if (v.nwc == 8) return pick_shape<8, MODE>(v.bdx, v.ch, v.kmax);
    if (v.nwc == 16) return pick_shape<16, MODE>(v.bdx, v.ch, v.kmax);
    return nullptr;
}

}  // namespace
}  // namespace dattn
