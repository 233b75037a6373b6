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
// spread over every partition, so each thread folds only a few pieces (the
// merge itself is merge::merge_task).  Launched with programmatic dependent
// launch: it may start while the decode kernel drains and waits on
// griddepcontrol.wait before touching the workspace.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "dattn_internal.h"
#include "ptx.cuh"
#include "merge.cuh"
#include "streamk.h"

namespace dattn {
namespace {

constexpr int kThreads = 128;
constexpr int kInlinePrefix = 4096;  // batches summed from current_pos in the combine

// INFLIGHT: piece loads each thread issues before folding them.  The host picks
// the smallest depth that covers a thread's expected pieces in one round; the
// shallow instances are bounded to 64 and 128 registers (8 and 4 CTAs per SM):
// tighter bounds, which let more of a large batch's merge CTAs be resident at
// once, spill and measured slower.
template <int INFLIGHT>
__global__ void __launch_bounds__(kThreads, INFLIGHT <= 2 ? 8 : (INFLIGHT <= 4 ? 4 : 1))
    combine_kernel(const CombineArgs a) {
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
    const long long Lb = merge::live_len(a.cur_pos, b, a.S);
    // Live positions before sequence b and in total.  For batches of up to
    // kInlinePrefix sequences they are summed here from current_pos (an input,
    // readable before the decode kernel finishes); larger batches read the
    // prefix sums the decode kernel wrote.
    long long before = 0, total = 0;
    if (a.B <= kInlinePrefix) {
        for (int i = tid; i < a.B; i += kThreads) {
            const long long L = merge::live_len(a.cur_pos, i, a.S);
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
    merge::merge_task<kThreads, INFLIGHT>(a.ws_acc, a.ws_ml, a.out, a.D, a.heads_per_cta, bh, c0, width, u,
                                hl, c_first, npieces, W, a.partitions, tid, sm_m, sm_l, sm_a,
                                [] { __syncthreads(); });
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
    if (a.inflight <= 2) return cudaLaunchKernelEx(&cfg, combine_kernel<2>, a);
    if (a.inflight <= 4) return cudaLaunchKernelEx(&cfg, combine_kernel<4>, a);
    return cudaLaunchKernelEx(&cfg, combine_kernel<8>, a);
}

}  // namespace dattn
