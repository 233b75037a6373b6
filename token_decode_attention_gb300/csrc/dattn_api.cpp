// dattn_api.cpp -- the C ABI declared in include/dattn.h.
//
// Host side of the library: argument validation (before anything is
// launched), the stream-K plan (tiling, pipeline depth, partition count), the
// library-owned workspace of dattn_decode_f16, status codes and per-thread
// error messages.  The arithmetic of the operation runs only in the CUDA
// kernels (decode_streamk.cu, combine.cu, split_calls.cu).
#include "dattn.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <unordered_map>

#include "dattn_internal.h"

namespace {

using dattn::DecodeVariant;

constexpr int kVersion = 10000;        // 1.0.0
constexpr int kMaxPartitions = 65535;  // CTAs of the decode grid
constexpr int kMaxHeadDim = 256;
constexpr int kMaxHeadsPerLaneGroup = 4;  // register slots per lane group (KMAX)
constexpr int kMaxRowBytesKV = 48 * 1024; // K+V bytes per position a CTA stages
// Tiling constants of the plan.  Each can be overridden at compile time
// (-DDATTN_<NAME>=value) to explore other configurations.
#ifndef DATTN_STAGE_BYTES_TWO_PER_SM
#define DATTN_STAGE_BYTES_TWO_PER_SM (32 * 1024)
#endif
#ifndef DATTN_STAGE_BYTES_ONE_PER_SM
#define DATTN_STAGE_BYTES_ONE_PER_SM (64 * 1024)
#endif
// At one CTA per SM a dense cache takes two stages of ~100 KB rather than
// three of 64 KB: about the same ring, fewer and larger copies and more
// positions per stage for the consumers.  Measured (split plan, graph replay,
// same runs): long 298-301 -> 294.5 us, ragged 150.1 -> 149.0 us, outlier
// 5705-5718 -> 5700-5708 us; few heads (rows of at most 4 KB) 5-8 %, e.g.
// B=64 H=8 ragged 46.5 -> 42.9 us, B=1 H=4 S=65536 21.4 -> 19.8 us.  Stages of
// 96 KB gave the 10 KB rows of 40 heads only two 80 KB stages: +0.7 %.  A paged
// cache gains only with small rows (its larger rows measured +0.3 to +0.9 %
// with ~100 KB stages), so its rows above DATTN_SMALL_ROW_BYTES keep 64 KB.
#ifndef DATTN_STAGE_BYTES_DENSE
#define DATTN_STAGE_BYTES_DENSE (100 * 1024)
#endif
// Measured (ragged lengths unless noted): with 2, B=4 H=8 D=128 S=2048 took
// 13.1 us against 12.1 with the smaller stages; with 4 the few-head gains above
// stay (B=1 H=1 S=131072 13.5 us, B=1 H=4 S=65536 19.8 us); with 8 or 16 they
// are lost (14.3 / 21.4 us) while B=4 H=8 D=256 (17.6 -> 17.0 us) and B=4 H=32
// (14.0 -> 13.3 us at 16) would gain.
#ifndef DATTN_BIG_STAGES_PER_SLOT
#define DATTN_BIG_STAGES_PER_SLOT 4
#endif
#ifndef DATTN_SMALL_ROW_BYTES
#define DATTN_SMALL_ROW_BYTES 4096
#endif
#ifndef DATTN_STAGE_BYTES_SMALL_ROWS
#define DATTN_STAGE_BYTES_SMALL_ROWS (96 * 1024)
#endif
#ifndef DATTN_RING_BYTES_TWO_PER_SM
#define DATTN_RING_BYTES_TWO_PER_SM (110 * 1024)
#endif
#ifndef DATTN_RING_BYTES_ONE_PER_SM
#define DATTN_RING_BYTES_ONE_PER_SM (200 * 1024)
#endif
#ifndef DATTN_DEEP_RING_POSITIONS
#define DATTN_DEEP_RING_POSITIONS (1LL << 40)
#endif
#ifndef DATTN_MIN_CONSUMER_WARPS
#define DATTN_MIN_CONSUMER_WARPS 8  // 16: always sixteen consumer warps per CTA
#endif
#ifndef DATTN_PREFETCH_STAGES
#define DATTN_PREFETCH_STAGES 2  // stages each CTA prefetches into L2 before its wait (0: none)
#endif
#ifndef DATTN_MIN_HEAD_GROUPS
#define DATTN_MIN_HEAD_GROUPS 1  // split the heads into at least this many groups
#endif
#ifndef DATTN_MIN_POSITIONS
#define DATTN_MIN_POSITIONS 16
#endif
// Cluster mode (one cluster of CTAs per (sequence, head group), merged in
// distributed shared memory; see DecodeArgs::cluster).
#ifndef DATTN_CLUSTER_MAX_BATCH
#define DATTN_CLUSTER_MAX_BATCH 1  // sequences up to which cluster mode is considered
#endif
#ifndef DATTN_CLUSTER_STAGE_BYTES
#define DATTN_CLUSTER_STAGE_BYTES (64 * 1024)  // K+V per pipeline stage
#endif
#ifndef DATTN_CLUSTER_MIN_CTA_BYTES
#define DATTN_CLUSTER_MIN_CTA_BYTES (32 * 1024)  // K+V capacity per CTA at least
#endif
#ifndef DATTN_CLUSTER_MAX_CAPACITY_BYTES
#define DATTN_CLUSTER_MAX_CAPACITY_BYTES (512LL << 20)  // K+V capacity up to which it is used
#endif
#ifndef DATTN_CLUSTER_PAGED_MIN_COPY_BYTES
// A paged cache takes the cluster plan only when one page of a head group (one
// tensor box or bulk copy) holds at least this much K, and only with as many
// CTAs as the plan of a dense cache of the same shape.  The copies are issued
// one per page; on GB300 a 7B-class step (128 CTAs of one head, 256 B rows)
// measured 30.6 us with 4 KB page boxes (16-position pages), 15.5 us with
// 16 KB and 14.9 us with 32 KB, and 64 CTAs of 8 heads (32 KB boxes of
// 16-position pages) 21.7 us, against 15.3-15.5 us for the split plan.
#define DATTN_CLUSTER_PAGED_MIN_COPY_BYTES (32 * 1024)
#endif
// The cluster plan streams with fewer CTAs than the split plan (whole clusters
// must be resident at once), and saves the merge kernel's ~1-2 us.  It is kept
// only where that trade wins on GB300: at most DATTN_CLUSTER_MAX_CTA_BYTES of
// K+V capacity per CTA, and at least DATTN_CLUSTER_MIN_CTA_FRACTION of the SMs
// busy unless the call is latency-bound (at most DATTN_CLUSTER_TINY_CTA_BYTES
// per CTA).  Measured B=1 (cluster vs split plan): 1 head, 16 CTAs, 100001
// live positions 48.0 vs 14.2 us; 2 heads, 32 CTAs 48.8 vs 21.1 us; 4 heads,
// 64 CTAs (2 MiB per CTA) 28.1 vs 21.5 us; 32 heads, 128 CTAs, 16384 positions
// (2 MiB per CTA) 33.7 vs 32.1 us at 12001 live positions, 40.4 vs 41.8 at
// 16384; and faster on the cluster plan from 96 CTAs at 1.4 MiB per CTA down.
#ifndef DATTN_CLUSTER_MAX_CTA_BYTES
#define DATTN_CLUSTER_MAX_CTA_BYTES (2LL << 20)
#endif
#ifndef DATTN_CLUSTER_MIN_CTA_FRACTION
#define DATTN_CLUSTER_MIN_CTA_FRACTION 0.6
#endif
#ifndef DATTN_CLUSTER_TINY_CTA_BYTES
#define DATTN_CLUSTER_TINY_CTA_BYTES (128LL << 10)
#endif
#ifndef DATTN_CLUSTER_MAX_SIZE
#define DATTN_CLUSTER_MAX_SIZE 16  // CTAs per cluster (8 is the portable limit)
#endif
#ifndef DATTN_CLUSTER_PREFER_SMALL
#define DATTN_CLUSTER_PREFER_SMALL 0  // on a tie in CTAs: 0 fewer head groups, 1 smaller clusters
#endif
#ifndef DATTN_CLUSTER_FORCE_GROUPS
#define DATTN_CLUSTER_FORCE_GROUPS 0  // > 0: only this many head groups (exploration)
#endif
#ifndef DATTN_CLUSTER_FORCE_SIZE
#define DATTN_CLUSTER_FORCE_SIZE 0  // > 0: only clusters of this many CTAs (exploration)
#endif
constexpr int kClusterMaxBatch = DATTN_CLUSTER_MAX_BATCH;
constexpr int kStageTargetBytes = DATTN_STAGE_BYTES_TWO_PER_SM;         // K+V per stage, 2 CTAs/SM
constexpr int kStageTargetBytesOnePerSm = DATTN_STAGE_BYTES_ONE_PER_SM;  // K+V per stage, 1 CTA/SM
constexpr int kTwoPerSmBudget = DATTN_RING_BYTES_TWO_PER_SM;  // ring bytes per CTA at 2 CTAs/SM
constexpr int kOnePerSmBudget = DATTN_RING_BYTES_ONE_PER_SM;  // ring bytes per CTA at 1 CTA/SM
constexpr int kMaxStages = 12;
// positions per CTA at two CTAs per SM below which one CTA per SM with a deep
// ring is used
constexpr long long kDeepRingPositions = DATTN_DEEP_RING_POSITIONS;
constexpr long long kMinPositions = DATTN_MIN_POSITIONS;  // per partition chosen by the library
constexpr int kStaticSmemReserve = 1024;  // the decode kernel's static shared memory

thread_local std::string g_last_error;

int fail(int status, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

int fail_cuda(cudaError_t e, const char *what) {
    return fail(DATTN_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- device info

struct DeviceInfo {
    int sms = 0;
    int max_smem_optin = 0;
    unsigned *err_word = nullptr;
};

std::mutex g_dev_mutex;
std::unordered_map<int, DeviceInfo> g_devices;

int current_device(int *dev) {
    const cudaError_t e = cudaGetDevice(dev);
    return e == cudaSuccess ? DATTN_OK : fail_cuda(e, "cudaGetDevice");
}

// Device properties and one-time kernel configuration for the current device.
int device_info(DeviceInfo *out) {
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    auto it = g_devices.find(dev);
    if (it != g_devices.end()) {
        *out = it->second;
        return DATTN_OK;
    }
    DeviceInfo di;
    cudaError_t e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute(SM count)");
    e = cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute(smem opt-in)");
    e = dattn::decode_configure_smem(di.max_smem_optin);
    if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute(decode kernel)");
    e = dattn::device_error_word(&di.err_word);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(error word)");
    g_devices[dev] = di;
    *out = di;
    return DATTN_OK;
}

// --------------------------------------------------------------------- plans

struct Plan {
    DecodeVariant v{};
    int HG = 0, NHG = 0, PHI = 0, P = 0, NST = 0, G = 0, active_warps = 0;
    int smem = 0, merge_offset = 0, bar_offset = 0, ctas_per_sm = 0, sms = 0;
    size_t prefix_bytes = 0, acc_bytes = 0, ws_bytes = 0;
    int combine_chunk = 0;  // channels per combine CTA
    int combine_inflight = 8;  // piece loads per combine thread per round
    // cluster mode (see DecodeArgs::cluster): CTAs per cluster (0 = stream-K)
    int cluster = 0, use_tmap = 0, rec_offset = 0, box_pos = 0;
};

int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }
static size_t round_up_sz(size_t x, size_t m) { return (x + m - 1) / m * m; }

int validate_dims(int B, int H, int D, int S) {
    if (B <= 0 || H <= 0 || D <= 0 || S <= 0)
        return fail(DATTN_ERR_INVALID_ARG,
                    "sizes must be positive (batch=%d n_heads=%d head_dim=%d seq_len=%d)", B, H,
                    D, S);
    if (D % 8 != 0 || D > kMaxHeadDim)
        return fail(DATTN_ERR_UNSUPPORTED, "head_dim=%d: must be a multiple of 8 and <= %d", D,
                    kMaxHeadDim);
    // element counts of the largest tensor must stay far inside int64
    const double elems = static_cast<double>(B) * S * H * D;
    if (elems > 4.0e18)
        return fail(DATTN_ERR_INVALID_ARG, "KV cache of %.3g elements is too large", elems);
    return DATTN_OK;
}

// (device, B, H, D, S, num_partitions, page_size: 0 dense, -1 paged of any page size)
using PlanKey = std::tuple<int, int, int, int, int, int, int>;
std::mutex g_plan_mutex;
std::map<PlanKey, Plan> g_plans;

// Number of partitions (CTAs) when the caller leaves it to the library: every
// resident CTA slot of the GPU, unless the batch's capacity is so small that a
// partition would hold less than min_pos positions (then fewer CTAs, to keep
// the partial states the combine must merge few).
int choose_partitions(const Plan &p, int B, int S) {
    const long long slots = static_cast<long long>(p.sms) * p.ctas_per_sm;
    const long long capacity = static_cast<long long>(B) * p.NHG * S;
    // At least a stage (and 8 positions) per partition when every head has its
    // own lane group; with several phases per head a partition also pays a
    // shared-memory merge per piece, so it keeps two stages (and
    // kMinPositions).  Either way a small batch still spreads over up to 32
    // partitions of a stage each.
    const long long min_pos = p.PHI == 1 ? std::max<long long>(8, p.P)
                                         : std::max<long long>(kMinPositions, 2LL * p.P);
    const long long by_work =
        std::max<long long>({1, capacity / min_pos, std::min<long long>(32, capacity / p.P)});
    return static_cast<int>(std::min<long long>({slots, by_work, kMaxPartitions}));
}

int make_cluster_plan(int B, int H, int D, int S, int page_size, const DeviceInfo &di, Plan *out);

int lcm_int(int x, int y) {
    int a = x, b = y;
    while (b != 0) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return x / a * y;
}

// The split (stream-K) plan with at least `min_groups` head groups, for a
// dense or a paged cache.
int split_plan(int B, int H, int D, int S, int num_partitions, int min_groups, bool paged,
               const DeviceInfo &di, Plan *out) {
    Plan p;
    p.sms = di.sms;
    // lanes per KV row and 8-element chunks per lane
    const int c8 = D / 8;
    int bdx, ch;
    if (c8 <= 8) {
        bdx = next_pow2(c8);
        ch = 1;
    } else if (c8 <= 16) {
        bdx = 8;
        ch = 2;
    } else {
        bdx = 16;
        ch = 2;
    }
    // Eight consumer warps (two CTAs per SM) while the heads fit their register
    // slots; otherwise sixteen (one CTA per SM, same warps per SM); beyond that
    // the heads are split into groups handled by different CTAs.
    const int kcap = ch == 2 ? 1 : 2;  // register slots per lane group
    int nwc = DATTN_MIN_CONSUMER_WARPS > 8 ? 16 : 8;
    if (H > nwc * (32 / bdx) * kcap) nwc = 16;
    const int nlg = nwc * (32 / bdx);  // lane groups per CTA
    const int hg_max = std::min(nlg * kcap, std::max(1, kMaxRowBytesKV / (D * 4)));
    p.NHG = std::max((H + hg_max - 1) / hg_max, std::min(H, min_groups));
    p.HG = (H + p.NHG - 1) / p.NHG;
    p.NHG = (H + p.HG - 1) / p.HG;  // no empty group
    p.PHI = p.HG >= nlg ? 1 : std::min(32, nlg / p.HG);
    const int kmax = (p.HG * p.PHI + nlg - 1) / nlg;
    p.v = DecodeVariant{bdx, ch, kmax, nwc};
    // warps whose first lane group holds a slot (slot s = lane group + k * nlg)
    p.active_warps = std::min(nwc, (p.HG * p.PHI + (32 / bdx) - 1) / (32 / bdx));
    const int row_bytes = p.HG * D * 2;
    // One CTA per SM with a deep ring of large stages (measured best on GB300
    // for every workload shape: a CTA alone keeps ~190 KB in flight, and large
    // bulk copies are the most efficient).  Two CTAs per SM with half the ring
    // remain available through DATTN_DEEP_RING_POSITIONS.
    const long long capacity_pos = static_cast<long long>(B) * p.NHG * S;
    const bool deep = dattn::decode_min_blocks(nwc) == 1 ||
                      capacity_pos < kDeepRingPositions * 2LL * di.sms;
    const long long slots = static_cast<long long>(di.sms) * (deep ? 1 : 2);
    auto stage_positions = [&](int target) {
        const int q = std::max(1, std::min(256, target / 2 / row_bytes));
        return std::max(p.PHI, q / p.PHI * p.PHI);
    };
    int P = stage_positions(deep ? kStageTargetBytesOnePerSm : kStageTargetBytes);
    // the larger stages, where the batch's capacity gives every CTA slot
    // DATTN_BIG_STAGES_PER_SLOT of them (a smaller batch is bound by latency
    // and keeps the smaller stages, more of them in flight)
    const int big_target = !deep                               ? 0
                           : !paged                             ? DATTN_STAGE_BYTES_DENSE
                           : row_bytes <= DATTN_SMALL_ROW_BYTES ? DATTN_STAGE_BYTES_SMALL_ROWS
                                                                : 0;
    if (big_target > 0) {
        const int Pb = stage_positions(big_target);
        if (capacity_pos >= slots * static_cast<long long>(DATTN_BIG_STAGES_PER_SLOT) * Pb) P = Pb;
    }
    // A batch too small to give every CTA slot two stages takes smaller stages,
    // for more partitions: such a decode is bound by latency, not by the
    // per-stage overhead that large stages amortise.
#ifndef DATTN_SMALL_BATCH_STAGES
#define DATTN_SMALL_BATCH_STAGES 1
#endif
    if (DATTN_SMALL_BATCH_STAGES) {
        while (P / 2 >= p.PHI && 2 * P > kMinPositions && capacity_pos < slots * 2LL * P)
            P = std::max(p.PHI, P / 2 / p.PHI * p.PHI);
    }
    p.P = P;
    const int stage_bytes = 2 * P * row_bytes;
    const int merge_bytes = p.PHI > 1 ? p.HG * p.PHI * (D + 2) * 4 : 0;
    const int ring_budget = deep ? kOnePerSmBudget - merge_bytes : kTwoPerSmBudget - merge_bytes;
    int nst = ring_budget / stage_bytes;
    if (nst < 2) nst = (di.max_smem_optin - 1024 - merge_bytes) / stage_bytes;
    p.NST = std::max(2, std::min(kMaxStages, nst));
    p.merge_offset = p.NST * stage_bytes;
    p.bar_offset = round_up(p.merge_offset + merge_bytes, 16);
    p.smem = p.bar_offset + p.NST * 16 + 16;
    if (p.smem > di.max_smem_optin - kStaticSmemReserve)
        return fail(DATTN_ERR_UNSUPPORTED, "shape needs %d B of shared memory (limit %d)",
                    p.smem, di.max_smem_optin);
    cudaError_t e = dattn::decode_occupancy(p.v, p.smem, &p.ctas_per_sm);
    if (e != cudaSuccess) return fail_cuda(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (p.ctas_per_sm < 1)
        return fail(DATTN_ERR_UNSUPPORTED, "decode kernel does not fit on an SM");
    p.G = num_partitions > 0 ? std::min(num_partitions, kMaxPartitions)
                             : choose_partitions(p, B, S);
    // partition arithmetic multiplies a partition index by the flattened
    // position count: keep it inside 64 bits
    const double capacity = static_cast<double>(B) * p.NHG * S;
    if (static_cast<double>(p.NHG) * S >= 2147483648.0)
        return fail(DATTN_ERR_UNSUPPORTED, "head_groups x seq_len must stay below 2^31");
    if (capacity * (p.G + 1.0) > 4.0e18)
        return fail(DATTN_ERR_UNSUPPORTED, "batch of %.3g positions is too large", capacity);
    if (p.G > 1) {
        const size_t units = static_cast<size_t>(B) * p.NHG;
        const size_t rows = (static_cast<size_t>(p.G) + units) * p.HG;
        p.prefix_bytes = round_up_sz((static_cast<size_t>(B) + 1) * sizeof(long long), 256);
        p.acc_bytes = round_up_sz(rows * D * sizeof(float), 256);
        p.ws_bytes = p.prefix_bytes + p.acc_bytes + rows * sizeof(float2);
        // Combine chunk: at most ~8 pieces per thread of a 128-thread CTA, given
        // the expected pieces per unit (G + U) / U.
        const double pieces = static_cast<double>(p.G + units) / static_cast<double>(units);
        int cw = std::min(256, next_pow2(D));
        while (cw > 8 && pieces * cw / 512.0 > 8.0) cw /= 2;
        p.combine_chunk = cw;
        // loads in flight per thread: a thread's expected pieces in one round
        const double per_thread = pieces / (128.0 / (cw / 4));
        p.combine_inflight = per_thread <= 2.0 ? 2 : (per_thread <= 4.0 ? 4 : 8);
    }
    *out = p;
    return DATTN_OK;
}


// page_size: 0 for a dense cache, the page size of a paged one, or -1 for a
// paged cache whose page size is not known (the split plan, which any paged
// call can run).
int make_plan(int B, int H, int D, int S, int num_partitions, int page_size, Plan *out) {
    if (int st = validate_dims(B, H, D, S)) return st;
    if (num_partitions < 0)
        return fail(DATTN_ERR_INVALID_ARG, "num_partitions=%d must be >= 0", num_partitions);
    DeviceInfo di;
    if (int st = device_info(&di)) return st;
    int dev = 0;
    if (int st = current_device(&dev)) return st;
    const PlanKey key{dev, B, H, D, S, num_partitions, page_size};
    {
        std::lock_guard<std::mutex> lock(g_plan_mutex);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) {
            *out = it->second;
            return DATTN_OK;
        }
    }
    Plan p;
    if (int st = split_plan(B, H, D, S, num_partitions, DATTN_MIN_HEAD_GROUPS, page_size != 0, di, &p))
        return st;
    // Few sequences (dense cache, library-chosen partitions): one cluster of
    // CTAs per (sequence, head group), merged in distributed shared memory,
    // when such a plan exists.
    if (num_partitions == 0 && page_size >= 0 && B <= kClusterMaxBatch) {
        Plan c;
        if (int st = make_cluster_plan(B, H, D, S, page_size, di, &c)) return st;
        if (c.cluster > 0 && page_size > 0) {
            // a paged cache keeps the dense plan's parallelism or takes the split plan
            Plan d;
            if (int st = make_cluster_plan(B, H, D, S, 0, di, &d)) return st;
            if (c.G < d.G) c.cluster = 0;
        }
        if (c.cluster > 0) p = c;
    }
    {
        std::lock_guard<std::mutex> lock(g_plan_mutex);
        g_plans[key] = p;
    }
    *out = p;
    return DATTN_OK;
}

// Cluster plan: unit (b, g) of HG = H / NHG heads goes to one cluster of C
// CTAs.  Among the head groupings whose K/V rows a tensor box can copy (or all
// heads, one contiguous span per position) and the cluster sizes of which
// B * NHG clusters fit on the GPU at once, take the one with the most CTAs
// while each CTA still holds DATTN_CLUSTER_MIN_CTA_BYTES of K+V capacity; on a
// tie, fewer head groups (longer rows).  out->cluster stays 0 when none fits.
int make_cluster_plan(int B, int H, int D, int S, int page_size, const DeviceInfo &di, Plan *out) {
    *out = Plan();
    const double cap_bytes = 4.0 * B * static_cast<double>(S) * H * D;  // K + V
    if (cap_bytes > static_cast<double>(DATTN_CLUSTER_MAX_CAPACITY_BYTES)) return DATTN_OK;
    // 32-bit box coordinate (a paged caller checks the rows of its pool)
    if (page_size == 0 && static_cast<double>(B) * S >= 2147483647.0) return DATTN_OK;
    // a paged cache: a stage is a whole number of pages and a page one tensor
    // box, whose height is at most 256 rows
    if (page_size < 0 || page_size > 256) return DATTN_OK;
    const int c8 = D / 8;
    int bdx, ch;
    if (c8 <= 8) {
        bdx = next_pow2(c8);
        ch = 1;
    } else if (c8 <= 16) {
        bdx = 8;
        ch = 2;
    } else {
        bdx = 16;
        ch = 2;
    }
    const int kcap = ch == 2 ? 1 : 2;
    Plan best;
    long long best_ctas = 0;
    for (int nhg = 1; nhg <= H; ++nhg) {
        if (H % nhg != 0) continue;
        if (DATTN_CLUSTER_FORCE_GROUPS > 0 && nhg != DATTN_CLUSTER_FORCE_GROUPS) continue;
        const int hg = H / nhg;
        if (hg * D * 4 > kMaxRowBytesKV) continue;
        int nwc = DATTN_MIN_CONSUMER_WARPS > 8 ? 16 : 8;
        if (hg > nwc * (32 / bdx) * kcap) nwc = 16;
        const int nlg = nwc * (32 / bdx);
        if (hg > nlg * kcap) continue;
        Plan p;
        p.sms = di.sms;
        p.NHG = nhg;
        p.HG = hg;
        p.PHI = hg >= nlg ? 1 : std::min(32, nlg / hg);
        const int kmax = (hg * p.PHI + nlg - 1) / nlg;
        p.v = DecodeVariant{bdx, ch, kmax, nwc};
        p.active_warps = std::min(nwc, (hg * p.PHI + (32 / bdx) - 1) / (32 / bdx));
        const int row_bytes = hg * D * 2;
        for (int C = DATTN_CLUSTER_MAX_SIZE; C >= 1; --C) {
            if (DATTN_CLUSTER_FORCE_SIZE > 0 && C != DATTN_CLUSTER_FORCE_SIZE) continue;
            const long long ctas = static_cast<long long>(B) * nhg * C;
            if (ctas > static_cast<long long>(di.sms)) continue;
            if (C > 1 && cap_bytes / static_cast<double>(ctas) < DATTN_CLUSTER_MIN_CTA_BYTES) continue;
            // a stage: ~DATTN_CLUSTER_STAGE_BYTES of K+V, no more than a CTA's
            // share of the capacity, a multiple of the phases (and of the page
            // size: the CTAs' ranges start on a page, so do the stages)
            const int quantum = page_size > 0 ? lcm_int(p.PHI, page_size) : p.PHI;
            if (quantum > 256) continue;
            const int share = (S + C - 1) / C;
            int P = std::max(1, std::min(256, DATTN_CLUSTER_STAGE_BYTES / 2 / row_bytes));
            P = std::min(P, std::max(share, quantum));
            P = std::max(quantum, P / quantum * quantum);
            if (P > 256) continue;
            // a head group's rows are copied as tensor boxes {D, HG, box}: a full
            // stage of a dense cache, a whole page of a paged one (the box's
            // shared-memory destination is 128-byte aligned)
            const bool grouped = hg < H;
            const int box = page_size > 0 ? page_size : P;
            if (grouped && (static_cast<long long>(box) * row_bytes) % 128 != 0) continue;
            if (page_size > 0 &&
                static_cast<long long>(page_size) * row_bytes < DATTN_CLUSTER_PAGED_MIN_COPY_BYTES)
                continue;
            const int merge_bytes = p.PHI > 1 ? hg * p.PHI * (D + 2) * 4 : 0;
            const int rec_bytes = hg * (D + 2) * 4;  // the CTA's record (m, l, acc) per head
            const int stage_bytes = 2 * P * row_bytes;
            const int avail = di.max_smem_optin - kStaticSmemReserve - merge_bytes - rec_bytes -
                              16 * kMaxStages - 64;
            const int nst = std::min(kMaxStages, avail / stage_bytes);
            if (nst < 2) continue;
            Plan q = p;
            q.P = P;
            q.NST = nst;
            q.merge_offset = nst * stage_bytes;
            q.rec_offset = round_up(q.merge_offset + merge_bytes, 16);
            q.bar_offset = round_up(q.rec_offset + rec_bytes, 16);
            q.smem = q.bar_offset + nst * 16 + 16;
            if (q.smem > di.max_smem_optin - kStaticSmemReserve) continue;
            int clusters = 0;
            cudaError_t e = dattn::decode_max_clusters(q.v, q.smem, C, page_size > 0, &clusters);
            if (e != cudaSuccess) {
                cudaGetLastError();  // this cluster size is not available: try the next
                continue;
            }
            if (clusters < B * nhg) continue;  // every cluster resident at once
            const bool better =
                ctas > best_ctas || (DATTN_CLUSTER_PREFER_SMALL && ctas == best_ctas && C < best.cluster);
            if (!better) continue;
            e = dattn::decode_occupancy(q.v, q.smem, &q.ctas_per_sm);
            if (e != cudaSuccess) return fail_cuda(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
            q.cluster = C;
            q.use_tmap = grouped ? 1 : 0;
            q.box_pos = box;
            q.G = static_cast<int>(ctas);
            q.ws_bytes = 0;
            best = q;
            best_ctas = ctas;
        }
    }
    if (best.cluster > 0) {
        const double cta_bytes = cap_bytes / static_cast<double>(best.G);
        const bool busy = best.G >= DATTN_CLUSTER_MIN_CTA_FRACTION * di.sms;
        if (cta_bytes > static_cast<double>(DATTN_CLUSTER_MAX_CTA_BYTES) ||
            (!busy && cta_bytes > static_cast<double>(DATTN_CLUSTER_TINY_CTA_BYTES)))
            best = Plan();  // the split plan streams faster
    }
    *out = best;
    return DATTN_OK;
}

int check_tensor(const void *p, const char *name) {
    if (p == nullptr) return fail(DATTN_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(p)) return fail(DATTN_ERR_MISALIGNED, "%s is not 16-byte aligned", name);
    return DATTN_OK;
}

int check_cur_pos(const uint32_t *cp) {
    if (cp == nullptr) return fail(DATTN_ERR_INVALID_ARG, "current_pos is NULL");
    if ((reinterpret_cast<uintptr_t>(cp) & 3u) != 0)
        return fail(DATTN_ERR_MISALIGNED, "current_pos is not 4-byte aligned");
    return DATTN_OK;
}

struct Paging {
    const int *table = nullptr;  // nullptr: dense [B, S, H, D] cache
    long long num_pages = 0;
    int page_size = 0, max_pages = 0;
};

// cuTensorMapEncodeTiled from the driver, found once through the runtime (the
// driver library is not linked).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// Tensor map of a cache [rows, H heads, D] (f16, innermost D) whose box is
// `box_rows` rows of one head group, {D, HG, box_rows}: the B*S positions of a
// dense cache and one stage, or the num_pages*page_size rows of a page pool
// and one page.
int encode_kv_box(CUtensorMap *map, const void *base, long long rows, int H, int D, int HG,
                  int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (enc == nullptr) return fail(DATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(H) * D * 2};  // bytes, dims 1 and 2
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(HG),
                               static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t unit[3] = {1, 1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims,
                           strides, box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return DATTN_OK;
}

int launch_decode(const Plan &p, const void *Q, const void *K, const void *V, void *out, int B,
                  int H, int D, int S, const uint32_t *cur_pos, void *workspace,
                  cudaStream_t stream, const Paging &pg = Paging()) {
    DeviceInfo di;
    if (int st = device_info(&di)) return st;
    char *ws = static_cast<char *>(workspace);
    dattn::DecodeArgs a{};
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.out = out;
    a.cur_pos = cur_pos;
    const bool split = p.G > 1 && p.cluster == 0;  // partial states go through the workspace
    a.ws_prefix = split ? reinterpret_cast<long long *>(ws) : nullptr;
    a.ws_acc = split ? reinterpret_cast<float *>(ws + p.prefix_bytes) : nullptr;
    a.ws_ml = split ? reinterpret_cast<float2 *>(ws + p.prefix_bytes + p.acc_bytes) : nullptr;
    a.err = di.err_word;
    a.block_table = pg.table;
    a.num_pages = pg.num_pages;
    a.page_size = pg.page_size;
    a.max_pages = pg.max_pages;
    a.B = B;
    a.H = H;
    a.D = D;
    a.S = S;
    a.heads_per_cta = p.HG;
    a.head_groups = p.NHG;
    a.phases = p.PHI;
    a.stage_pos = p.P;
    a.stages = p.NST;
    a.partitions = p.G;
    a.active_warps = p.active_warps;
    a.merge_offset = p.merge_offset;
    a.bar_offset = p.bar_offset;
    a.qscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    // dense or paged cache: prefetch the first stages into L2 before the wait on
    // the previous kernel
    a.prefetch_positions = DATTN_PREFETCH_STAGES > 0 ? DATTN_PREFETCH_STAGES * p.P : 0;
    // a window of a few pages is read by one thread (7b in 16-position pages,
    // a one-page window: 0.1 us faster than the warp); larger windows by one
    // lane per page
    a.prefetch_lanes =
        pg.table != nullptr && a.prefetch_positions >= 4LL * pg.page_size ? 32 : 1;
    a.cluster = p.cluster;
    a.use_tmap = p.use_tmap;
    a.rec_offset = p.rec_offset;
    a.box_pos = p.box_pos;
    if (p.use_tmap) {
        const long long rows = pg.table != nullptr ? pg.num_pages * pg.page_size
                                                   : static_cast<long long>(B) * S;
        if (int st = encode_kv_box(&a.tmap_k, K, rows, H, D, p.HG, p.box_pos)) return st;
        if (int st = encode_kv_box(&a.tmap_v, V, rows, H, D, p.HG, p.box_pos)) return st;
    }
    cudaError_t e = dattn::launch_decode(a, p.v, p.smem, stream);
    if (e != cudaSuccess) return fail_cuda(e, "decode kernel launch");
    if (p.G > 1 && p.cluster == 0) {
        dattn::CombineArgs c{};
        c.ws_acc = a.ws_acc;
        c.ws_ml = a.ws_ml;
        c.ws_prefix = a.ws_prefix;
        c.cur_pos = cur_pos;
        c.out = out;
        c.B = B;
        c.H = H;
        c.D = D;
        c.S = S;
        c.heads_per_cta = p.HG;
        c.head_groups = p.NHG;
        c.partitions = p.G;
        c.chunk = p.combine_chunk;
        c.inflight = p.combine_inflight;
        e = dattn::launch_combine(c, stream);
        if (e != cudaSuccess) return fail_cuda(e, "combine kernel launch");
    }
    return DATTN_OK;
}

// Library-owned workspaces of dattn_decode_f16, one per (device, stream).
struct OwnedWorkspace {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mutex;
std::map<std::pair<int, cudaStream_t>, OwnedWorkspace> g_workspaces;

}  // namespace

namespace dattn {
int set_last_error(int status, const char *message) { return fail(status, "%s", message); }
}  // namespace dattn

extern "C" {

int dattn_version(void) { return kVersion; }

const char *dattn_status_string(int status) {
    switch (status) {
        case DATTN_OK: return "DATTN_OK";
        case DATTN_ERR_INVALID_ARG: return "DATTN_ERR_INVALID_ARG";
        case DATTN_ERR_UNSUPPORTED: return "DATTN_ERR_UNSUPPORTED";
        case DATTN_ERR_MISALIGNED: return "DATTN_ERR_MISALIGNED";
        case DATTN_ERR_WORKSPACE: return "DATTN_ERR_WORKSPACE";
        case DATTN_ERR_CUDA: return "DATTN_ERR_CUDA";
        case DATTN_ERR_TIMEOUT: return "DATTN_ERR_TIMEOUT";
        case DATTN_ERR_BAD_PAGE: return "DATTN_ERR_BAD_PAGE";
        case DATTN_ERR_BAD_POSITION: return "DATTN_ERR_BAD_POSITION";
        default: return "DATTN_ERR_UNKNOWN";
    }
}

const char *dattn_last_error(void) { return g_last_error.c_str(); }

namespace {
void fill_plan(const Plan &p, dattn_plan *plan) {
    plan->partitions = p.G;
    plan->heads_per_cta = p.HG;
    plan->head_groups = p.NHG;
    plan->stage_positions = p.P;
    plan->stages = p.NST;
    plan->threads_per_cta = dattn::decode_threads(p.v.nwc);
    plan->smem_bytes = p.smem;
    plan->ctas_per_sm = p.ctas_per_sm;
    plan->sm_count = p.sms;
    plan->workspace_bytes = p.ws_bytes;
    plan->cluster_size = p.cluster;
}

// The paged call's plan key: its page size, or -1 (the split plan) when the
// pool's rows do not fit the 32-bit row coordinate of a tensor box.
int paged_plan(int batch, int n_heads, int head_dim, int page_size, int max_pages,
               long long num_pages, int num_partitions, Plan *p) {
    if (page_size <= 0 || max_pages <= 0 || num_pages <= 0)
        return fail(DATTN_ERR_INVALID_ARG,
                    "page_size=%d, max_pages=%d and num_pages=%lld must be positive", page_size,
                    max_pages, num_pages);
    const long long cap = static_cast<long long>(page_size) * max_pages;
    if (cap > 0x7fffffffLL)
        return fail(DATTN_ERR_UNSUPPORTED, "page_size x max_pages = %lld exceeds 2^31 - 1", cap);
    const bool box_rows_ok = static_cast<double>(num_pages) * page_size < 2147483647.0;
    return make_plan(batch, n_heads, head_dim, static_cast<int>(cap), num_partitions,
                     box_rows_ok ? page_size : -1, p);
}
}  // namespace

int dattn_decode_plan(int batch, int n_heads, int head_dim, int seq_len, int num_partitions,
                      dattn_plan *plan) {
    if (plan == nullptr) return fail(DATTN_ERR_INVALID_ARG, "plan is NULL");
    Plan p;
    if (int st = make_plan(batch, n_heads, head_dim, seq_len, num_partitions, 0, &p)) return st;
    fill_plan(p, plan);
    return DATTN_OK;
}

int dattn_decode_paged_plan(int batch, int n_heads, int head_dim, int page_size, int max_pages,
                            long long num_pages, int num_partitions, dattn_plan *plan) {
    if (plan == nullptr) return fail(DATTN_ERR_INVALID_ARG, "plan is NULL");
    Plan p;
    if (int st = paged_plan(batch, n_heads, head_dim, page_size, max_pages, num_pages,
                            num_partitions, &p))
        return st;
    fill_plan(p, plan);
    return DATTN_OK;
}

int dattn_decode_workspace_bytes(int batch, int n_heads, int head_dim, int seq_len,
                                 int num_partitions, size_t *bytes) {
    if (bytes == nullptr) return fail(DATTN_ERR_INVALID_ARG, "bytes is NULL");
    // enough for the dense call and for the paged call of the same capacity and
    // any page size (a cache of few sequences may take the cluster plan, which
    // needs none; the split plan covers every paged call)
    Plan p, q;
    if (int st = make_plan(batch, n_heads, head_dim, seq_len, num_partitions, 0, &p)) return st;
    if (int st = make_plan(batch, n_heads, head_dim, seq_len, num_partitions, -1, &q)) return st;
    *bytes = std::max(p.ws_bytes, q.ws_bytes);
    return DATTN_OK;
}

int dattn_decode_f16_ex(const void *Q, const void *K_cache, const void *V_cache, void *out,
                        int batch, int n_heads, int head_dim, int seq_len,
                        const uint32_t *current_pos, void *workspace, size_t workspace_bytes,
                        int num_partitions, dattn_stream_t stream) {
    if (int st = check_tensor(Q, "Q")) return st;
    if (int st = check_tensor(K_cache, "K_cache")) return st;
    if (int st = check_tensor(V_cache, "V_cache")) return st;
    if (int st = check_tensor(out, "out")) return st;
    if (int st = check_cur_pos(current_pos)) return st;
    if (int st = validate_dims(batch, n_heads, head_dim, seq_len)) return st;
    if (num_partitions < 0)
        return fail(DATTN_ERR_INVALID_ARG, "num_partitions=%d must be >= 0", num_partitions);
    Plan p;
    if (int st = make_plan(batch, n_heads, head_dim, seq_len, num_partitions, 0, &p)) return st;
    if (p.ws_bytes > 0) {
        if (workspace == nullptr)
            return fail(DATTN_ERR_WORKSPACE, "workspace of %zu bytes required, got NULL",
                        p.ws_bytes);
        if (!aligned16(workspace))
            return fail(DATTN_ERR_WORKSPACE, "workspace is not 16-byte aligned");
        if (workspace_bytes < p.ws_bytes)
            return fail(DATTN_ERR_WORKSPACE, "workspace of %zu bytes required, got %zu",
                        p.ws_bytes, workspace_bytes);
    }
    return launch_decode(p, Q, K_cache, V_cache, out, batch, n_heads, head_dim, seq_len,
                         current_pos, workspace, reinterpret_cast<cudaStream_t>(stream));
}

int dattn_decode_f16(const void *Q, const void *K_cache, const void *V_cache, void *out,
                     int batch, int n_heads, int head_dim, int seq_len,
                     const uint32_t *current_pos, dattn_stream_t stream) {
    if (int st = check_tensor(Q, "Q")) return st;
    if (int st = check_tensor(K_cache, "K_cache")) return st;
    if (int st = check_tensor(V_cache, "V_cache")) return st;
    if (int st = check_tensor(out, "out")) return st;
    if (int st = check_cur_pos(current_pos)) return st;
    Plan p;
    if (int st = make_plan(batch, n_heads, head_dim, seq_len, 0, 0, &p)) return st;
    void *ws = nullptr;
    if (p.ws_bytes > 0) {
        int dev = 0;
        if (int st = current_device(&dev)) return st;
        std::lock_guard<std::mutex> lock(g_ws_mutex);
        OwnedWorkspace &w = g_workspaces[{dev, reinterpret_cast<cudaStream_t>(stream)}];
        if (w.bytes < p.ws_bytes) {
            cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
            cudaError_t e = cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cap);
            if (e != cudaSuccess) return fail_cuda(e, "cudaStreamIsCapturing");
            if (cap != cudaStreamCaptureStatusNone)
                return fail(DATTN_ERR_WORKSPACE,
                            "the library workspace of this stream must grow to %zu bytes, which "
                            "cannot happen while the stream is being recorded; make one call on "
                            "this stream before recording",
                            p.ws_bytes);
            e = cudaDeviceSynchronize();
            if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize (workspace grow)");
            if (w.ptr != nullptr) cudaFree(w.ptr);
            w.ptr = nullptr;
            w.bytes = 0;
            e = cudaMalloc(&w.ptr, p.ws_bytes);
            if (e != cudaSuccess) return fail_cuda(e, "cudaMalloc (workspace)");
            w.bytes = p.ws_bytes;
        }
        ws = w.ptr;
    }
    return launch_decode(p, Q, K_cache, V_cache, out, batch, n_heads, head_dim, seq_len,
                         current_pos, ws, reinterpret_cast<cudaStream_t>(stream));
}

int dattn_decode_paged_f16(const void *Q, const void *K_pages, const void *V_pages, void *out,
                           int batch, int n_heads, int head_dim, int page_size, int max_pages,
                           long long num_pages, const int32_t *block_table,
                           const uint32_t *current_pos, void *workspace, size_t workspace_bytes,
                           int num_partitions, dattn_stream_t stream) {
    if (int st = check_tensor(Q, "Q")) return st;
    if (int st = check_tensor(K_pages, "K_pages")) return st;
    if (int st = check_tensor(V_pages, "V_pages")) return st;
    if (int st = check_tensor(out, "out")) return st;
    if (int st = check_cur_pos(current_pos)) return st;
    if (block_table == nullptr) return fail(DATTN_ERR_INVALID_ARG, "block_table is NULL");
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) != 0)
        return fail(DATTN_ERR_MISALIGNED, "block_table is not 4-byte aligned");
    if (page_size <= 0 || max_pages <= 0 || num_pages <= 0)
        return fail(DATTN_ERR_INVALID_ARG,
                    "page_size=%d, max_pages=%d and num_pages=%lld must be positive", page_size,
                    max_pages, num_pages);
    const long long cap = static_cast<long long>(page_size) * max_pages;
    if (cap > 0x7fffffffLL)
        return fail(DATTN_ERR_UNSUPPORTED, "page_size x max_pages = %lld exceeds 2^31 - 1", cap);
    if (static_cast<double>(num_pages) * page_size * n_heads * head_dim > 4.0e18)
        return fail(DATTN_ERR_INVALID_ARG, "page pool is too large");
    const int S = static_cast<int>(cap);
    if (int st = validate_dims(batch, n_heads, head_dim, S)) return st;
    if (num_partitions < 0)
        return fail(DATTN_ERR_INVALID_ARG, "num_partitions=%d must be >= 0", num_partitions);
    Plan p;
    if (int st = paged_plan(batch, n_heads, head_dim, page_size, max_pages, num_pages,
                            num_partitions, &p))
        return st;
    if (p.ws_bytes > 0) {
        if (workspace == nullptr)
            return fail(DATTN_ERR_WORKSPACE, "workspace of %zu bytes required, got NULL",
                        p.ws_bytes);
        if (!aligned16(workspace))
            return fail(DATTN_ERR_WORKSPACE, "workspace is not 16-byte aligned");
        if (workspace_bytes < p.ws_bytes)
            return fail(DATTN_ERR_WORKSPACE, "workspace of %zu bytes required, got %zu",
                        p.ws_bytes, workspace_bytes);
    }
    Paging pg;
    pg.table = block_table;
    pg.num_pages = num_pages;
    pg.page_size = page_size;
    pg.max_pages = max_pages;
    return launch_decode(p, Q, K_pages, V_pages, out, batch, n_heads, head_dim, S, current_pos,
                         workspace, reinterpret_cast<cudaStream_t>(stream), pg);
}

int dattn_qk_f16(const void *Q, const void *K_cache, void *scores, int batch, int n_heads,
                 int head_dim, int seq_len, const uint32_t *current_pos,
                 dattn_stream_t stream) {
    if (int st = check_tensor(Q, "Q")) return st;
    if (int st = check_tensor(K_cache, "K_cache")) return st;
    if (int st = check_tensor(scores, "scores")) return st;
    if (int st = check_cur_pos(current_pos)) return st;
    if (int st = validate_dims(batch, n_heads, head_dim, seq_len)) return st;
    const cudaError_t e = dattn::launch_qk(Q, K_cache, scores, batch, n_heads, head_dim, seq_len,
                                           current_pos, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DATTN_OK : fail_cuda(e, "qk kernel launch");
}

int dattn_pv_f16(const void *scores, const void *V_cache, void *out, int batch, int n_heads,
                 int head_dim, int seq_len, dattn_stream_t stream) {
    if (int st = check_tensor(scores, "scores")) return st;
    if (int st = check_tensor(V_cache, "V_cache")) return st;
    if (int st = check_tensor(out, "out")) return st;
    if (int st = validate_dims(batch, n_heads, head_dim, seq_len)) return st;
    const cudaError_t e = dattn::launch_pv(scores, V_cache, out, batch, n_heads, head_dim,
                                           seq_len, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DATTN_OK : fail_cuda(e, "pv kernel launch");
}

namespace {
int rope_append(const void *q_new, const void *k_new, const void *v_new, void *q_out, void *K,
                void *V, int batch, int n_heads, int head_dim, int seq_len, int rope_dims,
                double rope_base, int traditional, const uint32_t *current_pos,
                const Paging &pg, cudaStream_t stream) {
    if (int st = check_tensor(q_new, "q_new")) return st;
    if (int st = check_tensor(k_new, "k_new")) return st;
    if (int st = check_tensor(v_new, "v_new")) return st;
    if (int st = check_tensor(q_out, "q_out")) return st;
    if (int st = check_tensor(K, "K cache")) return st;
    if (int st = check_tensor(V, "V cache")) return st;
    if (int st = check_cur_pos(current_pos)) return st;
    if (int st = validate_dims(batch, n_heads, head_dim, seq_len)) return st;
    if (rope_dims < 2 || rope_dims > head_dim || rope_dims % 2 != 0)
        return fail(DATTN_ERR_INVALID_ARG, "rope_dims=%d must be even and in [2, head_dim=%d]",
                    rope_dims, head_dim);
    if (!(rope_base > 1.0) || !std::isfinite(rope_base))
        return fail(DATTN_ERR_INVALID_ARG, "rope_base must be a finite number above 1");
    DeviceInfo di;
    if (int st = device_info(&di)) return st;
    dattn::RopeAppendArgs a{};
    a.q_new = q_new;
    a.k_new = k_new;
    a.v_new = v_new;
    a.q_out = q_out;
    a.K = K;
    a.V = V;
    a.block_table = pg.table;
    a.num_pages = pg.num_pages;
    a.page_size = pg.page_size;
    a.max_pages = pg.max_pages;
    a.cur_pos = current_pos;
    a.err = di.err_word;
    a.B = batch;
    a.H = n_heads;
    a.D = head_dim;
    a.S = seq_len;
    a.rope_dims = rope_dims;
    a.traditional = traditional ? 1 : 0;
    // The table depends on (rope_dims, rope_base) only; a decode loop passes the
    // same pair every step, so the last one is kept per thread (long double is
    // software arithmetic on some hosts).
    struct TurnTable {
        int rope_dims = 0;
        double base = 0.0;
        unsigned long long frac[dattn::kRopeMaxPairs];
    };
    thread_local TurnTable table;
    if (table.rope_dims != rope_dims || table.base != rope_base) {
        // theta_i <= 1 < 2 pi, so theta_i / (2 pi) is a fraction of a turn below
        // 1/6; scaled by 2^64 in extended precision it fits in 63 bits.
        const long double two_pi = 6.283185307179586476925286766559005768L;
        for (int i = 0; i < rope_dims / 2; ++i) {
            const double theta = std::pow(rope_base, -2.0 * i / rope_dims);
            table.frac[i] = static_cast<unsigned long long>(
                std::llroundl(std::ldexp(static_cast<long double>(theta) / two_pi, 64)));
        }
        table.rope_dims = rope_dims;
        table.base = rope_base;
    }
    std::memcpy(a.turn_frac, table.frac, sizeof(unsigned long long) * (rope_dims / 2));
    // about four CTAs per SM of work, at most 8 heads per CTA
    const long long bh = static_cast<long long>(batch) * n_heads;
    a.heads_per_cta = static_cast<int>(
        std::max(1LL, std::min(8LL, bh / (4LL * std::max(di.sms, 1)))));
    const cudaError_t e = dattn::launch_rope_append(a, stream);
    return e == cudaSuccess ? DATTN_OK : fail_cuda(e, "rope/append kernel launch");
}
}  // namespace

int dattn_rope_append_f16(const void *q_new, const void *k_new, const void *v_new, void *q_out,
                          void *K_cache, void *V_cache, int batch, int n_heads, int head_dim,
                          int seq_len, int rope_dims, double rope_base, int traditional,
                          const uint32_t *current_pos, dattn_stream_t stream) {
    return rope_append(q_new, k_new, v_new, q_out, K_cache, V_cache, batch, n_heads, head_dim,
                       seq_len, rope_dims, rope_base, traditional, current_pos, Paging(),
                       reinterpret_cast<cudaStream_t>(stream));
}

int dattn_rope_append_paged_f16(const void *q_new, const void *k_new, const void *v_new,
                                void *q_out, void *K_pages, void *V_pages, int batch,
                                int n_heads, int head_dim, int page_size, int max_pages,
                                long long num_pages, const int32_t *block_table, int rope_dims,
                                double rope_base, int traditional, const uint32_t *current_pos,
                                dattn_stream_t stream) {
    if (block_table == nullptr) return fail(DATTN_ERR_INVALID_ARG, "block_table is NULL");
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) != 0)
        return fail(DATTN_ERR_MISALIGNED, "block_table is not 4-byte aligned");
    if (page_size <= 0 || max_pages <= 0 || num_pages <= 0)
        return fail(DATTN_ERR_INVALID_ARG,
                    "page_size=%d, max_pages=%d and num_pages=%lld must be positive", page_size,
                    max_pages, num_pages);
    const long long cap = static_cast<long long>(page_size) * max_pages;
    if (cap > 0x7fffffffLL)
        return fail(DATTN_ERR_UNSUPPORTED, "page_size x max_pages = %lld exceeds 2^31 - 1", cap);
    Paging pg;
    pg.table = block_table;
    pg.num_pages = num_pages;
    pg.page_size = page_size;
    pg.max_pages = max_pages;
    return rope_append(q_new, k_new, v_new, q_out, K_pages, V_pages, batch, n_heads, head_dim,
                       static_cast<int>(cap), rope_dims, rope_base, traditional, current_pos, pg,
                       reinterpret_cast<cudaStream_t>(stream));
}

int dattn_softmax_f32(const float *x, float *out, long long rows, int cols,
                      dattn_stream_t stream) {
    if (x == nullptr || out == nullptr) return fail(DATTN_ERR_INVALID_ARG, "x or out is NULL");
    if ((reinterpret_cast<uintptr_t>(x) & 3u) || (reinterpret_cast<uintptr_t>(out) & 3u))
        return fail(DATTN_ERR_MISALIGNED, "x and out must be 4-byte aligned");
    if (rows <= 0 || cols <= 0)
        return fail(DATTN_ERR_INVALID_ARG, "rows=%lld and cols=%d must be positive", rows, cols);
    if (static_cast<double>(rows) * cols > 4.0e18)
        return fail(DATTN_ERR_INVALID_ARG, "matrix is too large");
    if (cols > 1024 && rows > 0x7fffffffLL)
        return fail(DATTN_ERR_UNSUPPORTED, "at most 2^31-1 rows of more than 1024 columns");
    DeviceInfo di;
    if (int st = device_info(&di)) return st;
    const cudaError_t e = dattn::launch_softmax(x, out, rows, cols, di.err_word,
                                                reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DATTN_OK : fail_cuda(e, "softmax kernel launch");
}

int dattn_selftest_wait_timeout(dattn_stream_t stream) {
    DeviceInfo di;
    if (int st = device_info(&di)) return st;
    const cudaError_t e =
        dattn::launch_wait_timeout_selftest(di.err_word, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DATTN_OK : fail_cuda(e, "self-test kernel launch");
}

struct dattn_batch {
    cudaGraphExec_t exec = nullptr;
    size_t nodes = 0;
};

int dattn_batch_begin(dattn_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (s == nullptr)
        return fail(DATTN_ERR_INVALID_ARG, "batches need a created stream, not the legacy default");
    const cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    return e == cudaSuccess ? DATTN_OK : fail_cuda(e, "cudaStreamBeginCapture");
}

int dattn_batch_end(dattn_stream_t stream, dattn_batch **batch) {
    if (batch == nullptr) return fail(DATTN_ERR_INVALID_ARG, "batch is NULL");
    *batch = nullptr;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(s, &graph);
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamEndCapture");
    dattn_batch *b = new dattn_batch();
    e = cudaGraphGetNodes(graph, nullptr, &b->nodes);
    if (e == cudaSuccess) e = cudaGraphInstantiate(&b->exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
        delete b;
        return fail_cuda(e, "cudaGraphInstantiate");
    }
    *batch = b;
    return DATTN_OK;
}

int dattn_batch_launch(const dattn_batch *batch, dattn_stream_t stream) {
    if (batch == nullptr || batch->exec == nullptr)
        return fail(DATTN_ERR_INVALID_ARG, "batch is NULL");
    const cudaError_t e = cudaGraphLaunch(batch->exec, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DATTN_OK : fail_cuda(e, "cudaGraphLaunch");
}

long long dattn_batch_nodes(const dattn_batch *batch) {
    return batch == nullptr ? -1 : static_cast<long long>(batch->nodes);
}

int dattn_batch_destroy(dattn_batch *batch) {
    if (batch == nullptr) return DATTN_OK;
    cudaError_t e = cudaSuccess;
    if (batch->exec != nullptr) e = cudaGraphExecDestroy(batch->exec);
    delete batch;
    return e == cudaSuccess ? DATTN_OK : fail_cuda(e, "cudaGraphExecDestroy");
}

int dattn_device_error(int clear) {
    DeviceInfo di;
    if (int st = device_info(&di)) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceSynchronize");
    unsigned word = 0;
    e = cudaMemcpy(&word, di.err_word, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpy (error word)");
    if (clear && word != 0) {
        e = cudaMemset(di.err_word, 0, sizeof(unsigned));
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return fail_cuda(e, "cudaMemset (error word)");
    }
    const unsigned input_bits = dattn::kErrPageIndex | dattn::kErrAppendPosition;
    if (word & ~input_bits)
        return fail(DATTN_ERR_TIMEOUT, "a kernel gave up on a pipeline wait (code 0x%x)", word);
    if (word & dattn::kErrPageIndex)
        return fail(DATTN_ERR_BAD_PAGE,
                    "a block-table entry of a live position was outside [0, num_pages)");
    if (word & dattn::kErrAppendPosition)
        return fail(DATTN_ERR_BAD_POSITION, "an append position was outside the cache");
    return DATTN_OK;
}

}  // extern "C"
