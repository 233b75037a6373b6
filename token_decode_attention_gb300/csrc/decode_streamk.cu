// decode_streamk.cu -- launchers of the fused decode kernel
// (decode_kernel.cuh) and the instances of its split (stream-K) plan.  The
// cluster plan's instances are in decode_cluster.cu (dense caches) and
// decode_cluster_paged.cu (paged caches).
#include "decode_kernel.cuh"

namespace dattn {

__device__ unsigned g_device_error = 0;

// the cluster plan's instances (decode_cluster.cu, decode_cluster_paged.cu)
const void *decode_cluster_variant_fn(DecodeVariant v);
const void *decode_cluster_paged_variant_fn(DecodeVariant v);

namespace {

const void *variant_fn(DecodeVariant v, int mode) {
    switch (mode) {
        case kModeSplit: return variant_fn_of<kModeSplit>(v);
        case kModeCluster: return decode_cluster_variant_fn(v);
        case kModeClusterPaged: return decode_cluster_paged_variant_fn(v);
        default: return nullptr;
    }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, DecodeVariant v, int smem, cudaStream_t stream) {
    const int mode = a.cluster == 0 ? kModeSplit
                                    : (a.block_table != nullptr ? kModeClusterPaged : kModeCluster);
    const void *fn = variant_fn(v, mode);
    if (fn == nullptr || a.partitions <= 0) return cudaErrorInvalidValue;
    void *args[] = {const_cast<DecodeArgs *>(&a)};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.partitions));
    cfg.blockDim = dim3(decode_threads(v.nwc));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    // the kernel waits (griddepcontrol.wait) before its first global-memory access
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.cluster > 0) {
        if (a.cluster > kMaxCluster || a.partitions % a.cluster != 0) return cudaErrorInvalidValue;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(a.cluster);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t decode_occupancy(DecodeVariant v, int smem, int *ctas_per_sm) {
    const void *fn = variant_fn(v, kModeSplit);
    if (fn == nullptr) return cudaErrorInvalidValue;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, fn, decode_threads(v.nwc),
                                                         static_cast<size_t>(smem));
}

cudaError_t decode_max_clusters(DecodeVariant v, int smem, int cluster, bool paged, int *clusters) {
    const void *fn = variant_fn(v, paged ? kModeClusterPaged : kModeCluster);
    if (fn == nullptr || cluster < 1 || cluster > kMaxCluster) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cluster));
    cfg.blockDim = dim3(decode_threads(v.nwc));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(clusters, fn, &cfg);
}

cudaError_t decode_configure_smem(int max_smem) {
    static const DecodeVariant variants[] = {
        {1, 1, 1, 8},  {1, 1, 2, 8},  {2, 1, 1, 8},  {2, 1, 2, 8},  {4, 1, 1, 8},
        {4, 1, 2, 8},  {8, 1, 1, 8},  {8, 1, 2, 8},  {8, 2, 1, 8},  {16, 2, 1, 8},
        {1, 1, 1, 16}, {1, 1, 2, 16}, {2, 1, 1, 16}, {2, 1, 2, 16}, {4, 1, 1, 16},
        {4, 1, 2, 16}, {8, 1, 1, 16}, {8, 1, 2, 16}, {8, 2, 1, 16}, {16, 2, 1, 16}};
    for (const DecodeVariant &v : variants) {
        for (const int mode : {kModeSplit, kModeCluster, kModeClusterPaged}) {
            const void *fn = variant_fn(v, mode);
            // static and dynamic shared memory together may not exceed the opt-in limit
            cudaFuncAttributes attr{};
            cudaError_t e = cudaFuncGetAttributes(&attr, fn);
            if (e != cudaSuccess) return e;
            const int dyn = max_smem - static_cast<int>(attr.sharedSizeBytes);
            e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
            if (e != cudaSuccess) return e;
            // the cluster plan launches clusters of up to 16 CTAs
            if (mode != kModeSplit)
                e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

cudaError_t device_error_word(unsigned **ptr) {
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_device_error);
}

}  // namespace dattn
