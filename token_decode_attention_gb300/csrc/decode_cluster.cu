// decode_cluster.cu -- the instances of the fused decode kernel
// (decode_kernel.cuh) for the cluster plan over a dense cache: one
// thread-block cluster per (sequence, head group), partial states merged
// through distributed shared memory.  Kept apart from the other modes'
// instances so that they compile in parallel.
#include "decode_kernel.cuh"

namespace dattn {

const void *decode_cluster_variant_fn(DecodeVariant v) { return variant_fn_of<kModeCluster>(v); }

}  // namespace dattn
