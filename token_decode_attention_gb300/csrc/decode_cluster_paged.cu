// decode_cluster_paged.cu -- the instances of the fused decode kernel
// (decode_kernel.cuh) for the cluster plan over a paged cache: the CTAs of a
// cluster split the live positions of a (sequence, head group) at page
// boundaries, copy a head group's rows of each whole page as one tensor box,
// and merge their partial states through distributed shared memory.
#include "decode_kernel.cuh"

namespace dattn {

const void *decode_cluster_paged_variant_fn(DecodeVariant v) {
    return variant_fn_of<kModeClusterPaged>(v);
}

}  // namespace dattn
