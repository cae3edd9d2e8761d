// Instantiations of the multi-head latent attention core kernel (see cfa_mla.cuh).
#include "cfa_mla.cuh"

namespace cfa {

// heads_per_cluster <= 8: one head scored per warp; 16: two.
const void *mla_kernel_ptr(int heads_per_cluster) {
    if (heads_per_cluster <= kComputeWarps)
        return reinterpret_cast<const void *>(&mla_attention_kernel<1>);
    if (heads_per_cluster == 2 * kComputeWarps)
        return reinterpret_cast<const void *>(&mla_attention_kernel<2>);
    return nullptr;
}

}  // namespace cfa
