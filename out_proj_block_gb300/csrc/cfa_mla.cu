// The multi-head latent attention core kernel (see cfa_mla.cuh).
#include "cfa_mla.cuh"

namespace cfa {

// Any head-group size up to 16 runs the same kernel (the MMA's N is 16).
const void *mla_kernel_ptr(int heads_per_cluster) {
    if (heads_per_cluster < 2 || heads_per_cluster > kMlaMaxHG) return nullptr;
    return reinterpret_cast<const void *>(&mla_attention_kernel);
}

}  // namespace cfa
