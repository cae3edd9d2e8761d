// Instantiations of the fused kernel for head_dim 64.
#include "cfa_kernel.cuh"

namespace cfa {

const void *fused_kernel_d64(int maxb) {
    switch (maxb) {
        case 1: return reinterpret_cast<const void *>(&fused_decode_kernel<64, 1>);
        case 2: return reinterpret_cast<const void *>(&fused_decode_kernel<64, 2>);
        case 4: return reinterpret_cast<const void *>(&fused_decode_kernel<64, 4>);
        case 8: return reinterpret_cast<const void *>(&fused_decode_kernel<64, 8>);
        case 16: return reinterpret_cast<const void *>(&fused_decode_kernel<64, 16>);
        default: return nullptr;
    }
}

}  // namespace cfa
