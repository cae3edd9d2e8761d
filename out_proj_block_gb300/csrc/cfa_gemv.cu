// Instantiations of the decoder-layer kernels around the attention block.
#include "cfa_gemv.cuh"
#include "cfa_gemv_mma.cuh"

namespace cfa {

const void *gemv_kernel(int mode, int maxb, bool wide) {
    // 32 KB units are built for single-row batches only (the CUDA-core GEMV's
    // batch unless a plan forces this path for more rows).
#define CFA_GEMV_CASES(M)                                                                   \
    if (wide) return maxb == 1 ? reinterpret_cast<const void *>(&gemv_streamk_kernel<1, M, true>) \
                               : nullptr;                                                   \
    switch (maxb) {                                                                         \
        case 1: return reinterpret_cast<const void *>(&gemv_streamk_kernel<1, M, false>);   \
        case 2: return reinterpret_cast<const void *>(&gemv_streamk_kernel<2, M, false>);   \
        case 4: return reinterpret_cast<const void *>(&gemv_streamk_kernel<4, M, false>);   \
        case 8: return reinterpret_cast<const void *>(&gemv_streamk_kernel<8, M, false>);   \
        case 16: return reinterpret_cast<const void *>(&gemv_streamk_kernel<16, M, false>); \
        default: return nullptr;                                                            \
    }
    if (mode == kGemvSwiGLU) { CFA_GEMV_CASES(kGemvSwiGLU) }
    if (mode == kGemvResidual) { CFA_GEMV_CASES(kGemvResidual) }
    if (mode == kGemvPlain) { CFA_GEMV_CASES(kGemvPlain) }
    if (mode == kGemvNormPlain) { CFA_GEMV_CASES(kGemvNormPlain) }
#undef CFA_GEMV_CASES
    return nullptr;
}

const void *gemv_mma_kernel_ptr(int mode) {
    switch (mode) {
        case kGemvSwiGLU: return reinterpret_cast<const void *>(&gemv_mma_kernel<kGemvSwiGLU>);
        case kGemvResidual: return reinterpret_cast<const void *>(&gemv_mma_kernel<kGemvResidual>);
        case kGemvPlain: return reinterpret_cast<const void *>(&gemv_mma_kernel<kGemvPlain>);
        case kGemvNormPlain: return reinterpret_cast<const void *>(&gemv_mma_kernel<kGemvNormPlain>);
        default: return nullptr;
    }
}

const void *rmsnorm_kernel_ptr() { return reinterpret_cast<const void *>(&rmsnorm_kernel); }
const void *advance_kernel_ptr() { return reinterpret_cast<const void *>(&advance_positions_kernel); }

}  // namespace cfa
