// Instantiations of the fused kernel for head_dim 128.
#include "cfa_kernel.cuh"
#include "cfa_merge.cuh"

namespace cfa {

const void *fused_kernel_d128(int maxb) {
    switch (maxb) {
        case 1: return reinterpret_cast<const void *>(&fused_decode_kernel<128, 1>);
        case 2: return reinterpret_cast<const void *>(&fused_decode_kernel<128, 2>);
        case 4: return reinterpret_cast<const void *>(&fused_decode_kernel<128, 4>);
        case 8: return reinterpret_cast<const void *>(&fused_decode_kernel<128, 8>);
        case 16: return reinterpret_cast<const void *>(&fused_decode_kernel<128, 16>);
        default: return nullptr;
    }
}

const void *head_merge_kernel_ptr() { return reinterpret_cast<const void *>(&head_merge_kernel); }

// Exercises mbar_wait_bounded on a barrier nothing arrives on.
__global__ void selftest_wait_kernel(unsigned *status, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int timed_out;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        timed_out = 0;
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait_bounded<false>(smem_addr(&bar), 0, timeout_ns, &timed_out, status, kSiteSelftest);
}

const void *selftest_wait_kernel_ptr() {
    return reinterpret_cast<const void *>(&selftest_wait_kernel);
}

}  // namespace cfa
