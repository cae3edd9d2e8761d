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

// Copies n16 16-byte words src -> dst: the host entry point's transfer of x
// from, and of out to, device-mapped pinned host memory (zero-copy). Runs
// between the fused kernel's neighbours on the stream with programmatic
// dependent launch: it waits for the previous kernel before touching memory.
__global__ void __launch_bounds__(256) copy16_kernel(const uint4 *__restrict__ src,
                                                     uint4 *__restrict__ dst, int n16) {
    grid_dependency_wait();
    grid_dependents_launch();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += gridDim.x * blockDim.x)
        dst[i] = src[i];
}

const void *copy16_kernel_ptr() { return reinterpret_cast<const void *>(&copy16_kernel); }

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
