// cfa_merge.cuh -- the cross-head merge as its own kernel, for batches whose
// per-head output-projection partials are too large for one block to sum at
// the end of the fused kernel.
//
// Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命" (ClusterFusion
// framework analysis), written [CF §n]. The page adds every head's partial
// output projection into the result with atomicAdd [CF §3.2]; here the sum
// runs in a fixed head order, so results are bitwise reproducible.
#pragma once

#include <cuda_bf16.h>

#include "cfa_device.cuh"
#include "cfa_internal.h"
#include "cfa_tile.cuh"

namespace cfa {

// out[b][c] = bf16(resid[b][c] + sum over heads of partials[head][b][c]) for
// 4 columns per item: the heads in two halves [0, nh/2) and [nh/2, nh), each
// summed in ascending order by one of a pair of threads, then half 0 + half 1.
// Launched after the fused kernel on the same stream; it may start early
// (programmatic dependent launch) and waits for that kernel before reading.
__global__ void __launch_bounds__(kMergeThreads)
head_merge_kernel(const float *__restrict__ partials, int nh, int B, int H,
                  const uint16_t *__restrict__ resid, uint16_t *__restrict__ out) {
    grid_dependency_wait();
    grid_dependents_launch();
    const size_t head_stride = static_cast<size_t>(B) * H;
    const int items = B * (H / 4);
    const int idx = blockIdx.x * kMergeItemsPerBlock + (threadIdx.x >> 1);
    const int half = threadIdx.x & 1;
    const int hh = (nh + 1) / 2;
    const int e0 = half * hh, e1 = min(nh, e0 + hh);
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    if (idx < items) {
        const float *src = partials + 4 * static_cast<size_t>(idx);
        for (int e = e0; e < e1; e += 16) {
            float4 v[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
                v[k] = e + k < e1 ? __ldcg(reinterpret_cast<const float4 *>(src + (e + k) * head_stride))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                sum.x += v[k].x;
                sum.y += v[k].y;
                sum.z += v[k].z;
                sum.w += v[k].w;
            }
        }
    }
    float4 other;
    other.x = __shfl_xor_sync(0xffffffffu, sum.x, 1);
    other.y = __shfl_xor_sync(0xffffffffu, sum.y, 1);
    other.z = __shfl_xor_sync(0xffffffffu, sum.z, 1);
    other.w = __shfl_xor_sync(0xffffffffu, sum.w, 1);
    if (half != 0 || idx >= items) return;
    float4 tot = make_float4(sum.x + other.x, sum.y + other.y, sum.z + other.z, sum.w + other.w);
    if (resid) {
        const uint2 rv = *reinterpret_cast<const uint2 *>(resid + 4 * static_cast<size_t>(idx));
        tot.x += bf16_lo(rv.x);
        tot.y += bf16_hi(rv.x);
        tot.z += bf16_lo(rv.y);
        tot.w += bf16_hi(rv.y);
    }
    uint2 packed;
    packed.x = pack2_bf16(tot.x, tot.y);
    packed.y = pack2_bf16(tot.z, tot.w);
    *reinterpret_cast<uint2 *>(out + 4 * static_cast<size_t>(idx)) = packed;
}

}  // namespace cfa
