// cfa_tile.cuh -- shared-memory tile helpers used by every kernel of the
// library: bf16 packing, the stage-ring cursor, and the CUDA-core GEMV over a
// [rows x 64] bf16 weight tile with its fixed-order cross-warp reduction.
#pragma once

#include <cuda_bf16.h>

#include "cfa_device.cuh"
#include "cfa_internal.h"

namespace cfa {

__device__ __forceinline__ void unpack8_bf16(uint4 v, float *f) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}

// CPL consecutive bf16 weights from shared memory, widened to fp32.
template <int CPL>
__device__ __forceinline__ void load_weights(const uint8_t *p, float (&w)[CPL]) {
    if constexpr (CPL == 8) {
        unpack8_bf16(*reinterpret_cast<const uint4 *>(p), w);
    } else if constexpr (CPL == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        w[0] = bf16_lo(v.x); w[1] = bf16_hi(v.x); w[2] = bf16_lo(v.y); w[3] = bf16_hi(v.y);
    } else {
        const uint32_t v = *reinterpret_cast<const uint32_t *>(p);
        w[0] = bf16_lo(v); w[1] = bf16_hi(v);
    }
}

__device__ __forceinline__ float load_input(const uint16_t *p) { return bf16_bits(*p); }
__device__ __forceinline__ float load_input(const float *p) { return *p; }

// Position in the stage ring: stage index and the parity of the current pass.
struct RingCursor {
    int stage = 0;
    uint32_t phase = 0;
    bool wrapped = false;  // every stage has been filled at least once
    __device__ __forceinline__ void advance(int ns) {
        if (++stage == ns) {
            stage = 0;
            phase ^= 1u;
            wrapped = true;
        }
    }
};

// Columns each lane owns in a 64-column weight tile: wide vectors for small
// batches, narrow ones when the per-lane accumulators would not fit.
template <int MAXB>
struct GemvShape {
    static constexpr int CPL = MAXB <= 2 ? 8 : (MAXB <= 4 ? 4 : 2);  // columns per lane
    static constexpr int LPR = kTileCols / CPL;                      // lanes per tile row
    static constexpr int RPI = 32 / LPR;                             // rows per warp access
};

// acc[b][c] += sum over this warp's rows of in[b][row] * W[row][cg*CPL + c].
// Rows [warp*rpw, (warp+1)*rpw) of the tile belong to this warp; the lane
// takes every RPI-th of them. The tile is [rows][64] bf16 (128-byte rows).
template <int MAXB, typename InT>
__device__ __forceinline__ void gemv_tile(const uint8_t *tile, int rpw, const InT *in,
                                          int in_stride, int B, int warp, int lane,
                                          float (&acc)[MAXB][GemvShape<MAXB>::CPL]) {
    using S = GemvShape<MAXB>;
    const int cg = lane % S::LPR, rq = lane / S::LPR;
    const int r0 = warp * rpw;
#pragma unroll 4
    for (int j = rq; j < rpw; j += S::RPI) {
        const int row = r0 + j;
        float w[S::CPL];
        load_weights<S::CPL>(tile + row * (kTileCols * 2) + cg * (S::CPL * 2), w);
#pragma unroll
        for (int b = 0; b < MAXB; ++b) {
            if (b < B) {
                const float xv = load_input(in + b * in_stride + row);
#pragma unroll
                for (int c = 0; c < S::CPL; ++c) acc[b][c] = fmaf(xv, w[c], acc[b][c]);
            }
        }
    }
}

// Sums the per-lane partials of all compute warps into dst[b*dst_stride + c]
// (c < 64) in a fixed order. Uses `scratch` ([8][B][64] floats) and two
// compute-warp barriers.
template <int MAXB>
__device__ __forceinline__ void gemv_reduce(float (&acc)[MAXB][GemvShape<MAXB>::CPL], int B,
                                            int warp, int lane, int tid, float *scratch,
                                            float *dst, int dst_stride) {
    using S = GemvShape<MAXB>;
    const int cg = lane % S::LPR, rq = lane / S::LPR;
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
#pragma unroll
        for (int c = 0; c < S::CPL; ++c) {
#pragma unroll
            for (int off = S::LPR; off < 32; off <<= 1)
                acc[b][c] += __shfl_xor_sync(0xffffffffu, acc[b][c], off);
        }
    }
    if (rq == 0) {
#pragma unroll
        for (int b = 0; b < MAXB; ++b)
            if (b < B) {
#pragma unroll
                for (int c = 0; c < S::CPL; ++c)
                    scratch[(warp * B + b) * kTileCols + cg * S::CPL + c] = acc[b][c];
            }
    }
    compute_bar<kComputeThreads>();
    for (int idx = tid; idx < B * kTileCols; idx += kComputeThreads) {
        const int b = idx / kTileCols, c = idx % kTileCols;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < kComputeWarps; ++w) sum += scratch[(w * B + b) * kTileCols + c];
        dst[b * dst_stride + c] = sum;
    }
    compute_bar<kComputeThreads>();
}

}  // namespace cfa
