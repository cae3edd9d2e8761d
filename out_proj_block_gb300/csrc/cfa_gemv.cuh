// cfa_gemv.cuh -- the kernels that sit around the fused attention block in a
// decoder layer of the decode loop: a stream-K GEMV for the MLP projections
// (RMSNorm + gate/up + SwiGLU in one kernel, down projection + residual in
// another), a row RMSNorm, and the position counter of the loop.
//
// Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命" (ClusterFusion
// framework analysis), written [CF §n]. The page measures whole-model time
// per token of a Llama2-7B decoder [CF §3.3, §5.1] but describes only the
// attention block; the MLP and norms follow the Llama2 layer arrangement.
//
// The GEMV is HBM-bound at small batch: every weight byte is read once per
// token. Its work is cut into units of one 128-column tile x `rows` weight
// rows (16 KB of weights; 32 KB for a single batch row where K allows), and
// the units, taken tile by tile, are split evenly
// over a persistent grid -- so every SM streams the same number of bytes
// whatever the matrix shape ("stream-K"). Tiles are 128 columns (256 bytes of
// each weight row) because blocks stream different rows of the matrix at the
// same time: with 128-byte rows HBM delivered about 4.5 TB/s for this access
// pattern, with 256-byte rows about 6.6 TB/s (steady state, measured). A block
// accumulates its units of one tile in registers; a tile shared by several blocks is finished by the last of them
// to arrive (release/acquire counter), which sums the fp32 partials in block
// order -- deterministic, no float atomics. Weight tiles and input rows are
// streamed by one load warp through a ring of shared-memory stages with TMA,
// as in the attention kernel.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "cfa_device.cuh"
#include "cfa_internal.h"
#include "cfa_layer_params.h"
#include "cfa_tile.cuh"

namespace cfa {

// Units [0, U) split over P blocks: block i owns [floor(U i / P), floor(U (i+1) / P)).
__device__ __forceinline__ int unit_begin(long long i, long long U, long long P) {
    return static_cast<int>((U * i) / P);
}
// The block that owns unit u (the largest i with unit_begin(i) <= u).
__device__ __forceinline__ int unit_owner(long long u, long long U, long long P) {
    return static_cast<int>(((u + 1) * P - 1) / U);
}

// Warps split a [rows x 128] tile into two 64-column halves x four row
// quarters; each warp keeps the partial sums of its half over its rows.
constexpr int kGemvHalves = kGemvTileCols / kTileCols;
constexpr int kWarpsPerHalf = kComputeWarps / kGemvHalves;

// acc[b][c] += sum_j in[b * in_stride + j] * W[r0 + j][cg * CPL + c], j < RPW,
// over the rows of this warp; `half_tile` points at the warp's 64 columns of
// the tile (rows of `row_bytes` bytes). The lane takes every RPI-th row.
template <int MAXB, int RPW, typename InT>
__device__ __forceinline__ void gemv_rows(const uint8_t *half_tile, int row_bytes, int r0,
                                          const InT *in, int in_stride, int B, int lane,
                                          float (&acc)[MAXB][GemvShape<MAXB>::CPL]) {
    using S = GemvShape<MAXB>;
    const int cg = lane % S::LPR, rq = lane / S::LPR;
#pragma unroll
    for (int jj = 0; jj < RPW; jj += S::RPI) {
        const int j = jj + rq;
        float w[S::CPL];
        load_weights<S::CPL>(half_tile + (r0 + j) * row_bytes + cg * (S::CPL * 2), w);
#pragma unroll
        for (int b = 0; b < MAXB; ++b) {
            if (b < B) {
                const float xv = load_input(in + b * in_stride + j);
#pragma unroll
                for (int c = 0; c < S::CPL; ++c) acc[b][c] = fmaf(xv, w[c], acc[b][c]);
            }
        }
    }
}

// Sums the partials of the four warps of each column half, in warp order,
// into dst[b * dst_stride + col] for col < 128. Two compute-warp barriers.
template <int MAXB>
__device__ __forceinline__ void gemv_reduce_halves(float (&acc)[MAXB][GemvShape<MAXB>::CPL], int B,
                                                   int warp, int lane, int tid, float *scratch,
                                                   float *dst, int dst_stride) {
    using S = GemvShape<MAXB>;
    const int cg = lane % S::LPR, rq = lane / S::LPR;
#pragma unroll
    for (int b = 0; b < MAXB; ++b)
#pragma unroll
        for (int c = 0; c < S::CPL; ++c)
#pragma unroll
            for (int off = S::LPR; off < 32; off <<= 1)
                acc[b][c] += __shfl_xor_sync(0xffffffffu, acc[b][c], off);
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
    for (int idx = tid; idx < B * kGemvTileCols; idx += kComputeThreads) {
        const int b = idx / kGemvTileCols, col = idx % kGemvTileCols;
        const int half = col / kTileCols, c = col % kTileCols;
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < kWarpsPerHalf; ++q)
            sum += scratch[((half * kWarpsPerHalf + q) * B + b) * kTileCols + c];
        dst[b * dst_stride + col] = sum;
    }
    compute_bar<kComputeThreads>();
}

// The blocks that own units of tile t: [i_first, i_first + n_t).
__device__ __forceinline__ void gemv_tile_owners(const GemvParams &p, int t, int &i_first, int &n_t) {
    const long long U = p.units, P = p.nblocks;
    i_first = unit_owner(static_cast<long long>(t) * p.chunks, U, P);
    n_t = unit_owner(static_cast<long long>(t + 1) * p.chunks - 1, U, P) - i_first + 1;
}

// Floats per batch row of a tile partial: one or two matrices of 128 columns.
template <int MODE>
__host__ __device__ constexpr int gemv_nw() { return (MODE == kGemvSwiGLU ? 2 : 1) * kGemvTileCols; }

// This block's workspace slot for the partial of its k-th tile.
template <int MODE>
__device__ __forceinline__ float4 *gemv_slot(const GemvParams &p, int k) {
    return reinterpret_cast<float4 *>(
        p.partials + (static_cast<size_t>(blockIdx.x) * p.max_tiles + k) * p.B * gemv_nw<MODE>());
}

// Output columns [t*128, t*128 + 128) of tile t, as quads (b, c..c+3).
// A tile shared by n_t blocks is the sum of their fp32 partials in one
// fixed order, whichever warps compute it: sub_s = p_s + p_{s+4} + ... for
// s < 4 (ascending), total = (sub_0 + sub_1) + (sub_2 + sub_3), the four
// subs held by four adjacent lanes. This block's own partial is read from
// its tile buffer `tl`; a tile owned by one block is just that buffer.
// nthr threads (a multiple of 32) take the work items idx = (quad, s),
// ITEMS of them at a time with their loads in flight together (more items,
// more registers).
template <int MODE, int ITEMS>
__device__ __forceinline__ void gemv_finish_quads(const GemvParams &p, int t, int i_first, int n_t,
                                                  const float *tl, int ti, int nthr) {
    constexpr bool DUAL = MODE == kGemvSwiGLU;
    constexpr int NW = gemv_nw<MODE>();
    constexpr int V = 4;
    const int B = p.B;
    const int total = B * kGemvTileCols;  // a multiple of nthr: uniform trip counts
    const long long U = p.units, P = p.nblocks;
    // nthr is a multiple of 4, so every item of this thread has the same sub
    // (the lane within its quad): the partials it sums are the same blocks.
    const int sub = ti & 3;
    for (int idx0 = ti; idx0 < total; idx0 += ITEMS * nthr) {
        float4 a0[ITEMS], a1[ITEMS];
#pragma unroll
        for (int q = 0; q < ITEMS; ++q) {
            a0[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            a1[q] = a0[q];
        }
        // blocks j = sub, sub + 4, ... in ascending order; for each, the
        // partials of all ITEMS items are requested before any is used
        for (int j = sub; j < n_t; j += 4) {
            const int i = i_first + j;
            const bool own = i == static_cast<int>(blockIdx.x);
            const float *src = own ? tl
                                   : p.partials + (static_cast<size_t>(i) * p.max_tiles +
                                                   (t - unit_begin(i, U, P) / p.chunks)) * B * NW;
            float4 v0[ITEMS], v1[ITEMS];
#pragma unroll
            for (int q = 0; q < ITEMS; ++q) {
                const int idx = idx0 + q * nthr;
                const int o = idx >> 2;
                const int b = o / (kGemvTileCols / V), c = V * (o % (kGemvTileCols / V));
                v0[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                v1[q] = v0[q];
                if (idx < total) {
                    const float *e = src + b * NW + c;
                    if (own) {
                        v0[q] = *reinterpret_cast<const float4 *>(e);
                        if constexpr (DUAL) v1[q] = *reinterpret_cast<const float4 *>(e + kGemvTileCols);
                    } else {
                        v0[q] = __ldcg(reinterpret_cast<const float4 *>(e));
                        if constexpr (DUAL) v1[q] = __ldcg(reinterpret_cast<const float4 *>(e + kGemvTileCols));
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < ITEMS; ++q) {
                a0[q].x += v0[q].x; a0[q].y += v0[q].y; a0[q].z += v0[q].z; a0[q].w += v0[q].w;
                if constexpr (DUAL) {
                    a1[q].x += v1[q].x; a1[q].y += v1[q].y; a1[q].z += v1[q].z; a1[q].w += v1[q].w;
                }
            }
        }
#pragma unroll
        for (int q = 0; q < ITEMS; ++q) {
#pragma unroll
            for (int off = 1; off <= 2; off <<= 1) {
                a0[q].x += __shfl_xor_sync(0xffffffffu, a0[q].x, off);
                a0[q].y += __shfl_xor_sync(0xffffffffu, a0[q].y, off);
                a0[q].z += __shfl_xor_sync(0xffffffffu, a0[q].z, off);
                a0[q].w += __shfl_xor_sync(0xffffffffu, a0[q].w, off);
                if constexpr (DUAL) {
                    a1[q].x += __shfl_xor_sync(0xffffffffu, a1[q].x, off);
                    a1[q].y += __shfl_xor_sync(0xffffffffu, a1[q].y, off);
                    a1[q].z += __shfl_xor_sync(0xffffffffu, a1[q].z, off);
                    a1[q].w += __shfl_xor_sync(0xffffffffu, a1[q].w, off);
                }
            }
            const int idx = idx0 + q * nthr;
            const int o = idx >> 2;
            const int b = o / (kGemvTileCols / V), c = V * (o % (kGemvTileCols / V));
            // masked columns of a last half tile
            if (idx >= total || sub != 0 || t * kGemvTileCols + c >= p.N) continue;
            float v[V] = {a0[q].x, a0[q].y, a0[q].z, a0[q].w};
            const size_t o2 = static_cast<size_t>(b) * p.N + static_cast<size_t>(t) * kGemvTileCols + c;
            if constexpr (DUAL) {
                const float up[V] = {a1[q].x, a1[q].y, a1[q].z, a1[q].w};
#pragma unroll
                for (int e = 0; e < V; ++e) v[e] = v[e] / (1.0f + expf(-v[e])) * up[e];  // silu(gate) * up
            } else if constexpr (MODE == kGemvResidual) {
                const uint2 rv = __ldcg(reinterpret_cast<const uint2 *>(p.resid + o2));
                v[0] += bf16_lo(rv.x);
                v[1] += bf16_hi(rv.x);
                v[2] += bf16_lo(rv.y);
                v[3] += bf16_hi(rv.y);
            }
            uint2 packed;
            packed.x = pack2_bf16(v[0], v[1]);
            packed.y = pack2_bf16(v[2], v[3]);
            *reinterpret_cast<uint2 *>(p.y + o2) = packed;
        }
    }
}

// WIDE: units of 32 KB (128 weight rows, 64 of each matrix in SwiGLU mode)
// instead of 16 KB. One thread issuing copies moves more bytes per copy
// that way: a streaming probe at this kernel's shape (304 blocks, 256-byte
// box rows) read 5.6 TB/s with 5 stages of 16 KB and 6.3-6.7 TB/s with 2-3
// stages of 32 KB.
template <int MAXB, int MODE, bool WIDE>
__global__ void __launch_bounds__(kGemvThreads, MAXB >= 16 ? 1 : 2)
gemv_streamk_kernel(const __grid_constant__ CUtensorMap tm_w0,
                    const __grid_constant__ CUtensorMap tm_w1,
                    const __grid_constant__ CUtensorMap tm_x,
                    const GemvParams p) {
    constexpr bool DUAL = MODE == kGemvSwiGLU;          // gate and up side by side
    constexpr bool NORM = DUAL || MODE == kGemvNormPlain;  // RMSNorm of the input rows
    constexpr int NW = (DUAL ? 2 : 1) * kGemvTileCols;  // partial floats per batch row
    constexpr int STAGE = WIDE ? 2 * kStageBytes : kStageBytes;  // weight bytes per unit
    constexpr int BOX_BYTES = DUAL ? STAGE / 2 : STAGE;
    using GS = GemvShape<MAXB>;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    constexpr int R = (DUAL ? 32 : 64) * (WIDE ? 2 : 1);  // weight rows per unit
    constexpr int RPW = R / kWarpsPerHalf;              // weight rows per warp
    const int B = p.B;
    const int NS = p.nstages;
    const long long U = p.units, P = p.nblocks;
    const int u0 = unit_begin(blockIdx.x, U, P);
    const int u1 = unit_begin(blockIdx.x + 1, U, P);
    const int first_tile = u0 / p.chunks;

    const uint32_t bar_full0 = smem_addr(smem + p.off_bars);
    const uint32_t bar_empty0 = bar_full0 + 8u * NS;
    const uint32_t bar_tile_full0 = bar_full0 + 16u * NS;   // [2]: a reduced tile is in smem
    const uint32_t bar_tile_free0 = bar_tile_full0 + 16u;   // [2]: the epilogue warp is done with it
    volatile int *flags = reinterpret_cast<volatile int *>(smem + p.off_bars + 16 * NS + 32);
    volatile int *timed_out = flags;   // set by the first wait that gives up
    volatile int *is_last = flags + 1; // the block finishes its last tile

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full0 + 8u * s, 1);
            mbar_init(bar_empty0 + 8u * s, kComputeWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_tile_full0 + 8u * b, 1);
            mbar_init(bar_tile_free0 + 8u * b, 1);
        }
        *timed_out = 0;
        *is_last = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dependents_launch();

    const uint32_t stage_tx = STAGE + static_cast<uint32_t>(B * R * 2 + (NORM ? R * 2 : 0));

    if (warp == kComputeWarps) {
        // ---------------------------------------------------------------- load warp
        if (lane == 0) {
            const uint32_t ring = smem_addr(smem);
            const uint32_t xring = smem_addr(smem + p.off_xring);
            RingCursor cur;
            // Weight boxes of unit u: [R x 128] of W0 (and of W1 behind it).
            auto issue_w = [&](int u, int s) {
                const int t = u / p.chunks, k0 = (u % p.chunks) * R;
                const uint32_t dst = ring + s * STAGE, bar = bar_full0 + 8u * s;
                tma_load_2d(dst, &tm_w0, t * kGemvTileCols, k0, bar);
                if constexpr (DUAL) tma_load_2d(dst + BOX_BYTES, &tm_w1, t * kGemvTileCols, k0, bar);
            };
            // Input rows [k0, k0 + R) of every batch row (an earlier kernel's
            // output), plus the matching norm weights.
            auto issue_x = [&](int u, int s) {
                const int k0 = (u % p.chunks) * R;
                const uint32_t dst = xring + s * p.xstage_bytes, bar = bar_full0 + 8u * s;
                tma_load_2d(dst, &tm_x, k0, 0, bar);
                if constexpr (NORM) bulk_load_1d(dst + B * R * 2, p.norm_w + k0, R * 2, bar);
            };
            const int n = u1 - u0;
            const int n_pre = min(NS, n);
            // Weights do not depend on earlier kernels: request the first ring
            // of them before waiting for those kernels to finish.
            for (int i = 0; i < n_pre; ++i) {
                mbar_arrive_expect_tx(bar_full0 + 8u * i, stage_tx);
                issue_w(u0 + i, i);
            }
            grid_dependency_wait();
            for (int i = 0; i < n_pre; ++i) {
                issue_x(u0 + i, i);
                cur.advance(NS);
            }
            for (int i = n_pre; i < n; ++i) {
                if (cur.wrapped)
                    mbar_wait_bounded<false>(bar_empty0 + 8u * cur.stage, cur.phase ^ 1u,
                                             p.timeout_ns, timed_out, p.status, kSiteStageEmpty);
                const int s = cur.stage;
                mbar_arrive_expect_tx(bar_full0 + 8u * s, stage_tx);
                issue_w(u0 + i, s);
                issue_x(u0 + i, s);
                cur.advance(NS);
            }
            // Drain: no exit with copies of this block still in flight.
            // Each wait is bounded at kDrainTimeoutFactor times the normal
            // limit (a copy still pending then is not going to land). If one
            // gives up, the status word records the timeout and the block
            // exits anyway: a block that never exits would hang the GPU,
            // which is worse than a late copy into released shared memory.
            for (int s = 0; s < NS; ++s) {
                if (s >= cur.stage && !cur.wrapped) break;
                volatile int ignore = 0;
                mbar_wait_bounded<false>(bar_full0 + 8u * s, s < cur.stage ? cur.phase : cur.phase ^ 1u,
                                         kDrainTimeoutFactor * p.timeout_ns, &ignore, p.status,
                                         kSiteDrain);
            }
        } else {
            grid_dependency_wait();
        }
        return;
    }

    auto finish_quads = [&](int t, int i_first, int n_t, const float *tl, int ti, int nthr) {
        gemv_finish_quads<MODE, 1>(p, t, i_first, n_t, tl, ti, nthr);
    };
    auto tile_owners = [&](int t, int &i_first, int &n_t) { gemv_tile_owners(p, t, i_first, n_t); };
    auto slot_of = [&](int k) { return gemv_slot<MODE>(p, k); };

    float *tiles = reinterpret_cast<float *>(smem + p.off_tile);  // [2][B][NW]
    if (warp == kComputeWarps + 1) {
        // ----------------------------------------------------------- epilogue warp
        // Finishes every tile of this block but the last while the compute
        // warps stream on: the sole owner applies the epilogue at once; a
        // shared tile's partial goes to the workspace and the last block to
        // arrive sums them all. (The last tile is finished by the compute
        // warps themselves, with all their threads, once streaming is over.)
        grid_dependency_wait();
        const int t_last = (u1 - 1) / p.chunks;
        for (int t = first_tile, k = 0; t < t_last; ++t, ++k) {
            const int tb = k & 1;
            const float *tl = tiles + tb * B * NW;
            mbar_wait_bounded<false>(bar_tile_full0 + 8u * tb, (k >> 1) & 1, p.timeout_ns, timed_out,
                                     p.status, kSiteStageFull);
            int i_first, n_t;
            tile_owners(t, i_first, n_t);
            bool finish = true;
            if (n_t > 1) {
                float4 *slot = slot_of(k);
                const float4 *src = reinterpret_cast<const float4 *>(tl);
                for (int i = lane; i < B * NW / 4; i += 32) slot[i] = src[i];
                __syncwarp();
                unsigned last = 0;
                if (lane == 0) {
                    const unsigned prev = atomic_add_acq_rel_gpu(p.counters + t, 1u);
                    last = prev == static_cast<unsigned>(n_t - 1) ? 1u : 0u;
                    if (last) p.counters[t] = 0u;  // ready for the next launch
                }
                finish = __shfl_sync(0xffffffffu, last, 0) != 0;
            }
            if (finish) finish_quads(t, i_first, n_t, tl, lane, 32);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tile_free0 + 8u * tb);
        }
        return;
    }

    // ------------------------------------------------------------- compute warps
    const uint8_t *ring = smem;
    const uint8_t *xring = smem + p.off_xring;
    float *scratch = reinterpret_cast<float *>(smem + p.off_scratch);  // [8][B][64]
    float *inv_rms = reinterpret_cast<float *>(smem + p.off_misc);     // [B]
    const int half = warp / kWarpsPerHalf;                 // columns [64 half, 64 half + 64)
    const int r0 = (warp % kWarpsPerHalf) * RPW;           // this warp's first row
    float *xn = reinterpret_cast<float *>(smem + p.off_xn) + warp * B * RPW;  // [B][RPW]
    grid_dependency_wait();  // no dependent read or global write before this

    if constexpr (NORM) {
        // RMSNorm statistics: 1 / sqrt(mean_k x[b, k]^2 + eps) for every row,
        // in a fixed order (lane tree, then warps in order).
        for (int b = 0; b < B; ++b) {
            const uint4 *row = reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(b) * p.x_stride);
            float ss = 0.f;
#pragma unroll 4
            for (int i = tid; i < p.K / 8; i += kComputeThreads) {
                float f[8];
                unpack8_bf16(__ldcg(row + i), f);
#pragma unroll
                for (int c = 0; c < 8; ++c) ss = fmaf(f[c], f[c], ss);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if (lane == 0) scratch[warp * MAXB + b] = ss;
        }
        compute_bar<kComputeThreads>();
        if (tid < B) {
            float ss = 0.f;
            for (int w = 0; w < kComputeWarps; ++w) ss += scratch[w * MAXB + tid];
            inv_rms[tid] = 1.0f / sqrtf(ss / static_cast<float>(p.K) + p.eps);
        }
        compute_bar<kComputeThreads>();
    }

    float acc0[MAXB][GS::CPL];
    float acc1[MAXB][GS::CPL];
    auto zero = [&]() {
#pragma unroll
        for (int b = 0; b < MAXB; ++b)
#pragma unroll
            for (int c = 0; c < GS::CPL; ++c) {
                acc0[b][c] = 0.f;
                acc1[b][c] = 0.f;
            }
    };
    // This block is done with its k-th tile (tile t): reduce the warps'
    // partials into a free tile buffer. Tiles before the block's last go to the
    // epilogue warp; the last one is finished here by all compute threads.
    auto finish_tile = [&](int k, int t, bool last_tile) {
        const int tb = k & 1;
        if (k >= 2)
            mbar_wait_bounded<false>(bar_tile_free0 + 8u * tb, ((k >> 1) - 1) & 1, p.timeout_ns,
                                     timed_out, p.status, kSiteStageEmpty);
        float *tl = tiles + tb * B * NW;
        gemv_reduce_halves<MAXB>(acc0, B, warp, lane, tid, scratch, tl, NW);
        if constexpr (DUAL) gemv_reduce_halves<MAXB>(acc1, B, warp, lane, tid, scratch, tl + kGemvTileCols, NW);
        if (!last_tile) {
            if (tid == 0) mbar_arrive(bar_tile_full0 + 8u * tb);
            return;
        }
        int i_first, n_t;
        tile_owners(t, i_first, n_t);
        if (n_t > 1) {
            float4 *slot = slot_of(k);
            const float4 *src = reinterpret_cast<const float4 *>(tl);
            for (int i = tid; i < B * NW / 4; i += kComputeThreads) slot[i] = src[i];
            compute_bar<kComputeThreads>();
            if (tid == 0) {
                const unsigned prev = atomic_add_acq_rel_gpu(p.counters + t, 1u);
                const bool last = prev == static_cast<unsigned>(n_t - 1);
                if (last) p.counters[t] = 0u;  // ready for the next launch
                *is_last = last ? 1 : 0;
            }
            compute_bar<kComputeThreads>();
            if (!*is_last) return;
        }
        finish_quads(t, i_first, n_t, tl, tid, kComputeThreads);
    };

    zero();
    RingCursor cur;
    int k = 0;  // tiles of this block finished so far
    int t = first_tile;
    for (int u = u0; u < u1; ++u) {
        const int s = cur.stage;
        mbar_wait_bounded<false>(bar_full0 + 8u * s, cur.phase, p.timeout_ns, timed_out, p.status,
                                 kSiteStageFull);
        const uint16_t *xs = reinterpret_cast<const uint16_t *>(xring + s * p.xstage_bytes);
        const uint8_t *ws = ring + s * STAGE + half * (kTileCols * 2);
        if constexpr (NORM) {
            // This warp's rows of bf16(g * x * inv_rms): the operand of the
            // projection(s), rounded as a stored bf16 tensor would be.
            const uint16_t *gw = xs + B * R;
            for (int idx = lane; idx < B * RPW; idx += 32) {
                const int b = idx / RPW, j = idx % RPW;
                const float v = bf16_bits(gw[r0 + j]) * bf16_bits(xs[b * R + r0 + j]) * inv_rms[b];
                xn[b * RPW + j] = __bfloat162float(__float2bfloat16_rn(v));
            }
            __syncwarp();
            gemv_rows<MAXB, RPW>(ws, kGemvTileCols * 2, r0, xn, RPW, B, lane, acc0);
            if constexpr (DUAL)
                gemv_rows<MAXB, RPW>(ws + BOX_BYTES, kGemvTileCols * 2, r0, xn, RPW, B, lane, acc1);
        } else {
            gemv_rows<MAXB, RPW>(ws, kGemvTileCols * 2, r0, xs + r0, R, B, lane, acc0);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty0 + 8u * s);
        cur.advance(NS);
        if (u + 1 == u1 || (u + 1) % p.chunks == 0) {
            finish_tile(k++, t++, u + 1 == u1);
            zero();
        }
    }
}

// y[b] = bf16(g * x[b] / sqrt(mean(x[b]^2) + eps)); one block per row, n a
// multiple of 8, rows 16-byte aligned. Fixed-order reduction.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t *x, const uint16_t *g,
                                                      uint16_t *y, int n, float eps) {
    __shared__ float red[8];
    grid_dependents_launch();
    grid_dependency_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(blockIdx.x) * n);
    float ss = 0.f;
    for (int i = tid; i < n / 8; i += 256) {
        float f[8];
        unpack8_bf16(__ldcg(row + i), f);
#pragma unroll
        for (int c = 0; c < 8; ++c) ss = fmaf(f[c], f[c], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / static_cast<float>(n) + eps);
    const uint4 *gv = reinterpret_cast<const uint4 *>(g);
    uint4 *out = reinterpret_cast<uint4 *>(y + static_cast<size_t>(blockIdx.x) * n);
    for (int i = tid; i < n / 8; i += 256) {
        float f[8], w[8];
        unpack8_bf16(__ldcg(row + i), f);
        unpack8_bf16(__ldg(gv + i), w);
        uint4 o;
        o.x = pack2_bf16(w[0] * f[0] * inv, w[1] * f[1] * inv);
        o.y = pack2_bf16(w[2] * f[2] * inv, w[3] * f[3] * inv);
        o.z = pack2_bf16(w[4] * f[4] * inv, w[5] * f[5] * inv);
        o.w = pack2_bf16(w[6] * f[6] * inv, w[7] * f[7] * inv);
        out[i] = o;
    }
}

// The decode loop's position counters: pos[b] += 1 once every earlier kernel
// of the token has finished reading them.
__global__ void advance_positions_kernel(int *pos, int B) {
    grid_dependents_launch();
    grid_dependency_wait();
    if (static_cast<int>(threadIdx.x) < B) pos[threadIdx.x] += 1;
}

}  // namespace cfa
