// cfa_gemv_mma.cuh -- the stream-K GEMV of the decoder layer on the tcgen05
// tensor cores, for batches of 3 to 16 rows.
//
// At batch B the GEMV does 2B flops per weight byte; on the CUDA cores that is
// compute-bound from B = 4 on, while every weight byte still has to be read
// once. Here each unit of work -- one 128-column tile x 64 weight rows of one
// or two matrices -- is a dense contraction D[128 cols x 16] += W^T X^T:
//   A = the weight unit, read MN-major from two 128-byte-swizzled TMA boxes of
//       [64 rows x 64 cols] (M = 128 output columns, K = 16 rows per MMA),
//   B = the batch's 64 input values of those rows, one [16 x 64] K-major
//       swizzled box (rows past B are zero-filled by the TMA unit),
//   D = fp32 in TMEM, 16 columns per matrix, double-buffered per tile.
// Units, tiles, the split of the units over a persistent grid and the
// deterministic finishing of shared tiles are those of the CUDA-core kernel
// (cfa_gemv.cuh); only the inner product moved to the tensor cores.
//
// Warps: 0-3 read a finished tile's accumulators out of TMEM (warp w owns
// TMEM lanes 32w..32w+31 = output columns) and finish the tile (its partial to
// the workspace, and the fixed-order sum and epilogue if this block is the
// last of the tile's owners). Warp 4 issues the MMAs (one thread), warp 5 the
// TMA loads; in the RMSNorm modes warp 6 turns each input box into
// bf16(g x / rms(x)) in place before the MMAs read it. The accumulators are
// double-buffered, so the MMAs of the next tile run while a tile is finished.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "cfa_device.cuh"
#include "cfa_gemv.cuh"
#include "cfa_internal.h"
#include "cfa_layer_params.h"
#include "cfa_tile.cuh"

namespace cfa {

template <int MODE>
__global__ void __launch_bounds__(kGemvMmaThreads, 1)
gemv_mma_kernel(const __grid_constant__ CUtensorMap tm_w0,
                const __grid_constant__ CUtensorMap tm_w1,
                const __grid_constant__ CUtensorMap tm_x,
                const GemvParams p) {
    constexpr bool DUAL = MODE == kGemvSwiGLU;
    constexpr bool NORM = DUAL || MODE == kGemvNormPlain;
    constexpr int NMAT = DUAL ? 2 : 1;
    constexpr int NW = gemv_nw<MODE>();
    constexpr int WBYTES = NMAT * 2 * kGemvMmaBoxBytes;  // weights of one unit
    constexpr int R = kGemvMmaRows;
    constexpr int kReaderThreads = kGemvMmaReaders * 32;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.B;
    const int NS = p.nstages;
    const long long U = p.units, P = p.nblocks;
    const int u0 = unit_begin(blockIdx.x, U, P);
    const int u1 = unit_begin(blockIdx.x + 1, U, P);
    const int first_tile = u0 / p.chunks;
    const int SB = p.xstage_bytes;  // bytes of one stage: weights, input box, norm weights

    const uint32_t ring = smem_addr(smem);
    const uint32_t bar_full0 = smem_addr(smem + p.off_bars);
    const uint32_t bar_empty0 = bar_full0 + 8u * NS;        // released by the MMAs' commit
    const uint32_t bar_xready0 = bar_full0 + 16u * NS;      // input box normalized (RMSNorm modes)
    const uint32_t bar_acc_full0 = bar_full0 + 24u * NS;    // [2] a tile's accumulators are done
    const uint32_t bar_acc_free0 = bar_acc_full0 + 16u;     // [2] the readers are done with them
    volatile int *flags = reinterpret_cast<volatile int *>(smem + p.off_bars + 24 * NS + 32);
    volatile int *timed_out = flags;
    volatile int *is_last = flags + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + p.off_bars + 24 * NS + 40);

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full0 + 8u * s, 1);
            mbar_init(bar_empty0 + 8u * s, 1);
            mbar_init(bar_xready0 + 8u * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_acc_full0 + 8u * b, 1);
            mbar_init(bar_acc_free0 + 8u * b, kGemvMmaReaders);
        }
        *timed_out = 0;
        *is_last = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(smem_addr(tmem_slot), 64);  // tile k: columns 32 (k % 2) + 16 matrix
    tcgen05_fence_before();
    __syncthreads();
    grid_dependents_launch();
    tcgen05_fence_after();
    const uint32_t tmem = *tmem_slot;
    // A unit's last index within its tile, and whether it starts one.
    auto tile_end = [&](int u) { return u + 1 == u1 || (u + 1) % p.chunks == 0; };
    auto tile_start = [&](int u) { return u == u0 || u % p.chunks == 0; };

    float *tl = reinterpret_cast<float *>(smem + p.off_tile);  // [B][NW]: the tile being finished

    if (warp == kGemvMmaReaders + 1) {
        // ---------------------------------------------------------------- load warp
        if (lane == 0) {
            RingCursor cur;
            const uint32_t stage_tx = WBYTES + kGemvMmaXBytes + (NORM ? R * 2 : 0);
            auto issue_w = [&](int u, int s) {
                const int t = u / p.chunks, k0 = (u % p.chunks) * R;
                const uint32_t dst = ring + s * SB, bar = bar_full0 + 8u * s;
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        tma_load_2d(dst + (2 * m + h) * kGemvMmaBoxBytes, m ? &tm_w1 : &tm_w0,
                                    t * kGemvTileCols + h * 64, k0, bar);
            };
            auto issue_x = [&](int u, int s) {
                const int k0 = (u % p.chunks) * R;
                const uint32_t dst = ring + s * SB + WBYTES, bar = bar_full0 + 8u * s;
                tma_load_2d(dst, &tm_x, k0, 0, bar);
                if constexpr (NORM) bulk_load_1d(dst + kGemvMmaXBytes, p.norm_w + k0, R * 2, bar);
            };
            const int n = u1 - u0;
            const int n_pre = min(NS, n);
            for (int i = 0; i < n_pre; ++i) {  // weights do not depend on earlier kernels
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
            // No drain: the MMA warp waits for every stage loaded here, and the
            // block does not exit before its last MMAs have completed.
        } else {
            grid_dependency_wait();
        }
        return;
    }

    if (warp == kGemvMmaReaders) {
        // ----------------------------------------------------------------- MMA warp
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16(128, kMmaN, true, false);  // A MN-major
            RingCursor cur;
            int k = 0;  // tiles of this block
            for (int u = u0; u < u1; ++u) {
                const int s = cur.stage;
                mbar_wait_bounded<false>((NORM ? bar_xready0 : bar_full0) + 8u * s, cur.phase, p.timeout_ns,
                                         timed_out, p.status, kSiteStageFull);
                const bool first = tile_start(u);
                if (first && k >= 2)  // the readers are done with this accumulator buffer
                    mbar_wait_bounded<false>(bar_acc_free0 + 8u * (k & 1), ((k >> 1) - 1) & 1,
                                             p.timeout_ns, timed_out, p.status, kSiteStageEmpty);
                tcgen05_fence_after();
                const uint32_t st = ring + s * SB;
                const uint32_t d = tmem + 32u * (k & 1);
#pragma unroll
                for (int m = 0; m < NMAT; ++m)
#pragma unroll
                    for (int ks = 0; ks < R / 16; ++ks)
                        umma_bf16(d + 16u * m,
                                  umma_smem_desc(st + m * 2 * kGemvMmaBoxBytes + ks * 2048, kGemvMmaBoxBytes, 1024),
                                  umma_smem_desc(st + WBYTES + ks * 32, 16, 1024), idesc, !first || ks > 0);
                umma_commit(bar_empty0 + 8u * s);
                if (tile_end(u)) umma_commit(bar_acc_full0 + 8u * (k++ & 1));
                cur.advance(NS);
            }
        }
        __syncwarp();
        return;
    }

    if (warp == kGemvMmaReaders + 2) {
        // ------------------------------------------------------------- norm warp
        if constexpr (NORM) {
            const float *inv_rms = reinterpret_cast<const float *>(smem + p.off_misc);  // [B]
            // the readers compute the row statistics (1 / rms) and pass them on
            asm volatile("bar.sync 2, %0;" :: "n"(kReaderThreads + 32) : "memory");
            // Each stage's input box -> bf16(g x / rms(x)), in place: 16-byte
            // chunk c of box row (batch row) b, c = lane % 8, b = lane / 8 + 4 i.
            RingCursor cur;
            for (int u = u0; u < u1; ++u) {
                const int s = cur.stage;
                mbar_wait_bounded<false>(bar_full0 + 8u * s, cur.phase, p.timeout_ns, timed_out, p.status,
                                         kSiteStageFull);
                uint8_t *xb = smem + s * SB + WBYTES;
                const uint16_t *gw = reinterpret_cast<const uint16_t *>(xb + kGemvMmaXBytes);
                const int pc = lane & 7;  // physical chunk
#pragma unroll
                for (int i = 0; i < kMmaN / 4; ++i) {
                    const int b = (lane >> 3) + 4 * i;
                    const int lc = pc ^ (b & 7);  // logical chunk: columns 8 lc .. 8 lc + 7
                    if (b < B) {
                        uint4 *q = reinterpret_cast<uint4 *>(xb + b * 128 + pc * 16);
                        float f[8];
                        unpack8_bf16(*q, f);
                        const float inv = inv_rms[b];
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            o[e] = pack2_bf16(bf16_bits(gw[8 * lc + 2 * e]) * f[2 * e] * inv,
                                              bf16_bits(gw[8 * lc + 2 * e + 1]) * f[2 * e + 1] * inv);
                        *q = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
                fence_proxy_async_smem();  // the box is read by the tensor cores
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_xready0 + 8u * s);
                cur.advance(NS);
            }
        }
        return;
    }

    // ------------------------------------------------------------------ readers
    grid_dependency_wait();  // no dependent read or global write before this
    if constexpr (NORM) {
        // 1 / sqrt(mean_k x[b, k]^2 + eps) of every input row, in a fixed order
        // (per thread, per warp, then warps in order), for the norm warp. Each
        // thread keeps 16 loads in flight: 4 rows x 4 chunks of 8 values.
        float *red = reinterpret_cast<float *>(smem + p.off_scratch);  // [4 warps][16 rows]
        float *inv_rms = reinterpret_cast<float *>(smem + p.off_misc);  // [B]
        const int KC = p.K / 8;  // 16-byte chunks of a row
        for (int b0 = 0; b0 < B; b0 += 4) {
            float ss[4] = {0.f, 0.f, 0.f, 0.f};
            for (int i0 = tid; i0 < KC; i0 += 4 * kReaderThreads) {
                uint4 v[4][4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int i = i0 + j * kReaderThreads;
                        v[r][j] = b0 + r < B && i < KC
                                      ? __ldcg(reinterpret_cast<const uint4 *>(
                                                   p.x + static_cast<size_t>(b0 + r) * p.x_stride) + i)
                                      : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float f[8];
                        unpack8_bf16(v[r][j], f);
#pragma unroll
                        for (int c = 0; c < 8; ++c) ss[r] = fmaf(f[c], f[c], ss[r]);
                    }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss[r] += __shfl_xor_sync(0xffffffffu, ss[r], off);
                if (lane == 0 && b0 + r < B) red[warp * kMaxBatch + b0 + r] = ss[r];
            }
        }
        compute_bar<kReaderThreads>();
        if (tid < B) {
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < kGemvMmaReaders; ++w) tot += red[w * kMaxBatch + tid];
            inv_rms[tid] = 1.0f / sqrtf(tot / static_cast<float>(p.K) + p.eps);
        }
        asm volatile("bar.arrive 2, %0;" :: "n"(kReaderThreads + 32) : "memory");
    }
    // The block's k-th tile (tile t): accumulators -> tile buffer [B][NW],
    // then the partial to the workspace and, by the last owner, the finish.
    auto finish_tile = [&](int k, int t) {
        const int tb = k & 1;
        mbar_wait_bounded<false>(bar_acc_full0 + 8u * tb, (k >> 1) & 1, p.timeout_ns, timed_out, p.status,
                                 kSiteStageFull);
        tcgen05_fence_after();
        const int col = 32 * warp + lane;  // this thread's TMEM lane = output column
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            float v[16];
            tmem_ld_x16(tmem + (static_cast<uint32_t>(32 * warp) << 16) + 32u * tb + 16u * m, v);
#pragma unroll
            for (int b = 0; b < kMmaN; ++b)
                if (b < B) tl[b * NW + m * kGemvTileCols + col] = v[b];
        }
        tcgen05_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acc_free0 + 8u * tb);
        compute_bar<kReaderThreads>();
        int i_first, n_t;
        gemv_tile_owners(p, t, i_first, n_t);
        bool finish = true;
        if (n_t > 1) {
            float4 *slot = gemv_slot<MODE>(p, k);
            const float4 *src = reinterpret_cast<const float4 *>(tl);
            for (int i = tid; i < B * NW / 4; i += kReaderThreads) slot[i] = src[i];
            compute_bar<kReaderThreads>();
            if (tid == 0) {
                const unsigned prev = atomic_add_acq_rel_gpu(p.counters + t, 1u);
                const bool last = prev == static_cast<unsigned>(n_t - 1);
                if (last) p.counters[t] = 0u;  // ready for the next launch
                *is_last = last ? 1 : 0;
            }
            compute_bar<kReaderThreads>();
            finish = *is_last != 0;
        }
        if (finish) gemv_finish_quads<MODE, 8>(p, t, i_first, n_t, tl, tid, kReaderThreads);
        compute_bar<kReaderThreads>();  // the tile buffer and the flag are free again
    };

    int k = 0;
    int t = first_tile;
    for (int u = u0; u < u1; ++u)
        if (tile_end(u)) finish_tile(k++, t++);
    tcgen05_fence_before();
    compute_bar<kReaderThreads>();
    if (warp == 0) {
        tcgen05_fence_after();
        tmem_dealloc(tmem, 64);
    }
}

}  // namespace cfa
