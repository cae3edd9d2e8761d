// cfa_mla.cuh -- the attention core of a multi-head latent attention (MLA)
// decode step on one thread-block cluster per (sequence, head group).
//
// Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命" (ClusterFusion
// framework analysis), written [CF §n]. For DeepSeek's MLA the page partitions
// the latent key/value cache across clusters and changes ClusterReduce into a
// sparse reduction [CF §5.2]; it gives no further detail. The block's
// dimensions are DeepSeek-V2/V3's: latent 512, per-head nope / rope / value
// widths 128 / 64 / 128.
//
// All heads share one latent cache row per token ([c (512) | k_rope (64)]), so
// the kernel works on the absorbed form: with W_k, W_v the per-head key and
// value blocks of W_kvb [512, nh*256],
//   q~_h  = W_k,h q_nope,h            (512)      score_t = q~_h . c_t + rope(q_rope,h) . k_rope_t
//   o_h   = sum_t softmax_t c_t       (512)      v_h     = o_h . W_v,h   (128)
// which equals attention over the decompressed keys and values. The heads of a
// group share every latent byte, so the latent attention is a dense
// contraction and runs on the tensor cores.
//
// Grid: B x (nh / HG) x S clusters of C blocks; cluster (b, g, s) owns heads
// [g HG, (g+1) HG) of sequence b and split s of the latent rows: its block r
// attends rows [T q / (S C), T (q+1) / (S C)), q = s C + r, of T = L + 1 rows
// (the new token's row is the last). C (16, 8, 4 or 2) and S (1, 2 or 4) are
// chosen per step by the host among the shapes whose clusters are all
// resident at once; each block finishes HPB = HG / C heads. Warps: 8
// compute warps, a TMA warp streaming every operand through one ring of 32 KB
// stages (W_k blocks, cache tiles, W_v blocks, in the order they are used),
// and an MMA warp.
//  A  Absorption [CF §3.2 deferred projection]: block r computes q~ and the
//     rotated rope query of its HPB heads from their W_k blocks and sends
//     them to every block of the cluster (ClusterGather over DSMEM: one bulk
//     shared::cluster copy per peer, bytes counted on the peer's barrier), so
//     every block holds all HG queries; they become one bf16 operand of hi
//     and lo parts (about 16 bits together). The last block then builds the
//     new latent row (RMSNorm of the latent part, rope of the key part, bf16)
//     on chip while its first tile's scores are computed; one block appends
//     it.
//  B  Latent attention over the block's cached rows, 128 rows per tile, with
//     tcgen05 and TMEM accumulators: S^T = C [Qhi | Qlo]^T (M = 128 rows,
//     N = 32, K = 576; the row tile is the K-major A operand, straight from
//     its 128-byte-swizzled TMA boxes), a base-2 online softmax per head
//     across the tile (TMEM lane = row), P written as a bf16 K-major operand,
//     then O^T = C^T P^T (M = 4 x 128 latent dims, the same boxes read
//     MN-major, K = 128 rows), folded into fp32 registers. The MMA warp
//     issues the scores of tile t + 1 before the values of tile t, so the
//     softmax runs under the MMAs (scores, outputs and P double-buffered).
//     The latent boxes pass through the ring twice per tile (scores, then
//     values; the second pass hits L2). The new row is attended on CUDA cores.
//  C  Sparse ClusterReduce [CF §5.2]: a reduce-scatter over the cluster --
//     block r receives, for its own HPB heads only, every block's (m, l, o),
//     one bulk copy per head, and combines them in block order
//     (deterministic); then v_h = o_h W_v,h. With S > 1 splits, block r of
//     every split holds the same heads: each writes its v_h with its split's
//     max and sum to global memory, and the last of them to arrive combines
//     the S records in split order.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "cfa_device.cuh"
#include "cfa_internal.h"
#include "cfa_layer_params.h"
#include "cfa_tile.cuh"

namespace cfa {

// 8 consecutive fp32 TMEM columns of this warp's 32 lanes (one lane per thread).
__device__ __forceinline__ void mla_tmem_ld_x8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of element (row n, column k < 64) of a [rows x 64] K-major
// operand atom with 128-byte swizzle (16-byte chunks permuted by n mod 8).
__device__ __forceinline__ uint32_t mla_atom_off(int n, int k) {
    return static_cast<uint32_t>(n * 128 + (((k >> 3) ^ (n & 7)) << 4) + (k & 7) * 2);
}

// Bounded wait of every calling thread on a barrier phase (all threads poll:
// measured faster here than one polling lane per warp and a __syncwarp).
template <bool CLUSTER_SCOPE>
__device__ __forceinline__ void mla_wait(uint32_t bar, uint32_t parity, const MlaParams &p,
                                         volatile int *timed_out, unsigned site) {
    mbar_wait_bounded<CLUSTER_SCOPE>(bar, parity, p.timeout_ns, timed_out, p.status, site);
}

// Rotate-half rotation of (x0, x1) = dims (k, k + 32) by pos * inv_freq, the
// angle taken in fp64 and reduced to (-pi, pi] before the fp32 sine/cosine.
__device__ __forceinline__ void mla_rope(float &x0, float &x1, int pos, double inv_freq) {
    const double ang = static_cast<double>(pos) * inv_freq;
    const double red = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);
    float sn, cs;
    sincosf(static_cast<float>(red), &sn, &cs);
    const float y0 = x0 * cs - x1 * sn, y1 = x1 * cs + x0 * sn;
    x0 = y0;
    x1 = y1;
}

__global__ void __launch_bounds__(kMlaThreads, 1)
mla_attention_kernel(const __grid_constant__ MlaMaps maps,
                     const __grid_constant__ CUtensorMap tm_wkvb, const MlaParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = p.C, HG = p.HG, HPB = p.HPB, NS = p.nstages;
    const int r = static_cast<int>(cluster_ctarank());
    const int cluster = blockIdx.x / C;
    const int NG = p.nh / HG, S = p.S;
    const int b = cluster / (NG * S), g = (cluster / S) % NG, split = cluster % S;
    const int L = p.ctx_lens[b];
    const int T = L + 1;
    // rows of block r of split `split`: the (split C + r)-th of S C even parts
    const long long part = static_cast<long long>(split) * C + r, parts = static_cast<long long>(S) * C;
    const int row_s = static_cast<int>((static_cast<long long>(T) * part) / parts);
    const int row_e = static_cast<int>((static_cast<long long>(T) * (part + 1)) / parts);
    const int cache_e = min(row_e, L);                       // rows read from the cache
    const bool has_new = row_e == T;                         // this block attends the new row
    const int n_tiles = cache_e > row_s ? (cache_e - row_s + kMlaTileRows - 1) / kMlaTileRows : 0;
    constexpr int kSStages = (kMlaBoxes + 1) / 2;            // score pass: 5 stages (last: one box)
    constexpr int kVStages = kMlaKv / 128;                   // value pass: 4 stages of 128 dims

    float *qt = reinterpret_cast<float *>(smem + p.off_qt);      // [HG][576] scaled queries, fp32
    float *stat = reinterpret_cast<float *>(smem + p.off_stat);
    float *m_st = stat;               // [16] running max per head (base 2)
    float *l_st = stat + 16;          // [16] running sum
    float *alpha = stat + 32;         // [2 tiles][16] rescale of o
    float *red_max = stat + 64;       // [2 tiles][8 warps][16]
    float *red_sum = stat + 320;      // [2 tiles][8 warps][16]
    float *s_new = stat + 576;        // [16] score, then probability, of the new row
    float *recv = reinterpret_cast<float *>(smem + p.off_recv);  // [HPB][C][516], over qt
    float *ofin = reinterpret_cast<float *>(smem + p.off_ofin);  // [HPB][512]
    float *scr = reinterpret_cast<float *>(smem + p.off_scr);    // [8][128] + 64
    uint16_t *newrow = reinterpret_cast<uint16_t *>(smem + p.off_newrow);  // [576] bf16
    const uint32_t ring = smem_addr(smem + p.off_ring);
    const uint32_t qb = smem_addr(smem + p.off_qb);
    const uint32_t pb = smem_addr(smem + p.off_pb);
    const uint32_t bar_full0 = smem_addr(smem + p.off_bars);
    const uint32_t bar_empty0 = bar_full0 + 8u * NS;
    const uint32_t bar_q = bar_full0 + 16u * NS;      // every peer's queries have landed
    const uint32_t bar_red = bar_q + 8u;              // every peer's partials for my heads
    const uint32_t bar_qfree = bar_q + 16u;           // every peer is done with its fp32 queries
    const uint32_t bar_qready = bar_q + 24u;          // the query operand is built
    const uint32_t bar_s0 = bar_q + 32u;              // [2] a tile's scores are in TMEM
    const uint32_t bar_o0 = bar_q + 48u;              // [2] a tile's latent outputs are in TMEM
    const uint32_t bar_p0 = bar_q + 64u;              // [2] a tile's P is written, its scores read
    volatile int *timed_out = reinterpret_cast<volatile int *>(smem + p.off_bars + 16 * NS + 80);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + p.off_bars + 16 * NS + 88);

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full0 + 8u * s, 1);
            mbar_init(bar_empty0 + 8u * s, 1);     // released by the MMAs' commit
        }
        mbar_init(bar_q, 1);
        mbar_init(bar_red, 1);
        mbar_init(bar_qfree, C - 1);
        mbar_init(bar_qready, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar_s0 + 8u * i, 1);
            mbar_init(bar_o0 + 8u * i, 1);
            mbar_init(bar_p0 + 8u * i, 1);
        }
        *timed_out = 0;
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_q, static_cast<uint32_t>((C - 1) * HPB * kMlaRow * 4));
        mbar_arrive_expect_tx(bar_red, static_cast<uint32_t>((C - 1) * HPB * (kMlaKv + 4) * 4));
    }
    // TMEM: scores of tile t at columns 32 (t % 2) (hi part 0-15, lo part 16-31),
    // latent outputs at 64 + 64 (t % 2) + 16 v for latent block v
    if (warp == 0) tmem_alloc(smem_addr(tmem_slot), 256);
    tcgen05_fence_before();
    __syncthreads();
    cluster_arrive();  // barriers announced; waited for before the first push

    if (warp == kComputeWarps) {
        // ------------------------------------------------------------ load warp
        // Ring order (the compute side consumes in the same order): the W_k
        // blocks of this block's heads, the cache tiles (scores, then values,
        // per tile), the W_v blocks of its heads. Weight boxes are [256 x 64].
        if (lane == 0) {
            RingCursor cur;
            auto wait_slot = [&]() {
                if (cur.wrapped)
                    mbar_wait_bounded<false>(bar_empty0 + 8u * cur.stage, cur.phase ^ 1u,
                                             p.timeout_ns, timed_out, p.status, kSiteStageEmpty);
            };
            // [512 x 128] of W_kvb in 4 stages: W_k column-block major (each
            // half of q_nope is used for both row blocks), W_v row-block major
            auto weight_block = [&](int col0, bool col_major) {
                for (int a = 0; a < 2; ++a)
                    for (int c = 0; c < 2; ++c) {
                        const int rb = col_major ? c : a, cb = col_major ? a : c;
                        wait_slot();
                        const uint32_t full = bar_full0 + 8u * cur.stage;
                        mbar_arrive_expect_tx(full, static_cast<uint32_t>(kMlaStageBytes));
                        tma_load_2d(ring + cur.stage * kMlaStageBytes, &tm_wkvb, col0 + 64 * cb,
                                    kMlaWeightRows * rb, full);
                        cur.advance(NS);
                    }
            };
            // Weight blocks into L2 ahead of the ring (more bytes in flight than
            // it holds): W_k now, W_v once the W_k loads are out, so that it
            // does not queue in front of them.
            auto prefetch_block = [&](int col0) {
                for (int rb = 0; rb < 2; ++rb)
                    for (int cb = 0; cb < 2; ++cb) tma_prefetch_2d(&tm_wkvb, col0 + 64 * cb, kMlaWeightRows * rb);
            };
            // weights: independent of the previous kernel. The first head's
            // W_k goes straight into the ring; the other heads' into L2 behind it.
            weight_block((g * HG + r * HPB) * (kMlaNope + kMlaV), true);
            for (int i = 1; i < HPB; ++i) prefetch_block((g * HG + r * HPB + i) * (kMlaNope + kMlaV));
            for (int i = 1; i < HPB; ++i) weight_block((g * HG + r * HPB + i) * (kMlaNope + kMlaV), true);
            for (int i = 0; i < HPB; ++i)
                prefetch_block((g * HG + r * HPB + i) * (kMlaNope + kMlaV) + kMlaNope);
            grid_dependency_wait();  // cache rows may come from the previous step
            const CUtensorMap *tm = &maps.cache[b];
            auto stage_in = [&](int kc0, int nbox, int row) {
                wait_slot();
                const uint32_t full = bar_full0 + 8u * cur.stage;
                const uint32_t dst = ring + cur.stage * kMlaStageBytes;
                mbar_arrive_expect_tx(full, static_cast<uint32_t>(nbox * kMlaBoxBytes));
                for (int i = 0; i < nbox; ++i)
                    tma_load_2d(dst + i * kMlaBoxBytes, tm, (kc0 + i) * 64, row, full);
                cur.advance(NS);
            };
            // scores of tile t are computed while the softmax of tile t - 1 runs:
            // stages in the MMA warp's order S0, S1, V0, S2, V1, ...
            for (int t = 0; t <= n_tiles; ++t) {
                if (t < n_tiles)  // rows past the map's end read as zero
                    for (int sp = 0; sp < kSStages; ++sp)
                        stage_in(2 * sp, min(2, kMlaBoxes - 2 * sp), row_s + t * kMlaTileRows);
                if (t >= 1)
                    for (int vp = 0; vp < kVStages; ++vp) stage_in(2 * vp, 2, row_s + (t - 1) * kMlaTileRows);
            }
            for (int i = 0; i < HPB; ++i)
                weight_block((g * HG + r * HPB + i) * (kMlaNope + kMlaV) + kMlaNope, false);
            // no drain: the compute warps wait for every stage this warp loads
        } else {
            grid_dependency_wait();
        }
        __syncwarp();
        grid_dependents_launch();
        cluster_wait();
        cluster_sync_all();
        return;
    }

    if (warp == kComputeWarps + 1) {
        // ------------------------------------------------------------- MMA warp
        if (lane == 0 && n_tiles > 0) {
            RingCursor cur;
            for (int n = 0; n < 4 * HPB; ++n) cur.advance(NS);  // the W_k stages go to the compute warps
            mbar_wait_bounded<false>(bar_qready, 0, p.timeout_ns, timed_out, p.status, kSiteQExchange);
            tcgen05_fence_after();
            const uint32_t tmem = *tmem_slot;
            const uint32_t idesc_s = umma_idesc_bf16(128, 2 * kMlaMaxHG, false, false);  // A K-major
            const uint32_t idesc_o = umma_idesc_bf16(128, kMlaMaxHG, true, false);       // A MN-major
            auto stage_wait = [&]() {
                mbar_wait_bounded<false>(bar_full0 + 8u * cur.stage, cur.phase, p.timeout_ns, timed_out,
                                         p.status, kSiteStageFull);
                tcgen05_fence_after();
                return ring + cur.stage * kMlaStageBytes;
            };
            auto stage_free = [&]() {  // the stage is released once these MMAs have read it
                umma_commit(bar_empty0 + 8u * cur.stage);
                cur.advance(NS);
            };
            for (int t = 0; t <= n_tiles; ++t) {
                if (t < n_tiles) {
                    // S^T = C [Qhi | Qlo]^T over the 9 latent boxes: N = 32
                    const uint32_t d = tmem + 2 * kMlaMaxHG * (t & 1);
                    for (int sp = 0; sp < kSStages; ++sp) {
                        const uint32_t st = stage_wait();
                        for (int bx = 0; bx < 2 && 2 * sp + bx < kMlaBoxes; ++bx) {
                            const int kc = 2 * sp + bx;
#pragma unroll
                            for (int ks = 0; ks < 4; ++ks)
                                umma_bf16(d, umma_smem_desc(st + bx * kMlaBoxBytes + ks * 32, 16, 1024),
                                          umma_smem_desc(qb + kc * kMlaQAtomBytes + ks * 32, 16, 1024),
                                          idesc_s, kc > 0 || ks > 0);
                        }
                        stage_free();
                    }
                    umma_commit(bar_s0 + 8u * (t & 1));
                }
                if (t >= 1) {
                    // O^T = C^T P^T of tile u = t - 1, 4 latent blocks of 128 dims
                    const int u = t - 1;
                    mbar_wait_bounded<false>(bar_p0 + 8u * (u & 1), (u >> 1) & 1, p.timeout_ns, timed_out,
                                             p.status, kSiteStageFull);
                    tcgen05_fence_after();
                    const uint32_t d = tmem + 64 + 64 * (u & 1);
                    const uint32_t pt = pb + (u & 1) * 2 * kMlaAtomBytes;
                    for (int vp = 0; vp < kVStages; ++vp) {
                        const uint32_t st = stage_wait();
#pragma unroll
                        for (int ks = 0; ks < kMlaTileRows / 16; ++ks)
                            umma_bf16(d + 16 * vp, umma_smem_desc(st + ks * 2048, kMlaBoxBytes, 1024),
                                      umma_smem_desc(pt + (ks >> 2) * kMlaAtomBytes + (ks & 3) * 32, 16, 1024),
                                      idesc_o, ks > 0);
                        stage_free();
                    }
                    umma_commit(bar_o0 + 8u * (u & 1));
                }
            }
        }
        __syncwarp();
        grid_dependents_launch();
        cluster_wait();
        cluster_sync_all();
        return;
    }

    // --------------------------------------------------------------- compute
    tcgen05_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dependency_wait();
    // ---- A: absorbed queries of this block's heads, pushed to the cluster ----
    RingCursor cur;  // every compute thread follows the ring through phase A
    auto stage_ready = [&]() {
        mla_wait<false>(bar_full0 + 8u * cur.stage, cur.phase, p, timed_out, kSiteStageFull);
        return smem + p.off_ring + cur.stage * kMlaStageBytes;
    };
    auto stage_done = [&]() {  // every compute thread has read the stage
        compute_bar<kComputeThreads>();
        if (tid == 0) mbar_arrive(bar_empty0 + 8u * cur.stage);
        cur.advance(NS);
    };
    {
        // q_nope of this block's heads, [HPB][128], where the combined outputs
        // go in phase C
        float *qn_all = ofin;
        for (int k = tid; k < HPB * kMlaNope; k += kComputeThreads) {
            const int h = g * HG + r * HPB + k / kMlaNope;
            qn_all[k] = bf16_bits(p.q[static_cast<size_t>(b) * p.nh * kMlaQk + h * kMlaQk + k % kMlaNope]);
        }
        compute_bar<kComputeThreads>();
        for (int i = 0; i < HPB; ++i) {
            const int hl = r * HPB + i;             // head within the group
            const int h = g * HG + hl;
            const uint16_t *qh = p.q + static_cast<size_t>(b) * p.nh * kMlaQk + h * kMlaQk;
            const float *qn = qn_all + i * kMlaNope;
            float *dst = qt + hl * kMlaRow;
            // q~[j] = sum_c W_kvb[j, h*256 + c] q_nope[c]: thread tid takes latent
            // rows tid and tid + 256, a swizzled 128-byte box row per stage; the
            // 64 q_nope values of a column block stay in registers
            // (the stage loop is not unrolled: this code runs once per block, and
            // a smaller body costs fewer instruction fetches)
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll 1
            for (int cb = 0; cb < 2; ++cb) {
                float qr[64];
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float4 v = reinterpret_cast<const float4 *>(qn + 64 * cb)[c];
                    qr[4 * c] = v.x; qr[4 * c + 1] = v.y; qr[4 * c + 2] = v.z; qr[4 * c + 3] = v.w;
                }
#pragma unroll 1
                for (int rb = 0; rb < 2; ++rb) {
                    const uint8_t *st = stage_ready();
                    float sum = 0.f;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        float f[8];
                        unpack8_bf16(*reinterpret_cast<const uint4 *>(st + tid * 128 + ((c ^ (tid & 7)) << 4)), f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) sum = fmaf(f[e], qr[8 * c + e], sum);
                    }
                    stage_done();
                    if (rb == 0) acc0 += sum; else acc1 += sum;
                }
            }
            dst[tid] = acc0 * p.qscale;
            dst[tid + kComputeThreads] = acc1 * p.qscale;
            if (tid < kMlaRope / 2) {
                float x0 = bf16_bits(qh[kMlaNope + tid]), x1 = bf16_bits(qh[kMlaNope + tid + kMlaRope / 2]);
                if (p.rope) mla_rope(x0, x1, L, p.rope_inv_freq[tid]);
                dst[kMlaKv + tid] = x0 * p.qscale;
                dst[kMlaKv + tid + kMlaRope / 2] = x1 * p.qscale;
            }
            fence_proxy_async_smem();  // the rows are read by the bulk copies
            compute_bar<kComputeThreads>();
        }
        cluster_wait();  // every peer's barriers exist before the first copy
        // ClusterGather: my heads' 576 scaled query values, one bulk copy per peer
        if (tid < C && tid != r) {
            const uint32_t my0 = smem_addr(qt + r * HPB * kMlaRow);
            bulk_copy_to_rank(map_to_rank(my0, tid), my0, static_cast<uint32_t>(HPB * kMlaRow * 4),
                              map_to_rank(bar_q, tid));
        }
    }
    mla_wait<true>(bar_q, 0, p, timed_out, kSiteQExchange);

    // Queries as the B operand of the score MMA: [32 x 64] K-major swizzled
    // atoms, rows 0-15 the bf16 hi parts of the 16 heads, rows 16-31 the lo
    // parts (heads past HG are zero); and the running softmax state.
    for (int i = tid; i < kMlaMaxHG * (kMlaRow / 8); i += kComputeThreads) {
        const int n = i / (kMlaRow / 8), kc = i % (kMlaRow / 8);  // head, 8-element chunk
        float v[8];
        if (n < HG) {
            const float4 v0 = reinterpret_cast<const float4 *>(qt + n * kMlaRow)[2 * kc];
            const float4 v1 = reinterpret_cast<const float4 *>(qt + n * kMlaRow)[2 * kc + 1];
            v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w;
            v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * e]), h1 = __float2bfloat16_rn(v[2 * e + 1]);
            const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * e] - __bfloat162float(h0));
            const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * e + 1] - __bfloat162float(h1));
            hi[e] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                    (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
            lo[e] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
                    (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
        }
        uint8_t *atom = smem + p.off_qb + (kc >> 3) * kMlaQAtomBytes;
        *reinterpret_cast<uint4 *>(atom + mla_atom_off(n, (kc & 7) * 8)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(atom + mla_atom_off(kMlaMaxHG + n, (kc & 7) * 8)) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (tid < kMlaMaxHG) {
        m_st[tid] = -INFINITY;
        l_st[tid] = 0.f;
    }
    fence_proxy_async_smem();
    compute_bar<kComputeThreads>();
    if (tid == 0) mbar_arrive(bar_qready);
    // The new token's latent row (last block), built while the MMA warp issues
    // the first tile's scores: bf16 RMSNorm of the latent and bf16 rope of the
    // key; one block appends it to the cache. Then its score per head (base
    // 2) from the fp32 queries, which peers may overwrite only after this.
    if (has_new) {
        const uint16_t *ar = p.a + static_cast<size_t>(b) * p.a_stride + p.a_off;
        float ss = 0.f;
        for (int i = tid; i < kMlaKv; i += kComputeThreads) {
            const float v = bf16_bits(ar[i]);
            ss = fmaf(v, v, ss);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) scr[kMlaNope + warp] = ss;
        compute_bar<kComputeThreads>();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kComputeWarps; ++w) tot += scr[kMlaNope + w];
        const float inv = 1.0f / sqrtf(tot / static_cast<float>(kMlaKv) + p.eps);
        for (int i = tid; i < kMlaKv; i += kComputeThreads)
            newrow[i] = __bfloat16_as_ushort(__float2bfloat16_rn(bf16_bits(p.g_kv[i]) * bf16_bits(ar[i]) * inv));
        if (tid < kMlaRope / 2) {
            float x0 = bf16_bits(ar[kMlaKv + tid]), x1 = bf16_bits(ar[kMlaKv + tid + kMlaRope / 2]);
            if (p.rope) mla_rope(x0, x1, L, p.rope_inv_freq[tid]);
            newrow[kMlaKv + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(x0));
            newrow[kMlaKv + tid + kMlaRope / 2] = __bfloat16_as_ushort(__float2bfloat16_rn(x1));
        }
        compute_bar<kComputeThreads>();
        if (g == 0) {
            uint16_t *crow = p.cache + (static_cast<size_t>(b) * p.max_ctx + L) * kMlaRow;
            for (int i = tid; i < kMlaRow / 8; i += kComputeThreads)
                reinterpret_cast<uint4 *>(crow)[i] = reinterpret_cast<const uint4 *>(newrow)[i];
        }
        for (int h = warp; h < HG; h += kComputeWarps) {
            float s = 0.f;
            for (int k = lane; k < kMlaRow; k += 32) s = fmaf(qt[h * kMlaRow + k], bf16_bits(newrow[k]), s);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (lane == 0) s_new[h] = s;
        }
        compute_bar<kComputeThreads>();
    }
    // The fp32 queries are dead here; their space receives the peers' partials.
    if (tid == 0)
        for (int q = 0; q < C; ++q)
            if (q != r) mbar_arrive_remote(map_to_rank(bar_qfree, q));

    // ---- B: latent attention on the tensor cores --------------------------------
    // The MMA warp computes the scores of tile t + 1 while these warps run the
    // softmax of tile t. TMEM lanes 32 (warp % 4) + lane are this thread's tile
    // row (scores) and latent dim within a 128-dim block (outputs); warps 0-3
    // take heads 0-7 of the scores and latent blocks 0-1, warps 4-7 heads 8-15
    // and blocks 2-3.
    const int wq = warp & 3, wh = warp >> 2;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * wq) << 16);
    float acc[2][kMlaMaxHG];  // unnormalised o^T, latent dims 128 (2 wh + i) + 32 wq + lane
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int h = 0; h < kMlaMaxHG; ++h) acc[i][h] = 0.f;
    auto fold = [&](int u) {  // acc = acc alpha_u + O_u
        mla_wait<false>(bar_o0 + 8u * (u & 1), (u >> 1) & 1, p, timed_out, kSiteStageFull);
        tcgen05_fence_after();
        const float *al = alpha + kMlaMaxHG * (u & 1);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float o[16];
            tmem_ld_x16(tl + 64 + 64 * (u & 1) + 16 * (2 * wh + i), o);
#pragma unroll
            for (int h = 0; h < kMlaMaxHG; ++h) acc[i][h] = acc[i][h] * al[h] + o[h];
        }
        tcgen05_fence_before();
    };
    for (int t = 0; t < n_tiles; ++t) {
        const int nvalid = min(kMlaTileRows, cache_e - row_s - t * kMlaTileRows);
        float *rmax = red_max + 8 * kMlaMaxHG * (t & 1), *rsum = red_sum + 8 * kMlaMaxHG * (t & 1);
        mla_wait<false>(bar_s0 + 8u * (t & 1), (t >> 1) & 1, p, timed_out, kSiteStageFull);
        tcgen05_fence_after();
        // scores of tile row 32 wq + lane, heads 8 wh .. + 8 (base-2 units): hi + lo
        float sv[8], sl[8];
        mla_tmem_ld_x8(tl + 2 * kMlaMaxHG * (t & 1) + 8 * wh, sv);
        mla_tmem_ld_x8(tl + 2 * kMlaMaxHG * (t & 1) + kMlaMaxHG + 8 * wh, sl);
        const int row = 32 * wq + lane;
        const bool valid = row < nvalid;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            sv[j] += sl[j];
            float mx = valid ? sv[j] : -INFINITY;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (lane == 0) rmax[warp * 16 + j] = mx;
        }
        tcgen05_fence_before();
        compute_bar<kComputeThreads>();
        // probabilities against the new running max; P as the K-major B
        // operand of the value MMA (element (head, row))
        uint8_t *pt = smem + p.off_pb + (t & 1) * 2 * kMlaAtomBytes;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int h = 8 * wh + j;
            float tmax = rmax[(4 * wh) * 16 + j];
#pragma unroll
            for (int w = 1; w < 4; ++w) tmax = fmaxf(tmax, rmax[(4 * wh + w) * 16 + j]);
            const float m_new = fmaxf(m_st[h], tmax);
            const float pv = valid && h < HG ? fast_exp2(sv[j] - m_new) : 0.f;
            *reinterpret_cast<uint16_t *>(pt + (row >> 6) * kMlaAtomBytes + mla_atom_off(h, row & 63)) =
                __bfloat16_as_ushort(__float2bfloat16_rn(pv));
            float sm = pv;
#pragma unroll
            for (int off2 = 16; off2 > 0; off2 >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off2);
            if (lane == 0) rsum[warp * 16 + j] = sm;
        }
        fence_proxy_async_smem();  // P is read by the tensor cores
        compute_bar<kComputeThreads>();
        if (tid == 0) mbar_arrive(bar_p0 + 8u * (t & 1));
        // per-head state: new max, rescale factor, running sum (fixed warp order)
        if (tid < kMlaMaxHG) {
            const int h = tid, hw = h >> 3, j = h & 7;
            float tmax = rmax[(4 * hw) * 16 + j], tsum = rsum[(4 * hw) * 16 + j];
#pragma unroll
            for (int w = 1; w < 4; ++w) {
                tmax = fmaxf(tmax, rmax[(4 * hw + w) * 16 + j]);
                tsum += rsum[(4 * hw + w) * 16 + j];
            }
            const float m_old = m_st[h];
            const float m_new = fmaxf(m_old, tmax);
            const float al = fast_exp2(m_old - m_new);  // 0 while nothing was seen
            alpha[kMlaMaxHG * (t & 1) + h] = al;
            l_st[h] = l_st[h] * al + tsum;
            m_st[h] = m_new;
        }
        if (t >= 1) fold(t - 1);
    }
    if (n_tiles > 0) fold(n_tiles - 1);
    compute_bar<kComputeThreads>();
    // The new row, attended on CUDA cores: its score per head, the state
    // update, and its value folded into the partial output.
    if (has_new) {
        if (tid < HG) {
            const int h = tid;
            const float m_old = m_st[h];
            const float m_new = fmaxf(m_old, s_new[h]);
            const float al = fast_exp2(m_old - m_new), pn = fast_exp2(s_new[h] - m_new);
            alpha[h] = al;
            s_new[h] = pn;
            l_st[h] = l_st[h] * al + pn;
            m_st[h] = m_new;
        }
        compute_bar<kComputeThreads>();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float c = bf16_bits(newrow[128 * (2 * wh + i) + 32 * wq + lane]);
#pragma unroll
            for (int h = 0; h < kMlaMaxHG; ++h)
                if (h < HG) acc[i][h] = acc[i][h] * alpha[h] + s_new[h] * c;
        }
    }

    // ---- C: sparse ClusterReduce -- each head goes to the block that owns it --
    {
        // stage each head's (o^T [512], m, l, 0, 0) where the query operand was
        // (every MMA has completed), then one bulk copy per head to its owner
        float *stage = reinterpret_cast<float *>(smem + p.off_qb);  // [HG][516]
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int h = 0; h < kMlaMaxHG; ++h)
                if (h < HG) stage[h * (kMlaKv + 4) + 128 * (2 * wh + i) + 32 * wq + lane] = acc[i][h];
        if (tid < HG)
            *reinterpret_cast<float4 *>(stage + tid * (kMlaKv + 4) + kMlaKv) =
                make_float4(m_st[tid], l_st[tid], 0.f, 0.f);
        fence_proxy_async_smem();
        compute_bar<kComputeThreads>();
        mla_wait<true>(bar_qfree, 0, p, timed_out, kSiteSoftmaxExchange);
        if (tid < HG && tid / HPB != r) {
            const int h = tid, owner = h / HPB, slot = h % HPB;
            bulk_copy_to_rank(map_to_rank(smem_addr(recv + (slot * C + r) * (kMlaKv + 4)), owner),
                              smem_addr(stage + h * (kMlaKv + 4)), static_cast<uint32_t>((kMlaKv + 4) * 4),
                              map_to_rank(bar_red, owner));
        }
        for (int idx = tid; idx < HPB * (kMlaKv + 4) / 4; idx += kComputeThreads) {  // my own heads
            const int slot = idx / ((kMlaKv + 4) / 4), c = idx % ((kMlaKv + 4) / 4);
            reinterpret_cast<float4 *>(recv + (slot * C + r) * (kMlaKv + 4))[c] =
                reinterpret_cast<const float4 *>(stage + (r * HPB + slot) * (kMlaKv + 4))[c];
        }
        compute_bar<kComputeThreads>();  // own partials written
        mla_wait<true>(bar_red, 0, p, timed_out, kSiteSoftmaxExchange);
        // combine in block order: o = sum_r 2^(m_r - M) o_r / sum_r 2^(m_r - M) l_r,
        // the weights w_r = 2^(m_r - M) / L computed once per head
        float *wgt = scr;  // [HPB][16]
        float *split_ml = scr + kComputeWarps * kMlaV;  // [HPB][2]: (M, L) of this split
        if (warp < (HPB * kMlaMaxHG + 31) / 32) {  // 16 lanes per head, lane q for block q
            const int i = tid / kMlaMaxHG, q = tid % kMlaMaxHG;
            const bool act = i < HPB && q < C;
            const float *rv = recv + i * C * (kMlaKv + 4);
            const float mq = act ? rv[q * (kMlaKv + 4) + kMlaKv] : -INFINITY;
            float M = mq;
#pragma unroll
            for (int off = kMlaMaxHG / 2; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
            const float e = mq != -INFINITY ? fast_exp2(mq - M) : 0.f;
            const float lq = act ? rv[q * (kMlaKv + 4) + kMlaKv + 1] : 0.f;
            // block-order sum of e_q l_q: a fixed shuffle tree over the 16 lanes
            float Lsum = e * lq;
#pragma unroll
            for (int off = kMlaMaxHG / 2; off > 0; off >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, off);
            // (a split with no rows at all has Lsum = 0 and contributes nothing)
            if (i < HPB) wgt[i * kMlaMaxHG + q] = Lsum > 0.f ? e / Lsum : 0.f;  // 0 for q >= C
            if (i < HPB && q == 0) {  // this split's max and sum, for the combine of splits
                split_ml[2 * i] = M;
                split_ml[2 * i + 1] = Lsum;
            }
        }
        compute_bar<kComputeThreads>();
        for (int idx = tid; idx < HPB * kMlaKv; idx += kComputeThreads) {
            const int i = idx / kMlaKv, d = idx % kMlaKv;
            const float *rv = recv + i * C * (kMlaKv + 4) + d;
            const float *w = wgt + i * kMlaMaxHG;
            float o = 0.f;
#pragma unroll
            for (int q = 0; q < kMlaMaxHG; ++q)  // blocks past C have weight 0
                o = fmaf(w[q], rv[min(q, C - 1) * (kMlaKv + 4)], o);
            ofin[idx] = o;
        }
        compute_bar<kComputeThreads>();
        // v_h = o_h W_v,h from the ring's [256 x 64] W_v boxes: thread tid takes
        // the 8 value columns of 16-byte chunk tid % 8 in box rows tid / 8 + 32 k
        cur = RingCursor();
        for (int n = 0; n < 4 * HPB + (kSStages + kVStages) * n_tiles; ++n) cur.advance(NS);
        const int cc = tid & 7, rg = tid >> 3;
        for (int ii = 0; ii < HPB; ++ii) {
            const int h = g * HG + r * HPB + ii;
            float part[2][8];
#pragma unroll
            for (int cb = 0; cb < 2; ++cb)
#pragma unroll
                for (int e = 0; e < 8; ++e) part[cb][e] = 0.f;
#pragma unroll 1
            for (int sq = 0; sq < 4; ++sq) {  // stage (row block, column block) = (sq / 2, sq % 2)
                const int rb = sq >> 1;
                const uint8_t *st = stage_ready();
                float pk[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int k = 0; k < kMlaWeightRows / 32; ++k) {
                    const int row = rg + 32 * k;
                    const float oj = ofin[ii * kMlaKv + kMlaWeightRows * rb + row];
                    float f[8];
                    unpack8_bf16(*reinterpret_cast<const uint4 *>(st + row * 128 + ((cc ^ (row & 7)) << 4)), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) pk[e] = fmaf(oj, f[e], pk[e]);
                }
                stage_done();
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    if (sq & 1) part[1][e] += pk[e];
                    else part[0][e] += pk[e];
                }
            }
            // sum over the 32 row groups: 4 in a warp by shuffles, 8 warps in smem
#pragma unroll
            for (int cb = 0; cb < 2; ++cb)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float v = part[cb][e];
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    if (lane < 8) scr[warp * kMlaV + 64 * cb + 8 * cc + e] = v;
                }
            compute_bar<kComputeThreads>();
            if (tid < kMlaV) {
                float vsum = 0.f;
#pragma unroll
                for (int w = 0; w < kComputeWarps; ++w) vsum += scr[w * kMlaV + tid];
                if (S == 1) {
                    p.v[static_cast<size_t>(b) * p.nh * kMlaV + h * kMlaV + tid] =
                        __bfloat16_as_ushort(__float2bfloat16_rn(vsum));
                } else {  // this split's v_h (normalised by its own sum) with its (M, L)
                    float *rec = p.vpart + (static_cast<size_t>(b) * p.nh + h) * S * kMlaSplitRec +
                                 split * kMlaSplitRec;
                    rec[tid] = vsum;
                    if (tid < 2) rec[kMlaV + tid] = split_ml[2 * ii + tid];
                }
            }
            compute_bar<kComputeThreads>();
        }
        if (S > 1) {
            // Combine of the row splits [CF §5.2, the cache partitioned across
            // clusters]: block r of every split owns the same heads; the last
            // of them to get here sums the splits in split order,
            //   v_h = sum_s 2^(M_s - M) L_s v_s / sum_s 2^(M_s - M) L_s.
            // (A barrier follows the block's last store, so one thread's
            // release covers them.)
            volatile int *last = reinterpret_cast<volatile int *>(s_new);
            if (tid == 0) {
                unsigned *ctr = p.vcount + (static_cast<size_t>(b) * NG + g) * C + r;
                const bool is_last = atomic_add_acq_rel_gpu(ctr, 1u) == static_cast<unsigned>(S - 1);
                if (is_last) *ctr = 0u;  // ready for the next launch
                *last = is_last ? 1 : 0;
            }
            compute_bar<kComputeThreads>();
            if (*last) {
                for (int idx = tid; idx < HPB * kMlaV; idx += kComputeThreads) {
                    const int ii = idx / kMlaV, c = idx % kMlaV;
                    const int h = g * HG + r * HPB + ii;
                    const float *rec = p.vpart + (static_cast<size_t>(b) * p.nh + h) * S * kMlaSplitRec;
                    float M = -INFINITY;
                    for (int q = 0; q < S; ++q) M = fmaxf(M, __ldcg(rec + q * kMlaSplitRec + kMlaV));
                    float num = 0.f, den = 0.f;
                    for (int q = 0; q < S; ++q) {
                        const float mq = __ldcg(rec + q * kMlaSplitRec + kMlaV);
                        const float w = mq == -INFINITY
                                            ? 0.f
                                            : fast_exp2(mq - M) * __ldcg(rec + q * kMlaSplitRec + kMlaV + 1);
                        num = fmaf(w, __ldcg(rec + q * kMlaSplitRec + c), num);
                        den += w;
                    }
                    p.v[static_cast<size_t>(b) * p.nh * kMlaV + h * kMlaV + c] =
                        __bfloat16_as_ushort(__float2bfloat16_rn(num / den));
                }
            }
        }
    }
    if (warp == 0) {
        tcgen05_fence_after();
        tmem_dealloc(tmem, 256);
    }
    // The next kernel (the output projection) may start streaming its weights
    // now: launched earlier, its loads would compete with this kernel's.
    grid_dependents_launch();
    cluster_sync_all();  // no block leaves while a peer may still push into it
}

}  // namespace cfa
