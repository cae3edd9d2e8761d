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
// which equals attention over the decompressed keys and values.
//
// Grid: B x (nh / HG) clusters of C blocks; cluster (b, g) owns heads
// [g HG, (g+1) HG) of sequence b and block r of it owns the latent rows
// [T r / C, T (r+1) / C) of T = L + 1 rows (the new token's row is the last).
//  A  Absorption [CF §3.2 deferred projection]: block r computes q~ and the
//     rotated rope query of its HPB = HG / C heads (reading their W_k block
//     once) and pushes them to every block of the cluster (ClusterGather over
//     DSMEM, st.async + transaction counts), so every block holds all HG
//     queries. The last block builds the new latent row (RMSNorm of the
//     latent part, rope of the key part, bf16) on chip; one block appends it.
//  B  Latent attention over the block's rows for all HG heads: latent rows
//     arrive by TMA in 128-byte-swizzled [32 x 64] boxes through a stage
//     ring; per 32-row tile, each warp scores its heads (lane = row), keeps a
//     base-2 online softmax per head, and all warps accumulate the
//     unnormalised latent outputs o_h (head quad x 256 latent dims each).
//  C  Sparse ClusterReduce [CF §5.2]: a reduce-scatter over the cluster --
//     block r receives, for its own HPB heads only, every block's (m, l, o)
//     and combines them in block order (deterministic); then v_h = o_h W_v,h.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "cfa_device.cuh"
#include "cfa_internal.h"
#include "cfa_tile.cuh"

namespace cfa {

// Byte offset of row t, latent columns [64 kc + 8 j, +8) in a tile of
// [rows x 64] boxes with 128-byte swizzle (box_stride bytes apart).
__device__ __forceinline__ uint32_t mla_tile_off(int box_stride, int t, int kc, int j) {
    return static_cast<uint32_t>(kc * box_stride + t * 128 + ((j ^ (t & 7)) << 4));
}

// HPW: heads each warp scores (HG / 8, at least 1).
template <int HPW>
__global__ void __launch_bounds__(kThreads, 1)
mla_attention_kernel(const __grid_constant__ CUtensorMap tm_cache,
                     const __grid_constant__ CUtensorMap tm_wkvb, const MlaParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int C = p.C, HG = p.HG, HPB = p.HPB, NS = p.nstages;
    const int r = static_cast<int>(cluster_ctarank());
    const int cluster = blockIdx.x / C;
    const int NG = p.nh / HG;
    const int b = cluster / NG, g = cluster % NG;
    const int L = p.ctx_lens[b];
    const int T = L + 1;
    const int row_s = static_cast<int>((static_cast<long long>(T) * r) / C);
    const int row_e = static_cast<int>((static_cast<long long>(T) * (r + 1)) / C);
    const int cache_e = min(row_e, L);                       // rows read from the cache
    const bool has_new = row_e == T;                         // this block attends the new row
    const int n_tiles = cache_e > row_s ? (cache_e - row_s + kMlaTileRows - 1) / kMlaTileRows : 0;

    float *qt = reinterpret_cast<float *>(smem + p.off_qt);        // [HG][576] scaled queries
    float *pbuf = reinterpret_cast<float *>(smem + p.off_p);       // [32][HG] probabilities
    float *alpha = reinterpret_cast<float *>(smem + p.off_alpha);  // [HG] rescale of o
    float *recv = reinterpret_cast<float *>(smem + p.off_recv);    // [HPB][C][516]
    float *ofin = reinterpret_cast<float *>(smem + p.off_ofin);    // [HPB][512]
    float *scr = reinterpret_cast<float *>(smem + p.off_scr);      // [8][128] + 64
    uint8_t *newrow = smem + p.off_newrow;                         // 1-row tile (1152 B)
    const uint32_t bar_full0 = smem_addr(smem + p.off_bars);
    const uint32_t bar_empty0 = bar_full0 + 8u * NS;
    const uint32_t bar_q = bar_full0 + 16u * NS;      // every peer's queries have landed
    const uint32_t bar_red = bar_q + 8u;              // every peer's partials for my heads
    volatile int *timed_out = reinterpret_cast<volatile int *>(smem + p.off_bars + 16 * NS + 16);

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full0 + 8u * s, 1);
            mbar_init(bar_empty0 + 8u * s, kComputeWarps);
        }
        mbar_init(bar_q, 1);
        mbar_init(bar_red, 1);
        *timed_out = 0;
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_q, static_cast<uint32_t>((C - 1) * HPB * kMlaRow * 4));
        mbar_arrive_expect_tx(bar_red, static_cast<uint32_t>((C - 1) * HPB * (kMlaKv + 4) * 4));
    }
    __syncthreads();
    grid_dependents_launch();
    cluster_arrive();  // barriers announced; waited for before the first push

    if (warp == kComputeWarps) {
        // ------------------------------------------------------------ load warp
        if (lane == 0) {
            // W_v blocks of this block's heads, wanted at the end: warm L2 now.
            for (int i = 0; i < HPB; ++i) {
                const int h = g * HG + r * HPB + i;
                for (int y = 0; y < kMlaKv; y += 256)
                    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                                 :: "l"(reinterpret_cast<uint64_t>(&tm_wkvb)),
                                    "r"(h * (kMlaNope + kMlaV) + kMlaNope), "r"(y)
                                 : "memory");
            }
            grid_dependency_wait();  // cache rows may come from the previous step
            RingCursor cur;
            for (int i = 0; i < n_tiles; ++i) {
                if (cur.wrapped)
                    mbar_wait_bounded<false>(bar_empty0 + 8u * cur.stage, cur.phase ^ 1u,
                                             p.timeout_ns, timed_out, p.status, kSiteStageEmpty);
                const uint32_t full = bar_full0 + 8u * cur.stage;
                const uint32_t dst = smem_addr(smem + p.off_ring) + cur.stage * kMlaTileBytes;
                mbar_arrive_expect_tx(full, kMlaTileBytes);
                const int row = b * p.max_ctx + row_s + i * kMlaTileRows;
                for (int kc = 0; kc < kMlaBoxes; ++kc)
                    tma_load_2d(dst + kc * kMlaTileRows * 128, &tm_cache, kc * 64, row, full);
                cur.advance(NS);
            }
            for (int s = 0; s < NS; ++s) {  // drain
                if (s >= cur.stage && !cur.wrapped) break;
                volatile int ignore = 0;
                mbar_wait_bounded<false>(bar_full0 + 8u * s, s < cur.stage ? cur.phase : cur.phase ^ 1u,
                                         p.timeout_ns, &ignore, p.status, kSiteStageFull);
            }
        } else {
            grid_dependency_wait();
        }
        __syncwarp();
        cluster_wait();
        cluster_sync_all();
        return;
    }

    // --------------------------------------------------------------- compute
    grid_dependency_wait();
    // ---- A: absorbed queries of this block's heads, pushed to the cluster ----
    {
        float *qn = scr;  // [128] q_nope of the head being absorbed
        for (int i = 0; i < HPB; ++i) {
            const int hl = r * HPB + i;             // head within the group
            const int h = g * HG + hl;
            const uint16_t *qh = p.q + static_cast<size_t>(b) * p.nh * kMlaQk + h * kMlaQk;
            if (tid < kMlaNope) qn[tid] = bf16_bits(qh[tid]);
            compute_bar<kComputeThreads>();
            float *dst = qt + hl * kMlaRow;
            // q~[j] = sum_c W_kvb[j, h*256 + c] q_nope[c]: rows tid and tid + 256,
            // all 32 16-byte loads of both rows issued before any use
            {
                const size_t ld = static_cast<size_t>(p.nh) * (kMlaNope + kMlaV);
                const uint4 *w0 = reinterpret_cast<const uint4 *>(p.W_kvb + tid * ld + h * (kMlaNope + kMlaV));
                const uint4 *w1 = reinterpret_cast<const uint4 *>(p.W_kvb + (tid + kComputeThreads) * ld +
                                                                  h * (kMlaNope + kMlaV));
                uint4 r0[kMlaNope / 8], r1[kMlaNope / 8];
#pragma unroll
                for (int c8 = 0; c8 < kMlaNope / 8; ++c8) {
                    r0[c8] = __ldg(w0 + c8);
                    r1[c8] = __ldg(w1 + c8);
                }
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int c8 = 0; c8 < kMlaNope / 8; ++c8) {
                    float f0[8], f1[8];
                    unpack8_bf16(r0[c8], f0);
                    unpack8_bf16(r1[c8], f1);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        a0 = fmaf(f0[e], qn[c8 * 8 + e], a0);
                        a1 = fmaf(f1[e], qn[c8 * 8 + e], a1);
                    }
                }
                dst[tid] = a0 * p.qscale;
                dst[tid + kComputeThreads] = a1 * p.qscale;
            }
            // rope of the rope query at position L (rotate-half, angle in fp64)
            if (tid < kMlaRope / 2) {
                const int k = tid;
                float x0 = bf16_bits(qh[kMlaNope + k]), x1 = bf16_bits(qh[kMlaNope + k + kMlaRope / 2]);
                if (p.rope) {
                    const double ang = static_cast<double>(L) * p.rope_inv_freq[k];
                    const double red = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);
                    float sn, cs;
                    sincosf(static_cast<float>(red), &sn, &cs);
                    const float y0 = x0 * cs - x1 * sn, y1 = x1 * cs + x0 * sn;
                    x0 = y0;
                    x1 = y1;
                }
                dst[kMlaKv + k] = x0 * p.qscale;
                dst[kMlaKv + k + kMlaRope / 2] = x1 * p.qscale;
            }
            compute_bar<kComputeThreads>();
        }
        cluster_wait();  // every peer's barriers exist before the first push
        // ClusterGather: my heads' 576 scaled query values to every peer
        const int chunks = HPB * kMlaRow / 4;
        const uint32_t my0 = smem_addr(qt + r * HPB * kMlaRow);
        for (int idx = tid; idx < (C - 1) * chunks; idx += kComputeThreads) {
            const int pi = idx / chunks, c = idx % chunks;
            const int peer = pi < r ? pi : pi + 1;
            const float4 val = reinterpret_cast<const float4 *>(qt + r * HPB * kMlaRow)[c];
            push_16B(map_to_rank(my0 + 16u * c, peer), val, map_to_rank(bar_q, peer));
        }
    }
    // The new token's latent row (last block): bf16 RMSNorm of the latent and
    // bf16 rope of the key, in the one-row tile layout; one block appends it.
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
        uint16_t *nr = reinterpret_cast<uint16_t *>(newrow);  // row 0: plain 1152-byte row
        for (int i = tid; i < kMlaKv; i += kComputeThreads)
            nr[i] = __bfloat16_as_ushort(__float2bfloat16_rn(bf16_bits(p.g_kv[i]) * bf16_bits(ar[i]) * inv));
        if (tid < kMlaRope / 2) {
            const int k = tid;
            float x0 = bf16_bits(ar[kMlaKv + k]), x1 = bf16_bits(ar[kMlaKv + k + kMlaRope / 2]);
            if (p.rope) {
                const double ang = static_cast<double>(L) * p.rope_inv_freq[k];
                const double red = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);
                float sn, cs;
                sincosf(static_cast<float>(red), &sn, &cs);
                const float y0 = x0 * cs - x1 * sn, y1 = x1 * cs + x0 * sn;
                x0 = y0;
                x1 = y1;
            }
            nr[kMlaKv + k] = __bfloat16_as_ushort(__float2bfloat16_rn(x0));
            nr[kMlaKv + k + kMlaRope / 2] = __bfloat16_as_ushort(__float2bfloat16_rn(x1));
        }
        compute_bar<kComputeThreads>();
        if (g == 0) {
            uint16_t *crow = p.cache + (static_cast<size_t>(b) * p.max_ctx + L) * kMlaRow;
            for (int i = tid; i < kMlaRow / 8; i += kComputeThreads)
                reinterpret_cast<uint4 *>(crow)[i] = reinterpret_cast<const uint4 *>(nr)[i];
        }
    }
    mbar_wait_bounded<true>(bar_q, 0, p.timeout_ns, timed_out, p.status, kSiteQExchange);

    // ---- B: latent attention over this block's rows, all HG heads --------------
    const int h_sc = warp * HPW;                                    // first head this warp scores
    const bool scores_warp = h_sc < HG;
    float m_run[HPW], l_run[HPW];
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
        m_run[hh] = -INFINITY;
        l_run[hh] = 0.f;
    }
    const int hq = warp % 4;                   // output head quad
    const int dh = warp / 4;                   // output latent half
    float acc[4][8];
#pragma unroll
    for (int hh = 0; hh < 4; ++hh)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[hh][e] = 0.f;

    auto process_tile = [&](const uint8_t *tile, int box_stride, int nvalid) {
        // scores: lane = row, this warp's heads
        if (scores_warp) {
            // two partial sums per head (even / odd 8-column chunks) for ILP
            float s[HPW][2];
#pragma unroll
            for (int hh = 0; hh < HPW; ++hh) s[hh][0] = s[hh][1] = 0.f;
            if (lane < nvalid) {
#pragma unroll 1
                for (int kc = 0; kc < kMlaBoxes; ++kc) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float c8[8];
                        unpack8_bf16(*reinterpret_cast<const uint4 *>(tile + mla_tile_off(box_stride, lane, kc, j)), c8);
#pragma unroll
                        for (int hh = 0; hh < HPW; ++hh) {
                            const float4 *qv = reinterpret_cast<const float4 *>(qt + (h_sc + hh) * kMlaRow + kc * 64 + j * 8);
                            const float4 q0 = qv[0], q1 = qv[1];
                            float a = s[hh][j & 1];
                            a = fmaf(c8[0], q0.x, a);
                            a = fmaf(c8[1], q0.y, a);
                            a = fmaf(c8[2], q0.z, a);
                            a = fmaf(c8[3], q0.w, a);
                            a = fmaf(c8[4], q1.x, a);
                            a = fmaf(c8[5], q1.y, a);
                            a = fmaf(c8[6], q1.z, a);
                            a = fmaf(c8[7], q1.w, a);
                            s[hh][j & 1] = a;
                        }
                    }
                }
            }
#pragma unroll
            for (int hh = 0; hh < HPW; ++hh) {
                const float sv = s[hh][0] + s[hh][1];
                float mt = lane < nvalid ? sv : -INFINITY;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
                const float m_new = fmaxf(m_run[hh], mt);
                const float pr = lane < nvalid ? exp2f(sv - m_new) : 0.f;
                float ps = pr;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
                const float al = exp2f(m_run[hh] - m_new);  // 0 while nothing was seen
                l_run[hh] = l_run[hh] * al + ps;
                m_run[hh] = m_new;
                pbuf[lane * HG + h_sc + hh] = pr;
                if (lane == 0) alpha[h_sc + hh] = al;
            }
        }
        compute_bar<kComputeThreads>();
        // o_h += sum_t p[t][h] c_t: 4 heads x 8 latent dims per thread
        if (hq * 4 < HG) {
            const int kc = dh * 4 + lane / 8, j = lane % 8;
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                const float al = hq * 4 + hh < HG ? alpha[hq * 4 + hh] : 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[hh][e] *= al;
            }
            for (int t = 0; t < nvalid; ++t) {
                float c8[8];
                unpack8_bf16(*reinterpret_cast<const uint4 *>(tile + mla_tile_off(box_stride, t, kc, j)), c8);
                const float *pr = pbuf + t * HG + hq * 4;
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    const float pv = hq * 4 + hh < HG ? pr[hh] : 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[hh][e] = fmaf(pv, c8[e], acc[hh][e]);
                }
            }
        }
        compute_bar<kComputeThreads>();
    };

    RingCursor cur;
    for (int i = 0; i < n_tiles; ++i) {
        const int s = cur.stage;
        mbar_wait_bounded<false>(bar_full0 + 8u * s, cur.phase, p.timeout_ns, timed_out, p.status,
                                 kSiteStageFull);
        const int nvalid = min(kMlaTileRows, cache_e - row_s - i * kMlaTileRows);
        process_tile(smem + p.off_ring + s * kMlaTileBytes, kMlaTileRows * 128, nvalid);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty0 + 8u * s);
        cur.advance(NS);
    }
    if (has_new) process_tile(newrow, 128, 1);

    // ---- C: sparse ClusterReduce -- each head goes to the block that owns it --
    {
        // (m, l) of the heads this warp scored, then o of the heads this thread holds
        if (scores_warp && lane == 0) {
#pragma unroll
            for (int hh = 0; hh < HPW; ++hh) {
                const int h = h_sc + hh, owner = h / HPB, slot = h % HPB;
                float *dst = recv + (slot * C + r) * (kMlaKv + 4) + kMlaKv;
                const float4 st = make_float4(m_run[hh], l_run[hh], 0.f, 0.f);
                if (owner == r) {
                    *reinterpret_cast<float4 *>(dst) = st;
                } else {
                    push_16B(map_to_rank(smem_addr(dst), owner), st, map_to_rank(bar_red, owner));
                }
            }
        }
        if (hq * 4 < HG) {
            const int d0 = dh * 256 + lane * 8;
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
                const int h = hq * 4 + hh;
                if (h >= HG) continue;
                const int owner = h / HPB, slot = h % HPB;
                float *dst = recv + (slot * C + r) * (kMlaKv + 4) + d0;
                const float4 v0 = make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
                const float4 v1 = make_float4(acc[hh][4], acc[hh][5], acc[hh][6], acc[hh][7]);
                if (owner == r) {
                    reinterpret_cast<float4 *>(dst)[0] = v0;
                    reinterpret_cast<float4 *>(dst)[1] = v1;
                } else {
                    push_16B(map_to_rank(smem_addr(dst), owner), v0, map_to_rank(bar_red, owner));
                    push_16B(map_to_rank(smem_addr(dst + 4), owner), v1, map_to_rank(bar_red, owner));
                }
            }
        }
        compute_bar<kComputeThreads>();  // own partials written
        mbar_wait_bounded<true>(bar_red, 0, p.timeout_ns, timed_out, p.status, kSiteSoftmaxExchange);
        // combine in block order: o = sum_r 2^(m_r - M) o_r / sum_r 2^(m_r - M) l_r
        for (int i = 0; i < HPB; ++i) {
            const float *rv = recv + i * C * (kMlaKv + 4);
            float M = -INFINITY;
            for (int q = 0; q < C; ++q) M = fmaxf(M, rv[q * (kMlaKv + 4) + kMlaKv]);
            float Lsum = 0.f;
            for (int q = 0; q < C; ++q) {
                const float mq = rv[q * (kMlaKv + 4) + kMlaKv];
                if (mq != -INFINITY) Lsum += exp2f(mq - M) * rv[q * (kMlaKv + 4) + kMlaKv + 1];
            }
            const float inv = 1.0f / Lsum;
            for (int d = tid; d < kMlaKv; d += kComputeThreads) {
                float o = 0.f;
                for (int q = 0; q < C; ++q) {
                    const float mq = rv[q * (kMlaKv + 4) + kMlaKv];
                    if (mq != -INFINITY) o += exp2f(mq - M) * rv[q * (kMlaKv + 4) + d];
                }
                ofin[i * kMlaKv + d] = o * inv;
            }
        }
        compute_bar<kComputeThreads>();
        // v_h = o_h W_v,h: warp w sums rows j = w (mod 8), lane takes 4 columns
        for (int ii = 0; ii < HPB; ++ii) {
            const int h = g * HG + r * HPB + ii;
            float part[4] = {0.f, 0.f, 0.f, 0.f};
            const size_t ld = static_cast<size_t>(p.nh) * (kMlaNope + kMlaV);
            const uint16_t *wv0 = p.W_kvb + h * (kMlaNope + kMlaV) + kMlaNope + lane * 4;
            // rows j = warp + 8 i, i < 64: 16 loads in flight per round
#pragma unroll 1
            for (int i0 = 0; i0 < kMlaKv / kComputeWarps; i0 += 16) {
                uint2 wv[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    wv[i] = __ldg(reinterpret_cast<const uint2 *>(wv0 + (warp + (i0 + i) * kComputeWarps) * ld));
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float oj = ofin[ii * kMlaKv + warp + (i0 + i) * kComputeWarps];
                    part[0] = fmaf(oj, bf16_lo(wv[i].x), part[0]);
                    part[1] = fmaf(oj, bf16_hi(wv[i].x), part[1]);
                    part[2] = fmaf(oj, bf16_lo(wv[i].y), part[2]);
                    part[3] = fmaf(oj, bf16_hi(wv[i].y), part[3]);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) scr[warp * kMlaV + lane * 4 + e] = part[e];
            compute_bar<kComputeThreads>();
            if (tid < kMlaV) {
                float vsum = 0.f;
#pragma unroll
                for (int w = 0; w < kComputeWarps; ++w) vsum += scr[w * kMlaV + tid];
                p.v[static_cast<size_t>(b) * p.nh * kMlaV + h * kMlaV + tid] =
                    __bfloat16_as_ushort(__float2bfloat16_rn(vsum));
            }
            compute_bar<kComputeThreads>();
        }
    }
    cluster_sync_all();  // no block leaves while a peer may still push into it
}

}  // namespace cfa
