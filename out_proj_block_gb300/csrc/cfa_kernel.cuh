// cfa_kernel.cuh -- the fused decode-attention kernel for sm_103a.
//
// Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命" (ClusterFusion
// framework analysis), written [CF §n].
//
// One launch does the whole decode step of [CF §1.1] for every head and batch
// row. The grid is n_heads clusters of C blocks, one cluster per head
// [CF §3.2]. Each block has 8 compute warps and one load warp. The load warp
// streams every byte the block needs -- its slice of W_qkv, its slice of the
// K/V cache, its slice of W_o -- through one ring of 16 KB shared-memory
// stages with TMA (2-D tensor loads for weight tiles, 1-D bulk copies for
// contiguous cache rows), so loads for the next phase are already in flight
// while the compute warps wait on a cluster exchange [CF §3.3, §4.2].
//
// Phases of a block with cluster rank r (head h):
//  A  Deferred QKV projection [CF §3.2, §5.1]: the block owns one 64-column
//     group g of head h's Q, K and V column blocks ("split head_dim") and one
//     row group rg of the hidden dimension; it multiplies its rows of x by
//     its weight tile into partial q/k/v sums.
//  X1 Cluster gather/reduce of q, k, v [CF §3.1.2]: every block pushes its
//     partials into every other block's shared memory (st.async with
//     transaction counting on the receiver's mbarrier). Each block then sums
//     the row-group partials in rank order and concatenates the column
//     groups, so all blocks hold identical q, k_new, v_new. k_new and v_new
//     are rounded to bf16; rank 0 appends them to the caches.
//  B  Split-KV attention [CF §3.2]: the block owns cached positions
//     [L*r/C, L*(r+1)/C); the last rank also owns the new token, attended
//     from its on-chip copy. Each half- or quarter-warp keeps an online
//     softmax state (m, l, o) in base-2 units; the states are merged per
//     batch row at the end.
//  X2 ClusterReduce of the softmax statistics [CF §3.1.1, §3.2]: every block
//     pushes (m_r, l_r, o_r) to every other; each block takes m = max m_r and
//     sums the rescaled l_r and o_r in rank order, so all hold identical
//     attn = o / l.
//  C  Output projection [CF §3.2]: the block owns H/C output columns and
//     multiplies attn (head h's d rows of W_o) into fp32 partials, written to
//     a per-head workspace row.
//  D  Cross-head merge: instead of the page's atomicAdd merge [CF §3.2], the
//     last block to finish a column chunk (a release/acquire counter) sums
//     the n_heads partials in head order and writes bf16 out. Deterministic.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "cfa_device.cuh"
#include "cfa_internal.h"

namespace cfa {

__device__ __forceinline__ float dot8_bf16(const float (&q)[8], uint4 k) {
    float s = q[0] * bf16_lo(k.x);
    s = fmaf(q[1], bf16_hi(k.x), s);
    s = fmaf(q[2], bf16_lo(k.y), s);
    s = fmaf(q[3], bf16_hi(k.y), s);
    s = fmaf(q[4], bf16_lo(k.z), s);
    s = fmaf(q[5], bf16_hi(k.z), s);
    s = fmaf(q[6], bf16_lo(k.w), s);
    s = fmaf(q[7], bf16_hi(k.w), s);
    return s;
}

__device__ __forceinline__ void unpack8_bf16(uint4 v, float (&f)[8]) {
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

template <int D, int MAXB>
__global__ void __launch_bounds__(kThreads, 2)
fused_decode_kernel(const __grid_constant__ CUtensorMap tm_wqkv,
                    const __grid_constant__ CUtensorMap tm_wo,
                    const KernelParams p) {
    static_assert(D == 64 || D == 128, "head_dim must be 64 or 128");
    constexpr int TK = kStageBytes / (4 * D);            // cache rows per K (or V) tile
    constexpr int LPR = D / 8;                           // lanes per cache row (16 B each)
    constexpr int RPW = 32 / LPR;                        // rows a warp covers per step
    constexpr int NSTATE = kComputeWarps * RPW;          // online-softmax states per block
    constexpr int KV_STEPS = TK / (kComputeWarps * RPW); // steps per warp per tile
    constexpr int SMW = D + 4;                           // floats per softmax record
    static_assert(KV_STEPS * kComputeWarps * RPW == TK, "tile rows must split evenly");

    extern __shared__ __align__(1024) uint8_t smem[];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int r = static_cast<int>(cluster_ctarank());
    const int C = p.C;
    const int h = blockIdx.x / C;
    const int B = p.B;
    const int H = p.H;
    const int L = p.ctx_len;
    const int NS = p.nstages;

    const uint32_t bar_full0 = smem_addr(smem + p.off_bars);
    const uint32_t bar_empty0 = bar_full0 + 8u * NS;
    const uint32_t bar_qkv = bar_full0 + 16u * NS;
    const uint32_t bar_sm = bar_qkv + 8u;
    volatile int *flags = reinterpret_cast<volatile int *>(smem + p.off_bars + 16 * NS + 16);
    volatile int *timed_out = flags;      // set by the first wait that gives up
    volatile int *is_last = flags + 1;    // this block merges its column chunk

    const int g = r % p.G;                // column group in the projection
    const int rg = r / p.G;               // row group in the projection
    const int kv_s = static_cast<int>((static_cast<long long>(L) * r) / C);
    const int kv_e = static_cast<int>((static_cast<long long>(L) * (r + 1)) / C);
    const int n_kv_tiles = (kv_e - kv_s + TK - 1) / TK;
    const int col0 = r * p.ncols;
    const int n_out_tiles = p.ncols / kTileCols;
    const int qkv_payload = B * 3 * kTileCols;   // floats one block contributes
    const int sm_payload = B * SMW;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full0 + 8u * s, 1);
            mbar_init(bar_empty0 + 8u * s, kComputeWarps);
        }
        mbar_init(bar_qkv, 1);
        mbar_init(bar_sm, 1);
        *timed_out = 0;
        *is_last = 0;
        fence_mbar_init();
        // Each exchange barrier completes once every peer's bytes have landed.
        mbar_arrive_expect_tx(bar_qkv, static_cast<uint32_t>((C - 1) * qkv_payload * 4));
        mbar_arrive_expect_tx(bar_sm, static_cast<uint32_t>((C - 1) * sm_payload * 4));
    }
    cluster_sync_all();  // barriers initialised everywhere before any push

    if (warp == kComputeWarps) {
        // ------------------------------------------------------------ load warp
        if (lane == 0) {
            const uint32_t ring = smem_addr(smem);
            const uint32_t xring = smem_addr(smem + p.off_xring);
            const int xstage = B * p.TRA * 2;
            uint32_t it = 0;
            auto acquire = [&](uint32_t i) -> int {
                const int s = static_cast<int>(i % NS);
                if (i >= static_cast<uint32_t>(NS))
                    mbar_wait_bounded<false>(bar_empty0 + 8u * s, ((i / NS) - 1) & 1u,
                                             p.timeout_ns, timed_out, p.status, kSiteStageEmpty);
                return s;
            };
            // A: weight tiles [TRA rows x 64 cols] of Q, K, V plus the matching x rows
            for (int sec = 0; sec < 3; ++sec) {
                for (int t = 0; t < p.nA; ++t, ++it) {
                    const int s = acquire(it);
                    const uint32_t full = bar_full0 + 8u * s;
                    const int row = rg * p.R + t * p.TRA;
                    mbar_arrive_expect_tx(full, p.TRA * kTileCols * 2 + xstage);
                    tma_load_2d(ring + s * kStageBytes, &tm_wqkv,
                                sec * H + h * D + g * kTileCols, row, full);
                    for (int b = 0; b < B; ++b)
                        bulk_load_1d(xring + s * xstage + b * p.TRA * 2,
                                     p.x + static_cast<size_t>(b) * H + row, p.TRA * 2, full);
                }
            }
            // B: contiguous runs of cached K and V rows
            for (int b = 0; b < B; ++b) {
                const size_t base = (static_cast<size_t>(b) * p.nh + h) * p.max_ctx * D;
                for (int t = 0; t < n_kv_tiles; ++t, ++it) {
                    const int s = acquire(it);
                    const uint32_t full = bar_full0 + 8u * s;
                    const int t0 = kv_s + t * TK;
                    const int n = min(TK, kv_e - t0);
                    const uint32_t bytes = static_cast<uint32_t>(n * D * 2);
                    mbar_arrive_expect_tx(full, 2 * bytes);
                    bulk_load_1d(ring + s * kStageBytes, p.k_cache + base + static_cast<size_t>(t0) * D,
                                 bytes, full);
                    bulk_load_1d(ring + s * kStageBytes + TK * D * 2,
                                 p.v_cache + base + static_cast<size_t>(t0) * D, bytes, full);
                }
            }
            // C: W_o tiles [D rows x 64 cols] of this block's output columns
            for (int ct = 0; ct < n_out_tiles; ++ct, ++it) {
                const int s = acquire(it);
                const uint32_t full = bar_full0 + 8u * s;
                mbar_arrive_expect_tx(full, D * kTileCols * 2);
                tma_load_2d(ring + s * kStageBytes, &tm_wo, col0 + ct * kTileCols, h * D, full);
            }
            // Drain: the block may not exit with its own copies still in flight.
            const uint32_t issued = it;
            for (int s = 0; s < NS && static_cast<uint32_t>(s) < issued; ++s) {
                const uint32_t last = s + NS * ((issued - 1 - s) / NS);
                volatile int ignore = 0;
                mbar_wait_bounded<false>(bar_full0 + 8u * s, (last / NS) & 1u, p.timeout_ns,
                                         &ignore, p.status, kSiteStageFull);
            }
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- compute warps
        const uint8_t *ring = smem;
        const uint16_t *xring = reinterpret_cast<const uint16_t *>(smem + p.off_xring);
        float *qkv_recv = reinterpret_cast<float *>(smem + p.off_qkv_recv);  // [C][B][3][64]
        float *sm_recv = reinterpret_cast<float *>(smem + p.off_sm_recv);    // [C][B][SMW]
        float *qkv_full = reinterpret_cast<float *>(smem + p.off_qkv_full);  // [B][3][D]
        float *attn = reinterpret_cast<float *>(smem + p.off_attn);          // [B][D]
        float *scratch = reinterpret_cast<float *>(smem + p.off_scratch);
        uint32_t it = 0;
        auto wait_full = [&](uint32_t i) -> int {
            const int s = static_cast<int>(i % NS);
            mbar_wait_bounded<false>(bar_full0 + 8u * s, (i / NS) & 1u, p.timeout_ns, timed_out,
                                     p.status, kSiteStageFull);
            return s;
        };
        auto release = [&](int s) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty0 + 8u * s);
        };

        // ---- A: partial QKV projection ----------------------------------
        float *my_qkv = qkv_recv + static_cast<size_t>(r) * qkv_payload;
        {
            const int xstage = B * p.TRA;
            const int rpw = p.TRA / kComputeWarps;
            for (int sec = 0; sec < 3; ++sec) {
                float acc[MAXB][2];
#pragma unroll
                for (int b = 0; b < MAXB; ++b) acc[b][0] = acc[b][1] = 0.f;
                for (int t = 0; t < p.nA; ++t, ++it) {
                    const int s = wait_full(it);
                    const uint32_t *W = reinterpret_cast<const uint32_t *>(ring + s * kStageBytes);
                    const uint16_t *X = xring + s * xstage;
                    const int r0 = warp * rpw;
#pragma unroll 4
                    for (int i = 0; i < rpw; ++i) {
                        const int row = r0 + i;
                        const uint32_t w2 = W[row * 32 + lane];
                        const float w0 = bf16_lo(w2), w1 = bf16_hi(w2);
#pragma unroll
                        for (int b = 0; b < MAXB; ++b) {
                            if (b < B) {
                                const float xv = bf16_bits(X[b * p.TRA + row]);
                                acc[b][0] = fmaf(xv, w0, acc[b][0]);
                                acc[b][1] = fmaf(xv, w1, acc[b][1]);
                            }
                        }
                    }
                    release(s);
                }
                float2 *scr2 = reinterpret_cast<float2 *>(scratch);
#pragma unroll
                for (int b = 0; b < MAXB; ++b)
                    if (b < B) scr2[(warp * B + b) * 32 + lane] = make_float2(acc[b][0], acc[b][1]);
                compute_bar<kComputeThreads>();
                for (int idx = tid; idx < B * kTileCols; idx += kComputeThreads) {
                    const int b = idx / kTileCols, c = idx % kTileCols;
                    float sum = 0.f;
#pragma unroll
                    for (int w = 0; w < kComputeWarps; ++w) sum += scratch[(w * B + b) * kTileCols + c];
                    my_qkv[(b * 3 + sec) * kTileCols + c] = sum;
                }
                compute_bar<kComputeThreads>();
            }
        }

        // ---- X1: gather q/k/v partials across the cluster ----------------
        {
            const int chunks = qkv_payload / 4;
            const uint32_t my_addr = smem_addr(my_qkv);
            for (int idx = tid; idx < (C - 1) * chunks; idx += kComputeThreads) {
                const int pi = idx / chunks, c = idx % chunks;
                const int peer = pi < r ? pi : pi + 1;
                const float4 v = reinterpret_cast<const float4 *>(my_qkv)[c];
                push_16B(map_to_rank(my_addr + 16u * c, peer), v, map_to_rank(bar_qkv, peer));
            }
            mbar_wait_bounded<true>(bar_qkv, 0, p.timeout_ns, timed_out, p.status,
                                    kSiteQkvExchange);
            for (int idx = tid; idx < B * 3 * D; idx += kComputeThreads) {
                const int b = idx / (3 * D), rem = idx % (3 * D);
                const int sec = rem / D, j = rem % D;
                const int gg = j / kTileCols, c = j % kTileCols;
                float sum = 0.f;
                for (int q = 0; q < p.RG; ++q)
                    sum += qkv_recv[static_cast<size_t>(q * p.G + gg) * qkv_payload +
                                    (b * 3 + sec) * kTileCols + c];
                if (sec == 0) {
                    qkv_full[idx] = sum * p.qscale;
                } else {
                    const __nv_bfloat16 hb = __float2bfloat16_rn(sum);
                    qkv_full[idx] = __bfloat162float(hb);
                    if (r == 0) {
                        uint16_t *cache = sec == 1 ? p.k_cache : p.v_cache;
                        cache[((static_cast<size_t>(b) * p.nh + h) * p.max_ctx + L) * D + j] =
                            __bfloat16_as_ushort(hb);
                    }
                }
            }
            compute_bar<kComputeThreads>();
        }

        // ---- B: split-KV attention with per-lane-group online softmax ----
        float *my_sm = sm_recv + static_cast<size_t>(r) * sm_payload;
        {
            const int sub = lane / LPR, li = lane % LPR;
            float *st_o = scratch;                 // [NSTATE][D]
            float *st_m = scratch + NSTATE * D;    // [NSTATE]
            float *st_l = st_m + NSTATE;           // [NSTATE]
            for (int b = 0; b < B; ++b) {
                const float *qb = qkv_full + static_cast<size_t>(b) * 3 * D;
                float q8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) q8[k] = qb[8 * li + k];
                float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) o[k] = 0.f;
                if (r == C - 1 && warp == 0) {
                    // position L: the new token, from the on-chip bf16-rounded copy
                    float sc = 0.f;
#pragma unroll
                    for (int k = 0; k < 8; ++k) sc = fmaf(q8[k], qb[D + 8 * li + k], sc);
#pragma unroll
                    for (int off = LPR / 2; off > 0; off >>= 1)
                        sc += __shfl_xor_sync(0xffffffffu, sc, off);
                    if (sub == 0) {
                        m = sc;
                        l = 1.f;
#pragma unroll
                        for (int k = 0; k < 8; ++k) o[k] = qb[2 * D + 8 * li + k];
                    }
                }
                for (int t = 0; t < n_kv_tiles; ++t, ++it) {
                    const int s = wait_full(it);
                    const int nrows = min(TK, kv_e - kv_s - t * TK);
                    const uint4 *Kt = reinterpret_cast<const uint4 *>(ring + s * kStageBytes);
                    const uint4 *Vt = reinterpret_cast<const uint4 *>(ring + s * kStageBytes + TK * D * 2);
#pragma unroll
                    for (int j = 0; j < KV_STEPS; ++j) {
                        const int row = warp * (TK / kComputeWarps) + j * RPW + sub;
                        float sc = dot8_bf16(q8, Kt[row * LPR + li]);
#pragma unroll
                        for (int off = LPR / 2; off > 0; off >>= 1)
                            sc += __shfl_xor_sync(0xffffffffu, sc, off);
                        if (row < nrows) {
                            const float mn = fmaxf(m, sc);
                            const float cf = exp2f(m - mn);
                            const float pw = exp2f(sc - mn);
                            float v[8];
                            unpack8_bf16(Vt[row * LPR + li], v);
                            l = fmaf(l, cf, pw);
#pragma unroll
                            for (int k = 0; k < 8; ++k) o[k] = fmaf(pw, v[k], o[k] * cf);
                            m = mn;
                        }
                    }
                    release(s);
                }
                // merge the block's NSTATE states for batch row b
                const int sid = warp * RPW + sub;
#pragma unroll
                for (int k = 0; k < 8; ++k) st_o[sid * D + 8 * li + k] = o[k];
                if (li == 0) {
                    st_m[sid] = m;
                    st_l[sid] = l;
                }
                compute_bar<kComputeThreads>();
                for (int t = tid; t <= D; t += kComputeThreads) {
                    float M = -INFINITY;
                    for (int q = 0; q < NSTATE; ++q) M = fmaxf(M, st_m[q]);
                    float acc = 0.f;
                    for (int q = 0; q < NSTATE; ++q) {
                        const float f = st_m[q] == -INFINITY ? 0.f : exp2f(st_m[q] - M);
                        acc = fmaf(t < D ? st_o[q * D + t] : st_l[q], f, acc);
                    }
                    if (t < D) {
                        my_sm[b * SMW + 4 + t] = acc;
                    } else {
                        my_sm[b * SMW + 0] = M;
                        my_sm[b * SMW + 1] = acc;
                        my_sm[b * SMW + 2] = 0.f;
                        my_sm[b * SMW + 3] = 0.f;
                    }
                }
                compute_bar<kComputeThreads>();
            }
        }

        // ---- X2: ClusterReduce(max) then ClusterReduce(sum) ---------------
        {
            const int chunks = sm_payload / 4;
            const uint32_t my_addr = smem_addr(my_sm);
            for (int idx = tid; idx < (C - 1) * chunks; idx += kComputeThreads) {
                const int pi = idx / chunks, c = idx % chunks;
                const int peer = pi < r ? pi : pi + 1;
                const float4 v = reinterpret_cast<const float4 *>(my_sm)[c];
                push_16B(map_to_rank(my_addr + 16u * c, peer), v, map_to_rank(bar_sm, peer));
            }
            mbar_wait_bounded<true>(bar_sm, 0, p.timeout_ns, timed_out, p.status,
                                    kSiteSoftmaxExchange);
            for (int idx = tid; idx < B * D; idx += kComputeThreads) {
                const int b = idx / D, t = idx % D;
                float M = -INFINITY;
                for (int q = 0; q < C; ++q)
                    M = fmaxf(M, sm_recv[static_cast<size_t>(q) * sm_payload + b * SMW]);
                float num = 0.f, den = 0.f;
                for (int q = 0; q < C; ++q) {
                    const float *rec = sm_recv + static_cast<size_t>(q) * sm_payload + b * SMW;
                    const float f = rec[0] == -INFINITY ? 0.f : exp2f(rec[0] - M);
                    num = fmaf(rec[4 + t], f, num);
                    den = fmaf(rec[1], f, den);
                }
                attn[idx] = num / den;
            }
            compute_bar<kComputeThreads>();
        }

        // ---- C: output projection of this block's column chunk ------------
        {
            constexpr int rpw = D / kComputeWarps;
            float2 *scr2 = reinterpret_cast<float2 *>(scratch);
            for (int ct = 0; ct < n_out_tiles; ++ct, ++it) {
                const int s = wait_full(it);
                const uint32_t *W = reinterpret_cast<const uint32_t *>(ring + s * kStageBytes);
                float acc[MAXB][2];
#pragma unroll
                for (int b = 0; b < MAXB; ++b) acc[b][0] = acc[b][1] = 0.f;
                const int r0 = warp * rpw;
#pragma unroll 4
                for (int i = 0; i < rpw; ++i) {
                    const int row = r0 + i;
                    const uint32_t w2 = W[row * 32 + lane];
                    const float w0 = bf16_lo(w2), w1 = bf16_hi(w2);
#pragma unroll
                    for (int b = 0; b < MAXB; ++b) {
                        if (b < B) {
                            const float av = attn[b * D + row];
                            acc[b][0] = fmaf(av, w0, acc[b][0]);
                            acc[b][1] = fmaf(av, w1, acc[b][1]);
                        }
                    }
                }
                release(s);
#pragma unroll
                for (int b = 0; b < MAXB; ++b)
                    if (b < B) scr2[(warp * B + b) * 32 + lane] = make_float2(acc[b][0], acc[b][1]);
                compute_bar<kComputeThreads>();
                for (int idx = tid; idx < B * kTileCols; idx += kComputeThreads) {
                    const int b = idx / kTileCols, c = idx % kTileCols;
                    float sum = 0.f;
#pragma unroll
                    for (int w = 0; w < kComputeWarps; ++w) sum += scratch[(w * B + b) * kTileCols + c];
                    p.partials[(static_cast<size_t>(h) * B + b) * H + col0 + ct * kTileCols + c] = sum;
                }
                compute_bar<kComputeThreads>();
            }
        }

        // ---- D: deterministic cross-head merge ---------------------------
        __threadfence();
        compute_bar<kComputeThreads>();
        if (tid == 0) {
            const unsigned prev = atomicAdd(p.counters + r, 1u);
            *is_last = (prev == static_cast<unsigned>(p.nh - 1)) ? 1 : 0;
        }
        compute_bar<kComputeThreads>();
        if (*is_last) {
            __threadfence();
            const int n4 = p.ncols / 4;
            for (int idx = tid; idx < B * n4; idx += kComputeThreads) {
                const int b = idx / n4;
                const int c = col0 + 4 * (idx % n4);
                const float *src = p.partials + static_cast<size_t>(b) * H + c;
                const size_t head_stride = static_cast<size_t>(B) * H;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
                for (int hh = 0; hh < p.nh; ++hh) {
                    const float4 v = __ldcg(reinterpret_cast<const float4 *>(src + hh * head_stride));
                    acc.x += v.x;
                    acc.y += v.y;
                    acc.z += v.z;
                    acc.w += v.w;
                }
                uint2 packed;
                packed.x = pack2_bf16(acc.x, acc.y);
                packed.y = pack2_bf16(acc.z, acc.w);
                *reinterpret_cast<uint2 *>(p.out + static_cast<size_t>(b) * H + c) = packed;
            }
            if (tid == 0) p.counters[r] = 0u;  // ready for the next launch
        }
    }
    cluster_sync_all();  // no block leaves while a peer may still touch its shared memory
}

}  // namespace cfa
