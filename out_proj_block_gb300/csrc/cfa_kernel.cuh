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
//     its weight tiles into partial q/k/v sums.
//  X1 Cluster gather/reduce of q, k, v [CF §3.1.2]: every block pushes its
//     partials into every other block's shared memory (st.async with
//     transaction counting on the receiver's mbarrier). The q partials leave
//     as soon as the Q section is done, so the exchange overlaps the K and V
//     sections; the k/v partials leave after the V section and their exchange
//     overlaps attention. Each block sums the row-group partials in rank
//     order and concatenates the column groups, so all blocks hold identical
//     q, k_new, v_new. k_new and v_new are rounded to bf16; rank 0 appends
//     them to the caches.
//  B  Split-KV attention [CF §3.2]: the block owns cached positions
//     [L*r/C, L*(r+1)/C). Each warp keeps an online-softmax state in base-2
//     units with one running max for the whole warp (rescaled once per step,
//     only when the max grows); the states are merged per batch row at the
//     end.
//  X2 ClusterReduce of the softmax statistics [CF §3.1.1, §3.2]: every block
//     pushes (m_r, l_r, o_r) to every other; each block takes the max over
//     them and over the new token's score, then sums the rescaled l_r, o_r
//     and the new token's (1, v_new) in a fixed order, so all blocks hold
//     identical attn = o / l. The new token is thus one more split of the
//     softmax, attended from its on-chip bf16-rounded copy.
//  C  Output projection [CF §3.2]: the block owns H/C output columns and
//     multiplies attn (head h's d rows of W_o) into fp32 partials, written to
//     a per-head workspace row.
//  D  Cross-head merge: instead of the page's atomicAdd merge [CF §3.2], a
//     release/acquire counter per column chunk: the last head to finish the
//     chunk sums every head's partials into bf16 out. Fixed order,
//     deterministic. When that would read more than 256 KB through one block
//     (large batches), head_merge_kernel does the sum after the grid instead.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>

#include "cfa_device.cuh"
#include "cfa_internal.h"
#include "cfa_tile.cuh"

namespace cfa {

// Geometry of the tensor-core projection path (batches of 3..16 rows).
constexpr int kXStageMma = kXStageMmaBytes;      // x bytes per stage: two [16 x 64] swizzled boxes
constexpr uint32_t kAccQK = 0;                   // TMEM columns of the [Q|K] accumulator
constexpr uint32_t kAccV = kMmaN;                // TMEM columns of the V accumulator

// Reduce-scatter exchange of the q/k/v partials (kept out of line: it runs
// a few times per launch, and inlined it costs the kernel registers).
// Slice prg of sections [sec0, sec0 + nsec) of this block's partial
// `mine` [B][3][64] to the peer of row group prg in column group g, into its
// slot rg of the peer's slice buffer [RG][B][3][64 / RG].
static __device__ __noinline__ void rs_push_slices(const float *mine, uint32_t slices_addr,
                                                   uint32_t bar, int sec0, int nsec, int B, int RG,
                                                   int G, int g, int rg, int tid) {
    const int SL = kTileCols / RG;
    const int per_b = nsec * (SL / 4);  // 16-byte chunks per batch row
    const int chunks = B * per_b;
    for (int idx = tid; idx < (RG - 1) * chunks; idx += kComputeThreads) {
        const int pi = idx / chunks, c = idx % chunks;
        const int prg = pi < rg ? pi : pi + 1;
        const int b = c / per_b, w = c % per_b;
        const int sec = sec0 + w / (SL / 4), c4 = 4 * (w % (SL / 4));
        const float4 v = *reinterpret_cast<const float4 *>(mine + (b * 3 + sec) * kTileCols + prg * SL + c4);
        const int doff = ((rg * B + b) * 3 + sec) * SL + c4;
        push_16B(map_to_rank(slices_addr + 4u * doff, prg * G + g), v, map_to_rank(bar, prg * G + g));
    }
}

// Sum this block's slice of sections [sec0, sec0 + nsec) over the row groups
// in row-group order (the order of the gather exchange's sum, so both modes
// give the same bits) and store the raw sums into `full` [B][3][D] on every
// rank of the cluster, this one included; bar_ag counts the peers' bytes.
static __device__ __noinline__ void rs_reduce_gather(const float *mine, const float *slices,
                                                     float *full, uint32_t full_addr, uint32_t bar_ag,
                                                     int sec0, int nsec, int B, int D, int C, int RG,
                                                     int g, int rg, int r, int tid) {
    const int SL = kTileCols / RG;
    const int per_b = nsec * (SL / 4);
    for (int c = tid; c < B * per_b; c += kComputeThreads) {
        const int b = c / per_b, w = c % per_b;
        const int sec = sec0 + w / (SL / 4), c4 = 4 * (w % (SL / 4));
        float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q = 0; q < RG; ++q) {
            const float4 v = *reinterpret_cast<const float4 *>(
                q == rg ? mine + (b * 3 + sec) * kTileCols + rg * SL + c4
                        : slices + ((q * B + b) * 3 + sec) * SL + c4);
            sum.x += v.x;
            sum.y += v.y;
            sum.z += v.z;
            sum.w += v.w;
        }
        const int off = (b * 3 + sec) * D + g * kTileCols + rg * SL + c4;
        *reinterpret_cast<float4 *>(full + off) = sum;
        for (int q = 0; q < C; ++q)
            if (q != r) push_16B(map_to_rank(full_addr + 4u * off, q), sum, map_to_rank(bar_ag, q));
    }
}

template <int D, int MAXB>
__global__ void __launch_bounds__(kThreads, 2)
fused_decode_kernel(const __grid_constant__ CUtensorMap tm_wqkv,
                    const __grid_constant__ CUtensorMap tm_wo,
                    const __grid_constant__ CUtensorMap tm_x,
                    const KernelParams p) {
    static_assert(D == 64 || D == 128, "head_dim must be 64 or 128");
    // B >= 3: the projections are dense [64 x K] . [K x B] contractions and run
    // on the tensor cores (tcgen05, accumulators in TMEM); B <= 2: CUDA cores.
    constexpr bool MMA = MAXB >= 4;
    using GS = GemvShape<MAXB>;
    constexpr int TK = kStageBytes / (4 * D);     // cache rows per K (or V) tile
    constexpr int NV = D / 64;                    // 16-byte vectors per lane per cache row
    constexpr int DPL = 8 * NV;                   // head dims per lane
    constexpr int KV_RPS = 4;                     // cache rows per warp step (8 lanes each)
    constexpr int KV_STEPS = TK / (kComputeWarps * KV_RPS);
    constexpr int SMW = D + 4;                    // floats per softmax record
    static_assert(KV_STEPS * kComputeWarps * KV_RPS == TK, "tile rows must split evenly");

    extern __shared__ __align__(1024) uint8_t smem[];

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int r = static_cast<int>(cluster_ctarank());
    const int C = p.C;
    const int h = blockIdx.x / C;
    const int B = p.B;
    const int H = p.H;
    const int NS = p.nstages;

    const uint32_t bar_full0 = smem_addr(smem + p.off_bars);
    const uint32_t bar_empty0 = bar_full0 + 8u * NS;
    const uint32_t bar_qk = bar_full0 + 16u * NS;   // q and k partials from every peer
    const uint32_t bar_v = bar_qk + 8u;             // v partials from every peer
    const uint32_t bar_sm = bar_qk + 16u;           // softmax statistics from every peer
    const uint32_t bar_acc_a = bar_qk + 24u;        // projection accumulators ready (MMA path)
    const uint32_t bar_acc_c = bar_qk + 32u;        // out-projection accumulator groups (MMA path)
    const uint32_t bar_x = bar_qk + 40u;            // the block's x rows (CUDA-core path)
    const uint32_t bar_qk2 = bar_qk + 72u;          // reduce-scatter mode: every rank's q/k sums
    const uint32_t bar_v2 = bar_qk + 80u;           // reduce-scatter mode: every rank's v sums
    volatile int *flags = reinterpret_cast<volatile int *>(smem + p.off_bars + 16 * NS + 56);
    volatile int *timed_out = flags;      // set by the first wait that gives up
    volatile int *is_last = flags + 1;    // this block merges its column chunk
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + p.off_bars + 16 * NS + 64);

    const int g = r % p.G;                // column group in the projection
    const int rg = r / p.G;               // row group in the projection
    // Cached positions of sequence b before this token. Device-resident
    // lengths are read only after the grid dependency wait (an earlier kernel
    // may have written them); an out-of-range one is flagged in the status
    // word and the sequence is treated as having no cached rows and no row to
    // append (-1).
    auto seq_len = [&](int b) -> int {
        if (!p.lens_dev) return p.ctx_lens[b];
        const int v = p.lens_dev[b];
        if (v >= 0 && v < p.max_ctx) return v;
        if (tid == 0) atomicOr(p.status, kStatusBadLengthBit);
        return -1;
    };
    // Cached positions [kv_s, kv_e) of sequence b owned by this block.
    auto kv_range = [&](int b, int &s0, int &e0) {
        const long long Lb = max(seq_len(b), 0);
        s0 = static_cast<int>((Lb * r) / C);
        e0 = static_cast<int>((Lb * (r + 1)) / C);
    };
    const int col0 = r * p.ncols;
    const int n_out_tiles = p.ncols / kTileCols;
    // W_o in the ring: boxes of KROWS rows x 64 columns, TPS of them (adjacent
    // column tiles) side by side per stage. CUDA-core path: whole [D x 64]
    // tiles (16 KB at D = 128; two 8 KB ones at D = 64). Tensor-core path:
    // [64 x 64] boxes, two column tiles per stage, so the stage is one M = 128
    // operand; at D = 128 a column pair takes two stages (KP K-passes of 64
    // rows) accumulated into one TMEM slot.
    constexpr int KROWS = MMA ? 64 : D;
    constexpr int KP = D / KROWS;
    constexpr int kTileBytes = KROWS * kTileCols * 2;
    constexpr int TPS = kStageBytes / kTileBytes;
    const int n_out_groups = (n_out_tiles + TPS - 1) / TPS;   // column groups of TPS tiles
    const int n_out_units = n_out_groups * KP;                 // ring stages of phase C
    const int qkv_payload = B * 3 * kTileCols;   // floats one block contributes
    const int sm_payload = B * SMW;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar_full0 + 8u * s, 1);
            mbar_init(bar_empty0 + 8u * s, kComputeWarps);
        }
        mbar_init(bar_qk, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_sm, 1);
        mbar_init(bar_acc_a, 1);
        mbar_init(bar_acc_c, 1);
        mbar_init(bar_x, 1);
        mbar_init(bar_qk2, 1);
        mbar_init(bar_v2, 1);
        *timed_out = 0;
        *is_last = 0;
        fence_mbar_init();
        // Each exchange barrier completes once every peer's bytes have landed.
        if (p.rs) {
            // the slices of the peers of this block's column group, then every
            // rank's summed slice (C of them cover the head's D columns)
            const int sl = kTileCols / p.RG;
            mbar_arrive_expect_tx(bar_qk, static_cast<uint32_t>((p.RG - 1) * B * 2 * sl * 4));
            mbar_arrive_expect_tx(bar_v, static_cast<uint32_t>((p.RG - 1) * B * sl * 4));
            mbar_arrive_expect_tx(bar_qk2, static_cast<uint32_t>((C - 1) * B * 2 * sl * 4));
            mbar_arrive_expect_tx(bar_v2, static_cast<uint32_t>((C - 1) * B * sl * 4));
        } else {
            mbar_arrive_expect_tx(bar_qk, static_cast<uint32_t>((C - 1) * B * 2 * kTileCols * 4));
            mbar_arrive_expect_tx(bar_v, static_cast<uint32_t>((C - 1) * B * kTileCols * 4));
        }
        mbar_arrive_expect_tx(bar_sm, static_cast<uint32_t>((C - 1) * sm_payload * 4));
    }
    if constexpr (MMA) {
        if (warp == 0) tmem_alloc(smem_addr(tmem_slot), p.tmem_cols);
        tcgen05_fence_before();
    }
    __syncthreads();
    // The next kernel in the stream may be scheduled now; it waits for this
    // one to finish before touching anything this one writes.
    grid_dependents_launch();
    // Announce this block's barriers to the cluster; the matching wait comes
    // right before the first push, so loading starts without a cluster round trip.
    cluster_arrive();

    // Projection work items: CUDA-core path, 3 sections x nA tiles of [TRA x 64];
    // MMA path, n_qk stages of 64 rows of [Q | K] then n_v stages of 128 rows of V.
    const int n_a = MMA ? p.n_qk + p.n_v : 3 * p.nA;

    if (warp == kComputeWarps) {
        // ------------------------------------------------------------ load warp
        if (lane == 0) {
            const uint32_t ring = smem_addr(smem);
            const uint32_t xring = smem_addr(smem + p.off_xring);
            RingCursor cur;
            auto acquire = [&]() -> int {
                if (cur.wrapped)
                    mbar_wait_bounded<false>(bar_empty0 + 8u * cur.stage, cur.phase ^ 1u,
                                             p.timeout_ns, timed_out, p.status, kSiteStageEmpty);
                return cur.stage;
            };
            // A: weight tiles of this block's Q, K, V columns plus the matching x
            // rows. Weights do not depend on earlier kernels in the stream, so
            // the first ring of weight tiles is requested before waiting for
            // them; x (an earlier kernel's output) only after.
            const int n_pre = min(NS, n_a);
            auto a_bytes = [&](int i) -> uint32_t {
                if constexpr (MMA) return kStageBytes + (i < p.n_qk ? kXStageMma / 2 : kXStageMma);
                else return p.TRA * kTileCols * 2;
            };
            auto issue_w = [&](int i, int s) {
                const uint32_t dst = ring + s * kStageBytes, bar = bar_full0 + 8u * s;
                const int col = h * D + g * kTileCols;
                if constexpr (MMA) {
                    if (i < p.n_qk) {  // rows of Q and K side by side: one M=128 operand
                        const int row = rg * p.R + 64 * i;
                        tma_load_2d(dst, &tm_wqkv, col, row, bar);
                        tma_load_2d(dst + kStageBytes / 2, &tm_wqkv, H + col, row, bar);
                    } else {           // 128 rows of V as two 64-row halves
                        const int row = rg * p.R + 128 * (i - p.n_qk);
                        tma_load_2d(dst, &tm_wqkv, 2 * H + col, row, bar);
                        tma_load_2d(dst + kStageBytes / 2, &tm_wqkv, 2 * H + col, row + 64, bar);
                    }
                } else {
                    const int sec = i / p.nA, t = i % p.nA;
                    tma_load_2d(dst, &tm_wqkv, sec * H + col, rg * p.R + t * p.TRA, bar);
                }
            };
            auto issue_x = [&](int i, int s) {
                const uint32_t bar = bar_full0 + 8u * s;
                if constexpr (MMA) {
                    const uint32_t dst = xring + s * kXStageMma;
                    if (i < p.n_qk) {
                        tma_load_2d(dst, &tm_x, rg * p.R + 64 * i, 0, bar);
                    } else {
                        const int row = rg * p.R + 128 * (i - p.n_qk);
                        tma_load_2d(dst, &tm_x, row, 0, bar);
                        tma_load_2d(dst + kXStageMma / 2, &tm_x, row + 64, 0, bar);
                    }
                }
            };
            // CUDA-core path: the block's x rows [rg*R, rg*R + R) once, for all
            // stages. Without a programmatic dependency x is ready at launch and
            // is requested first (the first stage can then be used as soon as
            // it lands); otherwise only after the dependency wait.
            auto issue_x_rows = [&]() {
                if constexpr (!MMA) {
                    mbar_arrive_expect_tx(bar_x, static_cast<uint32_t>(B * p.R * 2));
                    for (int b = 0; b < B; ++b)
                        bulk_load_1d(xring + b * p.R * 2, p.x + static_cast<size_t>(b) * H + rg * p.R,
                                     p.R * 2, bar_x);
                }
            };
            if (!p.pdl && !p.x_direct) issue_x_rows();
            for (int i = 0; i < n_pre; ++i) {
                mbar_arrive_expect_tx(bar_full0 + 8u * i, a_bytes(i));
                issue_w(i, i);
            }
            grid_dependency_wait();
            if (p.pdl && !p.x_direct) issue_x_rows();
            for (int i = 0; i < n_pre; ++i) issue_x(i, i);
            for (int i = 0; i < n_pre; ++i) cur.advance(NS);
            for (int i = n_pre; i < n_a; ++i) {
                const int s = acquire();
                mbar_arrive_expect_tx(bar_full0 + 8u * s, a_bytes(i));
                issue_w(i, s);
                issue_x(i, s);
                cur.advance(NS);
            }
            // B: contiguous runs of cached K and V rows
            for (int b = 0; b < B; ++b) {
                const size_t base = (static_cast<size_t>(b) * p.nh + h) * p.max_ctx * D;
                int kv_s, kv_e;
                kv_range(b, kv_s, kv_e);
                const int n_kv_tiles = (kv_e - kv_s + TK - 1) / TK;
                for (int t = 0; t < n_kv_tiles; ++t) {
                    const int s = acquire();
                    const uint32_t full = bar_full0 + 8u * s;
                    const int t0 = kv_s + t * TK;
                    const int n = min(TK, kv_e - t0);
                    const uint32_t bytes = static_cast<uint32_t>(n * D * 2);
                    mbar_arrive_expect_tx(full, 2 * bytes);
                    bulk_load_1d(ring + s * kStageBytes, p.k_cache + base + static_cast<size_t>(t0) * D,
                                 bytes, full);
                    bulk_load_1d(ring + s * kStageBytes + TK * D * 2,
                                 p.v_cache + base + static_cast<size_t>(t0) * D, bytes, full);
                    cur.advance(NS);
                }
            }
            // C: W_o tiles [D rows x 64 cols] of this block's output columns,
            // TPS per stage
            for (int u = 0; u < n_out_units; ++u) {
                const int s = acquire();
                const uint32_t full = bar_full0 + 8u * s;
                const int grp = u / KP, kp = u % KP;
                const int nt = min(TPS, n_out_tiles - grp * TPS);
                mbar_arrive_expect_tx(full, static_cast<uint32_t>(nt * kTileBytes));
                for (int k = 0; k < nt; ++k)
                    tma_load_2d(ring + s * kStageBytes + k * kTileBytes, &tm_wo,
                                col0 + (grp * TPS + k) * kTileCols, h * D + kp * KROWS, full);
                cur.advance(NS);
            }
            // Drain: the block may not exit with its own copies still in flight.
            // Stages before the cursor were last filled in the current pass,
            // the others in the previous one (if the ring ever wrapped).
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
        __syncwarp();
        cluster_wait();
    } else {
        // --------------------------------------------------------- compute warps
        const uint8_t *ring = smem;
        float *qkv_recv = reinterpret_cast<float *>(smem + p.off_qkv_recv);  // [C][B][3][64]
        float *sm_recv = reinterpret_cast<float *>(smem + p.off_sm_recv);    // [C][B][SMW]
        float *qkv_full = reinterpret_cast<float *>(smem + p.off_qkv_full);  // [B][3][D], then s_new [B]
        float *attn = reinterpret_cast<float *>(smem + p.off_attn);          // [B][D]
        float *scratch = reinterpret_cast<float *>(smem + p.off_scratch);
        uint32_t tmem = 0;
        if constexpr (MMA) {
            tcgen05_fence_after();
            tmem = *tmem_slot;
        }
        grid_dependency_wait();  // no dependent read or global write before this
        RingCursor cur;
        auto wait_full = [&]() -> int {
            mbar_wait_bounded<false>(bar_full0 + 8u * cur.stage, cur.phase, p.timeout_ns, timed_out,
                                     p.status, kSiteStageFull);
            return cur.stage;
        };
        auto release = [&](int s) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty0 + 8u * s);
            cur.advance(NS);
        };
        // MMA path: warp 0's elected lane issues the MMAs of a stage and hands the
        // stage back with a commit (which counts as warp 0's arrival).
        auto release_after_mma = [&](int s) {
            if (lane == 0) umma_commit(bar_empty0 + 8u * s);
            __syncwarp();
            cur.advance(NS);
        };

        // ---- A: partial QKV projection; partials leave as soon as they exist --
        // Gather mode: every rank's partial [B][3][64] lands in its own slot of
        // qkv_recv on every peer. Reduce-scatter mode: this block's partial
        // sits at the start of qkv_recv and, behind it, the slices
        // [rg' SL, rg' SL + SL) that the RG - 1 peers of its column group
        // computed for the columns this block sums ([RG][B][3][SL]).
        float *my_qkv = p.rs ? qkv_recv : qkv_recv + static_cast<size_t>(r) * qkv_payload;
        const uint32_t my_qkv_addr = smem_addr(my_qkv);
        float *rs_recv = qkv_recv + qkv_payload;
        const uint32_t rs_recv_addr = smem_addr(rs_recv);
        const uint32_t qkv_full_addr = smem_addr(qkv_full);
        // Push sections [sec0, sec0 + nsec) of every batch row: gather mode,
        // the whole partial to every peer; reduce-scatter mode, slice rg' to
        // the peer of row group rg' in this block's column group.
        auto push_sections = [&](int sec0, int nsec, uint32_t bar) {
            if (p.rs) {
                rs_push_slices(my_qkv, rs_recv_addr, bar, sec0, nsec, B, p.RG, p.G, g, rg, tid);
                return;
            }
            const int per_b = nsec * (kTileCols / 4);  // 16-byte chunks per batch row
            const int chunks = B * per_b;
            for (int idx = tid; idx < (C - 1) * chunks; idx += kComputeThreads) {
                const int pi = idx / chunks, c = idx % chunks;
                const int peer = pi < r ? pi : pi + 1;
                const int off = ((c / per_b) * 3 + sec0) * kTileCols + 4 * (c % per_b);
                const float4 v = *reinterpret_cast<const float4 *>(my_qkv + off);
                push_16B(map_to_rank(my_qkv_addr + 4u * off, peer), v, map_to_rank(bar, peer));
            }
        };
        if constexpr (MMA) {
            const uint32_t idesc = umma_idesc_bf16(128, kMmaN, true, false);
            const uint32_t idesc_v = umma_idesc_bf16(128, 2 * kMmaN, true, false);
            const uint32_t ring_a = smem_addr(smem);
            const uint32_t xring_a = smem_addr(smem + p.off_xring);
            // Accumulator rows m (TMEM lanes) are weight columns: [Q | K] rows
            // 0..63 / 64..127; columns are batch rows. The V accumulator holds
            // the stages' first halves in rows 0..63, columns 0..15 and their
            // second halves in rows 64..127, columns 16..31. Read back by the
            // warps that own those lanes.
            auto read_acc = [&](uint32_t col, int nwarps, int sec_of_row64) {
                mbar_wait_bounded<false>(bar_acc_a, col == kAccQK ? 0u : 1u, p.timeout_ns, timed_out,
                                         p.status, kSiteStageFull);
                tcgen05_fence_after();
                if (warp < nwarps) {
                    float v[16];
                    tmem_ld_x16(tmem + (static_cast<uint32_t>(32 * warp) << 16) + col, v);
                    const int m = 32 * warp + lane;
                    const int sec = sec_of_row64 + (m >> 6), c = m & 63;
#pragma unroll
                    for (int b = 0; b < MAXB; ++b)
                        if (b < B) my_qkv[(b * 3 + sec) * kTileCols + c] = v[b];
                }
                tcgen05_fence_before();
                compute_bar<kComputeThreads>();
            };
            for (int i = 0; i < n_a; ++i) {
                const int s = wait_full();
                if (warp == 0) {
                    if (lane == 0) {
                        tcgen05_fence_after();
                        const uint32_t a0 = ring_a + s * kStageBytes;
                        const uint32_t b0 = xring_a + s * kXStageMma;
                        if (i < p.n_qk) {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                umma_bf16(tmem + kAccQK, umma_smem_desc(a0 + j * 2048, kStageBytes / 2, 1024),
                                          umma_smem_desc(b0 + j * 32, 16, 1024), idesc, i > 0 || j > 0);
                        } else {
                            // The stage's two 64-row halves of V side by side: A rows
                            // 64..127 are the second half's rows, B rows 16..31 its
                            // x rows (N = 32); the products of one half with the
                            // other's x land in accumulator quadrants never read.
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                umma_bf16(tmem + kAccV, umma_smem_desc(a0 + j * 2048, kStageBytes / 2, 1024),
                                          umma_smem_desc(b0 + j * 32, 16, 1024), idesc_v, i > p.n_qk || j > 0);
                        }
                        if (i == p.n_qk - 1 || i == n_a - 1) umma_commit(bar_acc_a);
                    }
                    release_after_mma(s);
                } else {
                    release(s);
                }
                if (i == p.n_qk - 1) {
                    read_acc(kAccQK, 4, 0);
                    cluster_wait();  // every peer's barriers are initialised
                    push_sections(0, 2, bar_qk);  // the q/k exchange overlaps the V stages
                }
            }
            {  // v = first halves + second halves (through shared memory)
                mbar_wait_bounded<false>(bar_acc_a, 1u, p.timeout_ns, timed_out, p.status, kSiteStageFull);
                tcgen05_fence_after();
                float *hv = scratch;  // [64 columns][16 batch rows]
                if (warp >= 2 && warp < 4) {
                    float v[16];
                    tmem_ld_x16(tmem + (static_cast<uint32_t>(32 * warp) << 16) + kAccV + kMmaN, v);
                    const int c = 32 * (warp - 2) + lane;
#pragma unroll
                    for (int b = 0; b < MAXB; ++b) hv[c * kMmaN + b] = v[b];
                }
                compute_bar<kComputeThreads>();
                if (warp < 2) {
                    float v[16];
                    tmem_ld_x16(tmem + (static_cast<uint32_t>(32 * warp) << 16) + kAccV, v);
                    const int c = 32 * warp + lane;
#pragma unroll
                    for (int b = 0; b < MAXB; ++b)
                        if (b < B) my_qkv[(b * 3 + 2) * kTileCols + c] = v[b] + hv[c * kMmaN + b];
                }
                tcgen05_fence_before();
                compute_bar<kComputeThreads>();
            }
            push_sections(2, 1, bar_v);  // the v exchange overlaps attention
        } else {
            const uint16_t *xrows = reinterpret_cast<const uint16_t *>(smem + p.off_xring);  // [B][R]
            const int rpw = p.TRA / kComputeWarps;
            if (p.x_direct) {
                // x in host-mapped memory: 16-byte plain loads of this block's
                // rows (not TMA), shared by every compute warp after a barrier
                const int n16 = p.R / 8;
                for (int idx = tid; idx < B * n16; idx += kComputeThreads) {
                    const int b = idx / n16, c = idx % n16;
                    const uint4 v = *reinterpret_cast<const uint4 *>(p.x + static_cast<size_t>(b) * H +
                                                                     rg * p.R + 8 * c);
                    *reinterpret_cast<uint4 *>(smem + p.off_xring + (static_cast<size_t>(b) * p.R + 8 * c) * 2) = v;
                }
                compute_bar<kComputeThreads>();
            } else {
                mbar_wait_bounded<false>(bar_x, 0, p.timeout_ns, timed_out, p.status, kSiteStageFull);
            }
            for (int sec = 0; sec < 3; ++sec) {
                float acc[MAXB][GS::CPL];
#pragma unroll
                for (int b = 0; b < MAXB; ++b)
#pragma unroll
                    for (int c = 0; c < GS::CPL; ++c) acc[b][c] = 0.f;
                for (int t = 0; t < p.nA; ++t) {
                    const int s = wait_full();
                    gemv_tile<MAXB>(ring + s * kStageBytes, rpw, xrows + t * p.TRA, p.R, B,
                                    warp, lane, acc);
                    release(s);
                }
                gemv_reduce<MAXB>(acc, B, warp, lane, tid, scratch, my_qkv + sec * kTileCols,
                                  3 * kTileCols);
                if (sec == 1) {
                    cluster_wait();  // every peer's barriers are initialised
                    push_sections(0, 2, bar_qk);  // the q/k exchange overlaps the V section
                }
            }
            push_sections(2, 1, bar_v);  // the v exchange overlaps attention
        }

        // Sum the row-group partials of section sec in rank order (column groups
        // concatenated) for batch row b and head dim j.
        auto gathered = [&](int b, int sec, int j) {
            const int gg = j / kTileCols, c = j % kTileCols;
            float sum = 0.f;
            for (int q = 0; q < p.RG; ++q)
                sum += qkv_recv[static_cast<size_t>(q * p.G + gg) * qkv_payload +
                                (b * 3 + sec) * kTileCols + c];
            return sum;
        };
        // bf16 k_new / v_new, kept on chip and appended to the cache by rank 0.
        auto append = [&](int b, int sec, int j, float val) {
            const __nv_bfloat16 hb = __float2bfloat16_rn(val);
            qkv_full[(b * 3 + sec) * D + j] = __bfloat162float(hb);
            const int Lb = seq_len(b);
            if (r == 0 && Lb >= 0) {
                uint16_t *cache = sec == 1 ? p.k_cache : p.v_cache;
                cache[((static_cast<size_t>(b) * p.nh + h) * p.max_ctx + Lb) * D + j] =
                    __bfloat16_as_ushort(hb);
            }
        };

        // Reduce-scatter mode: this block's slice summed into qkv_full on every rank.
        auto reduce_gather = [&](int sec0, int nsec, uint32_t bar_ag) {
            rs_reduce_gather(my_qkv, rs_recv, qkv_full, qkv_full_addr, bar_ag, sec0, nsec, B, D, C,
                             p.RG, g, rg, r, tid);
            compute_bar<kComputeThreads>();
        };

        // ---- X1 (q, k): the query for attention and the new key -------------
        // With rotary embedding, dims i and i + D/2 of q and k_new are rotated
        // by ctx_lens[b] * theta^(-2i/D) (rotate-half form); the angle is taken
        // in fp64 and reduced to (-pi, pi] before the fp32 sine and cosine.
        // The raw sums go to qkv_full first (reduce-scatter mode: by the
        // exchange itself) and are transformed in place (each element read and
        // written by the same thread).
        mbar_wait_bounded<true>(bar_qk, 0, p.timeout_ns, timed_out, p.status, kSiteQExchange);
        if (p.rs) {
            reduce_gather(0, 2, bar_qk2);
            mbar_wait_bounded<true>(bar_qk2, 0, p.timeout_ns, timed_out, p.status, kSiteQExchange);
        } else {
            // gather mode: the rank-order sums into qkv_full as well
            for (int idx = tid; idx < B * 2 * D; idx += kComputeThreads) {
                const int b = idx / (2 * D), rem = idx % (2 * D);
                qkv_full[b * 3 * D + rem] = gathered(b, rem / D, rem % D);
            }
            compute_bar<kComputeThreads>();
        }
        for (int idx = tid; idx < B * D; idx += kComputeThreads) {
            const int b = idx / D, rem = idx % D;
            const int sec = rem / (D / 2), i = rem % (D / 2);
            float y0 = qkv_full[(b * 3 + sec) * D + i];
            float y1 = qkv_full[(b * 3 + sec) * D + i + D / 2];
            if (p.rope) {
                const double ang = static_cast<double>(max(seq_len(b), 0)) * p.rope_inv_freq[i];
                const double red = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);
                float sn, cs;
                sincosf(static_cast<float>(red), &sn, &cs);
                const float x0 = y0, x1 = y1;
                y0 = x0 * cs - x1 * sn;
                y1 = x1 * cs + x0 * sn;
            }
            if (sec == 0) {
                qkv_full[b * 3 * D + i] = y0 * p.qscale;
                qkv_full[b * 3 * D + i + D / 2] = y1 * p.qscale;
            } else {
                append(b, 1, i, y0);
                append(b, 1, i + D / 2, y1);
            }
        }
        compute_bar<kComputeThreads>();

        // ---- B: split-KV attention over cached rows, one state per warp -----
        float *my_sm = sm_recv + static_cast<size_t>(r) * sm_payload;
        {
            // lane = 8 * rq + li: cache row rq of each 4-row step; 16-byte
            // vectors li and li + 8 of that row, i.e. dims [8li, 8li+8) and
            // [64 + 8li, 64 + 8li + 8) (the second only when D = 128).
            const int rq = lane >> 3, li = lane & 7;
            float *st_o = scratch;                          // [8][D]
            float *st_m = scratch + kComputeWarps * D;      // [8]
            float *st_l = st_m + kComputeWarps;             // [8]
            for (int b = 0; b < B; ++b) {
                const float *qb = qkv_full + static_cast<size_t>(b) * 3 * D;
                int kv_s, kv_e;
                kv_range(b, kv_s, kv_e);
                const int n_kv_tiles = (kv_e - kv_s + TK - 1) / TK;
                float q[DPL], o[DPL];
#pragma unroll
                for (int v = 0; v < NV; ++v)
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        q[8 * v + k] = qb[64 * v + 8 * li + k];
                        o[8 * v + k] = 0.f;
                    }
                float m = -INFINITY, l = 0.f;   // m is the same in every lane of the warp
                for (int t = 0; t < n_kv_tiles; ++t) {
                    const int s = wait_full();
                    const int nrows = min(TK, kv_e - kv_s - t * TK);
                    const uint4 *Kt = reinterpret_cast<const uint4 *>(ring + s * kStageBytes);
                    const uint4 *Vt = reinterpret_cast<const uint4 *>(ring + s * kStageBytes + TK * D * 2);
                    // Scores of all the warp's rows in this tile first (the steps
                    // are independent), then one running-max update for them all.
                    float sc[KV_STEPS];
                    float tmax = -INFINITY;
#pragma unroll
                    for (int j = 0; j < KV_STEPS; ++j) {
                        const int row = (warp * KV_STEPS + j) * KV_RPS + rq;
                        uint4 kr[NV];
#pragma unroll
                        for (int v = 0; v < NV; ++v) kr[v] = Kt[row * (D / 8) + 8 * v + li];
                        float s0 = 0.f, s1 = 0.f;
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            float kf[8];
                            unpack8_bf16(kr[v], kf);
#pragma unroll
                            for (int k = 0; k < 8; k += 2) {
                                s0 = fmaf(q[8 * v + k], kf[k], s0);
                                s1 = fmaf(q[8 * v + k + 1], kf[k + 1], s1);
                            }
                        }
                        float x = s0 + s1;
                        x += __shfl_xor_sync(0xffffffffu, x, 1);
                        x += __shfl_xor_sync(0xffffffffu, x, 2);
                        x += __shfl_xor_sync(0xffffffffu, x, 4);
                        sc[j] = row < nrows ? x : -INFINITY;
                        tmax = fmaxf(tmax, sc[j]);
                    }
                    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 8));
                    tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
                    if (tmax > m) {  // warp-uniform: rescale only when the max grows
                        const float cf = exp2f(m - tmax);
                        l *= cf;
#pragma unroll
                        for (int k = 0; k < DPL; ++k) o[k] *= cf;
                        m = tmax;
                    }
#pragma unroll
                    for (int j = 0; j < KV_STEPS; ++j) {
                        const int row = (warp * KV_STEPS + j) * KV_RPS + rq;
                        if (row < nrows) {
                            const float pw = exp2f(sc[j] - m);
                            l += pw;
#pragma unroll
                            for (int v = 0; v < NV; ++v) {
                                float vf[8];
                                unpack8_bf16(Vt[row * (D / 8) + 8 * v + li], vf);
#pragma unroll
                                for (int k = 0; k < 8; ++k) o[8 * v + k] = fmaf(pw, vf[k], o[8 * v + k]);
                            }
                        }
                    }
                    release(s);
                }
                // the warp's four row groups share m: add their l and o
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
#pragma unroll
                for (int k = 0; k < DPL; ++k) {
                    o[k] += __shfl_xor_sync(0xffffffffu, o[k], 8);
                    o[k] += __shfl_xor_sync(0xffffffffu, o[k], 16);
                }
                if (rq == 0) {
#pragma unroll
                    for (int v = 0; v < NV; ++v)
#pragma unroll
                        for (int k = 0; k < 8; ++k) st_o[warp * D + 64 * v + 8 * li + k] = o[8 * v + k];
                    if (li == 0) {
                        st_m[warp] = m;
                        st_l[warp] = l;
                    }
                }
                compute_bar<kComputeThreads>();
                // merge the 8 warp states of batch row b (fixed order)
                for (int t = tid; t <= D; t += kComputeThreads) {
                    float M = -INFINITY;
#pragma unroll
                    for (int w = 0; w < kComputeWarps; ++w) M = fmaxf(M, st_m[w]);
                    float acc = 0.f;
#pragma unroll
                    for (int w = 0; w < kComputeWarps; ++w) {
                        const float f = st_m[w] == -INFINITY ? 0.f : exp2f(st_m[w] - M);
                        acc = fmaf(t < D ? st_o[w * D + t] : st_l[w], f, acc);
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

        // ---- X2 push: this block's softmax statistics to every peer ---------
        {
            const int chunks = sm_payload / 4;
            const uint32_t my_addr = smem_addr(my_sm);
            for (int idx = tid; idx < (C - 1) * chunks; idx += kComputeThreads) {
                const int pi = idx / chunks, c = idx % chunks;
                const int peer = pi < r ? pi : pi + 1;
                const float4 v = reinterpret_cast<const float4 *>(my_sm)[c];
                push_16B(map_to_rank(my_addr + 16u * c, peer), v, map_to_rank(bar_sm, peer));
            }
        }

        // ---- X1 (v) while X2 is in flight: v_new, its cache append and the new
        //      token's score; the new token is one more split of the softmax,
        //      attended from its on-chip bf16-rounded copy.
        mbar_wait_bounded<true>(bar_v, 0, p.timeout_ns, timed_out, p.status, kSiteKvExchange);
        if (p.rs) {
            reduce_gather(2, 1, bar_v2);
            mbar_wait_bounded<true>(bar_v2, 0, p.timeout_ns, timed_out, p.status, kSiteKvExchange);
            for (int idx = tid; idx < B * D; idx += kComputeThreads)
                append(idx / D, 2, idx % D, qkv_full[(idx / D * 3 + 2) * D + idx % D]);
        } else {
            for (int idx = tid; idx < B * D; idx += kComputeThreads)
                append(idx / D, 2, idx % D, gathered(idx / D, 2, idx % D));
        }
        float *s_new = qkv_full + static_cast<size_t>(B) * 3 * D;  // [B]
        for (int b = warp; b < B; b += kComputeWarps) {
            const float *qb = qkv_full + static_cast<size_t>(b) * 3 * D;
            float sc = 0.f;
            for (int j = lane; j < D; j += 32) sc = fmaf(qb[j], qb[D + j], sc);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) sc += __shfl_xor_sync(0xffffffffu, sc, off);
            if (lane == 0) s_new[b] = sc;
        }
        compute_bar<kComputeThreads>();

        // ---- X2 combine: ClusterReduce(max) then ClusterReduce(sum) --------
        mbar_wait_bounded<true>(bar_sm, 0, p.timeout_ns, timed_out, p.status, kSiteSoftmaxExchange);
        for (int idx = tid; idx < B * D; idx += kComputeThreads) {
            const int b = idx / D, t = idx % D;
            float M = s_new[b];
            for (int q = 0; q < C; ++q)
                M = fmaxf(M, sm_recv[static_cast<size_t>(q) * sm_payload + b * SMW]);
            const float fn = exp2f(s_new[b] - M);
            float num = qkv_full[(b * 3 + 2) * D + t] * fn, den = fn;
            for (int q = 0; q < C; ++q) {
                const float *rec = sm_recv + static_cast<size_t>(q) * sm_payload + b * SMW;
                const float f = rec[0] == -INFINITY ? 0.f : exp2f(rec[0] - M);
                num = fmaf(rec[4 + t], f, num);
                den = fmaf(rec[1], f, den);
            }
            attn[idx] = num / den;
        }
        compute_bar<kComputeThreads>();

        // ---- C: output projection of this block's column chunk --------------
        const size_t head_stride = static_cast<size_t>(B) * H;
        if constexpr (MMA) {
            // attn^T as a K-major, 128-byte-swizzled bf16 operand of 32 rows per
            // 64-column atom: rows 0-15 the hi parts of the batch rows, 16-31
            // the lo parts, so one MMA (N = 32) carries ~16 mantissa bits of attn;
            // the two halves of each accumulator are added when read out.
            uint8_t *at = smem + p.off_attn_t;
            for (int idx = tid; idx < kMmaN * D; idx += kComputeThreads) {
                const int n = idx / D, k = idx % D;
                const float a = n < B ? attn[n * D + k] : 0.f;
                const __nv_bfloat16 hi = __float2bfloat16_rn(a);
                const __nv_bfloat16 lo = __float2bfloat16_rn(a - __bfloat162float(hi));
                const int kk = k & 63;
                uint8_t *atom = at + (k >> 6) * (2 * kMmaN * 128);
                const int in_row = (kk & 7) * 2;
                *reinterpret_cast<__nv_bfloat16 *>(atom + n * 128 + (((kk >> 3) ^ (n & 7)) << 4) + in_row) = hi;
                const int nl = kMmaN + n;
                *reinterpret_cast<__nv_bfloat16 *>(atom + nl * 128 + (((kk >> 3) ^ (nl & 7)) << 4) + in_row) = lo;
            }
            fence_proxy_async_smem();
            compute_bar<kComputeThreads>();
            const uint32_t idesc = umma_idesc_bf16(128, 2 * kMmaN, true, false);
            const uint32_t ring_a = smem_addr(smem);
            const uint32_t at_a = smem_addr(at);
            // One TMEM accumulator of 2 x 16 columns per column group of two
            // tiles (up to kbuf of them): the MMAs of consecutive stages are
            // issued back to back and read out in groups. A stage's A operand is
            // M = 128 weight columns, its two tiles side by side (a lone last
            // tile: its half repeated), K = 64 rows.
            const int kbuf = static_cast<int>(p.tmem_cols) / (2 * kMmaN);
            int group0 = 0, group_n = 0;
            uint32_t acc_phase = 0;
            auto flush = [&]() {
                if (warp == 0 && lane == 0) umma_commit(bar_acc_c);
                mbar_wait_bounded<false>(bar_acc_c, acc_phase, p.timeout_ns, timed_out, p.status,
                                         kSiteStageFull);
                acc_phase ^= 1u;
                tcgen05_fence_after();
                // Accumulator lanes 64k .. 64k+63 are the columns of the stage's
                // tile k: the warps of lane quarters 0-3 read them for even
                // stages, warps 4-7 (the same quarters) for odd ones; hi and lo
                // share one load wait.
                {
                    const int wq = warp & 3;
                    for (int u = group0 + (warp >> 2); u < group0 + group_n; u += 2) {
                        const int t = u * TPS + (wq >> 1);
                        if (t >= n_out_tiles) continue;  // a lone last tile: quarters 2, 3 unused
                        uint32_t vh[16], vl[16];
                        const uint32_t ta = tmem + (static_cast<uint32_t>(32 * wq) << 16) +
                                            static_cast<uint32_t>(2 * kMmaN * (u % kbuf));
                        tmem_ld_x16_nowait(ta, vh);
                        tmem_ld_x16_nowait(ta + kMmaN, vl);
                        tmem_wait_ld();
                        float *dst = p.partials + static_cast<size_t>(h) * head_stride + col0 +
                                     t * kTileCols + 32 * (wq & 1) + lane;
#pragma unroll
                        for (int b = 0; b < MAXB; ++b)
                            if (b < B) dst[static_cast<size_t>(b) * H] = __uint_as_float(vh[b]) + __uint_as_float(vl[b]);
                    }
                }
                tcgen05_fence_before();
                compute_bar<kComputeThreads>();  // the group's accumulators are free again
                group0 += group_n;
                group_n = 0;
            };
            static_assert(!MMA || TPS == 2, "tensor-core out-projection stages hold two tiles");
            for (int u = 0; u < n_out_units; ++u) {
                const int s = wait_full();
                const int grp = u / KP, kp = u % KP;
                if (warp == 0) {
                    if (lane == 0) {
                        tcgen05_fence_after();
                        const uint32_t a0 = ring_a + s * kStageBytes;
                        const uint32_t d = tmem + static_cast<uint32_t>(2 * kMmaN * (grp % kbuf));
                        const uint32_t half = grp * TPS + 1 < n_out_tiles ? static_cast<uint32_t>(kTileBytes) : 0u;
#pragma unroll
                        for (int j = 0; j < KROWS / 16; ++j) {
                            const uint64_t da = umma_smem_desc(a0 + j * 2048, half, 1024);
                            const int k0 = kp * KROWS + 16 * j;  // attn row of this K slice
                            const uint32_t boff = (k0 >> 6) * (2 * kMmaN * 128) + ((k0 & 63) >> 4) * 32;
                            umma_bf16(d, da, umma_smem_desc(at_a + boff, 16, 1024), idesc, kp > 0 || j > 0);
                        }
                    }
                    release_after_mma(s);
                } else {
                    release(s);
                }
                if (kp == KP - 1 && ++group_n == kbuf) flush();
            }
            if (group_n > 0) flush();
        } else {
            // A warp takes whole tiles (tile ct goes to warp ct % 8): all D rows
            // of its 64 columns, summed within the warp, so no block barrier
            // separates tiles. Every warp waits for each stage and releases it
            // (the ring's phases stay in order); only the owners of its tiles
            // read it.
            const int cg = lane % GS::LPR, rq = lane / GS::LPR;
            static_assert(MMA || KP == 1, "CUDA-core out-projection stages hold whole tiles");
            for (int u = 0; u < n_out_units; ++u) {
                const int s = wait_full();
                int k = 0;  // this warp's tile in the stage, if any (TPS <= 8 warps)
                while (k < TPS && (u * TPS + k >= n_out_tiles || (u * TPS + k) % kComputeWarps != warp)) ++k;
                if (k == TPS) {
                    release(s);
                    continue;
                }
                const int ct = u * TPS + k;
                float acc[MAXB][GS::CPL];
#pragma unroll
                for (int b = 0; b < MAXB; ++b)
#pragma unroll
                    for (int c = 0; c < GS::CPL; ++c) acc[b][c] = 0.f;
                gemv_tile<MAXB>(ring + s * kStageBytes + k * kTileBytes, D, attn, D, B, 0, lane, acc);
                release(s);
                // the warp's row groups, in a fixed shuffle order
#pragma unroll
                for (int b = 0; b < MAXB; ++b)
#pragma unroll
                    for (int c = 0; c < GS::CPL; ++c)
#pragma unroll
                        for (int off = GS::LPR; off < 32; off <<= 1)
                            acc[b][c] += __shfl_xor_sync(0xffffffffu, acc[b][c], off);
                if (rq == 0) {
                    float *dst = p.partials + static_cast<size_t>(h) * head_stride + col0 + ct * kTileCols +
                                 cg * GS::CPL;
#pragma unroll
                    for (int b = 0; b < MAXB; ++b)
                        if (b < B) {
#pragma unroll
                            for (int c = 0; c < GS::CPL; c += 4)
                                *reinterpret_cast<float4 *>(dst + static_cast<size_t>(b) * H + c) =
                                    make_float4(acc[b][c], acc[b][c + 1], acc[b][c + 2], acc[b][c + 3]);
                        }
                }
            }
            compute_bar<kComputeThreads>();  // every tile's partials are stored
        }

        // ---- D: deterministic cross-head merge ----------------------------------
        // The last head to finish this column chunk sums every head's partials
        // (in head order) into bf16 out. A barrier follows each block's last
        // store, so one thread's release covers the whole block's stores.
        // Plans whose merge would read more than 256 KB through one block
        // leave it to head_merge_kernel, launched after this grid.
        if (!p.merge_separate) {
            const int n4 = p.ncols / 4;
            unsigned *ctr = p.counters + r;
            if (tid == 0) {
                const unsigned prev = atomic_add_acq_rel_gpu(ctr, 1u);
                const bool last = prev == static_cast<unsigned>(p.nh - 1);
                if (last) *ctr = 0u;  // ready for the next launch
                *is_last = last ? 1 : 0;
            }
            compute_bar<kComputeThreads>();
            if (*is_last) {
                // Two threads per item (b, 4 columns): each sums half of the
                // heads in ascending order, 8 loads in flight at a time, then
                // half 0 + half 1.
                const int half = tid & 1, hh = (p.nh + 1) / 2;
                const int e0 = half * hh, e1 = min(p.nh, e0 + hh);
                for (int base = 0; base < B * n4; base += kComputeThreads / 2) {
                    const int idx = base + (tid >> 1);
                    const bool valid = idx < B * n4;
                    const int b = valid ? idx / n4 : 0;
                    const int c = col0 + 4 * (valid ? idx % n4 : 0);
                    const float *src = p.partials + static_cast<size_t>(b) * H + c;
                    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int i0 = e0; i0 < e1; i0 += 8) {
                        float4 v[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            v[i] = valid && i0 + i < e1
                                       ? __ldcg(reinterpret_cast<const float4 *>(src + (i0 + i) * head_stride))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            sum.x += v[i].x;
                            sum.y += v[i].y;
                            sum.z += v[i].z;
                            sum.w += v[i].w;
                        }
                    }
                    float4 other;
                    other.x = __shfl_xor_sync(0xffffffffu, sum.x, 1);
                    other.y = __shfl_xor_sync(0xffffffffu, sum.y, 1);
                    other.z = __shfl_xor_sync(0xffffffffu, sum.z, 1);
                    other.w = __shfl_xor_sync(0xffffffffu, sum.w, 1);
                    if (!valid || half) continue;
                    sum = make_float4(sum.x + other.x, sum.y + other.y, sum.z + other.z, sum.w + other.w);
                    if (p.resid) {  // residual stream: out = resid + attention block
                        const uint2 rv = *reinterpret_cast<const uint2 *>(p.resid + static_cast<size_t>(b) * H + c);
                        sum.x += bf16_lo(rv.x);
                        sum.y += bf16_hi(rv.x);
                        sum.z += bf16_lo(rv.y);
                        sum.w += bf16_hi(rv.y);
                    }
                    uint2 packed;
                    packed.x = pack2_bf16(sum.x, sum.y);
                    packed.y = pack2_bf16(sum.z, sum.w);
                    *reinterpret_cast<uint2 *>(p.out + static_cast<size_t>(b) * H + c) = packed;
                }
            }
        }
        if constexpr (MMA) {
            if (warp == 0) {
                tcgen05_fence_after();
                tmem_dealloc(tmem, p.tmem_cols);
            }
        }
    }
    cluster_sync_all();  // no block leaves while a peer may still touch its shared memory
}

}  // namespace cfa
