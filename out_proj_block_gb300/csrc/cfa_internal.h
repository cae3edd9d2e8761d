// cfa_internal.h -- launch parameters shared by the host side and the fused
// kernel. Not part of the public ABI (that is include/cfa.h).
#pragma once

#include <cstdint>

#include <cuda.h>

namespace cfa {

constexpr int kComputeWarps = 8;                   // warps doing arithmetic
constexpr int kComputeThreads = kComputeWarps * 32;
constexpr int kThreads = kComputeThreads + 32;     // + one load-issuing warp
constexpr int kStageBytes = 16384;                 // one pipeline stage
constexpr int kTileCols = 64;                      // weight tile width (128 bytes of bf16)
constexpr int kGemvTileCols = 128;                 // stream-K GEMV tile width (256 bytes)
constexpr int kGemvThreads = kComputeThreads + 64; // GEMV block: + load warp + epilogue warp
constexpr int kMaxCluster = 16;
constexpr int kMaxBatch = 16;
constexpr int kMaxRopePairs = 64;                  // head_dim / 2
constexpr int kMaxCounters = 4096;                 // merge counters; the status word follows
constexpr int kMmaN = 16;                          // batch rows per tensor-core MMA (zero-padded)
constexpr int kXStageMmaBytes = 2 * kMmaN * 128;   // x per stage on the tensor-core path

// Status word bits, written by kernels and read by cfa_plan_status.
constexpr unsigned kStatusTimeoutBit = 1u;
constexpr unsigned kStatusBadLengthBit = 2u;  // a device-resident length was out of range
constexpr unsigned kStatusSiteShift = 8;  // site code of the first timeout

// Site codes recorded with a timeout in the status word.
enum WaitSite : unsigned {
    kSiteStageFull = 1,
    kSiteStageEmpty = 2,
    kSiteQExchange = 3,
    kSiteSoftmaxExchange = 4,
    kSiteKvExchange = 5,
    kSiteSelftest = 15,
};

struct KernelParams {
    const uint16_t *x;     // [B][H] bf16
    uint16_t *k_cache;     // [B][nh][max_ctx][D] bf16
    uint16_t *v_cache;
    uint16_t *out;         // [B][H] bf16
    const uint16_t *resid; // [B][H] bf16 added to out before rounding, or null
    const int *lens_dev;   // [B] device-resident ctx_lens (read after the grid dependency
                           // wait), or null to use ctx_lens below
    float *partials;       // [nh][B][H] fp32 per-head output-projection partials
    float *group_sums;     // [ceil(nh / merge_group)][B][H] fp32 per-group sums
    unsigned *counters;    // [groups][C] then [C]: arrivals per column chunk, two levels
    unsigned *status;      // device status word
    int B, H, nh, max_ctx;
    int ctx_lens[kMaxBatch];   // cached positions of each sequence before this token
    int rope;                  // 1: rotate the new q and k (rotate-half form)
    double rope_inv_freq[kMaxRopePairs];  // theta^(-2i/D), i < D/2
    int C;                 // blocks per cluster (= per head)
    int G;                 // column groups of 64 inside one head's Q/K/V block: D/64 or fewer
    int RG;                // row groups of the hidden dimension: C / G
    int R;                 // hidden rows per block in the projection: H / RG
    int TRA;               // rows per projection tile
    int nA;                // projection tiles per Q/K/V block: R / TRA (CUDA-core path)
    int n_qk, n_v;         // tensor-core path: 64-row [Q|K] stages and 128-row V stages
    unsigned tmem_cols;    // tensor-core path: TMEM columns per block (power of two >= 32)
    int ncols;             // output columns per block in the out-projection: H / C
    int merge_group;       // heads per first-level merge group
    int nstages;           // pipeline depth
    int off_xring, off_qkv_recv, off_sm_recv, off_qkv_full, off_attn, off_attn_t, off_scratch,
        off_bars;
    unsigned long long timeout_ns;
    float qscale;          // log2(e) / sqrt(D)
};

// ------------------------------------------------------------ stream-K GEMV
// y[b, n] = epilogue( sum_k in[b, k] W[k, n] ) over 128-column tiles, with the
// (tile, row-chunk) units of work split evenly over a persistent grid.

enum GemvMode : int {
    kGemvSwiGLU = 0,    // two matrices (gate, up), RMSNorm of the input, silu(gate) * up
    kGemvResidual = 1,  // one matrix, residual added
    kGemvPlain = 2,     // one matrix, result stored as is
    kGemvNormPlain = 3, // one matrix, RMSNorm of the input, result stored as is
};

struct GemvParams {
    const uint16_t *x;       // [B][x_stride] bf16 input rows (the first K of each are used)
    const uint16_t *norm_w;  // [K] bf16 RMSNorm weight (SwiGLU mode)
    const uint16_t *resid;   // [B][N] bf16 residual (residual mode)
    uint16_t *y;             // [B][N] bf16 output
    float *partials;         // [nblocks][max_tiles][B][nmat * 128] fp32 tile partials
    unsigned *counters;      // [n_tiles] arrivals per tile
    unsigned *status;        // device status word
    int B, K, N;
    int x_stride;            // elements between input rows (>= K)
    int rows;                // weight rows per unit (and per stage): 32 (two matrices) or 64
    int chunks;              // units per tile: K / rows
    int n_tiles;             // ceil(N / 128); a last tile of 64 columns is masked
    int units;               // n_tiles * chunks
    int nblocks;             // grid size
    int max_tiles;           // tiles one block can touch
    int nstages;
    int xstage_bytes;        // bytes of one x (+ norm weight) stage
    int off_xring, off_xn, off_scratch, off_tile, off_misc, off_bars;
    float eps;
    unsigned long long timeout_ns;
};

// ---------------------------------------------------- multi-head latent attention

constexpr int kMlaKv = 512, kMlaNope = 128, kMlaRope = 64, kMlaV = 128;
constexpr int kMlaRow = kMlaKv + kMlaRope;          // 576 latent-row elements
constexpr int kMlaQk = kMlaNope + kMlaRope;         // 192 query / key width
constexpr int kMlaTileRows = 128;                   // latent rows per tile (MMA M)
constexpr int kMlaBoxes = kMlaRow / 64;             // 9 swizzled [128 x 64] boxes per tile
constexpr int kMlaBoxBytes = kMlaTileRows * 128;    // 16 KB
constexpr int kMlaStageBytes = 2 * kMlaBoxBytes;    // a stage holds two boxes
constexpr int kMlaMaxHG = 16;                       // heads per cluster = MMA N
constexpr int kMlaAtomBytes = kMlaMaxHG * 128;      // a [16 x 64] K-major swizzled atom
constexpr int kMlaWeightRows = 256;                 // a W_kvb box is [256 x 64] (one stage)
constexpr int kMlaQAtomBytes = 2 * kMlaAtomBytes;   // a [32 x 64] atom: hi rows, then lo rows
constexpr int kMlaThreads = kComputeThreads + 64;   // + load warp + MMA warp

struct MlaParams {
    const uint16_t *q;       // [B][nh*192] bf16: per head [q_nope | q_rope]
    const uint16_t *a;       // [B][a_stride] bf16: latent at a_off, rope key at a_off + 512
    const uint16_t *g_kv;    // [512] bf16 RMSNorm weight of the latent
    const uint16_t *W_kvb;   // [512][nh*256] bf16
    uint16_t *cache;         // [B][max_ctx][576] bf16
    uint16_t *v;             // [B][nh*128] bf16 output
    unsigned *status;
    int B, nh, max_ctx, a_stride, a_off;
    int ctx_lens[kMaxBatch];
    int rope;
    double rope_inv_freq[kMlaRope / 2];
    float eps;
    float qscale;            // log2(e) / sqrt(192): scores in base-2 units
    int HG, C, HPB;          // heads per cluster, blocks per cluster, heads per block
    int nstages;
    int off_ring, off_qb, off_pb, off_qt, off_newrow, off_stat, off_recv, off_ofin,
        off_scr, off_bars;
    unsigned long long timeout_ns;
};

// One latent-cache tensor map per sequence, limited to its cached rows, so a
// tile running past them reads zeros.
struct __align__(128) MlaMaps {
    CUtensorMap cache[kMaxBatch];
};

}  // namespace cfa
