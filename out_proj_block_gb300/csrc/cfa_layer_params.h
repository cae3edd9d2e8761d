// cfa_layer_params.h -- launch parameters of the decoder-layer kernels (the
// stream-K GEMV of the MLP and projections, and the multi-head latent
// attention core), shared by their host side and the kernels. Not part of the
// public ABI (that is include/cfa.h).
#pragma once

#include <cstdint>

#include <cuda.h>

#include "cfa_internal.h"

namespace cfa {

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
    int xstage_bytes;        // bytes of one x (+ norm weight) stage; on the tensor-core
                             // path, of one whole stage (weights, input box, norm weights)
    int off_xring, off_xn, off_scratch, off_tile, off_misc, off_bars;
    float eps;
    unsigned long long timeout_ns;
};

// The tensor-core GEMV: units of 64 weight rows, read as [64 x 64] swizzled
// boxes; the batch's input rows as one [16 x 64] box; 4 warps read TMEM and
// finish tiles, then one MMA warp, one TMA warp and one warp normalizing the
// input boxes (RMSNorm modes).
constexpr int kGemvMmaRows = 64;
constexpr int kGemvMmaBoxBytes = kGemvMmaRows * 128;
constexpr int kGemvMmaXBytes = kMmaN * 128;
constexpr int kGemvMmaReaders = 4;
constexpr int kGemvMmaThreads = (kGemvMmaReaders + 3) * 32;

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
constexpr int kMlaSplitRec = kMlaV + 4;             // per-split record: v_h [128], M, L, pad

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
    int S;                   // row splits: clusters per (sequence, head group)
    float *vpart;            // S > 1: [B][nh][S][kMlaSplitRec] per-split v_h, max, sum
    unsigned *vcount;        // S > 1: [B][nh / HG][C] arrivals of the splits
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
