// cfa_internal.h -- constants shared by every kernel and the launch
// parameters of the fused kernel. Not part of the public ABI (that is
// include/cfa.h); the decoder-layer kernels' parameters are in
// cfa_layer_params.h.
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
constexpr int kMergeThreads = 256;                 // head_merge_kernel: two threads per 4 columns
constexpr int kMergeItemsPerBlock = kMergeThreads / 2;
constexpr int kMmaN = 16;                          // batch rows per tensor-core MMA (zero-padded)
constexpr int kXStageMmaBytes = 2 * kMmaN * 128;   // x per stage on the tensor-core path

// Status word bits, written by kernels and read by cfa_plan_status.
constexpr unsigned kStatusTimeoutBit = 1u;
constexpr unsigned kStatusBadLengthBit = 2u;  // a device-resident length was out of range
constexpr unsigned kStatusSiteShift = 8;  // site code of the first timeout

// A load warp's final wait for its own copies in flight uses this many times
// the normal wait limit.
constexpr unsigned long long kDrainTimeoutFactor = 4;

// Site codes recorded with a timeout in the status word.
enum WaitSite : unsigned {
    kSiteStageFull = 1,
    kSiteStageEmpty = 2,
    kSiteQExchange = 3,
    kSiteSoftmaxExchange = 4,
    kSiteKvExchange = 5,
    kSiteDrain = 6,        // a load warp's final wait for its own copies
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
    unsigned *counters;    // [C]: arrivals per column chunk
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
    int merge_separate;    // 1: blocks only write their partials; head_merge_kernel sums them
    int pdl;               // 1: launched with programmatic dependent launch (may start before
                           // the previous kernel in the stream has finished)
    int x_direct;          // 1 (CUDA-core path only): x is read by the compute warps with plain
                           // loads (host-mapped pinned memory), not by TMA
    int rs;                // 1: q/k/v partials exchanged as a reduce-scatter then an all-gather
                           // of the sums; 0: every rank's whole partial to every peer
    int nstages;           // pipeline depth
    int off_xring, off_qkv_recv, off_sm_recv, off_qkv_full, off_attn, off_attn_t, off_scratch,
        off_bars;
    unsigned long long timeout_ns;
    float qscale;          // log2(e) / sqrt(D)
};

}  // namespace cfa
