// cfa_api.cu -- host side of the C ABI declared in include/cfa.h: plan
// creation and validation, shared-memory layout, tensor-map encoding and the
// cluster launch of the fused kernel.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "cfa.h"
#include "cfa_internal.h"

namespace cfa {
const void *fused_kernel_d128(int maxb);
const void *fused_kernel_d64(int maxb);
const void *selftest_wait_kernel_ptr();
const void *head_merge_kernel_ptr();
const void *copy16_kernel_ptr();
}  // namespace cfa

using cfa::KernelParams;

namespace {

thread_local cfa_status g_last_error = CFA_OK;

cfa_status fail(cfa_status s) {
    g_last_error = s;
    return s;
}

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxStages = 12;
constexpr int kMinStages = 2;
constexpr int kRsBelowStages = 4;

int align_up(int v, int a) { return (v + a - 1) / a * a; }

}  // namespace

struct cfa_plan {
    int B = 0, H = 0, nh = 0, D = 0, max_ctx = 0;
    int device = -1, num_sms = 0, smem_per_sm = 0, smem_optin = 0, smem_reserved = 0;
    int C = 0;
    int stages_override = 0;      // 0 = choose automatically
    int exchange = -1;            // q/k/v exchange: -1 automatic, 0 gather, 1 reduce-scatter
    bool overlap = true;          // programmatic dependent launch
    KernelParams kp{};            // everything but the per-call pointers
    int smem_bytes = 0;
    int coresident_clusters = 0;
    const void *kernel = nullptr;
    // workspace
    float *partials = nullptr;    // [nh][B][H]
    unsigned *words = nullptr;    // [0, kMaxCounters) merge counters, [kMaxCounters] status
    uint16_t *x_stage = nullptr;  // [B][H] for cfa_decode_step_host
    uint16_t *out_stage = nullptr;
    // cached tensor maps
    CUtensorMap tm_wqkv;  // 64-byte aligned by its own declaration
    CUtensorMap tm_wo;
    CUtensorMap tm_x;
    const void *tm_wqkv_src = nullptr;
    const void *tm_x_src = nullptr;
    const void *tm_wo_src = nullptr;
    int tm_wqkv_rows = 0;
    bool tm_mma = false;
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// Row-major bf16 matrix [rows][cols]; boxes of box_rows x box_cols elements.
cfa_status encode_2d(CUtensorMap *tm, const void *base, uint64_t cols, uint64_t rows,
                     uint32_t box_cols, uint32_t box_rows, bool swizzle128 = false) {
    auto fn = tensor_map_encoder();
    if (!fn) return CFA_ERR_CUDA;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), gdim,
                    gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? CFA_OK : CFA_ERR_CUDA;
}

// Tensor maps of one launch. The tensor-core path (kp.n_qk > 0) reads
// 128-byte-swizzled [64-row x 64-col] weight boxes and [16 x 64] x boxes;
// the CUDA-core path reads plain [TRA x 64] boxes and needs no x map.
cfa_status encode_w_qkv(CUtensorMap *tm, const void *W_qkv, int H, const KernelParams &kp) {
    const bool mma = kp.n_qk > 0;
    return encode_2d(tm, W_qkv, 3ull * H, H, cfa::kTileCols, static_cast<uint32_t>(kp.TRA), mma);
}
// W_o boxes: whole [D x 64] tiles on the CUDA-core path, [64 x 64] swizzled
// K slices on the tensor-core path.
cfa_status encode_w_o(CUtensorMap *tm, const void *W_o, int H, int D, const KernelParams &kp) {
    const bool mma = kp.n_qk > 0;
    return encode_2d(tm, W_o, H, H, cfa::kTileCols, static_cast<uint32_t>(mma ? 64 : D), mma);
}
cfa_status encode_x(CUtensorMap *tm, const void *x, int B, int H) {
    return encode_2d(tm, x, H, B, cfa::kTileCols, cfa::kMmaN, true);
}

const void *kernel_for(int D, int maxb) {
    return D == 128 ? cfa::fused_kernel_d128(maxb) : cfa::fused_kernel_d64(maxb);
}

// The shapes a plan accepts (the limits of cfa_plan_create).
cfa_status check_shape(int B, int hidden, int n_heads, int head_dim, int max_ctx) {
    if (B < 1 || hidden < 1 || n_heads < 1 || head_dim < 1 || max_ctx < 1 ||
        static_cast<long long>(n_heads) * head_dim != hidden)
        return CFA_ERR_INVALID_ARG;
    if ((head_dim != 64 && head_dim != 128) || B > 16 || hidden % 64 != 0 ||
        max_ctx > (1 << 22) || hidden > (1 << 16))
        return CFA_ERR_UNSUPPORTED;
    return CFA_OK;
}

// Work split, shared-memory layout and pipeline depth for cluster size C.
// Pure host arithmetic; no CUDA calls.
cfa_status make_layout(const cfa_plan *pl, int C, int stages_override, KernelParams *kp,
                       int *smem_out, int *maxb_out, int *blocks_per_sm_out = nullptr) {
    const int D = pl->D, B = pl->B, H = pl->H;
    if (C != 1 && C != 2 && C != 4 && C != 8 && C != 16) return CFA_ERR_UNSUPPORTED;
    const int G = D / cfa::kTileCols;  // 64-column groups per head block
    if (C < G) return CFA_ERR_UNSUPPORTED;
    const int RG = C / G;
    if (H % RG) return CFA_ERR_UNSUPPORTED;
    const int R = H / RG;
    int TRA = 128;
    while (TRA > 8 && R % TRA) TRA >>= 1;
    if (R % TRA || TRA < cfa::kComputeWarps) return CFA_ERR_UNSUPPORTED;
    if (H % C) return CFA_ERR_UNSUPPORTED;
    const int ncols = H / C;
    if (ncols % cfa::kTileCols) return CFA_ERR_UNSUPPORTED;
    int maxb = 1;
    while (maxb < B) maxb <<= 1;
    // B >= 3 runs the projections on the tensor cores: 64-row [Q|K] stages and
    // 128-row V stages, x staged by TMA as [16 x 64] swizzled boxes.
    const bool mma = maxb >= 4;
    if (mma) {
        if (R % 128) return CFA_ERR_UNSUPPORTED;
        TRA = 64;
    }

    // x: per stage on the tensor-core path; the block's whole x slice once otherwise.
    const int xstage = mma ? cfa::kXStageMmaBytes : 0;
    const int xrows = mma ? 0 : align_up(B * R * 2, 128);
    const int attn_t = mma ? 2 * (D / 64) * cfa::kMmaN * 128 : 0;
    // q/k/v partials: gather mode, every rank's [B][3][64] partial; reduce-
    // scatter mode, this block's partial plus the peers' slices of it (the
    // same size again), whatever C.
    auto qkv_recv_bytes = [&](int rs) { return (rs ? 2 : C) * B * 3 * cfa::kTileCols * 4; };
    const int sm_recv = C * B * (D + 4) * 4;
    const int qkv_full = B * (3 * D + 1) * 4;
    const int attn = B * D * 4;
    // scratch: CUDA-core GEMV reductions; the attention warp states; on the
    // tensor-core path also the second halves of the V accumulator [64][16]
    const int scratch = std::max({mma ? cfa::kTileCols * cfa::kMmaN * 4 : 0,
                                  mma ? 0 : cfa::kComputeWarps * B * cfa::kTileCols * 4,
                                  (cfa::kComputeWarps * D + 2 * cfa::kComputeWarps) * 4});
    // Stages of x ring needed to hold attn and its hi/lo operand (tensor-core
    // path; 0 = never alias).
    const int alias_stages = mma ? (align_up(attn, 1024) + attn_t + xstage - 1) / xstage : 0;
    const int attn_bytes = align_up(attn, 128) + align_up(attn_t, 1024);
    const int per_stage = cfa::kStageBytes + xstage + 16;
    const int grid = pl->nh * C;

    // Pipeline depth and blocks per SM for an exchange mode: as many blocks
    // per SM as the grid needs to cover the SMs (at most 4) while they get at
    // least kMinStages stages, else fewer blocks.
    auto depth = [&](int rs, int &ns_out, int &bps_out) {
        const int fixed_common = align_up(qkv_recv_bytes(rs), 128) + align_up(sm_recv, 128) +
                                 align_up(qkv_full, 128) + align_up(scratch, 128) + xrows +
                                 1024 /* alignment slack, barriers, flags */;
        int per_sm = (grid + pl->num_sms - 1) / std::max(pl->num_sms, 1);
        per_sm = std::min(std::max(per_sm, 1), 4);
        ns_out = 0;
        bps_out = 1;
        for (; per_sm >= 1 && ns_out < kMinStages; --per_sm) {
            const int budget =
                std::min(pl->smem_optin, pl->smem_per_sm / per_sm - pl->smem_reserved);
            ns_out = std::min(kMaxStages, (budget - fixed_common) / per_stage);
            if (!mma || ns_out < alias_stages)  // attn needs its own space
                ns_out = std::min(kMaxStages, (budget - fixed_common - attn_bytes) / per_stage);
            bps_out = per_sm;
        }
    };
    // The reduce-scatter exchange costs one more round of pushes between the
    // projection and attention. With the CUDA-core projections (B <= 2) the
    // step is short and that round costs more than deeper rings return (B=1:
    // 41.4 -> 43.1 us alone with 6 stages instead of 5); with the tensor-core
    // projections it pays (B=16: 238.7 -> 234.6 us with 7 stages instead of 5).
    // It is taken automatically where it fits more blocks on an SM than the
    // gather mode (the grid can then be resident at once: 64 heads of 64 at
    // B=16, C = 4, two blocks of 2 stages instead of one of 7, 139.7 ->
    // 103.2 us alone), and, at the same blocks per SM, where it gives more
    // stages on the tensor-core path or where the gather mode leaves fewer
    // than kRsBelowStages.
    int rs = pl->exchange > 0 ? 1 : 0;
    int NS = 0, blocks_per_sm = 1;
    depth(rs, NS, blocks_per_sm);
    if (pl->exchange < 0 && C > 1) {
        int ns1 = 0, bps1 = 1;
        depth(1, ns1, bps1);
        const bool more_blocks = bps1 > blocks_per_sm;
        const bool more_stages =
            bps1 == blocks_per_sm && ns1 > NS && (mma || NS < kRsBelowStages);
        if (more_blocks || more_stages) {
            rs = 1;
            NS = ns1;
            blocks_per_sm = bps1;
        }
    }
    const int qkv_recv = qkv_recv_bytes(rs);
    if (stages_override > 0) NS = stages_override;
    if (NS < kMinStages || NS > 64) return CFA_ERR_UNSUPPORTED;

    int off = NS * cfa::kStageBytes;
    KernelParams k{};
    k.off_xring = off;
    off = align_up(off + NS * xstage + xrows, 1024);
    // The tensor-core path reads x only in the projection phase, so attn and
    // its hi/lo operand (written after attention) reuse the x ring when it is
    // large enough.
    const bool alias_attn = mma && NS >= alias_stages;
    if (alias_attn) {
        k.off_attn = k.off_xring;
        k.off_attn_t = k.off_xring + align_up(attn, 1024);
    } else {
        k.off_attn_t = off;
        off = align_up(off + attn_t, 128);
    }
    k.off_qkv_recv = off;
    off = align_up(off + qkv_recv, 128);
    k.off_sm_recv = off;
    off = align_up(off + sm_recv, 128);
    k.off_qkv_full = off;
    off = align_up(off + qkv_full, 128);
    if (!alias_attn) {
        k.off_attn = off;
        off = align_up(off + attn, 128);
    }
    k.off_scratch = off;
    off = align_up(off + scratch, 128);
    k.off_bars = off;
    off += (2 * NS + 12) * 8;
    if (off > pl->smem_optin) return CFA_ERR_UNSUPPORTED;

    k.B = B;
    k.H = H;
    k.nh = pl->nh;
    k.max_ctx = pl->max_ctx;
    k.C = C;
    k.G = G;
    k.RG = RG;
    k.R = R;
    k.TRA = TRA;
    k.nA = R / TRA;
    k.n_qk = mma ? R / 64 : 0;
    k.n_v = mma ? R / 128 : 0;
    // TMEM: 48 columns for the projection accumulators ([Q|K] 16, V 32); the
    // out-projection keeps up to 16 tile accumulators of 32 columns (hi and lo
    // halves). Blocks that share an SM must fit its 512 columns together.
    unsigned cols = 64;
    if (mma) {
        const int want = std::min(ncols / cfa::kTileCols, 16) * 2 * cfa::kMmaN;
        while (static_cast<int>(cols) < want) cols <<= 1;
        const int resident = std::max(blocks_per_sm, (pl->smem_per_sm) / (off + pl->smem_reserved));
        while (cols > 64 && static_cast<int>(cols) * resident > 512) cols >>= 1;
    }
    k.tmem_cols = cols;
    k.ncols = ncols;
    // A separate merge kernel where one block would otherwise read more than
    // 256 KB of partials at the end of the fused kernel.
    k.merge_separate = 4ll * pl->nh * B * ncols > (256 << 10) ? 1 : 0;
    if (C > cfa::kMaxCounters) return CFA_ERR_UNSUPPORTED;
    k.nstages = NS;
    k.rs = rs;
    k.timeout_ns = kDefaultTimeoutNs;
    k.qscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(D)));
    *kp = k;
    *smem_out = off;
    *maxb_out = maxb;
    if (blocks_per_sm_out) *blocks_per_sm_out = blocks_per_sm;
    return CFA_OK;
}

cudaLaunchConfig_t launch_config(const cfa_plan *pl, const KernelParams &kp, int smem,
                                 cudaStream_t stream, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl->nh * kp.C, 1, 1);
    cfg.blockDim = dim3(cfa::kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kp.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Apply cluster size C to the plan if the device can run it.
cfa_status configure(cfa_plan *pl, int C, int stages_override) {
    KernelParams kp;
    int smem = 0, maxb = 1;
    cfa_status st = make_layout(pl, C, stages_override, &kp, &smem, &maxb);
    if (st != CFA_OK) return st;
    const void *kernel = kernel_for(pl->D, maxb);
    if (!kernel) return CFA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pl->smem_optin) != cudaSuccess ||
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
        cudaGetLastError();
        return CFA_ERR_CUDA;
    }
    // Whether the grid can be resident at once. Blocks per SM come from the
    // SM's own limits: shared memory, registers (allocated per warp in units of
    // 256), threads. The occupancy calls report one block per SM for the
    // tensor-core kernels at any shared memory size, though the SM holds two
    // (a timeline of such a launch shows two blocks resident on most SMs);
    // they do model how clusters pack into GPCs, which depends only on blocks
    // per SM. So the cluster count is the call's answer for the CUDA-core
    // kernel at a size that gives it the same blocks per SM, and the kernel's
    // own answer where that does not match.
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) {
        cudaGetLastError();
        return CFA_ERR_UNSUPPORTED;
    }
    const int warps = cfa::kThreads / 32;
    const int by_smem = pl->smem_per_sm / (smem + pl->smem_reserved);
    const int by_regs = 65536 / (warps * align_up(std::max(fa.numRegs, 1) * 32, 256));
    const int per_sm = std::min({by_smem, by_regs, 2048 / cfa::kThreads});
    // Clusters of `dim` blocks of function `fn` that the occupancy call fits.
    auto api_clusters = [&](const void *fn, int dim, int bytes) {
        cudaLaunchAttribute a[1];
        cudaLaunchConfig_t c = launch_config(pl, kp, bytes, nullptr, a);
        c.gridDim = dim3(pl->nh * dim, 1, 1);
        a[0].val.clusterDim.x = dim;
        int v = 0;
        if (cudaOccupancyMaxActiveClusters(&v, fn, &c) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        return v;
    };
    int clusters = api_clusters(kernel, C, smem);
    const void *ref = kernel_for(128, 1);
    const int ref_smem = std::min(pl->smem_optin, pl->smem_per_sm / std::max(per_sm, 1) -
                                                      pl->smem_reserved);
    if (clusters >= 1 && per_sm >= 1 && ref && ref != kernel &&
        cudaFuncSetAttribute(ref, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pl->smem_optin) == cudaSuccess &&
        cudaFuncSetAttribute(ref, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess &&
        api_clusters(ref, 1, ref_smem) == per_sm * pl->num_sms)
        clusters = std::max(clusters, api_clusters(ref, C, ref_smem));
    cudaGetLastError();
    if (clusters < 1) return CFA_ERR_UNSUPPORTED;
    pl->C = C;
    pl->kp = kp;
    pl->smem_bytes = smem;
    pl->kernel = kernel;
    pl->coresident_clusters = clusters;
    pl->tm_wqkv_src = nullptr;  // box shapes may have changed
    pl->tm_wo_src = nullptr;
    pl->tm_x_src = nullptr;
    return CFA_OK;
}

// Default cluster size. A grid whose clusters cannot all be resident at once
// runs in waves, each as slow as a whole step, so only sizes whose whole grid
// fits the device at once are taken while one exists: the smallest of those
// that gives every SM a block, else the largest of them. Failing that, the
// largest size that runs at all. Returns the size applied, or 0.
int choose_cluster(cfa_plan *pl) {
    const int candidates[5] = {1, 2, 4, 8, 16};
    int best = 0;  // largest co-resident size seen
    for (int C : candidates) {
        if (configure(pl, C, 0) != CFA_OK || pl->coresident_clusters < pl->nh) continue;
        best = C;
        if (pl->nh * C >= pl->num_sms) return C;
    }
    if (!best)
        for (int i = 4; i >= 0 && !best; --i)
            if (configure(pl, candidates[i], 0) == CFA_OK) best = candidates[i];
    if (best && pl->C != best && configure(pl, best, 0) != CFA_OK) return 0;
    return best;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

void free_workspace(cfa_plan *pl) {
    if (pl->partials) cudaFree(pl->partials);
    if (pl->words) cudaFree(pl->words);
    if (pl->x_stage) cudaFree(pl->x_stage);
    if (pl->out_stage) cudaFree(pl->out_stage);
    pl->partials = nullptr;
    pl->words = nullptr;
    pl->x_stage = pl->out_stage = nullptr;
}

}  // namespace

extern "C" {

const char *cfa_status_string(cfa_status s) {
    switch (s) {
        case CFA_OK: return "CFA_OK";
        case CFA_ERR_INVALID_ARG: return "CFA_ERR_INVALID_ARG";
        case CFA_ERR_UNSUPPORTED: return "CFA_ERR_UNSUPPORTED";
        case CFA_ERR_CUDA: return "CFA_ERR_CUDA";
        case CFA_ERR_TIMEOUT: return "CFA_ERR_TIMEOUT";
        case CFA_ERR_ALIGNMENT: return "CFA_ERR_ALIGNMENT";
    }
    return "CFA_ERR_UNKNOWN";
}

cfa_status cfa_last_error(void) { return g_last_error; }

cfa_plan *cfa_plan_create(int B, int hidden, int n_heads, int head_dim, int max_ctx) {
    const cfa_status shape = check_shape(B, hidden, n_heads, head_dim, max_ctx);
    if (shape != CFA_OK) {
        fail(shape);
        return nullptr;
    }
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    int major = 0, minor = 0, sms = 0, per_sm = 0, optin = 0, reserved = 0, cluster_ok = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&cluster_ok, cudaDevAttrClusterLaunch, dev) != cudaSuccess) {
        cudaGetLastError();
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    if (major != 10 || minor != 3 || !cluster_ok) {  // the library is built for sm_103a only
        fail(CFA_ERR_UNSUPPORTED);
        return nullptr;
    }
    cfa_plan *pl = new (std::nothrow) cfa_plan();
    if (!pl) {
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    pl->B = B;
    pl->H = hidden;
    pl->nh = n_heads;
    pl->D = head_dim;
    pl->max_ctx = max_ctx;
    pl->device = dev;
    pl->num_sms = sms;
    pl->smem_per_sm = per_sm;
    pl->smem_optin = optin;
    pl->smem_reserved = reserved;

    const size_t part_bytes = sizeof(float) * static_cast<size_t>(n_heads) * B * hidden;
    const size_t act_bytes = 2u * static_cast<size_t>(B) * hidden;
    if (cudaMalloc(&pl->partials, part_bytes) != cudaSuccess ||
        cudaMalloc(&pl->words, sizeof(unsigned) * (cfa::kMaxCounters + 16)) != cudaSuccess ||
        cudaMalloc(&pl->x_stage, act_bytes) != cudaSuccess ||
        cudaMalloc(&pl->out_stage, act_bytes) != cudaSuccess ||
        cudaMemset(pl->words, 0, sizeof(unsigned) * (cfa::kMaxCounters + 16)) != cudaSuccess) {
        cudaGetLastError();
        free_workspace(pl);
        delete pl;
        fail(CFA_ERR_CUDA);
        return nullptr;
    }

    if (!choose_cluster(pl)) {
        free_workspace(pl);
        delete pl;
        fail(CFA_ERR_UNSUPPORTED);
        return nullptr;
    }
    return pl;
}

void cfa_plan_destroy(cfa_plan *pl) {
    if (!pl) return;
    cudaDeviceSynchronize();
    free_workspace(pl);
    delete pl;
}

cfa_status cfa_plan_set_cluster_size(cfa_plan *pl, int C) {
    if (!pl) return fail(CFA_ERR_INVALID_ARG);
    const cfa_status st = configure(pl, C, pl->stages_override);
    return st == CFA_OK ? CFA_OK : fail(st);  // on error the plan is unchanged
}

cfa_status cfa_plan_set_stages(cfa_plan *pl, int stages) {
    if (!pl || stages < 0) return fail(CFA_ERR_INVALID_ARG);
    const cfa_status st = configure(pl, pl->C, stages);
    if (st != CFA_OK) return fail(st);  // on error the plan is unchanged
    pl->stages_override = stages;
    return CFA_OK;
}

cfa_status cfa_plan_set_qkv_exchange(cfa_plan *pl, int mode) {
    if (!pl || mode < -1 || mode > 1) return fail(CFA_ERR_INVALID_ARG);
    const int old = pl->exchange;
    pl->exchange = mode;
    const cfa_status st = configure(pl, pl->C, pl->stages_override);
    if (st != CFA_OK) {
        pl->exchange = old;  // on error the plan is unchanged
        return fail(st);
    }
    return CFA_OK;
}

cfa_status cfa_plan_set_overlap(cfa_plan *pl, int enable) {
    if (!pl) return fail(CFA_ERR_INVALID_ARG);
    pl->overlap = enable != 0;
    return CFA_OK;
}

int cfa_plan_cluster_size(const cfa_plan *pl) { return pl ? pl->C : -1; }

cfa_status cfa_plan_describe(const cfa_plan *pl, char *buf, int len) {
    if (!pl || !buf || len < 1) return fail(CFA_ERR_INVALID_ARG);
    const KernelParams &k = pl->kp;
    std::snprintf(buf, static_cast<size_t>(len),
                  "{\"B\": %d, \"hidden\": %d, \"n_heads\": %d, \"head_dim\": %d, "
                  "\"max_ctx\": %d, \"cluster_size\": %d, \"grid\": %d, \"block\": %d, "
                  "\"smem_bytes\": %d, \"stages\": %d, \"stage_bytes\": %d, "
                  "\"proj_rows_per_block\": %d, \"proj_tile_rows\": %d, "
                  "\"out_cols_per_block\": %d, \"coresident_clusters\": %d, \"num_sms\": %d, "
                  "\"overlap\": %d, \"merge\": \"%s\", \"launches_per_step\": %d, "
                  "\"qkv_exchange\": \"%s\"}",
                  pl->B, pl->H, pl->nh, pl->D, pl->max_ctx, pl->C, pl->nh * pl->C,
                  cfa::kThreads, pl->smem_bytes, k.nstages, cfa::kStageBytes, k.R, k.TRA,
                  k.ncols, pl->coresident_clusters, pl->num_sms, pl->overlap ? 1 : 0,
                  k.merge_separate ? "separate" : "flat",
                  k.merge_separate ? 2 : 1, k.rs ? "reduce_scatter" : "gather");
    return CFA_OK;
}

cfa_status cfa_plan_layout(int B, int hidden, int n_heads, int head_dim, int max_ctx, int C,
                           int exchange, int stages, int num_sms, int smem_per_sm,
                           int smem_optin, int smem_reserved, char *buf, int len) {
    if (!buf || len < 256) return fail(CFA_ERR_INVALID_ARG);
    const cfa_status shape = check_shape(B, hidden, n_heads, head_dim, max_ctx);
    if (shape != CFA_OK) return fail(shape);
    if (exchange < -1 || exchange > 1 || stages < 0 || stages > 64 || num_sms < 1 ||
        num_sms > 4096 || smem_per_sm < 1 || smem_per_sm > (1 << 20) || smem_optin < 1 ||
        smem_optin > smem_per_sm || smem_reserved < 0 || smem_reserved >= smem_per_sm)
        return fail(CFA_ERR_INVALID_ARG);
    cfa_plan pl;  // the fields the layout reads; no device memory, no CUDA call
    pl.B = B;
    pl.H = hidden;
    pl.nh = n_heads;
    pl.D = head_dim;
    pl.max_ctx = max_ctx;
    pl.num_sms = num_sms;
    pl.smem_per_sm = smem_per_sm;
    pl.smem_optin = smem_optin;
    pl.smem_reserved = smem_reserved;
    pl.exchange = exchange;
    KernelParams k{};
    int smem = 0, maxb = 1, bps = 1;
    const cfa_status st = make_layout(&pl, C, stages, &k, &smem, &maxb, &bps);
    if (st != CFA_OK) return fail(st);
    std::snprintf(buf, static_cast<size_t>(len),
                  "{\"cluster_size\": %d, \"grid\": %d, \"blocks_per_sm\": %d, \"stages\": %d, "
                  "\"smem_bytes\": %d, \"qkv_exchange\": \"%s\", \"tensor_cores\": %d, "
                  "\"tmem_cols\": %u, \"proj_rows_per_block\": %d, \"proj_tile_rows\": %d, "
                  "\"out_cols_per_block\": %d, \"merge\": \"%s\"}",
                  C, n_heads * C, bps, k.nstages, smem, k.rs ? "reduce_scatter" : "gather",
                  k.n_qk > 0 ? 1 : 0, k.n_qk > 0 ? k.tmem_cols : 0u, k.R, k.TRA, k.ncols,
                  k.merge_separate ? "separate" : "flat");
    return CFA_OK;
}

}  // extern "C"

namespace {

// The cross-head merge kernel behind a fused launch whose plan merges
// separately (same stream; programmatic dependent launch when `overlap`).
cudaError_t launch_head_merge(const KernelParams &kp, bool overlap, cudaStream_t stream) {
    const int items = kp.B * (kp.H / 4);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((items + cfa::kMergeItemsPerBlock - 1) / cfa::kMergeItemsPerBlock, 1, 1);
    cfg.blockDim = dim3(cfa::kMergeThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    const float *partials = kp.partials;
    int nh = kp.nh, B = kp.B, H = kp.H;
    const uint16_t *resid = kp.resid;
    uint16_t *out = kp.out;
    void *args[6] = {&partials, &nh, &B, &H, &resid, &out};
    return cudaLaunchKernelExC(&cfg, cfa::head_merge_kernel_ptr(), args);
}

// One launch of the fused kernel with the given tensor maps. lens (host,
// one per sequence) or lens_dev (device-resident, read by the kernel) gives
// the cached positions; resid (or null) is added to out.
cfa_status launch_fused(cfa_plan *pl, const CUtensorMap *tm_wqkv, const CUtensorMap *tm_wo,
                        const CUtensorMap *tm_x, const void *x, void *k_cache, void *v_cache,
                        const int *lens, const int *lens_dev, double rope_theta,
                        const void *resid, void *out, cudaStream_t stream, bool x_direct = false) {
    KernelParams kp = pl->kp;
    kp.x_direct = x_direct ? 1 : 0;
    kp.x = static_cast<const uint16_t *>(x);
    kp.k_cache = static_cast<uint16_t *>(k_cache);
    kp.v_cache = static_cast<uint16_t *>(v_cache);
    kp.out = static_cast<uint16_t *>(out);
    kp.resid = static_cast<const uint16_t *>(resid);
    kp.lens_dev = lens_dev;
    kp.partials = pl->partials;
    kp.counters = pl->words;
    kp.status = pl->words + cfa::kMaxCounters;
    for (int b = 0; b < pl->B; ++b) kp.ctx_lens[b] = lens ? lens[b] : 0;
    kp.rope = rope_theta > 0.0 ? 1 : 0;
    if (kp.rope)
        for (int i = 0; i < pl->D / 2; ++i)
            kp.rope_inv_freq[i] = std::pow(rope_theta, -2.0 * i / pl->D);

    kp.pdl = pl->overlap ? 1 : 0;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config(pl, kp, pl->smem_bytes, stream, attr);
    if (pl->overlap) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.numAttrs = 2;
    }
    CUtensorMap m_wqkv = *tm_wqkv, m_wo = *tm_wo, m_x = *tm_x;
    void *args[4] = {&m_wqkv, &m_wo, &m_x, &kp};
    if (cudaLaunchKernelExC(&cfg, pl->kernel, args) != cudaSuccess ||
        (kp.merge_separate && launch_head_merge(kp, pl->overlap, stream) != cudaSuccess)) {
        cudaGetLastError();
        return fail(CFA_ERR_CUDA);
    }
    return CFA_OK;
}

// The launch behind cfa_decode_step and cfa_decode_step_ex: lens[b] cached
// positions per sequence, rope_theta > 0 enables the rotary embedding.
// x_direct: x is in host-mapped memory and read with plain loads (CUDA-core
// path only).
cfa_status launch_step(cfa_plan *pl, const void *x, const void *W_qkv, const void *W_o,
                       void *k_cache, void *v_cache, const int *lens, double rope_theta,
                       void *out, void *stream, bool x_direct = false) {
    if (!pl || !x || !W_qkv || !W_o || !k_cache || !v_cache || !out || !lens)
        return fail(CFA_ERR_INVALID_ARG);
    for (int b = 0; b < pl->B; ++b)
        if (lens[b] < 0 || lens[b] >= pl->max_ctx) return fail(CFA_ERR_INVALID_ARG);
    if (!(rope_theta >= 0.0) || rope_theta > 1e30) return fail(CFA_ERR_INVALID_ARG);
    if (!aligned16(x) || !aligned16(W_qkv) || !aligned16(W_o) || !aligned16(k_cache) ||
        !aligned16(v_cache) || !aligned16(out))
        return fail(CFA_ERR_ALIGNMENT);
    const size_t H = static_cast<size_t>(pl->H);
    const size_t act = 2 * H * pl->B;
    const size_t cache = 2 * static_cast<size_t>(pl->B) * pl->nh * pl->max_ctx * pl->D;
    if (overlaps(out, act, x, act) || overlaps(out, act, W_qkv, 2 * H * 3 * H) ||
        overlaps(out, act, W_o, 2 * H * H) || overlaps(out, act, k_cache, cache) ||
        overlaps(out, act, v_cache, cache))
        return fail(CFA_ERR_INVALID_ARG);

    const bool mma = pl->kp.n_qk > 0;
    if (pl->tm_wqkv_src != W_qkv || pl->tm_wqkv_rows != pl->kp.TRA || pl->tm_mma != mma) {
        if (encode_w_qkv(&pl->tm_wqkv, W_qkv, pl->H, pl->kp) != CFA_OK) {
            pl->tm_wqkv_src = nullptr;
            return fail(CFA_ERR_CUDA);
        }
        pl->tm_wqkv_src = W_qkv;
        pl->tm_wqkv_rows = pl->kp.TRA;
        pl->tm_wo_src = nullptr;
        pl->tm_mma = mma;
    }
    if (pl->tm_wo_src != W_o) {
        if (encode_w_o(&pl->tm_wo, W_o, pl->H, pl->D, pl->kp) != CFA_OK) {
            pl->tm_wo_src = nullptr;
            return fail(CFA_ERR_CUDA);
        }
        pl->tm_wo_src = W_o;
    }
    if (mma && pl->tm_x_src != x) {
        if (encode_x(&pl->tm_x, x, pl->B, pl->H) != CFA_OK) {
            pl->tm_x_src = nullptr;
            return fail(CFA_ERR_CUDA);
        }
        pl->tm_x_src = x;
    }
    if (!mma) pl->tm_x = pl->tm_wqkv;  // unused by the CUDA-core path

    return launch_fused(pl, &pl->tm_wqkv, &pl->tm_wo, &pl->tm_x, x, k_cache, v_cache, lens,
                        nullptr, rope_theta, nullptr, out, static_cast<cudaStream_t>(stream), x_direct);
}

}  // namespace

extern "C" {

cfa_status cfa_decode_step(cfa_plan *pl, const void *x, const void *W_qkv, const void *W_o,
                           void *k_cache, void *v_cache, int ctx_len, void *out,
                           void *stream) {
    if (!pl) return fail(CFA_ERR_INVALID_ARG);
    int lens[cfa::kMaxBatch];
    for (int b = 0; b < pl->B; ++b) lens[b] = ctx_len;
    return launch_step(pl, x, W_qkv, W_o, k_cache, v_cache, lens, 0.0, out, stream);
}

cfa_status cfa_decode_step_ex(cfa_plan *pl, const void *x, const void *W_qkv, const void *W_o,
                              void *k_cache, void *v_cache, const int *ctx_lens,
                              double rope_theta, void *out, void *stream) {
    return launch_step(pl, x, W_qkv, W_o, k_cache, v_cache, ctx_lens, rope_theta, out, stream);
}

namespace {

// Device address of page-locked host memory the GPU can access (cudaHostAlloc,
// cudaHostRegister), or null for other host memory.
void *mapped_host_ptr(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// copy16_kernel of `bytes` (a multiple of 16) on the stream, overlapping its
// neighbours when the plan allows it.
cudaError_t launch_copy16(const void *src, void *dst, size_t bytes, bool overlap, cudaStream_t s) {
    const int n16 = static_cast<int>(bytes / 16);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min((n16 + 255) / 256, 152), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap ? 1 : 0;
    const uint4 *in = static_cast<const uint4 *>(src);
    uint4 *out = static_cast<uint4 *>(dst);
    int n = n16;
    void *args[3] = {&in, &out, &n};
    return cudaLaunchKernelExC(&cfg, cfa::copy16_kernel_ptr(), args);
}

}  // namespace

cfa_status cfa_decode_step_host(cfa_plan *pl, const void *x_host, const void *W_qkv,
                                const void *W_o, void *k_cache, void *v_cache, int ctx_len,
                                void *out_host, void *stream) {
    if (!pl || !x_host || !out_host) return fail(CFA_ERR_INVALID_ARG);
    if (ctx_len < 0 || ctx_len >= pl->max_ctx) return fail(CFA_ERR_INVALID_ARG);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t act = 2u * static_cast<size_t>(pl->B) * pl->H;
    // Page-locked, device-mapped buffers: the GPU reads x and writes out
    // itself, with no DMA transfer to set up. The step stores out straight into
    // the host buffer; on the CUDA-core path it also reads x there (plain
    // loads), on the tensor-core path a copy kernel stages x for its TMA loads.
    void *x_dev = mapped_host_ptr(x_host), *out_dev = mapped_host_ptr(out_host);
    if (x_dev && out_dev && aligned16(x_dev) && aligned16(out_dev)) {
        const bool direct = pl->kp.n_qk == 0;
        if (!direct && launch_copy16(x_dev, pl->x_stage, act, pl->overlap, s) != cudaSuccess) {
            cudaGetLastError();
            return fail(CFA_ERR_CUDA);
        }
        int lens[cfa::kMaxBatch];
        for (int b = 0; b < pl->B; ++b) lens[b] = ctx_len;
        const cfa_status st = launch_step(pl, direct ? x_dev : pl->x_stage, W_qkv, W_o, k_cache,
                                          v_cache, lens, 0.0, out_dev, s, direct);
        if (st != CFA_OK) return st;
        if (cudaStreamSynchronize(s) != cudaSuccess) {
            cudaGetLastError();
            return fail(CFA_ERR_CUDA);
        }
        return CFA_OK;
    }
    if (cudaMemcpyAsync(pl->x_stage, x_host, act, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        cudaGetLastError();
        return fail(CFA_ERR_CUDA);
    }
    const cfa_status st =
        cfa_decode_step(pl, pl->x_stage, W_qkv, W_o, k_cache, v_cache, ctx_len, pl->out_stage, s);
    if (st != CFA_OK) return st;
    if (cudaMemcpyAsync(out_host, pl->out_stage, act, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return fail(CFA_ERR_CUDA);
    }
    return CFA_OK;
}

cfa_status cfa_plan_status(cfa_plan *pl) {
    if (!pl) return fail(CFA_ERR_INVALID_ARG);
    unsigned word = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&word, pl->words + cfa::kMaxCounters, sizeof word, cudaMemcpyDeviceToHost) !=
            cudaSuccess ||
        cudaMemset(pl->words + cfa::kMaxCounters, 0, sizeof word) != cudaSuccess) {
        cudaGetLastError();
        return fail(CFA_ERR_CUDA);
    }
    if (word & cfa::kStatusTimeoutBit) return fail(CFA_ERR_TIMEOUT);
    if (word & cfa::kStatusBadLengthBit) return fail(CFA_ERR_INVALID_ARG);
    return CFA_OK;
}

cfa_status cfa_selftest_wait_timeout(int limit_us, void *stream) {
    if (limit_us < 1 || limit_us > (1 << 20)) return fail(CFA_ERR_INVALID_ARG);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned *word = nullptr;
    unsigned host = 0;
    if (cudaMalloc(&word, sizeof(unsigned)) != cudaSuccess) {
        cudaGetLastError();
        return fail(CFA_ERR_CUDA);
    }
    unsigned long long ns = static_cast<unsigned long long>(limit_us) * 1000ull;
    void *args[2] = {&word, &ns};
    cudaError_t e = cudaMemsetAsync(word, 0, sizeof(unsigned), s);
    if (e == cudaSuccess)
        e = cudaLaunchKernel(cfa::selftest_wait_kernel_ptr(), dim3(1), dim3(32), args, 0, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&host, word, sizeof host, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(word);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(CFA_ERR_CUDA);
    }
    return (host & cfa::kStatusTimeoutBit) ? CFA_ERR_TIMEOUT : CFA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode step without any device allocation.
//
// Some callers cannot allocate device memory once they are running: engines
// whose device memory is owned and budgeted by a host framework (plugins that
// are handed only their input and output buffers), and serving loops that
// forbid cudaMalloc after start-up because it can synchronize the device and
// can fail under memory pressure. For them, cfa_decode_step_noalloc runs the
// same fused kernel as cfa_decode_step but keeps its scratch (the per-column
// arrival counters, the status word and the fp32 per-head output-projection
// partials) in the file-scope array below, which every GPU that loads this
// library holds until the process exits.
// ---------------------------------------------------------------------------

namespace {

constexpr size_t kNoallocWordsBytes = (cfa::kMaxCounters + 64) * 4;  // counters + status word
constexpr size_t kNoallocPartialFloats = size_t(1) << 21;   // n_heads * B * hidden
constexpr size_t kNoallocBytes = kNoallocWordsBytes + kNoallocPartialFloats * sizeof(float);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mutex;
unsigned char *g_noalloc_ptr[kNoallocMaxDevices] = {};  // null until set up

// Once per device, with that device current: the array's device address (the
// host-side name is only a stand-in) and a zeroed counter/status region. A
// device counts as set up only when every step succeeded, so a call that
// failed here (inside a stream capture, say) leaves the next call to retry.
// Returns the address, or null.
unsigned char *noalloc_scratch(int dev) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev]) return g_noalloc_ptr[dev];
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e == cudaSuccess) e = cudaMemset(ptr, 0, kNoallocWordsBytes);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    g_noalloc_ptr[dev] = static_cast<unsigned char *>(ptr);
    return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" cfa_status cfa_decode_step_noalloc(int B, int hidden, int n_heads, int head_dim,
                                              int max_ctx, const void *x, const void *W_qkv,
                                              const void *W_o, void *k_cache, void *v_cache,
                                              int ctx_len, void *out, void *stream) {
    if (B < 1 || hidden < 1 || n_heads < 1 || head_dim < 1 || max_ctx < 1 ||
        static_cast<long long>(n_heads) * head_dim != hidden)
        return fail(CFA_ERR_INVALID_ARG);
    if ((head_dim != 64 && head_dim != 128) || B > 16 || hidden % 64 != 0 ||
        max_ctx > (1 << 22) || hidden > (1 << 16))
        return fail(CFA_ERR_UNSUPPORTED);
    const size_t noalloc_floats = static_cast<size_t>(n_heads) * B * hidden;
    if (noalloc_floats > kNoallocPartialFloats)
        return fail(CFA_ERR_UNSUPPORTED);  // scratch array too small for this shape
    if (!x || !W_qkv || !W_o || !k_cache || !v_cache || !out) return fail(CFA_ERR_INVALID_ARG);
    if (ctx_len < 0 || ctx_len >= max_ctx) return fail(CFA_ERR_INVALID_ARG);
    if (!aligned16(x) || !aligned16(W_qkv) || !aligned16(W_o) || !aligned16(k_cache) ||
        !aligned16(v_cache) || !aligned16(out))
        return fail(CFA_ERR_ALIGNMENT);
    const size_t H = static_cast<size_t>(hidden);
    const size_t act = 2 * H * B;
    const size_t cache = 2 * static_cast<size_t>(B) * n_heads * max_ctx * head_dim;
    if (overlaps(out, act, x, act) || overlaps(out, act, W_qkv, 2 * H * 3 * H) ||
        overlaps(out, act, W_o, 2 * H * H) || overlaps(out, act, k_cache, cache) ||
        overlaps(out, act, v_cache, cache))
        return fail(CFA_ERR_INVALID_ARG);

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoallocMaxDevices) {
        cudaGetLastError();
        return fail(CFA_ERR_CUDA);
    }
    unsigned char *scratch = noalloc_scratch(dev);
    if (!scratch) return fail(CFA_ERR_CUDA);

    // A plan object on the stack: same device queries, cluster-size choice and
    // shared-memory layout as cfa_plan_create, with no workspace behind it.
    cfa_plan pl;
    pl.B = B;
    pl.H = hidden;
    pl.nh = n_heads;
    pl.D = head_dim;
    pl.max_ctx = max_ctx;
    pl.device = dev;
    int major = 0, minor = 0, cluster_ok = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&cluster_ok, cudaDevAttrClusterLaunch, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&pl.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&pl.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                               dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&pl.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&pl.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess) {
        cudaGetLastError();
        return fail(CFA_ERR_CUDA);
    }
    if (major != 10 || minor != 3 || !cluster_ok) return fail(CFA_ERR_UNSUPPORTED);
    if (!choose_cluster(&pl)) return fail(CFA_ERR_UNSUPPORTED);

    CUtensorMap tm_wqkv, tm_wo, tm_x;
    if (encode_w_qkv(&tm_wqkv, W_qkv, hidden, pl.kp) != CFA_OK ||
        encode_w_o(&tm_wo, W_o, hidden, head_dim, pl.kp) != CFA_OK)
        return fail(CFA_ERR_CUDA);
    if (pl.kp.n_qk > 0) {
        if (encode_x(&tm_x, x, B, hidden) != CFA_OK) return fail(CFA_ERR_CUDA);
    } else {
        tm_x = tm_wqkv;  // unused by the CUDA-core path
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Counters must start at zero; the previous call may have been cut short.
    if (cudaMemsetAsync(scratch, 0, kNoallocWordsBytes, s) != cudaSuccess) {
        cudaGetLastError();
        return fail(CFA_ERR_CUDA);
    }
    KernelParams kp = pl.kp;
    kp.x = static_cast<const uint16_t *>(x);
    kp.k_cache = static_cast<uint16_t *>(k_cache);
    kp.v_cache = static_cast<uint16_t *>(v_cache);
    kp.out = static_cast<uint16_t *>(out);
    kp.counters = reinterpret_cast<unsigned *>(scratch);
    kp.status = reinterpret_cast<unsigned *>(scratch) + cfa::kMaxCounters;
    kp.partials = reinterpret_cast<float *>(scratch + kNoallocWordsBytes);
    for (int b = 0; b < B; ++b) kp.ctx_lens[b] = ctx_len;
    kp.rope = 0;
    kp.pdl = 0;  // launched without programmatic dependent launch
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = launch_config(&pl, kp, pl.smem_bytes, s, attr);
    void *args[4] = {&tm_wqkv, &tm_wo, &tm_x, &kp};
    if (cudaLaunchKernelExC(&cfg, pl.kernel, args) != cudaSuccess ||
        (kp.merge_separate && launch_head_merge(kp, false, s) != cudaSuccess)) {
        cudaGetLastError();
        return fail(CFA_ERR_CUDA);
    }
    return CFA_OK;
}

// ------------------------------------------------------------------------
// Internal entry points for the decoder-layer stack (cfa_stack.cu).

namespace cfa {

cfa_status plan_encode_layer(const cfa_plan *pl, const void *W_qkv, const void *W_o,
                             CUtensorMap *tm_wqkv, CUtensorMap *tm_wo) {
    if (encode_w_qkv(tm_wqkv, W_qkv, pl->H, pl->kp) != CFA_OK ||
        encode_w_o(tm_wo, W_o, pl->H, pl->D, pl->kp) != CFA_OK)
        return CFA_ERR_CUDA;
    return CFA_OK;
}

cfa_status plan_encode_input(const cfa_plan *pl, const void *x, CUtensorMap *tm_x) {
    std::memset(tm_x, 0, sizeof *tm_x);  // unused by the CUDA-core path
    if (pl->kp.n_qk > 0 && encode_x(tm_x, x, pl->B, pl->H) != CFA_OK) return CFA_ERR_CUDA;
    return CFA_OK;
}

cfa_status plan_launch_layer(cfa_plan *pl, const CUtensorMap *tm_wqkv, const CUtensorMap *tm_wo,
                             const CUtensorMap *tm_x, const void *x, void *k_cache,
                             void *v_cache, const int *lens_dev, double rope_theta,
                             const void *resid, void *out, cudaStream_t stream) {
    return launch_fused(pl, tm_wqkv, tm_wo, tm_x, x, k_cache, v_cache, nullptr, lens_dev,
                        rope_theta, resid, out, stream);
}

int plan_launches_per_step(const cfa_plan *pl) { return pl->kp.merge_separate ? 2 : 1; }

unsigned *plan_status_word(cfa_plan *pl) { return pl->words + kMaxCounters; }

cfa_status encode_bf16_2d(CUtensorMap *tm, const void *base, uint64_t cols, uint64_t rows,
                          uint32_t box_cols, uint32_t box_rows) {
    return encode_2d(tm, base, cols, rows, box_cols, box_rows, false);
}

cfa_status encode_bf16_2d_ex(CUtensorMap *tm, const void *base, uint64_t cols, uint64_t rows,
                             uint64_t row_stride, uint32_t box_cols, uint32_t box_rows,
                             bool swizzle128) {
    auto fn = tensor_map_encoder();
    if (!fn) return CFA_ERR_CUDA;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {row_stride * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), gdim,
                    gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? CFA_OK : CFA_ERR_CUDA;
}

cfa_status set_last_error(cfa_status s) { return fail(s); }

}  // namespace cfa
