// cfa_stack.cu -- host side of the decoder layer around the fused attention
// block: RMSNorm, the SwiGLU MLP (two stream-K GEMV launches), and the
// multi-layer decode loop, launched eagerly or recorded once into a CUDA graph
// and replayed token after token.
//
// Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命" (ClusterFusion
// framework analysis), written [CF §n]: the page reports time per output
// token of a whole Llama2-7B decoder [CF §3.3, §5.1]; a layer here is its
// fused attention block plus the Llama2-arrangement norms, residuals and MLP.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "cfa.h"
#include "cfa_host.h"
#include "cfa_internal.h"
#include "cfa_layer_params.h"

using cfa::GemvParams;

namespace {

constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s per device-side wait
constexpr int kMaxGemvStages = 12;

cfa_status fail(cfa_status s) { return cfa::set_last_error(s); }

int align_up(int v, int a) { return (v + a - 1) / a * a; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

struct Device {
    int id = -1, sms = 0, smem_per_sm = 0, smem_optin = 0, smem_reserved = 0;
};

cfa_status query_device(Device *d) {
    int major = 0, minor = 0;
    if (cudaGetDevice(&d->id) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d->id) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d->id) != cudaSuccess ||
        cudaDeviceGetAttribute(&d->sms, cudaDevAttrMultiProcessorCount, d->id) != cudaSuccess ||
        cudaDeviceGetAttribute(&d->smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                               d->id) != cudaSuccess ||
        cudaDeviceGetAttribute(&d->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d->id) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&d->smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock,
                               d->id) != cudaSuccess) {
        cudaGetLastError();
        return CFA_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return CFA_ERR_UNSUPPORTED;  // built for sm_103a only
    return CFA_OK;
}

// Launch with programmatic dependent launch allowed (the kernels wait for
// their predecessor before reading its output).
cfa_status launch_pdl(const void *kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                      void **args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelExC(&cfg, kernel, args) != cudaSuccess) {
        cudaGetLastError();
        return CFA_ERR_CUDA;
    }
    return CFA_OK;
}

cfa_status launch_rmsnorm(int B, int n, const void *x, const void *g, float eps, void *y,
                          cudaStream_t stream) {
    const uint16_t *xp = static_cast<const uint16_t *>(x);
    const uint16_t *gp = static_cast<const uint16_t *>(g);
    uint16_t *yp = static_cast<uint16_t *>(y);
    void *args[5] = {&xp, &gp, &yp, &n, &eps};
    return launch_pdl(cfa::rmsnorm_kernel_ptr(), dim3(B), dim3(256), 0, stream, args);
}

// ------------------------------------------------------------ stream-K GEMV plan

struct GemvPlan {
    GemvParams gp{};
    const void *kernel = nullptr;
    int smem = 0;
    int threads = 0;
    bool mma = false;             // the tensor-core kernel
    int resident = 0;             // blocks per SM the occupancy calculator allows
    size_t partial_floats = 0;
};

// Which kernel runs a GEMV of batch B: kGemvPathAuto takes the tensor cores
// from B = 2 on (measured at Llama2-7B MLP shapes: 53.9 vs 59.0 µs at B = 2,
// on par at B = 1), where the CUDA cores spend longer on the 2B flops per
// weight byte than HBM needs to deliver the byte.
constexpr int kGemvPathAuto = -1, kGemvPathCudaCores = 0, kGemvPathTensorCores = 1;

bool gemv_uses_mma(int path, int B) {
    if (path == kGemvPathCudaCores) return false;
    return path == kGemvPathTensorCores || B >= 2;
}

// Shared-memory layout, pipeline depth and grid of one stream-K GEMV.
// bps_req / ns_req > 0 ask for that many blocks per SM / stages.
cfa_status make_gemv(const Device &dev, int mode, int B, int K, int N, GemvPlan *out,
                     int bps_req = 0, int ns_req = 0, int path = kGemvPathAuto) {
    const bool dual = mode == cfa::kGemvSwiGLU;
    const bool norm = dual || mode == cfa::kGemvNormPlain;
    const bool mma = gemv_uses_mma(path, B);
    const int TW = cfa::kGemvTileCols;
    int maxb = 1;
    while (maxb < B) maxb <<= 1;
    // On the CUDA cores: 32 KB of weights per unit for a single batch row when
    // K divides into them (one issuing thread streams more with fewer,
    // larger copies), else 16 KB; on the tensor cores, 64 rows of each matrix
    // (16 or 32 KB).
    const int r_narrow = dual ? 32 : 64;
    const bool wide = !mma && maxb == 1 && K % (2 * r_narrow) == 0;
    const int R = mma ? cfa::kGemvMmaRows : r_narrow * (wide ? 2 : 1);
    const int unit_bytes = wide ? 2 * cfa::kStageBytes : cfa::kStageBytes;
    // N a multiple of 64: a last tile of 64 columns reads zeros past N and
    // stores nothing there.
    if (K < R || K % R || N < 64 || N % 64 || B > cfa::kMaxBatch) return CFA_ERR_UNSUPPORTED;
    const void *kernel = mma ? cfa::gemv_mma_kernel_ptr(mode) : cfa::gemv_kernel(mode, maxb, wide);
    if (!kernel) return CFA_ERR_UNSUPPORTED;
    const int threads = mma ? cfa::kGemvMmaThreads : cfa::kGemvThreads;
    const int NW = (dual ? 2 : 1) * TW;

    GemvParams p{};
    p.B = B;
    p.K = K;
    p.N = N;
    p.rows = R;
    p.chunks = K / R;
    p.n_tiles = (N + TW - 1) / TW;
    p.x_stride = K;
    p.units = p.n_tiles * p.chunks;
    int fixed = 0, per_stage = 0, xn = 0, scratch = 0;
    const int tile = align_up((mma ? 1 : 2) * B * NW * 4, 128);  // tile buffers
    const int misc = 128;
    if (mma) {
        // stage: weight boxes, the [16 x 64] input box, the norm weights
        p.xstage_bytes = align_up((dual ? 2 : 1) * 2 * cfa::kGemvMmaBoxBytes + cfa::kGemvMmaXBytes +
                                      (norm ? R * 2 : 0), 1024);
        scratch = norm ? align_up(cfa::kGemvMmaReaders * cfa::kMaxBatch * 4, 128) : 0;
        per_stage = p.xstage_bytes + 24;
        fixed = scratch + tile + misc + 64 + 1024;
    } else {
        p.xstage_bytes = align_up(B * R * 2 + (norm ? R * 2 : 0), 128);
        // per-warp normalized input rows: 8 warps x [B][R/4] floats
        xn = norm ? align_up(cfa::kComputeWarps * B * (R / 4) * 4, 128) : 0;
        scratch = align_up(cfa::kComputeWarps * B * cfa::kTileCols * 4, 128);
        per_stage = unit_bytes + p.xstage_bytes + 16;
        fixed = xn + scratch + tile + misc + 1024;  // + barriers, flags, slack
    }
    // Two blocks per SM with at least 64 KB of weight stages each (3 stages
    // on the tensor cores), else one deeper block.
    int bps = 2, NS = 0;
    for (; bps >= 1; --bps) {
        const int budget = std::min(dev.smem_optin, dev.smem_per_sm / bps - dev.smem_reserved);
        NS = std::min(kMaxGemvStages, (budget - fixed) / per_stage);
        if (NS >= (bps == 2 ? (mma ? 3 : 65536 / unit_bytes) : 2)) break;
    }
    if (bps_req > 0) {
        bps = bps_req;
        const int budget = std::min(dev.smem_optin, dev.smem_per_sm / bps - dev.smem_reserved);
        NS = std::min(kMaxGemvStages, (budget - fixed) / per_stage);
    }
    if (ns_req > 0) {
        if (ns_req > NS) return CFA_ERR_UNSUPPORTED;  // does not fit at this occupancy
        NS = ns_req;
    }
    if (bps < 1 || NS < 2) return CFA_ERR_UNSUPPORTED;
    int off = 0;
    if (mma) {
        off = NS * p.xstage_bytes;  // the ring: whole stages
        p.off_xring = 0;
        p.off_xn = off;
    } else {
        off = NS * unit_bytes;
        p.off_xring = off;
        off += NS * p.xstage_bytes;
        p.off_xn = off;
        off += xn;
    }
    p.off_scratch = off;
    off += scratch;
    p.off_tile = off;
    off += tile;
    p.off_misc = off;
    off += misc;
    p.off_bars = off;
    // stage barriers, tile barriers, flags (+ the TMEM address)
    off += mma ? 24 * NS + 64 : 16 * NS + 32 + 16;
    if (off > dev.smem_optin) return CFA_ERR_UNSUPPORTED;
    p.nstages = NS;
    p.timeout_ns = kTimeoutNs;

    // The attribute is per kernel and shared by every plan: set the device limit.
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dev.smem_optin) != cudaSuccess) {
        cudaGetLastError();
        return CFA_ERR_CUDA;
    }
    int resident = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kernel, threads, off) != cudaSuccess ||
        resident < 1) {
        cudaGetLastError();
        return CFA_ERR_UNSUPPORTED;
    }
    if (mma) {
        // The occupancy calculator answers one block per SM for the tensor-core
        // kernels whatever their size; two of the smaller ones do fit and run
        // together (measured: the down GEMV at B = 4 takes 57 instead of 64 µs).
        // Count what the SM holds instead: registers, shared memory, threads.
        cudaFuncAttributes fa{};
        if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) {
            cudaGetLastError();
            return CFA_ERR_CUDA;
        }
        const int warps = threads / 32;
        const int regs_per_warp = ((fa.numRegs * 32 + 255) / 256) * 256;
        const int by_regs = 65536 / (regs_per_warp * warps);
        const int by_smem = dev.smem_per_sm / (off + dev.smem_reserved);
        resident = std::max(1, std::min(by_regs, std::min(by_smem, 2048 / threads)));
    }
    // One persistent wave; every block owns an equal share of the units.
    p.nblocks = std::min(p.units, dev.sms * std::min(resident, bps));
    const int per_block = (p.units + p.nblocks - 1) / p.nblocks;
    p.max_tiles = (per_block + p.chunks - 1) / p.chunks + 1;
    out->gp = p;
    out->kernel = kernel;
    out->smem = off;
    out->threads = threads;
    out->mma = mma;
    out->resident = resident;
    out->partial_floats = static_cast<size_t>(p.nblocks) * p.max_tiles * B * NW;
    return CFA_OK;
}

// Tensor map of a GEMV weight W [K rows][N cols] for plan g: [rows x 128]
// boxes on the CUDA cores, [64 x 64] 128-byte-swizzled boxes on the tensor cores.
cfa_status gemv_map_w(const GemvPlan &g, CUtensorMap *tm, const void *W, int N, int K) {
    return g.mma ? cfa::encode_bf16_2d_ex(tm, W, N, K, N, 64, cfa::kGemvMmaRows, true)
                 : cfa::encode_bf16_2d(tm, W, N, K, cfa::kGemvTileCols, g.gp.rows);
}

// Tensor map of a GEMV's input rows x [B][stride] (first K of each) for plan
// g: [B x rows] boxes, or [16 x 64] swizzled boxes (rows past B read as zero).
cfa_status gemv_map_x(const GemvPlan &g, CUtensorMap *tm, const void *x, int K, int B, int stride) {
    return g.mma ? cfa::encode_bf16_2d_ex(tm, x, K, B, stride, 64, cfa::kMmaN, true)
                 : cfa::encode_bf16_2d_ex(tm, x, K, B, stride, g.gp.rows, B, false);
}

cfa_status launch_gemv(const GemvPlan &g, const GemvParams &p, const CUtensorMap *w0,
                       const CUtensorMap *w1, const CUtensorMap *x, cudaStream_t stream) {
    CUtensorMap m0 = *w0, m1 = *w1, mx = *x;
    GemvParams pp = p;
    void *args[4] = {&m0, &m1, &mx, &pp};
    return launch_pdl(g.kernel, dim3(p.nblocks), dim3(g.threads), static_cast<size_t>(g.smem),
                      stream, args);
}

}  // namespace

// ----------------------------------------------------------------------- MLP

struct cfa_mlp {
    int B = 0, H = 0, F = 0;
    Device dev;
    GemvPlan gu, dn;              // gate/up (+ norm, SwiGLU) and down (+ residual)
    int bps_req = 0, ns_req = 0;  // pipeline overrides (0: automatic)
    int path = -1;                // kGemvPath*: CUDA cores, tensor cores or by batch
    uint16_t *u = nullptr;        // [B][F] SwiGLU output
    float *partials = nullptr;    // gate/up partials, then down partials
    size_t partial_cap = 0;       // floats allocated
    unsigned *words = nullptr;    // gate/up counters, down counters, status word
    CUtensorMap tm_u;             // down projection's input rows
    // tensor maps cached by source pointer for cfa_mlp_step
    CUtensorMap tm_wg, tm_wu, tm_wd, tm_h;
    const void *src_wg = nullptr, *src_wu = nullptr, *src_wd = nullptr, *src_h = nullptr;
};

namespace {

unsigned *mlp_status_word(cfa_mlp *m) {
    return m->words + m->gu.gp.n_tiles + m->dn.gp.n_tiles;
}

cfa_status mlp_encode_weights(const cfa_mlp *m, const void *W_gate, const void *W_up,
                              const void *W_down, CUtensorMap *wg, CUtensorMap *wu,
                              CUtensorMap *wd) {
    if (gemv_map_w(m->gu, wg, W_gate, m->F, m->H) != CFA_OK ||
        gemv_map_w(m->gu, wu, W_up, m->F, m->H) != CFA_OK ||
        gemv_map_w(m->dn, wd, W_down, m->H, m->F) != CFA_OK)
        return CFA_ERR_CUDA;
    return CFA_OK;
}

cfa_status mlp_encode_input(const cfa_mlp *m, const void *h, CUtensorMap *tm) {
    return gemv_map_x(m->gu, tm, h, m->H, m->B, m->H);
}

// y = h + down(silu(gate(hn)) * up(hn)), hn = bf16(rmsnorm(h; norm_w)).
cfa_status mlp_launch(cfa_mlp *m, const CUtensorMap *wg, const CUtensorMap *wu,
                      const CUtensorMap *wd, const CUtensorMap *th, const void *h,
                      const void *norm_w, float eps, void *y, cudaStream_t stream) {
    unsigned *status = mlp_status_word(m);
    GemvParams a = m->gu.gp;
    a.x = static_cast<const uint16_t *>(h);
    a.norm_w = static_cast<const uint16_t *>(norm_w);
    a.y = m->u;
    a.partials = m->partials;
    a.counters = m->words;
    a.status = status;
    a.eps = eps;
    cfa_status st = launch_gemv(m->gu, a, wg, wu, th, stream);
    if (st != CFA_OK) return st;
    GemvParams d = m->dn.gp;
    d.x = m->u;
    d.resid = static_cast<const uint16_t *>(h);
    d.y = static_cast<uint16_t *>(y);
    d.partials = m->partials + m->gu.partial_floats;
    d.counters = m->words + m->gu.gp.n_tiles;
    d.status = status;
    return launch_gemv(m->dn, d, wd, wd, &m->tm_u, stream);
}

void mlp_free(cfa_mlp *m) {
    if (m->u) cudaFree(m->u);
    if (m->partials) cudaFree(m->partials);
    if (m->words) cudaFree(m->words);
    m->u = nullptr;
    m->partials = nullptr;
    m->words = nullptr;
}

// Rebuilds the MLP's two GEMV plans (the plan is unchanged on failure); the
// tensor maps depend on the kernel, so the cached ones are dropped.
cfa_status mlp_replan(cfa_mlp *m, int bps, int ns, int path) {
    GemvPlan gu, dn;
    cfa_status st = make_gemv(m->dev, cfa::kGemvSwiGLU, m->B, m->H, m->F, &gu, bps, ns, path);
    if (st == CFA_OK) st = make_gemv(m->dev, cfa::kGemvResidual, m->B, m->F, m->H, &dn, bps, ns, path);
    if (st != CFA_OK) return st;
    CUtensorMap tm_u;
    if (gemv_map_x(dn, &tm_u, m->u, m->F, m->B, m->F) != CFA_OK) return CFA_ERR_CUDA;
    const size_t need = gu.partial_floats + dn.partial_floats;
    if (need > m->partial_cap) {
        float *p = nullptr;
        if (cudaDeviceSynchronize() != cudaSuccess || cudaMalloc(&p, sizeof(float) * need) != cudaSuccess) {
            cudaGetLastError();
            return CFA_ERR_CUDA;
        }
        cudaFree(m->partials);
        m->partials = p;
        m->partial_cap = need;
    }
    // the counters keep their size: the tile counts do not depend on the kernel
    m->gu = gu;
    m->dn = dn;
    m->tm_u = tm_u;
    m->bps_req = bps;
    m->ns_req = ns;
    m->path = path;
    m->src_wg = m->src_wu = m->src_wd = m->src_h = nullptr;
    return CFA_OK;
}

// Reads and clears a device status word (synchronizes the device).
cfa_status read_status(unsigned *word) {
    unsigned v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&v, word, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(word, 0, sizeof v) != cudaSuccess) {
        cudaGetLastError();
        return CFA_ERR_CUDA;
    }
    if (v & cfa::kStatusTimeoutBit) return CFA_ERR_TIMEOUT;
    if (v & cfa::kStatusBadLengthBit) return CFA_ERR_INVALID_ARG;
    return CFA_OK;
}

}  // namespace

extern "C" {

cfa_status cfa_rmsnorm(int B, int n, const void *x, const void *g, float eps, void *y,
                       void *stream) {
    if (B < 1 || B > 65535 || n < 8 || n % 8 || n > (1 << 20) || !x || !g || !y ||
        !(eps >= 0.0f) || !std::isfinite(eps))
        return fail(CFA_ERR_INVALID_ARG);
    if (!aligned16(x) || !aligned16(g) || !aligned16(y)) return fail(CFA_ERR_ALIGNMENT);
    const size_t rows = 2u * static_cast<size_t>(B) * n;
    if (overlaps(y, rows, x, rows) || overlaps(y, rows, g, 2u * n)) return fail(CFA_ERR_INVALID_ARG);
    const cfa_status st = launch_rmsnorm(B, n, x, g, eps, y, static_cast<cudaStream_t>(stream));
    return st == CFA_OK ? CFA_OK : fail(st);
}

cfa_mlp *cfa_mlp_create(int B, int hidden, int ffn) {
    if (B < 1 || hidden < 1 || ffn < 1) {
        fail(CFA_ERR_INVALID_ARG);
        return nullptr;
    }
    if (B > cfa::kMaxBatch || hidden % 128 || hidden > (1 << 16) || ffn % 128 || ffn > (1 << 18)) {
        fail(CFA_ERR_UNSUPPORTED);
        return nullptr;
    }
    Device dev;
    cfa_status st = query_device(&dev);
    if (st != CFA_OK) {
        fail(st);
        return nullptr;
    }
    cfa_mlp *m = new (std::nothrow) cfa_mlp();
    if (!m) {
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    m->B = B;
    m->H = hidden;
    m->F = ffn;
    m->dev = dev;
    if ((st = make_gemv(dev, cfa::kGemvSwiGLU, B, hidden, ffn, &m->gu)) != CFA_OK ||
        (st = make_gemv(dev, cfa::kGemvResidual, B, ffn, hidden, &m->dn)) != CFA_OK) {
        delete m;
        fail(st);
        return nullptr;
    }
    const size_t nwords = static_cast<size_t>(m->gu.gp.n_tiles + m->dn.gp.n_tiles + 1);
    m->partial_cap = m->gu.partial_floats + m->dn.partial_floats;
    if (cudaMalloc(&m->u, 2u * static_cast<size_t>(B) * ffn) != cudaSuccess ||
        cudaMalloc(&m->partials, sizeof(float) * m->partial_cap) != cudaSuccess ||
        cudaMalloc(&m->words, sizeof(unsigned) * nwords) != cudaSuccess ||
        cudaMemset(m->words, 0, sizeof(unsigned) * nwords) != cudaSuccess) {
        cudaGetLastError();
        mlp_free(m);
        delete m;
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    if (gemv_map_x(m->dn, &m->tm_u, m->u, ffn, B, ffn) != CFA_OK) {
        mlp_free(m);
        delete m;
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    return m;
}

void cfa_mlp_destroy(cfa_mlp *m) {
    if (!m) return;
    cudaDeviceSynchronize();
    mlp_free(m);
    delete m;
}

cfa_status cfa_mlp_step(cfa_mlp *m, const void *h, const void *norm_w, float eps,
                        const void *W_gate, const void *W_up, const void *W_down, void *y,
                        void *stream) {
    if (!m || !h || !norm_w || !W_gate || !W_up || !W_down || !y || !(eps >= 0.0f) ||
        !std::isfinite(eps))
        return fail(CFA_ERR_INVALID_ARG);
    if (!aligned16(h) || !aligned16(norm_w) || !aligned16(W_gate) || !aligned16(W_up) ||
        !aligned16(W_down) || !aligned16(y))
        return fail(CFA_ERR_ALIGNMENT);
    const size_t act = 2u * static_cast<size_t>(m->B) * m->H;
    const size_t w = 2u * static_cast<size_t>(m->H) * m->F;
    if (overlaps(y, act, h, act) || overlaps(y, act, norm_w, 2u * m->H) ||
        overlaps(y, act, W_gate, w) || overlaps(y, act, W_up, w) || overlaps(y, act, W_down, w))
        return fail(CFA_ERR_INVALID_ARG);
    if (m->src_wg != W_gate || m->src_wu != W_up || m->src_wd != W_down) {
        m->src_wg = m->src_wu = m->src_wd = nullptr;
        if (mlp_encode_weights(m, W_gate, W_up, W_down, &m->tm_wg, &m->tm_wu, &m->tm_wd) != CFA_OK)
            return fail(CFA_ERR_CUDA);
        m->src_wg = W_gate;
        m->src_wu = W_up;
        m->src_wd = W_down;
    }
    if (m->src_h != h) {
        m->src_h = nullptr;
        if (mlp_encode_input(m, h, &m->tm_h) != CFA_OK) return fail(CFA_ERR_CUDA);
        m->src_h = h;
    }
    const cfa_status st = mlp_launch(m, &m->tm_wg, &m->tm_wu, &m->tm_wd, &m->tm_h, h, norm_w, eps,
                                     y, static_cast<cudaStream_t>(stream));
    return st == CFA_OK ? CFA_OK : fail(st);
}

cfa_status cfa_mlp_set_pipeline(cfa_mlp *m, int blocks_per_sm, int stages) {
    if (!m || blocks_per_sm < 0 || blocks_per_sm > 4 || stages < 0 || stages > kMaxGemvStages)
        return fail(CFA_ERR_INVALID_ARG);
    const cfa_status st = mlp_replan(m, blocks_per_sm, stages, m->path);
    return st == CFA_OK ? CFA_OK : fail(st);
}

cfa_status cfa_mlp_set_path(cfa_mlp *m, int path) {
    if (!m || path < kGemvPathAuto || path > kGemvPathTensorCores) return fail(CFA_ERR_INVALID_ARG);
    const cfa_status st = mlp_replan(m, m->bps_req, m->ns_req, path);
    return st == CFA_OK ? CFA_OK : fail(st);
}

cfa_status cfa_mlp_status(cfa_mlp *m) {
    if (!m) return fail(CFA_ERR_INVALID_ARG);
    const cfa_status st = read_status(mlp_status_word(m));
    return st == CFA_OK ? CFA_OK : fail(st);
}

cfa_status cfa_mlp_describe(const cfa_mlp *m, char *buf, int len) {
    if (!m || !buf || len < 1) return fail(CFA_ERR_INVALID_ARG);
    const GemvParams &a = m->gu.gp, &d = m->dn.gp;
    std::snprintf(buf, static_cast<size_t>(len),
                  "{\"B\": %d, \"hidden\": %d, \"ffn\": %d, \"tensor_cores\": %s, "
                  "\"gate_up\": {\"grid\": %d, \"units\": %d, \"rows_per_unit\": %d, "
                  "\"stages\": %d, \"smem_bytes\": %d, \"resident_per_sm\": %d}, "
                  "\"down\": {\"grid\": %d, \"units\": %d, \"rows_per_unit\": %d, "
                  "\"stages\": %d, \"smem_bytes\": %d, \"resident_per_sm\": %d}}",
                  m->B, m->H, m->F, m->gu.mma ? "true" : "false", a.nblocks, a.units, a.rows, a.nstages,
                  m->gu.smem, m->gu.resident, d.nblocks, d.units, d.rows, d.nstages, m->dn.smem,
                  m->dn.resident);
    return CFA_OK;
}

}  // extern "C"

// --------------------------------------------------------------------- stack

namespace {

struct StackLayer {
    const void *attn_norm = nullptr, *W_qkv = nullptr, *W_o = nullptr;
    const void *mlp_norm = nullptr, *W_gate = nullptr, *W_up = nullptr, *W_down = nullptr;
    void *k_cache = nullptr, *v_cache = nullptr;
    CUtensorMap tm_wqkv, tm_wo, tm_wg, tm_wu, tm_wd;
    bool set = false;
};

struct GraphKey {
    const void *x = nullptr;
    void *out = nullptr;
    int *pos = nullptr;
    double theta = 0.0;
    float eps = 0.0f;
    int advance = 0;
    cudaStream_t stream = nullptr;
    unsigned version = 0;
    bool operator==(const GraphKey &o) const {
        return x == o.x && out == o.out && pos == o.pos && theta == o.theta && eps == o.eps &&
               advance == o.advance && stream == o.stream && version == o.version;
    }
};

}  // namespace

struct cfa_stack {
    int L = 0, B = 0, H = 0, nh = 0, D = 0, F = 0, max_ctx = 0;
    cfa_plan *attn = nullptr;
    cfa_mlp *mlp = nullptr;
    std::vector<StackLayer> layers;
    uint16_t *xn = nullptr;   // [B][H] normalized attention input
    uint16_t *h = nullptr;    // [B][H] residual stream after attention
    uint16_t *xr = nullptr;   // [B][H] residual stream between layers
    CUtensorMap tm_xn, tm_h;
    unsigned version = 1;     // bumped whenever a layer changes
    cudaGraphExec_t exec = nullptr;
    GraphKey key;
};

namespace {

void stack_free(cfa_stack *s) {
    if (s->exec) cudaGraphExecDestroy(s->exec);
    s->exec = nullptr;
    if (s->attn) cfa_plan_destroy(s->attn);
    if (s->mlp) cfa_mlp_destroy(s->mlp);
    s->attn = nullptr;
    s->mlp = nullptr;
    if (s->xn) cudaFree(s->xn);
    if (s->h) cudaFree(s->h);
    if (s->xr) cudaFree(s->xr);
    s->xn = s->h = s->xr = nullptr;
}

cfa_status stack_check(const cfa_stack *s, const void *x, int *positions, double rope_theta,
                       float eps, void *out) {
    if (!s || !x || !positions || !out || !(eps >= 0.0f) || !std::isfinite(eps) ||
        !(rope_theta >= 0.0) || rope_theta > 1e30)
        return CFA_ERR_INVALID_ARG;
    for (const StackLayer &l : s->layers)
        if (!l.set) return CFA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || (reinterpret_cast<uintptr_t>(positions) & 3u))
        return CFA_ERR_ALIGNMENT;
    const size_t act = 2u * static_cast<size_t>(s->B) * s->H;
    if (overlaps(positions, sizeof(int) * s->B, out, act) ||
        overlaps(positions, sizeof(int) * s->B, x, act))
        return CFA_ERR_INVALID_ARG;
    return CFA_OK;
}

// Every kernel of one token, in stream order. x and out may be the same
// buffer: x is consumed by the first layer before the last layer writes out.
cfa_status stack_enqueue(cfa_stack *s, const void *x, int *positions, double rope_theta, float eps,
                         int advance, void *out, cudaStream_t stream) {
    const void *cur = x;
    for (int l = 0; l < s->L; ++l) {
        const StackLayer &ly = s->layers[l];
        cfa_status st = launch_rmsnorm(s->B, s->H, cur, ly.attn_norm, eps, s->xn, stream);
        if (st != CFA_OK) return st;
        st = cfa::plan_launch_layer(s->attn, &ly.tm_wqkv, &ly.tm_wo, &s->tm_xn, s->xn, ly.k_cache,
                                    ly.v_cache, positions, rope_theta, cur, s->h, stream);
        if (st != CFA_OK) return st;
        void *next = l == s->L - 1 ? out : s->xr;
        st = mlp_launch(s->mlp, &ly.tm_wg, &ly.tm_wu, &ly.tm_wd, &s->tm_h, s->h, ly.mlp_norm, eps,
                        next, stream);
        if (st != CFA_OK) return st;
        cur = next;
    }
    if (advance) {
        int B = s->B;
        void *args[2] = {&positions, &B};
        return launch_pdl(cfa::advance_kernel_ptr(), dim3(1), dim3(32), 0, stream, args);
    }
    return CFA_OK;
}

}  // namespace

extern "C" {

cfa_stack *cfa_stack_create(int n_layers, int B, int hidden, int n_heads, int head_dim, int ffn,
                            int max_ctx) {
    if (n_layers < 1 || n_layers > 4096 || B < 1 || hidden < 1 || n_heads < 1 ||
        head_dim < 1 || ffn < 1 || max_ctx < 1 ||
        static_cast<long long>(n_heads) * head_dim != hidden) {
        fail(CFA_ERR_INVALID_ARG);
        return nullptr;
    }
    cfa_stack *s = new (std::nothrow) cfa_stack();
    if (!s) {
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    s->L = n_layers;
    s->B = B;
    s->H = hidden;
    s->nh = n_heads;
    s->D = head_dim;
    s->F = ffn;
    s->max_ctx = max_ctx;
    s->attn = cfa_plan_create(B, hidden, n_heads, head_dim, max_ctx);
    if (!s->attn) {
        const cfa_status st = cfa_last_error();
        delete s;
        fail(st);
        return nullptr;
    }
    s->mlp = cfa_mlp_create(B, hidden, ffn);
    if (!s->mlp) {
        const cfa_status st = cfa_last_error();
        stack_free(s);
        delete s;
        fail(st);
        return nullptr;
    }
    const size_t act = 2u * static_cast<size_t>(B) * hidden;
    if (cudaMalloc(&s->xn, act) != cudaSuccess || cudaMalloc(&s->h, act) != cudaSuccess ||
        cudaMalloc(&s->xr, act) != cudaSuccess) {
        cudaGetLastError();
        stack_free(s);
        delete s;
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    if (cfa::plan_encode_input(s->attn, s->xn, &s->tm_xn) != CFA_OK ||
        mlp_encode_input(s->mlp, s->h, &s->tm_h) != CFA_OK) {
        stack_free(s);
        delete s;
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    s->layers.resize(static_cast<size_t>(n_layers));
    return s;
}

void cfa_stack_destroy(cfa_stack *s) {
    if (!s) return;
    cudaDeviceSynchronize();
    stack_free(s);
    delete s;
}

cfa_status cfa_stack_set_layer(cfa_stack *s, int layer, const void *attn_norm, const void *W_qkv,
                               const void *W_o, void *k_cache, void *v_cache,
                               const void *mlp_norm, const void *W_gate, const void *W_up,
                               const void *W_down) {
    if (!s || layer < 0 || layer >= s->L || !attn_norm || !W_qkv || !W_o || !k_cache ||
        !v_cache || !mlp_norm || !W_gate || !W_up || !W_down)
        return fail(CFA_ERR_INVALID_ARG);
    const void *ptrs[9] = {attn_norm, W_qkv, W_o, k_cache, v_cache, mlp_norm, W_gate, W_up, W_down};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(CFA_ERR_ALIGNMENT);
    StackLayer ly;
    if (cfa::plan_encode_layer(s->attn, W_qkv, W_o, &ly.tm_wqkv, &ly.tm_wo) != CFA_OK ||
        mlp_encode_weights(s->mlp, W_gate, W_up, W_down, &ly.tm_wg, &ly.tm_wu, &ly.tm_wd) != CFA_OK)
        return fail(CFA_ERR_CUDA);
    ly.attn_norm = attn_norm;
    ly.W_qkv = W_qkv;
    ly.W_o = W_o;
    ly.k_cache = k_cache;
    ly.v_cache = v_cache;
    ly.mlp_norm = mlp_norm;
    ly.W_gate = W_gate;
    ly.W_up = W_up;
    ly.W_down = W_down;
    ly.set = true;
    s->layers[static_cast<size_t>(layer)] = ly;
    ++s->version;
    return CFA_OK;
}

cfa_status cfa_stack_step(cfa_stack *s, const void *x, int *positions, double rope_theta,
                          float eps, int advance, void *out, void *stream) {
    cfa_status st = stack_check(s, x, positions, rope_theta, eps, out);
    if (st != CFA_OK) return fail(st);
    st = stack_enqueue(s, x, positions, rope_theta, eps, advance, out,
                       static_cast<cudaStream_t>(stream));
    return st == CFA_OK ? CFA_OK : fail(st);
}

cfa_status cfa_stack_step_graph(cfa_stack *s, const void *x, int *positions, double rope_theta,
                                float eps, int advance, void *out, void *stream) {
    cfa_status st = stack_check(s, x, positions, rope_theta, eps, out);
    if (st != CFA_OK) return fail(st);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    if (!cs) return fail(CFA_ERR_INVALID_ARG);  // the legacy default stream cannot be captured
    GraphKey k;
    k.x = x;
    k.out = out;
    k.pos = positions;
    k.theta = rope_theta;
    k.eps = eps;
    k.advance = advance ? 1 : 0;
    k.stream = cs;
    k.version = s->version;
    if (!s->exec || !(s->key == k)) {
        if (s->exec) {
            cudaGraphExecDestroy(s->exec);
            s->exec = nullptr;
        }
        if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
            cudaGetLastError();
            return fail(CFA_ERR_CUDA);
        }
        st = stack_enqueue(s, x, positions, rope_theta, eps, k.advance, out, cs);
        cudaGraph_t graph = nullptr;
        const cudaError_t end = cudaStreamEndCapture(cs, &graph);
        if (st != CFA_OK || end != cudaSuccess || !graph) {
            cudaGetLastError();
            if (graph) cudaGraphDestroy(graph);
            return fail(st != CFA_OK ? st : CFA_ERR_CUDA);
        }
        const cudaError_t inst = cudaGraphInstantiate(&s->exec, graph, 0);
        cudaGraphDestroy(graph);
        if (inst != cudaSuccess) {
            cudaGetLastError();
            s->exec = nullptr;
            return fail(CFA_ERR_CUDA);
        }
        s->key = k;
    }
    if (cudaGraphLaunch(s->exec, cs) != cudaSuccess) {
        cudaGetLastError();
        return fail(CFA_ERR_CUDA);
    }
    return CFA_OK;
}

cfa_status cfa_stack_status(cfa_stack *s) {
    if (!s) return fail(CFA_ERR_INVALID_ARG);
    const cfa_status a = cfa_plan_status(s->attn);
    const cfa_status m = cfa_mlp_status(s->mlp);
    if (a != CFA_OK) return fail(a);
    return m == CFA_OK ? CFA_OK : fail(m);
}

cfa_status cfa_stack_describe(const cfa_stack *s, char *buf, int len) {
    if (!s || !buf || len < 64) return fail(CFA_ERR_INVALID_ARG);
    char a[512], m[512];
    if (cfa_plan_describe(s->attn, a, sizeof a) != CFA_OK ||
        cfa_mlp_describe(s->mlp, m, sizeof m) != CFA_OK)
        return fail(CFA_ERR_INVALID_ARG);
    std::snprintf(buf, static_cast<size_t>(len),
                  "{\"n_layers\": %d, \"launches_per_token\": %d, \"attention\": %s, \"mlp\": %s}",
                  s->L, (3 + cfa::plan_launches_per_step(s->attn)) * s->L, a, m);
    return CFA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------- MLA

struct cfa_mla {
    int B = 0, H = 0, nh = 0, q_lora = 0, max_ctx = 0;
    Device dev;
    GemvPlan ga, gq, go;          // x.W_a, norm(cq).W_uq, v.W_o
    uint16_t *a = nullptr;        // [B][q_lora + 576]
    uint16_t *q = nullptr;        // [B][nh*192]
    uint16_t *v = nullptr;        // [B][nh*128]
    float *partials = nullptr;
    unsigned *words = nullptr;    // counters of the three GEMVs, GEMV status, kernel status
    float *vpart = nullptr;       // per-split v records when the rows are split across clusters
    unsigned *vcount = nullptr;   // their arrival counters
    CUtensorMap tm_aq, tm_v;      // inputs of the q and output GEMVs (fixed buffers)
    cfa::MlaParams mp{};
    int smem = 0;
    int coresident_clusters = 0;
    int fit_clusters[5] = {};     // clusters of C = 2, 4, 8, 16 blocks resident at once (0: no fit)
    int forced_splits = 0;        // cfa_mla_set_row_splits; 0: chosen per step
};

namespace {

constexpr int kMlaStages = 4;  // two-box (32 KB) stages of the latent ring

void mla_free(cfa_mla *m) {
    if (m->a) cudaFree(m->a);
    if (m->q) cudaFree(m->q);
    if (m->v) cudaFree(m->v);
    if (m->partials) cudaFree(m->partials);
    if (m->words) cudaFree(m->words);
    if (m->vpart) cudaFree(m->vpart);
    if (m->vcount) cudaFree(m->vcount);
    m->a = m->q = m->v = nullptr;
    m->partials = nullptr;
    m->words = nullptr;
    m->vpart = nullptr;
    m->vcount = nullptr;
}

constexpr int kMlaMaxSplits = 4;   // row splits per head group

// Shared memory of one attention block when a cluster has C blocks (HG / C
// heads each); sets C, HPB and the offsets in mp, returns the bytes.
int mla_layout(cfa::MlaParams &mp, int C) {
    const int HG = mp.HG;
    mp.C = C;
    mp.HPB = HG / C;
    int off = 0;
    mp.off_ring = off;                          // two-box stages (1024-aligned boxes)
    off += kMlaStages * cfa::kMlaStageBytes;
    mp.off_qb = off;                            // 9 swizzled [32 x 64] query atoms (hi, lo)
    off += cfa::kMlaBoxes * cfa::kMlaQAtomBytes;
    mp.off_pb = off;                            // P of two tiles: 2 x 2 atoms [16 heads x 64 rows]
    off += 4 * cfa::kMlaAtomBytes;
    mp.off_qt = off;                            // fp32 queries [HG][576], then
    mp.off_recv = off;                          // partials of my heads [HPB][C][516]
    off += align_up(std::max(HG * cfa::kMlaRow, mp.HPB * mp.C * (cfa::kMlaKv + 4)) * 4, 128);
    mp.off_newrow = off;
    off += align_up(cfa::kMlaRow * 2, 128);
    mp.off_stat = off;                          // m, l, 2 alpha, 2 x two [8][16] reductions, new row
    off += align_up(592 * 4, 128);
    mp.off_ofin = off;                          // combined latent outputs [HPB][512]
    off += align_up(mp.HPB * cfa::kMlaKv * 4, 128);
    mp.off_scr = off;
    off += align_up((cfa::kComputeWarps * cfa::kMlaV + 64) * 4, 128);
    mp.off_bars = off;
    off += 16 * kMlaStages + 128;
    return off;
}

int mla_fit(const cfa_mla *m, int C) { return m->fit_clusters[__builtin_ctz(static_cast<unsigned>(C)) - 1]; }

// Cluster size C and row splits S for a step whose longest sequence holds
// max_len cached rows: of the shapes whose grid fits on the GPU at once, the
// one with the least estimated attention-kernel time, 4.5 µs per head a block
// finishes (absorption, combine, W_v projection) + 3.5 µs per 128-row tile of
// its rows (the tile loop is bound by tensor-core instruction issue); both
// figures measured on GB300 at the DeepSeek-V3 shape. Ties: the larger C,
// then the fewer splits.
void mla_choose(cfa_mla *m, int max_len) {
    const int HG = m->mp.HG, n_groups = m->B * (m->nh / HG);
    int best_c = 0, best_s = 1;
    double best = 0.0;
    for (int C = HG; C >= 2; C /= 2) {
        if (mla_fit(m, C) < 1) continue;
        for (int S = 1; S <= kMlaMaxSplits; S *= 2) {
            if (mla_fit(m, C) < n_groups * S) break;
            const double rows = std::ceil((max_len + 1.0) / (C * S));
            const double cost = 4.5 * (HG / C) + 3.5 * std::ceil(rows / cfa::kMlaTileRows);
            if (!best_c || cost < best - 1e-9) {
                best = cost;
                best_c = C;
                best_s = S;
            }
        }
    }
    if (!best_c) return;  // keep the plan's configuration (a grid larger than one wave)
    if (best_c != m->mp.C) {
        m->smem = mla_layout(m->mp, best_c);
        m->coresident_clusters = mla_fit(m, best_c);
    }
    m->mp.S = best_s;
}

unsigned *mla_gemv_status(cfa_mla *m) {
    return m->words + m->ga.gp.n_tiles + m->gq.gp.n_tiles + m->go.gp.n_tiles;
}

GemvParams gemv_params(const GemvPlan &g, const void *x, const void *norm_w, const void *resid,
                       void *y, float *partials, unsigned *counters, unsigned *status, float eps) {
    GemvParams p = g.gp;
    p.x = static_cast<const uint16_t *>(x);
    p.norm_w = static_cast<const uint16_t *>(norm_w);
    p.resid = static_cast<const uint16_t *>(resid);
    p.y = static_cast<uint16_t *>(y);
    p.partials = partials;
    p.counters = counters;
    p.status = status;
    p.eps = eps;
    return p;
}

}  // namespace

extern "C" {

cfa_mla *cfa_mla_create(int B, int hidden, int n_heads, int q_lora, int max_ctx) {
    if (B < 1 || hidden < 1 || n_heads < 1 || q_lora < 1 || max_ctx < 1) {
        fail(CFA_ERR_INVALID_ARG);
        return nullptr;
    }
    int HG = 1;
    while (HG < cfa::kMlaMaxHG && n_heads % (2 * HG) == 0) HG *= 2;
    if (B > cfa::kMaxBatch || hidden % 64 || hidden > (1 << 16) || q_lora % 64 ||
        q_lora > (1 << 14) || HG < 2 || max_ctx > (1 << 22) || n_heads > 4096) {
        fail(CFA_ERR_UNSUPPORTED);
        return nullptr;
    }
    Device dev;
    cfa_status st = query_device(&dev);
    if (st != CFA_OK) {
        fail(st);
        return nullptr;
    }
    cfa_mla *m = new (std::nothrow) cfa_mla();
    if (!m) {
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    m->B = B;
    m->H = hidden;
    m->nh = n_heads;
    m->q_lora = q_lora;
    m->max_ctx = max_ctx;
    m->dev = dev;
    const int NA = q_lora + cfa::kMlaRow, NQ = n_heads * cfa::kMlaQk, NV = n_heads * cfa::kMlaV;
    if ((st = make_gemv(dev, cfa::kGemvPlain, B, hidden, NA, &m->ga)) != CFA_OK ||
        (st = make_gemv(dev, cfa::kGemvNormPlain, B, q_lora, NQ, &m->gq)) != CFA_OK ||
        (st = make_gemv(dev, cfa::kGemvPlain, B, NV, hidden, &m->go)) != CFA_OK) {
        delete m;
        fail(st);
        return nullptr;
    }
    m->gq.gp.x_stride = NA;  // the query GEMV reads the first q_lora columns of a

    // The attention kernel: one cluster of C blocks per (sequence, group of HG
    // heads); each block gathers and finishes HG / C heads.
    cfa::MlaParams &mp = m->mp;
    mp.B = B;
    mp.nh = n_heads;
    mp.max_ctx = max_ctx;
    mp.a_stride = NA;
    mp.a_off = q_lora;
    mp.HG = HG;
    mp.nstages = kMlaStages;
    mp.qscale = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(cfa::kMlaQk)));
    mp.timeout_ns = kTimeoutNs;
    auto layout = [&](int C) { return mla_layout(mp, C); };
    const void *kernel = cfa::mla_kernel_ptr(HG);
    if (!kernel ||
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.smem_optin) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
        cudaGetLastError();
        delete m;
        fail(CFA_ERR_UNSUPPORTED);
        return nullptr;
    }
    // How many clusters of each size C (blocks per head group, each finishing
    // HG / C heads) fit on the GPU at once; a 16-block cluster needs 16 SMs of
    // one GPC, and not every GPC has them. The shape of each step (C and the
    // row splits S) is chosen from these by mla_choose; the initial one is
    // that for a full cache, or, when no grid fits in one wave, the largest C
    // that runs at all, unsplit.
    {
        const int n_groups = B * (n_heads / HG);
        int fallback = 0;
        for (int C = HG; C >= 2; C /= 2) {
            if (layout(C) > dev.smem_optin) continue;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = C;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(n_groups * C);
            cfg.blockDim = dim3(cfa::kMlaThreads);
            cfg.dynamicSmemBytes = static_cast<size_t>(layout(C));
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
                cudaGetLastError();
                continue;
            }
            if (clusters < 1) continue;
            m->fit_clusters[__builtin_ctz(static_cast<unsigned>(C)) - 1] = clusters;
            if (!fallback) fallback = C;
        }
        if (!fallback) {
            delete m;
            fail(CFA_ERR_UNSUPPORTED);
            return nullptr;
        }
        m->smem = layout(fallback);
        m->coresident_clusters = mla_fit(m, fallback);
        mp.S = 1;
        mla_choose(m, max_ctx - 1);
    }

    const size_t nwords = static_cast<size_t>(m->ga.gp.n_tiles + m->gq.gp.n_tiles +
                                              m->go.gp.n_tiles + 2);
    const size_t pf = std::max(m->ga.partial_floats, std::max(m->gq.partial_floats, m->go.partial_floats));
    if (cudaMalloc(&m->a, 2u * static_cast<size_t>(B) * NA) != cudaSuccess ||
        cudaMalloc(&m->q, 2u * static_cast<size_t>(B) * NQ) != cudaSuccess ||
        cudaMalloc(&m->v, 2u * static_cast<size_t>(B) * NV) != cudaSuccess ||
        cudaMalloc(&m->partials, sizeof(float) * pf) != cudaSuccess ||
        cudaMalloc(&m->words, sizeof(unsigned) * nwords) != cudaSuccess ||
        cudaMemset(m->words, 0, sizeof(unsigned) * nwords) != cudaSuccess ||
        cudaMalloc(&m->vpart, sizeof(float) * static_cast<size_t>(B) * n_heads * kMlaMaxSplits *
                                  cfa::kMlaSplitRec) != cudaSuccess ||
        cudaMalloc(&m->vcount, sizeof(unsigned) * static_cast<size_t>(B) * n_heads) != cudaSuccess ||
        cudaMemset(m->vcount, 0, sizeof(unsigned) * static_cast<size_t>(B) * n_heads) != cudaSuccess) {
        cudaGetLastError();
        mla_free(m);
        delete m;
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    if (gemv_map_x(m->gq, &m->tm_aq, m->a, q_lora, B, NA) != CFA_OK ||
        gemv_map_x(m->go, &m->tm_v, m->v, NV, B, NV) != CFA_OK) {
        mla_free(m);
        delete m;
        fail(CFA_ERR_CUDA);
        return nullptr;
    }
    return m;
}

void cfa_mla_destroy(cfa_mla *m) {
    if (!m) return;
    cudaDeviceSynchronize();
    mla_free(m);
    delete m;
}

cfa_status cfa_mla_step(cfa_mla *m, const void *x, const void *W_a, const void *g_q,
                        const void *g_kv, const void *W_uq, const void *W_kvb, const void *W_o,
                        void *cache, const int *ctx_lens, double rope_theta, float eps, void *out,
                        void *stream) {
    if (!m || !x || !W_a || !g_q || !g_kv || !W_uq || !W_kvb || !W_o || !cache || !ctx_lens ||
        !out || !(eps >= 0.0f) || !std::isfinite(eps) || !(rope_theta >= 0.0) || rope_theta > 1e30)
        return fail(CFA_ERR_INVALID_ARG);
    for (int b = 0; b < m->B; ++b)
        if (ctx_lens[b] < 0 || ctx_lens[b] >= m->max_ctx) return fail(CFA_ERR_INVALID_ARG);
    const void *ptrs[9] = {x, W_a, g_q, g_kv, W_uq, W_kvb, W_o, cache, out};
    for (const void *ptr : ptrs)
        if (!aligned16(ptr)) return fail(CFA_ERR_ALIGNMENT);
    const size_t act = 2u * static_cast<size_t>(m->B) * m->H;
    const size_t cache_bytes = 2u * static_cast<size_t>(m->B) * m->max_ctx * cfa::kMlaRow;
    if (overlaps(out, act, x, act) || overlaps(out, act, cache, cache_bytes) ||
        overlaps(out, act, W_o, 2u * static_cast<size_t>(m->nh) * cfa::kMlaV * m->H))
        return fail(CFA_ERR_INVALID_ARG);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const int NA = m->q_lora + cfa::kMlaRow, NQ = m->nh * cfa::kMlaQk, NV = m->nh * cfa::kMlaV;

    // tensor maps of this call's operands (host work only)
    CUtensorMap tm_x, tm_wa, tm_wuq, tm_wo, tm_wkvb;
    cfa::MlaMaps maps;
    std::memset(&maps, 0, sizeof maps);
    bool enc_ok =
        gemv_map_x(m->ga, &tm_x, x, m->H, m->B, m->H) == CFA_OK &&
        gemv_map_w(m->ga, &tm_wa, W_a, NA, m->H) == CFA_OK &&
        gemv_map_w(m->gq, &tm_wuq, W_uq, NQ, m->q_lora) == CFA_OK &&
        gemv_map_w(m->go, &tm_wo, W_o, m->H, NV) == CFA_OK &&
        cfa::encode_bf16_2d_ex(&tm_wkvb, W_kvb, static_cast<uint64_t>(m->nh) * 256, cfa::kMlaKv,
                               static_cast<uint64_t>(m->nh) * 256, 64, cfa::kMlaWeightRows, true) == CFA_OK;
    // one map per sequence over its cached rows only: a tile running past
    // them reads zeros (never another row or a NaN-filled tail)
    for (int b = 0; b < m->B && enc_ok; ++b) {
        const uint16_t *base = static_cast<const uint16_t *>(cache) +
                               static_cast<size_t>(b) * m->max_ctx * cfa::kMlaRow;
        enc_ok = cfa::encode_bf16_2d_ex(&maps.cache[b], base, cfa::kMlaRow,
                                        std::max(ctx_lens[b], 1), cfa::kMlaRow, 64,
                                        cfa::kMlaTileRows, true) == CFA_OK;
    }
    if (!enc_ok)
        return fail(CFA_ERR_CUDA);

    unsigned *gst = mla_gemv_status(m);
    unsigned *ctr = m->words;
    // a = bf16(x . W_a)
    GemvParams pa = gemv_params(m->ga, x, nullptr, nullptr, m->a, m->partials, ctr, gst, eps);
    cfa_status st = launch_gemv(m->ga, pa, &tm_wa, &tm_wa, &tm_x, cs);
    if (st != CFA_OK) return fail(st);
    ctr += m->ga.gp.n_tiles;
    // q = bf16(bf16(rmsnorm(a[:, :q_lora]; g_q)) . W_uq)
    GemvParams pq = gemv_params(m->gq, m->a, g_q, nullptr, m->q, m->partials, ctr, gst, eps);
    if ((st = launch_gemv(m->gq, pq, &tm_wuq, &tm_wuq, &m->tm_aq, cs)) != CFA_OK) return fail(st);
    ctr += m->gq.gp.n_tiles;
    // v: the latent attention core
    if (!m->forced_splits) {
        int max_len = 0;
        for (int b = 0; b < m->B; ++b) max_len = std::max(max_len, ctx_lens[b]);
        mla_choose(m, max_len);
    }
    cfa::MlaParams mp = m->mp;
    mp.q = m->q;
    mp.a = m->a;
    mp.g_kv = static_cast<const uint16_t *>(g_kv);
    mp.W_kvb = static_cast<const uint16_t *>(W_kvb);
    mp.cache = static_cast<uint16_t *>(cache);
    mp.v = m->v;
    mp.vpart = m->vpart;
    mp.vcount = m->vcount;
    mp.status = gst + 1;
    mp.eps = eps;
    for (int b = 0; b < m->B; ++b) mp.ctx_lens[b] = ctx_lens[b];
    mp.rope = rope_theta > 0.0 ? 1 : 0;
    for (int i = 0; i < cfa::kMlaRope / 2; ++i)
        mp.rope_inv_freq[i] = mp.rope ? std::pow(rope_theta, -2.0 * i / cfa::kMlaRope) : 0.0;
    {
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = mp.C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(m->B * (m->nh / mp.HG) * mp.S * mp.C);
        cfg.blockDim = dim3(cfa::kMlaThreads);
        cfg.dynamicSmemBytes = static_cast<size_t>(m->smem);
        cfg.stream = cs;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        void *args[3] = {&maps, &tm_wkvb, &mp};
        if (cudaLaunchKernelExC(&cfg, cfa::mla_kernel_ptr(mp.HG), args) != cudaSuccess) {
            cudaGetLastError();
            return fail(CFA_ERR_CUDA);
        }
    }
    // out = bf16(v . W_o)
    GemvParams po = gemv_params(m->go, m->v, nullptr, nullptr, out, m->partials, ctr, gst, eps);
    if ((st = launch_gemv(m->go, po, &tm_wo, &tm_wo, &m->tm_v, cs)) != CFA_OK) return fail(st);
    return CFA_OK;
}

cfa_status cfa_mla_set_row_splits(cfa_mla *m, int splits) {
    if (!m || splits < 0 || splits > kMlaMaxSplits || (splits & (splits - 1)))
        return fail(CFA_ERR_INVALID_ARG);
    if (splits == 0) {  // back to the per-step choice
        m->forced_splits = 0;
        return CFA_OK;
    }
    // the largest cluster size whose split grid is resident at once
    const int n_groups = m->B * (m->nh / m->mp.HG);
    int C = m->mp.HG;
    while (C >= 2 && m->fit_clusters[__builtin_ctz(static_cast<unsigned>(C)) - 1] < n_groups * splits) C /= 2;
    if (C < 2) return fail(CFA_ERR_UNSUPPORTED);
    cudaDeviceSynchronize();
    m->smem = mla_layout(m->mp, C);
    m->coresident_clusters = mla_fit(m, C);
    m->mp.S = splits;
    m->forced_splits = splits;
    return CFA_OK;
}

cfa_status cfa_mla_status(cfa_mla *m) {
    if (!m) return fail(CFA_ERR_INVALID_ARG);
    cfa_status a = read_status(mla_gemv_status(m));
    cfa_status b = read_status(mla_gemv_status(m) + 1);
    if (a != CFA_OK) return fail(a);
    return b == CFA_OK ? CFA_OK : fail(b);
}

cfa_status cfa_mla_describe(const cfa_mla *m, char *buf, int len) {
    if (!m || !buf || len < 1) return fail(CFA_ERR_INVALID_ARG);
    std::snprintf(buf, static_cast<size_t>(len),
                  "{\"B\": %d, \"hidden\": %d, \"n_heads\": %d, \"q_lora\": %d, \"max_ctx\": %d, "
                  "\"heads_per_cluster\": %d, \"cluster_size\": %d, \"row_splits\": %d, "
                  "\"grid\": %d, \"smem_bytes\": %d, \"stages\": %d, \"coresident_clusters\": %d, "
                  "\"gemv_grids\": [%d, %d, %d]}",
                  m->B, m->H, m->nh, m->q_lora, m->max_ctx, m->mp.HG, m->mp.C, m->mp.S,
                  m->B * (m->nh / m->mp.HG) * m->mp.S * m->mp.C, m->smem, m->mp.nstages,
                  m->coresident_clusters, m->ga.gp.nblocks, m->gq.gp.nblocks, m->go.gp.nblocks);
    return CFA_OK;
}

}  // extern "C"
