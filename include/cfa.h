/*
 * cfa.h -- C ABI of the cluster-fused decode-attention library (libcfa.so).
 *
 * One call runs one decode step of a decoder attention block for a batch of
 * B sequences on one GPU, in a single kernel launch:
 *
 *   1. QKV projection of the new token      qkv[b] = x[b] . W_qkv
 *   2. KV append                            k_cache[b,h,ctx_len] = k[b,h]
 *                                           v_cache[b,h,ctx_len] = v[b,h]
 *   3. single-query attention with a max-subtracted softmax over the
 *      ctx_len cached keys plus the new one (scale 1/sqrt(head_dim))
 *   4. output projection                    out[b] = concat_h(attn[b,h]) . W_o
 *
 * This is the decoder block of the page "ClusterFusion框架解析：LLM推理优化的集群
 * 通信革命" (ClusterFusion framework analysis): the three stages of its §1.1,
 * fused the way its §3.2 describes (one thread-block cluster per head, the
 * cluster's blocks splitting head_dim and the KV length, q/k/v shared by a
 * cluster gather and the softmax statistics and partial outputs combined by
 * cluster reductions over distributed shared memory, §3.1). The page merges
 * its partial output projections with atomicAdd; this library merges them in
 * a fixed head order instead, so results are bitwise reproducible.
 *
 * Conventions shared by every call:
 *   - All tensors are bf16 (IEEE binary32 with the low 16 bits dropped),
 *     dense, row-major, and live in device memory owned by the caller. All
 *     arithmetic accumulates in fp32. Results are rounded to bf16 with
 *     round-to-nearest-even.
 *   - Weights are [in, out] and applied as x . W (the page's
 *     torch.mm(hidden_states, W_qkv) form, §1.1):
 *       W_qkv [hidden, 3*hidden]: columns [0,H) are Q, [H,2H) K, [2H,3H) V;
 *                                 head h owns columns [h*d, (h+1)*d) of each.
 *       W_o   [hidden, hidden]:   row block [h*d, (h+1)*d) multiplies head h.
 *   - Caches are [B, n_heads, max_ctx, head_dim]. Positions [0, ctx_len) are
 *     read; position ctx_len is written; all other positions are neither read
 *     nor written.
 *   - Every device pointer must be 16-byte aligned. `out` must not overlap an
 *     input. ctx_len is shared by all B sequences.
 *   - Calls are asynchronous on the given CUDA stream (NULL = legacy default
 *     stream) unless stated otherwise. A plan owns a small device workspace,
 *     so one plan must not run concurrently on two streams; use one plan per
 *     stream.
 *   - Functions that return cfa_status never abort the process. Host-side
 *     argument checks happen before anything is launched; an error leaves
 *     every buffer untouched.
 *
 * Supported shapes: hidden == n_heads * head_dim, head_dim in {64, 128},
 * 1 <= B <= 16, hidden a multiple of 64, 1 <= max_ctx <= 1<<22. Other shapes
 * return CFA_ERR_UNSUPPORTED.
 */
#ifndef CFA_H
#define CFA_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cfa_plan cfa_plan; /* opaque */

typedef enum cfa_status {
    CFA_OK = 0,
    CFA_ERR_INVALID_ARG = 1, /* NULL plan or pointer, ctx_len out of range, ... */
    CFA_ERR_UNSUPPORTED = 2, /* a shape or cluster size this build does not run */
    CFA_ERR_CUDA = 3,        /* a CUDA runtime call failed (no device, launch, ...) */
    CFA_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up (see cfa_plan_status) */
    CFA_ERR_ALIGNMENT = 5    /* a pointer is not 16-byte aligned */
} cfa_status;

/*
 * Create a plan for batch B, hidden size `hidden` = n_heads * head_dim and a
 * cache capacity of max_ctx positions, on the current CUDA device.
 * Chooses the cluster size (blocks per head) and the pipeline depth: of the
 * sizes whose whole grid is resident on the GPU at once, the smallest whose
 * grid gives every SM a block, else the largest; if no size is co-resident,
 * the largest that runs. Sets the kernel attributes, and allocates the plan's workspace (fp32 per-head
 * output-projection partials [n_heads, B, hidden], arrival counters of the
 * cross-head merge, a status word, and device staging
 * for cfa_decode_step_host).
 * Returns NULL on failure; cfa_last_error() then says why.
 */
cfa_plan *cfa_plan_create(int B, int hidden, int n_heads, int head_dim, int max_ctx);

/* Release the plan and its workspace. Synchronizes the device first. NULL is a no-op. */
void cfa_plan_destroy(cfa_plan *plan);

/*
 * One decode step (steps 1-4 above), launched on `stream` (a cudaStream_t).
 *   x       bf16 [B, hidden]               read
 *   W_qkv   bf16 [hidden, 3*hidden]        read
 *   W_o     bf16 [hidden, hidden]          read
 *   k_cache bf16 [B, n_heads, max_ctx, head_dim]  rows [0,ctx_len) read, row ctx_len written
 *   v_cache bf16 [B, n_heads, max_ctx, head_dim]  same
 *   ctx_len number of cached positions before this token, 0 <= ctx_len < max_ctx
 *   out     bf16 [B, hidden]               written
 * Re-running a step with the same ctx_len rewrites the same cache row with
 * the same value, so a step is idempotent.
 * The step is one kernel launch, or two when the plan merges the heads'
 * partial output projections in a separate kernel (large batches; see
 * cfa_plan_describe).
 * Launch overlap (on by default, see cfa_plan_set_overlap): the step is
 * launched with programmatic stream serialization, so it may be scheduled
 * while the previous kernel on the stream is still running. Before that
 * kernel has finished it only initialises shared memory and prefetches
 * weight tiles; x and the caches are read, and every buffer is written, only
 * afterwards. The weights must therefore not be written by kernels still in
 * flight on the stream.
 * Errors: CFA_ERR_INVALID_ARG (NULL pointer, ctx_len out of range),
 * CFA_ERR_ALIGNMENT, CFA_ERR_CUDA (launch failure). Faults raised while the
 * kernel runs surface at the next synchronizing call, as with any CUDA kernel.
 */
cfa_status cfa_decode_step(cfa_plan *plan, const void *x, const void *W_qkv,
                           const void *W_o, void *k_cache, void *v_cache,
                           int ctx_len, void *out, void *stream);

/*
 * The decode step with one context length per sequence and, optionally, a
 * rotary position embedding of the new token's q and k. This widens the
 * page's block (which names no positional encoding, §1.1) toward a
 * Llama2-style layer:
 *   ctx_lens   host array [B]: cached positions of sequence b before this
 *              token, each in [0, max_ctx); row ctx_lens[b] of sequence b is
 *              written, rows [0, ctx_lens[b]) are read.
 *   rope_theta 0 disables the rotation; > 0 rotates dims i and i + d/2 of
 *              q and k_new by ctx_lens[b] * rope_theta^(-2i/d) (rotate-half
 *              form; e.g. 10000 for Llama2). Cached keys are taken as
 *              already rotated, and the appended k row is the rotated one.
 * Other arguments as cfa_decode_step, which equals this call with every
 * ctx_lens[b] = ctx_len and rope_theta = 0. Errors: CFA_ERR_INVALID_ARG
 * also for a NULL ctx_lens, a length out of range or a negative theta.
 */
cfa_status cfa_decode_step_ex(cfa_plan *plan, const void *x, const void *W_qkv,
                              const void *W_o, void *k_cache, void *v_cache,
                              const int *ctx_lens, double rope_theta, void *out,
                              void *stream);

/*
 * The same step for a caller whose token activations live in host memory:
 * takes x_host (bf16 [B, hidden]) to the GPU, runs the step of
 * cfa_decode_step on `stream`, brings the result back to out_host
 * (bf16 [B, hidden]) and synchronizes `stream` before returning. Weights and
 * caches stay device pointers. With page-locked, device-mapped host buffers
 * (cudaHostAlloc / cudaHostRegister, 16-byte aligned) there is no DMA
 * transfer: the step writes out_host itself, and reads x_host itself at
 * B <= 2 (at B >= 3 a small copy kernel first stages x in the plan's device
 * buffer, which the step's tensor-map loads read). Other host memory goes
 * through cudaMemcpyAsync and the plan's staging buffers, and is slower.
 * Errors as cfa_decode_step.
 */
cfa_status cfa_decode_step_host(cfa_plan *plan, const void *x_host, const void *W_qkv,
                                const void *W_o, void *k_cache, void *v_cache,
                                int ctx_len, void *out_host, void *stream);

/*
 * The same decode step for callers that cannot allocate device memory while
 * they run: engines whose device memory is owned and budgeted by a host
 * framework (plugins that receive only their input and output buffers), and
 * serving loops that forbid cudaMalloc after start-up because it may
 * synchronize the device and may fail under memory pressure. The paper has no
 * counterpart to this entry point; it exists only for such callers.
 *
 * No plan is involved: the shape is passed directly, with the same meaning,
 * limits and cluster-size choice as cfa_plan_create, and the arguments after
 * it mean what they mean for cfa_decode_step. Nothing is allocated: the
 * kernel's scratch (arrival counters, status word and the fp32 per-head
 * output-projection partials) lives in one fixed array inside the library,
 * 8 MiB + 16.25 KiB, which every GPU that loads the library keeps until the
 * process exits. Shapes with n_heads * B * hidden > 2^21 do not fit and
 * return CFA_ERR_UNSUPPORTED before anything is launched.
 *
 * The first call on a device sets the array up (looks up its device address
 * and zeroes its counters, synchronizing that device once); make that first
 * call before any stream capture. If that set-up fails (CFA_ERR_CUDA), the
 * device is not marked as set up and the next call tries again. Every call then clears the counters with an
 * asynchronous memset on `stream` and launches the kernel (and the separate
 * head merge, where the plan would use one) there, without launch overlap. All calls on a device share the one array, so calls whose
 * kernels may run at the same time on that device (other streams, other host
 * threads) race and must be serialized by the caller. Device-side wait
 * timeouts are not reported by this entry point.
 * Errors: as cfa_plan_create and cfa_decode_step.
 */
cfa_status cfa_decode_step_noalloc(int B, int hidden, int n_heads, int head_dim, int max_ctx,
                                   const void *x, const void *W_qkv, const void *W_o,
                                   void *k_cache, void *v_cache, int ctx_len, void *out,
                                   void *stream);

/*
 * Override the cluster size (thread blocks per head): 1, 2, 4, 8 or 16.
 * CFA_ERR_UNSUPPORTED if the shape does not split evenly at that size, the
 * device cannot co-schedule such a cluster, or its shared memory does not fit.
 * The plan is unchanged on error.
 */
cfa_status cfa_plan_set_cluster_size(cfa_plan *plan, int cluster_size);

/*
 * Override the pipeline depth (number of 16 KB shared-memory stages per
 * block); 0 restores the automatic choice. CFA_ERR_UNSUPPORTED if the shared
 * memory does not fit or the depth is outside [2, 64]. The plan is unchanged
 * on error.
 */
cfa_status cfa_plan_set_stages(cfa_plan *plan, int stages);

/*
 * How the blocks of a head's cluster share their partial q, k and v (the
 * ClusterGather step, CF section 3.1.2 "QKV向量共享"). mode 0: every block
 * sends its whole partial [B][3][64] to every peer and each sums all of them
 * (one round of pushes; the receive buffer holds C partials). mode 1:
 * reduce-scatter then all-gather -- each block sums one slice of the columns
 * over the blocks of its column group and sends the sum to every peer (two
 * rounds; the receive buffer holds 2 partials whatever C, which leaves more
 * shared memory for pipeline stages). Both sum in the same order, so the
 * results are bit for bit the same. mode -1 (the default): mode 1 where it
 * fits more blocks on an SM than mode 0, or, at the same blocks per SM,
 * gives more stages and either the batch runs its projections on the tensor
 * cores (B >= 3) or mode 0 leaves fewer than 4 stages; else mode 0.
 * CFA_ERR_INVALID_ARG for another mode; CFA_ERR_UNSUPPORTED if the layout
 * does not fit. The plan is unchanged on error.
 */
cfa_status cfa_plan_set_qkv_exchange(cfa_plan *plan, int mode);

/*
 * Enable (1, the default) or disable (0) launch overlap for the following
 * steps. With overlap on, a step's prologue and first weight loads run under
 * the tail of the previous kernel in the stream (see cfa_decode_step); with
 * it off, the step starts only after that kernel has finished.
 */
cfa_status cfa_plan_set_overlap(cfa_plan *plan, int enable);

/* Current cluster size of the plan, or -1 for NULL. */
int cfa_plan_cluster_size(const cfa_plan *plan);

/*
 * Write a one-line JSON description of the plan (shape, cluster size, grid,
 * block, shared memory per block, pipeline stages, stage bytes, co-resident
 * clusters, the form of the cross-head merge -- "flat": the last head to
 * finish a column chunk sums every head's partials inside the fused kernel;
 * "separate": a second kernel, launched behind it on the same stream, sums
 * them, chosen when the flat form would read more than 256 KB through one
 * block -- "launches_per_step", 1 or 2, and "qkv_exchange", "gather" or
 * "reduce_scatter") into buf (NUL-terminated, truncated to len).
 * CFA_ERR_INVALID_ARG for NULL arguments.
 */
cfa_status cfa_plan_describe(const cfa_plan *plan, char *buf, int len);

/*
 * The layout a plan of this shape would use with cluster size C on a device
 * with the given limits, computed on the host with no device, no allocation
 * and no CUDA call: the same arithmetic as cfa_plan_create and
 * cfa_plan_set_cluster_size after they have read the device's attributes
 * (num_sms = multiprocessor count; smem_per_sm, smem_optin, smem_reserved =
 * shared memory per multiprocessor, the per-block opt-in maximum and the
 * per-block reservation, in bytes). exchange and stages are as in
 * cfa_plan_set_qkv_exchange (-1 automatic) and cfa_plan_set_stages (0
 * automatic). C itself is the caller's: the plan's automatic choice also
 * needs the device's answer on how many clusters of each size fit at once.
 * Writes one JSON line into buf (len >= 256): cluster_size, grid,
 * blocks_per_sm (the blocks an SM is sized to hold), stages, smem_bytes,
 * qkv_exchange, tensor_cores (1: the projections run on tcgen05, B >= 3),
 * tmem_cols, proj_rows_per_block, proj_tile_rows, out_cols_per_block and
 * merge ("flat" or "separate"). Errors: shapes as cfa_plan_create;
 * CFA_ERR_INVALID_ARG for out-of-range limits, exchange, stages or buffer;
 * CFA_ERR_UNSUPPORTED when C does not divide the work or the layout does not
 * fit the shared memory.
 */
cfa_status cfa_plan_layout(int B, int hidden, int n_heads, int head_dim, int max_ctx, int C,
                           int exchange, int stages, int num_sms, int smem_per_sm,
                           int smem_optin, int smem_reserved, char *buf, int len);

/*
 * Device-side status of the plan: synchronizes the device, reads and clears
 * the status word the kernels set when a bounded wait gives up. CFA_OK when
 * nothing happened, CFA_ERR_TIMEOUT after a timed-out wait,
 * CFA_ERR_INVALID_ARG after a device-resident position out of range (layer
 * stack), CFA_ERR_CUDA if the read itself fails.
 */
cfa_status cfa_plan_status(cfa_plan *plan);

/* Status of the last failed call on this thread (plan creation included). */
cfa_status cfa_last_error(void);

/* Static, human-readable name of a status code. */
const char *cfa_status_string(cfa_status status);

/*
 * Self-test of the bounded-wait mechanism every in-kernel wait uses: launches
 * one block that waits on a shared-memory barrier nothing ever arrives on,
 * giving up after limit_us microseconds, then reports through a status word.
 * Synchronizes `stream`. Returns CFA_ERR_TIMEOUT when the wait gave up as it
 * must, CFA_OK if it (wrongly) completed, CFA_ERR_CUDA on a CUDA error.
 * limit_us must be in [1, 1<<20]. No GPU fault or hang is involved.
 */
cfa_status cfa_selftest_wait_timeout(int limit_us, void *stream);

/* ==========================================================================
 * Decoder layers around the attention block, and the multi-layer decode loop.
 *
 * The page reports time per output token of a whole Llama2-7B decoder
 * [§3.3, §5.1] but describes only the attention block of a layer (§1.1). The
 * rest of a layer follows the Llama2 arrangement (a reading, not the page):
 *
 *   xn = bf16( rmsnorm(x; attn_norm) )
 *   h  = bf16( x + attention_block(xn) )          (the fused step above)
 *   hn = bf16( rmsnorm(h; mlp_norm) )
 *   y  = bf16( h + (bf16(silu(hn . W_gate) * (hn . W_up))) . W_down )
 *
 * rmsnorm(v; g)_i = g_i v_i / sqrt(mean_j v_j^2 + eps), silu(z) = z/(1+e^-z).
 * Same conventions as above: bf16 row-major tensors in caller-owned device
 * memory, weights [in, out] applied as v . W, fp32 accumulation, 16-byte
 * aligned pointers, asynchronous on `stream`, fixed-order (bitwise
 * reproducible) reductions.
 * ========================================================================== */

typedef struct cfa_mlp cfa_mlp;     /* opaque */
typedef struct cfa_stack cfa_stack; /* opaque */

/*
 * y[b] = bf16(g * x[b] / sqrt(mean(x[b]^2) + eps)) for b < B; x, y [B, n],
 * g [n]. n a multiple of 8 in [8, 1<<20], B in [1, 65535], eps >= 0 finite;
 * y must not overlap x or g. CFA_ERR_INVALID_ARG / CFA_ERR_ALIGNMENT before
 * any launch, CFA_ERR_CUDA if the launch fails.
 */
cfa_status cfa_rmsnorm(int B, int n, const void *x, const void *g, float eps, void *y,
                       void *stream);

/*
 * Plan for the MLP half of a layer at batch B: hidden a multiple of 64
 * (<= 65536), ffn a multiple of 128 (<= 1<<18), 1 <= B <= 16
 * (CFA_ERR_UNSUPPORTED otherwise). Allocates the [B, ffn] SwiGLU buffer, the
 * fp32 split partials and arrival counters of its two GEMVs, and a status
 * word. NULL on failure; cfa_last_error() says why.
 */
cfa_mlp *cfa_mlp_create(int B, int hidden, int ffn);

/* Release the plan (synchronizes the device first). NULL is a no-op. */
void cfa_mlp_destroy(cfa_mlp *mlp);

/*
 * y = h + down(silu(gate(hn)) * up(hn)) with hn = bf16(rmsnorm(h; norm_w)):
 *   h, y [B, hidden]; norm_w [hidden]; W_gate, W_up [hidden, ffn];
 *   W_down [ffn, hidden].
 * Two kernel launches (RMSNorm + gate/up + SwiGLU; down + residual). y must
 * not overlap h, norm_w or a weight. One plan must not run on two streams at
 * once. Errors as cfa_rmsnorm.
 */
cfa_status cfa_mlp_step(cfa_mlp *mlp, const void *h, const void *norm_w, float eps,
                        const void *W_gate, const void *W_up, const void *W_down, void *y,
                        void *stream);

/*
 * Override the MLP kernels' occupancy (blocks per SM, 1..4) and pipeline depth
 * (16 KB stages per block, 2..12); 0 keeps the automatic choice. For sweeps.
 * CFA_ERR_UNSUPPORTED if it does not fit (the plan is then unchanged).
 */
cfa_status cfa_mlp_set_pipeline(cfa_mlp *mlp, int blocks_per_sm, int stages);

/*
 * Choose the kernel of the MLP's two GEMVs: path -1 = by batch size (the
 * tcgen05 tensor-core kernel from B = 2 on, the CUDA-core kernel at B = 1), 0 =
 * CUDA cores, 1 = tensor cores. The result is the same to within fp32
 * summation order. Keeps the pipeline overrides of cfa_mlp_set_pipeline.
 * CFA_ERR_INVALID_ARG for another path; CFA_ERR_UNSUPPORTED if the shape does
 * not fit the kernel (the plan is then unchanged).
 */
cfa_status cfa_mlp_set_path(cfa_mlp *mlp, int path);

/* Synchronizes, reads and clears the plan's device status word (as cfa_plan_status). */
cfa_status cfa_mlp_status(cfa_mlp *mlp);

/* One-line JSON description of the plan's two GEMVs (grid, units, stages, shared memory). */
cfa_status cfa_mlp_describe(const cfa_mlp *mlp, char *buf, int len);

/*
 * A stack of n_layers decoder layers (shapes as cfa_plan_create and
 * cfa_mlp_create) for the decode loop. Owns one attention plan, one MLP plan
 * and three [B, hidden] activation buffers; the layers' weights and caches
 * stay the caller's. NULL on failure; cfa_last_error() says why.
 */
cfa_stack *cfa_stack_create(int n_layers, int B, int hidden, int n_heads, int head_dim, int ffn,
                            int max_ctx);

/* Release the stack (synchronizes the device first). NULL is a no-op. */
void cfa_stack_destroy(cfa_stack *stack);

/*
 * Bind layer `layer` (0-based) to its weights and caches: attn_norm,
 * mlp_norm [hidden]; W_qkv [hidden, 3*hidden]; W_o [hidden, hidden]; caches
 * [B, n_heads, max_ctx, head_dim]; W_gate, W_up [hidden, ffn]; W_down
 * [ffn, hidden]. The pointers must stay valid while the stack is used.
 * Rebinding a layer invalidates a recorded graph (it is recorded again on
 * the next cfa_stack_step_graph).
 */
cfa_status cfa_stack_set_layer(cfa_stack *stack, int layer, const void *attn_norm,
                               const void *W_qkv, const void *W_o, void *k_cache, void *v_cache,
                               const void *mlp_norm, const void *W_gate, const void *W_up,
                               const void *W_down);

/*
 * One token through every layer: x [B, hidden] in, out [B, hidden] out (x and
 * out may be the same buffer). positions: device int [B], the cached length
 * of every sequence, read by each layer's attention kernel on the device
 * (so a recorded graph serves every position); each must lie in
 * [0, max_ctx - 1]. A value outside that range is not caught on the host: the
 * kernels flag it in the status word (cfa_stack_status then returns
 * CFA_ERR_INVALID_ARG), read no cache rows and append nothing for that
 * sequence. advance != 0 adds 1 to every position after the last layer (the
 * decode loop's next token). rope_theta > 0 rotates q and the new k as in
 * cfa_decode_step_ex; eps is the RMSNorm epsilon. All layers must be bound.
 * 4 kernels per layer (+1 with advance).
 */
cfa_status cfa_stack_step(cfa_stack *stack, const void *x, int *positions, double rope_theta,
                          float eps, int advance, void *out, void *stream);

/*
 * The same token step, recorded into a CUDA graph on the first call (and
 * again whenever x, out, positions, rope_theta, eps, advance, the stream or a
 * layer binding changes) and replayed with one graph launch afterwards.
 * `stream` must not be the legacy default stream (CFA_ERR_INVALID_ARG).
 */
cfa_status cfa_stack_step_graph(cfa_stack *stack, const void *x, int *positions,
                                double rope_theta, float eps, int advance, void *out,
                                void *stream);

/* Synchronizes and reads (and clears) the status of both plans of the stack. */
cfa_status cfa_stack_status(cfa_stack *stack);

/* One-line JSON description (layers, launches per token, both plans). */
cfa_status cfa_stack_describe(const cfa_stack *stack, char *buf, int len);

/* ==========================================================================
 * Multi-head latent attention (MLA), the DeepSeek variant the page adapts
 * ClusterFusion to: the latent key/value cache partitioned across clusters,
 * combined by a sparse cluster reduction (§5.2). The page gives no formula or
 * dimension; the block is DeepSeek-V2/V3's attention with their widths:
 * latent 512, per-head nope / rope / value 128 / 64 / 128 (fixed here).
 *
 * One step for B sequences at positions ctx_lens[b] (weights [in, out]):
 *   a   = bf16(x . W_a)                    W_a  [hidden, q_lora + 576]
 *   q   = bf16(bf16(rmsnorm(a[:q_lora]; g_q)) . W_uq)     W_uq [q_lora, n_heads*192]
 *         per head: [q_nope (128) | q_rope (64)]
 *   row = [bf16(rmsnorm(a[q_lora:q_lora+512]; g_kv)) | bf16(rope(a[q_lora+512:], L))]
 *         appended to the latent cache at L    cache [B, max_ctx, 576]
 *   per head h, with W_kvb [512, n_heads*256] holding per head [W_k (128) | W_v (128)]:
 *     keys    k_t = [c_t . W_k,h | k_rope_t], values v_t = c_t . W_v,h  (c_t = latent of row t)
 *     o_h     = softmax_t((q_nope . k_nope_t + rope(q_rope) . k_rope_t) / sqrt(192)) . v
 *   out = bf16(bf16(concat_h o_h) . W_o)   W_o  [n_heads*128, hidden]
 * rope is the rotate-half form of cfa_decode_step_ex over the 64 rope dims
 * (rope_theta 0 disables it); rmsnorm as cfa_rmsnorm. The attention runs in
 * absorbed form (q_nope folded into W_k, values projected after the sum), one
 * thread-block cluster per (sequence, group of 16 heads) -- or two or four,
 * each over its share of the latent rows ("row splits", §5.2's cache
 * partitioned across clusters), chosen per step when that grid still fits on
 * the GPU at once; the last of them to finish combines them in split order,
 * so a given shape's results are bitwise reproducible.
 * ========================================================================== */

typedef struct cfa_mla cfa_mla; /* opaque */

/*
 * Plan for batch B (1..16), hidden a multiple of 64, n_heads even (the
 * cluster holds the largest power-of-two group of heads up to 16 that divides
 * n_heads), q_lora a multiple of 64, max_ctx latent rows per sequence.
 * Allocates the intermediate a, q, v buffers, GEMV workspace and status words.
 * NULL on failure; cfa_last_error() says why.
 */
cfa_mla *cfa_mla_create(int B, int hidden, int n_heads, int q_lora, int max_ctx);

/* Release the plan (synchronizes the device first). NULL is a no-op. */
void cfa_mla_destroy(cfa_mla *mla);

/*
 * One MLA decode step (4 kernel launches). ctx_lens: host array [B], each in
 * [0, max_ctx - 1]; row ctx_lens[b] of the cache is written, rows below it are
 * read. out must not overlap x, the cache or W_o. Errors as cfa_decode_step.
 */
cfa_status cfa_mla_step(cfa_mla *mla, const void *x, const void *W_a, const void *g_q,
                        const void *g_kv, const void *W_uq, const void *W_kvb, const void *W_o,
                        void *cache, const int *ctx_lens, double rope_theta, float eps,
                        void *out, void *stream);

/* Synchronizes, reads and clears the plan's device status words. */
cfa_status cfa_mla_status(cfa_mla *mla);

/* One-line JSON description (cluster shape, row splits, grid, shared memory,
 * GEMV grids). */
cfa_status cfa_mla_describe(const cfa_mla *mla, char *buf, int len);

/*
 * Fix the number of row splits (1, 2 or 4 clusters per sequence and head
 * group, each over its share of the latent rows) for every later step; the
 * cluster size becomes the largest whose grid then fits on the GPU at once.
 * 0 restores the default, a choice per step: of the shapes that fit at once,
 * the one with the least estimated attention time for the step's longest
 * sequence (long contexts split further). Synchronizes the device first.
 * CFA_ERR_INVALID_ARG for other values; CFA_ERR_UNSUPPORTED if no cluster size
 * fits.
 */
cfa_status cfa_mla_set_row_splits(cfa_mla *mla, int splits);

#ifdef __cplusplus
}
#endif

#endif /* CFA_H */
