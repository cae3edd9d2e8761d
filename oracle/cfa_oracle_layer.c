/*
 * cfa_oracle_layer.c -- fp64 CPU oracle for a stack of decoder layers built
 * around the attention block of cfa_oracle.c: the multi-layer decode loop
 * whose time per output token the page reports for Llama2-7B [CF §3.3, §5.1].
 *
 * TEST INFRASTRUCTURE, under the same rules as cfa_oracle.c: only the test
 * suite, the smoke check and the CPU baseline leg of the benchmark load it;
 * the CUDA library never links, calls or includes it.
 *
 * Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命" (ClusterFusion
 * framework analysis), written [CF §n].
 *
 * The page describes only the attention block of a layer [CF §1.1]. The rest
 * of a Llama2-style layer is a stand-in taken in the Llama2 arrangement
 * (pre-norm, two residual adds, SwiGLU MLP); this is a reading, not the page:
 *
 *   xn = bf16( rmsnorm(x; g_attn) )
 *   a  = attention block(xn)                      (cfa_oracle_decode_step_ex)
 *   h  = bf16( x + a )
 *   hn = bf16( rmsnorm(h; g_mlp) )
 *   u  = bf16( silu(hn . W_gate) * (hn . W_up) )
 *   y  = bf16( h + u . W_down )
 *
 * with rmsnorm(x; g)_i = g_i x_i / sqrt(mean_j x_j^2 + eps) and
 * silu(z) = z / (1 + e^-z). bf16(.) is round-to-nearest-even of the exact
 * value: xn, h, hn, u and y are the tensors a bf16 inference engine keeps
 * between stages (matmul operands and the residual stream). Everything else
 * is fp64. Weights are [in, out] row-major, applied as v . W, as for the
 * attention block.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Declared in cfa_oracle.c. */
int cfa_oracle_decode_step_ex(int B, int H, int nh, int d, int max_ctx, const int *ctx_lens,
                              double rope_theta, const uint16_t *x, const uint16_t *W_qkv,
                              const uint16_t *W_o, const uint16_t *k_cache,
                              const uint16_t *v_cache, double *out, double *k_new,
                              double *v_new, double *attn, int nthreads);

static double widen(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest bf16, ties to even, in one step (no detour
 * through float, which would round twice). bf16 has 8 significant bits and
 * float's exponent range: in the binade [2^(e-1), 2^e) its values are spaced
 * 2^(e-8); below 2^-126 the spacing stays 2^-133 (subnormals). Magnitudes that
 * round to 2^128 or more become infinity.
 */
uint16_t cfa_oracle_round_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    const uint16_t sign = signbit(v) ? 0x8000 : 0;
    const double a = fabs(v);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e;
    frexp(a, &e);               /* a = m 2^e, m in [0.5, 1) */
    int q = e - 8;
    if (q < -133)
        q = -133;
    const double n = nearbyint(ldexp(a, -q));   /* default mode: ties to even */
    const double r = ldexp(n, q);
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;
    const float f = (float)r;   /* exact: at most 8 significant bits, in range */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

void cfa_oracle_round_bf16_array(const double *src, uint16_t *dst, long n)
{
    for (long i = 0; i < n; ++i)
        dst[i] = cfa_oracle_round_bf16(src[i]);
}

/* y_i = g_i x_i / sqrt(mean_j x_j^2 + eps), all fp64. */
void cfa_oracle_rmsnorm(int n, const double *x, const double *g, double eps, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i)
        ss += x[i] * x[i];
    const double s = 1.0 / sqrt(ss / n + eps);
    for (int i = 0; i < n; ++i)
        y[i] = g[i] * x[i] * s;
}

double cfa_oracle_silu(double z)
{
    return z / (1.0 + exp(-z));
}

/* Row-wise bf16( rmsnorm(x[b]; g) ) of bf16 inputs: x, y [B][n], g [n]. */
int cfa_oracle_rmsnorm_bf16(int B, int n, const uint16_t *x, const uint16_t *g, double eps,
                            uint16_t *y)
{
    if (B < 1 || n < 1 || !(eps >= 0.0))
        return -1;
    double *xd = (double *)malloc(sizeof(double) * (size_t)n * 3);
    if (!xd)
        return -1;
    double *gd = xd + n, *yd = xd + 2 * (size_t)n;
    for (int i = 0; i < n; ++i)
        gd[i] = widen(g[i]);
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < n; ++i)
            xd[i] = widen(x[(size_t)b * n + i]);
        cfa_oracle_rmsnorm(n, xd, gd, eps, yd);
        cfa_oracle_round_bf16_array(yd, y + (size_t)b * n, n);
    }
    free(xd);
    return 0;
}

/*
 * The SwiGLU MLP with its pre-norm and residual, for every batch row:
 *   hn = bf16(rmsnorm(h; g)),  u = bf16(silu(hn . W_gate) * (hn . W_up)),
 *   delta = u . W_down (fp64),  y = bf16(h + delta).
 * h, y [B][H]; g [H]; W_gate, W_up [H][F]; W_down [F][H]; u [B][F] (bits,
 * may be NULL); delta [B][H] (may be NULL). Returns 0, or -1 on a bad
 * argument.
 */
int cfa_oracle_mlp(int B, int H, int F, double eps, const uint16_t *h, const uint16_t *g,
                   const uint16_t *W_gate, const uint16_t *W_up, const uint16_t *W_down,
                   uint16_t *u_out, double *delta, uint16_t *y, int nthreads)
{
    if (B < 1 || H < 1 || F < 1 || !(eps >= 0.0))
        return -1;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#else
    (void)nthreads;
#endif
    double *hd = (double *)malloc(sizeof(double) * (size_t)H);
    double *gd = (double *)malloc(sizeof(double) * (size_t)H);
    double *hn = (double *)malloc(sizeof(double) * (size_t)H);
    double *gate = (double *)malloc(sizeof(double) * (size_t)F);
    double *up = (double *)malloc(sizeof(double) * (size_t)F);
    double *u = (double *)malloc(sizeof(double) * (size_t)F);
    double *dl = (double *)malloc(sizeof(double) * (size_t)H);
    if (!hd || !gd || !hn || !gate || !up || !u || !dl) {
        free(hd); free(gd); free(hn); free(gate); free(up); free(u); free(dl);
        return -1;
    }
    for (int i = 0; i < H; ++i)
        gd[i] = widen(g[i]);
    const int CB = 256;  /* columns per parallel work item */
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i < H; ++i)
            hd[i] = widen(h[(size_t)b * H + i]);
        cfa_oracle_rmsnorm(H, hd, gd, eps, hn);
        for (int i = 0; i < H; ++i)
            hn[i] = widen(cfa_oracle_round_bf16(hn[i]));

        /* gate_j = sum_i hn_i W_gate[i, j]; up_j likewise. */
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
        for (int j0 = 0; j0 < F; j0 += CB) {
            const int j1 = j0 + CB < F ? j0 + CB : F;
            for (int j = j0; j < j1; ++j) {
                gate[j] = 0.0;
                up[j] = 0.0;
            }
            for (int i = 0; i < H; ++i) {
                const uint16_t *rg = W_gate + (size_t)i * F;
                const uint16_t *ru = W_up + (size_t)i * F;
                for (int j = j0; j < j1; ++j) {
                    gate[j] += hn[i] * widen(rg[j]);
                    up[j] += hn[i] * widen(ru[j]);
                }
            }
            for (int j = j0; j < j1; ++j) {
                const uint16_t bits = cfa_oracle_round_bf16(cfa_oracle_silu(gate[j]) * up[j]);
                u[j] = widen(bits);
                if (u_out)
                    u_out[(size_t)b * F + j] = bits;
            }
        }

        /* delta_k = sum_j u_j W_down[j, k]; y = bf16(h + delta). */
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
        for (int k0 = 0; k0 < H; k0 += CB) {
            const int k1 = k0 + CB < H ? k0 + CB : H;
            for (int k = k0; k < k1; ++k)
                dl[k] = 0.0;
            for (int j = 0; j < F; ++j) {
                const uint16_t *rd = W_down + (size_t)j * H;
                for (int k = k0; k < k1; ++k)
                    dl[k] += u[j] * widen(rd[k]);
            }
            for (int k = k0; k < k1; ++k) {
                if (delta)
                    delta[(size_t)b * H + k] = dl[k];
                y[(size_t)b * H + k] = cfa_oracle_round_bf16(hd[k] + dl[k]);
            }
        }
    }
    free(hd); free(gd); free(hn); free(gate); free(up); free(u); free(dl);
    return 0;
}

/*
 * One decoder layer for one token, in the order of the header comment.
 * Shapes: x, xn, h, y [B][H]; g_attn, g_mlp [H]; W_qkv [H][3H]; W_o [H][H];
 * caches [B][nh][max_ctx][d]; W_gate, W_up [H][F]; W_down [F][H]; u [B][F];
 * k_new, v_new [B][nh][d] (fp64, the rows to append at ctx_lens[b], k after
 * the rotary embedding). xn, h and u may be NULL. The caches are read, not
 * written. Returns 0, or -1 on a bad argument.
 */
int cfa_oracle_layer_step(int B, int H, int nh, int d, int F, int max_ctx, const int *ctx_lens,
                          double rope_theta, double eps, const uint16_t *x,
                          const uint16_t *g_attn, const uint16_t *W_qkv, const uint16_t *W_o,
                          const uint16_t *k_cache, const uint16_t *v_cache,
                          const uint16_t *g_mlp, const uint16_t *W_gate, const uint16_t *W_up,
                          const uint16_t *W_down, uint16_t *xn_out, uint16_t *h_out,
                          uint16_t *u_out, uint16_t *y, double *k_new, double *v_new,
                          int nthreads)
{
    if (B < 1 || H < 1 || F < 1 || nh < 1 || H != nh * d)
        return -1;
    const size_t BH = (size_t)B * H;
    uint16_t *xn = (uint16_t *)malloc(sizeof(uint16_t) * BH);
    uint16_t *hb = (uint16_t *)malloc(sizeof(uint16_t) * BH);
    double *a = (double *)malloc(sizeof(double) * BH);
    int rc = -1;
    if (!xn || !hb || !a)
        goto done;
    if (cfa_oracle_rmsnorm_bf16(B, H, x, g_attn, eps, xn) != 0)
        goto done;
    if (cfa_oracle_decode_step_ex(B, H, nh, d, max_ctx, ctx_lens, rope_theta, xn, W_qkv, W_o,
                                  k_cache, v_cache, a, k_new, v_new, NULL, nthreads) != 0)
        goto done;
    for (size_t i = 0; i < BH; ++i)
        hb[i] = cfa_oracle_round_bf16(widen(x[i]) + a[i]);
    if (cfa_oracle_mlp(B, H, F, eps, hb, g_mlp, W_gate, W_up, W_down, u_out, NULL, y,
                       nthreads) != 0)
        goto done;
    if (xn_out)
        memcpy(xn_out, xn, sizeof(uint16_t) * BH);
    if (h_out)
        memcpy(h_out, hb, sizeof(uint16_t) * BH);
    rc = 0;
done:
    free(xn);
    free(hb);
    free(a);
    return rc;
}
