/*
 * cfa_oracle.c -- fp64 CPU oracle for one decode step of a decoder attention
 * block (QKV projection -> KV append -> single-query attention -> output
 * projection).
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this library. The CUDA library never
 * links, calls or includes it, and this file includes nothing from the CUDA
 * library.
 *
 * Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命" (ClusterFusion
 * framework analysis), written [CF §n] below.
 *
 * What it computes is the plain definition of the block, in the order the
 * page gives its three stages [CF §1.1]: project the new token to q, k, v with
 * one merged matrix [CF §5.1], attend over the cached keys plus the new one
 * with a max-subtracted softmax, then project the per-head results with W_o.
 * The fused method of [CF §3.2] reaches this same value; only the order of
 * rounding differs, so no blocking, fusion or split is done here.
 *
 * Readings of points the page leaves open (each is also listed in the design
 * notes):
 *   - weights are [in, out] row-major and applied as x . W, following the
 *     page's torch.mm(hidden_states, W_qkv) form [CF §1.1];
 *   - W_qkv's 3H columns are [Q | K | V], head h owning columns
 *     [h*d, (h+1)*d) inside each block (merged QKV matrix, [CF §5.1]);
 *   - scale = 1/sqrt(head_dim); no RoPE, norm, bias or residual;
 *   - the new token is attended: T = ctx_len + 1 keys, the new k/v at
 *     position ctx_len;
 *   - one ctx_len shared by every batch row.
 * cfa_oracle_decode_step_ex widens the last two: one context length per batch
 * row, and an optional rotary embedding of the new q and k (rotate-half form
 * as in Llama2-style models).
 *
 * All inputs arrive as bf16 bit patterns (uint16) and are widened exactly to
 * double; every sum, product, exp and division is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an IEEE
 * binary32, so shifting into the high 16 bits gives the same real number. */
static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

void cfa_oracle_widen_bf16(const uint16_t *src, double *dst, long n)
{
    for (long i = 0; i < n; ++i)
        dst[i] = widen_bf16(src[i]);
}

/*
 * Single-query softmax attention over T keys, the "flash_attention" stage of
 * [CF §1.1] written out monolithically:
 *   s_t = scale * (q . K_t),  m = max_t s_t,
 *   a   = sum_t exp(s_t - m) V_t / sum_t exp(s_t - m).
 * q: [d], K, V: [T][d], a: [d]. T >= 1.
 */
void cfa_oracle_attention(int T, int d, const double *q, const double *K,
                          const double *V, double scale, double *a)
{
    double *w = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    double m = -INFINITY;
    for (int t = 0; t < T; ++t) {
        double s = 0.0;
        for (int i = 0; i < d; ++i)
            s += q[i] * K[(size_t)t * d + i];
        s *= scale;
        w[t] = s;
        if (s > m)
            m = s;
    }
    double denom = 0.0;
    for (int t = 0; t < T; ++t) {
        w[t] = exp(w[t] - m);
        denom += w[t];
    }
    for (int i = 0; i < d; ++i)
        a[i] = 0.0;
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < d; ++i)
            a[i] += w[t] * V[(size_t)t * d + i];
    for (int i = 0; i < d; ++i)
        a[i] /= denom;
    free(w);
}

/*
 * The per-split statistics of split-KV attention [CF §3.2]: one block of the
 * cluster owns the key range [t0, t1) and keeps
 *   m = max s_t,  l = sum exp(s_t - m),  o = sum exp(s_t - m) V_t.
 * An empty range gives m = -inf, l = 0, o = 0.
 */
void cfa_oracle_split_partial(int t0, int t1, int d, const double *q,
                              const double *K, const double *V, double scale,
                              double *m_out, double *l_out, double *o)
{
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        double s = 0.0;
        for (int i = 0; i < d; ++i)
            s += q[i] * K[(size_t)t * d + i];
        s *= scale;
        if (s > m)
            m = s;
    }
    double l = 0.0;
    for (int i = 0; i < d; ++i)
        o[i] = 0.0;
    if (t1 > t0) {
        for (int t = t0; t < t1; ++t) {
            double s = 0.0;
            for (int i = 0; i < d; ++i)
                s += q[i] * K[(size_t)t * d + i];
            double p = exp(s * scale - m);
            l += p;
            for (int i = 0; i < d; ++i)
                o[i] += p * V[(size_t)t * d + i];
        }
    }
    *m_out = m;
    *l_out = l;
}

/*
 * Combine of split partials in the page's two-step form [CF §3.1.1, §3.2]:
 * first a max-reduction of the m_r, then a sum-reduction of the rescaled
 * l_r and o_r:  m = max_r m_r,  l = sum_r l_r e^(m_r - m),
 * o = sum_r o_r e^(m_r - m),  a = o / l.
 * Splits with m_r = -inf (no keys) contribute nothing. At least one split
 * must hold a key. m, l: [n]; o: [n][d]; a: [d].
 */
void cfa_oracle_split_combine(int n, int d, const double *m, const double *l,
                              const double *o, double *a)
{
    double M = -INFINITY;
    for (int r = 0; r < n; ++r)
        if (m[r] > M)
            M = m[r];
    double L = 0.0;
    for (int i = 0; i < d; ++i)
        a[i] = 0.0;
    for (int r = 0; r < n; ++r) {
        if (m[r] == -INFINITY)
            continue;
        double f = exp(m[r] - M);
        L += l[r] * f;
        for (int i = 0; i < d; ++i)
            a[i] += o[(size_t)r * d + i] * f;
    }
    for (int i = 0; i < d; ++i)
        a[i] /= L;
}

/*
 * One decode step of the block for every batch row b and head h
 * [CF §1.1, §3.2, §5.1]:
 *   q, k, v    = x[b] . W_qkv restricted to head h's columns of Q, K, V;
 *   k_new, v_new (outputs) = k, v   (the row appended at position L);
 *   keys       = k_cache[b, h, 0..L-1] followed by k; values likewise;
 *   attn[b, h] = softmax attention of q over those L+1 keys;
 *   out[b]     = concat_h(attn[b, h]) . W_o.
 *
 * Layouts: x [B][H]; W_qkv [H][3H]; W_o [H][H]; k_cache, v_cache
 * [B][nh][max_ctx][d]; out [B][H]; k_new, v_new, attn [B][nh][d] (attn may be
 * NULL). The caches are read-only here: the oracle reports the appended row
 * instead of writing it.
 *
 * Returns 0 on success, -1 on a bad argument.
 */
int cfa_oracle_decode_step(int B, int H, int nh, int d, int max_ctx, int L,
                           const uint16_t *x, const uint16_t *W_qkv,
                           const uint16_t *W_o, const uint16_t *k_cache,
                           const uint16_t *v_cache, double *out,
                           double *k_new, double *v_new, double *attn,
                           int nthreads)
{
    if (B < 1 || nh < 1 || d < 1 || H != nh * d || L < 0 || L >= max_ctx)
        return -1;
    const int T = L + 1;
    const double scale = 1.0 / sqrt((double)d);
    double *a_all = (double *)malloc(sizeof(double) * (size_t)B * nh * d);
    if (!a_all)
        return -1;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#else
    (void)nthreads;
#endif

    /* Stages 1 and 2 for every (b, h). */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int bh = 0; bh < B * nh; ++bh) {
        const int b = bh / nh, h = bh % nh;
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        double *K = (double *)malloc(sizeof(double) * (size_t)T * d);
        double *V = (double *)malloc(sizeof(double) * (size_t)T * d);
        double *kk = K + (size_t)L * d;  /* the new key is row L */
        double *vv = V + (size_t)L * d;
        for (int j = 0; j < d; ++j) {
            q[j] = 0.0;
            kk[j] = 0.0;
            vv[j] = 0.0;
        }
        /* QKV projection of the new token: q_j = sum_i x_i W_qkv[i, col_j]. */
        for (int i = 0; i < H; ++i) {
            const double xi = widen_bf16(x[(size_t)b * H + i]);
            const uint16_t *row = W_qkv + (size_t)i * 3 * H;
            for (int j = 0; j < d; ++j) {
                q[j] += xi * widen_bf16(row[0 * H + h * d + j]);
                kk[j] += xi * widen_bf16(row[1 * H + h * d + j]);
                vv[j] += xi * widen_bf16(row[2 * H + h * d + j]);
            }
        }
        /* Cached keys/values at positions 0..L-1. */
        const size_t base = ((size_t)b * nh + h) * (size_t)max_ctx * d;
        for (int t = 0; t < L; ++t)
            for (int j = 0; j < d; ++j) {
                K[(size_t)t * d + j] = widen_bf16(k_cache[base + (size_t)t * d + j]);
                V[(size_t)t * d + j] = widen_bf16(v_cache[base + (size_t)t * d + j]);
            }
        for (int j = 0; j < d; ++j) {
            k_new[(size_t)bh * d + j] = kk[j];
            v_new[(size_t)bh * d + j] = vv[j];
        }
        cfa_oracle_attention(T, d, q, K, V, scale, a_all + (size_t)bh * d);
        free(q);
        free(K);
        free(V);
    }

    /* Stage 3: out[b, j] = sum over (h, i) of attn[b, h, i] W_o[h*d + i, j]. */
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int b = 0; b < B; ++b) {
        double *acc = out + (size_t)b * H;
        for (int j = 0; j < H; ++j)
            acc[j] = 0.0;
        for (int r = 0; r < H; ++r) {
            const double ar = a_all[(size_t)b * H + r];
            const uint16_t *row = W_o + (size_t)r * H;
            for (int j = 0; j < H; ++j)
                acc[j] += ar * widen_bf16(row[j]);
        }
    }
    if (attn)
        memcpy(attn, a_all, sizeof(double) * (size_t)B * nh * d);
    free(a_all);
    return 0;
}

/* Threads an OpenMP build would use for a request of n (1 without OpenMP). */
int cfa_oracle_threads(int n)
{
#ifdef _OPENMP
    return n < 1 ? 1 : n;
#else
    (void)n;
    return 1;
#endif
}

/*
 * Rotary position embedding, in the rotate-half form of Llama2-style models
 * (a reading: the ClusterFusion page names no positional encoding for its
 * block, [CF §1.1]). For i < d/2, with w_i = theta^(-2i/d) and angle a = pos w_i:
 *   y_i       = x_i cos a - x_{i+d/2} sin a
 *   y_{i+d/2} = x_{i+d/2} cos a + x_i sin a.
 * d must be even; y may not alias x.
 */
void cfa_oracle_rope(int d, const double *x, int pos, double theta, double *y)
{
    const int half = d / 2;
    for (int i = 0; i < half; ++i) {
        const double w = pow(theta, -2.0 * i / d);
        const double a = (double)pos * w;
        const double c = cos(a), s = sin(a);
        y[i] = x[i] * c - x[i + half] * s;
        y[i + half] = x[i + half] * c + x[i] * s;
    }
}

/*
 * The decode step with one context length per sequence and optional rotary
 * embedding of the new token's q and k at its own position ctx_lens[b]
 * (cached keys are taken as already rotated when they were appended).
 * rope_theta <= 0 disables the rotation. Everything else as
 * cfa_oracle_decode_step [CF §1.1, §3.2, §5.1]; k_new is reported after
 * rotation (the row that is appended).
 */
int cfa_oracle_decode_step_ex(int B, int H, int nh, int d, int max_ctx, const int *ctx_lens,
                              double rope_theta, const uint16_t *x, const uint16_t *W_qkv,
                              const uint16_t *W_o, const uint16_t *k_cache,
                              const uint16_t *v_cache, double *out, double *k_new,
                              double *v_new, double *attn, int nthreads)
{
    if (B < 1 || nh < 1 || d < 2 || (d & 1) || H != nh * d)
        return -1;
    for (int b = 0; b < B; ++b)
        if (ctx_lens[b] < 0 || ctx_lens[b] >= max_ctx)
            return -1;
    const double scale = 1.0 / sqrt((double)d);
    double *a_all = (double *)malloc(sizeof(double) * (size_t)B * nh * d);
    if (!a_all)
        return -1;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#else
    (void)nthreads;
#endif

#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int bh = 0; bh < B * nh; ++bh) {
        const int b = bh / nh, h = bh % nh;
        const int L = ctx_lens[b], T = L + 1;
        double *q0 = (double *)malloc(sizeof(double) * (size_t)d);
        double *k0 = (double *)malloc(sizeof(double) * (size_t)d);
        double *q = (double *)malloc(sizeof(double) * (size_t)d);
        double *K = (double *)malloc(sizeof(double) * (size_t)T * d);
        double *V = (double *)malloc(sizeof(double) * (size_t)T * d);
        double *kk = K + (size_t)L * d;
        double *vv = V + (size_t)L * d;
        for (int j = 0; j < d; ++j) {
            q0[j] = 0.0;
            k0[j] = 0.0;
            vv[j] = 0.0;
        }
        for (int i = 0; i < H; ++i) {
            const double xi = widen_bf16(x[(size_t)b * H + i]);
            const uint16_t *row = W_qkv + (size_t)i * 3 * H;
            for (int j = 0; j < d; ++j) {
                q0[j] += xi * widen_bf16(row[0 * H + h * d + j]);
                k0[j] += xi * widen_bf16(row[1 * H + h * d + j]);
                vv[j] += xi * widen_bf16(row[2 * H + h * d + j]);
            }
        }
        if (rope_theta > 0.0) {
            cfa_oracle_rope(d, q0, L, rope_theta, q);
            cfa_oracle_rope(d, k0, L, rope_theta, kk);
        } else {
            memcpy(q, q0, sizeof(double) * (size_t)d);
            memcpy(kk, k0, sizeof(double) * (size_t)d);
        }
        const size_t base = ((size_t)b * nh + h) * (size_t)max_ctx * d;
        for (int t = 0; t < L; ++t)
            for (int j = 0; j < d; ++j) {
                K[(size_t)t * d + j] = widen_bf16(k_cache[base + (size_t)t * d + j]);
                V[(size_t)t * d + j] = widen_bf16(v_cache[base + (size_t)t * d + j]);
            }
        for (int j = 0; j < d; ++j) {
            k_new[(size_t)bh * d + j] = kk[j];
            v_new[(size_t)bh * d + j] = vv[j];
        }
        cfa_oracle_attention(T, d, q, K, V, scale, a_all + (size_t)bh * d);
        free(q0);
        free(k0);
        free(q);
        free(K);
        free(V);
    }

#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (int b = 0; b < B; ++b) {
        double *acc = out + (size_t)b * H;
        for (int j = 0; j < H; ++j)
            acc[j] = 0.0;
        for (int r = 0; r < H; ++r) {
            const double ar = a_all[(size_t)b * H + r];
            const uint16_t *row = W_o + (size_t)r * H;
            for (int j = 0; j < H; ++j)
                acc[j] += ar * widen_bf16(row[j]);
        }
    }
    if (attn)
        memcpy(attn, a_all, sizeof(double) * (size_t)B * nh * d);
    free(a_all);
    return 0;
}
