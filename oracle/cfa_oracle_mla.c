/*
 * cfa_oracle_mla.c -- fp64 CPU oracle for one decode step of a multi-head
 * latent attention (MLA) block, the DeepSeek variant the page adapts
 * ClusterFusion to: the latent key/value cache partitioned across clusters,
 * combined by a sparse cluster reduction [CF §5.2].
 *
 * TEST INFRASTRUCTURE, under the same rules as cfa_oracle.c: only the test
 * suite, the smoke check and the CPU baseline leg of the benchmark load it;
 * the CUDA library never links, calls or includes it.
 *
 * Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命" (ClusterFusion
 * framework analysis), written [CF §n]. The page names MLA and its latent cache
 * but gives no formula or dimension; the block below is the DeepSeek-V2/V3
 * attention as published with those models, with their dimensions
 * (kv_lora = 512, per-head nope / rope / value widths 128 / 64 / 128). This is
 * a reading, written from the architecture, not from any code.
 *
 * For batch row b at position L = ctx_lens[b] (weights [in, out], applied as
 * v . W; bf16(.) = round-to-nearest-even at the points a bf16 engine stores):
 *
 *   a    = bf16( x . W_a )                       W_a [H, q_lora + 576]
 *   cq   = bf16( rmsnorm(a[0 : q_lora]; g_q) )
 *   q    = bf16( cq . W_uq )                     W_uq [q_lora, nh*192]
 *          head h: q_nope = q[h*192 : h*192+128], q_rope = q[h*192+128 : h*192+192]
 *   ckv  = bf16( rmsnorm(a[q_lora : q_lora+512]; g_kv) )
 *   kr   = bf16( rope(a[q_lora+512 : q_lora+576], L) )
 *   cache row L := [ckv | kr]                    cache [B, max_ctx, 576]
 *   for each head h, keys and values decompressed from the latent rows
 *   t = 0..L (row L is the new one):             W_kvb [512, nh*256]
 *     k_t = [ c_t . W_kvb[:, h*256 : h*256+128] | kr_t ]        (192)
 *     v_t =   c_t . W_kvb[:, h*256+128 : h*256+256]             (128)
 *     s_t = ( [q_nope | rope(q_rope, L)] . k_t ) / sqrt(192)
 *     o_h = sum_t softmax(s)_t v_t
 *   v    = bf16( concat_h o_h )                  [B, nh*128]
 *   out  = v . W_o                               W_o [nh*128, H]
 *
 * rope is the rotate-half rotation of the cfa_oracle.c reading (dims i and
 * i+32 of the 64 rope dims by pos * theta^(-2i/64)); rmsnorm is
 * g_i v_i / sqrt(mean v^2 + eps). The keys and values are written out per head
 * (the plain definition); the fused kernel reaches the same value through the
 * absorbed form, which no step here uses.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Defined in cfa_oracle.c / cfa_oracle_layer.c. */
void cfa_oracle_rope(int d, const double *x, int pos, double theta, double *y);
uint16_t cfa_oracle_round_bf16(double v);
void cfa_oracle_rmsnorm(int n, const double *x, const double *g, double eps, double *y);

#define MLA_KV 512
#define MLA_NOPE 128
#define MLA_ROPE 64
#define MLA_V 128
#define MLA_QK (MLA_NOPE + MLA_ROPE)
#define MLA_ROW (MLA_KV + MLA_ROPE)

static double wid(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double rnd(double v) { return wid(cfa_oracle_round_bf16(v)); }

/*
 * Single-query softmax attention with keys of width dk and values of width
 * dv (MLA's keys are 192 wide, its values 128):
 *   s_t = scale (q . K_t), m = max s_t, a = sum_t e^(s_t - m) V_t / sum_t e^(s_t - m).
 * q [dk], K [T][dk], V [T][dv], a [dv]; T >= 1.
 */
void cfa_oracle_attention_kv(int T, int dk, int dv, const double *q, const double *K,
                             const double *V, double scale, double *a)
{
    double *w = (double *)malloc(sizeof(double) * (size_t)T);
    double m = -INFINITY;
    for (int t = 0; t < T; ++t) {
        double s = 0.0;
        for (int i = 0; i < dk; ++i)
            s += q[i] * K[(size_t)t * dk + i];
        w[t] = s * scale;
        if (w[t] > m)
            m = w[t];
    }
    double den = 0.0;
    for (int t = 0; t < T; ++t) {
        w[t] = exp(w[t] - m);
        den += w[t];
    }
    for (int i = 0; i < dv; ++i)
        a[i] = 0.0;
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < dv; ++i)
            a[i] += w[t] * V[(size_t)t * dv + i];
    for (int i = 0; i < dv; ++i)
        a[i] /= den;
    free(w);
}

/*
 * The step of the header comment. out [B][H]; new_row [B][576] (the appended
 * latent row, after rounding); v [B][nh*128] (after rounding); attn_f64
 * [B][nh*128] (o before rounding, may be NULL). The cache is read, not
 * written. Returns 0, or -1 on a bad argument.
 */
int cfa_oracle_mla_step(int B, int H, int nh, int q_lora, int max_ctx, const int *ctx_lens,
                        double rope_theta, double eps, const uint16_t *x, const uint16_t *W_a,
                        const uint16_t *g_q, const uint16_t *g_kv, const uint16_t *W_uq,
                        const uint16_t *W_kvb, const uint16_t *W_o, const uint16_t *cache,
                        double *out, double *new_row, double *v_out, double *attn_f64,
                        int nthreads)
{
    if (B < 1 || H < 1 || nh < 1 || q_lora < 1 || max_ctx < 1 || !(eps >= 0.0))
        return -1;
    for (int b = 0; b < B; ++b)
        if (ctx_lens[b] < 0 || ctx_lens[b] >= max_ctx)
            return -1;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#else
    (void)nthreads;
#endif
    const int NA = q_lora + MLA_ROW;        /* columns of W_a */
    const int NQ = nh * MLA_QK;             /* columns of W_uq */
    const int NKV = nh * (MLA_NOPE + MLA_V); /* columns of W_kvb */
    const int NV = nh * MLA_V;
    const double scale = 1.0 / sqrt((double)MLA_QK);
    double *a = (double *)malloc(sizeof(double) * (size_t)NA);
    double *cq = (double *)malloc(sizeof(double) * (size_t)q_lora);
    double *gq = (double *)malloc(sizeof(double) * (size_t)q_lora);
    double *gkv = (double *)malloc(sizeof(double) * MLA_KV);
    double *q = (double *)malloc(sizeof(double) * (size_t)NQ);
    double *row = (double *)malloc(sizeof(double) * MLA_ROW);
    double *o = (double *)malloc(sizeof(double) * (size_t)NV);
    double *vr = (double *)malloc(sizeof(double) * (size_t)NV);
    int rc = -1;
    if (!a || !cq || !gq || !gkv || !q || !row || !o || !vr)
        goto done;
    for (int i = 0; i < q_lora; ++i)
        gq[i] = wid(g_q[i]);
    for (int i = 0; i < MLA_KV; ++i)
        gkv[i] = wid(g_kv[i]);

    for (int b = 0; b < B; ++b) {
        const int L = ctx_lens[b], T = L + 1;
        /* a = bf16(x . W_a) */
        for (int j = 0; j < NA; ++j)
            a[j] = 0.0;
        for (int i = 0; i < H; ++i) {
            const double xi = wid(x[(size_t)b * H + i]);
            const uint16_t *w = W_a + (size_t)i * NA;
            for (int j = 0; j < NA; ++j)
                a[j] += xi * wid(w[j]);
        }
        for (int j = 0; j < NA; ++j)
            a[j] = rnd(a[j]);
        /* cq = bf16(rmsnorm(a[:q_lora])); q = bf16(cq . W_uq) */
        cfa_oracle_rmsnorm(q_lora, a, gq, eps, cq);
        for (int i = 0; i < q_lora; ++i)
            cq[i] = rnd(cq[i]);
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
        for (int j0 = 0; j0 < NQ; j0 += 256) {
            const int j1 = j0 + 256 < NQ ? j0 + 256 : NQ;
            for (int j = j0; j < j1; ++j)
                q[j] = 0.0;
            for (int i = 0; i < q_lora; ++i) {
                const uint16_t *w = W_uq + (size_t)i * NQ;
                for (int j = j0; j < j1; ++j)
                    q[j] += cq[i] * wid(w[j]);
            }
            for (int j = j0; j < j1; ++j)
                q[j] = rnd(q[j]);
        }
        /* the new latent row: [bf16(rmsnorm(ckv)) | bf16(rope(kr, L))] */
        cfa_oracle_rmsnorm(MLA_KV, a + q_lora, gkv, eps, row);
        for (int i = 0; i < MLA_KV; ++i)
            row[i] = rnd(row[i]);
        if (rope_theta > 0.0)
            cfa_oracle_rope(MLA_ROPE, a + q_lora + MLA_KV, L, rope_theta, row + MLA_KV);
        else
            memcpy(row + MLA_KV, a + q_lora + MLA_KV, sizeof(double) * MLA_ROPE);
        for (int i = MLA_KV; i < MLA_ROW; ++i)
            row[i] = rnd(row[i]);
        if (new_row)
            memcpy(new_row + (size_t)b * MLA_ROW, row, sizeof(double) * MLA_ROW);

        /* per head: decompress keys / values from every latent row, attend */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
        for (int h = 0; h < nh; ++h) {
            double *qh = (double *)malloc(sizeof(double) * MLA_QK);
            double *K = (double *)malloc(sizeof(double) * (size_t)T * MLA_QK);
            double *V = (double *)malloc(sizeof(double) * (size_t)T * MLA_V);
            double *c = (double *)malloc(sizeof(double) * MLA_ROW);
            memcpy(qh, q + (size_t)h * MLA_QK, sizeof(double) * MLA_NOPE);
            if (rope_theta > 0.0)
                cfa_oracle_rope(MLA_ROPE, q + (size_t)h * MLA_QK + MLA_NOPE, L, rope_theta,
                                qh + MLA_NOPE);
            else
                memcpy(qh + MLA_NOPE, q + (size_t)h * MLA_QK + MLA_NOPE, sizeof(double) * MLA_ROPE);
            for (int t = 0; t < T; ++t) {
                if (t < L) {
                    const uint16_t *cr = cache + ((size_t)b * max_ctx + t) * MLA_ROW;
                    for (int i = 0; i < MLA_ROW; ++i)
                        c[i] = wid(cr[i]);
                } else {
                    memcpy(c, row, sizeof(double) * MLA_ROW);
                }
                double *kt = K + (size_t)t * MLA_QK;
                double *vt = V + (size_t)t * MLA_V;
                for (int j = 0; j < MLA_NOPE; ++j)
                    kt[j] = 0.0;
                for (int j = 0; j < MLA_V; ++j)
                    vt[j] = 0.0;
                for (int i = 0; i < MLA_KV; ++i) {
                    const uint16_t *w = W_kvb + (size_t)i * NKV + (size_t)h * (MLA_NOPE + MLA_V);
                    for (int j = 0; j < MLA_NOPE; ++j)
                        kt[j] += c[i] * wid(w[j]);
                    for (int j = 0; j < MLA_V; ++j)
                        vt[j] += c[i] * wid(w[MLA_NOPE + j]);
                }
                memcpy(kt + MLA_NOPE, c + MLA_KV, sizeof(double) * MLA_ROPE);
            }
            cfa_oracle_attention_kv(T, MLA_QK, MLA_V, qh, K, V, scale, o + (size_t)h * MLA_V);
            free(qh);
            free(K);
            free(V);
            free(c);
        }
        if (attn_f64)
            memcpy(attn_f64 + (size_t)b * NV, o, sizeof(double) * NV);
        for (int j = 0; j < NV; ++j)
            vr[j] = rnd(o[j]);
        if (v_out)
            memcpy(v_out + (size_t)b * NV, vr, sizeof(double) * NV);
        /* out = v . W_o */
        double *ob = out + (size_t)b * H;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
        for (int j0 = 0; j0 < H; j0 += 256) {
            const int j1 = j0 + 256 < H ? j0 + 256 : H;
            for (int j = j0; j < j1; ++j)
                ob[j] = 0.0;
            for (int i = 0; i < NV; ++i) {
                const uint16_t *w = W_o + (size_t)i * H;
                for (int j = j0; j < j1; ++j)
                    ob[j] += vr[i] * wid(w[j]);
            }
        }
    }
    rc = 0;
done:
    free(a); free(cq); free(gq); free(gkv); free(q); free(row); free(o); free(vr);
    return rc;
}
