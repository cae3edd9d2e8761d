"""Pins for the MLA part of the fp64 oracle, each against something other than
the oracle itself. CPU only.

A plausible slip and the pin that catches it:
  * wrong value width / key width mix-up      -> attention_kv against the pinned
                                                 attention routine
  * new latent row not attended or misbuilt   -> ctx_len = 0 closed form
  * wrong head column block of W_kvb (k vs v) -> linearity: doubling one head's
                                                 value columns doubles only it
  * rope / nope split of the key wrong        -> zero keys give the mean of the
                                                 decompressed values
  * cache indexing                            -> permutation invariance, NaN tail
  * anything else on tiny shapes              -> brute force with math.fsum

Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命", written [CF §n]
(§5.2 names MLA and the latent cache; the block is the DeepSeek-V2/V3 one).
"""
import math

import numpy as np
import pytest
import torch

from out_proj_block_gb300 import workloads

KV, NOPE, ROPE, V = 512, 128, 64, 128
ROW = KV + ROPE


def bits_to_f64(b):
    u = np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f64(t):
    return t.double().numpy()


def mla_inputs(B, H, nh, q_lora, L, max_ctx, seed, poison=False):
    wl = workloads.custom_mla(B, H, nh, q_lora, L, max_ctx=max_ctx)
    return workloads.make_mla_inputs(wl, seed=seed, poison_tail=poison)


def run(oracle, t, lens, theta=10000.0, eps=1e-6):
    return oracle.mla_step(t["x"], t["W_a"], t["g_q"], t["g_kv"], t["W_uq"], t["W_kvb"], t["W_o"],
                           t["cache"], lens, theta, eps)


def test_attention_kv_matches_the_pinned_attention(oracle):
    rng = np.random.default_rng(1)
    q, K = rng.standard_normal(24), rng.standard_normal((7, 24))
    Vv = rng.standard_normal((7, 24))
    np.testing.assert_allclose(oracle.attention_kv(q, K, Vv, 0.3), oracle.attention(q, K, Vv, 0.3),
                               rtol=1e-13)
    # narrower values: the same weights applied to the first 10 columns
    np.testing.assert_allclose(oracle.attention_kv(q, K, Vv[:, :10], 0.3),
                               oracle.attention(q, K, Vv, 0.3)[:10], rtol=1e-13)


def test_ctx0_attends_only_the_new_latent_row(oracle):
    B, H, nh, ql = 2, 64, 2, 32
    t = mla_inputs(B, H, nh, ql, 0, 8, seed=2)
    r = run(oracle, t, [0, 0])
    x, Wa = f64(t["x"]), f64(t["W_a"])
    a = bits_to_f64(oracle.round_bf16(x @ Wa))
    gkv = f64(t["g_kv"])
    for b in range(B):
        ckv = bits_to_f64(oracle.round_bf16(oracle.rmsnorm(a[b, ql:ql + KV], gkv, 1e-6)))
        kr = bits_to_f64(oracle.round_bf16(a[b, ql + KV:]))  # rope at position 0 is the identity
        np.testing.assert_array_equal(r["new_row"][b], np.concatenate([ckv, kr]))
        Wkvb = f64(t["W_kvb"])
        o = np.concatenate([ckv @ Wkvb[:, h * 256 + NOPE:(h + 1) * 256] for h in range(nh)])
        np.testing.assert_allclose(r["attn"][b], o, rtol=1e-12, atol=1e-14)
        v = bits_to_f64(oracle.round_bf16(o))
        np.testing.assert_allclose(r["out"][b], v @ f64(t["W_o"]), rtol=1e-12, atol=1e-14)


def test_one_heads_value_columns_scale_only_that_head(oracle):
    B, H, nh, ql, L = 1, 64, 3, 32, 5
    t = mla_inputs(B, H, nh, ql, L, 8, seed=3)
    base = run(oracle, t, [L])
    W = t["W_kvb"].float().clone()
    W[:, 1 * 256 + NOPE:2 * 256] *= 2  # exact in bf16
    t2 = dict(t, W_kvb=W.to(torch.bfloat16))
    r = run(oracle, t2, [L])
    a0, a1 = base["attn"].reshape(nh, V), r["attn"].reshape(nh, V)
    np.testing.assert_array_equal(a1[0], a0[0])
    np.testing.assert_array_equal(a1[2], a0[2])
    np.testing.assert_allclose(a1[1], 2 * a0[1], rtol=1e-13)


def test_zero_keys_give_the_mean_of_the_decompressed_values(oracle):
    B, H, nh, ql, L = 1, 64, 2, 32, 6
    t = mla_inputs(B, H, nh, ql, L, 8, seed=4)
    W = t["W_kvb"].float().clone()
    for h in range(nh):
        W[:, h * 256:h * 256 + NOPE] = 0       # no nope keys
    Wuq = t["W_uq"].float().clone()
    for h in range(nh):
        Wuq[:, h * 192 + NOPE:(h + 1) * 192] = 0  # no rope query: rope keys do not count
    t2 = dict(t, W_kvb=W.to(torch.bfloat16), W_uq=Wuq.to(torch.bfloat16))
    r = run(oracle, t2, [L])
    rows = np.vstack([f64(t["cache"][0, :L]), r["new_row"][0:1]])
    mean_c = rows[:, :KV].mean(axis=0)
    Wk = f64(t2["W_kvb"])
    want = np.concatenate([mean_c @ Wk[:, h * 256 + NOPE:(h + 1) * 256] for h in range(nh)])
    np.testing.assert_allclose(r["attn"][0], want, rtol=1e-12, atol=1e-14)


def test_cache_rows_permute_freely_and_the_tail_is_not_read(oracle):
    B, H, nh, ql, L = 1, 64, 2, 32, 7
    t = mla_inputs(B, H, nh, ql, L, 12, seed=5, poison=True)
    base = run(oracle, t, [L])
    assert np.isfinite(base["out"]).all()
    perm = torch.randperm(L, generator=torch.Generator().manual_seed(6))
    c = t["cache"].clone()
    c[0, :L] = t["cache"][0, perm]
    r = run(oracle, dict(t, cache=c), [L])
    np.testing.assert_allclose(r["out"], base["out"], rtol=1e-12, atol=1e-14)


def test_mla_brute_force_tiny(oracle):
    B, H, nh, ql, L, theta, eps = 1, 16, 2, 16, 2, 10000.0, 1e-6
    t = mla_inputs(B, H, nh, ql, L, 4, seed=7)
    r = run(oracle, t, [L], theta, eps)
    x, Wa, gq, gkv = f64(t["x"]), f64(t["W_a"]), f64(t["g_q"]), f64(t["g_kv"])
    Wuq, Wkvb, Wo, cache = f64(t["W_uq"]), f64(t["W_kvb"]), f64(t["W_o"]), f64(t["cache"])
    rb = lambda v: bits_to_f64(oracle.round_bf16(np.asarray(v, dtype=np.float64)))

    def rms(vv, g):
        s = math.sqrt(math.fsum(e * e for e in vv) / len(vv) + eps)
        return [g[i] * vv[i] / s for i in range(len(vv))]

    def rope(vv, pos):
        half = len(vv) // 2
        outv = list(vv)
        for i in range(half):
            ang = pos * theta ** (-2.0 * i / len(vv))
            outv[i] = vv[i] * math.cos(ang) - vv[i + half] * math.sin(ang)
            outv[i + half] = vv[i + half] * math.cos(ang) + vv[i] * math.sin(ang)
        return outv

    a = rb([math.fsum(x[0, i] * Wa[i, j] for i in range(H)) for j in range(ql + ROW)])
    cq = rb(rms(a[:ql], gq))
    q = rb([math.fsum(cq[i] * Wuq[i, j] for i in range(ql)) for j in range(nh * 192)])
    ckv = rb(rms(a[ql:ql + KV], gkv))
    kr = rb(rope(a[ql + KV:], L))
    rows = [list(cache[0, s]) for s in range(L)] + [list(ckv) + list(kr)]
    np.testing.assert_array_equal(r["new_row"][0], np.array(rows[L]))
    o = []
    for h in range(nh):
        qh = list(q[h * 192:h * 192 + NOPE]) + rope(list(q[h * 192 + NOPE:(h + 1) * 192]), L)
        ks, vs = [], []
        for c in rows:
            k = [math.fsum(c[i] * Wkvb[i, h * 256 + j] for i in range(KV)) for j in range(NOPE)]
            ks.append(k + c[KV:])
            vs.append([math.fsum(c[i] * Wkvb[i, h * 256 + NOPE + j] for i in range(KV))
                       for j in range(V)])
        s = [math.fsum(qh[j] * k[j] for j in range(192)) / math.sqrt(192) for k in ks]
        m = max(s)
        e = [math.exp(si - m) for si in s]
        den = math.fsum(e)
        o += [math.fsum(e[tt] * vs[tt][j] for tt in range(L + 1)) / den for j in range(V)]
    np.testing.assert_allclose(r["attn"][0], o, rtol=1e-11, atol=1e-13)
    v = rb(o)
    want = [math.fsum(v[i] * Wo[i, j] for i in range(nh * V)) for j in range(H)]
    np.testing.assert_allclose(r["out"][0], want, rtol=1e-11, atol=1e-13)


# The rotary frequencies of the 64 rope dims, omega_i = theta^(-2i/64), fixed
# by closed-form angles: at theta = 10000, pairs 8, 16 and 24 have the exact
# frequencies 10^-1, 10^-2 and 10^-3.
MLA_ROPE_PAIRS = [(8, 0.1), (16, 0.01), (24, 0.001)]


def _mla_zero_inputs(B, H, nh, q_lora, L, max_ctx):
    t = mla_inputs(B, H, nh, q_lora, L, max_ctx, seed=60)
    for k in ("x", "W_a", "W_uq", "W_kvb", "W_o", "cache"):
        t[k] = torch.zeros_like(t[k])
    t["g_q"] = torch.ones_like(t["g_q"])
    t["g_kv"] = torch.ones_like(t["g_kv"])
    return t


@pytest.mark.parametrize("i,w", MLA_ROPE_PAIRS)
@pytest.mark.parametrize("L", [1, 100, 4000])
def test_mla_key_rope_turns_by_the_closed_form_angle(oracle, i, w, L):
    """The new latent row's rope part is bf16(R(L) kr). With x = e_0 and W_a's
    row 0 = e at rope dim i, kr = e_i, so the row holds bf16(cos(L w_i)) at
    dim 512 + i and bf16(sin(L w_i)) at 512 + i + 32, zeros elsewhere."""
    H, q_lora = 64, 16
    t = _mla_zero_inputs(1, H, 1, q_lora, L, L + 1)
    t["x"][0, 0] = 1.0
    t["W_a"][0, q_lora + KV + i] = 1.0
    r = run(oracle, t, [L])
    a = L * w
    want = np.zeros(ROW)
    want[KV + i] = float(torch.tensor(math.cos(a)).to(torch.bfloat16))
    want[KV + i + ROPE // 2] = float(torch.tensor(math.sin(a)).to(torch.bfloat16))
    np.testing.assert_allclose(r["new_row"][0], want, rtol=0, atol=2.0 ** -9)


@pytest.mark.parametrize("i,w", MLA_ROPE_PAIRS)
def test_mla_query_rope_turns_by_the_closed_form_angle(oracle, i, w):
    """The query's rope part is rotated at the new token's position L. Setup
    (every other weight zero): q_rope = 8 e_i, q_nope = 0; cached row 0 holds
    latent e_0 (its value decompresses to all ones) and rope key e_i; cached
    rows 1..L-1 and the new row are zero. So the scores are
    s_0 = 8 cos(L w_i) / sqrt(192) and 0 for the L others, and every value dim
    of the head's output is e^(s_0) / (e^(s_0) + L)."""
    H, nh, q_lora, L = 64, 1, 16, 100
    t = _mla_zero_inputs(1, H, nh, q_lora, L, L + 1)
    t["x"][0, 0] = 1.0
    t["W_a"][0, 0] = 1.0          # a[0] = 1: cq = bf16(rmsnorm(e_0)) = 4 e_0 at q_lora 16
    t["W_uq"][0, NOPE + i] = 2.0  # q_rope = bf16(4 * 2) e_i = 8 e_i
    t["W_kvb"][0, NOPE:NOPE + V] = 1.0  # latent e_0 -> value of all ones
    t["cache"][0, 0, 0] = 1.0
    t["cache"][0, 0, KV + i] = 1.0
    r = run(oracle, t, [L])
    s0 = 8.0 * math.cos(L * w) / math.sqrt(NOPE + ROPE)
    p0 = math.exp(s0) / (math.exp(s0) + L)
    np.testing.assert_allclose(r["attn"][0], np.full(V, p0), rtol=1e-12)
