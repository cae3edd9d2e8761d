"""Pins for the decoder-layer part of the fp64 oracle (RMSNorm, SwiGLU MLP,
residuals, bf16 storage rounding, the multi-layer multi-token loop), each
against something other than the oracle itself. CPU only.

A plausible slip and the pin that catches it:
  * rounding twice (double -> float -> bf16)   -> the double-rounding trap
  * wrong tie or overflow rule                 -> torch's float->bf16 on floats,
                                                  hand-made ties, overflow cases
  * eps outside the sqrt, sum instead of mean  -> closed value with eps, unit
                                                  mean square
  * norm weight ignored or applied twice       -> linearity in g
  * silu on the wrong branch (up vs gate)      -> scalar closed form
  * gate/up/down index mismatch                -> permutation equivariance
  * activation after the down projection       -> doubling W_down doubles delta
  * residual dropped or taken from xn          -> zero-weight identities, the
                                                  scale-invariance test
  * appended row missing or at the wrong place -> NaN-poisoned cache tails
  * anything else in a tiny layer              -> brute force with math.fsum

Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命", written [CF §n]; the
norm/MLP part of a layer is the Llama2 arrangement, a reading (the page shows
only the attention block).
"""
import math

import numpy as np
import pytest
import torch

from out_proj_block_gb300 import workloads


def bits_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def torch_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def to_bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


# ------------------------------------------------------------- bf16 rounding


def test_round_matches_torch_on_float_values(oracle):
    g = torch.Generator().manual_seed(5)
    e = torch.randint(-140, 127, (20000,), generator=g).float()
    v = (torch.rand(20000, generator=g) + 1.0) * torch.pow(2.0, e)
    v[::2] *= -1
    v = torch.cat([v, torch.tensor([0.0, 1.0, -1.0, 2.0 ** -133, 3.3895314e38])])
    want = torch_bits(v.to(torch.bfloat16))
    got = oracle.round_bf16(v.double().numpy())
    np.testing.assert_array_equal(got, want)


def test_round_ties_to_even_and_no_double_rounding(oracle):
    r = oracle.round_bf16([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -30, -(1 + 2 ** -8)])
    assert list(r) == [0x3F80, 0x3F82, 0x3F81, 0xBF80]


def test_round_overflow_zero_nan(oracle):
    top = (2 - 2 ** -7) * 2.0 ** 127          # largest finite bf16
    half = (2 - 2 ** -8) * 2.0 ** 127         # halfway to 2^128: ties to the even 2^128
    r = oracle.round_bf16([top, half, np.nextafter(half, 0), -half, -0.0, 2.0 ** -134,
                           3 * 2.0 ** -134, float("nan")])
    assert list(r[:7]) == [0x7F7F, 0x7F80, 0x7F7F, 0xFF80, 0x8000, 0x0000, 0x0002]
    assert (r[7] & 0x7F80) == 0x7F80 and (r[7] & 0x7F) != 0


# ------------------------------------------------------------------ RMSNorm


def test_rmsnorm_eps_sits_inside_the_root(oracle):
    y = oracle.rmsnorm([1.0, 1.0, 1.0, 1.0], [1.0] * 4, eps=3.0)
    np.testing.assert_allclose(y, [0.5] * 4, rtol=1e-15)


def test_rmsnorm_unit_mean_square_and_scale_invariance(oracle):
    rng = np.random.default_rng(3)
    x = rng.standard_normal(333)
    g = np.ones(333)
    y = oracle.rmsnorm(x, g, 0.0)
    assert abs(np.mean(y * y) - 1.0) < 1e-14
    np.testing.assert_allclose(oracle.rmsnorm(7.5 * x, g, 0.0), y, rtol=1e-14)
    np.testing.assert_allclose(oracle.rmsnorm(-x, g, 0.0), -y, rtol=1e-15)
    # eps matters only against the mean square: x = 0 stays finite
    assert not oracle.rmsnorm(np.zeros(8), np.ones(8), 1e-5).any()


def test_rmsnorm_is_linear_in_the_weight(oracle):
    rng = np.random.default_rng(4)
    x, g1, g2 = rng.standard_normal((3, 64))
    np.testing.assert_allclose(oracle.rmsnorm(x, g1 * g2, 1e-3),
                               g1 * oracle.rmsnorm(x, g2, 1e-3), rtol=1e-13, atol=1e-15)


def test_rmsnorm_bf16_constant_rows_give_the_weight(oracle):
    g = to_bf16(np.linspace(0.5, 1.5, 40))
    x = to_bf16(np.vstack([np.full(40, 3.0), np.full(40, -0.125)]))
    y = oracle.rmsnorm_bf16(x, g, 0.0)
    np.testing.assert_array_equal(y[0], torch_bits(g))
    np.testing.assert_array_equal(y[1], torch_bits(-g))


# --------------------------------------------------------------------- SiLU


def test_silu_closed_forms(oracle):
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(math.log(3.0)) - 0.75 * math.log(3.0)) < 1e-15  # sigma(ln 3) = 3/4
    for z in (0.3, 1.7, 6.0, 25.0):
        assert abs(oracle.silu(z) - oracle.silu(-z) - z) < 1e-14 * max(1.0, z)
    assert 0 > oracle.silu(-40.0) > -1e-15
    assert abs(oracle.silu(40.0) - 40.0) < 1e-15


# ---------------------------------------------------------------------- MLP


def _mlp_inputs(B, H, F, seed):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn(B, H, generator=g).to(torch.bfloat16)
    nw = (1.0 + 0.1 * torch.randn(H, generator=g)).to(torch.bfloat16)
    Wg = (0.3 * torch.randn(H, F, generator=g)).to(torch.bfloat16)
    Wu = (0.3 * torch.randn(H, F, generator=g)).to(torch.bfloat16)
    Wd = (0.3 * torch.randn(F, H, generator=g)).to(torch.bfloat16)
    return h, nw, Wg, Wu, Wd


def test_mlp_scalar_closed_form(oracle):
    h, g = to_bf16([[2.0]]), to_bf16([1.5])
    Wg, Wu, Wd = to_bf16([[2.0]]), to_bf16([[0.5]]), to_bf16([[0.25]])
    r = oracle.mlp(h, g, Wg, Wu, Wd, eps=0.0)
    # hn = 1.5 * 2 / |2| = 1.5; gate = 3, up = 0.75; u = silu(3) * 0.75
    u = 3.0 / (1.0 + math.exp(-3.0)) * 0.75
    u_b = bits_to_f64(oracle.round_bf16([u]))[0]
    assert bits_to_f64(r["u"])[0, 0] == u_b
    assert r["delta"][0, 0] == u_b * 0.25
    assert bits_to_f64(r["y"])[0, 0] == bits_to_f64(oracle.round_bf16([2.0 + u_b * 0.25]))[0]


def test_mlp_zero_down_or_up_returns_residual(oracle):
    h, g, Wg, Wu, Wd = _mlp_inputs(2, 48, 80, seed=6)
    for args in ((Wg, Wu, torch.zeros_like(Wd)), (Wg, torch.zeros_like(Wu), Wd)):
        r = oracle.mlp(h, g, *args, eps=1e-5)
        np.testing.assert_array_equal(r["y"], torch_bits(h))
        assert not r["delta"].any()


def test_mlp_permuting_the_hidden_units_changes_nothing(oracle):
    h, g, Wg, Wu, Wd = _mlp_inputs(2, 40, 72, seed=7)
    perm = torch.randperm(72, generator=torch.Generator().manual_seed(8))
    a = oracle.mlp(h, g, Wg, Wu, Wd, eps=1e-5)
    b = oracle.mlp(h, g, Wg[:, perm], Wu[:, perm], Wd[perm, :], eps=1e-5)
    np.testing.assert_array_equal(b["u"], a["u"][:, perm.numpy()])
    np.testing.assert_allclose(b["delta"], a["delta"], rtol=1e-12, atol=1e-14)


def test_mlp_delta_is_linear_in_down(oracle):
    h, g, Wg, Wu, Wd = _mlp_inputs(1, 32, 64, seed=9)
    a = oracle.mlp(h, g, Wg, Wu, Wd, eps=1e-5)
    b = oracle.mlp(h, g, Wg, Wu, (Wd.float() * 2).to(torch.bfloat16), eps=1e-5)
    np.testing.assert_array_equal(b["delta"], 2 * a["delta"])


def test_mlp_brute_force_tiny(oracle):
    B, H, F, eps = 2, 6, 10, 1e-5
    h, g, Wg, Wu, Wd = _mlp_inputs(B, H, F, seed=10)
    r = oracle.mlp(h, g, Wg, Wu, Wd, eps=eps)
    hf, gf = h.double().numpy(), g.double().numpy()
    Wgf, Wuf, Wdf = Wg.double().numpy(), Wu.double().numpy(), Wd.double().numpy()
    for b in range(B):
        ms = math.fsum(v * v for v in hf[b]) / H
        hn = [gf[i] * hf[b, i] / math.sqrt(ms + eps) for i in range(H)]
        hn = bits_to_f64(oracle.round_bf16(hn))
        u = []
        for j in range(F):
            gate = math.fsum(hn[i] * Wgf[i, j] for i in range(H))
            up = math.fsum(hn[i] * Wuf[i, j] for i in range(H))
            u.append(gate / (1.0 + math.exp(-gate)) * up)
        u = bits_to_f64(oracle.round_bf16(u))
        np.testing.assert_array_equal(bits_to_f64(r["u"][b]), u)
        delta = [math.fsum(u[j] * Wdf[j, k] for j in range(F)) for k in range(H)]
        np.testing.assert_allclose(r["delta"][b], delta, rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- one layer


def _layer_inputs(B, H, nh, d, F, L, max_ctx, seed, poison=False):
    wl = workloads.custom_stack(1, B, H, nh, d, F, L, max_ctx=max_ctx)
    t = workloads.make_stack_inputs(wl, seed=seed, poison_tail=poison)
    return t["x"], t["layers"][0]


def test_layer_with_zero_output_weights_is_the_identity(oracle):
    x, layer = _layer_inputs(2, 64, 2, 32, 96, 5, 8, seed=11)
    layer = dict(layer, W_o=torch.zeros_like(layer["W_o"]), W_down=torch.zeros_like(layer["W_down"]))
    r = oracle.layer_step(x, layer, layer["k_cache"], layer["v_cache"], [5, 3], 10000.0, 1e-5)
    np.testing.assert_array_equal(r["y"], torch_bits(x))
    np.testing.assert_array_equal(r["h"], torch_bits(x))


def test_layer_wiring(oracle):
    """xn feeds the attention block, x (not xn) is the residual, h feeds the MLP."""
    B, H, nh, d, F, L = 2, 64, 2, 32, 96, 6
    x, layer = _layer_inputs(B, H, nh, d, F, L, 8, seed=12)
    lens = [L, 2]
    r = oracle.layer_step(x, layer, layer["k_cache"], layer["v_cache"], lens, 10000.0, 1e-5)
    xn = oracle.rmsnorm_bf16(x, layer["attn_norm"], 1e-5)
    np.testing.assert_array_equal(r["xn"], xn)
    att = oracle.decode_step_ex(xn, layer["W_qkv"], layer["W_o"], layer["k_cache"],
                                layer["v_cache"], lens, 10000.0)
    np.testing.assert_array_equal(r["h"], oracle.round_bf16(x.double().numpy() + att["out"]))
    np.testing.assert_array_equal(r["k_new"], att["k_new"])
    m = oracle.mlp(r["h"], layer["mlp_norm"], layer["W_gate"], layer["W_up"], layer["W_down"], 1e-5)
    np.testing.assert_array_equal(r["y"], m["y"])
    np.testing.assert_array_equal(r["u"], m["u"])


def test_layer_input_scale_reaches_only_the_residual(oracle):
    """rmsnorm makes the attention and the MLP input blind to the scale of x
    (eps = 0), so 4x gives the same xn and attention output and moves only the
    residual term."""
    x, layer = _layer_inputs(1, 64, 2, 32, 64, 4, 8, seed=13)
    x4 = (x.float() * 4).to(torch.bfloat16)
    a = oracle.layer_step(x, layer, layer["k_cache"], layer["v_cache"], [4], 0.0, 0.0)
    b = oracle.layer_step(x4, layer, layer["k_cache"], layer["v_cache"], [4], 0.0, 0.0)
    np.testing.assert_array_equal(a["xn"], b["xn"])
    np.testing.assert_array_equal(a["k_new"], b["k_new"])


# ------------------------------------------------- multi-layer decode loop


def test_stack_appends_each_layers_row_where_the_next_token_reads_it(oracle):
    wl = workloads.custom_stack(2, 2, 64, 2, 32, 96, 3, max_ctx=8)
    t = workloads.make_stack_inputs(wl, seed=14, poison_tail=True)
    caches = [(torch_bits(l["k_cache"]).copy(), torch_bits(l["v_cache"]).copy())
              for l in t["layers"]]
    x = torch_bits(t["x"])
    for step in range(4):  # tokens at positions 3, 4, 5, 6; rows >= position hold NaN
        lens = [3 + step, 3 + step]
        y, per = oracle.stack_step(x, t["layers"], caches, lens, 10000.0, 1e-5)
        assert np.isfinite(bits_to_f64(y)).all()
        for (kc, vc), r in zip(caches, per):
            np.testing.assert_array_equal(kc[:, :, 3 + step, :], oracle.round_bf16(r["k_new"]))
            np.testing.assert_array_equal(vc[:, :, 3 + step, :], oracle.round_bf16(r["v_new"]))
        x = y
    # the rows after the last token are still untouched (NaN)
    assert np.isnan(bits_to_f64(caches[0][0][:, :, 7, :])).all()


def test_stack_of_identity_layers_returns_x(oracle):
    wl = workloads.custom_stack(3, 1, 64, 2, 32, 64, 4, max_ctx=8)
    t = workloads.make_stack_inputs(wl, seed=15)
    layers = [dict(l, W_o=torch.zeros_like(l["W_o"]), W_down=torch.zeros_like(l["W_down"]))
              for l in t["layers"]]
    caches = [(torch_bits(l["k_cache"]).copy(), torch_bits(l["v_cache"]).copy()) for l in layers]
    y, _ = oracle.stack_step(t["x"], layers, caches, [4], 10000.0, 1e-5)
    np.testing.assert_array_equal(y, torch_bits(t["x"]))


def test_layer_threads_do_not_change_result(oracle):
    x, layer = _layer_inputs(2, 128, 4, 32, 192, 9, 16, seed=16)
    a = oracle.layer_step(x, layer, layer["k_cache"], layer["v_cache"], [9, 5], 10000.0, 1e-5, 1)
    b = oracle.layer_step(x, layer, layer["k_cache"], layer["v_cache"], [9, 5], 10000.0, 1e-5, 4)
    for k in ("xn", "h", "u", "y", "k_new", "v_new"):
        np.testing.assert_array_equal(a[k], b[k])
