"""Pins for the fp64 oracle, each against something other than the oracle itself.

Every test here runs on the CPU (no GPU marker). The pins are chosen so that a
plausible slip anywhere in the oracle fails at least one of them:

  * dropped new token / wrong append position  -> ctx_len=0 closed form,
    worked example, poison-tail test
  * wrong Q/K/V column block                    -> zero-Q, zero-K, zero-V tests
  * transposed weight                           -> ctx_len=0 closed form (numpy
    matmul with the [in, out] orientation), worked example
  * wrong scale or sign in the softmax          -> two-key sigmoid closed form,
    worked example
  * missing normalisation                       -> equal-values and mean tests
  * wrong cache indexing / head mix-up          -> permutation, head-isolation,
    identity-weight tests
  * wrong split combine                         -> split == monolithic for 1..8
    splits with empty splits

Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命", written [CF §n].
"""
import math
import os

import numpy as np
import pytest
import torch

from out_proj_block_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


def rand_inputs(B, H, nh, d, L, max_ctx, seed):
    wl = workloads.custom(B, H, nh, d, L, max_ctx=max_ctx)
    return workloads.make_inputs(wl, seed=seed)


def rel_err(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ---------------------------------------------------------------- exactness


def test_widen_bf16_exact(oracle):
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x7F80, 0x0001, 0x3EAB],
                    dtype=np.uint16)
    w = oracle.widen(bits)
    assert w[0] == 1.0 and w[1] == -2.0 and w[2] == 0.0
    assert math.copysign(1.0, w[3]) == -1.0 and w[3] == 0.0
    assert w[4] == math.inf
    assert w[5] == 2.0 ** -133  # smallest bf16 subnormal
    assert w[6] == float(torch.tensor(0x3EAB, dtype=torch.int16).view(torch.bfloat16).item())


# ------------------------------------------------------------- closed forms


def test_worked_example_closed_form(oracle):
    """Hand-derived example in tests/golden/worked_example_d2.txt [CF §1.1, §5.1]."""
    rows = {}
    with open(os.path.join(GOLDEN, "worked_example_d2.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, *v = line.split()
                rows[k] = [float(t) for t in v]
    x = bf16([rows["x"]])
    W_qkv = bf16([rows["W_qkv_row0"], rows["W_qkv_row1"]])
    W_o = bf16([rows["W_o_row0"], rows["W_o_row1"]])
    kc = torch.full((1, 1, 2, 2), float("nan")).to(torch.bfloat16)
    vc = kc.clone()
    kc[0, 0, 0] = bf16(rows["k_cache_pos0"])
    vc[0, 0, 0] = bf16(rows["v_cache_pos0"])
    r = oracle.decode_step(x, W_qkv, W_o, kc, vc, ctx_len=1)

    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    a0 = 2.0 * sig(-math.sqrt(2.0))
    a1 = 4.0 * sig(math.sqrt(2.0))
    np.testing.assert_allclose(r["k_new"][0, 0], [0.0, 1.0], rtol=0, atol=0)
    np.testing.assert_allclose(r["v_new"][0, 0], [2.0, 0.0], rtol=0, atol=0)
    np.testing.assert_allclose(r["attn"][0, 0], [a0, a1], rtol=1e-14, atol=0)
    np.testing.assert_allclose(r["out"][0], [a0 + 3 * a1, 2 * a0 + 4 * a1],
                               rtol=1e-14, atol=0)


@pytest.mark.parametrize("d", [4, 16, 128])
def test_two_key_sigmoid(oracle, d):
    """T=2: a = sigma(D) v1 + (1 - sigma(D)) v2, D = q.(k1 - k2)/sqrt(d).

    Fixes the 1/sqrt(d) scale and the sign of the exponent.
    """
    rng = np.random.default_rng(d)
    q = rng.standard_normal(d)
    K = rng.standard_normal((2, d))
    V = rng.standard_normal((2, d))
    scale = 1.0 / math.sqrt(d)
    delta = float(np.dot(q, K[0] - K[1])) / math.sqrt(d)
    s = 1.0 / (1.0 + math.exp(-delta))
    a = oracle.attention(q, K, V, scale)
    np.testing.assert_allclose(a, s * V[0] + (1 - s) * V[1], rtol=1e-13, atol=1e-15)


def test_ctx0_output_is_projected_new_value(oracle):
    """ctx_len = 0: the only key is the new one, so attn = v_new and
    out = (x . W_v) . W_o, with W_v = columns [2H, 3H) of W_qkv [CF §1.1]."""
    B, H, nh, d = 3, 64, 4, 16
    t = rand_inputs(B, H, nh, d, 0, 8, seed=1)
    r = oracle.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], 0)
    x, Wqkv, Wo = f64(t["x"]), f64(t["W_qkv"]), f64(t["W_o"])
    v = x @ Wqkv[:, 2 * H:3 * H]
    np.testing.assert_allclose(r["attn"].reshape(B, H), v, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["v_new"].reshape(B, H), v, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["k_new"].reshape(B, H), x @ Wqkv[:, H:2 * H],
                               rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(r["out"], v @ Wo, rtol=1e-11, atol=1e-13)


def test_identity_weights_return_x(oracle):
    """nh=1, H=d, W_q=W_k=W_v=W_o=I, ctx_len=0: out = x exactly."""
    d = 16
    rng = np.random.default_rng(5)
    x = bf16(rng.standard_normal((2, d)))
    eye = np.eye(d, dtype=np.float32)
    W_qkv = bf16(np.concatenate([eye, eye, eye], axis=1))
    W_o = bf16(eye)
    kc = torch.zeros(2, 1, 4, d, dtype=torch.bfloat16)
    r = oracle.decode_step(x, W_qkv, W_o, kc, kc.clone(), 0)
    np.testing.assert_array_equal(r["out"], f64(x))


# --------------------------------------------------- which column is which


def _zero_block(W_qkv: torch.Tensor, blk: int) -> torch.Tensor:
    H = W_qkv.shape[0]
    W = W_qkv.clone()
    W[:, blk * H:(blk + 1) * H] = 0
    return W


def _values(t, b, h, L, v_new):
    V = f64(t["v_cache"][b, h, :L])
    return np.concatenate([V, v_new[None]], axis=0)


def test_zero_key_block_gives_mean_of_values(oracle):
    """K block (columns [H, 2H)) zero and cached keys zero: every score is 0,
    the softmax is uniform and attn = mean of the L+1 values."""
    B, H, nh, d, L = 2, 64, 2, 32, 9
    t = rand_inputs(B, H, nh, d, L, 16, seed=2)
    W = _zero_block(t["W_qkv"], 1)
    kc = torch.zeros_like(t["k_cache"])
    r = oracle.decode_step(t["x"], W, t["W_o"], kc, t["v_cache"], L)
    for b in range(B):
        for h in range(nh):
            mean = _values(t, b, h, L, r["v_new"][b, h]).mean(axis=0)
            np.testing.assert_allclose(r["attn"][b, h], mean, rtol=1e-12, atol=1e-14)


def test_zero_query_block_gives_mean_of_values(oracle):
    """Q block (columns [0, H)) zero with random keys: q = 0, uniform softmax.
    A Q/K mix-up would project a non-zero query and fail."""
    B, H, nh, d, L = 1, 64, 2, 32, 7
    t = rand_inputs(B, H, nh, d, L, 16, seed=3)
    W = _zero_block(t["W_qkv"], 0)
    r = oracle.decode_step(t["x"], W, t["W_o"], t["k_cache"], t["v_cache"], L)
    for h in range(nh):
        mean = _values(t, 0, h, L, r["v_new"][0, h]).mean(axis=0)
        np.testing.assert_allclose(r["attn"][0, h], mean, rtol=1e-12, atol=1e-14)


def test_zero_value_block_and_cache_gives_zero(oracle):
    """V block (columns [2H, 3H)) zero and cached values zero: out = 0 exactly."""
    B, H, nh, d, L = 2, 64, 4, 16, 5
    t = rand_inputs(B, H, nh, d, L, 8, seed=4)
    W = _zero_block(t["W_qkv"], 2)
    r = oracle.decode_step(t["x"], W, t["W_o"], t["k_cache"],
                           torch.zeros_like(t["v_cache"]), L)
    assert np.all(r["out"] == 0.0)
    assert np.all(r["v_new"] == 0.0)


# ---------------------------------------------------------------- invariants


def test_equal_values_are_returned(oracle):
    """All value rows equal to u: attn = u whatever the scores (normalisation)."""
    rng = np.random.default_rng(7)
    d, T = 32, 50
    u = rng.standard_normal(d)
    a = oracle.attention(rng.standard_normal(d) * 3, rng.standard_normal((T, d)),
                         np.tile(u, (T, 1)), 1 / math.sqrt(d))
    np.testing.assert_allclose(a, u, rtol=1e-13, atol=1e-14)


def test_identical_keys_give_mean(oracle):
    rng = np.random.default_rng(8)
    d, T = 64, 33
    k = rng.standard_normal(d)
    V = rng.standard_normal((T, d))
    a = oracle.attention(rng.standard_normal(d), np.tile(k, (T, 1)), V, 1 / math.sqrt(d))
    np.testing.assert_allclose(a, V.mean(axis=0), rtol=1e-12, atol=1e-14)


def test_dominant_key(oracle):
    """One key with a score gap G over all others: |a - v*| <= (T-1) e^-G max|v|."""
    rng = np.random.default_rng(9)
    d, T, star = 32, 40, 17
    q = np.zeros(d); q[0] = 1.0
    K = rng.standard_normal((T, d)) * 0.1
    K[star, 0] = 60.0 * math.sqrt(d)  # score gap ~ 60
    V = rng.standard_normal((T, d))
    a = oracle.attention(q, K, V, 1 / math.sqrt(d))
    scores = K @ q / math.sqrt(d)
    gap = scores[star] - np.max(np.delete(scores, star))
    bound = (T - 1) * math.exp(-gap) * np.abs(V).max() * 2
    assert np.abs(a - V[star]).max() <= bound + 1e-15


def test_shift_invariance(oracle):
    """Adding one vector c to every key shifts every score by q.c/sqrt(d)."""
    rng = np.random.default_rng(10)
    d, T = 16, 21
    q, K, V = rng.standard_normal(d), rng.standard_normal((T, d)), rng.standard_normal((T, d))
    c = rng.standard_normal(d) * 5
    a0 = oracle.attention(q, K, V, 1 / math.sqrt(d))
    a1 = oracle.attention(q, K + c, V, 1 / math.sqrt(d))
    np.testing.assert_allclose(a1, a0, rtol=1e-11, atol=1e-13)


def test_cache_permutation_invariance(oracle):
    """Permuting the cached positions (same permutation for K and V) leaves the
    step unchanged: attention is a set function of the (key, value) pairs."""
    B, H, nh, d, L = 2, 128, 2, 64, 37
    t = rand_inputs(B, H, nh, d, L, 40, seed=11)
    r0 = oracle.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], L)
    perm = torch.randperm(L, generator=torch.Generator().manual_seed(3))
    kc, vc = t["k_cache"].clone(), t["v_cache"].clone()
    kc[:, :, :L] = t["k_cache"][:, :, perm]
    vc[:, :, :L] = t["v_cache"][:, :, perm]
    r1 = oracle.decode_step(t["x"], t["W_qkv"], t["W_o"], kc, vc, L)
    np.testing.assert_allclose(r1["out"], r0["out"], rtol=1e-12, atol=1e-14)


def test_rows_beyond_ctx_len_are_not_read(oracle):
    B, H, nh, d, L = 1, 64, 2, 32, 6
    wl = workloads.custom(B, H, nh, d, L, max_ctx=16)
    t = workloads.make_inputs(wl, seed=12, poison_tail=True)
    r = oracle.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], L)
    assert np.isfinite(r["out"]).all()


def test_head_isolation_and_per_head_assembly(oracle):
    """Each head's attention equals monolithic attention over its own q, keys and
    values, assembled here with numpy slicing; W_o with only head h's row block
    non-zero gives out = attn_h . W_o[h*d:(h+1)*d]."""
    B, H, nh, d, L = 2, 96, 3, 32, 11
    t = rand_inputs(B, H, nh, d, L, 16, seed=13)
    x, Wqkv = f64(t["x"]), f64(t["W_qkv"])
    for h in range(nh):
        Wo = t["W_o"].clone()
        Wo[:h * d] = 0
        Wo[(h + 1) * d:] = 0
        r = oracle.decode_step(t["x"], t["W_qkv"], Wo, t["k_cache"], t["v_cache"], L)
        for b in range(B):
            cols = slice(h * d, (h + 1) * d)
            q = x[b] @ Wqkv[:, cols]
            k = x[b] @ Wqkv[:, H:][:, cols]
            v = x[b] @ Wqkv[:, 2 * H:][:, cols]
            K = np.concatenate([f64(t["k_cache"][b, h, :L]), k[None]])
            V = np.concatenate([f64(t["v_cache"][b, h, :L]), v[None]])
            a = oracle.attention(q, K, V, 1 / math.sqrt(d))
            np.testing.assert_allclose(r["attn"][b, h], a, rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(r["out"][b], a @ f64(Wo)[cols], rtol=1e-11,
                                       atol=1e-14)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8])
def test_split_combine_equals_monolithic(oracle, n):
    """Split-KV partials combined by max-then-sum [CF §3.1.1, §3.2] reproduce the
    monolithic softmax for any split, including empty splits."""
    rng = np.random.default_rng(100 + n)
    d, T = 32, 29
    q, K, V = rng.standard_normal(d) * 2, rng.standard_normal((T, d)), rng.standard_normal((T, d))
    scale = 1 / math.sqrt(d)
    cuts = np.sort(rng.integers(0, T + 1, size=n - 1)) if n > 1 else np.array([], int)
    if n >= 3:
        cuts[1] = cuts[0]  # force an empty split
    bounds = [0, *cuts.tolist(), T]
    ms, ls, os_ = [], [], []
    for r in range(n):
        m, l, o = oracle.split_partial(q, K, V, bounds[r], bounds[r + 1], scale)
        if bounds[r] == bounds[r + 1]:
            assert m == -math.inf and l == 0.0 and not o.any()
        ms.append(m); ls.append(l); os_.append(o)
    a = oracle.split_combine(ms, ls, np.stack(os_))
    np.testing.assert_allclose(a, oracle.attention(q, K, V, scale), rtol=1e-12, atol=1e-14)


# ----------------------------------------------------- brute force, tiny


def _brute(x, Wqkv, Wo, kc, vc, L):
    """Exactly-rounded sums (math.fsum) over Python floats, tiny shapes only."""
    B, H = x.shape
    _, nh, _, d = kc.shape
    out = np.zeros((B, H))
    for b in range(B):
        a = []
        for h in range(nh):
            col = lambda blk, j: blk * H + h * d + j
            q = [math.fsum(x[b, i] * Wqkv[i, col(0, j)] for i in range(H)) for j in range(d)]
            k = [math.fsum(x[b, i] * Wqkv[i, col(1, j)] for i in range(H)) for j in range(d)]
            v = [math.fsum(x[b, i] * Wqkv[i, col(2, j)] for i in range(H)) for j in range(d)]
            keys = [list(kc[b, h, t]) for t in range(L)] + [k]
            vals = [list(vc[b, h, t]) for t in range(L)] + [v]
            s = [math.fsum(q[j] * kk[j] for j in range(d)) / math.sqrt(d) for kk in keys]
            m = max(s)
            e = [math.exp(si - m) for si in s]
            den = math.fsum(e)
            a += [math.fsum(e[t] * vals[t][j] for t in range(L + 1)) / den for j in range(d)]
        for j in range(H):
            out[b, j] = math.fsum(a[r] * Wo[r, j] for r in range(H))
    return out


@pytest.mark.parametrize("B,H,nh,d,L", [(1, 8, 2, 4, 3), (2, 12, 3, 4, 5), (1, 16, 1, 16, 0)])
def test_brute_force_tiny(oracle, B, H, nh, d, L):
    t = rand_inputs(B, H, nh, d, L, 8, seed=20 + L)
    r = oracle.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], L)
    ref = _brute(f64(t["x"]), f64(t["W_qkv"]), f64(t["W_o"]), f64(t["k_cache"]),
                 f64(t["v_cache"]), L)
    np.testing.assert_allclose(r["out"], ref, rtol=1e-12, atol=1e-15)


def test_threads_do_not_change_result(oracle):
    B, H, nh, d, L = 3, 128, 4, 32, 20
    t = rand_inputs(B, H, nh, d, L, 32, seed=30)
    r1 = oracle.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], L, 1)
    r4 = oracle.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], L, 4)
    for k in ("out", "k_new", "v_new", "attn"):
        np.testing.assert_array_equal(r1[k], r4[k])


def test_rejects_bad_arguments(oracle):
    t = rand_inputs(1, 64, 2, 32, 3, 4, seed=31)
    with pytest.raises(ValueError):
        oracle.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], 4)


# ------------------------------------- rotary embedding and ragged lengths


def test_rope_position_zero_is_identity(oracle):
    x = np.random.default_rng(40).standard_normal(128)
    np.testing.assert_array_equal(oracle.rope(x, 0, 10000.0), x)


@pytest.mark.parametrize("pos", [1, 7, 1000, 16383])
def test_rope_d2_is_a_plain_rotation(oracle, pos):
    """d = 2: one pair, frequency theta^0 = 1, so the angle is pos radians."""
    x = np.array([0.6, -1.3])
    c, s = math.cos(pos), math.sin(pos)
    np.testing.assert_allclose(oracle.rope(x, pos, 10000.0),
                               [x[0] * c - x[1] * s, x[1] * c + x[0] * s], rtol=0, atol=1e-15)


# The frequency schedule of the rotate-half reading, omega_i = theta^(-2i/d),
# fixed by angles written out in closed form (not by re-evaluating the
# oracle's own expression): with theta = 10000 and d = 8 the frequencies are
# exactly 10^-i, with d = 4 they are 1 and 10^-2. A schedule such as
# theta^(-i/d), or one pairing i with d-1-i, gives other angles.
ROPE_SCHEDULES = [
    # (d, theta, pos, [angle of pair i])
    (4, 10000.0, 1, [1.0, 0.01]),
    (4, 10000.0, 250, [250.0, 2.5]),
    (8, 10000.0, 4095, [4095.0, 409.5, 40.95, 4.095]),
    (8, 10000.0, 1, [1.0, 0.1, 0.01, 0.001]),
    (4, 500.0, 3, [3.0, 3.0 / math.sqrt(500.0)]),
    (6, 1000.0, 7, [7.0, 0.7, 0.07]),
]


@pytest.mark.parametrize("d,theta,pos,angles", ROPE_SCHEDULES)
def test_rope_frequency_schedule_closed_form(oracle, d, theta, pos, angles):
    """Basis vector e_i goes to cos(a_i) e_i + sin(a_i) e_(i+d/2), and e_(i+d/2)
    to -sin(a_i) e_i + cos(a_i) e_(i+d/2), with a_i = pos * theta^(-2i/d)."""
    half = d // 2
    for i, a in enumerate(angles):
        e = np.zeros(d)
        e[i] = 1.0
        want = np.zeros(d)
        want[i], want[i + half] = math.cos(a), math.sin(a)
        np.testing.assert_allclose(oracle.rope(e, pos, theta), want, rtol=0, atol=1e-12)
        e = np.zeros(d)
        e[i + half] = 1.0
        want = np.zeros(d)
        want[i], want[i + half] = -math.sin(a), math.cos(a)
        np.testing.assert_allclose(oracle.rope(e, pos, theta), want, rtol=0, atol=1e-12)


def test_rope_frequency_schedule_head_dim_128(oracle):
    """d = 128, theta = 10000: pair i turns by pos * 10^(-4i/64); pairs 16, 32
    and 48 have the exact frequencies 10^-1, 10^-2 and 10^-3."""
    d, pos = 128, 4095
    for i, w in ((0, 1.0), (16, 0.1), (32, 0.01), (48, 0.001)):
        e = np.zeros(d)
        e[i] = 1.0
        y = oracle.rope(e, pos, 10000.0)
        assert y[i] == pytest.approx(math.cos(pos * w), abs=1e-11)
        assert y[i + d // 2] == pytest.approx(math.sin(pos * w), abs=1e-11)


def test_rope_in_the_step_rotates_by_the_closed_form_angle(oracle):
    """Through decode_step_ex: one head, d = 4, the new key is x . W_k with
    x = e_0 and W_k's row 0 = e_1, so k_new = R(L) e_1 = cos(0.01 L) e_1 +
    sin(0.01 L) e_3 at theta = 10000 (pair 1's frequency is 10000^(-1/2))."""
    B, H, nh, d, L = 1, 4, 1, 4, 37
    t = rand_inputs(B, H, nh, d, L, 64, seed=45)
    x = np.zeros((B, H), np.float32)
    x[0, 0] = 1.0
    W = np.zeros((H, 3 * H), np.float32)
    W[0, H + 1] = 1.0
    t["x"], t["W_qkv"] = bf16(x), bf16(W)
    r = oracle.decode_step_ex(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], [L],
                              rope_theta=10000.0)
    a = 0.01 * L
    np.testing.assert_allclose(r["k_new"][0, 0], [0.0, math.cos(a), 0.0, math.sin(a)],
                               rtol=0, atol=1e-13)


def test_rope_pairs_dimension_i_with_i_plus_half(oracle):
    """Rotate-half convention: basis vector e_i only mixes with e_{i+d/2}."""
    d = 16
    for i in range(d // 2):
        e = np.zeros(d)
        e[i] = 1.0
        y = oracle.rope(e, 5, 10000.0)
        nz = set(np.nonzero(np.abs(y) > 1e-15)[0].tolist())
        assert nz <= {i, i + d // 2}


def test_rope_preserves_norm_and_relative_position(oracle):
    rng = np.random.default_rng(41)
    d = 128
    q, k = rng.standard_normal(d), rng.standard_normal(d)
    for pos in (3, 333, 4096):
        assert np.linalg.norm(oracle.rope(q, pos, 10000.0)) == pytest.approx(np.linalg.norm(q), rel=1e-13)
    base = np.dot(oracle.rope(q, 100, 10000.0), oracle.rope(k, 40, 10000.0))
    for shift in (1, 17, 2000):
        shifted = np.dot(oracle.rope(q, 100 + shift, 10000.0), oracle.rope(k, 40 + shift, 10000.0))
        assert shifted == pytest.approx(base, rel=1e-10, abs=1e-10)


def test_ex_without_rope_equals_uniform_step(oracle):
    B, H, nh, d, L = 3, 128, 2, 64, 20
    t = rand_inputs(B, H, nh, d, L, 32, seed=42)
    a = oracle.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], L)
    b = oracle.decode_step_ex(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], [L] * B)
    for key in ("out", "k_new", "v_new", "attn"):
        np.testing.assert_array_equal(a[key], b[key])


def test_ragged_rows_are_independent_sequences(oracle):
    """Each batch row with its own ctx_len equals a one-row step at that length."""
    B, H, nh, d = 3, 128, 2, 64
    lens = [0, 13, 31]
    t = rand_inputs(B, H, nh, d, 31, 32, seed=43)
    r = oracle.decode_step_ex(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], lens,
                              rope_theta=10000.0)
    for b, L in enumerate(lens):
        one = oracle.decode_step_ex(t["x"][b:b + 1], t["W_qkv"], t["W_o"], t["k_cache"][b:b + 1],
                                    t["v_cache"][b:b + 1], [L], rope_theta=10000.0)
        np.testing.assert_array_equal(r["out"][b], one["out"][0])


def test_rope_step_is_attention_over_rotated_q_and_new_key(oracle):
    """Assembled by hand: q and k_new projected with numpy, rotated at their
    position, attended against the cached (already rotated) keys."""
    B, H, nh, d = 2, 128, 2, 64
    lens = [9, 30]
    t = rand_inputs(B, H, nh, d, 30, 32, seed=44)
    r = oracle.decode_step_ex(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], lens,
                              rope_theta=500.0)
    x, Wqkv = f64(t["x"]), f64(t["W_qkv"])
    for b, L in enumerate(lens):
        for h in range(nh):
            cols = slice(h * d, (h + 1) * d)
            q = oracle.rope(x[b] @ Wqkv[:, cols], L, 500.0)
            k = oracle.rope(x[b] @ Wqkv[:, H:][:, cols], L, 500.0)
            v = x[b] @ Wqkv[:, 2 * H:][:, cols]
            K = np.concatenate([f64(t["k_cache"][b, h, :L]), k[None]])
            V = np.concatenate([f64(t["v_cache"][b, h, :L]), v[None]])
            np.testing.assert_allclose(r["k_new"][b, h], k, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(r["attn"][b, h], oracle.attention(q, K, V, 1 / math.sqrt(d)),
                                       rtol=1e-12, atol=1e-14)
