"""GPU parity of the multi-head latent attention step against the fp64 oracle,
through the C ABI.

Tolerance as for the attention block (relative L2 <= 5e-3, max abs <= 3e-2 on
unit-scale values; the max-abs bound is applied after dividing by
max(1, rms(ref))), separately for `out`, the value concat v (the input of the
output projection) and the appended latent row. Cache rows past each position
hold NaN, so a stray read shows as a non-finite result.
"""
import os

import numpy as np
import pytest
import torch

from out_proj_block_gb300 import workloads

pytestmark = pytest.mark.gpu

REL_L2 = 5e-3
MAX_ABS = 3e-2
NTHREADS = os.cpu_count() or 1
THETA = 10000.0
EPS = 1e-6


@pytest.fixture(scope="module")
def cfa():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from out_proj_block_gb300 import build
    build.build()
    from out_proj_block_gb300 import cfa as mod
    return mod


def check_close(name, got, ref, rel=REL_L2, max_abs=MAX_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    scale = max(1.0, float(np.sqrt(np.mean(ref * ref))))
    e_rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    e_abs = float(np.abs(got - ref).max()) / scale
    print(f"{name}: rel L2 {e_rel:.3e}, max abs/scale {e_abs:.3e}")
    assert e_rel <= rel and e_abs <= max_abs, (
        f"{name}: rel L2 {e_rel:.3e} (<= {rel}), max abs {e_abs:.3e} (<= {max_abs})")


def run_mla(cfa, oracle, wl, lens, seed=1, theta=THETA, splits=None):
    t = workloads.make_mla_inputs(wl, seed=seed, device="cpu")
    # NaN past each sequence's own position
    for b, L in enumerate(lens):
        t["cache"][b, L:] = float("nan")
    dev = {k: v.cuda() for k, v in t.items()}
    cache_before = dev["cache"].clone()
    out = torch.empty(wl.B, wl.hidden, dtype=torch.bfloat16, device="cuda")
    mla = cfa.Mla(wl.B, wl.hidden, wl.n_heads, wl.q_lora, wl.max_ctx)
    if splits is not None:
        mla.set_row_splits(splits)
    mla.step(dev["x"], dev, dev["cache"], lens, out, theta, EPS)
    torch.cuda.synchronize()
    assert mla.status() == cfa.CFA_OK
    ref = oracle.mla_step(t["x"], t["W_a"], t["g_q"], t["g_kv"], t["W_uq"], t["W_kvb"], t["W_o"],
                          t["cache"], lens, theta, EPS, NTHREADS)
    check_close("out", out.double().cpu().numpy(), ref["out"])
    rows = np.stack([dev["cache"][b, L].double().cpu().numpy() for b, L in enumerate(lens)])
    check_close("appended latent row", rows, ref["new_row"])
    # every other cache row is untouched
    after = dev["cache"].view(torch.int16).clone()
    before = cache_before.view(torch.int16).clone()
    for b, L in enumerate(lens):
        after[b, L] = 0
        before[b, L] = 0
    assert torch.equal(after, before)
    return mla, dev, out, ref


@pytest.mark.parametrize("B,H,nh,ql,L", [(1, 256, 2, 128, 64), (1, 512, 4, 128, 100),
                                         (2, 512, 16, 192, 257), (3, 1024, 32, 256, 33),
                                         (1, 256, 8, 64, 0), (2, 256, 4, 128, 1)])
def test_mla_matches_oracle(cfa, oracle, B, H, nh, ql, L):
    wl = workloads.custom_mla(B, H, nh, ql, L)
    lens = [max(0, L - 7 * b) for b in range(B)]
    run_mla(cfa, oracle, wl, lens, seed=B + nh + L)


def test_mla_many_heads_per_block(cfa, oracle):
    """More clusters than fit at 16 blocks each: smaller clusters, several
    heads finished per block."""
    wl = workloads.custom_mla(4, 1024, 128, 256, 100)
    lens = [100, 37, 64, 5]
    mla, _, _, _ = run_mla(cfa, oracle, wl, lens, seed=11)
    d = mla.describe()
    assert d["heads_per_cluster"] == 16 and d["cluster_size"] < 16
    assert d["coresident_clusters"] >= d["grid"] // d["cluster_size"]


@pytest.mark.parametrize("splits", [1, 2, 4])
@pytest.mark.parametrize("B,H,nh,ql,L", [(1, 512, 16, 128, 300), (2, 256, 4, 128, 0),
                                         (3, 1024, 32, 256, 77), (1, 256, 2, 64, 1)])
def test_mla_row_splits(cfa, oracle, B, H, nh, ql, L, splits):
    """One or two clusters per (sequence, head group), each over its share of
    the latent rows, the later of two combining them in split order: ctx 0
    (the first split has no rows), ctx 1, ragged lengths across sequences."""
    wl = workloads.custom_mla(B, H, nh, ql, L)
    lens = [max(0, L - 5 * b) for b in range(B)]
    probe = cfa.Mla(wl.B, wl.hidden, wl.n_heads, wl.q_lora, wl.max_ctx)
    try:
        probe.set_row_splits(splits)
    except cfa.CfaError:
        pytest.skip(f"{splits} row splits do not fit on this GPU for this shape")
    finally:
        probe.close()
    mla, dev, out, _ = run_mla(cfa, oracle, wl, lens, seed=20 + B + L, splits=splits)
    assert mla.describe()["row_splits"] == splits
    first = out.clone()
    for _ in range(2):  # the split counters are reset by the combining block
        mla.step(dev["x"], dev, dev["cache"], lens, out, THETA, EPS)
    torch.cuda.synchronize()
    assert mla.status() == cfa.CFA_OK
    assert torch.equal(first.view(torch.int16), out.view(torch.int16))


def test_mla_rejects_bad_row_splits(cfa):
    mla = cfa.Mla(1, 256, 4, 128, 64)
    for bad in (3, 8, -1):
        with pytest.raises(cfa.CfaError):
            mla.set_row_splits(bad)
    mla.set_row_splits(0)  # back to the per-step choice


def test_mla_long_context_splits_rows(cfa):
    """At ctx 16384 the per-step choice splits the latent rows over more
    blocks; the result equals the unsplit one within rounding."""
    wl = workloads.custom_mla(1, 512, 16, 128, 16384)
    t = {k: v.cuda() for k, v in workloads.make_mla_inputs(wl, seed=31).items()}
    outs, descs = [], []
    for splits in (0, 1):
        cache = t["cache"].clone()
        out = torch.empty(1, wl.hidden, dtype=torch.bfloat16, device="cuda")
        mla = cfa.Mla(1, wl.hidden, wl.n_heads, wl.q_lora, wl.max_ctx)
        if splits:
            mla.set_row_splits(splits)
        mla.step(t["x"], t, cache, [16384], out, THETA, EPS)
        torch.cuda.synchronize()
        assert mla.status() == cfa.CFA_OK
        outs.append(out.double().cpu().numpy())
        descs.append(mla.describe())
    assert descs[0]["row_splits"] > 1 and descs[1]["row_splits"] == 1
    check_close("auto vs unsplit", outs[0], outs[1])


def test_mla_without_rope(cfa, oracle):
    wl = workloads.custom_mla(1, 512, 16, 128, 300)
    run_mla(cfa, oracle, wl, [300], seed=9, theta=0.0)


def test_mla_v3_shape(cfa, oracle):
    """DeepSeek-V3-shaped block (hidden 7168, 128 heads, q_lora 1536) at ctx 4096,
    the benchmark's launch configuration."""
    wl = workloads.MLAS["mla_v3_b1_ctx4k"]
    mla, _, _, _ = run_mla(cfa, oracle, wl, list(wl.lens), seed=3)
    d = mla.describe()
    print(d)
    assert d["heads_per_cluster"] == 16
    # every cluster of the grid is resident at once
    assert d["coresident_clusters"] >= d["grid"] // d["cluster_size"]


def test_mla_is_deterministic(cfa, oracle):
    wl = workloads.custom_mla(2, 1024, 32, 256, 200)
    mla, dev, out, _ = run_mla(cfa, oracle, wl, [200, 150], seed=4)
    first = out.clone()
    for _ in range(3):
        mla.step(dev["x"], dev, dev["cache"], [200, 150], out, THETA, EPS)
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), out.view(torch.int16))


def test_mla_rejects_bad_arguments(cfa):
    with pytest.raises(cfa.CfaError):
        cfa.Mla(1, 256, 3, 128, 64)    # odd head count
    with pytest.raises(cfa.CfaError):
        cfa.Mla(1, 256, 4, 100, 64)    # q_lora not a multiple of 64
    wl = workloads.custom_mla(1, 256, 4, 128, 10)
    t = {k: v.cuda() for k, v in workloads.make_mla_inputs(wl).items()}
    mla = cfa.Mla(1, 256, 4, 128, wl.max_ctx)
    out = torch.empty(1, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cfa.CfaError):
        mla.step(t["x"], t, t["cache"], [wl.max_ctx], out)  # position out of range
