"""GPU parity: the fused CUDA kernel against the fp64 oracle, through the C ABI.

Tolerance (both for `out` and for the appended K/V rows, each compared with
the oracle's unrounded fp64 values): relative L2 error <= 5e-3 and max abs
error <= 3e-2. Cache rows other than row ctx_len must be bit-identical after
the call; rows past ctx_len are NaN-poisoned, so a stray read would also show
up as a non-finite output.
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


@pytest.fixture(scope="module")
def cfa():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from out_proj_block_gb300 import build
    build.build()
    from out_proj_block_gb300 import cfa as mod
    return mod


def rel_l2(got, ref):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


def check_close(name, got, ref):
    got = np.asarray(got, dtype=np.float64)
    assert np.isfinite(got).all(), f"{name}: non-finite values"
    e_rel = rel_l2(got, ref)
    e_abs = float(np.abs(got - ref).max())
    assert e_rel <= REL_L2 and e_abs <= MAX_ABS, (
        f"{name}: rel L2 {e_rel:.3e} (<= {REL_L2}), max abs {e_abs:.3e} (<= {MAX_ABS})")
    return e_rel, e_abs


def run_and_check(cfa, oracle, wl, seed=1, C=None, stages=None, check_untouched=True):
    t = workloads.make_inputs(wl, seed=seed, device="cuda", poison_tail=True)
    k_before = t["k_cache"].clone() if check_untouched else None
    v_before = t["v_cache"].clone() if check_untouched else None
    cpu = {k: v.cpu() for k, v in t.items()}
    L = wl.ctx_len
    out = torch.empty(wl.B, wl.hidden, dtype=torch.bfloat16, device="cuda")
    with cfa.Plan(wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.max_ctx,
                  cluster_size=C, stages=stages) as plan:
        plan.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], L, out)
        torch.cuda.synchronize()
        assert plan.status() == cfa.CFA_OK
        used_C = plan.cluster_size
    ref = oracle.decode_step(cpu["x"], cpu["W_qkv"], cpu["W_o"], cpu["k_cache"],
                             cpu["v_cache"], L, nthreads=NTHREADS)
    got = out.float().cpu().numpy()
    errs = {"out": check_close("out", got, ref["out"])}
    k_row = t["k_cache"][:, :, L].float().cpu().numpy()
    v_row = t["v_cache"][:, :, L].float().cpu().numpy()
    errs["k_new"] = check_close("k_new", k_row, ref["k_new"])
    errs["v_new"] = check_close("v_new", v_row, ref["v_new"])
    if check_untouched:
        for name, before, after in (("k", k_before, t["k_cache"]), ("v", v_before, t["v_cache"])):
            b = before.view(torch.int16).clone()
            a = after.view(torch.int16).clone()
            b[:, :, L] = 0
            a[:, :, L] = 0
            assert torch.equal(a, b), f"{name}_cache changed outside row ctx_len"
    return errs, used_C, out


# ------------------------------------------------ the benchmark configurations


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_workload_default_plan(cfa, oracle, name):
    wl = workloads.WORKLOADS[name]
    if wl.ctx_lens is not None or wl.rope_theta > 0:
        run_ex_and_check(cfa, oracle, wl, list(wl.lens), wl.rope_theta, seed=1)
        return
    errs, C, _ = run_and_check(cfa, oracle, wl, seed=1)
    print(f"{name}: C={C} out rel {errs['out'][0]:.2e} abs {errs['out'][1]:.2e}")


# --------------------------------------------- every cluster size, ragged tails


@pytest.mark.parametrize("C", [2, 4, 8, 16])
@pytest.mark.parametrize("B", [1, 3])
def test_cluster_sizes_head_dim_128(cfa, oracle, C, B):
    # ctx 301: 301 = 7 * 43, ragged against every split and against 32-row tiles
    wl = workloads.custom(B, 1024, 8, 128, 301, max_ctx=320)
    run_and_check(cfa, oracle, wl, seed=2 + C, C=C)


@pytest.mark.parametrize("C", [1, 2, 4, 8, 16])
def test_cluster_sizes_head_dim_64(cfa, oracle, C):
    wl = workloads.custom(2, 1024, 16, 64, 77, max_ctx=128)
    run_and_check(cfa, oracle, wl, seed=3 + C, C=C)


# ------------------------------------------------------------------ edge cases


@pytest.mark.parametrize("L", [0, 1, 3, 7, 63, 64, 65])
def test_short_contexts(cfa, oracle, L):
    """ctx_len = 0 (only the new token), ctx_len + 1 < cluster size (empty
    splits), and tile boundaries."""
    wl = workloads.custom(1, 512, 4, 128, L, max_ctx=96)
    run_and_check(cfa, oracle, wl, seed=10 + L, C=8)


def test_last_cache_row(cfa, oracle):
    """ctx_len = max_ctx - 1 writes the final row of the cache."""
    wl = workloads.custom(2, 512, 4, 128, 127, max_ctx=128)
    run_and_check(cfa, oracle, wl, seed=20, C=4)


def test_maximum_context(cfa, oracle):
    """The largest cache a plan accepts, max_ctx = 2^22, with ctx_len = 2^22 - 1:
    4,194,303 cached positions attended and the final row written, 4.3 GB of
    K/V cache (64-bit offsets everywhere). The oracle runs on one thread here
    (its per-head fp64 copies of K and V are 4.3 GB each)."""
    max_ctx = 1 << 22
    L = max_ctx - 1
    wl = workloads.custom(1, 256, 2, 128, L, max_ctx=max_ctx)
    t = workloads.make_inputs(wl, seed=21, device="cuda")
    out = torch.empty(1, wl.hidden, dtype=torch.bfloat16, device="cuda")
    k_last_before = t["k_cache"][:, :, L - 1].clone()
    with cfa.Plan(1, wl.hidden, wl.n_heads, wl.head_dim, max_ctx) as plan:
        plan.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], L, out)
        torch.cuda.synchronize()
        assert plan.status() == cfa.CFA_OK
    assert torch.equal(t["k_cache"][:, :, L - 1].view(torch.int16), k_last_before.view(torch.int16))
    cpu = {k: v.cpu() for k, v in t.items()}
    del t
    torch.cuda.empty_cache()
    ref = oracle.decode_step(cpu["x"], cpu["W_qkv"], cpu["W_o"], cpu["k_cache"], cpu["v_cache"], L,
                             nthreads=1)
    check_close("out", out.float().cpu().numpy(), ref["out"])
    check_close("k_new", cpu["k_cache"][:, :, L].float().numpy(), ref["k_new"])
    check_close("v_new", cpu["v_cache"][:, :, L].float().numpy(), ref["v_new"])


@pytest.mark.parametrize("B", [1, 2, 3, 5, 8, 9, 16])
def test_batch_sizes(cfa, oracle, B):
    wl = workloads.custom(B, 512, 4, 128, 150, max_ctx=192)
    run_and_check(cfa, oracle, wl, seed=30 + B, C=4)


@pytest.mark.parametrize("stages", [2, 3, 5])
def test_shallow_pipelines(cfa, oracle, stages):
    """Few stages force many ring wrap-arounds and phase changes mid-ring."""
    wl = workloads.custom(2, 1024, 8, 128, 500, max_ctx=512)
    run_and_check(cfa, oracle, wl, seed=40 + stages, C=4, stages=stages)


def test_spiky_keys_long_tile_count(cfa, oracle):
    wl = workloads.custom(1, 1024, 8, 128, 3000, max_ctx=3008, spiky_frac=0.05,
                          spiky_scale=4.0)
    run_and_check(cfa, oracle, wl, seed=50, C=2)


# ------------------------------------------------- the separate cross-head merge


@pytest.mark.parametrize("B,H,nh,D,L", [(16, 1536, 12, 128, 150), (9, 2048, 16, 128, 77),
                                        (16, 2048, 32, 64, 200)])
def test_separate_merge(cfa, oracle, B, H, nh, D, L):
    """Shapes whose cross-head merge would read more than 256 KB through one
    block merge in a second kernel: a head count that is not a power of two,
    head_dim 64, a batch of 9. Three launches on one plan, each step's merge
    overlapping the next step's start, give bit-identical outputs."""
    wl = workloads.custom(B, H, nh, D, L, max_ctx=L + 8)
    t = workloads.make_inputs(wl, seed=70 + B, device="cuda", poison_tail=True)
    cpu = {k: v.cpu() for k, v in t.items()}
    outs = []
    with cfa.Plan(wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.max_ctx, cluster_size=4) as plan:
        assert plan.describe()["merge"] == "separate"
        for _ in range(3):
            out = torch.empty(wl.B, wl.hidden, dtype=torch.bfloat16, device="cuda")
            plan.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], L, out)
            outs.append(out)
        torch.cuda.synchronize()
        assert plan.status() == cfa.CFA_OK
    ref = oracle.decode_step(cpu["x"], cpu["W_qkv"], cpu["W_o"], cpu["k_cache"], cpu["v_cache"], L,
                             nthreads=NTHREADS)
    check_close("out", outs[0].float().cpu().numpy(), ref["out"])
    assert all(torch.equal(outs[0].view(torch.int16), o.view(torch.int16)) for o in outs[1:])


def test_merge_forms_by_size(cfa):
    """B = 1 merges in the fused kernel (the last head to arrive); the batch-16
    benchmark shape merges in a second kernel."""
    with cfa.Plan(1, 4096, 32, 128, 4097) as plan:
        assert plan.describe()["merge"] == "flat"
        assert plan.describe()["launches_per_step"] == 1
    with cfa.Plan(16, 4096, 32, 128, 4097) as plan:
        assert plan.describe()["merge"] == "separate"
        assert plan.describe()["launches_per_step"] == 2


@pytest.mark.parametrize("B,H,nh,D", [
    (1, 4096, 32, 128), (16, 4096, 32, 128), (8, 4096, 64, 64),
    (2, 2048, 16, 128),   # C = 16 fills the SMs but only 14 clusters of 16 fit at once
    (8, 2048, 32, 64),    # C = 8 fills the SMs but only 15 clusters of 8 fit at once
    (16, 2048, 16, 128),
])
def test_default_cluster_size_keeps_the_grid_resident(cfa, B, H, nh, D):
    """The default plan never picks a cluster size whose grid would run in two
    waves; among co-resident sizes it takes the smallest that covers the SMs."""
    with cfa.Plan(B, H, nh, D, 320) as plan:
        d = plan.describe()
    C = d["cluster_size"]
    assert d["coresident_clusters"] >= nh, d
    if d["grid"] >= d["num_sms"]:
        assert C == 1 or nh * (C // 2) < d["num_sms"], d
    elif C < 16:
        # no larger size is co-resident
        try:
            with cfa.Plan(B, H, nh, D, 320, cluster_size=2 * C) as plan:
                assert plan.describe()["coresident_clusters"] < nh
        except cfa.CfaError:
            pass


@pytest.mark.parametrize("B,H,nh,D,L,C", [
    (1, 1024, 8, 128, 301, 8),    # two column groups, four row groups
    (2, 1024, 8, 128, 150, 2),    # one row group: nothing to reduce, only the gather
    (3, 1024, 8, 128, 97, 16),    # tensor-core projections, slices of 8 columns
    (8, 2048, 32, 64, 200, 4),    # head_dim 64 on the tensor cores
    (2, 1024, 16, 64, 77, 16),    # head_dim 64, sixteen row groups: slices of 4 columns
    (2, 512, 8, 64, 64, 1),       # a cluster of one block
])
def test_qkv_exchange_modes_are_bitwise_equal(cfa, oracle, B, H, nh, D, L, C):
    """The reduce-scatter exchange sums every slice over the row groups in the
    same order as the gather exchange, so out and the appended rows agree bit
    for bit; the reduce-scatter result is also held to the oracle."""
    wl = workloads.custom(B, H, nh, D, L, max_ctx=L + 16)
    t = workloads.make_inputs(wl, seed=80 + C, device="cuda", poison_tail=True)
    cpu = {k: v.cpu() for k, v in t.items()}
    res = {}
    for mode in (0, 1):
        out = torch.empty(B, H, dtype=torch.bfloat16, device="cuda")
        with cfa.Plan(B, H, nh, D, wl.max_ctx, cluster_size=C, qkv_exchange=mode) as plan:
            assert plan.describe()["qkv_exchange"] == ("reduce_scatter" if mode else "gather")
            plan.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], L, out)
            torch.cuda.synchronize()
            assert plan.status() == cfa.CFA_OK
        res[mode] = (out.view(torch.int16).clone(), t["k_cache"][:, :, L].view(torch.int16).clone(),
                     t["v_cache"][:, :, L].view(torch.int16).clone())
        t["k_cache"][:, :, L] = float("nan")
        t["v_cache"][:, :, L] = float("nan")
    for a, b, name in zip(res[0], res[1], ("out", "k_new", "v_new")):
        assert torch.equal(a, b), f"{name} differs between the two exchange modes"
    ref = oracle.decode_step(cpu["x"], cpu["W_qkv"], cpu["W_o"], cpu["k_cache"], cpu["v_cache"], L,
                             nthreads=NTHREADS)
    check_close("out", res[1][0].view(torch.bfloat16).float().cpu().numpy(), ref["out"])
    check_close("k_new", res[1][1].view(torch.bfloat16).float().cpu().numpy(), ref["k_new"])
    check_close("v_new", res[1][2].view(torch.bfloat16).float().cpu().numpy(), ref["v_new"])


def test_qkv_exchange_default_choice(cfa):
    """The reduce-scatter exchange is chosen on the tensor-core path (B >= 3)
    where it gives more pipeline stages (64 heads of 64 at B=8: 4 instead of
    3; B=16: 7 instead of 5); B=1 keeps the gather exchange."""
    for shape in ((8, 4096, 64, 64, 2112), (16, 4096, 32, 128, 4160)):
        with cfa.Plan(*shape) as plan:
            d = plan.describe()
            assert d["qkv_exchange"] == "reduce_scatter", (shape, d)
            plan.set_qkv_exchange(0)
            assert plan.describe()["stages"] < d["stages"], shape
    with cfa.Plan(1, 4096, 32, 128, 4160) as plan:
        assert plan.describe()["qkv_exchange"] == "gather"
    # 64 heads of 64 at B=16: only the reduce-scatter form fits two blocks per
    # SM at C = 4, which keeps that grid resident at once
    with cfa.Plan(16, 4096, 64, 64, 1088) as plan:
        d = plan.describe()
        assert d["cluster_size"] == 4 and d["qkv_exchange"] == "reduce_scatter", d
        assert d["coresident_clusters"] >= 64, d
    with cfa.Plan(1, 512, 4, 128, 64) as plan:
        with pytest.raises(cfa.CfaError):
            plan.set_qkv_exchange(2)


# ------------------------------------------------------ determinism and reuse


def test_deterministic_and_idempotent(cfa):
    wl = workloads.WORKLOADS["llama7b_b1_ctx1k"]
    t = workloads.make_inputs(wl, seed=5, device="cuda")
    outs, caches = [], []
    with cfa.Plan(wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.max_ctx) as plan:
        for _ in range(3):
            out = torch.empty(wl.B, wl.hidden, dtype=torch.bfloat16, device="cuda")
            plan.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"],
                             wl.ctx_len, out)
            torch.cuda.synchronize()
            outs.append(out.view(torch.int16).clone())
            caches.append(t["k_cache"][:, :, wl.ctx_len].view(torch.int16).clone())
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    assert all(torch.equal(caches[0], c) for c in caches[1:])


def test_cluster_size_does_not_change_result_beyond_rounding(cfa):
    wl = workloads.custom(1, 2048, 16, 128, 700, max_ctx=768)
    t = workloads.make_inputs(wl, seed=6, device="cuda")
    res = {}
    for C in (2, 4, 8, 16):
        out = torch.empty(1, wl.hidden, dtype=torch.bfloat16, device="cuda")
        with cfa.Plan(wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.max_ctx, cluster_size=C) as p:
            p.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"],
                          wl.ctx_len, out)
        res[C] = out.float().cpu().numpy()
    for C in (4, 8, 16):
        assert rel_l2(res[C], res[2]) < 5e-3


@pytest.mark.parametrize("pinned", [True, False])
def test_host_entry_point_matches_device(cfa, pinned):
    """Pinned host buffers take the zero-copy path (copy kernels), pageable
    ones the cudaMemcpyAsync path; both equal the device entry point."""
    wl = workloads.custom(3, 1024, 8, 128, 200, max_ctx=256)
    t = workloads.make_inputs(wl, seed=7, device="cuda")
    out_dev = torch.empty(wl.B, wl.hidden, dtype=torch.bfloat16, device="cuda")
    x_host = t["x"].cpu()
    out_host = torch.empty(wl.B, wl.hidden, dtype=torch.bfloat16)
    if pinned:
        x_host, out_host = x_host.pin_memory(), out_host.pin_memory()
    with cfa.Plan(wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.max_ctx) as plan:
        plan.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"],
                         wl.ctx_len, out_dev)
        plan.decode_step_host(x_host, t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"],
                              wl.ctx_len, out_host)
    torch.cuda.synchronize()
    assert torch.equal(out_host.view(torch.int16), out_dev.cpu().view(torch.int16))


# ------------------------------------------------------------- error handling


def test_runtime_argument_errors(cfa):
    wl = workloads.custom(1, 512, 4, 128, 10, max_ctx=64)
    t = workloads.make_inputs(wl, seed=8, device="cuda")
    out = torch.zeros(1, 512, dtype=torch.bfloat16, device="cuda")
    with cfa.Plan(1, 512, 4, 128, 64) as plan:
        h = plan.handle
        args = [t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"]]
        assert cfa.cfa_decode_step(h, *args, 64, out) == cfa.CFA_ERR_INVALID_ARG
        assert cfa.cfa_decode_step(h, *args, -1, out) == cfa.CFA_ERR_INVALID_ARG
        assert cfa.cfa_decode_step(h, t["x"].data_ptr() + 2, *args[1:], 10, out) == \
            cfa.CFA_ERR_ALIGNMENT
        assert cfa.cfa_decode_step(h, *args, 10, t["x"]) == cfa.CFA_ERR_INVALID_ARG  # aliasing
        assert cfa.cfa_plan_set_cluster_size(h, 3) == cfa.CFA_ERR_UNSUPPORTED
        assert cfa.cfa_plan_set_cluster_size(h, 1) == cfa.CFA_ERR_UNSUPPORTED  # d=128 needs >= 2
        assert cfa.cfa_plan_set_stages(h, 1) == cfa.CFA_ERR_UNSUPPORTED
        torch.cuda.synchronize()
        assert torch.count_nonzero(out) == 0  # nothing was launched
        assert plan.status() == cfa.CFA_OK


def test_bounded_wait_times_out_cleanly(cfa):
    """A wait on a barrier nothing arrives on gives up and reports a status;
    the context stays usable afterwards."""
    assert cfa.cfa_selftest_wait_timeout(2000) == cfa.CFA_ERR_TIMEOUT
    x = torch.ones(4, device="cuda")
    assert float(x.sum().item()) == 4.0


@pytest.mark.parametrize("overlap", [True, False])
def test_chained_steps_respect_dependencies(cfa, oracle, overlap):
    """Decode chain on one stream: step t+1 takes step t's `out` as its x and
    reads the cache row step t appended. With launch overlap on, each step may
    start before the previous one ends, so this checks that nothing dependent
    is read or written early. Every step is compared with the oracle on the
    exact inputs it saw (x and the cache as left by the earlier steps)."""
    wl = workloads.custom(2, 1024, 8, 128, 40, max_ctx=64)
    t = workloads.make_inputs(wl, seed=60, device="cuda", poison_tail=True)
    n_steps = 6
    xs = [t["x"]]
    outs = []
    with cfa.Plan(wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.max_ctx, overlap=overlap) as plan:
        for k in range(n_steps):
            out = torch.empty(wl.B, wl.hidden, dtype=torch.bfloat16, device="cuda")
            plan.decode_step(xs[-1], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"],
                             wl.ctx_len + k, out)
            outs.append(out)
            xs.append(out)
        torch.cuda.synchronize()
        assert plan.status() == cfa.CFA_OK
    W_qkv, W_o = t["W_qkv"].cpu(), t["W_o"].cpu()
    kc, vc = t["k_cache"].cpu(), t["v_cache"].cpu()
    for k in range(n_steps):
        ref = oracle.decode_step(xs[k].cpu(), W_qkv, W_o, kc, vc, wl.ctx_len + k,
                                 nthreads=NTHREADS)
        check_close(f"out[{k}]", outs[k].float().cpu().numpy(), ref["out"])
        check_close(f"k_new[{k}]", kc[:, :, wl.ctx_len + k].float().numpy(), ref["k_new"])


# ------------------------------------ per-sequence lengths and rotary embedding


def run_ex_and_check(cfa, oracle, wl, lens, theta, seed, C=None):
    t = workloads.make_inputs(wl, seed=seed, device="cuda", poison_tail=False)
    # rows past each sequence's own length are never read: poison them
    for b, L in enumerate(lens):
        t["k_cache"][b, :, L:] = float("nan")
        t["v_cache"][b, :, L:] = float("nan")
    k_before, v_before = t["k_cache"].clone(), t["v_cache"].clone()
    cpu = {k: v.cpu() for k, v in t.items()}
    out = torch.empty(wl.B, wl.hidden, dtype=torch.bfloat16, device="cuda")
    with cfa.Plan(wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.max_ctx, cluster_size=C) as plan:
        plan.decode_step_ex(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], lens, out,
                            rope_theta=theta)
        torch.cuda.synchronize()
        assert plan.status() == cfa.CFA_OK
    ref = oracle.decode_step_ex(cpu["x"], cpu["W_qkv"], cpu["W_o"], cpu["k_cache"],
                                cpu["v_cache"], lens, rope_theta=theta, nthreads=NTHREADS)
    check_close("out", out.float().cpu().numpy(), ref["out"])
    rows_k = np.stack([t["k_cache"][b, :, L].float().cpu().numpy() for b, L in enumerate(lens)])
    rows_v = np.stack([t["v_cache"][b, :, L].float().cpu().numpy() for b, L in enumerate(lens)])
    check_close("k_new", rows_k, ref["k_new"])
    check_close("v_new", rows_v, ref["v_new"])
    for name, before, after in (("k", k_before, t["k_cache"]), ("v", v_before, t["v_cache"])):
        b_ = before.view(torch.int16).clone()
        a_ = after.view(torch.int16).clone()
        for b, L in enumerate(lens):
            b_[b, :, L] = 0
            a_[b, :, L] = 0
        assert torch.equal(a_, b_), f"{name}_cache changed outside the appended rows"


@pytest.mark.parametrize("theta", [0.0, 10000.0])
@pytest.mark.parametrize("B,lens", [(1, [300]), (3, [0, 77, 301]), (5, [5, 64, 1, 200, 63])])
def test_ragged_lengths_and_rope(cfa, oracle, theta, B, lens):
    wl = workloads.custom(B, 1024, 8, 128, max(lens), max_ctx=320)
    run_ex_and_check(cfa, oracle, wl, lens, theta, seed=80 + B, C=4)


@pytest.mark.parametrize("C", [2, 8])
def test_rope_head_dim_64_and_long_positions(cfa, oracle, C):
    wl = workloads.custom(4, 1024, 16, 64, 4000, max_ctx=4096)
    run_ex_and_check(cfa, oracle, wl, [4000, 17, 2500, 4095], 10000.0, seed=90, C=C)


def test_ex_with_equal_lengths_matches_decode_step(cfa):
    wl = workloads.custom(2, 1024, 8, 128, 100, max_ctx=128)
    t = workloads.make_inputs(wl, seed=91, device="cuda")
    a = torch.empty(2, 1024, dtype=torch.bfloat16, device="cuda")
    b = torch.empty_like(a)
    with cfa.Plan(2, 1024, 8, 128, 128) as plan:
        plan.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], 100, a)
        plan.decode_step_ex(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"], [100, 100], b)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_ex_rejects_bad_lengths(cfa):
    with cfa.Plan(2, 512, 4, 128, 64) as plan:
        h = plan.handle
        assert cfa.cfa_decode_step_ex(h, 16, 16, 16, 16, 16, [3, 64], 0.0, 16) == cfa.CFA_ERR_INVALID_ARG
        assert cfa.cfa_decode_step_ex(h, 16, 16, 16, 16, 16, [3, -1], 0.0, 16) == cfa.CFA_ERR_INVALID_ARG
        assert cfa.cfa_decode_step_ex(h, 16, 16, 16, 16, 16, [3, 4], -1.0, 16) == cfa.CFA_ERR_INVALID_ARG
