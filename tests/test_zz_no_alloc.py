"""The allocation-free decode entry point, for callers that cannot allocate
device memory while they run (a host framework owns every device byte, or
cudaMalloc is forbidden after start-up because it may synchronize the device
and may fail under memory pressure).

The GPU test calls cfa_decode_step_noalloc through the C ABI twice in a row
(the second call finds the previous call's leftovers in the shared scratch
array) and compares each result with the plan-based cfa_decode_step on the
same inputs. Both run the same fused kernel with the same cluster size and
the same fixed-order merges, so `out` and the appended K/V rows must match
bit for bit: a scratch-aliasing slip (stale partials of the previous call in
one head, a counter left non-zero) cannot hide inside a tolerance. The first
call is also held to the oracle within the parity tolerance. This file is
collected last so that a run stopping at the first failure has run everything
else.
"""
import os

import numpy as np
import pytest
import torch

from out_proj_block_gb300 import workloads

REL_L2 = 5e-3
MAX_ABS = 3e-2
NTHREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def lib():
    from out_proj_block_gb300 import build
    build.build()
    from out_proj_block_gb300 import cfa
    return cfa


def _args(wl, t, ctx_len, out):
    return (wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.max_ctx, t["x"].data_ptr(),
            t["W_qkv"].data_ptr(), t["W_o"].data_ptr(), t["k_cache"].data_ptr(),
            t["v_cache"].data_ptr(), ctx_len, out.data_ptr(),
            torch.cuda.current_stream().cuda_stream)


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    """n_heads * B * hidden above 2^21 floats does not fit the fixed array; the
    call fails on the host before any CUDA work."""
    raw = lib._lib.cfa_decode_step_noalloc
    st = raw(16, 8192, 64, 128, 64, 16, 16, 16, 16, 16, 0, 16, None)
    assert st == lib.CFA_ERR_UNSUPPORTED


def _rel_l2(got, ref):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,nh,d,L", [
    (2, 2048, 16, 128, 300),   # CUDA-core projections, merge inside the fused kernel
    (16, 2048, 16, 128, 100),  # tensor-core projections, separate head-merge kernel
    (8, 2048, 32, 64, 200),    # head_dim 64 on the tensor-core path
    (1, 2048, 16, 128, 0),     # empty cache: the new token alone
    (4, 2048, 16, 128, 0),
])
def test_noalloc_matches_plan_entry_point_twice(lib, oracle, B, H, nh, d, L):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    wl = workloads.custom(B, H, nh, d, L, max_ctx=320)
    t = workloads.make_inputs(wl, seed=70, device="cuda", poison_tail=True)
    cpu = {k: v.cpu() for k, v in t.items()}
    ref_out = torch.empty(wl.B, wl.hidden, dtype=torch.bfloat16, device="cuda")
    with lib.Plan(wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.max_ctx) as plan:
        plan.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"],
                         wl.ctx_len, ref_out)
        torch.cuda.synchronize()
        assert plan.status() == lib.CFA_OK
    ref_k = t["k_cache"][:, :, L].clone()
    ref_v = t["v_cache"][:, :, L].clone()
    raw = lib._lib.cfa_decode_step_noalloc
    for call in range(2):
        out = torch.full((wl.B, wl.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
        t["k_cache"][:, :, L] = float("nan")
        t["v_cache"][:, :, L] = float("nan")
        st = raw(*_args(wl, t, wl.ctx_len, out))
        assert st == lib.CFA_OK, lib.cfa_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), (
            f"call {call}: out differs from cfa_decode_step")
        assert torch.equal(t["k_cache"][:, :, L].view(torch.int16), ref_k.view(torch.int16)), (
            f"call {call}: appended key row differs from cfa_decode_step")
        assert torch.equal(t["v_cache"][:, :, L].view(torch.int16), ref_v.view(torch.int16)), (
            f"call {call}: appended value row differs from cfa_decode_step")
        if call == 0:
            want = oracle.decode_step(cpu["x"], cpu["W_qkv"], cpu["W_o"], cpu["k_cache"],
                                      cpu["v_cache"], L, nthreads=NTHREADS)
            for name, got, ref in (("out", out, want["out"]),
                                   ("k_new", t["k_cache"][:, :, L], want["k_new"]),
                                   ("v_new", t["v_cache"][:, :, L], want["v_new"])):
                g = got.double().cpu().numpy()
                rel, mx = _rel_l2(g, ref), float(np.abs(g - ref).max())
                assert rel <= REL_L2 and mx <= MAX_ABS, (
                    f"{name}: rel L2 {rel:.3e}, max abs {mx:.3e} against the oracle")
