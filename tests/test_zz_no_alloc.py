"""The allocation-free decode entry point, for callers that cannot allocate
device memory while they run (a host framework owns every device byte, or
cudaMalloc is forbidden after start-up because it may synchronize the device
and may fail under memory pressure).

The GPU test calls cfa_decode_step_noalloc through the C ABI twice in a row
(the second call finds the previous call's leftovers in the shared scratch
array) and compares each result with the plan-based cfa_decode_step on the
same inputs, within the tolerance the parity tests use. This file is collected
last so that a run stopping at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

from out_proj_block_gb300 import workloads

REL_L2 = 5e-3
MAX_ABS = 3e-2


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


@pytest.mark.gpu
@pytest.mark.parametrize("B,L", [(2, 300), (16, 100)])
def test_noalloc_matches_plan_entry_point_twice(lib, B, L):
    """B = 16 merges the heads in the separate merge kernel."""
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    wl = workloads.custom(B, 2048, 16, 128, L, max_ctx=320)
    t = workloads.make_inputs(wl, seed=70, device="cuda")
    ref_out = torch.empty(wl.B, wl.hidden, dtype=torch.bfloat16, device="cuda")
    with lib.Plan(wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.max_ctx) as plan:
        plan.decode_step(t["x"], t["W_qkv"], t["W_o"], t["k_cache"], t["v_cache"],
                         wl.ctx_len, ref_out)
    torch.cuda.synchronize()
    ref = ref_out.float().cpu().numpy()
    raw = lib._lib.cfa_decode_step_noalloc
    for call in range(2):
        out = torch.full((wl.B, wl.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = raw(*_args(wl, t, wl.ctx_len, out))
        assert st == lib.CFA_OK, lib.cfa_status_string(st)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all(), f"call {call}: non-finite output"
        rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
        mx = float(np.abs(got - ref).max())
        assert rel <= REL_L2 and mx <= MAX_ABS, f"call {call}: rel {rel:.3e} max abs {mx:.3e}"
