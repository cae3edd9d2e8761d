"""The plan's layout arithmetic on the host, without a GPU (cfa_plan_layout):
the work split, ring depth, shared memory and exchange form a plan takes for a
cluster size on a device with given limits. These are the rules the GPU tests
see only through cfa_plan_describe; here they are pinned on the CPU.

Device limits are those a GB300 reports (152 multiprocessors, 228 KB of shared
memory per multiprocessor, 227 KB opt-in per block, 1 KB reserved per block).
"""
import itertools

import pytest

GB300 = dict(num_sms=152, smem_per_sm=233472, smem_optin=232448, smem_reserved=1024)


@pytest.fixture(scope="module")
def lib():
    from out_proj_block_gb300 import build
    build.build()
    from out_proj_block_gb300 import cfa
    return cfa


def layout(lib, B, H, nh, D, max_ctx, C, exchange=-1, stages=0, **limits):
    lim = dict(GB300, **limits)
    return lib.cfa_plan_layout(B, H, nh, D, max_ctx, C, exchange, stages, lim["num_sms"],
                               lim["smem_per_sm"], lim["smem_optin"], lim["smem_reserved"])


# The plans the GPU runs reported for the three measured configurations of the
# block (the bench line's plan description and the ncu summaries' dynamic
# shared memory per block).
MEASURED = [
    # (B, H, nh, D, max_ctx, C): stages, blocks per SM, exchange, smem bytes, merge
    ((1, 4096, 32, 128, 4160, 8), (5, 2, "gather", 100912, "flat")),
    ((16, 4096, 32, 128, 4160, 4), (7, 1, "reduce_scatter", 230864, "separate")),
    ((8, 4096, 64, 64, 2112, 4), (4, 2, "reduce_scatter", 113440, "separate")),
]


@pytest.mark.parametrize("shape,expect", MEASURED)
def test_layout_of_the_measured_plans(lib, shape, expect):
    st, got = layout(lib, *shape)
    assert st == lib.CFA_OK
    stages, bps, exchange, smem, merge = expect
    assert (got["stages"], got["blocks_per_sm"], got["qkv_exchange"], got["smem_bytes"],
            got["merge"]) == (stages, bps, exchange, smem, merge)
    assert got["grid"] == shape[2] * shape[5]
    assert got["tensor_cores"] == (1 if shape[0] >= 3 else 0)


SHAPES = [(4096, 32, 128), (4096, 64, 64), (2048, 16, 128), (1024, 16, 64)]
CASES = [(B, H, nh, D, C) for B, (H, nh, D), C in
         itertools.product([1, 2, 3, 4, 8, 16], SHAPES, [2, 4, 8, 16])]


def supported(lib, B, H, nh, D, C, **kw):
    st, got = layout(lib, B, H, nh, D, 1088, C, **kw)
    assert st in (lib.CFA_OK, lib.CFA_ERR_UNSUPPORTED), st
    return got


@pytest.mark.parametrize("B,H,nh,D,C", CASES)
def test_layout_fits_the_device(lib, B, H, nh, D, C):
    got = supported(lib, B, H, nh, D, C)
    if got is None:
        return
    G = D // 64                      # 64-column groups of a head's Q/K/V block
    assert got["smem_bytes"] <= GB300["smem_optin"]
    assert got["blocks_per_sm"] * (got["smem_bytes"] + GB300["smem_reserved"]) <= GB300["smem_per_sm"]
    assert 2 <= got["stages"] <= 12
    assert got["proj_rows_per_block"] * (C // G) == H
    assert got["out_cols_per_block"] * C == H
    assert got["tensor_cores"] == (1 if B >= 3 else 0)
    if got["tensor_cores"]:          # blocks that share an SM share its 512 TMEM columns
        assert got["tmem_cols"] * got["blocks_per_sm"] <= 512
    # the flat merge reads every head's fp32 partials of a column chunk through one block
    flat_bytes = 4 * nh * B * (H // C)
    assert got["merge"] == ("separate" if flat_bytes > 256 * 1024 else "flat")


@pytest.mark.parametrize("B,H,nh,D,C", CASES)
def test_automatic_exchange_follows_its_rule(lib, B, H, nh, D, C):
    """Automatic exchange: reduce-scatter where it fits more blocks on an SM
    than the gather form, or, at the same blocks per SM, more ring stages on
    the tensor-core path, or more stages where gather leaves fewer than 4."""
    auto = supported(lib, B, H, nh, D, C)
    gather = supported(lib, B, H, nh, D, C, exchange=0)
    rs = supported(lib, B, H, nh, D, C, exchange=1)
    if gather is None:               # only the reduce-scatter form can fit, if any
        assert auto == rs
        return
    if rs is None:
        assert auto == gather
        return
    more_blocks = rs["blocks_per_sm"] > gather["blocks_per_sm"]
    more_stages = (rs["blocks_per_sm"] == gather["blocks_per_sm"] and rs["stages"] > gather["stages"]
                   and (rs["tensor_cores"] == 1 or gather["stages"] < 4))
    assert auto == (rs if more_blocks or more_stages else gather)
    assert gather["qkv_exchange"] == "gather" and rs["qkv_exchange"] == "reduce_scatter"


def test_forced_stages_and_rejections(lib):
    st, got = layout(lib, 1, 4096, 32, 128, 4160, 8, stages=3)
    assert st == lib.CFA_OK and got["stages"] == 3
    # more stages than the shared memory holds; a cluster size that is not a power of two
    assert layout(lib, 1, 4096, 32, 128, 4160, 8, stages=20)[0] == lib.CFA_ERR_UNSUPPORTED
    assert layout(lib, 1, 4096, 32, 128, 4160, 3)[0] == lib.CFA_ERR_UNSUPPORTED
    # head_dim 128 needs its two 64-column groups in different blocks
    assert layout(lib, 1, 4096, 32, 128, 4160, 1)[0] == lib.CFA_ERR_UNSUPPORTED
    # shapes as cfa_plan_create
    assert layout(lib, 0, 4096, 32, 128, 4160, 8)[0] == lib.CFA_ERR_INVALID_ARG
    assert layout(lib, 1, 4096, 32, 100, 4160, 8)[0] == lib.CFA_ERR_INVALID_ARG
    assert layout(lib, 17, 4096, 32, 128, 4160, 8)[0] == lib.CFA_ERR_UNSUPPORTED
    # limits, exchange, stages out of range
    assert layout(lib, 1, 4096, 32, 128, 4160, 8, exchange=2)[0] == lib.CFA_ERR_INVALID_ARG
    assert layout(lib, 1, 4096, 32, 128, 4160, 8, stages=-1)[0] == lib.CFA_ERR_INVALID_ARG
    assert layout(lib, 1, 4096, 32, 128, 4160, 8, num_sms=0)[0] == lib.CFA_ERR_INVALID_ARG
    assert layout(lib, 1, 4096, 32, 128, 4160, 8, smem_optin=300000)[0] == lib.CFA_ERR_INVALID_ARG


def test_smaller_device_gets_fewer_stages_per_sm(lib):
    """With half the shared memory per SM the B=1 plan still fits, with fewer
    ring stages on each SM."""
    _, full = layout(lib, 1, 4096, 32, 128, 4160, 8)
    st, half = layout(lib, 1, 4096, 32, 128, 4160, 8, smem_per_sm=116736, smem_optin=115712)
    assert st == lib.CFA_OK
    assert half["blocks_per_sm"] * (half["smem_bytes"] + 1024) <= 116736
    assert half["blocks_per_sm"] * half["stages"] < full["blocks_per_sm"] * full["stages"]
