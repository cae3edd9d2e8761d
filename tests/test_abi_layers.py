"""The decoder-layer, decode-loop, MLA and no-alloc entry points of the C ABI
without a GPU: every argument check that include/cfa.h documents runs on the
host before any device call, so each bad call returns its documented status
code here, and a well-formed create call reaches the device query and reports
CFA_ERR_CUDA. Pointers are addresses inside one host buffer; every case below
fails before anything reads or writes through them."""
import ctypes

import pytest
import torch

# Host addresses stand in for device buffers here, so on a machine with a GPU a
# check that failed to fire would hand them to a kernel: the module runs only
# where there is no GPU to reach.
pytestmark = pytest.mark.skipif(torch.cuda.is_available(),
                                reason="host-only argument checks; a GPU is present")


@pytest.fixture(scope="module")
def lib():
    from out_proj_block_gb300 import build
    build.build()
    from out_proj_block_gb300 import cfa
    return cfa


@pytest.fixture(scope="module")
def arena():
    """A host buffer and a function giving the address of byte `off` in it,
    rounded up to 256 bytes first (so `off` itself sets the misalignment)."""
    buf = ctypes.create_string_buffer(1 << 20)
    base = (ctypes.addressof(buf) + 255) & ~255

    def at(off):
        return ctypes.c_void_p(base + off)

    at.buf = buf
    return at


# ------------------------------------------------------------------ RMSNorm


def test_rmsnorm_rejects_shapes_and_eps(lib, arena):
    x, g, y = arena(0), arena(65536), arena(131072)
    L = lib._lib
    assert L.cfa_rmsnorm(0, 64, x, g, 1e-5, y, None) == lib.CFA_ERR_INVALID_ARG      # B < 1
    assert L.cfa_rmsnorm(65536, 64, x, g, 1e-5, y, None) == lib.CFA_ERR_INVALID_ARG  # B too large
    assert L.cfa_rmsnorm(1, 60, x, g, 1e-5, y, None) == lib.CFA_ERR_INVALID_ARG      # n % 8
    assert L.cfa_rmsnorm(1, 4, x, g, 1e-5, y, None) == lib.CFA_ERR_INVALID_ARG       # n < 8
    assert L.cfa_rmsnorm(1, 64, None, g, 1e-5, y, None) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_rmsnorm(1, 64, x, None, 1e-5, y, None) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_rmsnorm(1, 64, x, g, 1e-5, None, None) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_rmsnorm(1, 64, x, g, -1.0, y, None) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_rmsnorm(1, 64, x, g, float("nan"), y, None) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_rmsnorm(1, 64, x, g, float("inf"), y, None) == lib.CFA_ERR_INVALID_ARG


def test_rmsnorm_rejects_misalignment_and_overlap(lib, arena):
    x, g, y = arena(0), arena(65536), arena(131072)
    L = lib._lib
    assert L.cfa_rmsnorm(1, 64, arena(8), g, 1e-5, y, None) == lib.CFA_ERR_ALIGNMENT
    assert L.cfa_rmsnorm(1, 64, x, arena(65538), 1e-5, y, None) == lib.CFA_ERR_ALIGNMENT
    assert L.cfa_rmsnorm(1, 64, x, g, 1e-5, arena(131080), None) == lib.CFA_ERR_ALIGNMENT
    # y over x (in place), y over the last bytes of x, y over the weight
    assert L.cfa_rmsnorm(1, 64, x, g, 1e-5, x, None) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_rmsnorm(2, 64, x, g, 1e-5, arena(240), None) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_rmsnorm(1, 64, x, g, 1e-5, arena(65536 + 64), None) == lib.CFA_ERR_INVALID_ARG


# ---------------------------------------------------------------------- MLP


@pytest.mark.parametrize("args,code", [
    ((0, 4096, 11008), 1),          # B < 1
    ((1, 0, 11008), 1),             # hidden < 1
    ((1, 4096, 0), 1),              # ffn < 1
    ((17, 4096, 11008), 2),         # B above 16
    ((1, 4032, 11008), 2),          # hidden not a multiple of 128
    ((1, 4096, 11000), 2),          # ffn not a multiple of 128
    ((1, 1 << 17, 11008), 2),       # hidden above 2^16
])
def test_mlp_create_rejects_bad_shapes(lib, args, code):
    assert lib._lib.cfa_mlp_create(*args) is None
    assert lib.cfa_last_error() == code


def test_mlp_create_without_gpu_reports_cuda_error(lib):
    assert lib._lib.cfa_mlp_create(1, 256, 512) is None
    assert lib.cfa_last_error() == lib.CFA_ERR_CUDA


def test_mlp_calls_reject_a_null_plan(lib, arena):
    L = lib._lib
    p = arena(0)
    assert L.cfa_mlp_step(None, p, p, 1e-5, p, p, p, p, None) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_mlp_set_pipeline(None, 1, 4) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_mlp_set_path(None, 0) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_mlp_status(None) == lib.CFA_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(256)
    assert L.cfa_mlp_describe(None, buf, 256) == lib.CFA_ERR_INVALID_ARG
    L.cfa_mlp_destroy(None)  # no-op


# --------------------------------------------------------- the decode loop


@pytest.mark.parametrize("args,code", [
    ((0, 1, 4096, 32, 128, 11008, 1088), 1),       # no layers
    ((4097, 1, 4096, 32, 128, 11008, 1088), 1),    # too many layers
    ((2, 0, 4096, 32, 128, 11008, 1088), 1),       # B < 1
    ((2, 1, 4096, 32, 100, 11008, 1088), 1),       # hidden != n_heads * head_dim
    ((2, 1, 4096, 32, 128, 0, 1088), 1),           # ffn < 1
    ((2, 1, 4096, 32, 128, 11008, 0), 1),          # max_ctx < 1
    ((2, 1, 3072, 32, 96, 11008, 1088), 2),        # head_dim 96 (attention plan)
    ((2, 17, 4096, 32, 128, 11008, 1088), 2),      # B above 16 (attention plan)
])
def test_stack_create_rejects_bad_shapes(lib, args, code):
    assert lib._lib.cfa_stack_create(*args) is None
    assert lib.cfa_last_error() == code


def test_stack_create_without_gpu_reports_cuda_error(lib):
    assert lib._lib.cfa_stack_create(2, 1, 256, 2, 128, 512, 128) is None
    assert lib.cfa_last_error() == lib.CFA_ERR_CUDA


def test_stack_calls_reject_a_null_stack(lib, arena):
    L = lib._lib
    p = arena(0)
    pos = arena(4096)
    assert L.cfa_stack_set_layer(None, 0, *([p] * 9)) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_stack_step(None, p, pos, 10000.0, 1e-5, 1, arena(8192), None) == \
        lib.CFA_ERR_INVALID_ARG
    assert L.cfa_stack_step_graph(None, p, pos, 10000.0, 1e-5, 1, arena(8192), None) == \
        lib.CFA_ERR_INVALID_ARG
    assert L.cfa_stack_status(None) == lib.CFA_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(256)
    assert L.cfa_stack_describe(None, buf, 256) == lib.CFA_ERR_INVALID_ARG
    L.cfa_stack_destroy(None)  # no-op


# ---------------------------------------------------------------------- MLA


@pytest.mark.parametrize("args,code", [
    ((0, 7168, 128, 1536, 4160), 1),         # B < 1
    ((1, 0, 128, 1536, 4160), 1),            # hidden < 1
    ((1, 7168, 0, 1536, 4160), 1),           # no heads
    ((1, 7168, 128, 0, 4160), 1),            # q_lora < 1
    ((1, 7168, 128, 1536, 0), 1),            # max_ctx < 1
    ((17, 7168, 128, 1536, 4160), 2),        # B above 16
    ((1, 7200, 128, 1536, 4160), 2),         # hidden not a multiple of 64
    ((1, 7168, 128, 1500, 4160), 2),         # q_lora not a multiple of 64
    ((1, 7168, 1, 1536, 4160), 2),           # one head: no head group of 2
    ((1, 7168, 127, 1536, 4160), 2),         # odd head count
    ((1, 7168, 128, 1536, (1 << 22) + 1), 2),
])
def test_mla_create_rejects_bad_shapes(lib, args, code):
    assert lib._lib.cfa_mla_create(*args) is None
    assert lib.cfa_last_error() == code


def test_mla_create_without_gpu_reports_cuda_error(lib):
    assert lib._lib.cfa_mla_create(1, 256, 2, 128, 128) is None
    assert lib.cfa_last_error() == lib.CFA_ERR_CUDA


def test_mla_calls_reject_a_null_plan(lib, arena):
    L = lib._lib
    p = arena(0)
    lens = (ctypes.c_int * 1)(5)
    assert L.cfa_mla_step(None, *([p] * 8), lens, 10000.0, 1e-6, arena(8192), None) == \
        lib.CFA_ERR_INVALID_ARG
    for splits in (0, 1, 2, 4):
        assert L.cfa_mla_set_row_splits(None, splits) == lib.CFA_ERR_INVALID_ARG
    assert L.cfa_mla_status(None) == lib.CFA_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(256)
    assert L.cfa_mla_describe(None, buf, 256) == lib.CFA_ERR_INVALID_ARG
    L.cfa_mla_destroy(None)  # no-op


# ------------------------------------------------------ the no-alloc step


def test_noalloc_rejects_bad_calls_before_the_device(lib, arena):
    L = lib._lib
    x, wq, wo, kc, vc, out = (arena(i * 16384) for i in range(6))

    def call(B=1, H=256, nh=2, d=128, max_ctx=128, ptrs=None, ctx_len=5):
        p = ptrs or (x, wq, wo, kc, vc)
        o = out if ptrs is None or len(ptrs) == 5 else ptrs[5]
        return L.cfa_decode_step_noalloc(B, H, nh, d, max_ctx, *p[:5], ctx_len, o, None)

    assert call(B=0) == lib.CFA_ERR_INVALID_ARG
    assert call(nh=3) == lib.CFA_ERR_INVALID_ARG                  # hidden != nh * d
    assert call(max_ctx=0) == lib.CFA_ERR_INVALID_ARG
    assert call(B=17) == lib.CFA_ERR_UNSUPPORTED
    assert call(H=192, nh=2, d=96) == lib.CFA_ERR_UNSUPPORTED     # head_dim 96
    assert call(max_ctx=(1 << 22) + 1) == lib.CFA_ERR_UNSUPPORTED
    # n_heads * B * hidden above 2^21 floats of scratch: 64 heads x 16 x 4096
    assert call(B=16, H=4096, nh=64, d=64) == lib.CFA_ERR_UNSUPPORTED
    assert call(ptrs=(x, None, wo, kc, vc)) == lib.CFA_ERR_INVALID_ARG
    assert call(ctx_len=-1) == lib.CFA_ERR_INVALID_ARG
    assert call(ctx_len=128) == lib.CFA_ERR_INVALID_ARG           # == max_ctx
    assert call(ptrs=(arena(8), wq, wo, kc, vc)) == lib.CFA_ERR_ALIGNMENT
    assert call(ptrs=(x, wq, wo, kc, arena(5 * 16384 + 4), out)) == lib.CFA_ERR_ALIGNMENT
    assert call(ptrs=(x, wq, wo, kc, vc, x)) == lib.CFA_ERR_INVALID_ARG  # out over x
