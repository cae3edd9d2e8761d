"""Python binding of libcfa.so (see include/cfa.h): same names, argument marshalling only.

Every step of the decode path runs inside the CUDA library. This module only
checks tensor dtypes, devices, shapes and contiguity, turns tensors into
pointers and CUDA streams into handles, and maps status codes to exceptions.
Importing it raises ImportError if the library has not been built; there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import json
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcfa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with out_proj_block_gb300.build.build() "
        "(nvcc, sm_103a). There is no fallback path.")

_lib = ctypes.CDLL(LIB_PATH)

_vp = ctypes.c_void_p
_i = ctypes.c_int

_lib.cfa_plan_create.restype = _vp
_lib.cfa_plan_create.argtypes = [_i, _i, _i, _i, _i]
_lib.cfa_plan_destroy.restype = None
_lib.cfa_plan_destroy.argtypes = [_vp]
_lib.cfa_decode_step.restype = _i
_lib.cfa_decode_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp]
_lib.cfa_decode_step_ex.restype = _i
_lib.cfa_decode_step_ex.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.POINTER(ctypes.c_int),
                                    ctypes.c_double, _vp, _vp]
_lib.cfa_decode_step_host.restype = _i
_lib.cfa_decode_step_host.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp]
_lib.cfa_decode_step_noalloc.restype = _i
_lib.cfa_decode_step_noalloc.argtypes = [_i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp]
_lib.cfa_plan_set_cluster_size.restype = _i
_lib.cfa_plan_set_cluster_size.argtypes = [_vp, _i]
_lib.cfa_plan_set_stages.restype = _i
_lib.cfa_plan_set_stages.argtypes = [_vp, _i]
_lib.cfa_plan_set_overlap.restype = _i
_lib.cfa_plan_set_overlap.argtypes = [_vp, _i]
_lib.cfa_plan_set_qkv_exchange.restype = _i
_lib.cfa_plan_set_qkv_exchange.argtypes = [_vp, _i]
_lib.cfa_plan_cluster_size.restype = _i
_lib.cfa_plan_cluster_size.argtypes = [_vp]
_lib.cfa_plan_describe.restype = _i
_lib.cfa_plan_describe.argtypes = [_vp, ctypes.c_char_p, _i]
_lib.cfa_plan_status.restype = _i
_lib.cfa_plan_status.argtypes = [_vp]
_lib.cfa_last_error.restype = _i
_lib.cfa_last_error.argtypes = []
_lib.cfa_status_string.restype = ctypes.c_char_p
_lib.cfa_status_string.argtypes = [_i]
_lib.cfa_selftest_wait_timeout.restype = _i
_lib.cfa_selftest_wait_timeout.argtypes = [_i, _vp]
_lib.cfa_rmsnorm.restype = _i
_lib.cfa_rmsnorm.argtypes = [_i, _i, _vp, _vp, ctypes.c_float, _vp, _vp]
_lib.cfa_mlp_create.restype = _vp
_lib.cfa_mlp_create.argtypes = [_i, _i, _i]
_lib.cfa_mlp_destroy.restype = None
_lib.cfa_mlp_destroy.argtypes = [_vp]
_lib.cfa_mlp_step.restype = _i
_lib.cfa_mlp_step.argtypes = [_vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp]
_lib.cfa_mlp_set_pipeline.restype = _i
_lib.cfa_mlp_set_pipeline.argtypes = [_vp, _i, _i]
_lib.cfa_mlp_set_path.restype = _i
_lib.cfa_mlp_set_path.argtypes = [_vp, _i]
_lib.cfa_mlp_status.restype = _i
_lib.cfa_mlp_status.argtypes = [_vp]
_lib.cfa_mlp_describe.restype = _i
_lib.cfa_mlp_describe.argtypes = [_vp, ctypes.c_char_p, _i]
_lib.cfa_stack_create.restype = _vp
_lib.cfa_stack_create.argtypes = [_i] * 7
_lib.cfa_stack_destroy.restype = None
_lib.cfa_stack_destroy.argtypes = [_vp]
_lib.cfa_stack_set_layer.restype = _i
_lib.cfa_stack_set_layer.argtypes = [_vp, _i] + [_vp] * 9
_lib.cfa_stack_step.restype = _i
_lib.cfa_stack_step.argtypes = [_vp, _vp, _vp, ctypes.c_double, ctypes.c_float, _i, _vp, _vp]
_lib.cfa_stack_step_graph.restype = _i
_lib.cfa_stack_step_graph.argtypes = [_vp, _vp, _vp, ctypes.c_double, ctypes.c_float, _i, _vp,
                                      _vp]
_lib.cfa_stack_status.restype = _i
_lib.cfa_stack_status.argtypes = [_vp]
_lib.cfa_mla_create.restype = _vp
_lib.cfa_mla_create.argtypes = [_i] * 5
_lib.cfa_mla_destroy.restype = None
_lib.cfa_mla_destroy.argtypes = [_vp]
_lib.cfa_mla_step.restype = _i
_lib.cfa_mla_step.argtypes = ([_vp] * 9 + [ctypes.POINTER(ctypes.c_int), ctypes.c_double,
                                           ctypes.c_float, _vp, _vp])
_lib.cfa_mla_status.restype = _i
_lib.cfa_mla_status.argtypes = [_vp]
_lib.cfa_mla_describe.restype = _i
_lib.cfa_mla_describe.argtypes = [_vp, ctypes.c_char_p, _i]
_lib.cfa_mla_set_row_splits.restype = _i
_lib.cfa_mla_set_row_splits.argtypes = [_vp, _i]
_lib.cfa_stack_describe.restype = _i
_lib.cfa_stack_describe.argtypes = [_vp, ctypes.c_char_p, _i]
_lib.cfa_plan_layout.restype = _i
_lib.cfa_plan_layout.argtypes = [_i] * 12 + [ctypes.c_char_p, _i]

CFA_OK = 0
CFA_ERR_INVALID_ARG = 1
CFA_ERR_UNSUPPORTED = 2
CFA_ERR_CUDA = 3
CFA_ERR_TIMEOUT = 4
CFA_ERR_ALIGNMENT = 5

EXPORTED_SYMBOLS = (
    "cfa_plan_create", "cfa_plan_destroy", "cfa_decode_step", "cfa_decode_step_ex",
    "cfa_decode_step_host",
    "cfa_decode_step_noalloc",
    "cfa_plan_set_cluster_size", "cfa_plan_set_stages", "cfa_plan_set_overlap",
    "cfa_plan_set_qkv_exchange",
    "cfa_plan_cluster_size",
    "cfa_plan_describe", "cfa_plan_layout", "cfa_plan_status", "cfa_last_error",
    "cfa_status_string",
    "cfa_selftest_wait_timeout",
    "cfa_rmsnorm", "cfa_mlp_create", "cfa_mlp_destroy", "cfa_mlp_step", "cfa_mlp_status",
    "cfa_mlp_set_pipeline", "cfa_mlp_set_path",
    "cfa_mlp_describe", "cfa_stack_create", "cfa_stack_destroy", "cfa_stack_set_layer",
    "cfa_stack_step", "cfa_stack_step_graph", "cfa_stack_status", "cfa_stack_describe",
    "cfa_mla_create", "cfa_mla_destroy", "cfa_mla_step", "cfa_mla_status", "cfa_mla_describe",
    "cfa_mla_set_row_splits",
)


class CfaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        super().__init__(f"{what}: {cfa_status_string(status)}" if what else cfa_status_string(status))


def cfa_status_string(status: int) -> str:
    return _lib.cfa_status_string(int(status)).decode()


def cfa_last_error() -> int:
    return int(_lib.cfa_last_error())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------- raw C-ABI calls


def cfa_plan_create(B: int, hidden: int, n_heads: int, head_dim: int, max_ctx: int) -> int:
    h = _lib.cfa_plan_create(B, hidden, n_heads, head_dim, max_ctx)
    if not h:
        raise CfaError(cfa_last_error(), "cfa_plan_create")
    return h


def cfa_plan_destroy(plan: int) -> None:
    _lib.cfa_plan_destroy(plan)


def cfa_decode_step(plan, x, W_qkv, W_o, k_cache, v_cache, ctx_len: int, out, stream=None) -> int:
    return int(_lib.cfa_decode_step(plan, _ptr(x), _ptr(W_qkv), _ptr(W_o), _ptr(k_cache),
                                    _ptr(v_cache), int(ctx_len), _ptr(out), _stream(stream)))


def cfa_decode_step_ex(plan, x, W_qkv, W_o, k_cache, v_cache, ctx_lens, rope_theta: float,
                       out, stream=None) -> int:
    lens = (ctypes.c_int * len(ctx_lens))(*[int(v) for v in ctx_lens])
    return int(_lib.cfa_decode_step_ex(plan, _ptr(x), _ptr(W_qkv), _ptr(W_o), _ptr(k_cache),
                                       _ptr(v_cache), lens, float(rope_theta), _ptr(out),
                                       _stream(stream)))


def cfa_decode_step_host(plan, x_host, W_qkv, W_o, k_cache, v_cache, ctx_len: int, out_host,
                         stream=None) -> int:
    return int(_lib.cfa_decode_step_host(plan, _ptr(x_host), _ptr(W_qkv), _ptr(W_o),
                                         _ptr(k_cache), _ptr(v_cache), int(ctx_len),
                                         _ptr(out_host), _stream(stream)))


def cfa_decode_step_noalloc(B: int, hidden: int, n_heads: int, head_dim: int, max_ctx: int,
                            x, W_qkv, W_o, k_cache, v_cache, ctx_len: int, out,
                            stream=None) -> int:
    """The decode step for callers that cannot allocate device memory (see
    include/cfa.h); its scratch is a fixed array inside the library."""
    return int(_lib.cfa_decode_step_noalloc(B, hidden, n_heads, head_dim, max_ctx, _ptr(x),
                                            _ptr(W_qkv), _ptr(W_o), _ptr(k_cache),
                                            _ptr(v_cache), int(ctx_len), _ptr(out),
                                            _stream(stream)))


def cfa_plan_set_cluster_size(plan, C: int) -> int:
    return int(_lib.cfa_plan_set_cluster_size(plan, int(C)))


def cfa_plan_set_stages(plan, stages: int) -> int:
    return int(_lib.cfa_plan_set_stages(plan, int(stages)))


def cfa_plan_set_overlap(plan, enable: bool) -> int:
    return int(_lib.cfa_plan_set_overlap(plan, 1 if enable else 0))


def cfa_plan_set_qkv_exchange(plan, mode: int) -> int:
    return int(_lib.cfa_plan_set_qkv_exchange(plan, int(mode)))


def cfa_plan_cluster_size(plan) -> int:
    return int(_lib.cfa_plan_cluster_size(plan))


def cfa_plan_describe(plan) -> dict:
    buf = ctypes.create_string_buffer(1024)
    st = _lib.cfa_plan_describe(plan, buf, len(buf))
    if st != CFA_OK:
        raise CfaError(st, "cfa_plan_describe")
    return json.loads(buf.value.decode())


def cfa_plan_layout(B: int, hidden: int, n_heads: int, head_dim: int, max_ctx: int, C: int,
                    exchange: int, stages: int, num_sms: int, smem_per_sm: int, smem_optin: int,
                    smem_reserved: int):
    """(status, layout dict or None): the layout a plan of this shape would use
    with cluster size C on a device with these limits, computed on the host."""
    buf = ctypes.create_string_buffer(1024)
    st = int(_lib.cfa_plan_layout(B, hidden, n_heads, head_dim, max_ctx, C, exchange, stages,
                                  num_sms, smem_per_sm, smem_optin, smem_reserved, buf,
                                  len(buf)))
    return st, (json.loads(buf.value.decode()) if st == CFA_OK else None)


def cfa_plan_status(plan) -> int:
    return int(_lib.cfa_plan_status(plan))


def cfa_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    return int(_lib.cfa_selftest_wait_timeout(int(limit_us), _stream(stream)))


# ---------------------------------------------------------- tensor-level API


class Plan:
    """Owns a cfa_plan; checks tensors and launches decode steps."""

    def __init__(self, B: int, hidden: int, n_heads: int, head_dim: int, max_ctx: int,
                 cluster_size: Optional[int] = None, stages: Optional[int] = None,
                 overlap: Optional[bool] = None, qkv_exchange: Optional[int] = None):
        self.B, self.hidden, self.n_heads, self.head_dim, self.max_ctx = (
            B, hidden, n_heads, head_dim, max_ctx)
        self.handle = cfa_plan_create(B, hidden, n_heads, head_dim, max_ctx)
        try:
            if cluster_size is not None:
                self.set_cluster_size(cluster_size)
            if qkv_exchange is not None:
                self.set_qkv_exchange(qkv_exchange)
            if stages is not None:
                self.set_stages(stages)
            if overlap is not None:
                self.set_overlap(overlap)
        except Exception:
            self.close()
            raise

    def close(self):
        if getattr(self, "handle", None):
            cfa_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def cluster_size(self) -> int:
        return cfa_plan_cluster_size(self.handle)

    def set_cluster_size(self, C: int) -> None:
        st = cfa_plan_set_cluster_size(self.handle, C)
        if st != CFA_OK:
            raise CfaError(st, f"cluster size {C}")

    def set_stages(self, n: int) -> None:
        st = cfa_plan_set_stages(self.handle, n)
        if st != CFA_OK:
            raise CfaError(st, f"stages {n}")

    def set_qkv_exchange(self, mode: int) -> None:
        """-1 automatic, 0 gather, 1 reduce-scatter (cfa_plan_set_qkv_exchange)."""
        st = cfa_plan_set_qkv_exchange(self.handle, mode)
        if st != CFA_OK:
            raise CfaError(st, f"qkv exchange {mode}")

    def set_overlap(self, enable: bool) -> None:
        st = cfa_plan_set_overlap(self.handle, enable)
        if st != CFA_OK:
            raise CfaError(st, "overlap")

    def describe(self) -> dict:
        return cfa_plan_describe(self.handle)

    def status(self) -> int:
        return cfa_plan_status(self.handle)

    def _check(self, x, W_qkv, W_o, k_cache, v_cache, out, host_io: bool):
        B, H, nh, d, mc = self.B, self.hidden, self.n_heads, self.head_dim, self.max_ctx
        want = {"W_qkv": (W_qkv, (H, 3 * H)), "W_o": (W_o, (H, H)),
                "k_cache": (k_cache, (B, nh, mc, d)), "v_cache": (v_cache, (B, nh, mc, d)),
                "x": (x, (B, H)), "out": (out, (B, H))}
        for name, (t, shape) in want.items():
            if t.dtype != torch.bfloat16:
                raise TypeError(f"{name} must be bf16")
            if tuple(t.shape) != shape:
                raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {shape}")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
            on_host = name in ("x", "out") and host_io
            if on_host == t.is_cuda:
                raise ValueError(f"{name} must be on the {'host' if on_host else 'GPU'}")

    def decode_step(self, x, W_qkv, W_o, k_cache, v_cache, ctx_len: int, out, stream=None):
        """One fused decode step on device tensors; asynchronous on `stream`."""
        self._check(x, W_qkv, W_o, k_cache, v_cache, out, host_io=False)
        st = cfa_decode_step(self.handle, x, W_qkv, W_o, k_cache, v_cache, ctx_len, out, stream)
        if st != CFA_OK:
            raise CfaError(st, "cfa_decode_step")
        return out

    def decode_step_ex(self, x, W_qkv, W_o, k_cache, v_cache, ctx_lens, out,
                       rope_theta: float = 0.0, stream=None):
        """Decode step with per-sequence lengths and optional rotary embedding."""
        self._check(x, W_qkv, W_o, k_cache, v_cache, out, host_io=False)
        if len(ctx_lens) != self.B:
            raise ValueError("ctx_lens needs one entry per batch row")
        st = cfa_decode_step_ex(self.handle, x, W_qkv, W_o, k_cache, v_cache, ctx_lens,
                                rope_theta, out, stream)
        if st != CFA_OK:
            raise CfaError(st, "cfa_decode_step_ex")
        return out

    def decode_step_host(self, x_host, W_qkv, W_o, k_cache, v_cache, ctx_len: int, out_host,
                         stream=None):
        """Same step with x and out in (preferably pinned) host memory; synchronous."""
        self._check(x_host, W_qkv, W_o, k_cache, v_cache, out_host, host_io=True)
        st = cfa_decode_step_host(self.handle, x_host, W_qkv, W_o, k_cache, v_cache, ctx_len,
                                  out_host, stream)
        if st != CFA_OK:
            raise CfaError(st, "cfa_decode_step_host")
        return out_host


# ----------------------------------------------- decoder layers and the loop


def cfa_rmsnorm(B: int, n: int, x, g, eps: float, y, stream=None) -> int:
    return int(_lib.cfa_rmsnorm(int(B), int(n), _ptr(x), _ptr(g), float(eps), _ptr(y),
                                _stream(stream)))


def cfa_mlp_create(B: int, hidden: int, ffn: int) -> int:
    h = _lib.cfa_mlp_create(B, hidden, ffn)
    if not h:
        raise CfaError(cfa_last_error(), "cfa_mlp_create")
    return h


def cfa_mlp_destroy(mlp: int) -> None:
    _lib.cfa_mlp_destroy(mlp)


def cfa_mlp_step(mlp, h, norm_w, eps: float, W_gate, W_up, W_down, y, stream=None) -> int:
    return int(_lib.cfa_mlp_step(mlp, _ptr(h), _ptr(norm_w), float(eps), _ptr(W_gate),
                                 _ptr(W_up), _ptr(W_down), _ptr(y), _stream(stream)))


def cfa_mlp_set_pipeline(mlp, blocks_per_sm: int, stages: int) -> int:
    return int(_lib.cfa_mlp_set_pipeline(mlp, int(blocks_per_sm), int(stages)))


# cfa_mlp_set_path: the MLP GEMVs' kernel
PATH_AUTO, PATH_CUDA_CORES, PATH_TENSOR_CORES = -1, 0, 1


def cfa_mlp_set_path(mlp, path: int) -> int:
    return int(_lib.cfa_mlp_set_path(mlp, int(path)))


def cfa_mlp_status(mlp) -> int:
    return int(_lib.cfa_mlp_status(mlp))


def cfa_mlp_describe(mlp) -> dict:
    buf = ctypes.create_string_buffer(1024)
    st = _lib.cfa_mlp_describe(mlp, buf, len(buf))
    if st != CFA_OK:
        raise CfaError(st, "cfa_mlp_describe")
    return json.loads(buf.value.decode())


def cfa_stack_create(n_layers: int, B: int, hidden: int, n_heads: int, head_dim: int, ffn: int,
                     max_ctx: int) -> int:
    h = _lib.cfa_stack_create(n_layers, B, hidden, n_heads, head_dim, ffn, max_ctx)
    if not h:
        raise CfaError(cfa_last_error(), "cfa_stack_create")
    return h


def cfa_stack_destroy(stack: int) -> None:
    _lib.cfa_stack_destroy(stack)


def cfa_stack_set_layer(stack, layer: int, attn_norm, W_qkv, W_o, k_cache, v_cache, mlp_norm,
                        W_gate, W_up, W_down) -> int:
    return int(_lib.cfa_stack_set_layer(stack, int(layer), _ptr(attn_norm), _ptr(W_qkv),
                                        _ptr(W_o), _ptr(k_cache), _ptr(v_cache), _ptr(mlp_norm),
                                        _ptr(W_gate), _ptr(W_up), _ptr(W_down)))


def cfa_stack_step(stack, x, positions, rope_theta: float, eps: float, advance: bool, out,
                   stream=None) -> int:
    return int(_lib.cfa_stack_step(stack, _ptr(x), _ptr(positions), float(rope_theta),
                                   float(eps), 1 if advance else 0, _ptr(out), _stream(stream)))


def cfa_stack_step_graph(stack, x, positions, rope_theta: float, eps: float, advance: bool, out,
                         stream=None) -> int:
    return int(_lib.cfa_stack_step_graph(stack, _ptr(x), _ptr(positions), float(rope_theta),
                                         float(eps), 1 if advance else 0, _ptr(out),
                                         _stream(stream)))


def cfa_stack_status(stack) -> int:
    return int(_lib.cfa_stack_status(stack))


def cfa_stack_describe(stack) -> dict:
    buf = ctypes.create_string_buffer(2048)
    st = _lib.cfa_stack_describe(stack, buf, len(buf))
    if st != CFA_OK:
        raise CfaError(st, "cfa_stack_describe")
    return json.loads(buf.value.decode())


def _check_tensor(name, t, shape, dtype=torch.bfloat16):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on the GPU")


def rmsnorm(x, g, eps: float, y, stream=None):
    """y = bf16(g * x / sqrt(mean(x^2) + eps)) row by row, on the GPU."""
    B, n = x.shape
    _check_tensor("x", x, (B, n))
    _check_tensor("g", g, (n,))
    _check_tensor("y", y, (B, n))
    st = cfa_rmsnorm(B, n, x, g, eps, y, stream)
    if st != CFA_OK:
        raise CfaError(st, "cfa_rmsnorm")
    return y


class Mlp:
    """Owns a cfa_mlp: y = h + down(silu(gate(hn)) * up(hn)), hn = rmsnorm(h)."""

    def __init__(self, B: int, hidden: int, ffn: int):
        self.B, self.hidden, self.ffn = B, hidden, ffn
        self.handle = cfa_mlp_create(B, hidden, ffn)

    def close(self):
        if getattr(self, "handle", None):
            cfa_mlp_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def describe(self) -> dict:
        return cfa_mlp_describe(self.handle)

    def set_pipeline(self, blocks_per_sm: int = 0, stages: int = 0) -> None:
        st = cfa_mlp_set_pipeline(self.handle, blocks_per_sm, stages)
        if st != CFA_OK:
            raise CfaError(st, f"pipeline {blocks_per_sm} x {stages}")

    def set_path(self, path: int) -> None:
        """PATH_AUTO (tensor cores from B = 2), PATH_CUDA_CORES or PATH_TENSOR_CORES."""
        st = cfa_mlp_set_path(self.handle, path)
        if st != CFA_OK:
            raise CfaError(st, f"path {path}")

    def status(self) -> int:
        return cfa_mlp_status(self.handle)

    def step(self, h, norm_w, W_gate, W_up, W_down, y, eps: float = 1e-5, stream=None):
        B, H, F = self.B, self.hidden, self.ffn
        for name, t, shape in (("h", h, (B, H)), ("norm_w", norm_w, (H,)),
                               ("W_gate", W_gate, (H, F)), ("W_up", W_up, (H, F)),
                               ("W_down", W_down, (F, H)), ("y", y, (B, H))):
            _check_tensor(name, t, shape)
        st = cfa_mlp_step(self.handle, h, norm_w, eps, W_gate, W_up, W_down, y, stream)
        if st != CFA_OK:
            raise CfaError(st, "cfa_mlp_step")
        return y


class Stack:
    """Owns a cfa_stack: n_layers decoder layers run token by token.

    layers: sequence of mappings with attn_norm, W_qkv, W_o, k_cache, v_cache,
    mlp_norm, W_gate, W_up, W_down (device bf16 tensors, kept referenced here
    so they outlive the stack's use of them)."""

    _KEYS = ("attn_norm", "W_qkv", "W_o", "k_cache", "v_cache", "mlp_norm", "W_gate", "W_up",
             "W_down")

    def __init__(self, n_layers: int, B: int, hidden: int, n_heads: int, head_dim: int,
                 ffn: int, max_ctx: int, layers=None):
        self.n_layers, self.B, self.hidden, self.n_heads, self.head_dim = (
            n_layers, B, hidden, n_heads, head_dim)
        self.ffn, self.max_ctx = ffn, max_ctx
        self.handle = cfa_stack_create(n_layers, B, hidden, n_heads, head_dim, ffn, max_ctx)
        self._layers = [None] * n_layers
        if layers is not None:
            for i, layer in enumerate(layers):
                self.set_layer(i, layer)

    def close(self):
        if getattr(self, "handle", None):
            cfa_stack_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def describe(self) -> dict:
        return cfa_stack_describe(self.handle)

    def status(self) -> int:
        return cfa_stack_status(self.handle)

    def set_layer(self, i: int, layer) -> None:
        B, H, nh, d, F, mc = (self.B, self.hidden, self.n_heads, self.head_dim, self.ffn,
                              self.max_ctx)
        shapes = {"attn_norm": (H,), "W_qkv": (H, 3 * H), "W_o": (H, H),
                  "k_cache": (B, nh, mc, d), "v_cache": (B, nh, mc, d), "mlp_norm": (H,),
                  "W_gate": (H, F), "W_up": (H, F), "W_down": (F, H)}
        for k in self._KEYS:
            _check_tensor(k, layer[k], shapes[k])
        st = cfa_stack_set_layer(self.handle, i, *[layer[k] for k in self._KEYS])
        if st != CFA_OK:
            raise CfaError(st, f"cfa_stack_set_layer({i})")
        self._layers[i] = {k: layer[k] for k in self._KEYS}

    def _check_io(self, x, positions, out):
        _check_tensor("x", x, (self.B, self.hidden))
        _check_tensor("out", out, (self.B, self.hidden))
        _check_tensor("positions", positions, (self.B,), torch.int32)

    def step(self, x, positions, out, rope_theta: float = 10000.0, eps: float = 1e-5,
             advance: bool = False, stream=None):
        """One token through every layer (eager launches)."""
        self._check_io(x, positions, out)
        st = cfa_stack_step(self.handle, x, positions, rope_theta, eps, advance, out, stream)
        if st != CFA_OK:
            raise CfaError(st, "cfa_stack_step")
        return out

    def step_graph(self, x, positions, out, rope_theta: float = 10000.0, eps: float = 1e-5,
                   advance: bool = False, stream=None):
        """One token through every layer, recorded once into a CUDA graph and
        replayed; `stream` must not be the legacy default stream."""
        self._check_io(x, positions, out)
        st = cfa_stack_step_graph(self.handle, x, positions, rope_theta, eps, advance, out,
                                  stream)
        if st != CFA_OK:
            raise CfaError(st, "cfa_stack_step_graph")
        return out


# ------------------------------------------------ multi-head latent attention

MLA_KV, MLA_NOPE, MLA_ROPE, MLA_V = 512, 128, 64, 128
MLA_ROW = MLA_KV + MLA_ROPE


def cfa_mla_create(B: int, hidden: int, n_heads: int, q_lora: int, max_ctx: int) -> int:
    h = _lib.cfa_mla_create(B, hidden, n_heads, q_lora, max_ctx)
    if not h:
        raise CfaError(cfa_last_error(), "cfa_mla_create")
    return h


def cfa_mla_destroy(mla: int) -> None:
    _lib.cfa_mla_destroy(mla)


def cfa_mla_step(mla, x, W_a, g_q, g_kv, W_uq, W_kvb, W_o, cache, ctx_lens, rope_theta: float,
                 eps: float, out, stream=None) -> int:
    lens = (ctypes.c_int * len(ctx_lens))(*[int(v) for v in ctx_lens])
    return int(_lib.cfa_mla_step(mla, _ptr(x), _ptr(W_a), _ptr(g_q), _ptr(g_kv), _ptr(W_uq),
                                 _ptr(W_kvb), _ptr(W_o), _ptr(cache), lens, float(rope_theta),
                                 float(eps), _ptr(out), _stream(stream)))


def cfa_mla_status(mla) -> int:
    return int(_lib.cfa_mla_status(mla))


def cfa_mla_describe(mla) -> dict:
    buf = ctypes.create_string_buffer(1024)
    st = _lib.cfa_mla_describe(mla, buf, len(buf))
    if st != CFA_OK:
        raise CfaError(st, "cfa_mla_describe")
    return json.loads(buf.value.decode())


def cfa_mla_set_row_splits(mla, splits: int) -> int:
    return int(_lib.cfa_mla_set_row_splits(mla, int(splits)))


class Mla:
    """Owns a cfa_mla: DeepSeek-style latent-attention decode steps."""

    _KEYS = ("W_a", "g_q", "g_kv", "W_uq", "W_kvb", "W_o")

    def __init__(self, B: int, hidden: int, n_heads: int, q_lora: int, max_ctx: int):
        self.B, self.hidden, self.n_heads, self.q_lora, self.max_ctx = (
            B, hidden, n_heads, q_lora, max_ctx)
        self.handle = cfa_mla_create(B, hidden, n_heads, q_lora, max_ctx)

    def close(self):
        if getattr(self, "handle", None):
            cfa_mla_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def describe(self) -> dict:
        return cfa_mla_describe(self.handle)

    def set_row_splits(self, splits: int):
        """1, 2 or 4 clusters per (sequence, head group), each over its share of
        the latent rows (0: chosen per step); raises CfaError if that grid does
        not fit at once."""
        st = cfa_mla_set_row_splits(self.handle, splits)
        if st != CFA_OK:
            raise CfaError(st, "cfa_mla_set_row_splits")

    def status(self) -> int:
        return cfa_mla_status(self.handle)

    def step(self, x, weights, cache, ctx_lens, out, rope_theta: float = 10000.0,
             eps: float = 1e-6, stream=None):
        B, H, nh, ql, mc = self.B, self.hidden, self.n_heads, self.q_lora, self.max_ctx
        shapes = {"W_a": (H, ql + MLA_ROW), "g_q": (ql,), "g_kv": (MLA_KV,),
                  "W_uq": (ql, nh * (MLA_NOPE + MLA_ROPE)), "W_kvb": (MLA_KV, nh * (MLA_NOPE + MLA_V)),
                  "W_o": (nh * MLA_V, H)}
        for k in self._KEYS:
            _check_tensor(k, weights[k], shapes[k])
        _check_tensor("x", x, (B, H))
        _check_tensor("out", out, (B, H))
        _check_tensor("cache", cache, (B, mc, MLA_ROW))
        if len(ctx_lens) != B:
            raise ValueError("ctx_lens needs one entry per batch row")
        st = cfa_mla_step(self.handle, x, *[weights[k] for k in self._KEYS], cache, ctx_lens,
                          rope_theta, eps, out, stream)
        if st != CFA_OK:
            raise CfaError(st, "cfa_mla_step")
        return out
