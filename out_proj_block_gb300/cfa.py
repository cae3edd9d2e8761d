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
    "cfa_plan_cluster_size",
    "cfa_plan_describe", "cfa_plan_status", "cfa_last_error", "cfa_status_string",
    "cfa_selftest_wait_timeout",
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


def cfa_plan_cluster_size(plan) -> int:
    return int(_lib.cfa_plan_cluster_size(plan))


def cfa_plan_describe(plan) -> dict:
    buf = ctypes.create_string_buffer(1024)
    st = _lib.cfa_plan_describe(plan, buf, len(buf))
    if st != CFA_OK:
        raise CfaError(st, "cfa_plan_describe")
    return json.loads(buf.value.decode())


def cfa_plan_status(plan) -> int:
    return int(_lib.cfa_plan_status(plan))


def cfa_selftest_wait_timeout(limit_us: int, stream=None) -> int:
    return int(_lib.cfa_selftest_wait_timeout(int(limit_us), _stream(stream)))


# ---------------------------------------------------------- tensor-level API


class Plan:
    """Owns a cfa_plan; checks tensors and launches decode steps."""

    def __init__(self, B: int, hidden: int, n_heads: int, head_dim: int, max_ctx: int,
                 cluster_size: Optional[int] = None, stages: Optional[int] = None,
                 overlap: Optional[bool] = None):
        self.B, self.hidden, self.n_heads, self.head_dim, self.max_ctx = (
            B, hidden, n_heads, head_dim, max_ctx)
        self.handle = cfa_plan_create(B, hidden, n_heads, head_dim, max_ctx)
        try:
            if cluster_size is not None:
                self.set_cluster_size(cluster_size)
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
