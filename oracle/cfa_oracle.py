"""ctypes wrapper around the fp64 C oracle in ``cfa_oracle.c``.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module. The product path (the
CUDA library and its binding) never imports it and fails loudly when its own
extension is missing instead of falling back here.

Cited page: "ClusterFusion框架解析：LLM推理优化的集群通信革命" (ClusterFusion
framework analysis), written [CF §n]. The arithmetic lives in the C file;
this module only moves arrays across the boundary.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "cfa_oracle.c"), os.path.join(_HERE, "cfa_oracle_layer.c"),
         os.path.join(_HERE, "cfa_oracle_mla.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libcfa_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when the compiler has it)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and all(os.path.getmtime(_LIB_PATH) >= os.path.getmtime(s) for s in _SRCS)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", *_SRCS, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.cfa_oracle_decode_step.restype = ctypes.c_int
            lib.cfa_oracle_decode_step.argtypes = (
                [ctypes.c_int] * 6 + [_u16p] * 5 + [_dp] * 4 + [ctypes.c_int])
            lib.cfa_oracle_attention.restype = None
            lib.cfa_oracle_attention.argtypes = [
                ctypes.c_int, ctypes.c_int, _dp, _dp, _dp, ctypes.c_double, _dp]
            lib.cfa_oracle_split_partial.restype = None
            lib.cfa_oracle_split_partial.argtypes = [
                ctypes.c_int, ctypes.c_int, ctypes.c_int, _dp, _dp, _dp,
                ctypes.c_double, _dp, _dp, _dp]
            lib.cfa_oracle_split_combine.restype = None
            lib.cfa_oracle_split_combine.argtypes = [
                ctypes.c_int, ctypes.c_int, _dp, _dp, _dp, _dp]
            lib.cfa_oracle_widen_bf16.restype = None
            lib.cfa_oracle_widen_bf16.argtypes = [_u16p, _dp, ctypes.c_long]
            lib.cfa_oracle_decode_step_ex.restype = ctypes.c_int
            lib.cfa_oracle_decode_step_ex.argtypes = (
                [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int), ctypes.c_double]
                + [_u16p] * 5 + [_dp] * 4 + [ctypes.c_int])
            lib.cfa_oracle_rope.restype = None
            lib.cfa_oracle_rope.argtypes = [ctypes.c_int, _dp, ctypes.c_int, ctypes.c_double, _dp]
            lib.cfa_oracle_round_bf16.restype = ctypes.c_uint16
            lib.cfa_oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.cfa_oracle_round_bf16_array.restype = None
            lib.cfa_oracle_round_bf16_array.argtypes = [_dp, _u16p, ctypes.c_long]
            lib.cfa_oracle_rmsnorm.restype = None
            lib.cfa_oracle_rmsnorm.argtypes = [ctypes.c_int, _dp, _dp, ctypes.c_double, _dp]
            lib.cfa_oracle_silu.restype = ctypes.c_double
            lib.cfa_oracle_silu.argtypes = [ctypes.c_double]
            lib.cfa_oracle_rmsnorm_bf16.restype = ctypes.c_int
            lib.cfa_oracle_rmsnorm_bf16.argtypes = [ctypes.c_int, ctypes.c_int, _u16p, _u16p,
                                                    ctypes.c_double, _u16p]
            lib.cfa_oracle_mlp.restype = ctypes.c_int
            lib.cfa_oracle_mlp.argtypes = (
                [ctypes.c_int] * 3 + [ctypes.c_double] + [_u16p] * 6 + [_dp, _u16p, ctypes.c_int])
            lib.cfa_oracle_layer_step.restype = ctypes.c_int
            lib.cfa_oracle_layer_step.argtypes = (
                [ctypes.c_int] * 6 + [ctypes.POINTER(ctypes.c_int), ctypes.c_double, ctypes.c_double]
                + [_u16p] * 10 + [_u16p] * 4 + [_dp, _dp, ctypes.c_int])
            lib.cfa_oracle_attention_kv.restype = None
            lib.cfa_oracle_attention_kv.argtypes = [ctypes.c_int] * 3 + [_dp] * 3 + [ctypes.c_double, _dp]
            lib.cfa_oracle_mla_step.restype = ctypes.c_int
            lib.cfa_oracle_mla_step.argtypes = (
                [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int), ctypes.c_double, ctypes.c_double]
                + [_u16p] * 8 + [_dp] * 4 + [ctypes.c_int])
            lib.cfa_oracle_threads.restype = ctypes.c_int
            lib.cfa_oracle_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def _bits(a) -> np.ndarray:
    """bf16 data as a contiguous uint16 array of bit patterns.

    Accepts a numpy uint16 array or a CPU torch bf16 tensor.
    """
    if isinstance(a, np.ndarray):
        if a.dtype != np.uint16:
            raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
        return np.ascontiguousarray(a)
    import torch  # only for tensor inputs
    if a.dtype != torch.bfloat16:
        raise TypeError("oracle inputs must be bf16")
    return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def widen(bits) -> np.ndarray:
    """Exact bf16 -> float64 widening of a bit-pattern array."""
    b = _bits(bits)
    out = np.empty(b.shape, dtype=np.float64)
    _load().cfa_oracle_widen_bf16(b.ctypes.data_as(_u16p),
                                  out.ctypes.data_as(_dp), b.size)
    return out


def threads_used(n: int) -> int:
    return int(_load().cfa_oracle_threads(int(n)))


def decode_step(x, W_qkv, W_o, k_cache, v_cache, ctx_len: int, nthreads: int = 1):
    """fp64 result of one decode step [CF §1.1, §3.2, §5.1].

    x [B, H], W_qkv [H, 3H], W_o [H, H], caches [B, nh, max_ctx, d] (bf16).
    Returns dict(out [B, H], k_new [B, nh, d], v_new [B, nh, d],
    attn [B, nh, d]) as float64 arrays.
    """
    xb, wq, wo, kc, vc = (_bits(t) for t in (x, W_qkv, W_o, k_cache, v_cache))
    B, H = xb.shape
    _, nh, max_ctx, d = kc.shape
    if wq.shape != (H, 3 * H) or wo.shape != (H, H) or vc.shape != kc.shape \
            or kc.shape[0] != B or nh * d != H:
        raise ValueError("inconsistent shapes")
    out = np.empty((B, H), np.float64)
    k_new = np.empty((B, nh, d), np.float64)
    v_new = np.empty((B, nh, d), np.float64)
    attn = np.empty((B, nh, d), np.float64)
    rc = _load().cfa_oracle_decode_step(
        B, H, nh, d, max_ctx, int(ctx_len),
        xb.ctypes.data_as(_u16p), wq.ctypes.data_as(_u16p), wo.ctypes.data_as(_u16p),
        kc.ctypes.data_as(_u16p), vc.ctypes.data_as(_u16p),
        out.ctypes.data_as(_dp), k_new.ctypes.data_as(_dp),
        v_new.ctypes.data_as(_dp), attn.ctypes.data_as(_dp), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return {"out": out, "k_new": k_new, "v_new": v_new, "attn": attn}


def attention(q, K, V, scale: float) -> np.ndarray:
    """Monolithic single-query softmax attention in fp64 [CF §1.1]."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    T, d = K.shape
    a = np.empty(d, np.float64)
    _load().cfa_oracle_attention(T, d, q.ctypes.data_as(_dp), K.ctypes.data_as(_dp),
                                 V.ctypes.data_as(_dp), float(scale),
                                 a.ctypes.data_as(_dp))
    return a


def split_partial(q, K, V, t0: int, t1: int, scale: float):
    """(m, l, o) of keys [t0, t1) [CF §3.2]."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    d = K.shape[1]
    m = ctypes.c_double()
    l = ctypes.c_double()
    o = np.empty(d, np.float64)
    _load().cfa_oracle_split_partial(int(t0), int(t1), d, q.ctypes.data_as(_dp),
                                     K.ctypes.data_as(_dp), V.ctypes.data_as(_dp),
                                     float(scale), ctypes.byref(m), ctypes.byref(l),
                                     o.ctypes.data_as(_dp))
    return m.value, l.value, o


def split_combine(m, l, o) -> np.ndarray:
    """Two-step max-then-sum combine of split partials [CF §3.1.1, §3.2]."""
    m, l, o = _f64(m), _f64(l), _f64(o)
    n, d = o.shape
    a = np.empty(d, np.float64)
    _load().cfa_oracle_split_combine(n, d, m.ctypes.data_as(_dp), l.ctypes.data_as(_dp),
                                     o.ctypes.data_as(_dp), a.ctypes.data_as(_dp))
    return a


def rope(x, pos: int, theta: float) -> np.ndarray:
    """Rotate-half rotary embedding of x [d] at position pos (fp64)."""
    x = _f64(x)
    y = np.empty_like(x)
    _load().cfa_oracle_rope(x.shape[0], x.ctypes.data_as(_dp), int(pos), float(theta),
                            y.ctypes.data_as(_dp))
    return y


def decode_step_ex(x, W_qkv, W_o, k_cache, v_cache, ctx_lens, rope_theta: float = 0.0,
                   nthreads: int = 1):
    """fp64 decode step with per-sequence context lengths and optional RoPE of
    the new q/k at position ctx_lens[b]. Same outputs as decode_step."""
    xb, wq, wo, kc, vc = (_bits(t) for t in (x, W_qkv, W_o, k_cache, v_cache))
    B, H = xb.shape
    _, nh, max_ctx, d = kc.shape
    lens = np.ascontiguousarray(np.asarray(ctx_lens, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("ctx_lens must have one entry per batch row")
    out = np.empty((B, H), np.float64)
    k_new = np.empty((B, nh, d), np.float64)
    v_new = np.empty((B, nh, d), np.float64)
    attn = np.empty((B, nh, d), np.float64)
    rc = _load().cfa_oracle_decode_step_ex(
        B, H, nh, d, max_ctx, lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
        float(rope_theta),
        xb.ctypes.data_as(_u16p), wq.ctypes.data_as(_u16p), wo.ctypes.data_as(_u16p),
        kc.ctypes.data_as(_u16p), vc.ctypes.data_as(_u16p),
        out.ctypes.data_as(_dp), k_new.ctypes.data_as(_dp),
        v_new.ctypes.data_as(_dp), attn.ctypes.data_as(_dp), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return {"out": out, "k_new": k_new, "v_new": v_new, "attn": attn}


# --------------------------------------------------------------------------
# Decoder layer stack (cfa_oracle_layer.c): RMSNorm, SwiGLU MLP, residuals.


def _u16(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint16)


def round_bf16(v) -> np.ndarray:
    """Round float64 values to bf16 bit patterns, nearest-even, in one step."""
    v = _f64(v)
    out = np.empty(v.shape, np.uint16)
    _load().cfa_oracle_round_bf16_array(v.ctypes.data_as(_dp), out.ctypes.data_as(_u16p), v.size)
    return out


def rmsnorm(x, g, eps: float) -> np.ndarray:
    """fp64 g * x / sqrt(mean(x^2) + eps) of one vector."""
    x, g = _f64(x), _f64(g)
    y = np.empty_like(x)
    _load().cfa_oracle_rmsnorm(x.shape[0], x.ctypes.data_as(_dp), g.ctypes.data_as(_dp),
                               float(eps), y.ctypes.data_as(_dp))
    return y


def silu(z: float) -> float:
    return float(_load().cfa_oracle_silu(float(z)))


def rmsnorm_bf16(x, g, eps: float) -> np.ndarray:
    """Row-wise bf16(rmsnorm(x[b]; g)) of bf16 inputs x [B, n], g [n]; bits out."""
    xb, gb = _bits(x), _bits(g)
    B, n = xb.shape
    if gb.shape != (n,):
        raise ValueError("norm weight must have one entry per column")
    y = np.empty((B, n), np.uint16)
    if _load().cfa_oracle_rmsnorm_bf16(B, n, xb.ctypes.data_as(_u16p), gb.ctypes.data_as(_u16p),
                                       float(eps), y.ctypes.data_as(_u16p)) != 0:
        raise ValueError("oracle rejected the arguments")
    return y


def mlp(h, g, W_gate, W_up, W_down, eps: float, nthreads: int = 1):
    """SwiGLU MLP with pre-norm and residual (see cfa_oracle_layer.c).

    Returns dict(u [B, F] bits, delta [B, H] fp64, y [B, H] bits)."""
    hb, gb, wg, wu, wd = (_bits(t) for t in (h, g, W_gate, W_up, W_down))
    B, H = hb.shape
    F = wg.shape[1]
    if gb.shape != (H,) or wg.shape != (H, F) or wu.shape != (H, F) or wd.shape != (F, H):
        raise ValueError("inconsistent shapes")
    u = np.empty((B, F), np.uint16)
    delta = np.empty((B, H), np.float64)
    y = np.empty((B, H), np.uint16)
    rc = _load().cfa_oracle_mlp(B, H, F, float(eps), hb.ctypes.data_as(_u16p),
                                gb.ctypes.data_as(_u16p), wg.ctypes.data_as(_u16p),
                                wu.ctypes.data_as(_u16p), wd.ctypes.data_as(_u16p),
                                u.ctypes.data_as(_u16p), delta.ctypes.data_as(_dp),
                                y.ctypes.data_as(_u16p), int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return {"u": u, "delta": delta, "y": y}


def layer_step(x, layer, k_cache, v_cache, ctx_lens, rope_theta: float, eps: float,
               nthreads: int = 1):
    """One decoder layer for one token (see cfa_oracle_layer.c).

    layer: mapping with attn_norm [H], W_qkv, W_o, mlp_norm [H], W_gate, W_up,
    W_down (bf16). Returns dict(xn, h, u, y as bits; k_new, v_new fp64)."""
    xb = _bits(x)
    kc, vc = _bits(k_cache), _bits(v_cache)
    g1, wq, wo, g2, wg, wu, wd = (_bits(layer[k]) for k in (
        "attn_norm", "W_qkv", "W_o", "mlp_norm", "W_gate", "W_up", "W_down"))
    B, H = xb.shape
    _, nh, max_ctx, d = kc.shape
    F = wg.shape[1]
    if (g1.shape != (H,) or g2.shape != (H,) or wq.shape != (H, 3 * H) or wo.shape != (H, H)
            or wg.shape != (H, F) or wu.shape != (H, F) or wd.shape != (F, H)
            or vc.shape != kc.shape or kc.shape[0] != B or nh * d != H):
        raise ValueError("inconsistent shapes")
    lens = np.ascontiguousarray(np.asarray(ctx_lens, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("ctx_lens must have one entry per batch row")
    xn = np.empty((B, H), np.uint16)
    hb = np.empty((B, H), np.uint16)
    u = np.empty((B, F), np.uint16)
    y = np.empty((B, H), np.uint16)
    k_new = np.empty((B, nh, d), np.float64)
    v_new = np.empty((B, nh, d), np.float64)
    ptrs = [a.ctypes.data_as(_u16p) for a in (xb, g1, wq, wo, kc, vc, g2, wg, wu, wd)]
    rc = _load().cfa_oracle_layer_step(
        B, H, nh, d, F, max_ctx, lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
        float(rope_theta), float(eps), *ptrs,
        xn.ctypes.data_as(_u16p), hb.ctypes.data_as(_u16p), u.ctypes.data_as(_u16p),
        y.ctypes.data_as(_u16p), k_new.ctypes.data_as(_dp), v_new.ctypes.data_as(_dp),
        int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return {"xn": xn, "h": hb, "u": u, "y": y, "k_new": k_new, "v_new": v_new}


def stack_step(x, layers, caches, ctx_lens, rope_theta: float, eps: float, nthreads: int = 1):
    """One token through every layer of a stack [CF §3.3, §5.1].

    caches: one (k_cache, v_cache) pair of uint16 bit arrays per layer; the
    bf16-rounded new rows are written into them at ctx_lens[b] (in place), as
    the decode loop appends them. Returns (y bits [B, H], per-layer results)."""
    cur = _bits(x)
    per_layer = []
    for layer, (kc, vc) in zip(layers, caches):
        r = layer_step(cur, layer, kc, vc, ctx_lens, rope_theta, eps, nthreads)
        for b, L in enumerate(ctx_lens):
            kc[b, :, L, :] = round_bf16(r["k_new"][b])
            vc[b, :, L, :] = round_bf16(r["v_new"][b])
        per_layer.append(r)
        cur = r["y"]
    return cur, per_layer


# --------------------------------------------------------------------------
# Multi-head latent attention (cfa_oracle_mla.c)

MLA_KV, MLA_NOPE, MLA_ROPE, MLA_V = 512, 128, 64, 128
MLA_QK = MLA_NOPE + MLA_ROPE
MLA_ROW = MLA_KV + MLA_ROPE


def attention_kv(q, K, V, scale: float) -> np.ndarray:
    """Single-query softmax attention with keys [T, dk] and values [T, dv]."""
    q, K, V = _f64(q), _f64(K), _f64(V)
    T, dk = K.shape
    dv = V.shape[1]
    a = np.empty(dv, np.float64)
    _load().cfa_oracle_attention_kv(T, dk, dv, q.ctypes.data_as(_dp), K.ctypes.data_as(_dp),
                                    V.ctypes.data_as(_dp), float(scale), a.ctypes.data_as(_dp))
    return a


def mla_step(x, W_a, g_q, g_kv, W_uq, W_kvb, W_o, cache, ctx_lens, rope_theta: float,
             eps: float, nthreads: int = 1):
    """fp64 MLA decode step (see cfa_oracle_mla.c).

    x [B, H]; W_a [H, q_lora + 576]; g_q [q_lora]; g_kv [512];
    W_uq [q_lora, nh*192]; W_kvb [512, nh*256]; W_o [nh*128, H];
    cache [B, max_ctx, 576]. Returns dict(out [B, H], new_row [B, 576],
    v [B, nh*128], attn [B, nh*128]) as float64 arrays."""
    xb, wa, gq, gkv, wuq, wkvb, wo, cb = (_bits(t) for t in (
        x, W_a, g_q, g_kv, W_uq, W_kvb, W_o, cache))
    B, H = xb.shape
    q_lora = gq.shape[0]
    nh = wuq.shape[1] // MLA_QK
    max_ctx = cb.shape[1]
    if (wa.shape != (H, q_lora + MLA_ROW) or gkv.shape != (MLA_KV,)
            or wuq.shape != (q_lora, nh * MLA_QK) or wkvb.shape != (MLA_KV, nh * (MLA_NOPE + MLA_V))
            or wo.shape != (nh * MLA_V, H) or cb.shape != (B, max_ctx, MLA_ROW)):
        raise ValueError("inconsistent shapes")
    lens = np.ascontiguousarray(np.asarray(ctx_lens, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("ctx_lens must have one entry per batch row")
    out = np.empty((B, H), np.float64)
    new_row = np.empty((B, MLA_ROW), np.float64)
    v = np.empty((B, nh * MLA_V), np.float64)
    attn = np.empty((B, nh * MLA_V), np.float64)
    ptrs = [t.ctypes.data_as(_u16p) for t in (xb, wa, gq, gkv, wuq, wkvb, wo, cb)]
    rc = _load().cfa_oracle_mla_step(
        B, H, nh, q_lora, max_ctx, lens.ctypes.data_as(ctypes.POINTER(ctypes.c_int)),
        float(rope_theta), float(eps), *ptrs, out.ctypes.data_as(_dp),
        new_row.ctypes.data_as(_dp), v.ctypes.data_as(_dp), attn.ctypes.data_as(_dp),
        int(nthreads))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return {"out": out, "new_row": new_row, "v": v, "attn": attn}
