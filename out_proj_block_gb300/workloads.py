"""Workload shapes and seeded synthetic inputs.

This module holds no arithmetic of the method: it only names the shapes and
draws seeded random bf16 tensors. Both the CUDA path (tests, bench, smoke) and
the fp64 oracle are fed from here, so the two sides see the same inputs.

Every workload is synthetic (no dataset, no trained weights):
x ~ N(0, 1), W_qkv and W_o ~ N(0, 0.02), cached K and V ~ N(0, 1), all rounded
to bf16. The long-context workload additionally multiplies 5% of the cached
key rows of every (batch, head) by 4, at positions drawn without replacement.
Cache rows at positions >= ctx_len are never part of the computation; they can
be filled with NaN so that a stray read shows up in the result.

Layer stacks (a decode loop over several decoder layers) add, per layer,
RMSNorm weights 1 + N(0, 0.1) and MLP weights W_gate, W_up, W_down
~ N(0, 0.02), all bf16, each layer with its own K/V cache.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import torch


def _round_up(v: int, m: int) -> int:
    return (v + m - 1) // m * m


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    hidden: int
    n_heads: int
    head_dim: int
    ctx_len: int
    max_ctx: int
    spiky_frac: float = 0.0
    spiky_scale: float = 1.0
    description: str = ""
    ctx_lens: Optional[Tuple[int, ...]] = None  # per-sequence lengths; None = ctx_len for all
    rope_theta: float = 0.0                     # > 0: rotary embedding of the new q, k

    @property
    def lens(self) -> Tuple[int, ...]:
        return self.ctx_lens if self.ctx_lens is not None else (self.ctx_len,) * self.B

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes the step must move from HBM: both weights plus the cached K/V
        rows that are read (the appended row, x and out are not counted)."""
        H = self.hidden
        return (2 * H * 3 * H + 2 * H * H
                + sum(self.lens) * 2 * self.n_heads * self.head_dim * 2)

    @property
    def flops(self) -> int:
        H, B = self.hidden, self.B
        return (2 * B * H * 3 * H + 2 * B * H * H
                + sum(L + 1 for L in self.lens) * self.n_heads * self.head_dim * 4)

    def as_config(self) -> Dict[str, object]:
        cfg = {"workload": self.name, "B": self.B, "hidden": self.hidden,
               "n_heads": self.n_heads, "head_dim": self.head_dim,
               "ctx_len": self.ctx_len, "max_ctx": self.max_ctx}
        if self.ctx_lens is not None:
            cfg["ctx_lens"] = list(self.ctx_lens)
        if self.rope_theta > 0:
            cfg["rope_theta"] = self.rope_theta
        return cfg


def _wl(name, B, H, nh, d, L, desc, spiky_frac=0.0, spiky_scale=1.0, max_ctx=None,
        ctx_lens=None, rope_theta=0.0):
    top = max(ctx_lens) if ctx_lens else L
    return Workload(name, B, H, nh, d, L,
                    max_ctx if max_ctx is not None else _round_up(top + 1, 64),
                    spiky_frac, spiky_scale, desc,
                    tuple(ctx_lens) if ctx_lens else None, rope_theta)


WORKLOADS: Dict[str, Workload] = {w.name: w for w in [
    _wl("tiny", 1, 256, 2, 128, 64,
        "tiny block: B=1, hidden 256, 2 heads x 128, ctx_len 64", max_ctx=128),
    _wl("llama7b_b1_ctx1k", 1, 4096, 32, 128, 1024,
        "Llama2-7B-shaped block, B=1, ctx_len 1024"),
    _wl("llama7b_b1_ctx4k", 1, 4096, 32, 128, 4096,
        "Llama2-7B-shaped block, B=1, ctx_len 4096"),
    _wl("llama7b_b16_ctx4k", 16, 4096, 32, 128, 4096,
        "Llama2-7B-shaped block, B=16, ctx_len 4096, per-sequence caches"),
    _wl("llama7b_b1_ctx16k_spiky", 1, 4096, 32, 128, 16384,
        "Llama2-7B-shaped block, B=1, ctx_len 16384, 5% of keys x4",
        spiky_frac=0.05, spiky_scale=4.0),
    _wl("hd64_b8_ctx2k", 8, 4096, 64, 64, 2048,
        "hidden 4096, 64 heads x 64, B=8, ctx_len 2048"),
    # Widened steps: per-sequence lengths and rotary embedding (base 10000).
    _wl("llama7b_b1_ctx4k_rope", 1, 4096, 32, 128, 4096,
        "Llama2-7B-shaped block, B=1, ctx_len 4096, RoPE", rope_theta=10000.0),
    _wl("llama7b_b16_ragged_rope", 16, 4096, 32, 128, 4096,
        "Llama2-7B-shaped block, B=16, ctx_lens 1024..6784 (step 384), RoPE",
        ctx_lens=[1024 + 384 * i for i in range(16)], rope_theta=10000.0),
]}


def custom(B: int, hidden: int, n_heads: int, head_dim: int, ctx_len: int,
           max_ctx: Optional[int] = None, name: str = "custom",
           spiky_frac: float = 0.0, spiky_scale: float = 1.0) -> Workload:
    return _wl(name, B, hidden, n_heads, head_dim, ctx_len,
               f"{name}: B={B}, hidden {hidden}, {n_heads}x{head_dim}, ctx_len {ctx_len}",
               spiky_frac, spiky_scale, max_ctx)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std: float, device, seed: int) -> torch.Tensor:
    t = torch.randn(*shape, generator=_gen(device, seed), device=device,
                    dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def make_inputs(wl: Workload, seed: int = 0, device="cpu",
                poison_tail: bool = False) -> Dict[str, torch.Tensor]:
    """Seeded bf16 inputs of workload ``wl`` on ``device``.

    Each tensor has its own sub-seed, so a tensor does not depend on which
    other tensors were drawn. ``poison_tail`` fills cache rows at positions
    >= ctx_len with NaN.
    """
    device = torch.device(device)
    B, H, nh, d, L, mc = wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.ctx_len, wl.max_ctx
    s = 1000003 * (seed + 1)
    x = _normal((B, H), 1.0, device, s + 1)
    W_qkv = _normal((H, 3 * H), 0.02, device, s + 2)
    W_o = _normal((H, H), 0.02, device, s + 3)
    k_cache = _normal((B, nh, mc, d), 1.0, device, s + 4)
    v_cache = _normal((B, nh, mc, d), 1.0, device, s + 5)
    if wl.spiky_frac > 0.0 and L > 0:
        n_spiky = max(1, int(round(wl.spiky_frac * L)))
        g = _gen("cpu", s + 6)
        for b in range(B):
            for h in range(nh):
                pos = torch.randperm(L, generator=g)[:n_spiky].to(device)
                k_cache[b, h, pos] = k_cache[b, h, pos] * wl.spiky_scale
    if poison_tail:
        for b, Lb in enumerate(wl.lens):
            if Lb < mc:
                k_cache[b, :, Lb:, :] = float("nan")
                v_cache[b, :, Lb:, :] = float("nan")
    return {"x": x, "W_qkv": W_qkv, "W_o": W_o, "k_cache": k_cache, "v_cache": v_cache}


# --------------------------------------------------------------------------
# Layer stacks: the decode loop over n_layers decoder layers.


@dataclasses.dataclass(frozen=True)
class StackWorkload:
    name: str
    n_layers: int
    B: int
    hidden: int
    n_heads: int
    head_dim: int
    ffn: int
    ctx_len: int
    max_ctx: int
    rope_theta: float = 10000.0
    eps: float = 1e-5
    description: str = ""

    @property
    def lens(self) -> Tuple[int, ...]:
        return (self.ctx_len,) * self.B

    @property
    def layer_weight_bytes(self) -> int:
        H, F = self.hidden, self.ffn
        return 2 * (3 * H * H + H * H + 3 * H * F)

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes one token must move from HBM: every layer's weight matrices plus
        the cached K/V rows it reads (norm weights, activations and the appended
        rows are not counted)."""
        kv = sum(self.lens) * 2 * self.n_heads * self.head_dim * 2
        return self.n_layers * (self.layer_weight_bytes + kv)

    def as_config(self) -> Dict[str, object]:
        return {"workload": self.name, "n_layers": self.n_layers, "B": self.B,
                "hidden": self.hidden, "n_heads": self.n_heads, "head_dim": self.head_dim,
                "ffn": self.ffn, "ctx_len": self.ctx_len, "max_ctx": self.max_ctx,
                "rope_theta": self.rope_theta, "eps": self.eps}


def _sw(name, n_layers, B, H, nh, d, F, L, desc, max_ctx=None, rope_theta=10000.0, eps=1e-5):
    return StackWorkload(name, n_layers, B, H, nh, d, F, L,
                         max_ctx if max_ctx is not None else _round_up(L + 1, 64),
                         rope_theta, eps, desc)


STACKS: Dict[str, StackWorkload] = {w.name: w for w in [
    _sw("stack_tiny", 2, 1, 256, 2, 128, 512, 64,
        "2 tiny layers: hidden 256, 2 heads x 128, ffn 512, ctx_len 64", max_ctx=128),
    _sw("llama7b_2l_b1_ctx1k", 2, 1, 4096, 32, 128, 11008, 1024,
        "2 Llama2-7B-shaped layers (SwiGLU MLP, ffn 11008), B=1, ctx_len 1024"),
    _sw("llama7b_2l_b16_ctx1k", 2, 16, 4096, 32, 128, 11008, 1024,
        "2 Llama2-7B-shaped layers (SwiGLU MLP, ffn 11008), B=16, ctx_len 1024"),
    _sw("llama7b_32l_b1_ctx1k", 32, 1, 4096, 32, 128, 11008, 1024,
        "32 Llama2-7B-shaped layers (SwiGLU MLP, ffn 11008), B=1, ctx_len 1024"),
    _sw("llama7b_32l_b16_ctx1k", 32, 16, 4096, 32, 128, 11008, 1024,
        "32 Llama2-7B-shaped layers (SwiGLU MLP, ffn 11008), B=16, ctx_len 1024"),
]}


def custom_stack(n_layers: int, B: int, hidden: int, n_heads: int, head_dim: int, ffn: int,
                 ctx_len: int, max_ctx: Optional[int] = None, rope_theta: float = 10000.0,
                 eps: float = 1e-5, name: str = "custom_stack") -> StackWorkload:
    return _sw(name, n_layers, B, hidden, n_heads, head_dim, ffn, ctx_len,
               f"{name}: {n_layers} layers, B={B}, hidden {hidden}, {n_heads}x{head_dim}, "
               f"ffn {ffn}, ctx_len {ctx_len}", max_ctx, rope_theta, eps)


def make_stack_inputs(wl: StackWorkload, seed: int = 0, device="cpu",
                      poison_tail: bool = False) -> Dict[str, object]:
    """Seeded bf16 inputs of a layer stack: x [B, H] and one dict per layer
    (attn_norm, W_qkv, W_o, mlp_norm, W_gate, W_up, W_down, k_cache, v_cache).
    ``poison_tail`` fills cache rows at positions >= ctx_len with NaN."""
    device = torch.device(device)
    B, H, nh, d, F, L, mc = (wl.B, wl.hidden, wl.n_heads, wl.head_dim, wl.ffn, wl.ctx_len,
                             wl.max_ctx)
    s = 7000003 * (seed + 1)
    x = _normal((B, H), 1.0, device, s + 1)
    layers = []
    for l in range(wl.n_layers):
        t = s + 100 * (l + 1)
        layer = {
            "attn_norm": (_normal((H,), 0.1, device, t + 1).float() + 1.0).to(torch.bfloat16),
            "W_qkv": _normal((H, 3 * H), 0.02, device, t + 2),
            "W_o": _normal((H, H), 0.02, device, t + 3),
            "mlp_norm": (_normal((H,), 0.1, device, t + 4).float() + 1.0).to(torch.bfloat16),
            "W_gate": _normal((H, F), 0.02, device, t + 5),
            "W_up": _normal((H, F), 0.02, device, t + 6),
            "W_down": _normal((F, H), 0.02, device, t + 7),
            "k_cache": _normal((B, nh, mc, d), 1.0, device, t + 8),
            "v_cache": _normal((B, nh, mc, d), 1.0, device, t + 9),
        }
        if poison_tail and L < mc:
            layer["k_cache"][:, :, L:, :] = float("nan")
            layer["v_cache"][:, :, L:, :] = float("nan")
        layers.append(layer)
    return {"x": x, "layers": layers}


# --------------------------------------------------------------------------
# Multi-head latent attention (DeepSeek-V2/V3 dimensions: latent 512, per-head
# nope / rope / value widths 128 / 64 / 128). Inputs: x ~ N(0, 1); W_a, W_uq,
# W_kvb, W_o ~ N(0, 0.02); norm weights 1 + N(0, 0.1); latent cache rows
# ~ N(0, 1); all bf16.

MLA_KV, MLA_NOPE, MLA_ROPE, MLA_V = 512, 128, 64, 128
MLA_ROW = MLA_KV + MLA_ROPE


@dataclasses.dataclass(frozen=True)
class MlaWorkload:
    name: str
    B: int
    hidden: int
    n_heads: int
    q_lora: int
    ctx_len: int
    max_ctx: int
    rope_theta: float = 10000.0
    eps: float = 1e-6
    description: str = ""

    @property
    def lens(self) -> Tuple[int, ...]:
        return (self.ctx_len,) * self.B

    @property
    def weight_bytes(self) -> int:
        H, nh, ql = self.hidden, self.n_heads, self.q_lora
        return 2 * (H * (ql + MLA_ROW) + ql * nh * (MLA_NOPE + MLA_ROPE)
                    + MLA_KV * nh * (MLA_NOPE + MLA_V) + nh * MLA_V * H)

    @property
    def algorithmic_bytes(self) -> int:
        """Every weight once plus the latent cache rows read."""
        return self.weight_bytes + sum(self.lens) * MLA_ROW * 2

    @property
    def attention_flops(self) -> int:
        """Multiply-adds x 2 of the latent attention in absorbed form:
        q absorption, scores over 576 dims, latent output, value projection."""
        nh = self.n_heads
        per_b = [nh * (2 * MLA_KV * MLA_NOPE + (L + 1) * (MLA_ROW + MLA_KV) + MLA_KV * MLA_V)
                 for L in self.lens]
        return 2 * sum(per_b)

    def as_config(self) -> Dict[str, object]:
        return {"workload": self.name, "B": self.B, "hidden": self.hidden,
                "n_heads": self.n_heads, "q_lora": self.q_lora, "kv_lora": MLA_KV,
                "qk_nope": MLA_NOPE, "qk_rope": MLA_ROPE, "v_head": MLA_V,
                "ctx_len": self.ctx_len, "max_ctx": self.max_ctx,
                "rope_theta": self.rope_theta, "eps": self.eps}


def _mw(name, B, H, nh, ql, L, desc, max_ctx=None, rope_theta=10000.0, eps=1e-6):
    return MlaWorkload(name, B, H, nh, ql, L,
                       max_ctx if max_ctx is not None else _round_up(L + 1, 64),
                       rope_theta, eps, desc)


MLAS: Dict[str, MlaWorkload] = {w.name: w for w in [
    _mw("mla_tiny", 1, 256, 2, 128, 64, "MLA, hidden 256, 2 heads, q_lora 128, ctx_len 64",
        max_ctx=128),
    _mw("mla_v3_b1_ctx4k", 1, 7168, 128, 1536, 4096,
        "DeepSeek-V3-shaped MLA (hidden 7168, 128 heads, q_lora 1536), B=1, ctx_len 4096"),
    _mw("mla_v3_b1_ctx16k", 1, 7168, 128, 1536, 16384,
        "DeepSeek-V3-shaped MLA (hidden 7168, 128 heads, q_lora 1536), B=1, ctx_len 16384"),
    _mw("mla_v3_b4_ctx4k", 4, 7168, 128, 1536, 4096,
        "DeepSeek-V3-shaped MLA (hidden 7168, 128 heads, q_lora 1536), B=4, ctx_len 4096"),
]}


def custom_mla(B: int, hidden: int, n_heads: int, q_lora: int, ctx_len: int,
               max_ctx: Optional[int] = None, name: str = "custom_mla") -> MlaWorkload:
    return _mw(name, B, hidden, n_heads, q_lora, ctx_len,
               f"{name}: B={B}, hidden {hidden}, {n_heads} heads, q_lora {q_lora}, "
               f"ctx_len {ctx_len}", max_ctx)


def make_mla_inputs(wl: MlaWorkload, seed: int = 0, device="cpu",
                    poison_tail: bool = False) -> Dict[str, torch.Tensor]:
    """Seeded bf16 inputs of an MLA step: x [B, H], W_a [H, q_lora + 576],
    g_q [q_lora], g_kv [512], W_uq [q_lora, nh*192], W_kvb [512, nh*256],
    W_o [nh*128, H], cache [B, max_ctx, 576]. ``poison_tail`` fills cache rows
    at positions >= ctx_len with NaN."""
    device = torch.device(device)
    B, H, nh, ql, L, mc = wl.B, wl.hidden, wl.n_heads, wl.q_lora, wl.ctx_len, wl.max_ctx
    s = 3000017 * (seed + 1)
    t = {
        "x": _normal((B, H), 1.0, device, s + 1),
        "W_a": _normal((H, ql + MLA_ROW), 0.02, device, s + 2),
        "g_q": (_normal((ql,), 0.1, device, s + 3).float() + 1.0).to(torch.bfloat16),
        "g_kv": (_normal((MLA_KV,), 0.1, device, s + 4).float() + 1.0).to(torch.bfloat16),
        "W_uq": _normal((ql, nh * (MLA_NOPE + MLA_ROPE)), 0.02, device, s + 5),
        "W_kvb": _normal((MLA_KV, nh * (MLA_NOPE + MLA_V)), 0.02, device, s + 6),
        "W_o": _normal((nh * MLA_V, H), 0.02, device, s + 7),
        "cache": _normal((B, mc, MLA_ROW), 1.0, device, s + 8),
    }
    if poison_tail and L < mc:
        t["cache"][:, L:, :] = float("nan")
    return t
