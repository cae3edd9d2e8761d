"""The seeded synthetic inputs and the byte counts every GB/s figure is computed
from. CPU only.

The roofline unit of a step is the bytes it must move from HBM: both weight
matrices once plus the cached rows it reads (the appended row, x and out are
not counted). The figures below are summed by hand from the shapes; the small
cases are also checked against the bytes of the tensors the generator draws.
"""
import dataclasses

import pytest
import torch

from out_proj_block_gb300 import workloads

MB = 1e6


# --------------------------------------------------------------- byte counts


@pytest.mark.parametrize("name,expected", [
    # 2 B x (H x 3H + H x H) + 2 B x 2 (K and V) x nh x d x (rows read)
    ("tiny", 2 * (256 * 768 + 256 * 256) + 4 * 2 * 128 * 64),                      # 589,824
    ("llama7b_b1_ctx1k", 2 * 4 * 4096 ** 2 + 4 * 4096 * 1024),                     # 150,994,944
    ("llama7b_b1_ctx4k", 2 * 4 * 4096 ** 2 + 4 * 4096 * 4096),                     # 201,326,592
    ("llama7b_b16_ctx4k", 2 * 4 * 4096 ** 2 + 16 * 4 * 4096 * 4096),               # 1,207,959,552
    ("llama7b_b1_ctx16k_spiky", 2 * 4 * 4096 ** 2 + 4 * 4096 * 16384),             # 402,653,184
    ("hd64_b8_ctx2k", 2 * 4 * 4096 ** 2 + 8 * 4 * 4096 * 2048),                    # 402,653,184
    ("llama7b_b1_ctx4k_rope", 2 * 4 * 4096 ** 2 + 4 * 4096 * 4096),
    # lengths 1024 + 384 i, i < 16: 16 x 1024 + 384 x 120 = 62,464 rows
    ("llama7b_b16_ragged_rope", 2 * 4 * 4096 ** 2 + 4 * 4096 * 62464),             # 1,157,627,904
])
def test_attention_block_bytes(name, expected):
    assert workloads.WORKLOADS[name].algorithmic_bytes == expected


def test_headline_figures_in_megabytes():
    w = workloads.WORKLOADS
    assert round(w["llama7b_b1_ctx4k"].algorithmic_bytes / MB, 1) == 201.3
    assert round(w["llama7b_b1_ctx1k"].algorithmic_bytes / MB, 1) == 151.0
    assert round(w["llama7b_b16_ctx4k"].algorithmic_bytes / MB, 1) == 1208.0
    assert round(w["llama7b_b16_ragged_rope"].algorithmic_bytes / MB, 1) == 1157.6


@pytest.mark.parametrize("name,expected", [
    # per layer: W_qkv + W_o (4 H^2) + gate, up, down (3 H F), bf16, + K/V rows read
    ("llama7b_32l_b1_ctx1k", 32 * (2 * (4 * 4096 ** 2 + 3 * 4096 * 11008) + 4 * 4096 * 1024)),
    ("llama7b_32l_b16_ctx1k",
     32 * (2 * (4 * 4096 ** 2 + 3 * 4096 * 11008) + 16 * 4 * 4096 * 1024)),
    ("llama7b_2l_b1_ctx1k", 2 * (2 * (4 * 4096 ** 2 + 3 * 4096 * 11008) + 4 * 4096 * 1024)),
])
def test_decode_loop_bytes(name, expected):
    assert workloads.STACKS[name].algorithmic_bytes == expected


# DeepSeek-V3 MLA: W_a [7168, 1536 + 576], W_uq [1536, 128 x 192],
# W_kvb [512, 128 x 256], W_o [128 x 128, 7168], bf16; 576 bf16 per cached row.
V3_WEIGHTS = 2 * (7168 * 2112 + 1536 * 128 * 192 + 512 * 128 * 256 + 128 * 128 * 7168)


def test_mla_bytes():
    m = workloads.MLAS
    assert V3_WEIGHTS == 374_210_560
    assert m["mla_v3_b1_ctx4k"].weight_bytes == V3_WEIGHTS
    assert m["mla_v3_b1_ctx4k"].algorithmic_bytes == V3_WEIGHTS + 4096 * 1152
    assert m["mla_v3_b1_ctx16k"].algorithmic_bytes == V3_WEIGHTS + 16384 * 1152
    assert m["mla_v3_b4_ctx4k"].algorithmic_bytes == V3_WEIGHTS + 4 * 4096 * 1152
    assert round(m["mla_v3_b1_ctx4k"].algorithmic_bytes / MB, 1) == 378.9
    assert round(m["mla_v3_b1_ctx16k"].algorithmic_bytes / MB, 1) == 393.1


def test_bytes_equal_the_tensors_a_step_reads():
    """Ragged lengths, including an empty cache: weights plus rows [0, L_b)."""
    wl = dataclasses.replace(workloads.WORKLOADS["tiny"], B=3, ctx_lens=(0, 5, 63))
    t = workloads.make_inputs(wl, seed=3)
    read = t["W_qkv"].nbytes + t["W_o"].nbytes
    for b, L in enumerate(wl.lens):
        read += t["k_cache"][b, :, :L].nbytes + t["v_cache"][b, :, :L].nbytes
    assert wl.algorithmic_bytes == read

    m = workloads.MLAS["mla_tiny"]
    t = workloads.make_mla_inputs(m, seed=3)
    weights = sum(t[k].nbytes for k in ("W_a", "W_uq", "W_kvb", "W_o"))
    assert m.weight_bytes == weights
    assert m.algorithmic_bytes == weights + t["cache"][0, :m.ctx_len].nbytes


# ------------------------------------------------------------ the recipe


def test_max_ctx_is_the_next_multiple_of_64_above_the_longest_sequence():
    w = workloads.WORKLOADS
    assert w["tiny"].max_ctx == 128  # fixed for the tiny case
    assert w["llama7b_b1_ctx1k"].max_ctx == 1088
    assert w["llama7b_b1_ctx4k"].max_ctx == 4160
    assert w["llama7b_b1_ctx16k_spiky"].max_ctx == 16448
    assert w["llama7b_b16_ragged_rope"].max_ctx == 6848   # longest 6784
    assert workloads.custom(1, 256, 2, 128, 63).max_ctx == 64
    assert workloads.custom(1, 256, 2, 128, 64).max_ctx == 128


def test_ragged_lengths():
    w = workloads.WORKLOADS["llama7b_b16_ragged_rope"]
    assert w.lens == tuple(1024 + 384 * i for i in range(16))
    assert w.rope_theta == 10000.0


def test_inputs_are_seeded_bf16_and_drawn_per_tensor():
    wl = workloads.custom(2, 256, 2, 128, 40, max_ctx=64)
    a = workloads.make_inputs(wl, seed=5)
    b = workloads.make_inputs(wl, seed=5)
    c = workloads.make_inputs(wl, seed=6)
    for k in a:
        assert a[k].dtype == torch.bfloat16
        assert torch.equal(a[k].view(torch.int16), b[k].view(torch.int16)), k
        assert not torch.equal(a[k], c[k]), k
    # one sub-seed per tensor: a longer cache leaves x and the weights as they were
    longer = workloads.make_inputs(workloads.custom(2, 256, 2, 128, 100, max_ctx=128), seed=5)
    for k in ("x", "W_qkv", "W_o"):
        assert torch.equal(a[k], longer[k]), k


def test_input_distributions():
    wl = workloads.custom(4, 1024, 8, 128, 500, max_ctx=512)
    t = workloads.make_inputs(wl, seed=0)
    for k, std in (("x", 1.0), ("W_qkv", 0.02), ("W_o", 0.02), ("k_cache", 1.0), ("v_cache", 1.0)):
        v = t[k].double()
        assert abs(v.mean().item()) < 0.02 * std, k
        assert abs(v.std().item() / std - 1.0) < 0.02, k


def test_spiky_keys_scale_exactly_five_percent_of_each_heads_rows():
    base = workloads.custom(2, 256, 2, 128, 400, max_ctx=448)
    spiky = workloads.custom(2, 256, 2, 128, 400, max_ctx=448, spiky_frac=0.05, spiky_scale=4.0)
    a = workloads.make_inputs(base, seed=2)
    s = workloads.make_inputs(spiky, seed=2)
    assert torch.equal(a["v_cache"], s["v_cache"])
    for b in range(2):
        for h in range(2):
            ka, ks = a["k_cache"][b, h].float(), s["k_cache"][b, h].float()
            changed = (ka != ks).any(dim=1).nonzero().flatten().tolist()
            assert len(changed) == 20                      # round(0.05 x 400)
            assert max(changed) < 400                       # only cached rows
            assert torch.equal(ks[changed], 4.0 * ka[changed])  # x4 is exact in bf16
    # different rows for different heads
    pick = lambda b, h: set((a["k_cache"][b, h] != s["k_cache"][b, h]).any(1).nonzero().flatten().tolist())
    assert pick(0, 0) != pick(0, 1)


def test_poisoned_tail_starts_at_each_length():
    wl = dataclasses.replace(workloads.WORKLOADS["tiny"], B=3, ctx_lens=(0, 5, 63))
    t = workloads.make_inputs(wl, seed=1, poison_tail=True)
    for name in ("k_cache", "v_cache"):
        for b, L in enumerate(wl.lens):
            rows = t[name][b].float()
            assert torch.isfinite(rows[:, :L]).all()
            assert torch.isnan(rows[:, L:]).all()
    m = workloads.MLAS["mla_tiny"]
    t = workloads.make_mla_inputs(m, seed=1, poison_tail=True)
    assert torch.isfinite(t["cache"][:, :m.ctx_len].float()).all()
    assert torch.isnan(t["cache"][:, m.ctx_len:].float()).all()


def test_norm_weights_are_one_plus_small_noise():
    s = workloads.make_stack_inputs(workloads.STACKS["stack_tiny"], seed=0)
    for layer in s["layers"]:
        for k in ("attn_norm", "mlp_norm"):
            g = layer[k].double()
            assert abs(g.mean().item() - 1.0) < 0.03
            assert 0.05 < g.std().item() < 0.15
    m = workloads.make_mla_inputs(workloads.MLAS["mla_tiny"], seed=0)
    assert abs(m["g_kv"].double().mean().item() - 1.0) < 0.03
