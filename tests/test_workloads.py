"""Workload shapes and the seeded input generator (CPU only)."""
import math

import torch

from sparse_mixture_experts_54_b300 import inputs


def test_mixtral_parameter_counts_closed_form():
    # Shapes: 32 layers, d=4096, 32 heads of 128, 8 KV heads, n=8 SwiGLU experts with
    # d_ff=14336 (xyznot "Method"), vocab 32000 (zikao35 part 04), top-2.
    # The pages state 46.7B total and 12.9B active parameters (aiqianji section 2.1.2).
    w = inputs.workload("prefill_t4096")
    L, d, F, n, K = 32, w.d, w.d_ff, w.n_experts, w.k
    heads, kv_heads, hd, vocab = 32, 8, 128, 32000
    expert = 3 * d * F
    attn = d * heads * hd + 2 * d * kv_heads * hd + heads * hd * d
    gate = d * n
    norms = 2 * d
    emb = 2 * vocab * d
    total = L * (n * expert + attn + gate + norms) + emb
    active = L * (K * expert + attn + gate + norms) + emb
    assert round(total / 1e9, 1) == 46.7
    assert round(active / 1e9, 1) == 12.9
    # expert-only weights of the 32-layer stack: ~45B parameters, ~90 GB in bf16
    assert round(L * n * expert / 1e9) == 45 and round(L * n * expert * 2 / 1e9) == 90


def test_generator_is_seeded_and_shaped():
    w = inputs.workload("tiny_fp32")
    a = inputs.make_layer(w)
    b = inputs.make_layer(w)
    for k in ("x", "Wg", "W1", "W3", "W2"):
        assert torch.equal(a[k], b[k])
    assert a["x"].shape == (64, 128) and a["x"].dtype == torch.float32
    assert a["W1"].shape == (8, 256, 128) and a["W2"].shape == (8, 128, 256)
    assert a["bias"] is None
    c = inputs.make_layer(w, seed=1)
    assert not torch.equal(a["x"], c["x"])
    # distributions: sigma of W1 ~ 1/sqrt(d), W2 ~ 1/sqrt(d_ff), router 0.02
    assert abs(a["W1"].std().item() * math.sqrt(128) - 1) < 0.02
    assert abs(a["W2"].std().item() * math.sqrt(256) - 1) < 0.02
    assert abs(a["Wg"].std().item() / 0.02 - 1) < 0.1


def test_bf16_rows_unit_rms_and_locality():
    w = inputs.workload("skewed_t32768", T=512, d=256, d_ff=512)
    x = inputs.make_x(w)
    assert x.dtype == torch.bfloat16
    rms = x.float().pow(2).mean(1).sqrt()
    assert torch.all((rms - 1).abs() < 0.01)
    # about half the rows are the previous row plus small noise
    diff = (x[1:].float() - x[:-1].float()).pow(2).mean(1).sqrt()
    frac_close = (diff < 0.5).float().mean().item()
    assert 0.4 < frac_close < 0.6
    Wg, b = inputs.make_router(w)
    assert b.tolist() == [1.5, 0.5, 0, 0, 0, 0, -0.5, -1]


def test_to_oracle_keeps_bits():
    t = torch.tensor([1.0, -2.0, 0.25], dtype=torch.bfloat16)
    assert inputs.to_oracle(t).tolist() == [0x3F80, 0xC000, 0x3E80]


def test_sample_tokens():
    s = inputs.sample_tokens(4096, 512)
    assert s.numel() == 512 and torch.all(s[1:] > s[:-1]) and s.max() < 4096
    assert torch.equal(s, inputs.sample_tokens(4096, 512))
    assert torch.equal(inputs.sample_tokens(10, 50), torch.arange(10))
