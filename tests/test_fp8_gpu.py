"""moe_forward_fp8 (e4m3 expert weights, fp32 row scales) on the GPU, both kernels.

* Default (MOE_OPT_FP8_WIDEN = 0): the weight bytes go straight into the e4m3
  tensor-core MMA against token rows split into hi/lo e4m3 rows.  Checked
  against the fp64 oracle on the oracle's own dequantisation of the bytes, and
  against the bf16 path on the dequantised weights, both within the bf16 bound.
* Widening (MOE_OPT_FP8_WIDEN = 1): with power-of-two scales the dequantised
  weights s * q are exact in bf16, and the kernels must reproduce, bit for bit,
  the bf16 weight-streaming path run on those weights; also checked against the
  oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, check_route, reference_selection, y_to_numpy
from sparse_mixture_experts_54_b300 import _lib, inputs
from sparse_mixture_experts_54_b300.layer import MoELayer

pytestmark = pytest.mark.gpu

NAMES = ("W1", "W3", "W2")


def quantize_layer(layer, all_codes=True, scale_factor=1.0):
    """(q, s) per expert tensor; with all_codes, rows 0 and 5 of every expert hold
    every finite e4m3 byte (zeros, subnormals, the largest), ascending / descending."""
    q, s = {}, {}
    codes = inputs.every_e4m3_code(layer["x"].device)
    for name in NAMES:
        q[name], s[name] = inputs.quantize_e4m3_rows(layer[name])
        s[name] = s[name] * scale_factor
        if all_codes:
            m = min(q[name].shape[-1], codes.numel())
            q[name][:, 0, :m] = codes[:m]
            q[name][:, 5, -m:] = codes.flip(0)[:m]
    return q, s


def oracle_y(x, Wg, bias, q, s, K, toks, gpu_idx):
    xo, Wgo, bo = inputs.to_oracle(x), inputs.to_oracle(Wg), inputs.to_oracle(bias)
    W = []
    for n in NAMES:   # one expert at a time: the fp64 temporaries of a Mixtral expert are ~0.5 GB each
        qn, sn = q[n].cpu().numpy(), s[n].cpu().numpy()
        W.append(np.stack([oracle.dequantize_e4m3_rows(qn[e], sn[e]).astype(np.float32) for e in range(qn.shape[0])]))
    logits = oracle.router_logits(xo, Wgo, bo)
    idx, gate = oracle.select_topk(logits, K)
    idx_u, gate_u, near = reference_selection(dict(logits=logits, idx=idx, gate=gate), gpu_idx, K)
    return oracle.moe_tokens(xo, *W, idx_u, gate_u, toks), logits, idx, gate


def run_both(w, layer, q, s, widen=1):
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, bias=layer["bias"])
    m.set_option(_lib.MOE_OPT_FORCE_PATH, 2)
    m.set_option(_lib.MOE_OPT_FP8_WIDEN, widen)
    # the bf16 weight-streaming path with the uniform K split the fp8 kernels use,
    # so that the widened kernels' partial sums are grouped like its own
    m.set_option(_lib.MOE_OPT_DECODE_STREAMK, 0)
    r = m.route(layer["x"], layer["Wg"])
    y8 = m.forward_fp8(layer["x"], layer["Wg"], q["W1"], s["W1"], q["W3"], s["W3"], q["W2"], s["W2"])
    deq = {n: inputs.dequantize_e4m3_rows(q[n], s[n]) for n in NAMES}
    y16 = m.forward(layer["x"], layer["Wg"], deq["W1"], deq["W3"], deq["W2"])
    torch.cuda.synchronize()
    assert m.status() == 0, _lib.moe_error_string(m.status())
    return m, y8, y16, r["topk_idx"].cpu().numpy(), r["topk_w"].cpu().numpy()


FP8_CASES = [
    # T, d, F, n, K
    (1, 256, 256, 8, 2),
    (5, 512, 384, 8, 2),
    (32, 256, 256, 8, 2),
    (64, 512, 256, 8, 2),
    (200, 512, 384, 8, 2),
    (100, 256, 256, 4, 1),
    (77, 256, 384, 8, 3),
    (120, 768, 640, 16, 2),
    (256, 256, 256, 8, 2),
    (16, 256, 256, 8, 8),
    (24, 6144, 256, 8, 2),      # the longest rows the router's staged W_g allows at 8 experts
]


@pytest.mark.parametrize("T,d,F,n,K", FP8_CASES)
def test_fp8_widened_equals_bf16_on_dequantised_weights(T, d, F, n, K):
    w = inputs.Workload("fp8", T=T, d=d, d_ff=F, n_experts=n, k=K, seed=300 + T + d)
    layer = inputs.make_layer(w, "cuda")
    q, s = quantize_layer(layer)
    m, y8, y16, gidx, gw = run_both(w, layer, q, s, widen=1)
    assert torch.equal(y8, y16)
    y_ref, logits, idx, gate = oracle_y(layer["x"], layer["Wg"], layer["bias"], q, s, K, np.arange(T), gidx)
    check_route(gidx, gw, logits, idx, gate, K)
    assert_close(y_to_numpy(y8), y_ref, "bf16")


@pytest.mark.parametrize("T,d,F,n,K", FP8_CASES)
def test_fp8_mma_matches_oracle_and_bf16_path(T, d, F, n, K):
    w = inputs.Workload("fp8", T=T, d=d, d_ff=F, n_experts=n, k=K, seed=300 + T + d)
    layer = inputs.make_layer(w, "cuda")
    q, s = quantize_layer(layer)
    m, y8, y16, gidx, gw = run_both(w, layer, q, s, widen=0)
    y_ref, logits, idx, gate = oracle_y(layer["x"], layer["Wg"], layer["bias"], q, s, K, np.arange(T), gidx)
    check_route(gidx, gw, logits, idx, gate, K)
    err, bound = assert_close(y_to_numpy(y8), y_ref, "bf16")
    assert_close(y_to_numpy(y8), y_to_numpy(y16), "bf16")
    print(f"fp8 e4m3 MMA T={T} d={d} F={F} n={n} K={K}: max err {err:.3e} (bound {bound:.3e})")


@pytest.mark.parametrize("widen", [0, 1])
def test_fp8_all_tokens_to_one_expert_pair_and_deterministic(widen):
    # 200 tokens on experts (5, 2): 224 token columns per item (448 hi/lo columns,
    # two MMAs per K step, for the e4m3 MMA); W1 and W3 run as separate items
    w = inputs.Workload("fp8_skew", T=200, d=256, d_ff=384, bias=(0, 0, 50, 0, 0, 100, 0, 0), seed=8)
    layer = inputs.make_layer(w, "cuda")
    q, s = quantize_layer(layer)
    m, y8, y16, gidx, gw = run_both(w, layer, q, s, widen=widen)
    assert np.all(gidx == [5, 2])
    if widen:
        assert torch.equal(y8, y16)
    else:
        y_ref, *_ = oracle_y(layer["x"], layer["Wg"], layer["bias"], q, s, w.k, np.arange(w.T), gidx)
        assert_close(y_to_numpy(y8), y_ref, "bf16")
    y8b = m.forward_fp8(layer["x"], layer["Wg"], q["W1"], s["W1"], q["W3"], s["W3"], q["W2"], s["W2"])
    assert torch.equal(y8, y8b)


@pytest.mark.parametrize("widen", [0, 1])
def test_fp8_scales_not_powers_of_two(widen):
    # s * 0.75: the row scale multiplies the fp32 accumulator (one rounding), so
    # only the tolerance against the oracle holds, not bitwise equality
    w = inputs.Workload("fp8_s", T=48, d=512, d_ff=384, seed=44)
    layer = inputs.make_layer(w, "cuda")
    q, s = quantize_layer(layer, scale_factor=0.75)
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, bias=layer["bias"])
    m.set_option(_lib.MOE_OPT_FP8_WIDEN, widen)
    r = m.route(layer["x"], layer["Wg"])
    y8 = m.forward_fp8(layer["x"], layer["Wg"], q["W1"], s["W1"], q["W3"], s["W3"], q["W2"], s["W2"])
    torch.cuda.synchronize()
    assert m.status() == 0
    gidx = r["topk_idx"].cpu().numpy()
    y_ref, *_ = oracle_y(layer["x"], layer["Wg"], layer["bias"], q, s, w.k, np.arange(w.T), gidx)
    assert_close(y_to_numpy(y8), y_ref, "bf16")


@pytest.mark.parametrize("widen", [0, 1])
def test_fp8_batches_above_256_run_in_chunks(widen):
    # 600 tokens = chunks of 256, 256, 88; each chunk equals a separate call
    w = inputs.Workload("fp8_chunks", T=600, d=256, d_ff=256, seed=12)
    layer = inputs.make_layer(w, "cuda")
    q, s = quantize_layer(layer)
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, bias=layer["bias"])
    m.set_option(_lib.MOE_OPT_FP8_WIDEN, widen)
    args = (layer["Wg"], q["W1"], s["W1"], q["W3"], s["W3"], q["W2"], s["W2"])
    y = m.forward_fp8(layer["x"], *args)
    parts = [m.forward_fp8(layer["x"][a:b].contiguous(), *args) for a, b in ((0, 256), (256, 512), (512, 600))]
    torch.cuda.synchronize()
    assert m.status() == 0
    assert torch.equal(y, torch.cat(parts))
    gidx = m.route(layer["x"], layer["Wg"])["topk_idx"].cpu().numpy()
    y_ref, *_ = oracle_y(layer["x"], layer["Wg"], layer["bias"], q, s, w.k, np.arange(w.T), gidx)
    assert_close(y_to_numpy(y), y_ref, "bf16")


def test_fp8_argument_errors():
    m = MoELayer(256, 256, 8, 2)
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    Wg = torch.zeros((8, 256), dtype=torch.float32, device="cuda")
    q = torch.zeros((8, 256, 256), dtype=torch.uint8, device="cuda")
    s = torch.ones((8, 256), dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    st = torch.cuda.current_stream().cuda_stream
    # a null scale pointer, a misaligned weight pointer
    assert _lib.moe_forward_fp8(m.ctx, x.data_ptr(), Wg.data_ptr(), q.data_ptr(), None, q.data_ptr(), s.data_ptr(),
                                q.data_ptr(), s.data_ptr(), y.data_ptr(), 4, st) == _lib.MOE_ERR_INVALID
    assert _lib.moe_forward_fp8(m.ctx, x.data_ptr(), Wg.data_ptr(), q.data_ptr() + 1, s.data_ptr(), q.data_ptr(),
                                s.data_ptr(), q.data_ptr(), s.data_ptr(), y.data_ptr(), 4, st) == _lib.MOE_ERR_INVALID
    assert _lib.moe_forward_fp8(m.ctx, x.data_ptr(), Wg.data_ptr(), q.data_ptr(), s.data_ptr(), q.data_ptr(),
                                s.data_ptr(), q.data_ptr(), s.data_ptr(), y.data_ptr(), 0, st) == _lib.MOE_OK
    m32 = MoELayer(256, 256, 8, 2, dtype=torch.float32)   # fp8 weights serve bf16 layers only
    x32 = torch.zeros((4, 256), dtype=torch.float32, device="cuda")
    assert _lib.moe_forward_fp8(m32.ctx, x32.data_ptr(), Wg.data_ptr(), q.data_ptr(), s.data_ptr(), q.data_ptr(),
                                s.data_ptr(), q.data_ptr(), s.data_ptr(), x32.data_ptr(), 4,
                                st) == _lib.MOE_ERR_UNSUPPORTED


@pytest.fixture(scope="module")
def mixtral_fp8():
    """The Mixtral-shape experts quantised to e4m3 with power-of-two row scales,
    and the oracle's own fp64 dequantisation of those bytes.  Every dequantised
    weight is exactly a bf16 value (4 significant bits times a power of two), so
    it is handed to the oracle as bf16 bit patterns; the conversion is checked
    to be exact."""
    w = inputs.workload("decode_t32")
    W1, W3, W2 = inputs.make_experts(w, "cuda")
    q, s = {}, {}
    for name, t in zip(NAMES, (W1, W3, W2)):
        q[name], s[name] = inputs.quantize_e4m3_rows(t)
    del W1, W3, W2
    torch.cuda.empty_cache()
    # the oracle's decoding of every byte value, gathered per weight (the same
    # values as oracle.dequantize_e4m3_rows, without its per-element decode of
    # 1.4 G bytes)
    table = oracle.decode_e4m3(np.arange(256, dtype=np.uint8))
    host = []
    for n in NAMES:
        qn, sn = q[n].cpu().numpy(), s[n].cpu().numpy()
        bits = np.empty(qn.shape, dtype=np.uint16)
        for e in range(qn.shape[0]):   # one expert at a time: fp64 temporaries of ~0.5 GB
            v = (sn[e].astype(np.float64)[:, None] * table[qn[e]]).astype(np.float32)
            u = v.view(np.uint32)
            assert not np.any(u & 0xFFFF), "dequantised weight not exact in bf16"
            bits[e] = (u >> 16).astype(np.uint16)
        host.append(bits)
    return w, q, s, tuple(host)


@pytest.mark.parametrize("T", [1, 8, 32, 128, 256])
def test_mixtral_decode_fp8(mixtral_fp8, T):
    """Mixtral shape, every token, both kernels against the oracle run on its own
    decoding of the e4m3 bytes; the widening kernel bitwise equal to the bf16
    weight-streaming path (uniform K split) on the dequantised weights, the e4m3
    MMA within the bf16 bound of it."""
    w, q, s, host = mixtral_fp8
    x = inputs.make_x(w, "cuda", seed=None if T == 32 else 60 + T, T=T)
    Wg, b = inputs.make_router(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, bias=b)
    m.set_option(_lib.MOE_OPT_FORCE_PATH, 2)
    r = m.route(x, Wg)
    ys = {}
    for widen in (0, 1):
        m.set_option(_lib.MOE_OPT_FP8_WIDEN, widen)
        ys[widen] = m.forward_fp8(x, Wg, q["W1"], s["W1"], q["W3"], s["W3"], q["W2"], s["W2"])
    deq = {n: inputs.dequantize_e4m3_rows(q[n], s[n]) for n in NAMES}
    m.set_option(_lib.MOE_OPT_DECODE_STREAMK, 0)   # the uniform K split of the fp8 kernels
    y16 = m.forward(x, Wg, deq["W1"], deq["W3"], deq["W2"])
    torch.cuda.synchronize()
    assert m.status() == 0
    assert torch.equal(ys[1], y16)
    del deq
    gidx, gw = r["topk_idx"].cpu().numpy(), r["topk_w"].cpu().numpy()
    xo, Wgo, bo = inputs.to_oracle(x), inputs.to_oracle(Wg), inputs.to_oracle(b)
    logits = oracle.router_logits(xo, Wgo, bo)
    idx, gate = oracle.select_topk(logits, w.k)
    near = check_route(gidx, gw, logits, idx, gate, w.k)
    idx_u, gate_u, _ = reference_selection(dict(logits=logits, idx=idx, gate=gate), gidx, w.k)
    y_ref = oracle.moe_tokens(xo, *host, idx_u, gate_u, np.arange(T))
    for widen in (0, 1):
        err, bound = assert_close(y_to_numpy(ys[widen]), y_ref, "bf16")
        print(f"fp8 decode T={T} {'widened' if widen else 'e4m3 MMA'}: max err {err:.3e} (bound {bound:.3e}), "
              f"near ties {near}")
    assert_close(y_to_numpy(ys[0]), y_to_numpy(y16), "bf16")
    m.close()
