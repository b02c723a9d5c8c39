"""moe_forward_noalloc: the allocation-free forward entry point.

It serves callers that cannot call cudaMalloc (a process whose device memory
belongs to another allocator, or one that must not allocate once serving), so
its scratch is a fixed array inside the library.  Checked here through the C
ABI against the existing moe_forward entry point and against the fp64 oracle
directly (it runs other kernels than moe_forward: the separate router,
dispatch, gather and combine kernels and single-CTA GEMMs), on two calls in a
row (the second call reuses the array the first one left behind), plus its
size limit, recomputed here from the formula the header documents.
This file is collected last on purpose: it must pass alone in a fresh process
and after every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, check_route, reference_selection, y_to_numpy
from sparse_mixture_experts_54_b300 import _lib, inputs
from sparse_mixture_experts_54_b300.layer import MoELayer

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20


def documented_bytes(T, d, d_ff, n, k, es):
    """Scratch one call needs, as include/moe.h states it: 256-byte-rounded regions
    of 4*k*T bytes (four of them), (3n+2)*4 bytes, k*T*d*es, k*T*d_ff*es and
    k*T*d*4 bytes."""
    up = lambda v: (v + 255) // 256 * 256
    R = k * T
    return 4 * up(4 * R) + up((3 * n + 2) * 4) + up(R * d * es) + up(R * d_ff * es) + up(R * d * 4)


def noalloc(layer, w, y, status, T=None):
    dt = _lib.MOE_F32 if w.dtype == "f32" else _lib.MOE_BF16
    b = layer["bias"]
    return _lib.moe_forward_noalloc(layer["x"].data_ptr(), layer["Wg"].data_ptr(), 0 if b is None else b.data_ptr(),
                                    layer["W1"].data_ptr(), layer["W3"].data_ptr(), layer["W2"].data_ptr(),
                                    y.data_ptr(), layer["x"].shape[0] if T is None else T, w.d, w.d_ff,
                                    w.n_experts, w.k, dt, status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def oracle_check(layer, w, ys, toks, gpu_idx):
    """The noalloc outputs against the fp64 oracle on the listed tokens (routing
    taken from moe_route on the same inputs, near ties switched to its experts)."""
    x, Wg, W1, W3, W2, b = (inputs.to_oracle(layer[k]) for k in ("x", "Wg", "W1", "W3", "W2", "bias"))
    logits = oracle.router_logits(x, Wg, b)
    idx, gate = oracle.select_topk(logits, w.k)
    idx_u, gate_u, near = reference_selection(dict(logits=logits, idx=idx, gate=gate), gpu_idx, w.k)
    y_ref = oracle.moe_tokens(x, W1, W3, W2, idx_u, gate_u, toks)
    for y in ys:
        assert_close(y_to_numpy(y)[toks], y_ref, w.dtype)
    return logits, idx, gate, near


CASES = [
    inputs.workload("tiny_fp32"),
    inputs.Workload("noalloc_f32_n4_k3", T=90, d=128, d_ff=192, n_experts=4, k=3, dtype="f32",
                    router_sigma=0.05, rms_normalise_x=False, seed=23),
    inputs.Workload("noalloc_bf16", T=300, d=512, d_ff=384, seed=21),
    inputs.Workload("noalloc_bias", T=129, d=256, d_ff=256, bias=(0, 0, 1.5, 0, 0, 0.5, 0, 0), seed=22),
    inputs.workload("decode_t32"),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_noalloc_matches_moe_forward_and_oracle_on_two_calls(w):
    layer = inputs.make_layer(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, dtype=w.torch_dtype, bias=layer["bias"])
    y_ref = m.forward(layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    r = m.route(layer["x"], layer["Wg"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y1 = torch.full_like(y_ref, float("nan"))
    y2 = torch.full_like(y_ref, float("nan"))
    assert noalloc(layer, w, y1, status) == _lib.MOE_OK
    assert noalloc(layer, w, y2, status) == _lib.MOE_OK
    torch.cuda.synchronize()
    assert status.item() == 0 and m.status() == 0
    ref = y_to_numpy(y_ref)
    for y in (y1, y2):
        assert_close(y_to_numpy(y), ref, w.dtype)
    gidx, gw = r["topk_idx"].cpu().numpy(), r["topk_w"].cpu().numpy()
    logits, idx, gate, near = oracle_check(layer, w, (y1, y2), np.arange(w.T), gidx)
    check_route(gidx, gw, logits, idx, gate, w.k)
    m.close()


def test_noalloc_mixtral_shape_at_its_largest_batch():
    """bf16 at d=4096, d_ff=14336, k=2: T=314 is the largest batch the array
    holds (its last region, the per-slot outputs, ends 104,192 bytes before the
    end of the 32 MiB) and runs; T=315 is refused before any launch."""
    w = inputs.workload("decode_t32", T=314)
    assert documented_bytes(314, w.d, w.d_ff, 8, 2, 2) <= SCRATCH_BYTES < documented_bytes(315, w.d, w.d_ff, 8, 2, 2)
    assert SCRATCH_BYTES - documented_bytes(314, w.d, w.d_ff, 8, 2, 2) == 104192
    layer = inputs.make_layer(w, "cuda", seed=31)
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k)
    y_ref = m.forward(layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    r = m.route(layer["x"], layer["Wg"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y1 = torch.full_like(y_ref, float("nan"))
    y2 = torch.full_like(y_ref, float("nan"))
    assert noalloc(layer, w, y1, status) == _lib.MOE_OK
    assert noalloc(layer, w, y2, status) == _lib.MOE_OK
    torch.cuda.synchronize()
    assert status.item() == 0
    for y in (y1, y2):
        assert_close(y_to_numpy(y), y_to_numpy(y_ref), "bf16")
    # the last tokens write the end of the array; check them and a seeded sample
    toks = np.union1d(inputs.sample_tokens(w.T, 16, seed=5).numpy(), np.arange(w.T - 8, w.T))
    oracle_check(layer, w, (y1, y2), toks, r["topk_idx"].cpu().numpy())
    # one token more does not fit
    x315 = torch.zeros((315, w.d), dtype=torch.bfloat16, device="cuda")
    y315 = torch.empty_like(x315)
    rc = _lib.moe_forward_noalloc(x315.data_ptr(), layer["Wg"].data_ptr(), 0, layer["W1"].data_ptr(),
                                  layer["W3"].data_ptr(), layer["W2"].data_ptr(), y315.data_ptr(), 315, w.d, w.d_ff,
                                  8, 2, _lib.MOE_BF16, 0, torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.MOE_ERR_SCRATCH_LIMIT
    m.close()


def test_noalloc_allocates_no_device_memory():
    w = CASES[2]
    layer = inputs.make_layer(w, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    assert noalloc(layer, w, y, status) == _lib.MOE_OK    # first call on this device: symbol lookup
    torch.cuda.synchronize()
    for rep in range(2):
        free0, _ = torch.cuda.mem_get_info()
        stats0 = torch.cuda.memory_stats()
        for _ in range(3):
            assert noalloc(layer, w, y, status) == _lib.MOE_OK
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        stats1 = torch.cuda.memory_stats()
        assert free1 == free0, f"round {rep}: device free memory changed by {free1 - free0} bytes"
        for key in ("allocation.all.allocated", "segment.all.allocated", "allocated_bytes.all.allocated"):
            assert stats1.get(key, 0) == stats0.get(key, 0), f"round {rep}: torch allocator counter {key} moved"
    assert status.item() == 0


def test_noalloc_rejects_calls_beyond_its_scratch():
    w = inputs.workload("prefill_t4096")
    x = torch.zeros((315, w.d), dtype=torch.bfloat16, device="cuda")
    Wg = torch.zeros((8, w.d), dtype=torch.float32, device="cuda")
    y = torch.empty_like(x)
    dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")   # never read: rejected before any launch
    s = torch.cuda.current_stream().cuda_stream
    rc = _lib.moe_forward_noalloc(x.data_ptr(), Wg.data_ptr(), 0, dummy.data_ptr(), dummy.data_ptr(),
                                  dummy.data_ptr(), y.data_ptr(), 315, w.d, w.d_ff, 8, 2, _lib.MOE_BF16, 0, s)
    assert rc == _lib.MOE_ERR_SCRATCH_LIMIT
    assert _lib.moe_error_string(rc) == "MOE_ERR_SCRATCH_LIMIT"
    # fp32 at a small shape: the documented formula decides acceptance there too
    d, F, n, k = 128, 256, 8, 2
    T_max = max(T for T in range(1, 20000) if documented_bytes(T, d, F, n, k, 4) <= SCRATCH_BYTES)
    x32 = torch.zeros((T_max + 1, d), dtype=torch.float32, device="cuda")
    rc = _lib.moe_forward_noalloc(x32.data_ptr(), Wg.data_ptr(), 0, dummy.data_ptr(), dummy.data_ptr(),
                                  dummy.data_ptr(), x32.data_ptr(), T_max + 1, d, F, n, k, _lib.MOE_F32, 0, s)
    assert rc == _lib.MOE_ERR_SCRATCH_LIMIT
    # bad arguments are refused before the size check
    assert _lib.moe_forward_noalloc(x.data_ptr(), Wg.data_ptr(), 0, 0, 0, 0, y.data_ptr(), 4, w.d, w.d_ff, 8, 2,
                                    _lib.MOE_BF16, 0, s) == _lib.MOE_ERR_INVALID
