"""moe_forward_noalloc: the allocation-free forward entry point.

It serves callers that cannot call cudaMalloc (a process whose device memory
belongs to another allocator, or one that must not allocate once serving), so
its scratch is a fixed array inside the library.  Checked here through the C
ABI against the existing moe_forward entry point, on two calls in a row (the
second call reuses the array the first one left behind), plus its size limit.
This file is collected last on purpose: it must pass alone in a fresh process
and after every other test.
"""
import numpy as np
import pytest
import torch

from parity import assert_close, y_to_numpy
from sparse_mixture_experts_54_b300 import _lib, inputs
from sparse_mixture_experts_54_b300.layer import MoELayer

pytestmark = pytest.mark.gpu


def noalloc(layer, w, y, status):
    dt = _lib.MOE_F32 if w.dtype == "f32" else _lib.MOE_BF16
    b = layer["bias"]
    return _lib.moe_forward_noalloc(layer["x"].data_ptr(), layer["Wg"].data_ptr(), 0 if b is None else b.data_ptr(),
                                    layer["W1"].data_ptr(), layer["W3"].data_ptr(), layer["W2"].data_ptr(),
                                    y.data_ptr(), layer["x"].shape[0], w.d, w.d_ff, w.n_experts, w.k, dt,
                                    status.data_ptr(), torch.cuda.current_stream().cuda_stream)


CASES = [
    inputs.workload("tiny_fp32"),
    inputs.Workload("noalloc_bf16", T=300, d=512, d_ff=384, seed=21),
    inputs.Workload("noalloc_bias", T=129, d=256, d_ff=256, bias=(0, 0, 1.5, 0, 0, 0.5, 0, 0), seed=22),
    inputs.workload("decode_t32"),
]


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_noalloc_matches_moe_forward_on_two_calls(w):
    layer = inputs.make_layer(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, dtype=w.torch_dtype, bias=layer["bias"])
    y_ref = m.forward(layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
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
    m.close()


def test_noalloc_allocates_no_device_memory():
    w = CASES[1]
    layer = inputs.make_layer(w, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.empty((w.T, w.d), dtype=torch.bfloat16, device="cuda")
    assert noalloc(layer, w, y, status) == _lib.MOE_OK    # first call on this device: symbol lookup
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert noalloc(layer, w, y, status) == _lib.MOE_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
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
    # bad arguments are refused before the size check
    assert _lib.moe_forward_noalloc(x.data_ptr(), Wg.data_ptr(), 0, 0, 0, 0, y.data_ptr(), 4, w.d, w.d_ff, 8, 2,
                                    _lib.MOE_BF16, 0, s) == _lib.MOE_ERR_INVALID
