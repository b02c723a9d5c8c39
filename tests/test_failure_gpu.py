"""Failure detection without faulting the GPU: a bounded wait that runs out
reports MOE_ERR_TIMEOUT and leaves the context usable; host-side injection of
a workspace allocation failure; argument errors."""
import pytest
import torch

from sparse_mixture_experts_54_b300 import _lib, inputs
from sparse_mixture_experts_54_b300.layer import MoELayer

pytestmark = pytest.mark.gpu


def tiny():
    w = inputs.workload("tiny_fp32")
    return w, inputs.make_layer(w, "cuda")


def test_bounded_wait_times_out_and_context_survives():
    w, layer = tiny()
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, dtype=torch.float32)
    s = torch.cuda.current_stream().cuda_stream
    args = (layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    y0 = m.forward(*args).clone()            # workspace exists before the timeout
    assert _lib.moe_selftest_wait_timeout(m.ctx, 2000, s) == _lib.MOE_OK   # nothing ever arrives: 2 ms limit
    torch.cuda.synchronize()
    assert m.status() == _lib.MOE_ERR_TIMEOUT
    m.clear_status()                         # also resets the kernels' barrier words and counters
    assert m.status() == _lib.MOE_OK
    y = m.forward(*args)
    torch.cuda.synchronize()
    assert m.status() == _lib.MOE_OK and torch.equal(y, y0)


def test_injected_workspace_failure_reports_oom(monkeypatch):
    w, layer = tiny()
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, dtype=torch.float32)
    monkeypatch.setenv("MOE_FAIL_WORKSPACE_ALLOC", "1")
    with pytest.raises(_lib.MoEError) as ei:
        m.forward(layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    assert ei.value.code == _lib.MOE_ERR_OOM
    monkeypatch.delenv("MOE_FAIL_WORKSPACE_ALLOC")
    y = m.forward(layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()


def test_argument_errors():
    w, layer = tiny()
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, dtype=torch.float32)
    s = torch.cuda.current_stream().cuda_stream
    x = layer["x"]
    # misaligned x, negative T, NULL weights
    assert _lib.moe_forward(m.ctx, x.data_ptr() + 4, layer["Wg"].data_ptr(), layer["W1"].data_ptr(),
                            layer["W3"].data_ptr(), layer["W2"].data_ptr(), x.data_ptr(), 4, s) == _lib.MOE_ERR_INVALID
    assert _lib.moe_forward(m.ctx, x.data_ptr(), layer["Wg"].data_ptr(), 0, 0, 0, x.data_ptr(), 4, s) == \
        _lib.MOE_ERR_INVALID
    assert _lib.moe_route(m.ctx, x.data_ptr(), layer["Wg"].data_ptr(), -1, 0, 0, 0, 0, 0, s) == _lib.MOE_ERR_INVALID
    assert _lib.moe_set_dtype(m.ctx, 7) == _lib.MOE_ERR_INVALID
    assert _lib.moe_set_option(m.ctx, 99, 1) == _lib.MOE_ERR_INVALID
    assert _lib.moe_selftest_wait_timeout(m.ctx, 0, s) == _lib.MOE_ERR_INVALID
    assert m.status() == _lib.MOE_OK


def test_workspace_bytes_and_reserve():
    m = MoELayer(4096, 14336, 8, 2)
    b = m.workspace_bytes(4096)
    R = 8192
    assert b >= R * 4096 * 2 + R * 14336 * 2 + R * 4096 * 4
    m.reserve(64)
    assert m.workspace_bytes(64) < b
