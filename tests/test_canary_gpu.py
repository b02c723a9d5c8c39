"""Out-of-bounds writes: every entry point's output is a slice of a larger
buffer whose rows before and after hold a sentinel; after the call (on each
kernel path) those guard rows must be unchanged."""
import numpy as np
import pytest
import torch

from sparse_mixture_experts_54_b300 import _lib, inputs
from sparse_mixture_experts_54_b300.layer import MoELayer

pytestmark = pytest.mark.gpu

GUARD = 64            # rows of sentinel before and after
SENTINEL = -12345.0   # exactly representable in bf16


def guarded(T, d, dtype, fill=None):
    buf = torch.full((T + 2 * GUARD, d), SENTINEL, dtype=dtype, device="cuda")
    if fill is not None:
        buf[GUARD:GUARD + T] = fill
    return buf, buf[GUARD:GUARD + T]


def assert_guards(buf, T):
    assert torch.all(buf[:GUARD] == SENTINEL), "write before the output"
    assert torch.all(buf[GUARD + T:] == SENTINEL), "write after the output"


@pytest.mark.parametrize("T,path,pair", [(300, 1, 1), (300, 1, 2), (40, 2, 0), (129, 0, 0)])
def test_forward_writes_only_its_output(T, path, pair):
    w = inputs.Workload("canary", T=T, d=512, d_ff=384, seed=T)
    layer = inputs.make_layer(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k)
    m.set_option(_lib.MOE_OPT_FORCE_PATH, path)
    if pair:
        m.set_option(_lib.MOE_OPT_GEMM_PAIR, pair)
    buf, y = guarded(T, w.d, torch.bfloat16)
    m.forward(layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"], y=y)
    torch.cuda.synchronize()
    assert m.status() == 0
    assert_guards(buf, T)
    assert not torch.any(y == SENTINEL)


@pytest.mark.parametrize("T", [40, 300])
def test_block_and_stack_write_only_h(T):
    w = inputs.Workload("canary_blk", T=T, d=256, d_ff=256, seed=T + 1)
    layer = inputs.make_layer(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k)
    buf, h = guarded(T, w.d, torch.bfloat16, fill=layer["x"])
    lw = (layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    m.block_forward(h, *lw)
    m.stack_forward(h, [lw, lw])
    torch.cuda.synchronize()
    assert m.status() == 0
    assert_guards(buf, T)


def test_fp32_and_host_and_noalloc_paths_write_only_their_outputs():
    w = inputs.workload("tiny_fp32")
    layer = inputs.make_layer(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, dtype=torch.float32)
    buf, y = guarded(w.T, w.d, torch.float32)
    m.forward(layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"], y=y)
    torch.cuda.synchronize()
    assert_guards(buf, w.T)
    # host output (pinned), bf16
    wb = inputs.Workload("canary_host", T=200, d=256, d_ff=256, seed=7)
    lb = inputs.make_layer(wb, "cuda")
    mb = MoELayer(wb.d, wb.d_ff, wb.n_experts, wb.k)
    hbuf = torch.full((wb.T + 2 * GUARD, wb.d), SENTINEL, dtype=torch.bfloat16).pin_memory()
    mb.forward_host(lb["x"].cpu().pin_memory(), lb["Wg"], lb["W1"], lb["W3"], lb["W2"], hbuf[GUARD:GUARD + wb.T])
    torch.cuda.synchronize()
    assert_guards(hbuf, wb.T)
    # allocation-free entry point
    nbuf, ny = guarded(wb.T, wb.d, torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _lib.moe_forward_noalloc(lb["x"].data_ptr(), lb["Wg"].data_ptr(), None, lb["W1"].data_ptr(),
                                  lb["W3"].data_ptr(), lb["W2"].data_ptr(), ny.data_ptr(), wb.T, wb.d, wb.d_ff,
                                  wb.n_experts, wb.k, _lib.MOE_BF16, status.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == _lib.MOE_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_guards(nbuf, wb.T)
