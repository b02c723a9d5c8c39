"""The forward calls' NVTX ranges, recorded through an NVTX injection library.

A profiler that records NVTX attaches to a process through the variable
NVTX_INJECTION64_PATH: the first NVTX call loads the named library and lets it
fill the range functions.  This test builds such a library (a few lines of C
that log pushes and pops to a file), runs moe_forward on its grouped path,
moe_block_forward on its weight-streaming path and one moe_forward_fp8 call in
a child process with it attached, and checks the nesting: one range per call
holding one range per stage, named as the stages of moe_stage_times.
"""
import os
import subprocess
import sys
import textwrap

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu

INJECTION_C = r"""
#include <stdio.h>
#include <stdlib.h>
#include <nvtx3/nvToolsExt.h>

static FILE* g_out;
static int log_push(const char* msg) { fprintf(g_out, "push %s\n", msg ? msg : "(null)"); fflush(g_out); return 0; }
static int log_pop(void) { fprintf(g_out, "pop\n"); fflush(g_out); return 0; }

int InitializeInjectionNvtx2(NvtxGetExportTableFunc_t get_table) {
    const NvtxExportTableCallbacks* cb = (const NvtxExportTableCallbacks*)get_table(NVTX_ETID_CALLBACKS);
    NvtxFunctionTable table = 0;
    unsigned int size = 0;
    if (!cb || !cb->GetModuleFunctionTable(NVTX_CB_MODULE_CORE, &table, &size)) return 0;
    if (size <= NVTX_CBID_CORE_RangePop) return 0;
    g_out = fopen(getenv("MOE_TEST_NVTX_LOG"), "w");
    if (!g_out) return 0;
    *table[NVTX_CBID_CORE_RangePushA] = (NvtxFunctionPointer)log_push;
    *table[NVTX_CBID_CORE_RangePop] = (NvtxFunctionPointer)log_pop;
    return 1;
}
"""

CHILD = textwrap.dedent("""
    import sys, torch
    sys.path.insert(0, {root!r})
    from sparse_mixture_experts_54_b300 import _lib, inputs
    from sparse_mixture_experts_54_b300.layer import MoELayer
    w = inputs.Workload("nvtx", T=300, d=256, d_ff=256, seed=3)
    layer = inputs.make_layer(w, "cuda")
    args = (layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    x40 = layer["x"][:40].contiguous()
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k)
    m.forward(layer["x"], *args)                    # grouped GEMMs
    h = x40.clone()
    m.block_forward(h, *args, 1e-5)                 # weight-streaming kernels, residual block
    q = [inputs.quantize_e4m3_rows(layer[n]) for n in ("W1", "W3", "W2")]
    m.forward_fp8(x40, layer["Wg"], q[0][0], q[0][1], q[1][0], q[1][1], q[2][0], q[2][1])
    torch.cuda.synchronize()
    assert m.status() == 0
    print("child ok")
""")


def parse(lines):
    """Nested ranges as (name, [children]) trees from push/pop lines."""
    root = ("", [])
    stack = [root]
    for ln in lines:
        if ln.startswith("push "):
            node = (ln[5:], [])
            stack[-1][1].append(node)
            stack.append(node)
        elif ln == "pop":
            assert len(stack) > 1, "pop without push"
            stack.pop()
    assert len(stack) == 1, "unbalanced ranges"
    return root[1]


def test_forward_calls_emit_one_nvtx_range_per_stage(tmp_path):
    lib = tmp_path / "libnvtx_log.so"
    src = tmp_path / "nvtx_log.c"
    src.write_text(INJECTION_C)
    subprocess.check_call(["gcc", "-shared", "-fPIC", "-O1", "-I/usr/local/cuda/include", "-o", str(lib), str(src)])
    log = tmp_path / "ranges.txt"
    env = dict(os.environ, NVTX_INJECTION64_PATH=str(lib), MOE_TEST_NVTX_LOG=str(log))
    out = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], env=env, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stdout + out.stderr
    calls = parse(log.read_text().split("\n"))
    stages = ["route", "expert_w1w3_swiglu", "expert_w2_gate", "combine"]
    assert [c[0] for c in calls] == ["moe_forward", "moe_forward", "moe_forward_fp8"]
    for name, children in calls:
        assert [c[0] for c in children] == stages, (name, children)
        assert all(not c[1] for c in children)
