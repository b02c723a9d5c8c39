"""The whole MoE layer on the GPU (through the C ABI) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity import (EDGE_ROWS, EDGE_ROWS_FINE, assert_close, check_dispatch, check_route, dispatch_sample,
                    reference_selection, y_to_numpy)
from sparse_mixture_experts_54_b300 import _lib, inputs
from sparse_mixture_experts_54_b300.layer import MoELayer

pytestmark = pytest.mark.gpu


def oracle_y(layer, w, toks, gpu_idx):
    x, Wg, W1, W3, W2, b = (inputs.to_oracle(layer[k]) for k in ("x", "Wg", "W1", "W3", "W2", "bias"))
    logits = oracle.router_logits(x, Wg, b)
    idx, gate = oracle.select_topk(logits, w.k)
    ref = dict(logits=logits, idx=idx, gate=gate)
    idx_u, gate_u, near = reference_selection(ref, gpu_idx, w.k)
    y = oracle.moe_tokens(x, W1, W3, W2, idx_u, gate_u, toks)
    return y, ref, near


def run_layer(w, layer, path=0, pair=0, streamk=1):
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, dtype=w.torch_dtype, bias=layer["bias"])
    if path:
        m.set_option(_lib.MOE_OPT_FORCE_PATH, path)
    if pair:
        m.set_option(_lib.MOE_OPT_GEMM_PAIR, pair)
    if not streamk:
        m.set_option(_lib.MOE_OPT_DECODE_STREAMK, 0)
    r = m.route(layer["x"], layer["Wg"])
    y = m.forward(layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    torch.cuda.synchronize()
    assert m.status() == 0, _lib.moe_error_string(m.status())
    return m, y, r["topk_idx"].cpu().numpy(), r["topk_w"].cpu().numpy()


def test_tiny_fp32_full_parity():
    w = inputs.workload("tiny_fp32")
    layer = inputs.make_layer(w, "cuda")
    m, y, gidx, gw = run_layer(w, layer)
    y_ref, ref, near = oracle_y(layer, w, np.arange(w.T), gidx)
    check_route(gidx, gw, ref["logits"], ref["idx"], ref["gate"], w.k)
    err, bound = assert_close(y_to_numpy(y), y_ref, "f32")
    print(f"tiny fp32: max err {err:.3e} (bound {bound:.3e}), near ties {near}")


SMALL_BF16 = [
    # T, d, F, n, K
    (1, 256, 128, 8, 2),
    (5, 256, 256, 8, 2),
    (64, 256, 384, 8, 2),
    (129, 512, 256, 8, 2),
    (1000, 512, 384, 8, 2),
    (300, 256, 256, 4, 1),
    (257, 256, 256, 8, 3),
    (200, 768, 640, 16, 2),
    (200, 256, 256, 8, 8),      # K = n: dense routing, every token to every expert
    (150, 256, 256, 2, 2),      # two experts, both taken
]


# grouped GEMM kernels: 1 = single CTA (128-row tiles), 2 = CTA pairs (256-row tiles)
GEMM_KINDS = [1, 2]


@pytest.mark.parametrize("pair", GEMM_KINDS)
@pytest.mark.parametrize("T,d,F,n,K", SMALL_BF16)
def test_bf16_small_shapes(T, d, F, n, K, pair):
    w = inputs.Workload("small", T=T, d=d, d_ff=F, n_experts=n, k=K, seed=T + d)
    layer = inputs.make_layer(w, "cuda")
    m, y, gidx, gw = run_layer(w, layer, path=1, pair=pair)
    y_ref, ref, near = oracle_y(layer, w, np.arange(T), gidx)
    check_route(gidx, gw, ref["logits"], ref["idx"], ref["gate"], K)
    assert_close(y_to_numpy(y), y_ref, "bf16")


@pytest.mark.parametrize("pair", GEMM_KINDS)
def test_bf16_all_tokens_one_expert_pair(pair):
    # every token to experts (5, 2): two groups of 700 rows (6 single-CTA tiles or
    # 3 pair tiles each, ragged), all other experts empty
    w = inputs.Workload("skew", T=700, d=256, d_ff=256, bias=(0, 0, 50, 0, 0, 100, 0, 0), seed=3)
    layer = inputs.make_layer(w, "cuda")
    m, y, gidx, gw = run_layer(w, layer, path=1, pair=pair)
    assert np.all(gidx == [5, 2])
    y_ref, ref, near = oracle_y(layer, w, np.arange(w.T), gidx)
    assert_close(y_to_numpy(y), y_ref, "bf16")


@pytest.mark.parametrize("T", [128, 129, 256, 257, 384, 513])
def test_pair_tile_boundaries(T):
    # K=1 with every token on expert 3: one group of exactly T rows, so the pair
    # tiles end on, just past and inside a 128/256-row boundary
    w = inputs.Workload("edge", T=T, d=256, d_ff=384, k=1, bias=(0, 0, 0, 80, 0, 0, 0, 0), seed=T)
    layer = inputs.make_layer(w, "cuda")
    _, y1, gidx, _ = run_layer(w, layer, path=1, pair=1)
    _, y2, _, _ = run_layer(w, layer, path=1, pair=2)
    assert np.all(gidx[:, 0] == 3)
    y_ref, ref, near = oracle_y(layer, w, np.arange(T), gidx)
    assert_close(y_to_numpy(y2), y_ref, "bf16")
    assert_close(y_to_numpy(y1), y_ref, "bf16")


def test_pair_and_single_cta_agree_and_are_deterministic():
    w = inputs.Workload("pair_vs_single", T=1500, d=512, d_ff=640, seed=21)
    layer = inputs.make_layer(w, "cuda")
    _, y1, _, _ = run_layer(w, layer, path=1, pair=1)
    _, y2, _, _ = run_layer(w, layer, path=1, pair=2)
    _, y3, _, _ = run_layer(w, layer, path=1, pair=2)
    assert torch.equal(y2, y3)
    assert_close(y_to_numpy(y2), y_to_numpy(y1).astype(np.float64), "bf16")


def test_bf16_fp32_fallback_shape_rejected():
    m = MoELayer(200, 256, 8, 2)   # d not a multiple of 256: no tensor-core tiling
    x = torch.zeros((4, 200), dtype=torch.bfloat16, device="cuda")
    Wg = torch.zeros((8, 200), dtype=torch.float32, device="cuda")
    W = torch.zeros((8, 256, 200), dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros((8, 200, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.MoEError) as ei:
        m.forward(x, Wg, W, W, W2)
    assert ei.value.code == _lib.MOE_ERR_UNSUPPORTED


def test_empty_batch_is_noop():
    w = inputs.workload("tiny_fp32")
    layer = inputs.make_layer(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, dtype=torch.float32)
    x = torch.empty((0, w.d), dtype=torch.float32, device="cuda")
    y = m.forward(x, layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    torch.cuda.synchronize()
    assert y.shape == (0, w.d) and m.status() == 0


def test_forward_is_bitwise_deterministic_and_host_entry_matches():
    w = inputs.Workload("det", T=1000, d=512, d_ff=384, seed=11)
    layer = inputs.make_layer(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k)
    y1 = m.forward(layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"]).clone()
    y2 = m.forward(layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"]).clone()
    xh = layer["x"].cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    m.forward_host(xh, layer["Wg"], layer["W1"], layer["W3"], layer["W2"], yh)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert torch.equal(y1.cpu(), yh)
    assert m.status() == 0


def test_host_entry_back_to_back_calls_keep_their_own_inputs():
    # consecutive host-buffer calls stage their inputs in alternating buffers on the
    # context's copy stream; with no synchronisation between them each result must
    # still be exactly the device-path result for its own input
    w = inputs.Workload("host_pipe", T=700, d=512, d_ff=384, seed=17)
    layer = inputs.make_layer(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k)
    args = (layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    xs = [inputs.make_x(w, "cuda", seed=100 + i) for i in range(5)]
    refs = [m.forward(x, *args).clone() for x in xs]
    xh = [x.cpu().pin_memory() for x in xs]
    yh = [torch.empty_like(h).pin_memory() for h in xh]
    torch.cuda.synchronize()
    for i in range(5):
        m.forward_host(xh[i], *args, yh[i])
    torch.cuda.synchronize()
    assert m.status() == 0
    for i in range(5):
        assert torch.equal(yh[i], refs[i].cpu()), f"call {i}"


@pytest.mark.parametrize("pinned,direct", [(True, 1), (True, 0), (False, 1)])
def test_host_entry_output_routes(pinned, direct):
    # y written by the last kernel straight into pinned host memory, or copied back
    # (pageable output, or the option off): all give the device path's result
    w = inputs.Workload("host_out", T=300, d=512, d_ff=384, seed=19)
    layer = inputs.make_layer(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k)
    m.set_option(_lib.MOE_OPT_HOST_OUTPUT, direct)
    args = (layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    ref = m.forward(layer["x"], *args).cpu()
    xh = layer["x"].cpu()
    yh = torch.empty_like(xh)
    if pinned:
        xh, yh = xh.pin_memory(), yh.pin_memory()
    m.forward_host(xh, *args, yh)
    torch.cuda.synchronize()
    assert m.status() == 0
    assert torch.equal(yh, ref)


@pytest.mark.parametrize("T", [600, 40])
def test_forward_replays_from_a_cuda_graph(T):
    # the routing kernel's barrier words and the combine's counters return to zero
    # after every call, so a captured call replays correctly; each replay must match
    # an eager call on the same input bit for bit (grouped path at T=600, weight
    # streaming at T=40)
    w = inputs.Workload("graph", T=T, d=512, d_ff=384, seed=23 + T)
    layer = inputs.make_layer(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k)
    m.reserve(T)
    args = (layer["Wg"], layer["W1"], layer["W3"], layer["W2"])
    x = layer["x"].clone()
    y = torch.empty_like(x)
    m.forward(x, *args, y=y)                 # outside capture: kernel attributes, device queries
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        m.forward(x, *args, y=y)
    for i in range(3):
        x.copy_(inputs.make_x(w, "cuda", seed=300 + i))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, m.forward(x, *args)), f"replay {i}"
    assert m.status() == 0


# ----------------------------------------------------------------------------- Mixtral shape
# d = 4096, d_ff = 14336, 8 experts, top-2 (xyznot "Method"; aiqianji 2.1.2), with
# the seeded weight and token distributions of the workloads.  The oracle's fp64
# routing covers every token; its expert outputs cover the tokens each case
# lists.  One oracle result serves every kernel configuration of a case.
@pytest.fixture(scope="module")
def mixtral_experts():
    w = inputs.workload("decode_t32")
    W1, W3, W2 = inputs.make_experts(w, "cuda")
    host = tuple(inputs.to_oracle(t) for t in (W1, W3, W2))
    return (W1, W3, W2), host


class MixtralCase:
    """One Mixtral-shape batch: the GPU's routing and dispatch checked against the
    oracle (indices bit-exact except near ties, dispatch bit-exact on the GPU's
    own indices), the tokens to check and the oracle's outputs for them."""

    def __init__(self, name, experts, T=None, seed=None, n_random=None, edges=EDGE_ROWS_FINE):
        w = inputs.workload(name) if T is None else inputs.workload(name, T=T)
        (self.W1, self.W3, self.W2), (h1, h3, h2) = experts
        self.w = w
        self.x = inputs.make_x(w, "cuda", seed=seed)
        self.Wg, self.b = inputs.make_router(w, "cuda")
        m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, bias=self.b)
        r = m.route(self.x, self.Wg)
        torch.cuda.synchronize()
        gidx, gw = r["topk_idx"].cpu().numpy(), r["topk_w"].cpu().numpy()
        counts, offsets, perm = (r[k].cpu().numpy() for k in ("counts", "offsets", "perm"))
        m.close()
        xo, Wgo, bo = inputs.to_oracle(self.x), inputs.to_oracle(self.Wg), inputs.to_oracle(self.b)
        logits = oracle.router_logits(xo, Wgo, bo)
        idx, gate = oracle.select_topk(logits, w.k)
        self.near = check_route(gidx, gw, logits, idx, gate, w.k)
        check_dispatch(gidx, counts, offsets, perm, w.n_experts)
        if n_random is None:
            self.toks, self.info = np.arange(w.T), dict(all_tokens=w.T)
        else:
            self.toks, self.info = dispatch_sample(counts, offsets, perm, w.k, w.T, n_random, edges=edges)
        self.counts = counts.tolist()
        idx_u, gate_u, _ = reference_selection(dict(logits=logits, idx=idx, gate=gate), gidx, w.k)
        self.y_ref = oracle.moe_tokens(xo, h1, h3, h2, idx_u, gate_u, self.toks)

    def check(self, path=0, pair=0, streamk=1):
        w = self.w
        layer = dict(x=self.x, Wg=self.Wg, bias=self.b, W1=self.W1, W3=self.W3, W2=self.W2)
        m, y, gidx, _ = run_layer(w, layer, path, pair, streamk)
        m.close()
        err, bound = assert_close(y_to_numpy(y)[self.toks], self.y_ref, "bf16")
        print(f"{w.name} T={w.T} path={path} pair={pair}: {len(self.toks)} tokens checked {self.info}, "
              f"loads {self.counts}, max err {err:.3e} (bound {bound:.3e}), near ties {self.near}")
        return err


@pytest.fixture(scope="module")
def prefill_case(mixtral_experts):
    # 512 seeded tokens + the smallest expert group + every tile edge and tail
    return MixtralCase("prefill_t4096", mixtral_experts, n_random=512)


@pytest.fixture(scope="module")
def skewed_case(mixtral_experts):
    return MixtralCase("skewed_t32768", mixtral_experts, n_random=512, edges=EDGE_ROWS)


@pytest.mark.parametrize("pair", [0, 1, 2], ids=["default", "single_cta", "cta_pairs"])
def test_mixtral_prefill_t4096(prefill_case, pair):
    prefill_case.check(pair=pair)


@pytest.mark.parametrize("pair", [0, 1, 2], ids=["default", "single_cta", "cta_pairs"])
def test_mixtral_skewed_t32768(skewed_case, pair):
    case = skewed_case
    assert max(case.counts) > 0.3 * sum(case.counts)   # the hot expert takes > 30% of the rows
    case.check(pair=pair)


_DECODE_CASES = {}


@pytest.fixture(scope="module")
def decode_cases(mixtral_experts):
    """Mixtral-shape decode batches, every token checked, built on first use."""
    def get(T):
        if T not in _DECODE_CASES:
            _DECODE_CASES[T] = MixtralCase("decode_t32", mixtral_experts, T=T, seed=None if T == 32 else 40 + T)
        return _DECODE_CASES[T]
    yield get
    _DECODE_CASES.clear()


# (T, forced path): 0 = the default for that T (weight streaming up to T = 128,
# grouped GEMMs above), 1 = grouped GEMMs, 2 = weight streaming
MIXTRAL_DECODE = [(1, 0), (32, 0), (32, 1), (128, 0), (128, 1), (256, 0), (256, 2)]


@pytest.mark.parametrize("T,path", MIXTRAL_DECODE, ids=[f"T{T}-path{p}" for T, p in MIXTRAL_DECODE])
def test_mixtral_decode_sweep(decode_cases, T, path):
    decode_cases(T).check(path=path)


@pytest.mark.parametrize("T", [8, 32, 128])
def test_mixtral_decode_uniform_k_split(decode_cases, T):
    # the weight-streaming kernels with the uniform K split at the Mixtral shape
    decode_cases(T).check(path=2, streamk=0)


# ----------------------------------------------------------------------------- decode (weight-streaming) path
DECODE_CASES = [
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
    (16, 256, 256, 8, 8),       # K = n on the weight-streaming path
]


@pytest.mark.parametrize("T,d,F,n,K", DECODE_CASES)
def test_decode_path_matches_oracle(T, d, F, n, K):
    w = inputs.Workload("dec", T=T, d=d, d_ff=F, n_experts=n, k=K, seed=100 + T + d)
    layer = inputs.make_layer(w, "cuda")
    m, y, gidx, gw = run_layer(w, layer, path=2)
    y_ref, ref, near = oracle_y(layer, w, np.arange(T), gidx)
    check_route(gidx, gw, ref["logits"], ref["idx"], ref["gate"], K)
    assert_close(y_to_numpy(y), y_ref, "bf16")


@pytest.mark.parametrize("T,d,F,n,K", DECODE_CASES)
def test_decode_uniform_k_split_matches_oracle(T, d, F, n, K):
    # the weight-streaming kernels with K split uniformly into items (the stream-K
    # split is the default, checked above): same layer, partial sums grouped otherwise
    w = inputs.Workload("dec", T=T, d=d, d_ff=F, n_experts=n, k=K, seed=100 + T + d)
    layer = inputs.make_layer(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, dtype=w.torch_dtype, bias=layer["bias"])
    m.set_option(_lib.MOE_OPT_FORCE_PATH, 2)
    ys = []
    for sk in (0, 1):
        m.set_option(_lib.MOE_OPT_DECODE_STREAMK, sk)
        ys.append(m.forward(layer["x"], layer["Wg"], layer["W1"], layer["W3"], layer["W2"]))
    torch.cuda.synchronize()
    assert m.status() == 0, _lib.moe_error_string(m.status())
    r = m.route(layer["x"], layer["Wg"])
    gidx = r["topk_idx"].cpu().numpy()
    y_ref, ref, near = oracle_y(layer, w, np.arange(T), gidx)
    assert_close(y_to_numpy(ys[0]), y_ref, "bf16")
    assert_close(y_to_numpy(ys[0]), y_to_numpy(ys[1]), "bf16")
    m.close()


def test_decode_all_tokens_to_one_expert_pair():
    # 200 tokens on experts (5, 2): N = 224 token columns per item, other experts skipped
    w = inputs.Workload("dec_skew", T=200, d=256, d_ff=384, bias=(0, 0, 50, 0, 0, 100, 0, 0), seed=4)
    layer = inputs.make_layer(w, "cuda")
    m, y, gidx, gw = run_layer(w, layer, path=2)
    assert np.all(gidx == [5, 2])
    y_ref, ref, near = oracle_y(layer, w, np.arange(w.T), gidx)
    assert_close(y_to_numpy(y), y_ref, "bf16")


def test_decode_and_grouped_paths_agree_and_are_deterministic():
    w = inputs.Workload("dec_vs_grp", T=48, d=512, d_ff=384, seed=9)
    layer = inputs.make_layer(w, "cuda")
    _, y_dec, _, _ = run_layer(w, layer, path=2)
    _, y_dec2, _, _ = run_layer(w, layer, path=2)
    _, y_grp, _, _ = run_layer(w, layer, path=1)
    assert torch.equal(y_dec, y_dec2)
    assert_close(y_to_numpy(y_dec), y_to_numpy(y_grp), "bf16")
