"""Pins for the fp64 oracle against what the pages and the mathematics fix.

Each test ties one part of the oracle to something other than itself: values
the pages print (slide router example, code blocks A/B/C of the aiqianji code
walkthrough), closed forms worked by hand, brute-force restatements written
independently here in numpy from the formulas, and invariants.  A dropped
term, a wrong sign, a transposed weight or a wrong index in the oracle fails
at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden


# ----------------------------------------------------------------------------- helpers
def f32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def np_widen(a):
    """Widen through torch's own dtype conversion (independent of the oracle's C code)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    return a.astype(np.float64)


def np_silu(z):
    return z / (1.0 + np.exp(-z))


def np_expert(x, W1, W3, W2, e):
    """SwiGLU expert with nn.Linear layouts: W2 (SiLU(W1 x) * (W3 x))."""
    return (np_silu(x @ W1[e].T) * (x @ W3[e].T)) @ W2[e].T


def rand_layer(rng, T, d, F, n, bf16=False):
    x = rng.standard_normal((T, d)).astype(np.float32)
    Wg = (rng.standard_normal((n, d)) * 0.5).astype(np.float32)
    W1 = (rng.standard_normal((n, F, d)) / math.sqrt(d)).astype(np.float32)
    W3 = (rng.standard_normal((n, F, d)) / math.sqrt(d)).astype(np.float32)
    W2 = (rng.standard_normal((n, d, F)) / math.sqrt(F)).astype(np.float32)
    if bf16:
        def tobf(a):
            return torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        x, W1, W3, W2 = (tobf(a) for a in (x, W1, W3, W2))
    return x, Wg, W1, W3, W2


# ----------------------------------------------------------------------------- widening
def test_bf16_widening_exact():
    bits = np.array([0x3F80, 0xC000, 0x3E80, 0x7F7F, 0x0001, 0x8000, 0x4049], dtype=np.uint16)
    got = oracle.widen(bits)
    want = np_widen(bits)
    assert np.array_equal(got, want)
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 0.25
    assert got[3] == 3.3895313892515355e38 and got[4] == 2.0 ** -133


# ----------------------------------------------------------------------------- gate (a2)
def test_slide_router_example_reading_a():
    keyed, _ = read_golden("slide_router_example.txt")
    logits = np.array([keyed["logits"]])
    idx, gate = oracle.select_topk(logits, 2)
    assert idx[0].tolist() == [int(v) for v in keyed["top2_experts"]]
    # closed form: Softmax over the two kept logits 1.4 and 0.6
    g1 = 1.0 / (1.0 + math.exp(-(1.4 - 0.6)))
    assert abs(gate[0, 0] - g1) < 1e-12 and abs(gate[0, 1] - (1.0 - g1)) < 1e-12
    assert abs(gate[0, 0] - 0.68997) < 1e-5 and abs(gate[0, 1] - 0.31003) < 1e-5
    tol = keyed["weight_tolerance_vs_slide"][0]
    assert np.all(np.abs(gate[0] - np.array(keyed["slide_weights"])) < tol)


def test_slide_router_example_reading_b():
    # Full-softmax probabilities 0.6 and 0.3 (the rest share 0.1): the gate over the
    # kept logits must equal those probabilities renormalised, 2/3 and 1/3.
    keyed, _ = read_golden("slide_router_example.txt")
    p_hi, p_lo = keyed["reading_b_probabilities"]
    p = np.full(8, (1.0 - p_hi - p_lo) / 6.0)
    p[2], p[5] = p_hi, p_lo
    idx, gate = oracle.select_topk(np.log(p)[None, :], 2)
    assert idx[0].tolist() == [2, 5]
    assert abs(gate[0, 0] - 2.0 / 3.0) < 1e-12 and abs(gate[0, 1] - 1.0 / 3.0) < 1e-12


def test_code_block_A_round_trip():
    _, rows = read_golden("routing_weights_code_block_A.txt")
    rows = np.array(rows)
    assert rows.shape == (16, 2)
    # properties of the printed rows themselves
    assert np.all(np.abs(rows.sum(1) - 1.0) <= 1e-4)
    assert np.all(rows[:, 0] >= rows[:, 1]) and np.all(rows[:, 1] > 0)
    assert np.array_equal(rows[0], rows[8]) and np.array_equal(rows[3], rows[12])
    # round trip: the logit gap ln(w1/w2) fed back through the oracle gives the row back
    rng = np.random.default_rng(0)
    for w1, w2 in rows:
        a, b = rng.choice(8, size=2, replace=False)
        base = rng.uniform(-2, 2)
        l = np.full(8, base - 10.0) + rng.uniform(0, 1, 8)
        l[a] = base + math.log(w1 / w2)
        l[b] = base
        idx, gate = oracle.select_topk(l[None, :], 2)
        assert idx[0].tolist() == [a, b]
        assert abs(gate[0, 0] - w1) <= 5e-5 and abs(gate[0, 1] - w2) <= 5e-5


@pytest.mark.parametrize("K", [1, 2, 3, 8])
def test_gate_identity_paper_vs_code_walkthrough(K):
    # Paper form: softmax over the top-K logits.  Code walkthrough form (aiqianji 3.1.1
    # steps 4-6): softmax over all n, take the top K, divide by their sum.
    rng = np.random.default_rng(K)
    l = rng.standard_normal((2000, 8)) * 3
    idx, gate = oracle.select_topk(l, K)
    p = np.exp(l - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :K]
    w = np.take_along_axis(p, order, 1)
    w /= w.sum(1, keepdims=True)
    assert np.array_equal(order, idx)
    assert np.max(np.abs(w - gate)) < 1e-14
    assert np.max(np.abs(gate.sum(1) - 1.0)) < 1e-14
    assert np.all(np.diff(gate, axis=1) <= 0)


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(1)
    l = np.round(rng.standard_normal((3000, 8)), 1)   # coarse values: many exact ties
    l[0] = 1.0                                         # all equal
    l[1] = [0, 2, 2, 1, 2, 0, 0, 0]
    for K in (1, 2, 4):
        idx, _ = oracle.select_topk(l, K)
        for t in range(l.shape[0]):
            brute = sorted(range(8), key=lambda e: (-l[t, e], e))[:K]
            assert idx[t].tolist() == brute
    idx, gate = oracle.select_topk(l[:2], 2)
    assert idx[0].tolist() == [0, 1] and np.allclose(gate[0], [0.5, 0.5], atol=0)
    assert idx[1].tolist() == [1, 2]


# ----------------------------------------------------------------------------- dispatch (a3)
def test_dispatch_code_blocks_B_C():
    keyed, _ = read_golden("dispatch_code_blocks_BC.txt")
    T = int(keyed["T"][0])
    mask = np.array([keyed["mask_rank0"], keyed["mask_rank1"]], dtype=int)
    E = 3
    # Build selections consistent with the printed mask for expert E; other tokens use
    # experts != E.
    idx = np.zeros((T, 2), dtype=np.int32)
    rng = np.random.default_rng(2)
    for t in range(T):
        others = [e for e in range(8) if e != E]
        a, b = rng.choice(others, size=2, replace=False)
        idx[t] = [a, b]
        for r in range(2):
            if mask[r, t]:
                idx[t, r] = E
                if idx[t, 1 - r] == E:
                    idx[t, 1 - r] = others[0]
    # the page's expert_mask = one_hot(selected).permute(2,1,0) slice for E, restated
    one_hot = (idx[:, :, None] == np.arange(8)[None, None, :]).astype(int)
    assert np.array_equal(one_hot.transpose(2, 1, 0)[E], mask)
    counts, offsets, perm = oracle.dispatch(idx, 8)
    seg = perm[offsets[E]:offsets[E + 1]]
    assert (seg // 2).tolist() == [int(v) for v in keyed["top_x"]]
    assert (seg % 2).tolist() == [int(v) for v in keyed["idx"]]


@pytest.mark.parametrize("T,n,K", [(1, 8, 2), (37, 8, 2), (500, 8, 2), (64, 4, 4), (100, 16, 1)])
def test_dispatch_invariants_and_where_listing(T, n, K):
    rng = np.random.default_rng(T + n + K)
    l = rng.standard_normal((T, n))
    idx, _ = oracle.select_topk(l, K)
    counts, offsets, perm = oracle.dispatch(idx, n)
    assert counts.sum() == K * T
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(np.sort(perm), np.arange(K * T))
    flat = idx.reshape(-1)
    for e in range(n):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)       # stable: ascending flat order t*K+k
        # torch.where over the (K, T) mask slice lists the same (rank, token) pairs
        mask = (idx == e).T
        r, tok = np.nonzero(mask)
        assert sorted(zip(tok.tolist(), r.tolist())) == sorted(zip((seg // K).tolist(), (seg % K).tolist()))


# ----------------------------------------------------------------------------- experts + combine (a4-a6)
@pytest.mark.parametrize("bf16", [False, True])
def test_dense_masked_brute_force(bf16):
    # y = sum_{i=0}^{n-1} G(x)_i E_i(x) with G = Softmax(TopK(l)), TopK setting the rest
    # to -inf: every expert is evaluated for every token, the masked ones weigh exactly 0.
    rng = np.random.default_rng(3 + bf16)
    T, d, F, n, K = 7, 6, 10, 8, 2
    x, Wg, W1, W3, W2 = rand_layer(rng, T, d, F, n, bf16)
    xd, W1d, W3d, W2d = (np_widen(a) for a in (x, W1, W3, W2))
    l = xd @ Wg.astype(np.float64).T
    kth = np.sort(l, axis=1)[:, -K][:, None]
    masked = np.where(l >= kth, l, -np.inf)
    G = np.exp(masked - masked.max(1, keepdims=True))
    G /= G.sum(1, keepdims=True)
    y_dense = sum(G[:, [e]] * np_expert(xd, W1d, W3d, W2d, e) for e in range(n))
    ref = oracle.moe_forward(x, Wg, W1, W3, W2, K)
    assert np.allclose(ref["logits"], l, rtol=0, atol=1e-12)
    scale = np.abs(y_dense).max()
    assert np.max(np.abs(ref["y"] - y_dense)) <= 1e-12 * scale


def test_identical_experts_with_K_equal_n_is_one_ffn():
    rng = np.random.default_rng(4)
    T, d, F, n = 9, 5, 12, 4
    x, Wg, W1, W3, W2 = rand_layer(rng, T, d, F, n)
    W1[:] = W1[0]
    W3[:] = W3[0]
    W2[:] = W2[0]
    ref = oracle.moe_forward(x, Wg, W1, W3, W2, K=n)
    xd = x.astype(np.float64)
    ffn = (np_silu(xd @ W1[0].T.astype(np.float64)) * (xd @ W3[0].T.astype(np.float64))) @ W2[0].T.astype(np.float64)
    assert np.max(np.abs(ref["y"] - ffn)) <= 1e-12 * np.abs(ffn).max()


def test_K1_routes_to_argmax_expert_with_gate_one():
    rng = np.random.default_rng(5)
    T, d, F, n = 11, 6, 9, 8
    x, Wg, W1, W3, W2 = rand_layer(rng, T, d, F, n)
    ref = oracle.moe_forward(x, Wg, W1, W3, W2, K=1)
    xd = x.astype(np.float64)
    am = np.argmax(xd @ Wg.astype(np.float64).T, axis=1)
    assert np.array_equal(ref["idx"][:, 0], am)
    assert np.all(ref["gate"] == 1.0)
    W1d, W3d, W2d = (w.astype(np.float64) for w in (W1, W3, W2))
    want = np.stack([np_expert(xd[t:t + 1], W1d, W3d, W2d, am[t])[0] for t in range(T)])
    assert np.max(np.abs(ref["y"] - want)) <= 1e-12 * np.abs(want).max()


def test_linear_in_W2():
    rng = np.random.default_rng(6)
    x, Wg, W1, W3, W2 = rand_layer(rng, 6, 8, 16, 8)
    a = oracle.moe_forward(x, Wg, W1, W3, W2, 2)["y"]
    b = oracle.moe_forward(x, Wg, W1, W3, (W2 * 2).astype(np.float32), 2)["y"]
    assert np.array_equal(b, 2 * a)


def test_hand_worked_single_expert():
    # n=1, K=1, d=2, F=1:  a = 0.5*1 + 0.25*2 = 1,  b = 1*1 - 1*2 = -1,
    # h = SiLU(1) * (-1) = -1/(1+e^-1),  y = [2h, 3h].
    x = f32([[1.0, 2.0]])
    Wg = f32([[1.0, 1.0]])
    W1 = f32([[[0.5, 0.25]]])
    W3 = f32([[[1.0, -1.0]]])
    W2 = f32([[[2.0], [3.0]]])
    ref = oracle.moe_forward(x, Wg, W1, W3, W2, K=1)
    h = -0.7310585786300049
    assert np.allclose(ref["y"][0], [2 * h, 3 * h], rtol=0, atol=1e-15)


def test_hand_worked_two_experts_two_slots():
    # n=2, K=2, d=2, F=2.  Router logits l = [0, ln 3] -> expert 1 first, gates 3/4, 1/4.
    # Expert e: W1 = I, W3 = 2I (e=0) or -I (e=1), W2 = [[1,0],[0,1]] (e=0), [[0,1],[1,0]] (e=1).
    x = f32([[1.0, -2.0]])
    Wg = f32([[0.0, 0.0], [-math.log(3.0), 0.0]])
    Wg[1, 0] = f32([math.log(3.0)])[0]  # logit_1 = x0 * ln3 = ln3
    W1 = f32([[[1, 0], [0, 1]], [[1, 0], [0, 1]]])
    W3 = f32([[[2, 0], [0, 2]], [[-1, 0], [0, -1]]])
    W2 = f32([[[1, 0], [0, 1]], [[0, 1], [1, 0]]])
    ref = oracle.moe_forward(x, Wg, W1, W3, W2, K=2)
    assert ref["idx"][0].tolist() == [1, 0]
    l1 = float(np.float32(math.log(3.0)))
    g1 = 1.0 / (1.0 + math.exp(-l1))
    assert abs(ref["gate"][0, 0] - g1) < 1e-15 and abs(g1 - 0.75) < 1e-7
    s1, sm2 = 1.0 / (1.0 + math.exp(-1.0)), -2.0 / (1.0 + math.exp(2.0))
    e0 = np.array([s1 * 2.0, sm2 * -4.0])          # SiLU(x) * 2x
    e1 = np.array([sm2 * 2.0, s1 * -1.0])          # swap(SiLU(x) * -x)
    want = g1 * e1 + (1.0 - g1) * e0
    assert np.allclose(ref["y"][0], want, rtol=0, atol=1e-14)


def test_silu_limits_through_one_expert():
    # d=1, F=1, W1 = z, W3 = 1, W2 = 1, x = 1: y = SiLU(z).
    for z, want in [(0.0, 0.0), (30.0, 30.0), (-30.0, 0.0)]:
        ref = oracle.moe_forward(f32([[1.0]]), f32([[1.0]]), f32([[[z]]]), f32([[[1.0]]]), f32([[[1.0]]]), 1)
        assert abs(ref["y"][0, 0] - want) < 1e-10
    zs = [0.3, 1.7, 4.0]
    pos = [oracle.moe_forward(f32([[1.0]]), f32([[1.0]]), f32([[[z]]]), f32([[[1.0]]]), f32([[[1.0]]]), 1)["y"][0, 0] for z in zs]
    neg = [oracle.moe_forward(f32([[1.0]]), f32([[1.0]]), f32([[[-z]]]), f32([[[1.0]]]), f32([[[1.0]]]), 1)["y"][0, 0] for z in zs]
    for z, p, m in zip(zs, pos, neg):
        assert abs((p - m) - float(np.float32(z))) < 1e-12     # SiLU(z) - SiLU(-z) = z
        assert 0 < p < float(np.float32(z))


def test_router_bias_shifts_logits():
    rng = np.random.default_rng(7)
    x, Wg, W1, W3, W2 = rand_layer(rng, 20, 8, 8, 8)
    b = f32([1.5, 0.5, 0, 0, 0, 0, -0.5, -1])
    l0 = oracle.router_logits(x, Wg)
    l1 = oracle.router_logits(x, Wg, b)
    assert np.allclose(l1 - l0, b.astype(np.float64)[None, :], atol=1e-12)
    xd = x.astype(np.float64)
    assert np.allclose(l0, xd @ Wg.astype(np.float64).T, rtol=0, atol=1e-12)


def test_expert_rows_match_tokens_with_unit_gate():
    rng = np.random.default_rng(8)
    x, Wg, W1, W3, W2 = rand_layer(rng, 10, 8, 12, 4, bf16=True)
    toks = np.array([0, 3, 9])
    out = oracle.expert_rows(x, W1, W3, W2, 2, toks)
    want = np_expert(np_widen(x)[toks], np_widen(W1), np_widen(W3), np_widen(W2), 2)
    assert np.max(np.abs(out - want)) <= 1e-12 * np.abs(want).max()


def test_threads_do_not_change_results():
    rng = np.random.default_rng(9)
    x, Wg, W1, W3, W2 = rand_layer(rng, 33, 16, 24, 8, bf16=True)
    a = oracle.moe_forward(x, Wg, W1, W3, W2, 2, nthreads=1)["y"]
    b = oracle.moe_forward(x, Wg, W1, W3, W2, 2, nthreads=4)["y"]
    assert np.array_equal(a, b)


# ----------------------------------------------------------------------------- residual stack
def tobf_bits(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_round_bf16_matches_torch_on_fp32_values():
    # For values that are exact in fp32, rounding straight to bf16 is what torch's
    # fp32 -> bf16 conversion does (round to nearest, ties to even).
    rng = np.random.default_rng(11)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 1.0, 37.0)]).astype(np.float32)
    assert np.array_equal(oracle.round_bf16(v.astype(np.float64)), tobf_bits(v))


def test_round_bf16_closed_forms():
    # bf16 keeps 8 significant bits: between 1 and 2 the spacing is 2^-7.
    cases = {
        1.0: 0x3F80,
        1.0 + 2.0 ** -8: 0x3F80,                 # exact tie -> even (1.0)
        1.0 + 3 * 2.0 ** -8: 0x3F82,             # exact tie -> even (1 + 2^-6)
        1.0 + 2.0 ** -8 + 2.0 ** -30: 0x3F81,    # just above the tie -> up; an fp32 detour would give 1.0
        -2.5: 0xC020,
        0.0: 0x0000,
    }
    got = oracle.round_bf16(np.array(list(cases.keys())))
    assert [int(g) for g in got] == list(cases.values())


def test_rms_norm_hand_worked():
    # rows [3, 4]: mean square 12.5 -> [3, 4] / sqrt(12.5 + eps); a constant row c -> 1/sqrt(1 + eps/c^2)
    eps = 1e-5
    h = f32([[3.0, 4.0], [2.0, 2.0]])
    u = oracle.rms_norm(h, eps)
    assert np.allclose(u[0], np.array([3.0, 4.0]) / math.sqrt(12.5 + eps), rtol=0, atol=1e-15)
    assert np.allclose(u[1], 1.0 / math.sqrt(1.0 + eps / 4.0), rtol=0, atol=1e-15)
    # scale invariance (up to eps): RMSNorm(5h) == RMSNorm(h) when eps = 0
    assert np.allclose(oracle.rms_norm(f32([[3.0, 4.0]]) * 5, 0.0), oracle.rms_norm(f32([[3.0, 4.0]]), 0.0),
                       rtol=0, atol=1e-15)


def test_block_is_residual_plus_dense_masked_moe_of_rounded_norm():
    # h_new = h + sum_i G(u)_i E_i(u), u = bf16(h / rms(h)): brute force over all experts in numpy.
    rng = np.random.default_rng(12)
    T, d, F, n, K, eps = 9, 8, 12, 8, 2, 1e-5
    _, Wg, W1, W3, W2 = rand_layer(rng, T, d, F, n, bf16=True)
    h = tobf_bits(rng.standard_normal((T, d)) * 3.0)
    hd = np_widen(h)
    u = tobf_bits(hd / np.sqrt(np.mean(hd * hd, axis=1, keepdims=True) + eps))
    ud, W1d, W3d, W2d = (np_widen(a) for a in (u, W1, W3, W2))
    l = ud @ Wg.astype(np.float64).T
    kth = np.sort(l, axis=1)[:, -K][:, None]
    masked = np.where(l >= kth, l, -np.inf)
    G = np.exp(masked - masked.max(1, keepdims=True))
    G /= G.sum(1, keepdims=True)
    y = sum(G[:, [e]] * np_expert(ud, W1d, W3d, W2d, e) for e in range(n))
    ref = oracle.block_forward(h, Wg, W1, W3, W2, K, eps)
    assert np.array_equal(ref["u"], u)
    assert np.max(np.abs(ref["h_new"] - (hd + y))) <= 1e-12 * np.abs(hd + y).max()
    assert np.array_equal(ref["h_bits"], oracle.round_bf16(hd + y))


def test_block_with_zero_W2_is_identity():
    rng = np.random.default_rng(13)
    _, Wg, W1, W3, W2 = rand_layer(rng, 5, 8, 12, 8, bf16=True)
    h = tobf_bits(rng.standard_normal((5, 8)))
    ref = oracle.block_forward(h, Wg, W1, W3, np.zeros_like(W2), 2, 1e-5)
    assert np.array_equal(ref["h_bits"], h)
    assert np.all(ref["y"] == 0.0)
