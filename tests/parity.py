"""Comparison helpers shared by the GPU parity tests (test-side logic only).

Tolerances, derived from the layer's arithmetic: fp32 accumulation over K = d
or d_ff products of bf16 operands, with the SwiGLU product H rounded once to
bf16 before the W2 GEMM, so the expected relative error of y is a few bf16 ulps
(2^-8) spread over d_ff terms, well inside 1e-2 of the output's RMS:
  * routing indices and dispatch order: bit-exact, except near-tie tokens whose
    fp64 oracle logits have two neighbours among the top K+1 closer than 1e-6
    (fp32 on the GPU may order them either way); those are counted;
  * bf16: max|y - y_ref| <= 1e-2 * rms(y_ref), on top of the rounding of the
    stored bf16 result itself (at most half an ulp, <= 2^-8 |y_ref|, elementwise);
  * fp32: max|y - y_ref| <= 1e-5 * max|y_ref|.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_mixture_experts_54_b300 import inputs

TIE_EPS = 1e-6
BF16_TOL = 1e-2
F32_TOL = 1e-5


def near_tie_mask(logits: np.ndarray, K: int, eps: float = TIE_EPS) -> np.ndarray:
    """True for tokens whose sorted fp64 logits have a gap < eps among ranks 1..K+1."""
    s = -np.sort(-logits, axis=1)
    m = min(K + 1, logits.shape[1])
    gaps = s[:, : m - 1] - s[:, 1:m]
    return np.any(gaps < eps, axis=1)


def check_route(gpu_idx: np.ndarray, gpu_w: np.ndarray, ref_logits: np.ndarray, ref_idx: np.ndarray,
                ref_gate: np.ndarray, K: int, w_tol: float = 2e-6):
    """Bit-exact indices except near ties; gates within w_tol.  Returns the near-tie count."""
    near = near_tie_mask(ref_logits, K)
    far = ~near
    bad = np.nonzero(np.any(gpu_idx[far] != ref_idx[far], axis=1))[0]
    assert bad.size == 0, f"{bad.size} non-tie tokens routed differently, first {np.nonzero(far)[0][bad[:5]]}"
    err = np.max(np.abs(gpu_w[far] - ref_gate[far])) if far.any() else 0.0
    assert err <= w_tol, f"gate error {err}"
    # near-tie tokens must still pick valid, distinct experts with gates summing to 1
    if near.any():
        gi = gpu_idx[near]
        assert np.all((gi >= 0) & (gi < ref_logits.shape[1]))
        assert all(len(set(r.tolist())) == K for r in gi)
        assert np.max(np.abs(gpu_w[near].sum(1) - 1.0)) < 1e-5
    return int(near.sum())


def check_dispatch(gpu_idx, counts, offsets, perm, n):
    """Dispatch is a pure function of the indices: compare with the oracle's on the GPU's own indices."""
    c, o, p = oracle.dispatch(gpu_idx.astype(np.int32), n)
    assert np.array_equal(counts.astype(np.int64), c)
    assert np.array_equal(offsets.astype(np.int64), o)
    assert np.array_equal(perm.astype(np.int64), p)


def reference_selection(ref: dict, gpu_idx: np.ndarray, K: int):
    """Oracle selection, with near-tie tokens switched to the GPU's experts (gates recomputed in fp64)."""
    idx = ref["idx"].copy()
    gate = ref["gate"].copy()
    near = near_tie_mask(ref["logits"], K)
    for t in np.nonzero(near)[0]:
        idx[t] = gpu_idx[t]
        l = ref["logits"][t, gpu_idx[t]]
        w = np.exp(l - l.max())
        gate[t] = w / w.sum()
    return idx, gate, int(near.sum())


BF16_STORE = 2.0 ** -8   # half an ulp of bf16, relative


def assert_close(y_gpu: np.ndarray, y_ref: np.ndarray, dtype: str):
    """Returns (max error beyond the output's own storage rounding, bound)."""
    y_gpu = y_gpu.astype(np.float64)
    assert np.all(np.isfinite(y_gpu)), "non-finite output"
    diff = np.abs(y_gpu - y_ref)
    if dtype == "f32":
        bound = F32_TOL * np.max(np.abs(y_ref))
        err = np.max(diff)
    else:
        bound = BF16_TOL * np.sqrt(np.mean(y_ref ** 2))
        err = np.max(diff - BF16_STORE * np.abs(y_ref))
    assert err <= bound, f"max abs err {err:.3e} > bound {bound:.3e} (raw max {np.max(diff):.3e})"
    return err, bound


def y_to_numpy(y: torch.Tensor) -> np.ndarray:
    return y.detach().float().cpu().numpy().astype(np.float64)


def oracle_args(layer: dict):
    return tuple(inputs.to_oracle(layer[k]) for k in ("x", "Wg", "W1", "W3", "W2")) + (inputs.to_oracle(layer["bias"]),)


# Row boundaries inside a 256-row block of one expert's rows that the tiled
# kernels treat differently: 32-row epilogue quadrants, the 64-row halves of a
# CTA pair's 128-row tail tile, 128-row single-CTA tiles and the two CTAs of a
# 256-row pair tile.
EDGE_ROWS_FINE = (0, 31, 32, 63, 64, 95, 96, 127, 128, 255)
EDGE_ROWS = (0, 127, 128, 255)


def dispatch_sample(counts, offsets, perm, K: int, T: int, n_random: int, seed: int = 0,
                    edges=EDGE_ROWS_FINE):
    """Tokens for a sampled check at full size, picked from the GPU's own
    expert-contiguous order (which check_dispatch has already compared with the
    oracle's), so that every tiling boundary of every expert is covered:

    * n_random seeded tokens;
    * every token of the smallest non-empty expert group;
    * the tokens at the ``edges`` rows of every 256-row block of every expert;
    * every row of each expert's last 128-row tile (its ragged tail, including
      the most loaded expert's).

    Returns (sorted token numbers, dict of how many rows each rule picked)."""
    counts = np.asarray(counts, dtype=np.int64)
    offsets = np.asarray(offsets, dtype=np.int64)
    perm = np.asarray(perm, dtype=np.int64)
    rows_edge, rows_tail, rows_small = [], [], []
    for e in range(counts.size):
        c, o = int(counts[e]), int(offsets[e])
        if c == 0:
            continue
        for b in range(0, c, 256):
            rows_edge += [o + b + r for r in edges if b + r < c]
        last = (c - 1) // 128 * 128
        rows_tail += list(range(o + last, o + c))
    nz = np.nonzero(counts)[0]
    small = int(nz[np.argmin(counts[nz])])
    rows_small = list(range(int(offsets[small]), int(offsets[small] + counts[small])))
    rows = np.asarray(sorted(set(rows_edge) | set(rows_tail) | set(rows_small)), dtype=np.int64)
    toks = set((perm[rows] // K).tolist()) | set(inputs.sample_tokens(T, n_random, seed).tolist())
    info = dict(random=min(n_random, T), edge_rows=len(set(rows_edge)), tail_rows=len(set(rows_tail)),
                smallest_expert=small, smallest_rows=len(rows_small))
    return np.asarray(sorted(toks), dtype=np.int64), info
