"""fp64 CPU oracle for the Mixtral sparse MoE feed-forward layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
library under ``sparse_mixture_experts_54_b300`` never imports it, and this
package imports nothing from the library: the two share no code.

The arithmetic lives in ``moe_oracle.c`` (plain C loops in double precision,
one token per thread, OpenMP across tokens).  This module only marshals numpy
arrays to it.  Stored element types are passed through unchanged: bf16 tensors
travel as ``numpy.uint16`` bit patterns, fp32 as ``numpy.float32``; the C code
widens them exactly to double.

Every function here is pinned by ``tests/test_oracle_pins.py`` against what the
pages fix (the slide router example, the printed routing weights and dispatch
lists of the code walkthrough, closed forms and brute-force restatements).
The printed final hidden states of code block E (aiqianji, section 3.2.5)
need trained weights: that value is *parity unpinned*.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lib = None

BF16 = 0
F32 = 1


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/libmoe_oracle.so with gcc (no GPU needed)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared",
               "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        lib.oracle_router_logits.argtypes = [P, I, P, P, I64, I, I, P]
        lib.oracle_select_topk.argtypes = [P, I64, I, I, P, P]
        lib.oracle_dispatch.argtypes = [P, I64, I, I, P, P, P]
        lib.oracle_expert_rows.argtypes = [P, I, P, P, P, I, I, I, I, P, I64, P, P]
        lib.oracle_moe_tokens.argtypes = [P, I, P, P, P, I, I, I, I, I, P, P, P, I64, P, I, P]
        lib.oracle_widen.argtypes = [P, I, I64, I64, P]
        lib.oracle_max_threads.argtypes = []
        for f in ("oracle_router_logits", "oracle_select_topk", "oracle_dispatch",
                  "oracle_expert_rows", "oracle_moe_tokens", "oracle_max_threads"):
            getattr(lib, f).restype = I
        lib.oracle_widen.restype = None
        _lib = lib
    return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"oracle takes bf16 bit patterns (uint16) or float32, got {a.dtype}")


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def widen(a: np.ndarray) -> np.ndarray:
    """Exact fp64 value of stored bf16 (uint16 bits) or fp32 elements."""
    a = np.ascontiguousarray(a)
    out = np.empty(a.shape, dtype=np.float64)
    _load().oracle_widen(_ptr(a), _dtype_code(a), 0, a.size, _ptr(out))
    return out


def router_logits(x: np.ndarray, Wg: np.ndarray, bias: Optional[np.ndarray] = None) -> np.ndarray:
    """l[t][e] = x[t] . W_g[e] (+ bias[e]) in fp64; W_g is [n][d] fp32."""
    x = np.ascontiguousarray(x)
    Wg = np.ascontiguousarray(Wg, dtype=np.float32)
    T, d = x.shape
    n = Wg.shape[0]
    assert Wg.shape == (n, d)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty((T, n), dtype=np.float64)
    rc = _load().oracle_router_logits(_ptr(x), _dtype_code(x), _ptr(Wg), None if b is None else _ptr(b),
                                      T, d, n, _ptr(out))
    assert rc == 0, rc
    return out


def select_topk(logits: np.ndarray, K: int):
    """Top-K experts per token (descending, ties -> lower index) and their softmax gates."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    T, n = logits.shape
    idx = np.empty((T, K), dtype=np.int32)
    gate = np.empty((T, K), dtype=np.float64)
    rc = _load().oracle_select_topk(_ptr(logits), T, n, K, _ptr(idx), _ptr(gate))
    assert rc == 0, rc
    return idx, gate


def dispatch(idx: np.ndarray, n: int):
    """counts[n], offsets[n+1] (exclusive scan) and perm[K*T] (flat t*K+k, by expert, stable)."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, K = idx.shape
    counts = np.empty(n, dtype=np.int64)
    offsets = np.empty(n + 1, dtype=np.int64)
    perm = np.empty(T * K, dtype=np.int64)
    rc = _load().oracle_dispatch(_ptr(idx), T, K, n, _ptr(counts), _ptr(offsets), _ptr(perm))
    assert rc == 0, rc
    return counts, offsets, perm


def expert_rows(x, W1, W3, W2, e: int, toks) -> np.ndarray:
    """E_e(x[t]) for each t in toks, no gate: fp64 [len(toks)][d]."""
    x = np.ascontiguousarray(x)
    W1, W3, W2 = (np.ascontiguousarray(w) for w in (W1, W3, W2))
    n, F, d = W1.shape
    toks = np.ascontiguousarray(toks, dtype=np.int64)
    out = np.empty((toks.size, d), dtype=np.float64)
    scratch = np.empty(d + F, dtype=np.float64)
    rc = _load().oracle_expert_rows(_ptr(x), _dtype_code(x), _ptr(W1), _ptr(W3), _ptr(W2),
                                    _dtype_code(W1), d, F, e, _ptr(toks), toks.size, _ptr(out),
                                    _ptr(scratch))
    assert rc == 0, rc
    return out


def moe_tokens(x, W1, W3, W2, idx, gate, toks, nthreads: Optional[int] = None) -> np.ndarray:
    """y[s] = sum_k gate[t][k] * E_{idx[t][k]}(x[t]) for t = toks[s]; fp64 [len(toks)][d]."""
    x = np.ascontiguousarray(x)
    W1, W3, W2 = (np.ascontiguousarray(w) for w in (W1, W3, W2))
    assert W1.dtype == W3.dtype == W2.dtype
    n, F, d = W1.shape
    assert W3.shape == (n, F, d) and W2.shape == (n, d, F) and x.shape[1] == d
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float64)
    K = idx.shape[1]
    toks = np.ascontiguousarray(toks, dtype=np.int64)
    nthreads = max_threads() if nthreads is None else int(nthreads)
    y = np.empty((toks.size, d), dtype=np.float64)
    scratch = np.empty(max(nthreads, 1) * (2 * d + F), dtype=np.float64)
    rc = _load().oracle_moe_tokens(_ptr(x), _dtype_code(x), _ptr(W1), _ptr(W3), _ptr(W2),
                                   _dtype_code(W1), d, F, n, K, _ptr(idx), _ptr(gate), _ptr(toks),
                                   toks.size, _ptr(y), nthreads, _ptr(scratch))
    assert rc == 0, rc
    return y


def moe_forward(x, Wg, W1, W3, W2, K: int, bias=None, toks=None, nthreads: Optional[int] = None):
    """Whole layer in fp64: router, top-K gate, dispatch and y for ``toks`` (all tokens if None).

    Returns a dict with logits [T][n], idx [T][K], gate [T][K], counts, offsets,
    perm and y [len(toks)][d].
    """
    logits = router_logits(x, Wg, bias)
    idx, gate = select_topk(logits, K)
    counts, offsets, perm = dispatch(idx, Wg.shape[0])
    if toks is None:
        toks = np.arange(x.shape[0], dtype=np.int64)
    y = moe_tokens(x, W1, W3, W2, idx, gate, toks, nthreads)
    return dict(logits=logits, idx=idx, gate=gate, counts=counts, offsets=offsets, perm=perm,
                y=y, toks=np.asarray(toks, dtype=np.int64))


# ----------------------------------------------------------------------------- the residual stack
# The pages' block diagram (DL reading-group slides, "Architecture - 全体") repeats,
# 32 times (xyznot "Method"), RMSNorm -> attention -> RMSNorm -> MoE, each with a
# residual connection.  The MoE half of a block, as built here:
#     u = RMSNorm(h) = h / sqrt(mean_j h_j^2 + eps)      (unit gain; the pages only name it)
#     h <- h + MoE(u)
# with the hidden state h and the MoE input u stored in bf16, as the model's
# activations are.  The oracle follows its own trajectory in fp64, rounding
# to bf16 exactly where the definition stores a value.

def round_bf16(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 (ties to even), directly -- no detour
    through fp32, whose own rounding could move a value onto a bf16 tie.  Returns
    the bit patterns (uint16).  Normal-range values only (|v| in [2^-126, 2^127))
    or zero; that covers every activation here."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                      # v = m * 2^e, 0.5 <= |m| < 1
    q = np.rint(m * 256.0)                  # 8 significant bits, ties to even
    r = np.ldexp(q / 256.0, e)              # exact: q has at most 9 bits
    bits = np.ascontiguousarray(r.astype(np.float32)).view(np.uint32)
    return (bits >> 16).astype(np.uint16)


def rms_norm(h: np.ndarray, eps: float) -> np.ndarray:
    """fp64 RMSNorm with unit gain of stored rows h [S][d] (bf16 bits or fp32)."""
    h64 = widen(h)
    ms = np.mean(h64 * h64, axis=1, keepdims=True)
    return h64 / np.sqrt(ms + eps)


def _store_like(v: np.ndarray, h: np.ndarray) -> np.ndarray:
    """fp64 values stored in h's element type: bf16 bits (rounded to nearest even)
    or fp32 (numpy's conversion, also to nearest even)."""
    if h.dtype == np.uint16:
        return round_bf16(v)
    return v.astype(np.float32)


def block_forward(h: np.ndarray, Wg, W1, W3, W2, K: int, eps: float, bias=None, nthreads: Optional[int] = None):
    """One residual block on the given rows h [S][d] (bf16 bits or fp32): the MoE
    of RMSNorm(h) stored in h's element type, added to h in fp64.

    Returns dict(u=the stored MoE input, logits, idx, gate, y=MoE(u) fp64,
    h_new=h + y in fp64 (before the storage rounding), h_bits=h_new stored)."""
    u = _store_like(rms_norm(h, eps), h)
    logits = router_logits(u, Wg, bias)
    idx, gate = select_topk(logits, K)
    y = moe_tokens(u, W1, W3, W2, idx, gate, np.arange(u.shape[0]), nthreads)
    h_new = widen(h) + y
    return dict(u=u, logits=logits, idx=idx, gate=gate, y=y, h_new=h_new, h_bits=_store_like(h_new, h))


# --------------------------------------------------------------------------- fp8 expert weights
# Not part of the method on the pages: an input format of the library's
# fp8-weight entry point.  A weight is scale[row] * q, q an OCP e4m3 byte.

def decode_e4m3(q: np.ndarray) -> np.ndarray:
    """Exact fp64 value of OCP FP8 E4M3 bytes (uint8): sign bit, 4 exponent bits
    with bias 7, 3 mantissa bits; exponent field 0 is subnormal (M/8 * 2^-6);
    the all-ones pattern S.1111.111 is NaN (the format has no infinities)."""
    q = np.asarray(q, dtype=np.uint8)
    sign = np.where(q & 0x80, -1.0, 1.0)
    E = ((q >> 3) & 0xF).astype(np.int64)
    M = (q & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + M / 8.0, E - 7)
    sub = np.ldexp(M / 8.0, -6)
    v = sign * np.where(E == 0, sub, normal)
    return np.where((E == 15) & (M == 7), np.nan, v)


def dequantize_e4m3_rows(q: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """W[..., r, j] = scale[..., r] * e4m3(q[..., r, j]) in fp64."""
    return np.asarray(scale, dtype=np.float64)[..., None] * decode_e4m3(q)
