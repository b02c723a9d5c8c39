"""The fp8 (OCP E4M3) weight format of moe_forward_fp8, on the CPU: the
oracle's decoder against the format's definition and against torch's own
float8_e4m3fn, and the properties of the seeded row quantiser."""
import math

import numpy as np
import torch

import oracle
from sparse_mixture_experts_54_b300 import inputs

# byte -> value fixed by the format: bias 7, 3 mantissa bits, E = 0 subnormal
CLOSED_FORMS = {
    0x00: 0.0,
    0x38: 1.0,                 # E = 7, M = 0
    0x3C: 1.5,                 # M = 4: 1 + 4/8
    0x40: 2.0,
    0x7E: 448.0,               # E = 15, M = 6: the largest finite value
    0x08: 2.0 ** -6,           # smallest normal
    0x01: 2.0 ** -9,           # smallest subnormal: 1/8 * 2^-6
    0x07: 7 * 2.0 ** -9,       # largest subnormal
    0xB8: -1.0,
    0xFE: -448.0,
}


def test_decode_closed_forms():
    v = oracle.decode_e4m3(np.array(list(CLOSED_FORMS), dtype=np.uint8))
    assert np.array_equal(v, np.array(list(CLOSED_FORMS.values())))
    assert math.copysign(1.0, float(oracle.decode_e4m3(np.uint8(0x80)))) == -1.0   # negative zero
    assert np.isnan(oracle.decode_e4m3(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_decode_matches_torch_float8_e4m3fn():
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.decode_e4m3(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(lib))
    ok = ~np.isnan(mine)
    assert np.array_equal(mine[ok], lib[ok])


def test_decode_order_and_sign_symmetry():
    pos = oracle.decode_e4m3(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)
    neg = oracle.decode_e4m3(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -pos)
    # spacing: one step of M is 2^(E-10) for normals, 2^-9 for subnormals
    assert pos[0x39] - pos[0x38] == 2.0 ** -3
    assert pos[0x02] - pos[0x01] == 2.0 ** -9


def test_every_code_helper():
    codes = inputs.every_e4m3_code().numpy()
    assert len(codes) == 254 and 0x7F not in codes and 0xFF not in codes
    assert not np.isnan(oracle.decode_e4m3(codes)).any()


def test_dequantize_rows_broadcasts_the_row_scale():
    q = np.array([[[0x38, 0x40], [0xB8, 0x01]]], dtype=np.uint8)          # [1][2][2]
    s = np.array([[0.5, 8.0]], dtype=np.float32)
    assert np.array_equal(oracle.dequantize_e4m3_rows(q, s), [[[0.5, 1.0], [-8.0, 8.0 * 2.0 ** -9]]])


def test_quantizer_scales_range_and_error():
    g = torch.Generator().manual_seed(5)
    W = torch.randn((3, 40, 512), generator=g) * 0.02
    W[1, 7] = 0.0                                             # a zero row
    W[2, 3] = torch.linspace(-448.0, 448.0, 512) * 2.0 ** -3  # amax / 448 an exact power of two
    q, s = inputs.quantize_e4m3_rows(W)
    assert q.dtype == torch.uint8 and s.dtype == torch.float32 and s.shape == W.shape[:-1]
    m, _ = np.frexp(s.numpy())
    assert np.all(m == 0.5)                                   # every scale a power of two
    assert s[1, 7] == 1.0 and not q[1, 7].any()
    assert s[2, 3] == 2.0 ** -3                               # no needless round-up
    vals = oracle.decode_e4m3(q.numpy())
    assert not np.isnan(vals).any() and np.abs(vals).max() <= 448.0
    # the largest element of each row is above 448/2 before rounding, so at least 224 after
    amax_q = np.abs(vals).max(axis=-1)
    nz = W.abs().amax(-1).numpy() > 0
    assert np.all(amax_q[nz] >= 224.0)
    deq = oracle.dequantize_e4m3_rows(q.numpy(), s.numpy())
    W64 = W.double().numpy()
    # nearest rounding: |error| <= half a step, 2^-4 relative for normals, 2^-10 * s for subnormals
    bound = np.maximum(np.abs(W64) * 2.0 ** -4, s.double().numpy()[..., None] * 2.0 ** -10)
    assert np.all(np.abs(deq - W64) <= bound)
    # the torch-side dequantisation equals the oracle's (both exact)
    assert np.array_equal(inputs.dequantize_e4m3_rows(q, s, torch.float32).double().numpy(), deq)


def test_widening_recipe_against_the_format():
    """The fp8 kernels widen a byte pair (b0, b1) to two bf16 with integer steps:
    f = b0 << 8 | b1 << 24, m = (b0 & 0x7f) | (b1 & 0x7f) << 16, r = f - 240 m
    (mod 2^32), each 16-bit half of r read as bf16 and multiplied by 2^120.  Here
    that recipe, restated on the host for every pair of finite codes, must give
    the oracle's decoding of the bytes exactly (zeros and subnormals included)."""
    codes = inputs.every_e4m3_code().numpy().astype(np.uint32)
    b0, b1 = np.meshgrid(codes, codes, indexing="ij")
    b0, b1 = b0.ravel(), b1.ravel()
    f = (b0 << 8) | (b1 << 24)
    m = (b0 & 0x7F) | ((b1 & 0x7F) << 16)
    r = (f - np.uint32(240) * m) & np.uint32(0xFFFFFFFF)
    lo = (r & 0xFFFF).astype(np.uint32) << 16          # bf16 bits -> fp32 bits
    hi = (r >> 16).astype(np.uint32) << 16
    v_lo = lo.view(np.float32).astype(np.float64) * 2.0 ** 120
    v_hi = hi.view(np.float32).astype(np.float64) * 2.0 ** 120
    assert np.array_equal(v_lo, oracle.decode_e4m3(b0.astype(np.uint8)))
    assert np.array_equal(v_hi, oracle.decode_e4m3(b1.astype(np.uint8)))
    # the sign of zero survives too
    assert np.array_equal(np.signbit(v_lo), np.signbit(oracle.decode_e4m3(b0.astype(np.uint8))))


def split_recipe(v: np.ndarray):
    """The e4m3-MMA kernels' token split, restated on the host: for a row v (bf16
    values), s = 2^k with max|v| * s in (224, 448]; hi = e4m3(s v), lo = e4m3(s v - hi),
    e4m3 rounding to nearest even (torch's conversion).  Returns (s, hi, lo) as
    exact fp64 values (the byte values through the oracle's decoding)."""
    mx = float(np.max(np.abs(v)))
    m, e = np.frexp(448.0 / mx)                 # 448/mx = m 2^e, 0.5 <= m < 1
    s = 2.0 ** (e - 1)                          # the largest power of two <= 448/mx
    sv = torch.from_numpy((v * s).astype(np.float32))
    hi_b = sv.to(torch.float8_e4m3fn)
    hi = hi_b.float()
    lo_b = (sv - hi).to(torch.float8_e4m3fn)
    dec = lambda b: oracle.decode_e4m3(b.view(torch.uint8).numpy())
    return s, dec(hi_b), dec(lo_b)


def test_token_split_recipe_is_exact_above_a_quarter():
    """Every bf16 value is hi + lo of two e4m3 values after the row's power-of-two
    scale, exactly when |s v| >= 1/4, and within 2^-10 (half of e4m3's smallest
    step) below; the scale puts the row's largest magnitude in (224, 448]."""
    # every finite bf16 bit pattern of magnitude in [2^-30, 448), as rows under
    # several row maxima
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    v = (bits << 16).view(np.float32).astype(np.float64)
    v = v[np.isfinite(v) & (np.abs(v) < 448.0) & ((np.abs(v) >= 2.0 ** -30) | (v == 0.0))]
    for row_max in (1.0, 3.75, 4.5, 100.0, 447.0):
        row = np.concatenate([v[np.abs(v) <= row_max], [row_max]])
        s, hi, lo = split_recipe(row)
        assert 224.0 < np.max(np.abs(row)) * s <= 448.0
        sv = row * s
        err = np.abs(hi + lo - sv)
        big = np.abs(sv) >= 0.25
        assert np.all(err[big] == 0.0)
        assert np.all(err[~big] <= 2.0 ** -10)
