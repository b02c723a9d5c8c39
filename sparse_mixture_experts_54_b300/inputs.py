"""Seeded synthetic inputs for the MoE layer workloads.

This module only draws random tensors with the shapes and distributions of the
workloads; it holds none of the layer's arithmetic.  Both the CUDA path (via
the tests and the benchmark) and the CPU oracle receive the very same values:
tensors are drawn once, on one device, and copied.

Workloads (Mixtral 8x7B shapes: d = 4096, d_ff = 14336, 8 experts, top-2):

* ``tiny_fp32``      T=64, d=128, d_ff=256, fp32 everything.  x ~ N(0,1),
                     W_g ~ N(0, 0.02), W1, W3 ~ N(0, 1/sqrt(d)), W2 ~ N(0, 1/sqrt(d_ff)).
* ``decode_t32``     T=32, bf16 x (N(0,1) rows scaled to unit RMS) and bf16
                     expert weights N(0, 1/sqrt(fan_in)); fp32 router N(0, 1/sqrt(d)).
* ``prefill_t4096``  T=4096, same distributions.
* ``skewed_t32768``  T=32768, same distributions plus a per-expert router bias
                     [1.5, 0.5, 0, 0, 0, 0, -0.5, -1]; with probability 1/2 a
                     token's row repeats the previous token's row plus N(0, 0.1)
                     noise (consecutive-token locality), then rows are scaled to
                     unit RMS and rounded to bf16.
* ``stack32``        32 layers of the decode/prefill shapes, layer l seeded
                     with 1000 + l.

Standard deviations are written as sigma in N(0, sigma).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    d_ff: int
    n_experts: int = 8
    k: int = 2
    dtype: str = "bf16"            # element type of x, W1, W3, W2 and y
    router_sigma: Optional[float] = None   # None -> 1/sqrt(d)
    bias: Optional[Sequence[float]] = None
    locality_p: float = 0.0        # probability that row t repeats row t-1 (+ noise)
    locality_sigma: float = 0.1
    rms_normalise_x: bool = True
    seed: int = 0
    notes: str = ""

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


MIXTRAL = dict(d=4096, d_ff=14336, n_experts=8, k=2)

WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", T=64, d=128, d_ff=256, dtype="f32", router_sigma=0.02,
                          rms_normalise_x=False, notes="fp32 parity case"),
    "decode_t32": Workload("decode_t32", T=32, **MIXTRAL, notes="decode regime, weight streaming"),
    "prefill_t4096": Workload("prefill_t4096", T=4096, **MIXTRAL, notes="prefill regime"),
    "skewed_t32768": Workload("skewed_t32768", T=32768, **MIXTRAL,
                              bias=(1.5, 0.5, 0.0, 0.0, 0.0, 0.0, -0.5, -1.0), locality_p=0.5,
                              notes="skewed, locally correlated routing at 32k context"),
}

STACK_LAYERS = 32
STACK_DECODE_T = (1, 8, 32, 128, 256)
STACK_PREFILL_T = 8192


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    if overrides:
        w = Workload(**{**w.__dict__, **overrides})
    return w


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, sigma: float, dtype, device, g) -> torch.Tensor:
    # Drawn in fp32, scaled, then stored in the workload's element type.
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(sigma)
    return t.to(dtype)


def make_x(w: Workload, device="cpu", seed: Optional[int] = None, T: Optional[int] = None) -> torch.Tensor:
    """Token rows x [T][d] in the workload's element type."""
    T = w.T if T is None else T
    g = _gen(device, (w.seed if seed is None else seed) * 7919 + 1)
    x = torch.randn((T, w.d), generator=g, device=device, dtype=torch.float32)
    if w.locality_p > 0.0 and T > 1:
        repeat = torch.rand((T,), generator=g, device=device) < w.locality_p
        repeat[0] = False
        noise = torch.randn((T, w.d), generator=g, device=device, dtype=torch.float32) * w.locality_sigma
        # Row t = row t-1 + noise[t] where repeat[t].  A run of repeats starting
        # after fresh row s gives row t = x[s] + sum_{u=s+1..t} noise[u].
        noise = noise * repeat[:, None].to(torch.float32)
        csum = torch.cumsum(noise, dim=0)
        ar = torch.arange(T, device=device)
        start = torch.cummax(torch.where(repeat, torch.zeros_like(ar), ar), dim=0).values
        x = x[start] + (csum - csum[start])
    if w.rms_normalise_x:
        x = x / torch.sqrt((x * x).mean(dim=1, keepdim=True))
    return x.to(w.torch_dtype).contiguous()


def make_router(w: Workload, device="cpu", seed: Optional[int] = None):
    """Router weight W_g [n][d] fp32 and optional bias [n] fp32."""
    g = _gen(device, (w.seed if seed is None else seed) * 7919 + 2)
    sigma = w.router_sigma if w.router_sigma is not None else 1.0 / math.sqrt(w.d)
    Wg = _normal((w.n_experts, w.d), sigma, torch.float32, device, g).contiguous()
    b = None
    if w.bias is not None:
        b = torch.tensor(list(w.bias), dtype=torch.float32, device=device)
    return Wg, b


def make_experts(w: Workload, device="cpu", seed: Optional[int] = None):
    """Expert weights W1, W3 [n][d_ff][d] and W2 [n][d][d_ff] in the workload's element type."""
    s = w.seed if seed is None else seed
    dt = w.torch_dtype
    g = _gen(device, s * 7919 + 3)
    W1 = torch.empty((w.n_experts, w.d_ff, w.d), dtype=dt, device=device)
    W3 = torch.empty_like(W1)
    W2 = torch.empty((w.n_experts, w.d, w.d_ff), dtype=dt, device=device)
    # One expert at a time keeps the fp32 staging buffer small at Mixtral shape.
    for e in range(w.n_experts):
        W1[e] = _normal((w.d_ff, w.d), 1.0 / math.sqrt(w.d), dt, device, g)
        W3[e] = _normal((w.d_ff, w.d), 1.0 / math.sqrt(w.d), dt, device, g)
        W2[e] = _normal((w.d, w.d_ff), 1.0 / math.sqrt(w.d_ff), dt, device, g)
    return W1, W3, W2


def make_layer(w: Workload, device="cpu", seed: Optional[int] = None, T: Optional[int] = None) -> dict:
    """Everything one MoE layer call needs, drawn from ``seed`` (default: the workload's)."""
    x = make_x(w, device, seed, T)
    Wg, b = make_router(w, device, seed)
    W1, W3, W2 = make_experts(w, device, seed)
    return dict(x=x, Wg=Wg, bias=b, W1=W1, W3=W3, W2=W2)


def to_oracle(t: Optional[torch.Tensor]):
    """Host numpy view with the stored bits: bf16 -> uint16 bit patterns, fp32 -> float32."""
    if t is None:
        return None
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)


def sample_tokens(T: int, count: int, seed: int = 0) -> torch.Tensor:
    """A seeded, sorted sample of distinct token numbers in [0, T)."""
    if count >= T:
        return torch.arange(T, dtype=torch.int64)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 12345)
    return torch.randperm(T, generator=g)[:count].sort().values


E4M3_MAX = 448.0


def quantize_e4m3_rows(W: torch.Tensor):
    """fp8 expert weights for ``moe_forward_fp8``: per weight row (last axis
    reduced) the smallest power-of-two scale s with max|W_row| / s <= 448, and
    q = e4m3(W_row / s) (torch's round-to-nearest cast; the division is exact).
    Returns (q as torch.uint8 bytes, s as float32), on W's device.  Rows of zeros
    get s = 1.  With power-of-two scales the dequantised weights s * q are exact
    in bf16, so the fp8 path can be checked against the bf16 path bit for bit."""
    Wf = W.float()
    amax = Wf.abs().amax(dim=-1)
    m, e = torch.frexp(amax / E4M3_MAX)          # amax / 448 = m * 2^e, 0.5 <= m < 1
    e = torch.where(m == 0.5, e - 1, e)          # an exact power of two needs no round-up
    s = torch.where(amax > 0, torch.ldexp(torch.ones_like(amax), e), torch.ones_like(amax))
    q = (Wf / s[..., None]).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), s.contiguous()


def dequantize_e4m3_rows(q: torch.Tensor, s: torch.Tensor, dtype=torch.bfloat16) -> torch.Tensor:
    """s[..., None] * e4m3(q) in ``dtype`` (exact in bf16 for power-of-two s)."""
    return (s[..., None] * q.view(torch.float8_e4m3fn).float()).to(dtype)


def every_e4m3_code(device="cpu") -> torch.Tensor:
    """The 254 non-NaN e4m3 bytes, ascending: zeros, subnormals, normals, both signs."""
    return torch.tensor([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=torch.uint8, device=device)
