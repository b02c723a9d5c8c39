"""Torch-facing wrapper of the C ABI: device memory and streams come from
PyTorch, every step of the layer runs in the library's CUDA kernels."""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dev_ptr(t: Optional[torch.Tensor], dtype=None, name: str = "") -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


class MoELayer:
    """Mixtral sparse MoE FFN: y = sum_{top-k experts} softmax-gate * SwiGLU_e(x).

    Weights are caller-owned torch tensors (nn.Linear layouts): W_g [n][d] fp32,
    W1/W3 [n][d_ff][d], W2 [n][d][d_ff] in ``dtype`` (torch.bfloat16 or torch.float32).
    """

    def __init__(self, d: int, d_ff: int, n_experts: int = 8, k: int = 2, dtype=torch.bfloat16,
                 bias: Optional[torch.Tensor] = None):
        self.d, self.d_ff, self.n, self.k = d, d_ff, n_experts, k
        self.dtype = dtype
        ctx = _lib.moe_create(d, d_ff, n_experts, k)
        if not ctx:
            raise _lib.MoEError(_lib.MOE_ERR_INVALID, "moe_create")
        self.ctx = ctx
        _lib.check(_lib.moe_set_dtype(ctx, _lib.MOE_F32 if dtype == torch.float32 else _lib.MOE_BF16),
                   "moe_set_dtype")
        self._bias = None
        if bias is not None:
            self.set_bias(bias)

    def set_bias(self, bias: Optional[torch.Tensor]):
        self._bias = bias
        _lib.check(_lib.moe_set_router_bias(self.ctx, _dev_ptr(bias, torch.float32, "bias")), "moe_set_router_bias")

    def set_option(self, option: int, value: int):
        _lib.check(_lib.moe_set_option(self.ctx, option, int(value)), "moe_set_option")

    def reserve(self, T_max: int):
        _lib.check(_lib.moe_reserve(self.ctx, T_max), "moe_reserve")

    def workspace_bytes(self, T: int) -> int:
        return _lib.moe_workspace_bytes(self.ctx, T)

    def route(self, x: torch.Tensor, Wg: torch.Tensor, stream=None) -> dict:
        T = x.shape[0]
        dev = x.device
        out = dict(
            topk_idx=torch.empty((T, self.k), dtype=torch.int32, device=dev),
            topk_w=torch.empty((T, self.k), dtype=torch.float32, device=dev),
            counts=torch.empty((self.n,), dtype=torch.int32, device=dev),
            offsets=torch.empty((self.n + 1,), dtype=torch.int32, device=dev),
            perm=torch.empty((T * self.k,), dtype=torch.int32, device=dev),
        )
        _lib.check(_lib.moe_route(self.ctx, _dev_ptr(x, self.dtype, "x"), _dev_ptr(Wg, torch.float32, "W_g"), T,
                                  out["topk_idx"].data_ptr(), out["topk_w"].data_ptr(), out["counts"].data_ptr(),
                                  out["offsets"].data_ptr(), out["perm"].data_ptr(), _stream_handle(stream)),
                   "moe_route")
        return out

    def router_logits(self, x: torch.Tensor, Wg: torch.Tensor, stream=None) -> torch.Tensor:
        T = x.shape[0]
        logits = torch.empty((T, self.n), dtype=torch.float32, device=x.device)
        _lib.check(_lib.moe_router_logits(self.ctx, _dev_ptr(x, self.dtype, "x"), _dev_ptr(Wg, torch.float32, "W_g"),
                                          T, logits.data_ptr(), _stream_handle(stream)), "moe_router_logits")
        return logits

    def forward(self, x, Wg, W1, W3, W2, y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.d), dtype=self.dtype, device=x.device)
        _lib.check(_lib.moe_forward(self.ctx, _dev_ptr(x, self.dtype, "x"), _dev_ptr(Wg, torch.float32, "W_g"),
                                    _dev_ptr(W1, self.dtype, "W1"), _dev_ptr(W3, self.dtype, "W3"),
                                    _dev_ptr(W2, self.dtype, "W2"), _dev_ptr(y, self.dtype, "y"), T,
                                    _stream_handle(stream)), "moe_forward")
        return y

    __call__ = forward

    def forward_host(self, x_host: torch.Tensor, Wg, W1, W3, W2, y_host: torch.Tensor, stream=None):
        """x_host / y_host: CPU tensors (pinned for asynchronous copies)."""
        if x_host.is_cuda or y_host.is_cuda:
            raise ValueError("forward_host takes host tensors")
        T = x_host.shape[0]
        _lib.check(_lib.moe_forward_host(self.ctx, x_host.data_ptr(), _dev_ptr(Wg, torch.float32, "W_g"),
                                         _dev_ptr(W1, self.dtype, "W1"), _dev_ptr(W3, self.dtype, "W3"),
                                         _dev_ptr(W2, self.dtype, "W2"), y_host.data_ptr(), T,
                                         _stream_handle(stream)), "moe_forward_host")
        return y_host

    def forward_fp8(self, x, Wg, W1q, W1_scale, W3q, W3_scale, W2q, W2_scale, y: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
        """y = MoE(x) with e4m3 expert weights (torch.float8_e4m3fn or their bytes as torch.uint8)
        and fp32 row scales: W1 = W1_scale[..., None] * W1q, likewise W3 and W2 (bf16 layers only)."""
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.d), dtype=self.dtype, device=x.device)
        q = {}
        for name, t in (("W1q", W1q), ("W3q", W3q), ("W2q", W2q)):
            if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
                raise ValueError(f"{name} must be torch.float8_e4m3fn or torch.uint8, got {t.dtype}")
            q[name] = _dev_ptr(t, None, name)
        _lib.check(_lib.moe_forward_fp8(self.ctx, _dev_ptr(x, self.dtype, "x"), _dev_ptr(Wg, torch.float32, "W_g"),
                                        q["W1q"], _dev_ptr(W1_scale, torch.float32, "W1_scale"),
                                        q["W3q"], _dev_ptr(W3_scale, torch.float32, "W3_scale"),
                                        q["W2q"], _dev_ptr(W2_scale, torch.float32, "W2_scale"),
                                        _dev_ptr(y, self.dtype, "y"), T, _stream_handle(stream)), "moe_forward_fp8")
        return y

    def block_forward(self, h: torch.Tensor, Wg, W1, W3, W2, eps: float = 1e-5, stream=None) -> torch.Tensor:
        """In place: h <- h + MoE(RMSNorm(h)) (one residual block of a stack)."""
        T = h.shape[0]
        _lib.check(_lib.moe_block_forward(self.ctx, _dev_ptr(h, self.dtype, "h"), float(eps),
                                          _dev_ptr(Wg, torch.float32, "W_g"), _dev_ptr(W1, self.dtype, "W1"),
                                          _dev_ptr(W3, self.dtype, "W3"), _dev_ptr(W2, self.dtype, "W2"), T,
                                          _stream_handle(stream)), "moe_block_forward")
        return h

    def stack_forward(self, h: torch.Tensor, layers, eps: float = 1e-5, stream=None) -> torch.Tensor:
        """In place over the layers in order; ``layers`` is a sequence of (W_g, W1, W3, W2)."""
        import ctypes
        L = len(layers)
        arrs = [(ctypes.c_void_p * max(L, 1))() for _ in range(4)]
        for l, (Wg, W1, W3, W2) in enumerate(layers):
            arrs[0][l] = _dev_ptr(Wg, torch.float32, "W_g")
            arrs[1][l] = _dev_ptr(W1, self.dtype, "W1")
            arrs[2][l] = _dev_ptr(W3, self.dtype, "W3")
            arrs[3][l] = _dev_ptr(W2, self.dtype, "W2")
        T = h.shape[0]
        _lib.check(_lib.moe_stack_forward(self.ctx, _dev_ptr(h, self.dtype, "h"), float(eps), L,
                                          *(ctypes.addressof(a) for a in arrs), T, _stream_handle(stream)),
                   "moe_stack_forward")
        return h

    def stage_times(self) -> tuple:
        """(dict stage -> mean ms per call, calls) for calls made with MOE_OPT_STAGE_TIMING on."""
        import ctypes
        ms = (ctypes.c_float * 16)()
        calls = ctypes.c_int(0)
        n = _lib.moe_stage_times(self.ctx, ctypes.addressof(ms), 16, ctypes.addressof(calls))
        if n < 0:
            raise _lib.MoEError(n, "moe_stage_times")
        return {_lib.moe_stage_name(i): float(ms[i]) for i in range(n)}, calls.value

    def status(self) -> int:
        return _lib.moe_status(self.ctx)

    def clear_status(self):
        _lib.moe_clear_status(self.ctx)

    def close(self):
        if getattr(self, "ctx", None):
            _lib.moe_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
