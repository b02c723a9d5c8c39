"""ctypes binding of libmoe_b300.so: one Python function per C entry point of
include/moe.h, same names, argument marshalling only.

Pointers are passed as Python ints (device or host addresses) and streams as
the raw ``cudaStream_t`` value (``torch.cuda.Stream.cuda_stream``; 0 for the
legacy default stream).  Loading fails loudly when the library has not been
built: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

MOE_OK = 0
MOE_ERR_INVALID = -1
MOE_ERR_CUDA = -2
MOE_ERR_OOM = -3
MOE_ERR_TIMEOUT = -4
MOE_ERR_UNSUPPORTED = -5
MOE_ERR_BOUNDS = -6
MOE_ERR_SCRATCH_LIMIT = -7

MOE_BF16 = 0
MOE_F32 = 1

MOE_OPT_DECODE_MAX_T = 1
MOE_OPT_WAIT_LIMIT_US = 2
MOE_OPT_FORCE_PATH = 3
MOE_OPT_STAGE_TIMING = 4
MOE_OPT_GEMM_PAIR = 5
MOE_OPT_HOST_OUTPUT = 6
MOE_OPT_FP8_WIDEN = 7
MOE_OPT_DECODE_STREAMK = 8

# Every entry point declared in include/moe.h, with its ctypes signature.
_P = ctypes.c_void_p
_I = ctypes.c_int
_LL = ctypes.c_longlong
SIGNATURES = {
    "moe_create": (_P, [_I, _I, _I, _I]),
    "moe_set_dtype": (_I, [_P, _I]),
    "moe_set_router_bias": (_I, [_P, _P]),
    "moe_set_option": (_I, [_P, _I, _LL]),
    "moe_reserve": (_I, [_P, _I]),
    "moe_workspace_bytes": (ctypes.c_size_t, [_P, _I]),
    "moe_route": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P]),
    "moe_router_logits": (_I, [_P, _P, _P, _I, _P, _P]),
    "moe_forward": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P]),
    "moe_forward_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _P]),
    "moe_block_forward": (_I, [_P, _P, ctypes.c_float, _P, _P, _P, _P, _I, _P]),
    "moe_stack_forward": (_I, [_P, _P, ctypes.c_float, _I, _P, _P, _P, _P, _I, _P]),
    "moe_forward_fp8": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P]),
    "moe_status": (_I, [_P]),
    "moe_clear_status": (_I, [_P]),
    "moe_selftest_wait_timeout": (_I, [_P, _LL, _P]),
    "moe_forward_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P]),
    "moe_stage_times": (_I, [_P, _P, _I, _P]),
    "moe_stage_name": (ctypes.c_char_p, [_I]),
    "moe_error_string": (ctypes.c_char_p, [_I]),
    "moe_destroy": (None, [_P]),
}

_lib = None


class MoEError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {error_string(code)} ({code})" if what else f"{error_string(code)} ({code})")


def load():
    """Load the shared library (raises if it is missing: build it with __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing; build it with `python -m "
                               "sparse_mixture_experts_54_b300.build` (there is no fallback path)")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def check(code: int, what: str = "") -> int:
    if code != MOE_OK:
        raise MoEError(code, what)
    return code


def error_string(code: int) -> str:
    try:
        return load().moe_error_string(code).decode()
    except Exception:  # library not loadable: still name the code
        return str(code)


def _p(v):
    return None if v is None or v == 0 else int(v)


def moe_create(d: int, d_ff: int, n_experts: int, k: int):
    return load().moe_create(d, d_ff, n_experts, k)


def moe_set_dtype(ctx, dtype: int) -> int:
    return load().moe_set_dtype(ctx, dtype)


def moe_set_router_bias(ctx, b_g) -> int:
    return load().moe_set_router_bias(ctx, _p(b_g))


def moe_set_option(ctx, option: int, value: int) -> int:
    return load().moe_set_option(ctx, option, value)


def moe_reserve(ctx, T_max: int) -> int:
    return load().moe_reserve(ctx, T_max)


def moe_workspace_bytes(ctx, T: int) -> int:
    return load().moe_workspace_bytes(ctx, T)


def moe_route(ctx, x, W_g, T, topk_idx, topk_w, counts, offsets, perm, stream) -> int:
    return load().moe_route(ctx, _p(x), _p(W_g), T, _p(topk_idx), _p(topk_w), _p(counts), _p(offsets),
                            _p(perm), _p(stream))


def moe_router_logits(ctx, x, W_g, T, logits, stream) -> int:
    return load().moe_router_logits(ctx, _p(x), _p(W_g), T, _p(logits), _p(stream))


def moe_forward(ctx, x, W_g, W1, W3, W2, y, T, stream) -> int:
    return load().moe_forward(ctx, _p(x), _p(W_g), _p(W1), _p(W3), _p(W2), _p(y), T, _p(stream))


def moe_forward_host(ctx, x_host, W_g, W1, W3, W2, y_host, T, stream) -> int:
    return load().moe_forward_host(ctx, _p(x_host), _p(W_g), _p(W1), _p(W3), _p(W2), _p(y_host), T, _p(stream))


def moe_block_forward(ctx, h, eps, W_g, W1, W3, W2, T, stream) -> int:
    return load().moe_block_forward(ctx, _p(h), float(eps), _p(W_g), _p(W1), _p(W3), _p(W2), T, _p(stream))


def moe_stack_forward(ctx, h, eps, n_layers, W_g, W1, W3, W2, T, stream) -> int:
    """W_g, W1, W3, W2: addresses of host arrays of n_layers device pointers."""
    return load().moe_stack_forward(ctx, _p(h), float(eps), n_layers, _p(W_g), _p(W1), _p(W3), _p(W2), T,
                                    _p(stream))


def moe_forward_fp8(ctx, x, W_g, W1q, W1_scale, W3q, W3_scale, W2q, W2_scale, y, T, stream) -> int:
    return load().moe_forward_fp8(ctx, _p(x), _p(W_g), _p(W1q), _p(W1_scale), _p(W3q), _p(W3_scale), _p(W2q),
                                  _p(W2_scale), _p(y), T, _p(stream))


def moe_status(ctx) -> int:
    return load().moe_status(ctx)


def moe_clear_status(ctx) -> int:
    return load().moe_clear_status(ctx)


def moe_selftest_wait_timeout(ctx, wait_limit_us: int, stream) -> int:
    return load().moe_selftest_wait_timeout(ctx, wait_limit_us, _p(stream))


def moe_forward_noalloc(x, W_g, b_g, W1, W3, W2, y, T, d, d_ff, n_experts, k, dtype, status, stream) -> int:
    return load().moe_forward_noalloc(_p(x), _p(W_g), _p(b_g), _p(W1), _p(W3), _p(W2), _p(y), T, d, d_ff,
                                      n_experts, k, dtype, _p(status), _p(stream))


def moe_stage_times(ctx, ms, max_stages: int, calls) -> int:
    return load().moe_stage_times(ctx, _p(ms), max_stages, _p(calls))


def moe_stage_name(i: int):
    r = load().moe_stage_name(i)
    return None if r is None else r.decode()


def moe_error_string(code: int) -> str:
    return load().moe_error_string(code).decode()


def moe_destroy(ctx) -> None:
    if ctx:
        load().moe_destroy(ctx)
