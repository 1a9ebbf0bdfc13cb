"""ctypes binding of libcompkv.so: the C-ABI calls under the same names.

Argument marshalling only: pointers are passed as integers (device addresses
or host addresses), streams as cudaStream_t handles.  Every step of the decode
path runs in the library's CUDA kernels; there is no Python or CPU fallback,
and loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_int, c_int64, c_size_t, c_void_p

from ._build import HEADER, LIB

COMPKV_OK = 0
STATUS_NAMES = {
    0: "COMPKV_OK", 1: "COMPKV_ERR_INVALID_ARG", 2: "COMPKV_ERR_UNSUPPORTED_SHAPE",
    3: "COMPKV_ERR_CAPACITY", 4: "COMPKV_ERR_CUDA", 5: "COMPKV_ERR_TIMEOUT",
    6: "COMPKV_ERR_BAD_SELECTION", 7: "COMPKV_ERR_INTERNAL",
}


class compkv_config(ctypes.Structure):
    _fields_ = [("num_layers", c_int), ("batch", c_int), ("num_kv_heads", c_int),
                ("group_size", c_int), ("head_dim", c_int), ("block_size", c_int),
                ("r", c_int), ("budget_tokens", c_int), ("max_tokens", c_int),
                ("capacity_tokens", POINTER(c_int)), ("variant", c_int)]


# ablation bits of compkv_config.variant (include/compkv.h)
VARIANT_FIRST_ORDER_MASS = 1
VARIANT_NO_VARIANCE_FACTOR = 2
VARIANT_NO_COMPENSATION = 4


class compkv_buffers(ctypes.Structure):
    _fields_ = [("k", c_void_p), ("v", c_void_p), ("kbar", c_void_p), ("vbar", c_void_p),
                ("dbar", c_void_p), ("seq_len", c_void_p), ("scratch", c_void_p),
                ("scratch_bytes", c_size_t)]


class CompKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None

# (name, restype, argtypes) of every entry point declared in include/compkv.h
_SIGNATURES = [
    ("compkv_rows_per_layer", c_int64, [POINTER(compkv_config)]),
    ("compkv_scratch_bytes", c_size_t, [POINTER(compkv_config)]),
    ("compkv_init", c_int, [POINTER(compkv_config), POINTER(compkv_buffers), POINTER(c_void_p)]),
    ("compkv_row_offset", c_int, [c_void_p, c_int, c_int, c_int, POINTER(c_int64), POINTER(c_int)]),
    ("compkv_prefill", c_int, [c_void_p, c_int, POINTER(c_int), c_void_p]),
    ("compkv_append", c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p]),
    ("compkv_score_select", c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p]),
    ("compkv_attend", c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p]),
    ("compkv_decode", c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    ("compkv_decode_host", c_int, [c_void_p, c_int, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    ("compkv_decode_static", c_int, [POINTER(compkv_config), POINTER(compkv_buffers), c_int, c_void_p, c_void_p,
                                     c_void_p, c_void_p, c_void_p, c_void_p]),
    ("compkv_device_status", c_int, [c_void_p, c_void_p]),
    ("compkv_launch_count", c_int64, [c_void_p]),
    ("compkv_selftest_wait_timeout", c_int, [c_void_p, c_void_p]),
    ("compkv_profile_enable", c_int, [c_void_p, c_int]),
    ("compkv_trace", c_int, [c_void_p, c_void_p, c_size_t]),
    ("compkv_profile_read", c_int, [c_void_p, c_int, POINTER(ctypes.c_double), POINTER(c_int64)]),
    ("compkv_last_error", c_char_p, []),
    ("compkv_status_string", c_char_p, [c_int]),
    ("compkv_destroy", None, [c_void_p]),
]


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is not built; run block_sparse_kv_summary_gb300.build() first")
        L = ctypes.CDLL(LIB)
        for name, res, args in _SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def library_path() -> str:
    return LIB


def header_path() -> str:
    return HEADER


def compkv_last_error() -> str:
    return lib().compkv_last_error().decode()


def compkv_status_string(status: int) -> str:
    return lib().compkv_status_string(status).decode()


def _check(status: int, what: str):
    if status != COMPKV_OK:
        raise CompKVError(status, f"{what}: {compkv_last_error()}")


def make_config(num_layers, batch, num_kv_heads, group_size, head_dim, r, budget_tokens,
                max_tokens=0, capacity_tokens=None, block_size=16, variant=0) -> compkv_config:
    cfg = compkv_config(num_layers, batch, num_kv_heads, group_size, head_dim, block_size, r,
                        budget_tokens, max_tokens, None, variant)
    if capacity_tokens is not None:
        arr = (c_int * len(capacity_tokens))(*capacity_tokens)
        cfg.capacity_tokens = ctypes.cast(arr, POINTER(c_int))
        cfg._keep = arr  # keep the host array alive with the struct
    return cfg


def compkv_rows_per_layer(cfg: compkv_config) -> int:
    return lib().compkv_rows_per_layer(ctypes.byref(cfg))


def compkv_scratch_bytes(cfg: compkv_config) -> int:
    return lib().compkv_scratch_bytes(ctypes.byref(cfg))


def compkv_init(cfg: compkv_config, bufs: compkv_buffers) -> int:
    ctx = c_void_p()
    _check(lib().compkv_init(ctypes.byref(cfg), ctypes.byref(bufs), ctypes.byref(ctx)), "compkv_init")
    return ctx.value


def compkv_row_offset(ctx, layer, seq, head):
    row, cap = c_int64(), c_int()
    _check(lib().compkv_row_offset(ctx, layer, seq, head, ctypes.byref(row), ctypes.byref(cap)),
           "compkv_row_offset")
    return row.value, cap.value


def compkv_prefill(ctx, layer, lens, stream):
    arr = (c_int * len(lens))(*lens)
    _check(lib().compkv_prefill(ctx, layer, arr, stream), "compkv_prefill")


def compkv_append(ctx, layer, k_new, v_new, stream):
    _check(lib().compkv_append(ctx, layer, k_new, v_new, stream), "compkv_append")


def compkv_score_select(ctx, layer, q, sel, scores, stream):
    _check(lib().compkv_score_select(ctx, layer, q, sel, scores, stream), "compkv_score_select")


def compkv_attend(ctx, layer, q, sel, out, stream):
    _check(lib().compkv_attend(ctx, layer, q, sel, out, stream), "compkv_attend")


def compkv_decode(ctx, layer, q, k_new, v_new, out, sel, stream):
    _check(lib().compkv_decode(ctx, layer, q, k_new, v_new, out, sel, stream), "compkv_decode")


def compkv_decode_host(ctx, layer, q, k_new, v_new, out, sel, stream):
    """compkv_decode from host buffers to host buffers (addresses of host memory); synchronises."""
    _check(lib().compkv_decode_host(ctx, layer, q, k_new, v_new, out, sel, stream), "compkv_decode_host")


class PreparedDecode:
    """compkv_decode with the context and stream bound once: each call passes
    plain addresses (ints) and pays only the ctypes call and the library's own
    checks."""

    def __init__(self, ctx, stream):
        self._fn = lib().compkv_decode
        self._ctx = c_void_p(ctx)
        self._stream = c_void_p(stream)

    def __call__(self, layer, q, k_new, v_new, out, sel=None):
        st = self._fn(self._ctx, layer, q, k_new, v_new, out, sel, self._stream)
        if st != COMPKV_OK:
            raise CompKVError(st, f"compkv_decode: {compkv_last_error()}")


COMPKV_STATIC_SCRATCH_BYTES = 16 << 20


def compkv_decode_static(cfg, bufs, layer, q, k_new, v_new, out, sel, stream):
    """compkv_decode without a context, on the library's own static scratch
    (bufs.scratch is ignored); see include/compkv.h."""
    _check(lib().compkv_decode_static(ctypes.byref(cfg), ctypes.byref(bufs), layer, q, k_new, v_new, out, sel,
                                      stream), "compkv_decode_static")


def compkv_device_status(ctx, stream) -> int:
    """Synchronise, read and clear the device status word; returns the status code."""
    return lib().compkv_device_status(ctx, stream)


def compkv_selftest_wait_timeout(ctx, stream):
    """Enqueue the bounded-wait self-test (its wait runs out and records a timeout)."""
    _check(lib().compkv_selftest_wait_timeout(ctx, stream), "compkv_selftest_wait_timeout")


def compkv_launch_count(ctx) -> int:
    return lib().compkv_launch_count(ctx)


KERNEL_FAMILIES = {"prefill": 0, "append": 1, "score": 2, "attend": 4, "decode": 5,
                   "k_stream": 6, "k_post": 7}


def compkv_profile_enable(ctx, enable):
    """enable: False/0 off, True/1 per API call, 2 per call and per kernel of a chain."""
    _check(lib().compkv_profile_enable(ctx, int(enable)), "compkv_profile_enable")


def compkv_profile_read(ctx, family):
    """(total device ms, launches) of a kernel family since the last read."""
    fam = KERNEL_FAMILIES[family] if isinstance(family, str) else int(family)
    ms, n = ctypes.c_double(), c_int64()
    _check(lib().compkv_profile_read(ctx, fam, ctypes.byref(ms), ctypes.byref(n)), "compkv_profile_read")
    return ms.value, n.value


def compkv_trace(ctx, buf, nbytes):
    """Record the fused kernel's work items into device buffer `buf` (0: off)."""
    _check(lib().compkv_trace(ctx, buf, nbytes), "compkv_trace")


def compkv_destroy(ctx):
    lib().compkv_destroy(ctx)
