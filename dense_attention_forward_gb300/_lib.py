"""ctypes binding of include/attn.h (argument marshalling only)."""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn.so")
SELFTEST_PATH = os.path.join(PKG, "libattn_selftest.so")
TEST_HOOKS_PATH = os.path.join(PKG, "libattn_testhooks.so")

ATTN_OK = 0
# Rows (B * H * S) the library's own staging array holds for attn_fwd_host_noalloc; the same
# number as ATTN_NOALLOC_MAX_ROWS in include/attn.h.
NOALLOC_MAX_ROWS = 32768
STATUS_NAMES = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED_DIM",
    3: "ATTN_ERR_MISALIGNED", 4: "ATTN_ERR_UNSUPPORTED_DEVICE", 5: "ATTN_ERR_LAUNCH",
    6: "ATTN_ERR_TIMEOUT",
}

# Every symbol include/attn.h declares, with its ctypes signature.
SIGNATURES = {
    "attn_fwd": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int, ctypes.c_float, ctypes.c_void_p]),
    "attn_fwd_ex": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                   ctypes.c_void_p]),
    "attn_fwd_strided": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                        ctypes.POINTER(ctypes.c_longlong),
                                        ctypes.POINTER(ctypes.c_longlong),
                                        ctypes.POINTER(ctypes.c_longlong),
                                        ctypes.POINTER(ctypes.c_longlong), ctypes.c_int,
                                        ctypes.c_int, ctypes.c_void_p]),
    "attn_fwd_causal": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                       ctypes.c_void_p]),
    "attn_fwd_host": (ctypes.c_int, [ctypes.c_void_p] * 10 + [ctypes.c_int] * 4 +
                      [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "attn_fwd_host_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4 +
                              [ctypes.c_float, ctypes.c_int, ctypes.c_void_p]),
    "attn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "attn_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint), ctypes.c_int]),
    "attn_version": (ctypes.c_int, []),
}

# The test-hook build's extra symbol (include/attn_test_hooks.h).
TEST_HOOK_SIGNATURES = {
    "attn_fwd_withhold": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                         ctypes.c_int, ctypes.c_void_p]),
}

_lib = None
_selftest = None
_test_hooks = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str = "attn_fwd"):
        self.status = status
        super().__init__(f"{what} failed: {STATUS_NAMES.get(status, status)} "
                         f"({lib().attn_status_string(status).decode()})")


def lib():
    """The loaded libattn.so. Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -m dense_attention_forward_gb300.build "
                "or __graft_entry__.build()); the attention path has no CPU fallback")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def test_hooks_lib():
    """libattn_testhooks.so (the kernels with -DATTN_TEST_HOOKS), for the tests of the bounded
    waits. It carries its own copy of the device status word: read it through this handle."""
    global _test_hooks
    if _test_hooks is None:
        if not os.path.exists(TEST_HOOKS_PATH):
            raise RuntimeError(f"{TEST_HOOKS_PATH} is missing: build it first")
        h = ctypes.CDLL(TEST_HOOKS_PATH)
        for name, (res, args) in {**SIGNATURES, **TEST_HOOK_SIGNATURES}.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _test_hooks = h
    return _test_hooks


def selftest_lib():
    global _selftest
    if _selftest is None:
        if not os.path.exists(SELFTEST_PATH):
            raise RuntimeError(f"{SELFTEST_PATH} is missing: build it first")
        h = ctypes.CDLL(SELFTEST_PATH)
        h.attn_selftest_gemm.restype = ctypes.c_int
        h.attn_selftest_gemm.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_int, ctypes.c_void_p]
        h.attn_selftest_elementwise.restype = ctypes.c_int
        h.attn_selftest_elementwise.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_void_p]
        _selftest = h
    return _selftest


def attn_fwd(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int | None, B: int, H: int,
             S: int, D: int, scale: float, stream: int | None) -> int:
    """Direct call of the C entry point with raw addresses; returns the status code."""
    return lib().attn_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, S, D, scale, stream)


def attn_fwd_ex(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int | None, B: int, H: int,
                S: int, D: int, scale: float, rebase_threshold_log2: int, stream: int | None) -> int:
    """Direct call of attn_fwd_ex (rebase threshold 0, 1 or 8); returns the status code."""
    return lib().attn_fwd_ex(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, S, D, scale,
                             rebase_threshold_log2, stream)


def attn_fwd_strided(q_ptr: int, k_ptr: int, v_ptr: int, o_ptr: int, lse_ptr: int | None, B: int,
                     H: int, S: int, D: int, scale: float, q_strides, k_strides, v_strides,
                     o_strides, rebase_threshold_log2: int, causal: int, stream: int | None) -> int:
    """Direct call of attn_fwd_strided; each *_strides is (batch, head, seq) in elements."""
    arr = ctypes.c_longlong * 3
    return lib().attn_fwd_strided(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, S, D, scale,
                                  arr(*q_strides), arr(*k_strides), arr(*v_strides),
                                  arr(*o_strides), rebase_threshold_log2, causal, stream)


def device_status(reset: bool = True) -> int:
    word = ctypes.c_uint(0)
    st = lib().attn_device_status(ctypes.byref(word), 1 if reset else 0)
    if st != ATTN_OK:
        raise AttnError(st, "attn_device_status")
    return word.value


_ROLES = {1: "TMA producer", 2: "MMA issue", 3: "softmax", 4: "O correction"}


def check_device_status(reset: bool = True) -> None:
    """Raise AttnError(ATTN_ERR_TIMEOUT) if a kernel gave up a bounded wait since the word was
    last cleared (call after synchronising the streams that ran the kernels)."""
    word = device_status(reset)
    if word != 0:
        role = _ROLES.get((word >> 8) & 0xFF, "unknown role")
        idx = word & 0xFF
        what = f"mbarrier {idx}" if idx < 18 else f"S-seen count of Q tile {idx - 18}"
        raise AttnError(6, f"kernel (status word {word:#010x}: {role}, {what})")
