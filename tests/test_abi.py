"""The C-ABI library: it loads, exports every symbol include/attn.h declares, and rejects bad
arguments on the host before any CUDA call. CPU only (no compute calls)."""
import ctypes
import os
import re
import subprocess

import pytest

import dense_attention_forward_gb300 as attn
from dense_attention_forward_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")

# Fake, never dereferenced device addresses (16-byte aligned, disjoint).
Q, K, V, O, L = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\s*\*)\s*(attn_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from dense_attention_forward_gb300 import build
        build.build()
    return _lib.lib()


def test_header_declares_the_boundary():
    assert declared_symbols() == ["attn_device_status", "attn_fwd", "attn_fwd_causal", "attn_fwd_ex",
                                  "attn_fwd_host", "attn_fwd_host_noalloc", "attn_fwd_strided",
                                  "attn_status_string", "attn_version"]


def test_product_library_exports_exactly_the_product_abi(lib):
    """libattn.so's dynamic symbol table holds the entry points of attn.h and no other attn_*
    function: the test hook and the trace calls live in their own builds."""
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm is not available")
    exported = sorted({ln.split()[-1] for ln in out.stdout.splitlines()
                       if ln.split() and ln.split()[-1].startswith("attn_")})
    assert exported == declared_symbols()


def test_test_hook_build_exports_both_headers(lib):
    from dense_attention_forward_gb300 import build
    hook_header = os.path.join(ROOT, "include", "attn_test_hooks.h")
    hook_syms = sorted(set(re.findall(r"^\s*int\s+(attn_\w+)\s*\(", open(hook_header).read(), re.M)))
    assert hook_syms == ["attn_fwd_withhold"] == sorted(_lib.TEST_HOOK_SIGNATURES)
    hl = ctypes.CDLL(build.build_test_hooks())
    for name in declared_symbols() + hook_syms:
        assert hasattr(hl, name), name
    assert not hasattr(lib, "attn_fwd_withhold")


def test_check_device_status_decodes_a_timeout_word(monkeypatch):
    # The binding's decoding of a non-zero status word (of the form the kernel writes when a
    # bounded wait runs out) into ATTN_ERR_TIMEOUT naming the role and the barrier.
    monkeypatch.setattr(_lib, "device_status", lambda reset=True: 0xA77E0000 | (3 << 8) | 7)
    with pytest.raises(attn.AttnError) as e:
        _lib.check_device_status()
    assert e.value.status == 6 and "softmax" in str(e.value) and "mbarrier 7" in str(e.value)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert set(declared_symbols()) == set(_lib.SIGNATURES)


def test_trace_build_exports_both_headers(lib):
    """libattn_trace.so (built on demand) exports attn.h and attn_trace.h; libattn.so does not
    export the trace entry points."""
    from dense_attention_forward_gb300 import build
    trace_header = os.path.join(ROOT, "include", "attn_trace.h")
    trace_syms = sorted(set(re.findall(r"^\s*int\s+(attn_\w+)\s*\(", open(trace_header).read(), re.M)))
    assert trace_syms == ["attn_trace_clear", "attn_trace_read"]
    tl = ctypes.CDLL(build.build_trace())
    for name in declared_symbols() + trace_syms:
        assert hasattr(tl, name), name
    for name in trace_syms:
        assert not hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.attn_version() >> 16 == 1
    for code in range(7):
        assert lib.attn_status_string(code).decode()
    assert lib.attn_status_string(99) == b"unknown status"


def call(lib, q=Q, k=K, v=V, o=O, lse=L, B=1, H=1, S=256, D=128, scale=0.088):
    return lib.attn_fwd(q, k, v, o, lse, B, H, S, D, scale, None)


@pytest.mark.parametrize("kw,expected", [
    (dict(D=64), 2), (dict(D=256), 2),
    (dict(q=None), 1), (dict(k=None), 1), (dict(v=None), 1), (dict(o=None), 1),
    (dict(B=0), 1), (dict(H=-1), 1), (dict(S=0), 1),
    (dict(scale=0.0), 1), (dict(scale=-0.1), 1), (dict(scale=float("inf")), 1),
    (dict(scale=float("nan")), 1),
    (dict(q=Q + 8), 3), (dict(o=O + 2), 3), (dict(lse=L + 2), 3),
    (dict(o=Q), 1), (dict(o=K + 256), 1), (dict(lse=O + 1024), 1), (dict(lse=V), 1),
    (dict(B=65536, H=65536), 1), (dict(B=1 << 20, H=1 << 10, S=4096), 1),
])
def test_argument_errors_are_reported_before_any_cuda_call(lib, kw, expected):
    assert call(lib, **kw) == expected


@pytest.mark.parametrize("thr,expected", [(2, 1), (-1, 1), (-8, 1), (16, 1), (7, 1)])
def test_bad_rebase_threshold(lib, thr, expected):
    assert lib.attn_fwd_ex(Q, K, V, O, L, 1, 1, 256, 128, 0.088, thr, None) == expected


def test_ex_validates_like_attn_fwd(lib):
    assert lib.attn_fwd_ex(Q, K, V, O, L, 1, 1, 256, 64, 0.088, 8, None) == 2
    assert lib.attn_fwd_ex(Q, K, V, Q, L, 1, 1, 256, 128, 0.088, 0, None) == 1


def strided(lib, qs, ks=None, vs=None, os_=None, B=2, H=3, S=256, q=Q, o=O, lse=L, causal=0):
    arr = ctypes.c_longlong * 3
    ks, vs, os_ = ks or qs, vs or qs, os_ or qs
    return lib.attn_fwd_strided(q, K, V, o, lse, B, H, S, 128, 0.088, arr(*qs), arr(*ks), arr(*vs),
                                arr(*os_), 0, causal, None)


BHSD = (3 * 256 * 128, 256 * 128, 128)
BSHD = (256 * 3 * 128, 128, 3 * 128)


@pytest.mark.parametrize("kw,expected", [
    (dict(qs=(0, 256 * 128, 128)), 1),                       # zero stride
    (dict(qs=(-1, 256 * 128, 128)), 1),                      # negative
    (dict(qs=(3 * 256 * 128, 256 * 128, 132)), 3),           # not a multiple of 16 bytes
    (dict(qs=BHSD, os_=(128, 128, 128)), 1),                 # output rows would collide
    (dict(qs=BHSD, os_=(256 * 128, 256 * 128, 128)), 1),     # batch and head overlap in o
    (dict(qs=BSHD, o=Q + 128 * 2), 1),                       # o inside q's span
    (dict(qs=BHSD, causal=2), 1),                            # causal is 0 or 1
    (dict(qs=BHSD, causal=-1), 1),
])
def test_strided_argument_errors(lib, kw, expected):
    assert strided(lib, **kw) == expected


def test_strided_null_strides(lib):
    arr = ctypes.c_longlong * 3
    assert lib.attn_fwd_strided(Q, K, V, O, L, 1, 1, 256, 128, 0.088, None, arr(*BHSD), arr(*BHSD),
                                arr(*BHSD), 0, 0, None) == 1


@pytest.mark.parametrize("kw,expected", [
    (dict(D=64), 2), (dict(q=None), 1), (dict(S=0), 1), (dict(scale=-1.0), 1), (dict(o=O + 2), 3),
    (dict(o=V), 1),
])
def test_causal_argument_errors(lib, kw, expected):
    a = dict(q=Q, k=K, v=V, o=O, lse=L, B=1, H=1, S=256, D=128, scale=0.088)
    a.update(kw)
    assert lib.attn_fwd_causal(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["S"], a["D"],
                               a["scale"], None) == expected


@pytest.mark.parametrize("S,token,expected", [
    (256, -1, 1), (256, -5, 1), (256, 4, 1), (300, 6, 1), (256, 3, 4), (300, 5, 4),
])
def test_withhold_token_range(S, token, expected):
    """The test hook accepts only a token the CTAs walk (2 per 128-key tile); a valid call
    reaches the device check, which fails here without a GPU."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    from dense_attention_forward_gb300 import build
    build.build_test_hooks()
    hl = _lib.test_hooks_lib()
    assert hl.attn_fwd_withhold(Q, K, V, O, L, 1, 1, S, 128, 0.088, token, None) == expected


# Fake host addresses (never dereferenced: every case fails before a copy is enqueued).
QH, KH, VH, OH, LH = 0x61000000, 0x62000000, 0x63000000, 0x64000000, 0x65000000


@pytest.mark.parametrize("kw,expected", [
    (dict(q_h=None), 1), (dict(k_h=None), 1), (dict(v_h=None), 1), (dict(o_h=None), 1),
    (dict(lse_h=None), 1), (dict(lse_d=None), 1), (dict(D=64), 2), (dict(S=0), 1), (dict(causal=2), 1),
    (dict(o_d=Q), 1), (dict(q_d=Q + 8), 3),
    # q_d, k_d, v_d are copy destinations: no two may overlap (256 rows x 256 B = 64 KB each)
    (dict(k_d=Q), 1), (dict(v_d=K), 1), (dict(v_d=Q + 65536 - 16), 1), (dict(k_d=V - 65536 + 16), 1),
])
def test_host_entry_argument_errors(lib, kw, expected):
    a = dict(q_h=QH, k_h=KH, v_h=VH, o_h=OH, lse_h=LH, q_d=Q, k_d=K, v_d=V, o_d=O, lse_d=L,
             B=1, H=1, S=256, D=128, scale=0.088, causal=0)
    a.update(kw)
    assert lib.attn_fwd_host(a["q_h"], a["k_h"], a["v_h"], a["o_h"], a["lse_h"], a["q_d"], a["k_d"], a["v_d"],
                             a["o_d"], a["lse_d"], a["B"], a["H"], a["S"], a["D"], a["scale"], a["causal"],
                             None) == expected


def test_host_entry_without_lse_and_without_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # Valid arguments reach the device check (nothing is enqueued without a GPU).
    assert lib.attn_fwd_host(QH, KH, VH, OH, None, Q, K, V, O, None, 1, 1, 256, 128, 0.088, 0, None) == 4
    # Adjacent (touching, not overlapping) device buffers are valid too.
    n = 256 * 128 * 2
    assert lib.attn_fwd_host(QH, KH, VH, OH, None, Q, Q + n, Q + 2 * n, O, None, 1, 1, 256, 128, 0.088, 0,
                             None) == 4


def test_no_device_is_reported(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call(lib) == 4  # ATTN_ERR_UNSUPPORTED_DEVICE, nothing launched
    assert lib.attn_fwd_causal(Q, K, V, O, L, 1, 1, 256, 128, 0.088, None) == 4
    word = ctypes.c_uint(7)
    assert lib.attn_device_status(ctypes.byref(word), 0) == 4
    assert lib.attn_device_status(None, 0) == 1


def test_status_check_without_a_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(attn.AttnError) as e:
        attn.check_device_status()
    assert e.value.status == 4  # the word cannot be read: ATTN_ERR_UNSUPPORTED_DEVICE


def test_python_wrapper_rejects_cpu_and_wrong_dtype():
    import torch
    x = torch.zeros(1, 1, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.fwd(x, x, x)
    y = torch.zeros(1, 1, 8, 128, dtype=torch.float32)
    with pytest.raises((TypeError, ValueError)):
        attn.fwd(y, y, y)


def test_fwd_host_rejects_bad_device_buffers():
    """fwd_host checks a caller-supplied dev tuple before any C call: count, shape, dtype,
    contiguity, then that the buffers are CUDA tensors."""
    import torch
    B, H, S, D = 1, 2, 40, 128
    q = torch.zeros(B, H, S, D, dtype=torch.bfloat16)
    good = [torch.empty(B, H, S, D, dtype=torch.bfloat16) for _ in range(4)] + [torch.empty(B, H, S)]
    bad = {
        "count": tuple(good[:4]),
        "shape": (torch.empty(B, H, S - 1, D, dtype=torch.bfloat16),) + tuple(good[1:]),
        "dtype": tuple(good[:3]) + (torch.empty(B, H, S, D),) + (good[4],),
        "lse shape": tuple(good[:4]) + (torch.empty(B, H, S + 1),),
        "contiguity": (torch.empty(B, S, H, D, dtype=torch.bfloat16).transpose(1, 2),) + tuple(good[1:]),
        "not cuda": tuple(good),
    }
    for what, dev in bad.items():
        with pytest.raises(ValueError):
            attn.fwd_host(q, q, q, out=torch.empty(B, H, S, D, dtype=torch.bfloat16),
                          lse=torch.empty(B, H, S), dev=dev)
