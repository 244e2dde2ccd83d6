"""Host-only checks of the C ABI: the library builds and loads, exports every
entry point include/kda.h declares, and rejects bad arguments with the right
status before anything reaches a GPU.  No kernel is launched here."""
import ctypes
import os
import re

import pytest

from kimi_delta_attention_08_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, NULLP, SHAPE, ARG, MISALIGNED, WS = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_entry_points():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", src)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_entry_points()
    assert set(_lib.EXPORTS) <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for s in range(0, 10):
        assert lib.kda_status_string(s)
    assert lib.kda_status_string(99) == b"unknown status"


def test_workspace_size(lib):
    n = ctypes.c_size_t(0)
    assert lib.kda_get_workspace_size(8 * 4096, 32, ctypes.byref(n)) == OK
    assert n.value >= 256
    small = n.value
    assert lib.kda_get_workspace_size(1 << 20, 64, ctypes.byref(n)) == OK and n.value >= small
    assert lib.kda_get_workspace_size(-1, 4, ctypes.byref(n)) == SHAPE
    assert lib.kda_get_workspace_size(10, -1, ctypes.byref(n)) == SHAPE
    assert lib.kda_get_workspace_size(10, 4, None) == NULLP


class FakeCall:
    """kda_fwd arguments with fake (never dereferenced) aligned device pointers."""

    def __init__(self, lib):
        self.lib = lib
        self.a = dict(q=0x10000, k=0x20000, v=0x30000, g=0x40000, beta=0x50000, scale=0.1,
                      out=0x60000, A_log=0x70000, dt_bias=0x80000, lower_bound=-5.0,
                      init=None, fin=None, cu=None, B=2, T=128, H=4, N=0, sdt=0,
                      ws=0x100000, ws_bytes=1 << 40, opts=None, stream=None)

    def __call__(self, **kw):
        a = dict(self.a, **kw)
        P = lambda x: None if x is None else ctypes.c_void_p(x)
        opts = a["opts"]
        return self.lib.kda_fwd(P(a["q"]), P(a["k"]), P(a["v"]), P(a["g"]), P(a["beta"]),
                                a["scale"], P(a["out"]), P(a["A_log"]), P(a["dt_bias"]),
                                a["lower_bound"], P(a["init"]), P(a["fin"]), P(a["cu"]),
                                a["B"], a["T"], a["H"], a["N"], a["sdt"], P(a["ws"]),
                                a["ws_bytes"], ctypes.byref(opts) if opts is not None else None,
                                P(a["stream"]))


def test_fwd_rejects_null_pointers(lib):
    call = FakeCall(lib)
    for nm in ("q", "k", "v", "g", "beta", "out", "A_log", "dt_bias", "ws"):
        assert call(**{nm: None}) == NULLP, nm


def test_fwd_rejects_bad_shapes(lib):
    call = FakeCall(lib)
    assert call(B=0) == SHAPE
    assert call(T=-1) == SHAPE
    assert call(H=0) == SHAPE
    assert call(cu=0x90000, B=2, N=3) == SHAPE          # varlen needs B == 1
    assert call(cu=0x90000, B=1, N=0) == SHAPE
    assert call(B=1, T=1 << 31) == SHAPE                # token coordinate range


def test_fwd_rejects_bad_args(lib):
    call = FakeCall(lib)
    assert call(lower_bound=0.1) == ARG                 # outside [-5, 0]
    assert call(lower_bound=-5.5) == ARG
    assert call(lower_bound=float("nan")) == ARG
    assert call(scale=float("inf")) == ARG
    assert call(sdt=2) == ARG
    o = _lib.kda_options()
    o.cp_mode = 7
    assert call(opts=o) == ARG
    o = _lib.kda_options()
    o.reserved[1] = 1
    assert call(opts=o) == ARG
    o = _lib.kda_options()
    o.debug_stall = 2                                   # only 0 or 1
    assert call(opts=o) == ARG
    o = _lib.kda_options()
    o.g_dtype = 2                                       # only bf16 (0) and fp32 (1)
    assert call(opts=o) == ARG
    o = _lib.kda_options()
    o.path = 3
    assert call(opts=o) == ARG


def test_fwd_rejects_misalignment(lib):
    call = FakeCall(lib)
    assert call(q=0x10008) == MISALIGNED
    assert call(out=0x60002) == MISALIGNED
    assert call(init=0x90004) == MISALIGNED
    assert call(ws=0x100040) == MISALIGNED             # workspace needs 128 B


def test_fwd_rejects_small_workspace(lib):
    call = FakeCall(lib)
    assert call(ws_bytes=16) == WS


def test_valid_call_without_gpu_does_not_succeed(lib):
    """With all host checks passed, the call needs a device: on a GPU-less host
    it reports a CUDA / device error instead of pretending to run."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert FakeCall(lib)() in (6, 7)


def test_fwd_grouped_value_heads_validation(lib):
    """num_v_heads must be 0 (= H) or a positive multiple of H, and the workspace
    is sized by the value heads."""
    call = FakeCall(lib)
    for hv, want in ((-4, SHAPE), (6, SHAPE), (2, SHAPE)):
        o = _lib.kda_options()
        o.num_v_heads = hv                              # H = 4
        assert call(opts=o) == want, hv
    n4, n16 = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.kda_get_workspace_size(2 * 128, 4, ctypes.byref(n4)) == OK
    assert lib.kda_get_workspace_size(2 * 128, 16, ctypes.byref(n16)) == OK
    o = _lib.kda_options()
    o.num_v_heads = 16
    assert call(opts=o, ws_bytes=n4.value) == WS or n16.value <= n4.value
    assert call(opts=o, ws_bytes=n16.value) != WS
