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
    assert lib.kda_get_workspace_size(1 << 31, 4, ctypes.byref(n)) == SHAPE   # kda_fwd's bound
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
    assert call(B=1 << 40, T=1 << 40) == SHAPE          # B * T would overflow int64
    assert call(B=1 << 31, T=0) == SHAPE


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


class FakeBwdCall:
    """kda_bwd arguments with fake (never dereferenced) aligned device pointers."""

    def __init__(self, lib):
        self.lib = lib
        self.a = dict(q=0x10000, k=0x20000, v=0x30000, g=0x40000, beta=0x50000, scale=0.1,
                      A_log=0x70000, dt_bias=0x80000, lower_bound=-5.0, init=None,
                      dout=0x60000, dfin=None, cu=None, dq=0x110000, dk=0x120000, dv=0x130000,
                      dg=0x140000, dbeta=0x150000, dA_log=0x160000, ddt_bias=0x170000,
                      dinit=None, B=2, T=128, H=4, N=0, sdt=0, ws=0x1000000, ws_bytes=1 << 40,
                      opts=None, stream=None)

    def __call__(self, **kw):
        a = dict(self.a, **kw)
        P = lambda x: None if x is None else ctypes.c_void_p(x)
        opts = a["opts"]
        return self.lib.kda_bwd(P(a["q"]), P(a["k"]), P(a["v"]), P(a["g"]), P(a["beta"]),
                                a["scale"], P(a["A_log"]), P(a["dt_bias"]), a["lower_bound"],
                                P(a["init"]), P(a["dout"]), P(a["dfin"]), P(a["cu"]), P(a["dq"]),
                                P(a["dk"]), P(a["dv"]), P(a["dg"]), P(a["dbeta"]),
                                P(a["dA_log"]), P(a["ddt_bias"]), P(a["dinit"]), a["B"], a["T"],
                                a["H"], a["N"], a["sdt"], P(a["ws"]), a["ws_bytes"],
                                ctypes.byref(opts) if opts is not None else None, P(a["stream"]))


def test_bwd_workspace_size(lib):
    """Grows with tokens and sequences, counts value heads, adds per-value-head dq /
    dk partials only for grouped heads; bad shapes and a null result are errors."""
    n = lambda T, N, H, HV: (lambda s: (lib.kda_bwd_get_workspace_size(T, N, H, HV, ctypes.byref(s)),
                                        s.value))(ctypes.c_size_t(0))
    st, base = n(8 * 4096, 8, 32, 0)
    assert st == OK and base > 8 * 4096 // 16 * 32 * 128 * 128 * 4   # checkpoints alone
    assert n(8 * 4096, 8, 32, 32) == (OK, base)                       # HV = H is the default
    assert n(2 * 8 * 4096, 16, 32, 0)[1] > base
    st, grouped = n(8 * 4096, 8, 16, 32)
    assert st == OK and grouped > base                                # + dq / dk partials
    assert n(0, 0, 4, 0)[0] == OK                                     # empty problem
    for bad in ((-1, 1, 4, 0), (10, -1, 4, 0), (10, 1, 0, 0), (10, 1, 4, -4), (10, 1, 4, 6),
                (1 << 31, 1, 4, 0)):
        assert n(*bad)[0] == SHAPE, bad
    assert lib.kda_bwd_get_workspace_size(10, 1, 4, 0, None) == NULLP


def test_bwd_rejects_null_pointers(lib):
    call = FakeBwdCall(lib)
    for nm in ("q", "k", "v", "g", "beta", "dout", "dq", "dk", "dv", "dg", "dbeta", "A_log",
               "dt_bias", "dA_log", "ddt_bias", "ws"):
        assert call(**{nm: None}) == NULLP, nm


def test_bwd_token_pointers_may_be_null_without_tokens(lib):
    """T = 0: the per-token tensors are not needed, so null passes the host checks
    (on a GPU-less host the call then stops at the device check)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    call = FakeBwdCall(lib)
    nulls = {nm: None for nm in ("q", "k", "v", "g", "beta", "dout", "dq", "dk", "dv", "dg",
                                 "dbeta")}
    assert call(T=0, **nulls) in (6, 7)


def test_bwd_rejects_bad_shapes_and_args(lib):
    call = FakeBwdCall(lib)
    assert call(B=0) == SHAPE
    assert call(T=-1) == SHAPE
    assert call(H=0) == SHAPE
    assert call(cu=0x90000, B=2, N=3) == SHAPE          # varlen needs B == 1
    assert call(cu=0x90000, B=1, N=0) == SHAPE
    assert call(B=1, T=1 << 31) == SHAPE
    assert call(B=1 << 40, T=1 << 40) == SHAPE          # B * T would overflow int64
    assert call(lower_bound=0.5) == ARG
    assert call(lower_bound=float("nan")) == ARG
    assert call(scale=float("nan")) == ARG
    assert call(sdt=3) == ARG
    for field, val, want in (("num_v_heads", 6, SHAPE), ("num_v_heads", -1, SHAPE),
                             ("g_dtype", 2, ARG), ("debug_stall", 2, ARG)):
        o = _lib.kda_options()
        setattr(o, field, val)
        assert call(opts=o) == want, (field, val)
    o = _lib.kda_options()
    o.reserved[0] = 1
    assert call(opts=o) == ARG
    o = _lib.kda_options()
    o.path, o.debug_stall = 2, 1                        # the stall hook is chunked-path only
    assert call(opts=o) == ARG


def test_bwd_rejects_misalignment_and_small_workspace(lib):
    call = FakeBwdCall(lib)
    assert call(dq=0x110004) == MISALIGNED             # fp32 gradients written as float4
    assert call(dg=0x140008) == MISALIGNED
    assert call(dinit=0x180004) == MISALIGNED
    assert call(dout=0x60002) == MISALIGNED
    assert call(ws=0x1000040) == MISALIGNED            # workspace needs 128 B
    assert call(q=0x10008) == MISALIGNED               # the chunked path's tensor maps: 16 B
    assert call(v=0x30008) == MISALIGNED
    o = _lib.kda_options()
    o.path = 2                                          # token by token: 8 B is enough
    assert call(q=0x10008, opts=o) != MISALIGNED
    need = ctypes.c_size_t(0)
    assert lib.kda_bwd_get_workspace_size(2 * 128, 2, 4, 0, ctypes.byref(need)) == OK
    assert call(ws_bytes=need.value - 1) == WS
    o = _lib.kda_options()
    o.num_v_heads = 8                                   # grouped heads need more
    assert call(opts=o, ws_bytes=need.value) == WS


# ------------------------------------------------------- chunk start states ----
def test_chunk_states_size(lib):
    n = ctypes.c_size_t(0)
    assert lib.kda_get_chunk_states_size(8 * 4096, 8, 32, ctypes.byref(n)) == OK
    assert n.value == (8 * 4096 // 64 + 2 * 8 + 1) * 32 * 128 * 128 * 2
    assert lib.kda_get_chunk_states_size(0, 1, 2, ctypes.byref(n)) == OK
    assert n.value == 3 * 2 * 128 * 128 * 2
    assert lib.kda_get_chunk_states_size(-1, 1, 2, ctypes.byref(n)) == SHAPE
    assert lib.kda_get_chunk_states_size(10, -1, 2, ctypes.byref(n)) == SHAPE
    assert lib.kda_get_chunk_states_size(1 << 31, 1, 2, ctypes.byref(n)) == SHAPE
    assert lib.kda_get_chunk_states_size(10, 1, 2, None) == NULLP


def _states_opts(lib, total, N, HV, path=0, addr=0x2000000, short=0):
    need = ctypes.c_size_t(0)
    assert lib.kda_get_chunk_states_size(total, N, HV, ctypes.byref(need)) == OK
    o = _lib.kda_options()
    o.path = path
    o.chunk_states = addr
    o.chunk_states_bytes = need.value - short
    return o


def test_fwd_chunk_states_checks(lib):
    """The forward writes chunk states on the chunked path only, into a buffer of
    at least kda_get_chunk_states_size bytes at a 16-byte boundary."""
    call = FakeCall(lib)
    assert call(opts=_states_opts(lib, 2 * 128, 2, 4, path=2)) == ARG
    assert call(opts=_states_opts(lib, 2 * 128, 2, 4, addr=0x2000008)) == MISALIGNED
    assert call(opts=_states_opts(lib, 2 * 128, 2, 4, short=1)) == WS
    o = _states_opts(lib, 2 * 128, 2, 4)
    assert call(opts=o) not in (ARG, MISALIGNED, WS)


def test_bwd_chunk_states_checks(lib):
    call = FakeBwdCall(lib)
    assert call(opts=_states_opts(lib, 2 * 128, 2, 4, path=2)) == ARG
    assert call(opts=_states_opts(lib, 2 * 128, 2, 4, addr=0x2000008)) == MISALIGNED
    assert call(opts=_states_opts(lib, 2 * 128, 2, 4, short=1)) == WS
    assert call(opts=_states_opts(lib, 2 * 128, 2, 4)) not in (ARG, MISALIGNED, WS)


def test_chunk_states_slot_bound(lib):
    """Every slot that the forward writes and the backward reads, floor(bos_n / 64)
    + 2n + c for chunk c of sequence n, lies below the slot count that
    kda_get_chunk_states_size provides, for random packed lengths (empty and
    one-token sequences included)."""
    import numpy as np
    rng = np.random.default_rng(5)
    HV = 3
    for trial in range(200):
        N = int(rng.integers(1, 40))
        lengths = rng.choice([0, 1, 2, 63, 64, 65, 127, 128, 129, 500, 4097], size=N)
        bos = np.concatenate([[0], np.cumsum(lengths)[:-1]])
        total = int(lengths.sum())
        n = ctypes.c_size_t(0)
        assert lib.kda_get_chunk_states_size(total, N, HV, ctypes.byref(n)) == OK
        slots = n.value // (HV * 128 * 128 * 2)
        for i, (b, L) in enumerate(zip(bos, lengths)):
            nch = (int(L) + 63) // 64
            if nch:
                assert int(b) // 64 + 2 * i + nch - 1 < slots, (trial, i)
