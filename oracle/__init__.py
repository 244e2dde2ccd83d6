"""fp64 CPU oracle of the Kimi Delta Attention (KDA) forward pass and its backward.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg import this package; the product path (the CUDA library and
its Python binding) never does, and shares no code with it.

The arithmetic lives in ``kda_oracle.c`` (plain fp64 C, see its header for the
passages each step follows).  This module only builds that file with gcc,
decodes the bf16 / fp32 input bits exactly into fp64, and marshals arrays.

Pins: every function here is pinned by ``tests/test_oracle_pins.py`` against
closed forms, brute force on tiny inputs, special cases and invariants; the
backward by ``tests/test_oracle_bwd_pins.py`` against central differences of the
forward.  ``chunked_bwd.py`` (numpy) holds the reverse mode in the chunked WY
form, pinned there against the token-level reverse mode.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lib = None

KD = 128


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into oracle/_build/liboracle.so (portable flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
           "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.kda_oracle_prep.restype = None
        lib.kda_oracle_prep.argtypes = [ctypes.c_int64, ctypes.c_int32] + [P] * 6 + [
            ctypes.c_double] + [P] * 4
        lib.kda_oracle_fwd.restype = ctypes.c_int
        lib.kda_oracle_fwd.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int32, P] + [
            P] * 7 + [ctypes.c_double, ctypes.c_double, P, P, P, ctypes.c_int32, ctypes.c_int32]
        lib.kda_oracle_bwd.restype = ctypes.c_int
        lib.kda_oracle_bwd.argtypes = ([ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                        ctypes.c_int32, P] + [P] * 7 +
                                       [ctypes.c_double, ctypes.c_double] + [P] * 11 +
                                       [ctypes.c_int32])
        _lib = lib
    return _lib


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 numbers given as their uint16 bit patterns."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_f64(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float64)


def _as_f64(x, name):
    a = np.asarray(x)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    if a.dtype == np.float32:
        return f32_to_f64(a)
    if a.dtype == np.float64:
        return np.ascontiguousarray(a)
    raise TypeError(f"{name}: expected uint16 (bf16 bits), float32 or float64, got {a.dtype}")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def prep(q, k, g, beta, A_log, dt_bias, lower_bound):
    """Elementwise prep. q,k,g: [tok,H,128]; beta: [tok,H].  Returns fp64
    (qn, kn, log_alpha, beta_sig) with the same shapes."""
    q, k, g, beta = (_as_f64(x, n) for x, n in ((q, "q"), (k, "k"), (g, "g"), (beta, "beta")))
    A_log, dt_bias = _as_f64(A_log, "A_log"), _as_f64(dt_bias, "dt_bias")
    n_tok, H = beta.shape
    qn, kn, la = (np.empty_like(q) for _ in range(3))
    bs = np.empty_like(beta)
    _load().kda_oracle_prep(n_tok, H, _ptr(q), _ptr(k), _ptr(g), _ptr(beta), _ptr(A_log),
                            _ptr(dt_bias), float(lower_bound), _ptr(qn), _ptr(kn), _ptr(la),
                            _ptr(bs))
    return qn, kn, la, bs


def fwd(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, initial_state=None,
        cu_seqlens=None, want_final=True, chunk=0, nthreads=None):
    """KDA forward in fp64.

    q, k: [B,T,HK,128] or packed [T_total,HK,128]; v, g: [B,T,H,128] or
    [T_total,H,128] (bf16 bits as uint16, float32 or float64), H a multiple of HK:
    value head h reads q/k head h // (H // HK) (grouped value heads; HK = H is
    the plain case); beta: [B,T,H] or [T_total,H]; A_log [H]; dt_bias [H,128];
    initial_state [N,H,V,K] (bf16 bits / fp32 / fp64) or None; cu_seqlens int64
    [N+1] (packed tokens, B must be 1) or None (then N = B, each of length T).
    chunk = 0 runs the token recurrence, chunk > 0 the chunked WY form.

    Returns (out fp64 with q's leading shape, final_state fp64 [N,H,V,K] or None,
    threads used).
    """
    qa = _as_f64(q, "q")
    lead = qa.shape[:-2]
    HK = qa.shape[-2]
    H = np.asarray(v).shape[-2]
    if qa.shape[-1] != KD:
        raise ValueError("head dim must be 128")
    if HK < 1 or H % HK != 0:
        raise ValueError("value heads must be a multiple of q/k heads")
    T_total = int(np.prod(lead))
    if cu_seqlens is None:
        if len(lead) == 2:
            B, T = lead
        else:
            B, T = 1, lead[0]
        cu = np.arange(0, B * T + 1, T if T > 0 else 1, dtype=np.int64)[: B + 1]
        if T == 0:
            cu = np.zeros(B + 1, dtype=np.int64)
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = len(cu) - 1
    if cu[0] != 0 or cu[-1] != T_total or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0, end at T_total and be non-decreasing")
    flat = lambda x, n, nh: _as_f64(x, n).reshape(T_total, nh, KD)
    qf, kf = flat(qa, "q", HK), flat(k, "k", HK)
    vf, gf = flat(v, "v", H), flat(g, "g", H)
    bf = _as_f64(beta, "beta").reshape(T_total, H)
    A = _as_f64(A_log, "A_log").reshape(H)
    dtb = _as_f64(dt_bias, "dt_bias").reshape(H, KD)
    init = None
    if initial_state is not None:
        init = _as_f64(initial_state, "initial_state").reshape(N, H, KD, KD)
    out = np.zeros((T_total, H, KD), dtype=np.float64)
    fin = np.zeros((N, H, KD, KD), dtype=np.float64) if want_final else None
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    used = _load().kda_oracle_fwd(T_total, H, HK, N, _ptr(cu), _ptr(qf), _ptr(kf), _ptr(vf),
                                  _ptr(gf), _ptr(bf), _ptr(A), _ptr(dtb), float(lower_bound),
                                  float(scale), _ptr(init), _ptr(out), _ptr(fin), int(chunk),
                                  int(nthreads))
    return out.reshape(*lead, H, KD), fin, used


def bwd(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale, dout, initial_state=None,
        dfinal_state=None, cu_seqlens=None, nthreads=None):
    """Reverse mode of :func:`fwd` in fp64: gradients of L = <dout, out> +
    <dfinal_state, final_state> with respect to every input.

    Inputs as for :func:`fwd`; dout has v's shape, dfinal_state the state shape
    [N, H, V, K] (None = zero).  Returns a dict with dq, dk (q's shape), dv, dg
    (v's shape), dbeta (beta's shape), dA_log [H], ddt_bias [H, 128] and
    dinitial_state [N, H, V, K] (the gradient with respect to the initial state,
    whether one was given or not)."""
    qa = _as_f64(q, "q")
    lead = qa.shape[:-2]
    HK = qa.shape[-2]
    H = np.asarray(v).shape[-2]
    if HK < 1 or H % HK != 0:
        raise ValueError("value heads must be a multiple of q/k heads")
    T_total = int(np.prod(lead))
    if cu_seqlens is None:
        B, T = (lead if len(lead) == 2 else (1, lead[0]))
        cu = np.arange(0, B * T + 1, T if T > 0 else 1, dtype=np.int64)[: B + 1]
        if T == 0:
            cu = np.zeros(B + 1, dtype=np.int64)
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = len(cu) - 1
    flat = lambda x, n, nh: _as_f64(x, n).reshape(T_total, nh, KD)
    qf, kf = flat(qa, "q", HK), flat(k, "k", HK)
    vf, gf = flat(v, "v", H), flat(g, "g", H)
    bf = _as_f64(beta, "beta").reshape(T_total, H)
    A = _as_f64(A_log, "A_log").reshape(H)
    dtb = _as_f64(dt_bias, "dt_bias").reshape(H, KD)
    do = flat(dout, "dout", H)
    init = None if initial_state is None else _as_f64(initial_state, "initial_state").reshape(N, H, KD, KD)
    dfin = None if dfinal_state is None else _as_f64(dfinal_state, "dfinal_state").reshape(N, H, KD, KD)
    dq, dk = np.zeros_like(qf), np.zeros_like(kf)
    dv, dg = np.zeros_like(vf), np.zeros_like(gf)
    dbeta = np.zeros_like(bf)
    dA, ddt = np.zeros(H), np.zeros((H, KD))
    dinit = np.zeros((N, H, KD, KD))
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    _load().kda_oracle_bwd(T_total, H, HK, N, _ptr(cu), _ptr(qf), _ptr(kf), _ptr(vf), _ptr(gf),
                           _ptr(bf), _ptr(A), _ptr(dtb), float(lower_bound), float(scale),
                           _ptr(init), _ptr(do), _ptr(dfin), _ptr(dq), _ptr(dk), _ptr(dv),
                           _ptr(dg), _ptr(dbeta), _ptr(dA), _ptr(ddt), _ptr(dinit), int(nthreads))
    shp = lambda x, nh: x.reshape(*lead, nh, KD)
    return {"dq": shp(dq, HK), "dk": shp(dk, HK), "dv": shp(dv, H), "dg": shp(dg, H),
            "dbeta": dbeta.reshape(*lead, H), "dA_log": dA, "ddt_bias": ddt,
            "dinitial_state": dinit}
