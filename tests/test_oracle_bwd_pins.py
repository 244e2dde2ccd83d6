"""Pins of the fp64 oracle's backward pass against the forward oracle alone:
central finite differences of L = <dout, out> + <dfinal, final_state> along a
random direction of every input, compared with <gradient, direction>.  A dropped
term, a wrong sign or a transposed index anywhere in the reverse pass changes at
least one of these directional derivatives.  CPU only.

Cases: 70 tokens (crossing the backward's 64-token recomputation block), and
grouped value heads (HV = 3 per q/k head) over varlen sequences including an
empty one."""
import numpy as np
import pytest

import oracle
from kimi_delta_attention_08_gb300 import synth

KD = 128
INPUTS = ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state")
GRAD = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "A_log": "dA_log",
        "dt_bias": "ddt_bias", "initial_state": "dinitial_state"}


def as_f64(w):
    T = w.tensors
    x = {}
    for nm in INPUTS:
        a = T[nm]
        x[nm] = (oracle.bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64))
    return x


def loss(w, x, dout, dfin):
    out, fin, _ = oracle.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["A_log"],
                             x["dt_bias"], w.lower_bound, w.scale, x["initial_state"],
                             w.cu_seqlens)
    return float(np.sum(out * dout) + np.sum(fin * dfin))


@pytest.mark.parametrize("case", ["plain_T70", "grouped_varlen"])
def test_backward_matches_central_differences(case):
    if case == "plain_T70":
        w = synth.make("bwd_pin", 1, 70, 2, init="randn", lower_bound=-2.0, seed=71)
    else:
        w = synth.make("bwd_pin_gva", 1, 0, 1, HV=3, lengths=[7, 0, 13], init="randn",
                       lower_bound=-2.0, seed=72)
    x = as_f64(w)
    rng = np.random.default_rng(7)
    dout = rng.standard_normal(x["v"].shape)
    dfin = rng.standard_normal(x["initial_state"].shape)
    grads = oracle.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["A_log"], x["dt_bias"],
                       w.lower_bound, w.scale, dout, x["initial_state"], dfin, w.cu_seqlens)
    for nm in INPUTS:
        e = rng.standard_normal(x[nm].shape)
        step = 1e-5
        xp = dict(x); xp[nm] = x[nm] + step * e
        xm = dict(x); xm[nm] = x[nm] - step * e
        fd = (loss(w, xp, dout, dfin) - loss(w, xm, dout, dfin)) / (2 * step)
        an = float(np.sum(grads[GRAD[nm]].reshape(e.shape) * e))
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), f"{case} {nm}: fd {fd!r} vs grad {an!r}"


def test_backward_no_dout_no_dfinal_is_zero():
    """Zero cotangents give exactly zero gradients."""
    w = synth.make("bwd_zero", 1, 20, 1, init="randn", seed=73)
    x = as_f64(w)
    g = oracle.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["A_log"], x["dt_bias"],
                   w.lower_bound, w.scale, np.zeros(x["v"].shape), x["initial_state"])
    assert all(np.all(v == 0.0) for v in g.values())


# ------------------------------------------- chunked (WY-form) reverse mode --
@pytest.mark.parametrize("case,chunk", [("plain_T70", 1), ("plain_T70", 5), ("plain_T70", 16),
                                        ("plain_T70", 64), ("grouped_varlen", 16),
                                        ("saturated_C64", 64), ("no_decay", 16)])
def test_chunked_backward_matches_token_backward(case, chunk):
    """The chunked form of the reverse mode (oracle.chunked_bwd, the form a chunked
    tensor-core backward evaluates) against the token-level reverse mode, itself
    pinned by central differences above: every gradient to 1e-9 of its largest
    magnitude, for chunk lengths 1 to 64 (blocks crossing, and ragged at, the
    sequence ends), grouped value heads with an fp32 gate and a bf16 state over
    varlen sequences with an empty one, gates saturated at lower_bound = -5 with
    64-token blocks (decay factors to e^+-320 inside a block), and no decay."""
    from oracle.chunked_bwd import bwd_chunked
    if case == "plain_T70":
        w = synth.make("cbwd_pin", 2, 70, 2, init="randn", lower_bound=-2.0, seed=73)
    elif case == "grouped_varlen":
        w = synth.make("cbwd_pin_gva", 1, 0, 1, HV=3, lengths=[7, 0, 40, 1], init="randn",
                       g_dtype="fp32", state_dtype="bf16", lower_bound=-2.0, seed=74)
    elif case == "saturated_C64":
        w = synth.make("cbwd_pin_sat", 1, 130, 2, init="randn", lower_bound=-5.0, seed=75)
        w.tensors["g"][:] = np.uint16(0x42C8)          # bf16 100.0: log alpha = -5
    else:
        w = synth.make("cbwd_pin_nodecay", 1, 70, 2, init="randn", lower_bound=0.0, seed=76)
    T = w.tensors
    rng = np.random.default_rng(8)
    dout = rng.standard_normal(T["v"].shape)
    dfin = rng.standard_normal((w.N, w.HV, KD, KD))
    args = (T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"], T["dt_bias"], w.lower_bound,
            w.scale, dout, T["initial_state"], dfin, w.cu_seqlens)
    ref = oracle.bwd(*args)
    got = bwd_chunked(*args, chunk=chunk)
    for nm in GRAD.values():
        r = np.asarray(ref[nm], dtype=np.float64)
        gq = np.asarray(got[nm], dtype=np.float64).reshape(r.shape)
        den = np.abs(r).max()
        e = np.abs(gq - r).max() / (den if den > 0 else 1.0)
        assert e <= 1e-9, f"{case} C={chunk} {nm}: {e:.3e}"
