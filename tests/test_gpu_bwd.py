"""GPU parity of the token-by-token backward (kda_bwd, path "recurrent") against
the fp64 oracle's reverse mode (itself pinned by central differences of the
forward oracle), on the same input bits.  Tolerance: every gradient within BWD_TOL of the oracle's, relative
to that gradient's largest magnitude (fp32 recurrence over at most a few hundred
tokens here), and bitwise reproducibility."""
import numpy as np
import pytest

from kimi_delta_attention_08_gb300 import synth
from tests.kda_testutil import device_inputs, to_torch_bf16, to_torch_f32

import oracle

pytestmark = pytest.mark.gpu

BWD_TOL = 2e-5  # measured: <= 1.5e-6 on every case here (fp32 recurrence, fp64 oracle)
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias", "dinitial_state")


def cotangents(w, seed):
    """Seeded dout (bf16, out's shape) and dfinal (state dtype) for workload w."""
    HV = w.n_vheads
    dout = synth.normal_bf16((w.B, w.T, HV, 128), seed, 9)
    df = synth.normal_f32((w.N, HV, 128, 128), seed, 10)
    if w.state_dtype == "bf16":
        df = synth.f32_to_bf16_bits(df)
    return dout, df


def run_both(w, use_init=True, use_dfinal=True, seed=0):
    import kimi_delta_attention_08_gb300 as kda
    T = w.tensors
    dout, df = cotangents(w, seed)
    d = device_inputs(w)
    dd = to_torch_bf16(dout, "cuda")
    dfin = None
    if use_dfinal:
        dfin = to_torch_bf16(df, "cuda") if w.state_dtype == "bf16" else to_torch_f32(df, "cuda")
    g = kda.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, d["A_log"], d["dt_bias"],
                    w.lower_bound, dd, d["initial_state"] if use_init else None, dfin,
                    d["cu_seqlens"], path="recurrent")
    st = kda.kda_get_device_status(g["workspace"])
    assert st == 0, kda.status_string(st)
    ref = oracle.bwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"], T["dt_bias"],
                     w.lower_bound, w.scale, dout, T["initial_state"] if use_init else None,
                     df if use_dfinal else None, w.cu_seqlens)
    return g, ref


def check(w, **kw):
    g, ref = run_both(w, **kw)
    return compare(w.name, g, ref)


def compare(name, g, ref):
    errs = {}
    for nm in NAMES:
        got = g[nm].cpu().numpy().astype(np.float64).reshape(ref[nm].shape)
        assert np.all(np.isfinite(got)), f"{name} {nm}: non-finite"
        den = np.abs(ref[nm]).max()
        errs[nm] = float(np.abs(got - ref[nm]).max() / (den if den > 0 else 1.0))
    print(f"{name}: " + " ".join(f"{k} {v:.1e}" for k, v in errs.items()))
    bad = {k: v for k, v in errs.items() if v > BWD_TOL}
    assert not bad, f"{name}: {bad} (all: {errs})"
    return errs


@pytest.mark.parametrize("T", [1, 64, 150])
def test_bwd_batched(kda_lib, T):
    check(synth.make(f"bwd_T{T}", 2, T, 2, init="randn", lower_bound=-2.0, seed=80 + T))


def test_bwd_grouped_heads_varlen_fp32_gate_bf16_state(kda_lib):
    w = synth.make("bwd_gva", 1, 0, 1, HV=3, lengths=[7, 0, 70, 1], g_dtype="fp32",
                   state_dtype="bf16", init="randn", seed=90)
    check(w)


def test_bwd_no_states(kda_lib):
    check(synth.make("bwd_nostate", 2, 90, 2, init="none", seed=91), use_init=False,
          use_dfinal=False)


def test_bwd_slow_decay_default_bound(kda_lib):
    check(synth.make("bwd_lb5", 1, 130, 2, init="randn", lower_bound=-5.0, seed=92))


def test_bwd_no_decay_gives_zero_gate_gradients(kda_lib):
    """lower_bound = 0 makes alpha = 1 for every gate value: the gate, dt_bias and
    A_log gradients are exactly zero, the rest match the oracle."""
    import torch
    w = synth.make("bwd_lb0", 1, 80, 2, init="randn", lower_bound=0.0, seed=94)
    g, ref = run_both(w)
    compare(w.name, g, ref)
    for nm in ("dg", "dA_log", "ddt_bias"):
        assert int(torch.count_nonzero(g[nm])) == 0, nm


BF16_BITS = {100.0: 0x42C8, -100.0: 0xC2C8, 30.0: 0x41F0, -30.0: 0xC1F0}


def test_bwd_degenerate_rows(kda_lib):
    """Zero q and k rows (the l2 norm's reverse at r = 1 / sqrt(1e-6)), beta driven
    to 0 and 1 by the sigmoid, and gates saturated at both ends (log alpha =
    lower_bound = -5, and alpha = 1), across a block boundary; q and k rows
    scaled by 2^40 (the l2 norm removes the scale; its reverse divides by it)."""
    w = synth.make("bwd_degenerate", 1, 70, 2, init="randn", lower_bound=-5.0, seed=95)
    T = w.tensors
    T["q"][0, 5:9] = 0
    T["k"][0, 7:11] = 0
    big = np.float32(2.0 ** 40)
    for nm, rows in (("q", [14, 33]), ("k", [15, 33])):
        T[nm][0, rows] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(T[nm][0, rows]) * big)
    T["beta"][0, 12:16] = BF16_BITS[30.0]
    T["beta"][0, 16:18] = BF16_BITS[-30.0]
    T["g"][0, 20:40, 0] = BF16_BITS[100.0]    # head 0: saturated decay (alpha = e^-5)
    T["g"][0, 40:60, 1] = BF16_BITS[-100.0]   # head 1: no decay
    check(w)


@pytest.mark.parametrize("HV", [2, 4])
def test_bwd_deterministic(kda_lib, HV):
    import torch
    w = synth.make("bwd_det", 2, 100, 2, HV=HV, init="randn", seed=93)
    g1, _ = run_both(w)
    g2, _ = run_both(w)
    for nm in NAMES:
        assert torch.equal(g1[nm].view(torch.int32), g2[nm].view(torch.int32)), nm


def test_bwd_mid_size_whole_tensors(kda_lib):
    """B=4, T=2048, H=8 (64 units, more than one 16-token block per CTA pass):
    every gradient compared over the whole tensor."""
    check(synth.make("bwd_mid_B4_T2048_H8", 4, 2048, 8, init="randn", seed=96))


def test_bwd_full_size_sampled(kda_lib):
    """The benchmark's backward workload (B=8, T=4096, H=32, fp32 states) in the
    benchmark's launch configuration; the per-unit gradients of sampled (sequence,
    head) units against the oracle run on just that unit's tokens."""
    import kimi_delta_attention_08_gb300 as kda
    w = synth.prefill()
    T = w.tensors
    dout, df = cotangents(w, 5)
    d = device_inputs(w)
    g = kda.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, d["A_log"], d["dt_bias"],
                    w.lower_bound, to_torch_bf16(dout, "cuda"), d["initial_state"],
                    to_torch_f32(df, "cuda"), path="recurrent")
    assert kda.kda_get_device_status(g["workspace"]) == 0
    for n, h in [(0, 0), (3, 17), (7, 31)]:
        sl = lambda x: x[n:n + 1, :, h:h + 1]
        ref = oracle.bwd(sl(T["q"]), sl(T["k"]), sl(T["v"]), sl(T["g"]), T["beta"][n:n + 1, :, h:h + 1],
                         T["A_log"][h:h + 1], T["dt_bias"][h:h + 1], w.lower_bound, w.scale,
                         sl(dout), T["initial_state"][n:n + 1, h:h + 1], df[n:n + 1, h:h + 1])
        for nm in ("dq", "dk", "dv", "dg", "dbeta", "dinitial_state"):
            got = g[nm][n:n + 1, :, h:h + 1] if nm != "dinitial_state" else g[nm][n:n + 1, h:h + 1]
            got = got.cpu().numpy().astype(np.float64).reshape(ref[nm].shape)
            den = np.abs(ref[nm]).max()
            e = float(np.abs(got - ref[nm]).max() / (den if den > 0 else 1.0))
            print(f"unit {(n, h)} {nm}: {e:.1e}")
            assert e <= BWD_TOL, f"unit {(n, h)} {nm}: {e:.2e}"


@pytest.mark.parametrize("pattern", ["shared", "alternating"])
def test_bwd_adversarial_keys(kda_lib, pattern):
    """beta near 1 (logit 8), almost no decay (lower_bound = -0.001) and every
    token's key the same direction up to 1 % noise (or alternating in sign): the
    recurrence's most key-sensitive regime.  The backward runs in fp32 token by
    token and keeps its usual tolerance.  (Logits are kept off saturation: at
    sigmoid(30) fp32 gives exactly 1 and a zero beta gradient where the exact one
    is 1e-13 in scale, which a relative bound cannot judge.)"""
    w = synth.make(f"bwd_adv_{pattern}", 1, 150, 2, init="randn", lower_bound=-0.001, seed=96)
    T = w.tensors
    rng = np.random.default_rng(96)
    base = rng.standard_normal((1, 1, 2, 128))
    sign = (np.where(np.arange(150) % 2 == 0, 1.0, -1.0)[None, :, None, None]
            if pattern == "alternating" else 1.0)
    k = sign * base + 0.01 * rng.standard_normal((1, 150, 2, 128))
    T["k"] = synth.f32_to_bf16_bits(k.astype(np.float32))
    T["beta"][:] = np.uint16(0x4100)   # bf16 8.0
    check(w)
