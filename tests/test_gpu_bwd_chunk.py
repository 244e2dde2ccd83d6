"""GPU parity of the chunked tensor-core backward (kda_bwd, path "auto" /
"chunked") against the fp64 oracle's reverse mode (pinned by central differences
of the forward oracle), on the same input bits.  Tolerance: CHUNK_BWD_TOL of
tests/kda_testutil.py (bf16 MMA operands; the token-summed dA_log and dt_bias
gradients against their summed absolute per-token terms)."""
from types import SimpleNamespace

import numpy as np
import pytest

from kimi_delta_attention_08_gb300 import synth
from tests.kda_testutil import bwd_chunk_errors, device_inputs, to_torch_bf16, to_torch_f32

import oracle

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias", "dinitial_state")


def cotangents(w, seed):
    HV = w.n_vheads
    dout = synth.normal_bf16((w.B, w.T, HV, 128), seed, 9)
    df = synth.normal_f32((w.N, HV, 128, 128), seed, 10)
    if w.state_dtype == "bf16":
        df = synth.f32_to_bf16_bits(df)
    return dout, df


def run_chunked(w, use_init=True, use_dfinal=True, seed=0, path="chunked"):
    import kimi_delta_attention_08_gb300 as kda
    dout, df = cotangents(w, seed)
    d = device_inputs(w)
    dfin = None
    if use_dfinal:
        dfin = to_torch_bf16(df, "cuda") if w.state_dtype == "bf16" else to_torch_f32(df, "cuda")
    g = kda.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, d["A_log"], d["dt_bias"],
                    w.lower_bound, to_torch_bf16(dout, "cuda"),
                    d["initial_state"] if use_init else None, dfin, d["cu_seqlens"], path=path)
    st = kda.kda_get_device_status(g["workspace"])
    assert st == 0, kda.status_string(st)
    return g, dout, df


def oracle_bwd(w, dout, df, use_init=True, use_dfinal=True):
    T = w.tensors
    return oracle.bwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"], T["dt_bias"],
                      w.lower_bound, w.scale, dout, T["initial_state"] if use_init else None,
                      df if use_dfinal else None, w.cu_seqlens)


def check(w, use_init=True, use_dfinal=True, seed=0):
    g, dout, df = run_chunked(w, use_init, use_dfinal, seed)
    ref = oracle_bwd(w, dout, df, use_init, use_dfinal)
    got = {nm: g[nm].cpu().numpy() for nm in NAMES}
    errs, lim = bwd_chunk_errors(w, got, ref)
    print(f"{w.name}: " + " ".join(f"{k} {v:.1e}" for k, v in errs.items()))
    bad = {k: v for k, v in errs.items() if not v <= lim[k]}
    assert not bad, f"{w.name}: {bad} (all: {errs})"
    return g


@pytest.mark.parametrize("T", [1, 64, 150, 300])
def test_chunk_bwd_batched(kda_lib, T):
    """One chunk, an exact chunk, a ragged tail, several chunks."""
    check(synth.make(f"cbwd_T{T}", 2, T, 2, init="randn", lower_bound=-2.0, seed=80 + T))


@pytest.mark.parametrize("lb", [-5.0, -0.05])
def test_chunk_bwd_decay_range(kda_lib, lb):
    """The default bound (saturated gates decay by e^-5 per token: the pair factors
    span 2^+-115 around the reference points) and almost no decay."""
    check(synth.make(f"cbwd_lb{lb}", 2, 256, 2, init="randn", lower_bound=lb, seed=7))


def test_chunk_bwd_grouped_heads_varlen_fp32_gate_bf16_state(kda_lib):
    w = synth.make("cbwd_gva", 1, 0, 1, HV=3, lengths=[7, 0, 70, 1, 130], g_dtype="fp32",
                   state_dtype="bf16", init="randn", seed=90)
    check(w)


def test_chunk_bwd_no_states(kda_lib):
    check(synth.make("cbwd_nostate", 2, 90, 2, init="none", seed=91), use_init=False,
          use_dfinal=False)


def test_chunk_bwd_long_sequence_no_initial_state(kda_lib):
    check(synth.make("cbwd_T1000", 1, 1000, 2, init="none", seed=12), use_init=False)


def test_chunk_bwd_no_decay_gives_zero_gate_gradients(kda_lib):
    """lower_bound = 0: alpha = 1 for every gate value, and the gate, dt_bias and
    A_log gradients are exactly zero."""
    import torch
    w = synth.make("cbwd_lb0", 1, 150, 2, init="randn", lower_bound=0.0, seed=94)
    g = check(w)
    for nm in ("dg", "dA_log", "ddt_bias"):
        assert int(torch.count_nonzero(g[nm])) == 0, nm


BF16_BITS = {100.0: 0x42C8, -100.0: 0xC2C8, 30.0: 0x41F0, -30.0: 0xC1F0}


def test_chunk_bwd_degenerate_rows(kda_lib):
    """Zero q and k rows, beta driven to 0 and 1, gates saturated at both ends
    across a chunk boundary, and q / k rows scaled by 2^40."""
    w = synth.make("cbwd_degenerate", 1, 140, 2, init="randn", lower_bound=-5.0, seed=95)
    T = w.tensors
    T["q"][0, 5:9] = 0
    T["k"][0, 7:11] = 0
    big = np.float32(2.0 ** 40)
    for nm, rows in (("q", [14, 70]), ("k", [15, 70])):
        T[nm][0, rows] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(T[nm][0, rows]) * big)
    T["beta"][0, 12:16] = BF16_BITS[30.0]
    T["beta"][0, 16:18] = BF16_BITS[-30.0]
    T["g"][0, 40:90, 0] = BF16_BITS[100.0]    # head 0: saturated decay (alpha = e^-5)
    T["g"][0, 40:90, 1] = BF16_BITS[-100.0]   # head 1: no decay
    check(w)


@pytest.mark.parametrize("HV", [2, 4])
def test_chunk_bwd_deterministic(kda_lib, HV):
    import torch
    w = synth.make("cbwd_det", 2, 200, 2, HV=HV, init="randn", seed=93)
    g1, _, _ = run_chunked(w)
    g2, _, _ = run_chunked(w)
    for nm in NAMES:
        assert torch.equal(g1[nm].view(torch.int32), g2[nm].view(torch.int32)), nm


def test_chunk_bwd_auto_path_is_chunked(kda_lib):
    """The default path gives the chunked path's bits."""
    import torch
    w = synth.make("cbwd_auto", 1, 100, 2, init="randn", seed=97)
    g1, _, _ = run_chunked(w, path="chunked")
    g2, _, _ = run_chunked(w, path="auto")
    for nm in NAMES:
        assert torch.equal(g1[nm].view(torch.int32), g2[nm].view(torch.int32)), nm


def test_chunk_bwd_mid_size_whole_tensors(kda_lib):
    """B=4, T=2048, H=8: 32 chunks per unit, 32 units; every gradient over the
    whole tensor."""
    check(synth.make("cbwd_mid_B4_T2048_H8", 4, 2048, 8, init="randn", seed=96))


def test_chunk_bwd_full_size_sampled(kda_lib):
    """The benchmark's backward workload (B=8, T=4096, H=32, fp32 states) in the
    benchmark's launch configuration; sampled (sequence, head) units against the
    oracle run on just that unit's tokens."""
    import kimi_delta_attention_08_gb300 as kda
    w = synth.prefill()
    T = w.tensors
    dout, df = cotangents(w, 5)
    d = device_inputs(w)
    g = kda.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, d["A_log"], d["dt_bias"],
                    w.lower_bound, to_torch_bf16(dout, "cuda"), d["initial_state"],
                    to_torch_f32(df, "cuda"))
    assert kda.kda_get_device_status(g["workspace"]) == 0
    for n, h in [(0, 0), (3, 17), (7, 31)]:
        sl = lambda x: x[n:n + 1, :, h:h + 1]
        wu = SimpleNamespace(n_vheads=1, tensors={
            "q": sl(T["q"]), "k": sl(T["k"]), "v": sl(T["v"]), "g": sl(T["g"]),
            "beta": T["beta"][n:n + 1, :, h:h + 1], "A_log": T["A_log"][h:h + 1],
            "dt_bias": T["dt_bias"][h:h + 1], "initial_state": T["initial_state"][n:n + 1, h:h + 1]})
        ref = oracle.bwd(wu.tensors["q"], wu.tensors["k"], wu.tensors["v"], wu.tensors["g"],
                         wu.tensors["beta"], wu.tensors["A_log"], wu.tensors["dt_bias"],
                         w.lower_bound, w.scale, sl(dout), wu.tensors["initial_state"],
                         df[n:n + 1, h:h + 1])
        got = {}
        for nm in ("dq", "dk", "dv", "dg", "dbeta"):
            got[nm] = g[nm][n:n + 1, :, h:h + 1].cpu().numpy()
        got["dinitial_state"] = g["dinitial_state"][n:n + 1, h:h + 1].cpu().numpy()
        got["dA_log"], got["ddt_bias"] = ref["dA_log"], ref["ddt_bias"]  # sums over all units
        errs, lim = bwd_chunk_errors(wu, got, ref)
        print(f"unit {(n, h)}: " + " ".join(f"{k} {v:.1e}" for k, v in errs.items()))
        bad = {k: v for k, v in errs.items() if not v <= lim[k]}
        assert not bad, f"unit {(n, h)}: {bad}"


@pytest.mark.parametrize("what,e,gbits", [("v", 14, 0x42C8), ("v", 16, 0x42C8), ("init", 16, 0x42C8),
                                          ("v", 14, 0x4100)])
def test_chunk_bwd_large_values_saturated_decay(kda_lib, what, e, gbits):
    """Gates at (bf16 100: log alpha = lower_bound = -5 exactly) or near (bf16 8)
    saturation, so the pair products' decay factors span 2^+-115, with v or the
    initial state scaled by 2^e: the operand [dMq; dP] grows with the values, and
    only its power-of-two rescaling keeps those products inside fp32."""
    w = synth.make(f"cbwd_big_{what}{e}_{gbits:x}", 1, 192, 2, init="randn", lower_bound=-5.0,
                   seed=31)
    T = w.tensors
    T["g"][:] = np.uint16(gbits)
    if what == "v":
        T["v"] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(T["v"]) * np.float32(2.0 ** e))
    else:
        T["initial_state"] = (T["initial_state"] * np.float32(2.0 ** e)).astype(np.float32)
    check(w)


def test_chunk_bwd_irregular_varlen_whole_tensors(kda_lib):
    """The irregular varlen workload (H = 16; eight sequences of 1 .. 65,537 tokens,
    ragged last chunks, one of 1,025 chunks; bf16 states): every gradient over the
    whole tensor against the oracle."""
    check(synth.irregular_varlen())


# --------------------------------------------------- edge cases, both paths ----
@pytest.mark.parametrize("path", ["chunked", "recurrent"])
def test_bwd_bad_cu_seqlens_reported(kda_lib, path):
    """A cu_seqlens that runs backwards: the status word reports KDA_ERR_BAD_SEQLENS
    and the skipped unit adds nothing to the token-summed gradients."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    w = synth.make("cbwd_bad_cu", 1, 0, 2, lengths=[100, 50, 50], init="randn", seed=46)
    dout, df = cotangents(w, 46)
    d = device_inputs(w)
    cu = torch.tensor([0, 100, 60, 200], dtype=torch.int64, device="cuda")
    g = kda.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, d["A_log"], d["dt_bias"],
                    w.lower_bound, to_torch_bf16(dout, "cuda"), d["initial_state"],
                    to_torch_f32(df, "cuda"), cu, path=path)
    assert kda.kda_get_device_status(g["workspace"]) == 9          # KDA_ERR_BAD_SEQLENS
    assert bool(torch.isfinite(g["dA_log"]).all()) and bool(torch.isfinite(g["ddt_bias"]).all())


@pytest.mark.parametrize("path", ["chunked", "recurrent"])
@pytest.mark.parametrize("state_dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("varlen", [False, True])
def test_bwd_empty_input_passes_dfinal_through(kda_lib, path, state_dtype, varlen):
    """No tokens (T = 0, or one varlen sequence of length 0): dinitial_state is the
    final-state gradient, exactly, and the token-summed gradients are zero."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    if varlen:
        w = synth.make("cbwd_empty_varlen", 1, 0, 2, lengths=[0], init="randn",
                       state_dtype=state_dtype, seed=47)
    else:
        w = synth.make("cbwd_empty", 3, 0, 2, init="randn", state_dtype=state_dtype, seed=48)
    dout, df = cotangents(w, 47)
    d = device_inputs(w)
    dfin = to_torch_bf16(df, "cuda") if state_dtype == "bf16" else to_torch_f32(df, "cuda")
    g = kda.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, d["A_log"], d["dt_bias"],
                    w.lower_bound, to_torch_bf16(dout, "cuda"), d["initial_state"], dfin,
                    d["cu_seqlens"], path=path)
    assert kda.kda_get_device_status(g["workspace"]) == 0
    assert g["dq"].numel() == 0
    assert torch.equal(g["dinitial_state"], dfin.float())
    for nm in ("dA_log", "ddt_bias"):
        assert int(torch.count_nonzero(g[nm])) == 0, nm


# ------------------------------------ chunk start states from the forward ----
def fwd_with_states(w, d, **kw):
    import torch
    import kimi_delta_attention_08_gb300 as kda
    HV = w.n_vheads
    out = torch.full_like(d["v"], float("nan"))
    init = d["initial_state"]
    fin = None if init is None else torch.empty_like(init)
    ws = kda.make_workspace(w.B * w.T, HV)
    cs = kda.make_chunk_states(w.B * w.T, w.N, HV)
    kda.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, out, d["A_log"], d["dt_bias"],
                w.lower_bound, init, fin, d["cu_seqlens"], ws, chunk_states=cs, **kw)
    assert kda.kda_get_device_status(ws) == 0
    return out, fin, cs


def bwd_given(w, d, dout, df, cs):
    import kimi_delta_attention_08_gb300 as kda
    dfin = to_torch_bf16(df, "cuda") if w.state_dtype == "bf16" else to_torch_f32(df, "cuda")
    g = kda.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, d["A_log"], d["dt_bias"],
                    w.lower_bound, to_torch_bf16(dout, "cuda"), d["initial_state"], dfin,
                    d["cu_seqlens"], chunk_states=cs)
    assert kda.kda_get_device_status(g["workspace"]) == 0
    return g


@pytest.mark.parametrize("case", ["batched", "gva_varlen"])
def test_bwd_reads_forward_chunk_states(kda_lib, case):
    """A backward given the chunk states that the forward wrote gives the bits of
    the backward that runs its own state-checkpoint pass, and writing them leaves
    the forward's outputs unchanged."""
    import torch
    from tests.kda_testutil import run_gpu
    if case == "batched":
        w = synth.make("cbwd_cs", 2, 300, 2, init="randn", seed=71)
    else:
        w = synth.make("cbwd_cs_gva", 1, 0, 1, HV=3, lengths=[7, 0, 70, 1, 130], g_dtype="fp32",
                       state_dtype="bf16", init="randn", seed=72)
    d = device_inputs(w)
    out, fin, cs = fwd_with_states(w, d)
    out0, fin0 = run_gpu(w, inputs=d)
    assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
    dout, df = cotangents(w, 73)
    g1 = bwd_given(w, d, dout, df, cs)
    g2, _, _ = run_chunked(w, seed=73)
    for nm in NAMES:
        assert torch.equal(g1[nm].view(torch.int32), g2[nm].view(torch.int32)), nm


def test_bwd_reads_chunk_states_of_a_split_sequence(kda_lib):
    """The forward splits a 4,096-token sequence into segments (FORCE, 16 chunks
    each): every segment writes its chunks' start states, the later segments from
    their merged start states; the backward given them meets the oracle."""
    w = synth.make("cbwd_cs_split", 1, 4096, 2, init="randn", seed=74)
    d = device_inputs(w)
    _, _, cs = fwd_with_states(w, d, cp_mode="force", seg_chunks=16)
    dout, df = cotangents(w, 75)
    g = bwd_given(w, d, dout, df, cs)
    ref = oracle_bwd(w, dout, df)
    got = {nm: g[nm].cpu().numpy() for nm in NAMES}
    errs, lim = bwd_chunk_errors(w, got, ref)
    print(f"{w.name}: " + " ".join(f"{k} {v:.1e}" for k, v in errs.items()))
    bad = {k: v for k, v in errs.items() if not v <= lim[k]}
    assert not bad, f"{w.name}: {bad} (all: {errs})"


def test_bwd_reads_chunk_states_split_varlen_grouped_heads(kda_lib):
    """Chunk states written through a forced segment split of packed sequences with
    grouped value heads, an fp32 gate and bf16 states; the backward given them meets
    the oracle on whole tensors."""
    w = synth.make("cbwd_cs_split_gva", 1, 0, 1, HV=2, lengths=[5, 700, 0, 1300, 64],
                   g_dtype="fp32", state_dtype="bf16", init="randn", seed=76)
    d = device_inputs(w)
    _, _, cs = fwd_with_states(w, d, cp_mode="force", seg_chunks=4)
    dout, df = cotangents(w, 77)
    g = bwd_given(w, d, dout, df, cs)
    ref = oracle_bwd(w, dout, df)
    got = {nm: g[nm].cpu().numpy() for nm in NAMES}
    errs, lim = bwd_chunk_errors(w, got, ref)
    print(f"{w.name}: " + " ".join(f"{k} {v:.1e}" for k, v in errs.items()))
    bad = {k: v for k, v in errs.items() if not v <= lim[k]}
    assert not bad, f"{w.name}: {bad} (all: {errs})"
