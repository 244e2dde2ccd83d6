"""GPU parity of the token-by-token path (decode steps and short prompts) against
the fp64 oracle, with the tolerances of the chunked path and, since every step
is fp32 here, a tighter state bound."""
import numpy as np
import pytest

from kimi_delta_attention_08_gb300 import synth
from tests.kda_testutil import OUT_TOL, STATE_TOL, compare, run_gpu

import oracle

pytestmark = pytest.mark.gpu

REC_STATE_TOL = 1e-4  # fp32 state, fp32 arithmetic throughout
# Outputs: each within one bf16 rounding of the fp64 value (half an ulp is at most
# 2^-8 of the value) plus fp32 noise of 1e-4 of the largest output.
REC_OUT_REL, REC_OUT_ABS = 2.0 ** -8, 1e-4


def out_rounding_ratio(out, ref_out):
    """max |out - ref| / (2^-8 |ref| + 1e-4 max|ref|) over all outputs: at most 1
    when every output is the bf16 rounding of the exact value, up to fp32 noise."""
    from tests.kda_testutil import bf16_tensor_to_f64
    o = bf16_tensor_to_f64(out).reshape(ref_out.shape)
    bound = REC_OUT_REL * np.abs(ref_out) + REC_OUT_ABS * np.abs(ref_out).max()
    return float((np.abs(o - ref_out) / bound).max())


def oracle_run(w, use_init=True):
    T = w.tensors
    out, fin, _ = oracle.fwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"], T["dt_bias"],
                             w.lower_bound, w.scale, T["initial_state"] if use_init else None,
                             w.cu_seqlens)
    return out, fin


def check(w, state_tol=STATE_TOL, **kw):
    out, fin = run_gpu(w, **kw)
    ref_out, ref_fin = oracle_run(w, kw.get("use_init", True))
    e_out, e_st = compare(out, fin, ref_out, ref_fin, label=w.name)
    assert e_out <= OUT_TOL, f"{w.name}: out max-rel error {e_out:.3e}"
    assert e_st <= state_tol, f"{w.name}: state rel-L2 error {e_st:.3e}"
    if kw.get("path") == "recurrent":
        r = out_rounding_ratio(out, ref_out)
        print(f"{w.name}: output error / bf16 rounding bound {r:.3f}")
        assert r <= 1.0, f"{w.name}: output beyond one bf16 rounding ({r:.3f} of the bound)"
    return e_out, e_st


@pytest.mark.parametrize("T", [1, 2, 7, 16, 17, 33])
def test_decode_batched(kda_lib, T):
    """The recurrent kernel on batched short input (one and several token blocks)."""
    w = synth.make(f"decode_T{T}", 24, T, 8, init="randn", seed=300 + T)
    check(w, path="recurrent", state_tol=REC_STATE_TOL)


@pytest.mark.parametrize("T", [1, 16, 17])
def test_decode_batched_auto(kda_lib, T):
    """AUTO picks a path by length; either meets the shared tolerances."""
    check(synth.make(f"decode_auto_T{T}", 24, T, 8, init="randn", seed=320 + T))


def test_decode_many_units_per_cta(kda_lib):
    """More (sequence, head) units than SMs: every persistent CTA walks several
    units through its double buffer."""
    w = synth.make("decode_many", 80, 3, 8, init="randn", seed=318)
    check(w, path="recurrent", state_tol=REC_STATE_TOL)


def test_decode_bf16_state(kda_lib):
    w = synth.make("decode_bf16", 16, 4, 8, init="randn", state_dtype="bf16", seed=311)
    check(w, path="recurrent")


def test_decode_no_initial_state(kda_lib):
    w = synth.make("decode_noinit", 8, 3, 4, init="randn", seed=312)
    check(w, use_init=False, path="recurrent", state_tol=REC_STATE_TOL)


def test_recurrent_forced_varlen(kda_lib):
    w = synth.make("rec_varlen", 1, 0, 4, lengths=[3, 0, 16, 40, 1, 130], init="randn", seed=313)
    check(w, path="recurrent", state_tol=REC_STATE_TOL)


def test_recurrent_forced_long_slow_decay(kda_lib):
    w = synth.make("rec_long", 2, 300, 4, init="randn", lower_bound=-0.01, seed=314)
    check(w, path="recurrent", state_tol=REC_STATE_TOL)


def test_recurrent_and_chunked_agree(kda_lib):
    import torch
    w = synth.make("rec_vs_chunk", 6, 16, 8, init="randn", seed=315)
    o_r, f_r = run_gpu(w, path="recurrent")
    o_c, f_c = run_gpu(w, path="chunked")
    ref_out, ref_fin = oracle_run(w)
    for o, f in ((o_r, f_r), (o_c, f_c)):
        e_out, e_st = compare(o, f, ref_out, ref_fin)
        assert e_out <= OUT_TOL and e_st <= STATE_TOL
    d = (o_r.float() - o_c.float()).abs().max().item() / max(float(np.abs(ref_out).max()), 1e-30)
    assert d <= 2 * OUT_TOL


def test_recurrent_beta_zero_exact(kda_lib):
    """beta = 0 (bf16 -inf logits) and no initial state: the state stays zero and
    every output is exactly zero."""
    w = synth.make("rec_beta0", 4, 5, 4, init="none", seed=316)
    w.tensors["beta"][:] = np.uint16(0xFF80)      # bf16 -inf -> beta = 0
    out, fin = run_gpu(w, path="recurrent")
    assert float(out.float().abs().max()) == 0.0 and float(fin.abs().max()) == 0.0


def test_recurrent_deterministic(kda_lib):
    import torch
    w = synth.make("rec_det", 32, 9, 8, init="randn", seed=317)
    o1, f1 = run_gpu(w, path="recurrent")
    o2, f2 = run_gpu(w, path="recurrent")
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(f1.view(torch.int32), f2.view(torch.int32))
