"""GPU parity: the CUDA path against the fp64 oracle, element by element, on the
same seeded inputs (tolerances: max|out-ref| <= 1e-2 max|ref|, final-state
relative L2 <= 5e-3)."""
import numpy as np
import pytest

from kimi_delta_attention_08_gb300 import synth
from tests.kda_testutil import OUT_TOL, STATE_TOL, compare, device_inputs, run_gpu

import oracle

pytestmark = pytest.mark.gpu


def oracle_run(w, use_init=True):
    T = w.tensors
    out, fin, _ = oracle.fwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"], T["dt_bias"],
                             w.lower_bound, w.scale, T["initial_state"] if use_init else None,
                             w.cu_seqlens)
    return out, fin


def check(w, label=None, **kw):
    out, fin = run_gpu(w, **kw)
    ref_out, ref_fin = oracle_run(w, kw.get("use_init", True))
    e_out, e_st = compare(out, fin, ref_out, ref_fin, label=label or w.name)
    assert e_out <= OUT_TOL, f"{w.name}: out max-rel error {e_out:.3e}"
    assert e_st <= STATE_TOL, f"{w.name}: state rel-L2 error {e_st:.3e}"
    return e_out, e_st


def test_tiny_ref(kda_lib):
    check(synth.tiny_ref())


def test_batched_small(kda_lib):
    check(synth.batched_small())


@pytest.mark.parametrize("T", [1, 17, 63, 64, 65, 130, 333])
def test_ragged_lengths(kda_lib, T):
    check(synth.make(f"ragged_T{T}", 1, T, 3, init="randn", seed=100 + T))


def test_varlen_small(kda_lib):
    w = synth.make("varlen_small", 1, 0, 4, lengths=[5, 0, 64, 130, 1, 77], init="randn",
                   state_dtype="bf16", seed=7)
    check(w)


# ---------------------------------------------------------------- states ----
@pytest.mark.parametrize("use_init,final", [(True, True), (True, False), (False, True),
                                             (False, False)])
def test_state_presence_combinations(kda_lib, use_init, final):
    """Either state may be present without the other."""
    w = synth.make("states", 1, 200, 2, init="randn", seed=31)
    out, fin = run_gpu(w, use_init=use_init, final=final)
    ref_out, ref_fin = oracle_run(w, use_init=use_init)
    e_out, e_st = compare(out, fin, ref_out, ref_fin if final else None)
    assert e_out <= OUT_TOL and e_st <= STATE_TOL
    assert (fin is None) == (not final)


def test_bf16_state_batched(kda_lib):
    check(synth.make("bf16_state", 2, 300, 4, init="randn", state_dtype="bf16", seed=32))


# -------------------------------------------------------- special inputs ----
def test_beta_zero_gives_exact_zero(kda_lib):
    w = synth.make("beta0", 2, 130, 3, init="none", seed=33)
    w.tensors["beta"][:] = np.uint16(0xFF80)      # bf16 -inf -> beta = 0
    out, fin = run_gpu(w)
    assert float(out.float().abs().max()) == 0.0 and float(fin.abs().max()) == 0.0


def test_alpha_one(kda_lib):
    check(synth.make("alpha1", 1, 256, 2, init="randn", lower_bound=0.0, seed=34))


def test_slow_decay(kda_lib):
    """lower_bound -0.01: memory spans thousands of tokens, so long-range state
    error is exercised (not a published workload)."""
    check(synth.make("slow_decay", 1, 2048, 4, init="randn", lower_bound=-0.01, seed=35))


def test_deterministic_bitwise(kda_lib):
    import torch
    w = synth.make("determinism", 2, 640, 8, init="randn", seed=36)
    o1, f1 = run_gpu(w)
    o2, f2 = run_gpu(w)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(f1.view(torch.int32), f2.view(torch.int32))


# ------------------------------------------------- full-size workloads ----
# The three large workloads, each in the launch configuration the benchmark uses,
# compared with the oracle over the whole output and the whole final state.

def test_prefill_full_size(kda_lib):
    """B=8, T=4096, H=32, fp32 state, zero initial state passed explicitly."""
    w = synth.prefill()
    check(w, label=f"full:{w.name}")


@pytest.mark.parametrize("cp_mode", ["auto", "off"])
def test_irregular_varlen_full_size(kda_lib, cp_mode):
    """H=16, eight sequences of 1 .. 65,537 tokens, bf16 states."""
    w = synth.irregular_varlen()
    check(w, label=f"full:{w.name} cp={cp_mode}", cp_mode=cp_mode)


@pytest.mark.parametrize("cp_mode", ["auto", "off"])
def test_long_sequence_full_size(kda_lib, cp_mode):
    """H=8, 65,536 + 5 x 1,024 tokens, fp32 states; AUTO splits the long sequence."""
    w = synth.long_sequence()
    check(w, label=f"full:{w.name} cp={cp_mode}", cp_mode=cp_mode)


# ----------------------------------------------------- state hand-off ----
@pytest.mark.parametrize("state_dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("cp_mode,seg_chunks", [("off", 0), ("force", 2)])
def test_state_handoff_matches_one_run(kda_lib, state_dtype, cp_mode, seg_chunks):
    """Checkpoint / resume: [0, T1) with the kernel's own final state fed as the
    initial state of [T1, T), against the oracle's single run over [0, T)."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    from tests.kda_testutil import device_inputs
    w = synth.make(f"handoff_{state_dtype}_{cp_mode}", 2, 1000, 4, init="randn",
                   state_dtype=state_dtype, seed=47)
    d = device_inputs(w)
    T1 = 437                                  # ragged on both sides of the split
    sdt = torch.bfloat16 if state_dtype == "bf16" else torch.float32
    outs, state = [], d["initial_state"]
    for lo, hi in ((0, T1), (T1, w.T)):
        part = {nm: (d[nm][:, lo:hi].contiguous() if nm in ("q", "k", "v", "g", "beta") else d[nm])
                for nm in d}
        out = torch.full_like(part["v"], float("nan"))
        fin = torch.full((w.N, w.H, 128, 128), float("nan"), dtype=sdt, device="cuda")
        ws = kda.make_workspace(w.B * (hi - lo), w.H)
        kda.kda_fwd(part["q"], part["k"], part["v"], part["g"], part["beta"], w.scale, out,
                    part["A_log"], part["dt_bias"], w.lower_bound, state, fin, None, ws,
                    cp_mode=cp_mode, seg_chunks=seg_chunks, path="chunked")
        assert kda.kda_get_device_status(ws) == 0
        outs.append(out)
        state = fin
    out = torch.cat(outs, dim=1)
    ref_out, ref_fin = oracle_run(w)
    e_out, e_st = compare(out, state, ref_out, ref_fin, label=w.name)
    assert e_out <= OUT_TOL, f"{w.name}: out max-rel error {e_out:.3e}"
    assert e_st <= STATE_TOL, f"{w.name}: state rel-L2 error {e_st:.3e}"


# ------------------------------------------------------ segment scan (CP) ----
@pytest.mark.parametrize("seg_chunks", [1, 2, 3])
def test_segment_scan_forced_small(kda_lib, seg_chunks):
    """Every sequence with >= 2 chunks is split into segments of seg_chunks chunks:
    prescan (M_s, B_s), merge, rerun.  Same tolerances as the serial path."""
    w = synth.make("cp_small", 1, 0, 3, lengths=[300, 1, 520, 64, 0, 200], init="randn",
                   seed=41)
    check(w, cp_mode="force", seg_chunks=seg_chunks)


def test_segment_scan_slow_decay(kda_lib):
    w = synth.make("cp_slow", 1, 0, 2, lengths=[1500, 700], init="randn", lower_bound=-0.05,
                   seed=42)
    check(w, cp_mode="force", seg_chunks=4)


def test_segment_scan_matches_serial(kda_lib):
    import torch
    w = synth.make("cp_vs_serial", 2, 1024, 4, init="randn", seed=43)
    o_ser, f_ser = run_gpu(w, cp_mode="off")
    o_cp, f_cp = run_gpu(w, cp_mode="force", seg_chunks=3)
    ref_o, ref_f = oracle_run(w)
    for o, f in ((o_ser, f_ser), (o_cp, f_cp)):
        e_out, e_st = compare(o, f, ref_o, ref_f)
        assert e_out <= OUT_TOL and e_st <= STATE_TOL
    diff = (o_ser.float() - o_cp.float()).abs().max().item()
    assert diff <= 2 * OUT_TOL * float(np.abs(ref_o).max())


def test_segment_scan_deterministic(kda_lib):
    import torch
    w = synth.make("cp_det", 1, 0, 4, lengths=[2000, 37, 900], init="randn", seed=44)
    o1, f1 = run_gpu(w, cp_mode="force", seg_chunks=5)
    o2, f2 = run_gpu(w, cp_mode="force", seg_chunks=5)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(f1.view(torch.int32), f2.view(torch.int32))


def test_bad_cu_seqlens_reported(kda_lib):
    import torch
    import kimi_delta_attention_08_gb300 as kda
    from tests.kda_testutil import device_inputs
    w = synth.make("bad_cu", 1, 0, 2, lengths=[100, 50, 50], seed=45)
    d = device_inputs(w)
    d["cu_seqlens"] = torch.tensor([0, 100, 60, 200], dtype=torch.int64, device="cuda")
    out = torch.zeros_like(d["q"])
    ws = kda.make_workspace(200, w.H)
    kda.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, out, d["A_log"],
                d["dt_bias"], w.lower_bound, None, None, d["cu_seqlens"], ws)
    assert kda.kda_get_device_status(ws) == 9          # KDA_ERR_BAD_SEQLENS
    assert float(out.float().abs().max()) == 0.0       # nothing was written


# ----------------------------------------------------------- extreme gates ----
BF16_100 = np.uint16(0x42C8)        # bf16 100.0
BF16_M100 = np.uint16(0xC2C8)       # bf16 -100.0


@pytest.mark.parametrize("path", ["chunked", "recurrent"])
def test_saturated_gates(kda_lib, path):
    """Every gate at lower_bound = -5 (sigmoid(exp(A_log)(100 + dt_bias)) = 1): the
    in-chunk decay factors span about 2^+-115 around the reference points and the
    state decays by e^-5 per token."""
    w = synth.make("gates_saturated", 2, 200, 4, init="randn", seed=61)
    w.tensors["g"][:] = BF16_100
    check(w, path=path)


@pytest.mark.parametrize("path", ["chunked", "recurrent"])
def test_mixed_extreme_gates(kda_lib, path):
    """Even channels decay at e^-5 per token, odd channels not at all (g = -100
    gives sigmoid 0, alpha = 1): per-channel decay ranges as far apart as the gate
    allows, in one tile."""
    w = synth.make("gates_mixed", 2, 200, 4, init="randn", seed=62)
    g = w.tensors["g"]
    g[..., 0::2] = BF16_100
    g[..., 1::2] = BF16_M100
    check(w, path=path)


# ------------------------------------------------------------- empty input ----
@pytest.mark.parametrize("path", ["chunked", "recurrent"])
@pytest.mark.parametrize("state_dtype", ["fp32", "bf16"])
def test_empty_batch_keeps_initial_state(kda_lib, path, state_dtype):
    """T = 0: the token tensors are empty (NULL data pointers) and the final state
    equals the initial state bit for bit."""
    import torch
    from tests.kda_testutil import device_inputs
    w = synth.make("empty", 3, 0, 4, init="randn", state_dtype=state_dtype, seed=63)
    d = device_inputs(w)
    out, fin = run_gpu(w, inputs=d, path=path)
    assert out.numel() == 0
    bits = torch.int16 if state_dtype == "bf16" else torch.int32
    assert torch.equal(fin.view(bits), d["initial_state"].view(bits))


def test_varlen_only_empty_sequence(kda_lib):
    import torch
    from tests.kda_testutil import device_inputs
    w = synth.make("empty_varlen", 1, 0, 2, lengths=[0], init="randn", seed=64)
    d = device_inputs(w)
    out, fin = run_gpu(w, inputs=d)
    assert torch.equal(fin.view(torch.int32), d["initial_state"].view(torch.int32))


# ----------------------------------------------- large-magnitude values ----
@pytest.mark.parametrize("path", ["chunked", "recurrent"])
@pytest.mark.parametrize("log2_scale", [10, 14, 16])
def test_large_values_saturated_gates(kda_lib, path, log2_scale):
    """Every gate saturated at lower_bound = -5 (the in-chunk decay factors then
    span the widest range the gate allows) with v and the initial state scaled by
    2^10, 2^14 and 2^16: the products of the state update must not overflow fp32.
    The scaling is exact in bf16 and fp32, and the tolerances are relative."""
    w = synth.make(f"large_v_2^{log2_scale}_{path}", 2, 200, 4, init="randn", seed=65)
    Tn = w.tensors
    f = np.float32(2.0 ** log2_scale)
    Tn["v"] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(Tn["v"]) * f)
    Tn["initial_state"] = Tn["initial_state"] * f
    Tn["g"][:] = BF16_100
    check(w, path=path)


# --------------------------------------------------------- degenerate rows ----
@pytest.mark.parametrize("path", ["chunked", "recurrent"])
def test_degenerate_rows(kda_lib, path):
    """Rows the preprocessing has to survive, across a chunk boundary: q and k rows
    of zeros (the l2 norm maps them to zero), beta driven to exactly 0 and 1 (bf16
    -inf / +inf logits), and q, k rows scaled by 2^40 (the l2 norm removes the
    scale; the scaling is exact in bf16)."""
    w = synth.make("degenerate_rows", 2, 150, 4, init="randn", seed=66)
    Tn = w.tensors
    q, k, beta = Tn["q"], Tn["k"], Tn["beta"]
    q[:, [5, 62, 63, 64]] = 0
    k[:, [5, 63, 64, 65, 127]] = 0
    beta[:, [10, 64, 100]] = np.uint16(0xFF80)     # -inf -> beta = 0
    beta[:, [11, 65, 101]] = np.uint16(0x7F80)     # +inf -> beta = 1
    big = np.float32(2.0 ** 40)
    for x, rows in ((q, [20, 66, 130]), (k, [21, 66, 131])):
        x[:, rows] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(x[:, rows]) * big)
    check(w, path=path)


# ----------------------------------------------------------- planner limits ----
@pytest.mark.parametrize("path", ["chunked", "auto"])
def test_varlen_many_short_sequences(kda_lib, path):
    """400 packed sequences of 0 to 9 tokens (many empty or single-token): the
    device planner's unit tables and longest-first order over 1,200 units."""
    lengths = [int(x) for x in np.random.default_rng(67).integers(0, 10, size=400)]
    w = synth.make("varlen_many_short", 1, 0, 3, lengths=lengths, init="randn", seed=67)
    check(w, path=path)


@pytest.mark.parametrize("cp_mode", ["auto", "off"])
def test_segment_cap_doubles_segment_length(kda_lib, cp_mode):
    """Nine sequences of 4,096 tokens with H = 8: the automatic split wants 4
    segments of 16 chunks each, 288 segment-heads, above the planner's cap of 256,
    so it doubles the segment length (2 segments each).  Same tolerances with and
    without the split."""
    w = synth.make("segment_cap", 1, 0, 8, lengths=[4096] * 9, init="randn", seed=68)
    check(w, label=f"{w.name} cp={cp_mode}", cp_mode=cp_mode)


# ------------------------------------------------------ adversarial keys ----
def _adversarial_keys(pattern):
    w = synth.make(f"adv_keys_{pattern}", 2, 200, 3, init="randn", seed=69)
    Tn = w.tensors
    rng = np.random.default_rng(69)
    B_, T_, H_ = w.B, w.T, w.H
    base = rng.standard_normal((B_, 1, H_, 128))
    if pattern == "shared":
        k = base + 0.01 * rng.standard_normal((B_, T_, H_, 128))
    elif pattern == "alternating":
        sign = np.where(np.arange(T_) % 2 == 0, 1.0, -1.0)[None, :, None, None]
        k = sign * base + 0.01 * rng.standard_normal((B_, T_, H_, 128))
    else:
        other = rng.standard_normal((B_, 1, H_, 128))
        c = rng.standard_normal((B_, T_, H_, 2))
        k = c[..., :1] * base + c[..., 1:] * other
    Tn["k"] = synth.f32_to_bf16_bits(k.astype(np.float32))
    Tn["beta"][:] = np.uint16(0x41F0)   # bf16 30.0: beta = sigmoid(30) ~ 1
    Tn["g"][:] = BF16_M100              # alpha = 1
    return w


def _bf16_key_sensitivity(w):
    """The error the bf16 representation of the normalized keys alone causes: the
    fp64 oracle on keys replaced by bf16(k / sqrt(|k|^2 + 1e-6)) against the oracle
    on the exact keys (max-rel out, rel-L2 state).  Computed by the oracle only."""
    T = w.tensors
    args = (T["v"], T["g"], T["beta"], T["A_log"], T["dt_bias"], w.lower_bound, w.scale,
            T["initial_state"])
    o0, s0, _ = oracle.fwd(T["q"], T["k"], *args)
    k = synth.bf16_bits_to_f32(T["k"]).astype(np.float64)
    kb = synth.f32_to_bf16_bits((k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)).astype(np.float32))
    o1, s1, _ = oracle.fwd(T["q"], kb, *args)
    return (float(np.abs(o1 - o0).max() / np.abs(o0).max()),
            float(np.linalg.norm(s1 - s0) / np.linalg.norm(s0)))


@pytest.mark.parametrize("pattern", ["shared", "alternating", "rank2"])
@pytest.mark.parametrize("path", ["chunked", "recurrent"])
def test_adversarial_keys(kda_lib, pattern, path):
    """Keys that make the recurrence as sensitive to the keys as it gets: beta = 1
    (logit 30), no decay (g = -100), and every token's key the same direction up to
    1 % noise, alternating between a direction and its negative, or drawn from a
    two-dimensional subspace.  Each step then projects the state onto nearly the
    same hyperplane, and a key perturbation of relative size eps moves the outputs
    by a growing multiple of eps.

    The token-by-token path keeps the normalized keys in fp32 and meets the usual
    tolerances.  The chunked path forms its key products from bf16 normalized keys
    (relative rounding 2^-9, as any bf16 tensor-core formulation of the chunked form
    does); that representation alone, fed to the fp64 oracle, moves the outputs by
    about 1e-2 and the state by about 2e-2 here.  The chunked path is held to the
    usual tolerances plus 1.5 times that oracle-measured sensitivity."""
    w = _adversarial_keys(pattern)
    if path == "recurrent":
        check(w, path=path)
        return
    sens_out, sens_st = _bf16_key_sensitivity(w)
    out, fin = run_gpu(w, path=path)
    ref_out, ref_fin = oracle_run(w)
    # not in the run's summary of margins, which holds every case to the usual bar
    e_out, e_st = compare(out, fin, ref_out, ref_fin)
    print(f"{w.name} (chunked): out {e_out:.2e} state {e_st:.2e}; bf16-key sensitivity "
          f"out {sens_out:.2e} state {sens_st:.2e}")
    assert e_out <= OUT_TOL + 1.5 * sens_out, (e_out, sens_out)
    assert e_st <= STATE_TOL + 1.5 * sens_st, (e_st, sens_st)


@pytest.mark.parametrize("path", ["chunked", "recurrent"])
def test_beta_one_no_decay_long(kda_lib, path):
    """beta = 1 and no decay over 2,000 tokens with random keys: the state is
    rewritten along a new key every token and nothing fades, the regime with the
    longest memory.  Random keys keep the recurrence well conditioned (the bf16
    key representation alone moves the oracle by under 3e-3), so the usual
    tolerances apply."""
    w = synth.make("beta1_nodecay", 1, 2000, 2, init="randn", seed=5)
    w.tensors["beta"][:] = np.uint16(0x41F0)   # bf16 30.0: beta ~ 1
    w.tensors["g"][:] = BF16_M100              # alpha = 1
    check(w, path=path)


# ---------------------------------------------------------- in-place state ----
@pytest.mark.parametrize("case,path,cp_mode", [("batched", "chunked", "auto"),
                                               ("varlen", "chunked", "force"),
                                               ("batched", "recurrent", "auto")])
@pytest.mark.parametrize("state_dtype", ["fp32", "bf16"])
def test_state_updated_in_place(kda_lib, case, path, cp_mode, state_dtype):
    """final_state may be the initial_state buffer itself (a streaming caller
    updating its state in place): every unit reads its initial state before it
    writes its final state, and with the segment scan the initial state is read
    in the prescan launch only.  Same bits as with separate buffers."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    if case == "batched":
        w = synth.make(f"inplace_{case}", 3, 300, 4, init="randn", state_dtype=state_dtype, seed=75)
    else:
        w = synth.make(f"inplace_{case}", 1, 0, 3, lengths=[900, 0, 1, 300], init="randn",
                       state_dtype=state_dtype, seed=75)
    d = device_inputs(w)
    ws = kda.make_workspace(w.B * w.T, w.HV)
    ref_out = torch.empty_like(d["v"])
    ref_fin = torch.empty_like(d["initial_state"])
    kda.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, ref_out, d["A_log"],
                d["dt_bias"], w.lower_bound, d["initial_state"], ref_fin, d["cu_seqlens"], ws,
                cp_mode=cp_mode, path=path)
    state = d["initial_state"].clone()
    out = torch.empty_like(d["v"])
    kda.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, out, d["A_log"],
                d["dt_bias"], w.lower_bound, state, state, d["cu_seqlens"], ws,
                cp_mode=cp_mode, path=path)
    torch.cuda.synchronize()
    assert kda.kda_get_device_status(ws) == 0
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(state.view(torch.int16), ref_fin.view(torch.int16))


@pytest.mark.parametrize("path", ["chunked", "recurrent"])
def test_varlen_twenty_thousand_sequences(kda_lib, path):
    """20,000 packed sequences of 0 to 3 tokens with H = 2: 40,000 units through the
    device planner's loops (chunked path) or the persistent kernel's unit walk
    (token-by-token path)."""
    lengths = [int(x) for x in np.random.default_rng(76).integers(0, 4, size=20000)]
    w = synth.make("varlen_20k", 1, 0, 2, lengths=lengths, init="randn", seed=76)
    check(w, path=path)
