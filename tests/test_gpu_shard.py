"""GPU parity of the sequence-sharded forward (kimi_delta_attention_08_gb300.shard):
the transition entry point against the oracle run from the identity with zero
values (M) and from zero (B), the compose entry point against the fold written
out in fp64, and two shards of one batch run one after the other in this process
(their pieces passed by hand, as the all-gather would) against the oracle's
single run over the whole sequences."""
import numpy as np
import pytest

from kimi_delta_attention_08_gb300 import synth
from tests.kda_testutil import OUT_TOL, STATE_TOL, compare, device_inputs

import oracle

pytestmark = pytest.mark.gpu


def _slice(d, lo, hi):
    return {nm: (d[nm][:, lo:hi].contiguous() if nm in ("q", "k", "v", "g", "beta") else d[nm])
            for nm in d}


def test_transition_matches_oracle_affine_form(kda_lib):
    """M = final state from the identity with v = 0; B = final state from zero."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    w = synth.make("transition", 2, 300, 3, init="none", seed=71)
    d = device_inputs(w)
    M = torch.full((w.N, w.H, 128, 128), float("nan"), device="cuda")
    Bo = torch.full_like(M, float("nan"))
    ws = kda.make_workspace(w.B * w.T, w.H)
    kda.kda_fwd_transition(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                           w.lower_bound, M, Bo, None, ws)
    assert kda.kda_get_device_status(ws) == 0
    T = w.tensors
    eye = np.broadcast_to(np.eye(128), (w.N, w.H, 128, 128)).copy()
    _, ref_M, _ = oracle.fwd(T["q"], T["k"], np.zeros(T["v"].shape), T["g"], T["beta"],
                             T["A_log"], T["dt_bias"], w.lower_bound, w.scale, eye)
    _, ref_B, _ = oracle.fwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"],
                             T["dt_bias"], w.lower_bound, w.scale, None)
    for got, ref, nm in ((M, ref_M, "M"), (Bo, ref_B, "B")):
        g = got.cpu().numpy().astype(np.float64)
        e = np.linalg.norm(g - ref) / np.linalg.norm(ref)
        print(f"transition {nm}: rel-L2 {e:.2e}")
        assert e <= STATE_TOL, f"{nm}: rel-L2 {e:.3e}"


def test_compose_matches_fold(kda_lib):
    """S_out = fold X <- X M[r] + B[r] from S_in, against the fold in fp64."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    R, ns = 3, 5
    M = synth.normal_f32((R, ns, 128, 128), 72, 1, scale=0.05)
    B = synth.normal_f32((R, ns, 128, 128), 72, 2)
    S0 = synth.normal_f32((ns, 128, 128), 72, 3)
    for s_in in (S0, None):
        out = torch.empty((ns, 128, 128), device="cuda")
        kda.kda_compose_states(torch.from_numpy(M).cuda(), torch.from_numpy(B).cuda(), out,
                               None if s_in is None else torch.from_numpy(s_in).cuda())
        X = np.zeros((ns, 128, 128)) if s_in is None else s_in.astype(np.float64)
        for r in range(R):
            X = X @ M[r].astype(np.float64) + B[r]
        e = np.abs(out.cpu().numpy() - X).max() / np.abs(X).max()
        assert e <= 1e-5, e


@pytest.mark.parametrize("T,cuts,HV", [(2600, (437,), None), (6000, (300, 301, 2000), None),
                                       (3000, (1000,), 8)])
def test_two_and_four_shards_in_process(kda_lib, T, cuts, HV):
    """Shards of every sequence run in rank order in one process, pieces passed
    by hand.  Four shards: one of a single token (the token-by-token path) and a
    last one of 4,000 tokens on 8 (sequence, head) units, where kda_fwd's
    automatic plan splits the shard into segments: the intracard segment scan
    nested inside a rank's shard.  The third case has two value heads per q/k
    head and an fp32 gate."""
    import torch
    from kimi_delta_attention_08_gb300 import shard
    w = synth.make(f"shards_{len(cuts) + 1}" + ("_gva" if HV else ""), 2, T, 4, init="randn",
                   seed=73, HV=HV, g_dtype="fp32" if HV else "bf16")
    d = device_inputs(w)
    bounds = [0, *cuts, w.T]
    parts = [_slice(d, lo, hi) for lo, hi in zip(bounds[:-1], bounds[1:])]
    outs = [torch.full_like(p["v"], float("nan")) for p in parts]
    pieces = []
    for r, p in enumerate(parts):
        pieces.append(shard.shard_piece(r, p["q"], p["k"], p["v"], p["g"], p["beta"], w.scale,
                                        outs[r], p["A_log"], p["dt_bias"], w.lower_bound,
                                        d["initial_state"] if r == 0 else None))
    pieces = torch.stack(pieces)
    fin = None
    for r, p in enumerate(parts):
        f = torch.full((w.N, w.HV, 128, 128), float("nan"), device="cuda")
        shard.shard_finish(r, pieces, p["q"], p["k"], p["v"], p["g"], p["beta"], w.scale,
                           outs[r], p["A_log"], p["dt_bias"], w.lower_bound, f)
        fin = f
    out = torch.cat(outs, dim=1)
    T = w.tensors
    ref_out, ref_fin, _ = oracle.fwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"],
                                     T["dt_bias"], w.lower_bound, w.scale, T["initial_state"])
    e_out, e_st = compare(out, fin, ref_out, ref_fin, label=w.name)
    assert e_out <= OUT_TOL and e_st <= STATE_TOL, (e_out, e_st)


def test_transition_grouped_heads_fp32_gate_varlen(kda_lib):
    """The transition entry point on packed sequences (one empty, one of a single
    token, ragged tails) with two value heads per q/k head and an fp32 gate: M and
    B against the oracle; the empty sequence's map is the identity and zero."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    w = synth.make("transition_gva_varlen", 1, 0, 2, lengths=[700, 0, 1, 130, 64], HV=4,
                   g_dtype="fp32", init="none", seed=74)
    d = device_inputs(w)
    M = torch.full((w.N, w.HV, 128, 128), float("nan"), device="cuda")
    Bo = torch.full_like(M, float("nan"))
    ws = kda.make_workspace(w.B * w.T, w.HV)
    kda.kda_fwd_transition(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                           w.lower_bound, M, Bo, d["cu_seqlens"], ws)
    assert kda.kda_get_device_status(ws) == 0
    T = w.tensors
    eye = np.broadcast_to(np.eye(128), (w.N, w.HV, 128, 128)).copy()
    _, ref_M, _ = oracle.fwd(T["q"], T["k"], np.zeros(T["v"].shape), T["g"], T["beta"],
                             T["A_log"], T["dt_bias"], w.lower_bound, w.scale, eye,
                             cu_seqlens=w.cu_seqlens)
    _, ref_B, _ = oracle.fwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"],
                             T["dt_bias"], w.lower_bound, w.scale, None, cu_seqlens=w.cu_seqlens)
    Mg, Bg = M.cpu().numpy().astype(np.float64), Bo.cpu().numpy().astype(np.float64)
    assert np.array_equal(Mg[1], eye[1]) and not np.any(Bg[1]), "empty sequence"
    for g, ref, nm in ((Mg, ref_M, "M"), (Bg, ref_B, "B")):
        e = np.linalg.norm(g - ref) / np.linalg.norm(ref)
        print(f"transition (grouped heads, fp32 gate, varlen) {nm}: rel-L2 {e:.2e}")
        assert e <= STATE_TOL, f"{nm}: rel-L2 {e:.3e}"
