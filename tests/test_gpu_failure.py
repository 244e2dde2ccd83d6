"""Failure detection on the GPU without a fault: a bounded wait is made to run out
on purpose with the test-only `debug_stall` option (the token-by-token kernel
never fetches a CTA's third unit; the chunk kernel's prep group never hands a
chunk to the factor group), so nothing ever completes the awaited barrier.  The
call must come back, the device status must read KDA_ERR_DEVICE_TIMEOUT, and the
CUDA context must stay usable: the next normal call is checked against the
oracle."""
import time

import pytest

from kimi_delta_attention_08_gb300 import synth
from tests.kda_testutil import OUT_TOL, STATE_TOL, compare, device_inputs, run_gpu

import oracle

pytestmark = pytest.mark.gpu

KDA_ERR_DEVICE_TIMEOUT = 8


@pytest.mark.parametrize("path", ["recurrent", "chunked"])
def test_bounded_wait_expires_reports_timeout_and_context_survives(kda_lib, path):
    import torch
    import kimi_delta_attention_08_gb300 as kda
    # recurrent: 64 x 32 = 2048 (sequence, head) units, several per SM, so every CTA
    # has a third unit; chunked: 8 units of 4 chunks, one wave
    w = (synth.make("stall", 64, 1, 32, init="randn", seed=500) if path == "recurrent"
         else synth.make("stall_chunked", 2, 256, 4, init="randn", seed=501))
    d = device_inputs(w)
    out = torch.zeros_like(d["v"])
    fin = torch.zeros((w.N, w.H, 128, 128), dtype=torch.float32, device="cuda")
    ws = kda.make_workspace(w.B * w.T, w.H)
    t0 = time.time()
    kda.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, out, d["A_log"],
                d["dt_bias"], w.lower_bound, d["initial_state"], fin, None, ws,
                path=path, debug_stall=1)
    status = kda.kda_get_device_status(ws)  # synchronises
    elapsed = time.time() - t0
    assert status == KDA_ERR_DEVICE_TIMEOUT, kda.status_string(status)
    assert elapsed < 10.0, f"the bounded wait took {elapsed:.1f} s"

    # same context, normal call: correct results and a clean status
    T = w.tensors
    ref_out, ref_fin, _ = oracle.fwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"],
                                     T["dt_bias"], w.lower_bound, w.scale, T["initial_state"])
    o2, f2 = run_gpu(w, path=path)
    e_out, e_st = compare(o2, f2, ref_out, ref_fin)
    assert e_out <= OUT_TOL and e_st <= (1e-4 if path == "recurrent" else STATE_TOL)


def test_bwd_chunked_bounded_wait_expires_and_context_survives(kda_lib):
    """The chunked backward's stall hook: the reverse kernel never issues a chunk's
    first MMAs, so the wait for them expires on every CTA.  The call comes back with
    KDA_ERR_DEVICE_TIMEOUT in the status word, and the next normal backward on the
    same context matches the oracle."""
    import kimi_delta_attention_08_gb300 as kda
    from tests.kda_testutil import bwd_chunk_errors, to_torch_bf16, to_torch_f32
    w = synth.make("stall_bwd", 2, 256, 4, init="randn", seed=502)
    T = w.tensors
    dout = synth.normal_bf16((w.B, w.T, w.H, 128), 7, 9)
    df = synth.normal_f32((w.N, w.H, 128, 128), 7, 10)
    d = device_inputs(w)
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, d["A_log"], d["dt_bias"],
            w.lower_bound, to_torch_bf16(dout, "cuda"), d["initial_state"], to_torch_f32(df, "cuda"))
    t0 = time.time()
    g = kda.kda_bwd(*args, path="chunked", debug_stall=1)
    status = kda.kda_get_device_status(g["workspace"])
    elapsed = time.time() - t0
    assert status == KDA_ERR_DEVICE_TIMEOUT, kda.status_string(status)
    assert elapsed < 10.0, f"the bounded wait took {elapsed:.1f} s"

    g2 = kda.kda_bwd(*args, path="chunked")
    assert kda.kda_get_device_status(g2["workspace"]) == 0
    ref = oracle.bwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"], T["dt_bias"],
                     w.lower_bound, w.scale, dout, T["initial_state"], df)
    errs, lim = bwd_chunk_errors(w, {nm: g2[nm].cpu().numpy() for nm in ref}, ref)
    assert all(errs[k] <= lim[k] for k in errs), errs
