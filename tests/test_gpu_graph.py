"""kda_fwd and kda_bwd inside a CUDA graph: the library only enqueues work on the
caller's stream (status-header memset, the device-side planner, the kernels), so
a call can be captured once and replayed.  A replay on new inputs, copied into
the captured buffers, must give the bits of a direct call on the same inputs."""
import numpy as np
import pytest

from kimi_delta_attention_08_gb300 import synth
from tests.kda_testutil import device_inputs

pytestmark = pytest.mark.gpu


def _call(kda, d, w, out, fin, ws, cp_mode):
    kda.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, out, d["A_log"],
                d["dt_bias"], w.lower_bound, d["initial_state"], fin, d["cu_seqlens"], ws,
                cp_mode=cp_mode)


@pytest.mark.parametrize("case", ["batched", "varlen_segment_scan"])
def test_graph_replay_matches_direct_calls(kda_lib, case):
    import torch
    import kimi_delta_attention_08_gb300 as kda
    if case == "batched":
        mk = lambda seed: synth.make("graph_batched", 2, 300, 4, init="randn", seed=seed)
        cp_mode = "auto"
    else:
        mk = lambda seed: synth.make("graph_varlen", 1, 0, 2, lengths=[2000, 1, 0, 130],
                                     init="randn", seed=seed)
        cp_mode = "force"
    w0 = mk(80)
    d = device_inputs(w0)                                 # the captured buffers
    out = torch.empty_like(d["v"])
    fin = torch.empty((w0.N, w0.HV, 128, 128), dtype=torch.float32, device="cuda")
    ws = kda.make_workspace(w0.B * w0.T, w0.HV)
    _call(kda, d, w0, out, fin, ws, cp_mode)              # first call outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _call(kda, d, w0, out, fin, ws, cp_mode)
    for seed in (81, 82):
        w = mk(seed)
        fresh = device_inputs(w)
        for nm in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state"):
            d[nm].copy_(fresh[nm])
        graph.replay()
        torch.cuda.synchronize()
        assert kda.kda_get_device_status(ws) == 0
        ref_out = torch.empty_like(out)
        ref_fin = torch.empty_like(fin)
        ws2 = kda.make_workspace(w.B * w.T, w.HV)
        _call(kda, fresh, w, ref_out, ref_fin, ws2, cp_mode)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"out, seed {seed}"
        assert torch.equal(fin.view(torch.int32), ref_fin.view(torch.int32)), f"state, seed {seed}"


def test_graph_replay_backward(kda_lib):
    """kda_bwd captured once (its outputs and workspace come from the graph's memory
    pool) and replayed on new inputs and cotangents: the bits of direct calls."""
    import torch
    import kimi_delta_attention_08_gb300 as kda
    from tests.kda_testutil import to_torch_bf16, to_torch_f32
    mk = lambda seed: synth.make("graph_bwd", 2, 150, 2, init="randn", lower_bound=-2.0, seed=seed)

    def cot(w, seed):
        rng = np.random.default_rng(seed)
        dout = synth.f32_to_bf16_bits(rng.standard_normal(w.tensors["v"].shape).astype(np.float32))
        df = rng.standard_normal((w.N, w.HV, 128, 128)).astype(np.float32)
        return to_torch_bf16(dout, "cuda"), to_torch_f32(df, "cuda")

    w0 = mk(83)
    d = device_inputs(w0)
    dout, dfin = cot(w0, 83)
    call = lambda dd, do, df: kda.kda_bwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], w0.scale,
                                          dd["A_log"], dd["dt_bias"], w0.lower_bound, do,
                                          dd["initial_state"], df)
    call(d, dout, dfin)                                   # first call outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g = call(d, dout, dfin)
    for seed in (84, 85):
        w = mk(seed)
        fresh = device_inputs(w)
        do2, df2 = cot(w, seed)
        for nm in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state"):
            d[nm].copy_(fresh[nm])
        dout.copy_(do2)
        dfin.copy_(df2)
        graph.replay()
        torch.cuda.synchronize()
        ref = call(fresh, do2, df2)
        torch.cuda.synchronize()
        for nm in ("dq", "dk", "dv", "dg", "dbeta", "dA_log", "ddt_bias", "dinitial_state"):
            assert torch.equal(g[nm].view(torch.int32), ref[nm].view(torch.int32)), (nm, seed)
