"""kda_fwd inside a CUDA graph: the library only enqueues work on the caller's
stream (status-header memset, the device-side planner, the kernels), so a call
can be captured once and replayed.  A replay on new inputs, copied into the
captured buffers, must give the bits of a direct call on the same inputs."""
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
