"""kda_fwd_static_scratch: the forward for callers that cannot allocate device
memory (a host framework that owns all device memory and passes a plugin only
its input and output buffers, or a runtime with a fixed memory budget).  It runs
kda_fwd with its workspace in a file-scope device array.

The GPU test calls it through the C ABI twice in a row on a problem that uses
the workspace scratch (schedule tables and segment-scan state slots) and checks
each call against kda_fwd with a caller-allocated workspace.  This file is
collected last so a run that stops at the first failure has run every other
test already; it also passes when run alone in a fresh process."""
import ctypes

import numpy as np
import pytest

from kimi_delta_attention_08_gb300 import _lib, synth
from tests.kda_testutil import OUT_TOL, STATE_TOL, device_inputs, run_gpu

KDA_OK, KDA_ERR_NULL_POINTER, KDA_ERR_INVALID_SHAPE, KDA_ERR_MISALIGNED = 0, 1, 2, 4
KDA_ERR_WORKSPACE_TOO_SMALL, KDA_ERR_DEVICE_TIMEOUT = 5, 8


def _call_static(lib, w, d, out, fin, cp_mode, seg_chunks, debug_stall=0):
    import torch
    opts = _lib.kda_options()
    opts.debug_stall = debug_stall
    opts.cp_mode = {"auto": 0, "off": 1, "force": 2}[cp_mode]
    opts.seg_chunks = seg_chunks
    HV = d["v"].shape[2]
    opts.num_v_heads = HV if HV != w.H else 0
    opts.g_dtype = 1 if d["g"].dtype == torch.float32 else 0
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    q = d["q"]
    B, T = q.shape[0], q.shape[1]
    stream = torch.cuda.current_stream().cuda_stream
    return lib.kda_fwd_static_scratch(
        P(d["q"]), P(d["k"]), P(d["v"]), P(d["g"]), P(d["beta"]), float(w.scale), P(out),
        P(d["A_log"]), P(d["dt_bias"]), float(w.lower_bound), P(d["initial_state"]), P(fin),
        P(d["cu_seqlens"]), B, T, w.H, w.N, 1 if w.state_dtype == "bf16" else 0,
        ctypes.byref(opts), ctypes.c_void_p(stream))


def test_static_scratch_rejects_oversized_problem():
    from kimi_delta_attention_08_gb300 import build
    build.build()
    lib = _lib.load()
    fake = lambda a: ctypes.c_void_p(a)
    st = lib.kda_fwd_static_scratch(
        fake(0x10000), fake(0x20000), fake(0x30000), fake(0x40000), fake(0x50000), 0.1,
        fake(0x60000), fake(0x70000), fake(0x80000), -5.0, None, None, None,
        1, 1 << 30, 64, 1, 0, None, None)
    assert st == KDA_ERR_WORKSPACE_TOO_SMALL


def test_static_scratch_argument_errors_are_kda_fwds():
    """A call that kda_fwd rejects for its arguments gets kda_fwd's status, not the
    size limit's, even when the problem is also too large for the array; and the
    status accessor checks its pointer.  No kernel runs."""
    from kimi_delta_attention_08_gb300 import build
    build.build()
    lib = _lib.load()
    fake = lambda a: ctypes.c_void_p(a)
    ptrs = [fake(0x10000 * i) for i in range(1, 10)]

    def call(B, T, H, opts=None, A_log=ptrs[6], q=ptrs[0]):
        return lib.kda_fwd_static_scratch(q, ptrs[1], ptrs[2], ptrs[3], ptrs[4], 0.1, ptrs[5],
                                          A_log, ptrs[7], -5.0, None, None, None, B, T, H, B, 0,
                                          opts, None)
    assert call(1, 1 << 31, 64) == KDA_ERR_INVALID_SHAPE           # B*T >= 2^31
    assert call(1, 1 << 30, 64, A_log=None) == KDA_ERR_NULL_POINTER
    assert call(1, 1 << 30, 64, q=fake(0x10008)) == KDA_ERR_MISALIGNED
    opts = _lib.kda_options()
    opts.num_v_heads = 65                                          # not a multiple of H
    assert call(1, 1 << 30, 64, opts=ctypes.byref(opts)) == KDA_ERR_INVALID_SHAPE
    assert call(1, 1 << 30, 64) == KDA_ERR_WORKSPACE_TOO_SMALL
    assert lib.kda_static_scratch_device_status(None, None) == KDA_ERR_NULL_POINTER


@pytest.mark.gpu
def test_static_scratch_reports_device_status(kda_lib):
    """Device-side errors of a static-scratch call are readable: a bounded wait made
    to run out on purpose (debug_stall, no fault) reads back as a timeout; the next
    normal call reads back KDA_OK and matches kda_fwd with a caller workspace."""
    import torch
    w = synth.make("static_stall", 2, 256, 4, init="randn", seed=53)
    d = device_inputs(w)
    out = torch.zeros_like(d["q"])
    fin = torch.zeros((w.N, w.H, 128, 128), dtype=torch.float32, device="cuda")
    st = ctypes.c_int(-1)
    assert _call_static(kda_lib, w, d, out, fin, "off", 0, debug_stall=1) == KDA_OK
    assert kda_lib.kda_static_scratch_device_status(ctypes.byref(st), None) == KDA_OK
    assert st.value == KDA_ERR_DEVICE_TIMEOUT
    ref_out, ref_fin = run_gpu(w, inputs=d, cp_mode="off")
    assert _call_static(kda_lib, w, d, out, fin, "off", 0) == KDA_OK
    assert kda_lib.kda_static_scratch_device_status(ctypes.byref(st), None) == KDA_OK
    assert st.value == KDA_OK
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(fin.view(torch.int32), ref_fin.view(torch.int32))


@pytest.mark.gpu
def test_static_scratch_matches_caller_workspace(kda_lib):
    import torch
    w = synth.make("static_scratch", 1, 0, 3, lengths=[300, 1, 520, 64, 0, 200],
                   init="randn", seed=51)
    d = device_inputs(w)
    ref_out, ref_fin = run_gpu(w, inputs=d, cp_mode="force", seg_chunks=2)
    torch.cuda.synchronize()
    ro = ref_out.float().cpu().numpy()
    rf = ref_fin.float().cpu().numpy()
    for call in range(2):
        out = torch.full_like(d["q"], float("nan"))
        fin = torch.full((w.N, w.H, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
        st = _call_static(kda_lib, w, d, out, fin, "force", 2)
        assert st == KDA_OK, f"call {call}: status {st}"
        torch.cuda.synchronize()
        o = out.float().cpu().numpy()
        f = fin.cpu().numpy()
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(f))
        e_out = np.abs(o - ro).max() / np.abs(ro).max()
        e_st = np.linalg.norm(f - rf) / np.linalg.norm(rf)
        assert e_out <= OUT_TOL, f"call {call}: out differs by {e_out:.3e}"
        assert e_st <= STATE_TOL, f"call {call}: state differs by {e_st:.3e}"


@pytest.mark.gpu
def test_static_scratch_grouped_heads_fp32_gate(kda_lib):
    """Grouped value heads (H = 2, HV = 6) and an fp32 gate through the segment scan:
    the static array is sized by the value heads, and the result equals kda_fwd
    with a caller workspace bit for bit (same plan, same kernels)."""
    import torch
    w = synth.make("static_gva", 1, 0, 2, HV=6, g_dtype="fp32", lengths=[300, 1, 520, 0, 200],
                   init="randn", seed=52)
    d = device_inputs(w)
    ref_out, ref_fin = run_gpu(w, inputs=d, cp_mode="force", seg_chunks=2)
    out = torch.full_like(d["v"], float("nan"))
    fin = torch.full((w.N, 6, 128, 128), float("nan"), dtype=torch.float32, device="cuda")
    assert _call_static(kda_lib, w, d, out, fin, "force", 2) == KDA_OK
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(fin.view(torch.int32), ref_fin.view(torch.int32))
