"""GPU parity of grouped value heads (HV a multiple of the q/k heads H) and of
the fp32 gate input, on both kernels, against the fp64 oracle with the shared
tolerances; plus bitwise identities that pin the head mapping and the gate
read independently of the oracle:
  - grouped input equals the plain input with q/k repeated per value head;
  - an fp32 gate whose values are on the bf16 grid equals the bf16 gate."""
import numpy as np
import pytest

from kimi_delta_attention_08_gb300 import synth
from tests.kda_testutil import OUT_TOL, STATE_TOL, compare, device_inputs, run_gpu

import oracle

pytestmark = pytest.mark.gpu

REC_STATE_TOL = 1e-4  # token-by-token path: fp32 throughout


def oracle_run(w, use_init=True):
    T = w.tensors
    out, fin, _ = oracle.fwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"], T["dt_bias"],
                             w.lower_bound, w.scale, T["initial_state"] if use_init else None,
                             w.cu_seqlens)
    return out, fin


def check(w, state_tol=STATE_TOL, **kw):
    out, fin = run_gpu(w, **kw)
    ref_out, ref_fin = oracle_run(w)
    e_out, e_st = compare(out, fin, ref_out, ref_fin)
    assert e_out <= OUT_TOL, f"{w.name}: out max-rel error {e_out:.3e}"
    assert e_st <= state_tol, f"{w.name}: state rel-L2 error {e_st:.3e}"
    return out, fin


# ------------------------------------------------------------ chunked path --
@pytest.mark.parametrize("H,HV,T", [(2, 6, 200), (4, 32, 130), (1, 3, 65), (1, 64, 130)])
def test_chunked_grouped_heads(kda_lib, H, HV, T):
    check(synth.make(f"gva_H{H}_HV{HV}", 2, T, H, HV=HV, init="randn", seed=400 + HV),
          path="chunked")


@pytest.mark.parametrize("T", [1, 63, 64, 200, 333])
def test_chunked_fp32_gate(kda_lib, T):
    check(synth.make(f"g32_T{T}", 2, T, 3, g_dtype="fp32", init="randn", seed=410 + T),
          path="chunked")


def test_chunked_grouped_fp32_gate_varlen_bf16_state(kda_lib):
    w = synth.make("gva_g32_varlen", 1, 0, 2, HV=8, g_dtype="fp32", state_dtype="bf16",
                   lengths=[5, 0, 64, 130, 1, 77], init="randn", seed=420)
    check(w, path="chunked")


@pytest.mark.parametrize("cp_mode", ["auto", "force"])
def test_grouped_fp32_gate_segment_scan(kda_lib, cp_mode):
    """A long sequence split into segments (prescan, merge, rerun) with both
    variants on."""
    w = synth.make("gva_g32_cp", 1, 0, 2, HV=4, g_dtype="fp32",
                   lengths=[40 * 64 + 17, 300], init="randn", lower_bound=-0.3, seed=421)
    check(w, cp_mode=cp_mode, seg_chunks=8 if cp_mode == "force" else 0)


# -------------------------------------------------------- recurrent path ----
@pytest.mark.parametrize("T", [1, 7, 16, 33])
def test_recurrent_grouped_fp32_gate(kda_lib, T):
    w = synth.make(f"rec_gva_g32_T{T}", 24, T, 2, HV=8, g_dtype="fp32", init="randn",
                   seed=430 + T)
    check(w, path="recurrent", state_tol=REC_STATE_TOL)


def test_recurrent_grouped_varlen(kda_lib):
    w = synth.make("rec_gva_varlen", 1, 0, 4, HV=16, lengths=[3, 0, 16, 40, 1],
                   init="randn", seed=431)
    check(w, path="recurrent", state_tol=REC_STATE_TOL)


# ---------------------------------------------------- bitwise identities ----
def _repeated(w):
    """The plain problem whose q/k heads are w's repeated per value head."""
    G = w.n_vheads // w.H
    p = synth.make(w.name + "_plain", w.B, w.T, w.n_vheads, lengths=w.lengths,
                   state_dtype=w.state_dtype, init="randn", lower_bound=w.lower_bound,
                   seed=w.seed, g_dtype=w.g_dtype)
    for nm in ("v", "g", "beta", "A_log", "dt_bias", "initial_state"):
        p.tensors[nm] = w.tensors[nm]
    p.tensors["q"] = np.repeat(w.tensors["q"], G, axis=-2)
    p.tensors["k"] = np.repeat(w.tensors["k"], G, axis=-2)
    return p


@pytest.mark.parametrize("path", ["chunked", "recurrent"])
def test_grouped_equals_repeated_qk_bitwise(kda_lib, path):
    import torch
    w = synth.make("gva_bits", 3, 150, 2, HV=6, init="randn", seed=440)
    o1, f1 = run_gpu(w, path=path)
    o2, f2 = run_gpu(_repeated(w), path=path)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(f1.view(torch.int32), f2.view(torch.int32))


@pytest.mark.parametrize("path", ["chunked", "recurrent"])
def test_fp32_gate_on_bf16_grid_equals_bf16_gate_bitwise(kda_lib, path):
    import torch
    w = synth.make("g_grid", 2, 150, 4, init="randn", seed=441)
    o1, f1 = run_gpu(w, path=path)
    d = device_inputs(w)
    d["g"] = d["g"].float()  # exact: every bf16 value is an fp32 value
    w.g_dtype = "fp32"
    o2, f2 = run_gpu(w, path=path, inputs=d)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(f1.view(torch.int32), f2.view(torch.int32))


# ------------------------------------------------ full size, sampled units --
def test_gva_fp32_gate_full_size_sampled(kda_lib):
    """The benchmark's grouped-head workload (B=8, T=4096, H=16, HV=32, fp32 gate)
    in the benchmark's launch configuration; sampled (sequence, value head) units
    against the oracle run on just those (q/k from the unit's key head)."""
    w = synth.make("gva_B8_T4096_H16_HV32_g32", 8, 4096, 16, HV=32, g_dtype="fp32",
                   init="zero", seed=6)
    out, fin = run_gpu(w)
    T = w.tensors
    G = w.n_vheads // w.H
    for n, h in [(0, 0), (0, 1), (3, 17), (7, 31), (5, 2)]:
        sl = slice(n * w.T, (n + 1) * w.T)
        hk = h // G
        flat = lambda nm, nh, hh: T[nm].reshape(-1, nh, *T[nm].shape[3:])[sl, hh:hh + 1][None]
        ro, rf, _ = oracle.fwd(flat("q", w.H, hk), flat("k", w.H, hk), flat("v", w.n_vheads, h),
                               flat("g", w.n_vheads, h),
                               T["beta"].reshape(-1, w.n_vheads)[sl, h:h + 1][None],
                               T["A_log"][h:h + 1], T["dt_bias"][h:h + 1], w.lower_bound, w.scale,
                               T["initial_state"][n:n + 1, h:h + 1])
        o = out.reshape(-1, w.n_vheads, 128)[sl, h].unsqueeze(1)[None]
        e_out, e_st = compare(o, fin[n:n + 1, h:h + 1], ro, rf)
        assert e_out <= OUT_TOL, f"unit {(n, h)}: out {e_out:.3e}"
        assert e_st <= STATE_TOL, f"unit {(n, h)}: state {e_st:.3e}"
