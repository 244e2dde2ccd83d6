"""Helpers shared by the tests: move a seeded workload to the GPU, run the CUDA
path through the binding, and compare with the oracle's fp64 result."""
from __future__ import annotations

import numpy as np

from kimi_delta_attention_08_gb300 import synth

OUT_TOL = 1e-2     # max|out - ref| <= 1e-2 * max|ref|
STATE_TOL = 5e-3   # ||S - S_ref||_F <= 5e-3 * ||S_ref||_F

# (case, out max-rel error, state rel-L2 error) of every parity comparison in the
# run; conftest prints the full-size cases and the worst case at the end, so the
# margins against the tolerances show in the run's output.
PARITY_LOG = []


def to_torch_bf16(bits, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_torch_f32(x, device):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)


def bf16_tensor_to_f64(t):
    import torch
    return t.detach().float().cpu().numpy().astype(np.float64)


def device_inputs(w, device="cuda"):
    T = w.tensors
    d = {nm: to_torch_bf16(T[nm], device) for nm in ("q", "k", "v", "beta")}
    d["g"] = (to_torch_f32(T["g"], device) if getattr(w, "g_dtype", "bf16") == "fp32"
              else to_torch_bf16(T["g"], device))
    d["A_log"] = to_torch_f32(T["A_log"], device)
    d["dt_bias"] = to_torch_f32(T["dt_bias"], device)
    init = T["initial_state"]
    if init is None:
        d["initial_state"] = None
    elif w.state_dtype == "bf16":
        d["initial_state"] = to_torch_bf16(init, device)
    else:
        d["initial_state"] = to_torch_f32(init, device)
    cu = w.cu_seqlens
    import torch
    d["cu_seqlens"] = None if cu is None else torch.from_numpy(cu).to(device)
    return d


def run_gpu(w, device="cuda", cp_mode="auto", seg_chunks=0, final=True, inputs=None,
            use_init=True, out=None, workspace=None, path="auto"):
    import torch
    import kimi_delta_attention_08_gb300 as kda
    d = inputs if inputs is not None else device_inputs(w, device)
    q = d["q"]
    HV = d["v"].shape[2]  # value heads (= q's heads unless grouped)
    if out is None:
        out = torch.full_like(d["v"], float("nan"))
    sdt = torch.bfloat16 if w.state_dtype == "bf16" else torch.float32
    fin = torch.full((w.N, HV, 128, 128), float("nan"), dtype=sdt, device=q.device) if final else None
    if workspace is None:
        workspace = kda.make_workspace(q.shape[0] * q.shape[1], HV, q.device)
    kda.kda_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], w.scale, out, d["A_log"], d["dt_bias"],
                w.lower_bound, d["initial_state"] if use_init else None, fin, d["cu_seqlens"],
                workspace, cp_mode=cp_mode, seg_chunks=seg_chunks, path=path)
    st = kda.kda_get_device_status(workspace)
    if st != 0:
        raise RuntimeError(f"device status {st}: {kda.status_string(st)}")
    return out, fin


def compare(out, fin, ref_out, ref_fin, label=None):
    """(max|out-ref|/max|ref|, rel-L2 of the final state); out/fin are torch.
    With a label, the pair is added to PARITY_LOG."""
    o = bf16_tensor_to_f64(out).reshape(ref_out.shape)
    denom = np.abs(ref_out).max()
    e_out = float(np.abs(o - ref_out).max() / (denom if denom > 0 else 1.0))
    e_st = 0.0
    if fin is not None and ref_fin is not None:
        f = fin.detach().float().cpu().numpy().astype(np.float64)
        nr = np.linalg.norm(ref_fin)
        e_st = float(np.linalg.norm(f - ref_fin) / (nr if nr > 0 else 1.0))
        if not np.all(np.isfinite(f)):
            e_st = float("inf")
    if not np.all(np.isfinite(o)):
        e_out = float("inf")
    if label is not None:
        PARITY_LOG.append((label, e_out, e_st if fin is not None and ref_fin is not None else None))
    return e_out, e_st


# Tolerance of the chunked (tensor-core) backward.  Its MMA operands are bf16
# (relative rounding 2^-9) and every gradient passes through two to four such
# products, with fp32 accumulation; an emulation of the kernel's arithmetic in
# numpy reproduces its errors to two digits, at most 1.2e-2 of a gradient's
# largest magnitude on the cases of tests/test_gpu_bwd_chunk.py.  The sums over
# tokens (dA_log per head, dt_bias per channel) are sums of per-token terms
# (dg, and dg (g + dt_bias) for A_log) whose own accuracy the dg bound fixes;
# each is checked by the triangle inequality against the oracle's terms:
# |sum_kernel - sum_oracle| <= sum_t |term_kernel - term_oracle| + fp32 rounding
# of the sum (1e-4 of the summed magnitudes: sequential fp32 sums of up to a few
# thousand terms), reported as a ratio (<= 1 passes).
CHUNK_BWD_TOL = 2e-2
BWD_TOKEN_NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dinitial_state")


def bwd_chunk_errors(w, got, ref):
    """Errors of the chunked backward's gradients `got` (numpy, any shape) against
    the oracle's `ref`: per-token tensors and dinitial_state relative to their
    largest magnitude (limit CHUNK_BWD_TOL); dA_log and ddt_bias as the ratio of
    their error to the triangle bound (limit 1).  Returns (errs, limits)."""
    import oracle
    errs, limits = {}, {}
    for nm in BWD_TOKEN_NAMES:
        g = np.asarray(got[nm], dtype=np.float64).reshape(ref[nm].shape)
        limits[nm] = CHUNK_BWD_TOL
        if not np.all(np.isfinite(g)):
            errs[nm] = float("inf")
            continue
        den = np.abs(ref[nm]).max()
        errs[nm] = float(np.abs(g - ref[nm]).max() / (den if den > 0 else 1.0))
    HV = w.n_vheads
    dg_r = ref["dg"].reshape(-1, HV, 128)
    dg_k = np.asarray(got["dg"], dtype=np.float64).reshape(-1, HV, 128)
    gx = oracle._as_f64(w.tensors["g"], "g").reshape(-1, HV, 128)
    dtb = np.asarray(w.tensors["dt_bias"], dtype=np.float64).reshape(HV, 128)
    xa = gx + dtb[None]
    terms = {"dA_log": (dg_k * xa, dg_r * xa, (0, 2)), "ddt_bias": (dg_k, dg_r, (0,))}
    for nm, (tk, tr, ax) in terms.items():
        g = np.asarray(got[nm], dtype=np.float64).reshape(ref[nm].shape)
        limits[nm] = 1.0
        if not np.all(np.isfinite(g)):
            errs[nm] = float("inf")
            continue
        bound = np.abs(tk - tr).sum(axis=ax) + 1e-4 * np.abs(tk).sum(axis=ax) + 1e-30
        errs[nm] = float(np.max(np.abs(g - ref[nm]) / bound))
    return errs, limits
