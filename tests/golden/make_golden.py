"""Writes the stored expected values under tests/golden/ from the fp64 oracle
alone (oracle/ and the seeded input generators; nothing from the CUDA path).

    python tests/golden/make_golden.py

The pages print no numeric worked example, so these fixtures are regression
pins of the oracle: tests/test_golden.py recomputes them and any change to the
oracle's arithmetic shows up as a mismatch.  Regenerate only together with such
a change, and name in the commit the passage (or its reading) that justifies it.

Method followed (page titles and sections):
- the recurrence and the per-channel gate: "How FlashKDA Integrates with CUTLASS
  for High-Performance GEMM Operations", "Kernel Launch Pipeline and Template
  Dispatching" (the KDA recurrence), with the gate form, l2 norm and sigmoid read
  as the oracle states them;
- the in-kernel preprocessing flags and lower_bound range: "How to Use FlashKDA as
  a Backend for flash-linear-attention: Complete Integration Guide", "Running
  Inference with chunk_kda" and "Kernel API and Tensor Requirements";
- varlen and the state layout [N, H, V, K]: the same guide, "State Handling and
  Variable-Length Batches";
- the backward: reverse mode of that forward (the pages' kernels are forward
  only, "feat(kda): SM90 FlashKDA prefill, intracard CP, and backend dispatch",
  commit notes).
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from kimi_delta_attention_08_gb300 import synth  # noqa: E402

NCH = 16  # channels of each per-token vector that are stored


def cases():
    """(file stem, workload, dout seed) of every fixture."""
    yield ("plain_T5_H1", synth.make("golden_plain", 1, 5, 1, init="randn", lower_bound=-2.0,
                                     seed=61), 62)
    yield ("varlen_grouped_fp32g", synth.make("golden_varlen", 1, 0, 1, HV=2, lengths=[3, 0, 2],
                                              init="randn", g_dtype="fp32", lower_bound=-5.0,
                                              seed=63), 64)


def compute(w, dseed):
    """The stored quantities of workload w: forward outputs and final states, and
    the backward's gradients for seeded cotangents."""
    T = w.tensors
    HV = w.n_vheads
    out, fin, _ = oracle.fwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"],
                             T["dt_bias"], w.lower_bound, w.scale, T["initial_state"],
                             w.cu_seqlens, want_final=True)
    dout = synth.normal_bf16(out.shape, dseed, 9)
    dfin = synth.normal_f32((w.N, HV, 128, 128), dseed, 10)
    g = oracle.bwd(T["q"], T["k"], T["v"], T["g"], T["beta"], T["A_log"], T["dt_bias"],
                   w.lower_bound, w.scale, dout, T["initial_state"], dfin, w.cu_seqlens)
    vals = {
        "out": out[..., :NCH],
        "final_state_row_sums": fin[..., :NCH, :].sum(axis=-1),  # value rows v < 16
    }
    for nm in ("dq", "dk", "dv", "dg"):
        vals[nm] = g[nm][..., :NCH]
    vals["dbeta"] = g["dbeta"]
    vals["dA_log"] = g["dA_log"]
    vals["ddt_bias"] = g["ddt_bias"][..., :NCH]
    vals["dinitial_state_row_sums"] = g["dinitial_state"][..., :NCH, :].sum(axis=-1)
    return {k: np.ascontiguousarray(v, dtype=np.float64) for k, v in vals.items()}


def write(stem, w, dseed):
    vals = compute(w, dseed)
    path = os.path.join(HERE, f"{stem}.txt")
    with open(path, "w") as f:
        f.write(f"# fp64 oracle values for workload {w.name}: B={w.B} T={w.T} H={w.H} "
                f"HV={w.n_vheads} lengths={w.lengths} state={w.state_dtype} "
                f"g={w.g_dtype} lower_bound={w.lower_bound} seed={w.seed}; "
                f"cotangent seed {dseed}\n")
        f.write("# written by tests/golden/make_golden.py (oracle/ only); per-token vectors "
                "keep their first 16 channels, states the sums of their first 16 value rows\n")
        for k, v in vals.items():
            f.write(f"{k} {' '.join(str(d) for d in v.shape)} : "
                    + " ".join(f"{x:.15g}" for x in v.ravel()) + "\n")
    return path


def read(path):
    vals = {}
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            head, data = line.split(":", 1)
            parts = head.split()
            shape = tuple(int(x) for x in parts[1:])
            vals[parts[0]] = np.array([float(x) for x in data.split()]).reshape(shape)
    return vals


if __name__ == "__main__":
    for stem, w, dseed in cases():
        print(write(stem, w, dseed))
