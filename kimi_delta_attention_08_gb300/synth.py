"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and rounds them to the storage types; it holds
none of the attention arithmetic.  Both the CUDA path and the CPU oracle receive
the exact same bits from here.

Generator: numpy's Philox-4x32-10 counter-based bit generator (Salmon et al.,
"Parallel random numbers: as easy as 1, 2, 3", SC'11), keyed per (seed, tensor
stream, block) through a SeedSequence, with numpy's standard-normal transform.
Blocks of 2**22 values are drawn independently, so generation can run on
several host threads and still give the same bits.  fp32 -> bf16 uses
round-to-nearest-even on the bit pattern.

The five workloads follow the shapes, dtypes and distributions of the FlashKDA
usage examples ("How FlashKDA Integrates with CUTLASS ...", section "Practical
Implementation Example"; "How to Use FlashKDA as a Backend ...", section
"Running Inference with chunk_kda"): q, k, v, g ~ N(0,1) bf16 [B,T,H,128],
beta ~ N(0,1) bf16 [B,T,H], A_log ~ N(0,1) fp32 [H], dt_bias ~ N(0,1) fp32
[H,128]; initial states are 0.1 N(0,1).

Grouped value heads (HV > H): q and k keep H heads, while v, g, beta, A_log,
dt_bias and the states get HV heads.  An fp32 gate keeps the generator's fp32
values unrounded.  With HV = H and a bf16 gate every tensor is bit-identical to
the plain workload of the same seed.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

KD = 128
_BLOCK = 1 << 22
_STREAMS = {"q": 1, "k": 2, "v": 3, "g": 4, "beta": 5, "A_log": 6, "dt_bias": 7, "init": 8}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits.
    NaN is not expected from the generator."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _fill_normal(out: np.ndarray, seed: int, stream: int, threads: int) -> None:
    flat = out.reshape(-1)
    nblk = (flat.size + _BLOCK - 1) // _BLOCK

    def work(b):
        lo, hi = b * _BLOCK, min(flat.size, (b + 1) * _BLOCK)
        rng = np.random.Generator(np.random.Philox(np.random.SeedSequence([seed, stream, b])))
        rng.standard_normal(out=flat[lo:hi], dtype=np.float32)

    if nblk <= 1 or threads <= 1:
        for b in range(nblk):
            work(b)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, range(nblk)))


def normal_f32(shape, seed: int, stream: int, scale: float = 1.0, threads: int | None = None):
    out = np.empty(shape, dtype=np.float32)
    _fill_normal(out, seed, stream, threads or min(16, os.cpu_count() or 1))
    if scale != 1.0:
        out *= np.float32(scale)
    return out


def normal_bf16(shape, seed: int, stream: int, scale: float = 1.0, threads: int | None = None):
    return f32_to_bf16_bits(normal_f32(shape, seed, stream, scale, threads))


@dataclass
class Workload:
    """One seeded problem.  Tensors are numpy: bf16 as uint16 bits, fp32 as float32."""
    name: str
    B: int
    T: int
    H: int
    lengths: list | None          # varlen sequence lengths (then B == 1, T == sum)
    state_dtype: str              # "fp32" | "bf16"
    init: str                     # "none" | "zero" | "randn"
    final: bool
    lower_bound: float
    scale: float
    seed: int
    tensors: dict = field(default_factory=dict)
    HV: int = 0                   # value heads (0: same as H)
    g_dtype: str = "bf16"         # "bf16" | "fp32"

    @property
    def n_vheads(self) -> int:
        return self.HV if self.HV else self.H

    @property
    def N(self) -> int:
        return len(self.lengths) if self.lengths is not None else self.B

    @property
    def total_tokens(self) -> int:
        return self.B * self.T

    @property
    def cu_seqlens(self):
        if self.lengths is None:
            return None
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int64)

    def seq_bounds(self):
        """(bos, eos) of every sequence over the packed token axis."""
        if self.lengths is None:
            return [(b * self.T, (b + 1) * self.T) for b in range(self.B)]
        cu = self.cu_seqlens
        return [(int(cu[i]), int(cu[i + 1])) for i in range(len(cu) - 1)]


def make(name, B, T, H, *, lengths=None, state_dtype="fp32", init="none", final=True,
         lower_bound=-5.0, scale=1.0 / math.sqrt(128.0), seed=0, threads=None, HV=None,
         g_dtype="bf16") -> Workload:
    if lengths is not None:
        assert B == 1
        T = int(sum(lengths))
    HV = H if HV is None else int(HV)
    assert HV >= H and HV % H == 0 and g_dtype in ("bf16", "fp32")
    w = Workload(name, B, T, H, list(lengths) if lengths is not None else None, state_dtype,
                 init, final, float(lower_bound), float(scale), int(seed), HV=HV,
                 g_dtype=g_dtype)
    s = w.seed
    for nm in ("q", "k"):
        w.tensors[nm] = normal_bf16((B, T, H, KD), s, _STREAMS[nm], threads=threads)
    w.tensors["v"] = normal_bf16((B, T, HV, KD), s, _STREAMS["v"], threads=threads)
    if g_dtype == "fp32":
        w.tensors["g"] = normal_f32((B, T, HV, KD), s, _STREAMS["g"], threads=threads)
    else:
        w.tensors["g"] = normal_bf16((B, T, HV, KD), s, _STREAMS["g"], threads=threads)
    w.tensors["beta"] = normal_bf16((B, T, HV), s, _STREAMS["beta"], threads=threads)
    w.tensors["A_log"] = normal_f32((HV,), s, _STREAMS["A_log"])
    w.tensors["dt_bias"] = normal_f32((HV, KD), s, _STREAMS["dt_bias"])
    N = w.N
    if init == "randn":
        st = normal_f32((N, HV, KD, KD), s, _STREAMS["init"], scale=0.1, threads=threads)
        w.tensors["initial_state"] = f32_to_bf16_bits(st) if state_dtype == "bf16" else st
    elif init == "zero":
        z = np.zeros((N, HV, KD, KD), dtype=np.float32)
        w.tensors["initial_state"] = f32_to_bf16_bits(z) if state_dtype == "bf16" else z
    else:
        w.tensors["initial_state"] = None
    return w


# The five seeded workloads (seed = workload index, starting at 0).
def tiny_ref(**kw):
    return make("tiny_ref_B1_T64_H2", 1, 64, 2, state_dtype="fp32", init="none", final=True,
                lower_bound=-5.0, scale=1.0 / math.sqrt(128.0), seed=0, **kw)


def batched_small(**kw):
    return make("batched_small_B2_T256_H16", 2, 256, 16, state_dtype="fp32", init="randn",
                final=True, lower_bound=-3.0, scale=0.125, seed=1, **kw)


def prefill(B=8, T=4096, H=32, seed=2, **kw):
    return make(f"prefill_B{B}_T{T}_H{H}", B, T, H, state_dtype="fp32", init="zero",
                final=True, lower_bound=-5.0, scale=1.0 / math.sqrt(128.0), seed=seed, **kw)


VARLEN_LENGTHS = [1023, 1025, 1, 17, 4096, 65537, 2048, 333]


def irregular_varlen(lengths=None, H=16, **kw):
    return make("irregular_varlen_H16_N8", 1, 0, H, lengths=lengths or VARLEN_LENGTHS,
                state_dtype="bf16", init="randn", final=True, lower_bound=-5.0,
                scale=1.0 / math.sqrt(128.0), seed=3, **kw)


LONGSEQ_LENGTHS = [65536, 1024, 1024, 1024, 1024, 1024]


def long_sequence(lengths=None, H=8, **kw):
    return make("long_seq_segment_scan_H8", 1, 0, H, lengths=lengths or LONGSEQ_LENGTHS,
                state_dtype="fp32", init="zero", final=True, lower_bound=-5.0,
                scale=1.0 / math.sqrt(128.0), seed=4, **kw)
