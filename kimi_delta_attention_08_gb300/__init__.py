"""GB300 (sm_103a) Kimi Delta Attention forward: Python binding of libkda.

The binding only marshals arguments: it checks that each tensor already has the
dtype, device and layout the C ABI documents (it never converts), reads the
sizes off the shapes, and calls the entry point of the same name in
include/kda.h.  Every step of the computation runs in the library's kernels.
"""
from __future__ import annotations

import ctypes

from . import _lib

__all__ = ["KdaError", "kda_fwd", "kda_bwd", "kda_fwd_transition", "kda_compose_states",
           "kda_get_workspace_size", "kda_get_device_status", "make_workspace",
           "make_bwd_workspace", "make_chunk_states", "kda_get_chunk_states_size",
           "status_string", "CP_MODES", "PATHS"]

KDA_OK = 0
CP_MODES = {"auto": 0, "off": 1, "force": 2, None: 0, True: 2, False: 1}
# kernel choice: chunked (WY) form, or the token-by-token recurrence for short inputs
PATHS = {"auto": 0, "chunked": 1, "recurrent": 2}
STATE_FP32, STATE_BF16 = 0, 1
GATE_BF16, GATE_FP32 = 0, 1


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def status_string(status: int) -> str:
    return _lib.load().kda_status_string(int(status)).decode()


def kda_get_workspace_size(total_tokens: int, H: int) -> int:
    n = ctypes.c_size_t(0)
    st = _lib.load().kda_get_workspace_size(int(total_tokens), int(H), ctypes.byref(n))
    if st != KDA_OK:
        raise KdaError(st, "kda_get_workspace_size")
    return int(n.value)


def make_workspace(total_tokens: int, H: int, device=None):
    """Workspace for kda_fwd; H is the number of value heads (v's head count)."""
    import torch
    return torch.empty(kda_get_workspace_size(total_tokens, H), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def kda_get_chunk_states_size(total_tokens: int, N: int, HV: int) -> int:
    n = ctypes.c_size_t(0)
    st = _lib.load().kda_get_chunk_states_size(int(total_tokens), int(N), int(HV), ctypes.byref(n))
    if st != KDA_OK:
        raise KdaError(st, "kda_get_chunk_states_size")
    return int(n.value)


def make_chunk_states(total_tokens: int, N: int, HV: int, device=None):
    """Buffer for the chunk start states that kda_fwd(..., chunk_states=buf) writes
    and kda_bwd(..., chunk_states=buf) reads (include/kda.h, kda_options)."""
    import torch
    return torch.empty(kda_get_chunk_states_size(total_tokens, N, HV), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def _set_chunk_states(opts, buf, dev):
    if buf is None:
        return
    import torch
    _need(buf, "chunk_states", torch.uint8, dev, 1)
    opts.chunk_states = buf.data_ptr()
    opts.chunk_states_bytes = buf.numel()


def _need(t, name, dtype, device, ndim=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype} (no implicit conversion)")
    if t.device != device:
        raise ValueError(f"{name}: expected device {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous (no implicit copy)")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: expected {ndim} dims, got shape {tuple(t.shape)}")


def kda_fwd(q, k, v, g, beta, scale, out, A_log, dt_bias, lower_bound, initial_state=None,
            final_state=None, cu_seqlens=None, workspace=None, *, cp_mode="auto",
            seg_chunks: int = 0, path="auto", stream=None, debug_stall: int = 0,
            chunk_states=None) -> None:
    """Enqueue the KDA forward (see include/kda.h, kda_fwd) on `stream`
    (default: torch's current stream).  `out` and `final_state` are written, and
    with chunk_states (make_chunk_states) every chunk's start state for kda_bwd.

    q, k: [B, T, H, 128] bf16; v, out: [B, T, HV, 128] bf16 with HV a multiple of
    H (grouped value heads when HV > H); g: [B, T, HV, 128] bf16 or float32;
    beta [B, T, HV]; A_log [HV]; dt_bias [HV, 128]; states [N, HV, 128, 128]."""
    import torch
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q: must be a CUDA tensor")
    bf16, f32 = torch.bfloat16, torch.float32
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _need(t, nm, bf16, dev, 4)
    if g.dtype not in (bf16, f32):
        raise TypeError(f"g: expected bfloat16 or float32, got {g.dtype} (no implicit conversion)")
    _need(g, "g", g.dtype, dev, 4)
    B, T, H, D = q.shape
    HV = v.shape[2]
    if tuple(k.shape) != (B, T, H, D):
        raise ValueError(f"k: shape {tuple(k.shape)} != q's {(B, T, H, D)}")
    if HV < H or HV % H != 0:
        raise ValueError(f"v: {HV} value heads is not a multiple of q's {H} heads")
    for t, nm in ((v, "v"), (g, "g"), (out, "out")):
        if tuple(t.shape) != (B, T, HV, D):
            raise ValueError(f"{nm}: shape {tuple(t.shape)} != {(B, T, HV, D)}")
    _need(beta, "beta", bf16, dev, 3)
    if tuple(beta.shape) != (B, T, HV):
        raise ValueError(f"beta: shape {tuple(beta.shape)} != {(B, T, HV)}")
    _need(A_log, "A_log", f32, dev, 1)
    _need(dt_bias, "dt_bias", f32, dev, 2)
    if tuple(A_log.shape) != (HV,) or tuple(dt_bias.shape) != (HV, D):
        raise ValueError("A_log must be [HV] and dt_bias [HV, 128]")
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int64, dev, 1)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    sdt = None
    for t, nm in ((initial_state, "initial_state"), (final_state, "final_state")):
        if t is None:
            continue
        if sdt is None:
            sdt = t.dtype
        if t.dtype not in (f32, bf16) or t.dtype != sdt:
            raise TypeError(f"{nm}: states must both be float32 or both bfloat16")
        _need(t, nm, sdt, dev, 4)
        if tuple(t.shape) != (N, HV, D, D):
            raise ValueError(f"{nm}: expected shape {(N, HV, D, D)}, got {tuple(t.shape)}")
    if workspace is None:
        raise ValueError("workspace: required (make_workspace(B*T, HV) allocates one)")
    _need(workspace, "workspace", torch.uint8, dev, 1)
    opts = _lib.kda_options()
    if cp_mode not in CP_MODES:
        raise ValueError(f"cp_mode must be one of {list(CP_MODES)}")
    opts.cp_mode = CP_MODES[cp_mode]
    opts.seg_chunks = int(seg_chunks)
    if path not in PATHS:
        raise ValueError(f"path must be one of {list(PATHS)}")
    opts.path = PATHS[path]
    opts.num_v_heads = HV if HV != H else 0
    opts.g_dtype = GATE_FP32 if g.dtype == f32 else GATE_BF16
    opts.debug_stall = int(debug_stall)  # timeout tests only (see include/kda.h)
    _set_chunk_states(opts, chunk_states, dev)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = _lib.load().kda_fwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(out), _ptr(A_log),
        _ptr(dt_bias), float(lower_bound), _ptr(initial_state), _ptr(final_state),
        _ptr(cu_seqlens), B, T, H, N, STATE_BF16 if sdt == bf16 else STATE_FP32,
        _ptr(workspace), workspace.numel(), ctypes.byref(opts), ctypes.c_void_p(sh))
    if st != KDA_OK:
        raise KdaError(st, "kda_fwd")


def kda_fwd_transition(q, k, v, g, beta, A_log, dt_bias, lower_bound, M_out, B_out,
                       cu_seqlens=None, workspace=None, *, stream=None) -> None:
    """Enqueue the affine form of the forward over each sequence (include/kda.h,
    kda_fwd_transition): M_out / B_out (float32 [N, HV, 128, 128]) receive the
    transition and the offset, S_end = M S_start + B, in the state layout."""
    import torch
    dev = q.device
    bf16, f32 = torch.bfloat16, torch.float32
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, nm, bf16, dev, 4)
    if g.dtype not in (bf16, f32):
        raise TypeError(f"g: expected bfloat16 or float32, got {g.dtype} (no implicit conversion)")
    _need(g, "g", g.dtype, dev, 4)
    B, T, H, D = q.shape
    HV = v.shape[2]
    if tuple(k.shape) != (B, T, H, D) or HV < H or HV % H != 0:
        raise ValueError("k must match q, and v's heads must be a multiple of q's")
    for t, nm in ((v, "v"), (g, "g")):
        if tuple(t.shape) != (B, T, HV, D):
            raise ValueError(f"{nm}: shape {tuple(t.shape)} != {(B, T, HV, D)}")
    _need(beta, "beta", bf16, dev, 3)
    _need(A_log, "A_log", f32, dev, 1)
    _need(dt_bias, "dt_bias", f32, dev, 2)
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int64, dev, 1)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    for t, nm in ((M_out, "M_out"), (B_out, "B_out")):
        _need(t, nm, f32, dev, 4)
        if tuple(t.shape) != (N, HV, D, D):
            raise ValueError(f"{nm}: expected shape {(N, HV, D, D)}, got {tuple(t.shape)}")
    if workspace is None:
        raise ValueError("workspace: required (make_workspace(B*T, HV) allocates one)")
    _need(workspace, "workspace", torch.uint8, dev, 1)
    opts = _lib.kda_options()
    opts.num_v_heads = HV if HV != H else 0
    opts.g_dtype = GATE_FP32 if g.dtype == f32 else GATE_BF16
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = _lib.load().kda_fwd_transition(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(A_log), _ptr(dt_bias),
        float(lower_bound), _ptr(cu_seqlens), B, T, H, N, _ptr(M_out), _ptr(B_out),
        _ptr(workspace), workspace.numel(), ctypes.byref(opts), ctypes.c_void_p(sh))
    if st != KDA_OK:
        raise KdaError(st, "kda_fwd_transition")


def kda_compose_states(M, B, S_out, S_in=None, *, stream=None) -> None:
    """Enqueue S_out = fold of X <- X M[r] + B[r] from X = S_in (zero if None)
    (include/kda.h, kda_compose_states).  M, B: float32 [R, *state_shape]; S_in,
    S_out: float32 state_shape = [..., 128, 128]."""
    import torch
    dev = S_out.device
    f32 = torch.float32
    _need(M, "M", f32, dev)
    _need(B, "B", f32, dev)
    _need(S_out, "S_out", f32, dev)
    if S_in is not None:
        _need(S_in, "S_in", f32, dev)
        if S_in.shape != S_out.shape:
            raise ValueError("S_in and S_out must have the same shape")
    if tuple(M.shape) != tuple(B.shape) or tuple(M.shape[1:]) != tuple(S_out.shape):
        raise ValueError("M and B must be [R, *S_out.shape]")
    if S_out.shape[-2:] != (128, 128):
        raise ValueError("states must end in [128, 128]")
    R = M.shape[0]
    ns = S_out.numel() // (128 * 128)
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = _lib.load().kda_compose_states(_ptr(M), _ptr(B), int(R), int(ns), _ptr(S_in),
                                        _ptr(S_out), ctypes.c_void_p(sh))
    if st != KDA_OK:
        raise KdaError(st, "kda_compose_states")


def make_bwd_workspace(total_tokens: int, N: int, H: int, HV: int = 0, device=None):
    """Workspace for kda_bwd (H: q/k heads, HV: value heads, 0 = H)."""
    import torch
    n = ctypes.c_size_t(0)
    st = _lib.load().kda_bwd_get_workspace_size(int(total_tokens), int(N), int(H), int(HV),
                                                ctypes.byref(n))
    if st != KDA_OK:
        raise KdaError(st, "kda_bwd_get_workspace_size")
    return torch.empty(int(n.value), dtype=torch.uint8,
                       device=device if device is not None else "cuda")


def kda_bwd(q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, dout, initial_state=None,
            dfinal_state=None, cu_seqlens=None, workspace=None, *, path="auto", stream=None,
            debug_stall: int = 0, chunk_states=None):
    """Enqueue the backward pass (include/kda.h, kda_bwd) for the forward call with
    the same inputs, given dout (bf16, out's shape) and optionally the gradient of
    the final state.  Returns a dict of fp32 gradients dq, dk, dv, dg, dbeta,
    dA_log, ddt_bias and dinitial_state (allocated here with torch).
    path: "auto" / "chunked" (tensor cores, bf16 operands) or "recurrent" (token
    by token, fp32).  chunk_states: the buffer that a kda_fwd of the same inputs
    filled (chunked path); the backward then skips its own state-checkpoint pass."""
    import torch
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("q: must be a CUDA tensor")
    bf16, f32 = torch.bfloat16, torch.float32
    for t, nm in ((q, "q"), (k, "k"), (v, "v"), (dout, "dout")):
        _need(t, nm, bf16, dev, 4)
    if g.dtype not in (bf16, f32):
        raise TypeError(f"g: expected bfloat16 or float32, got {g.dtype} (no implicit conversion)")
    _need(g, "g", g.dtype, dev, 4)
    B, T, H, D = q.shape
    HV = v.shape[2]
    if tuple(k.shape) != (B, T, H, D) or HV < H or HV % H != 0:
        raise ValueError("k must match q, and v's heads must be a multiple of q's")
    for t, nm in ((v, "v"), (g, "g"), (dout, "dout")):
        if tuple(t.shape) != (B, T, HV, D):
            raise ValueError(f"{nm}: shape {tuple(t.shape)} != {(B, T, HV, D)}")
    _need(beta, "beta", bf16, dev, 3)
    _need(A_log, "A_log", f32, dev, 1)
    _need(dt_bias, "dt_bias", f32, dev, 2)
    if tuple(beta.shape) != (B, T, HV) or tuple(A_log.shape) != (HV,) or \
            tuple(dt_bias.shape) != (HV, D):
        raise ValueError("beta must be [B, T, HV], A_log [HV] and dt_bias [HV, 128]")
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int64, dev, 1)
        N = cu_seqlens.numel() - 1
    else:
        N = B
    sdt = None
    for t, nm in ((initial_state, "initial_state"), (dfinal_state, "dfinal_state")):
        if t is None:
            continue
        if sdt is None:
            sdt = t.dtype
        if t.dtype not in (f32, bf16) or t.dtype != sdt:
            raise TypeError(f"{nm}: states must both be float32 or both bfloat16")
        _need(t, nm, sdt, dev, 4)
        if tuple(t.shape) != (N, HV, D, D):
            raise ValueError(f"{nm}: expected shape {(N, HV, D, D)}, got {tuple(t.shape)}")
    if workspace is None:
        workspace = make_bwd_workspace(B * T, N, H, HV, dev)
    _need(workspace, "workspace", torch.uint8, dev, 1)
    grads = {"dq": torch.empty((B, T, H, D), dtype=f32, device=dev),
             "dk": torch.empty((B, T, H, D), dtype=f32, device=dev),
             "dv": torch.empty((B, T, HV, D), dtype=f32, device=dev),
             "dg": torch.empty((B, T, HV, D), dtype=f32, device=dev),
             "dbeta": torch.empty((B, T, HV), dtype=f32, device=dev),
             "dA_log": torch.empty((HV,), dtype=f32, device=dev),
             "ddt_bias": torch.empty((HV, D), dtype=f32, device=dev),
             "dinitial_state": torch.empty((N, HV, D, D), dtype=f32, device=dev)}
    opts = _lib.kda_options()
    opts.num_v_heads = HV if HV != H else 0
    opts.g_dtype = GATE_FP32 if g.dtype == f32 else GATE_BF16
    opts.path = PATHS[path]
    opts.debug_stall = int(debug_stall)  # timeout tests only (see include/kda.h)
    _set_chunk_states(opts, chunk_states, dev)  # states a kda_fwd of these inputs wrote
    if stream is None:
        stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    G = grads
    st = _lib.load().kda_bwd(
        _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(A_log), _ptr(dt_bias),
        float(lower_bound), _ptr(initial_state), _ptr(dout), _ptr(dfinal_state), _ptr(cu_seqlens),
        _ptr(G["dq"]), _ptr(G["dk"]), _ptr(G["dv"]), _ptr(G["dg"]), _ptr(G["dbeta"]),
        _ptr(G["dA_log"]), _ptr(G["ddt_bias"]), _ptr(G["dinitial_state"]), B, T, H, N,
        STATE_BF16 if sdt == bf16 else STATE_FP32, _ptr(workspace), workspace.numel(),
        ctypes.byref(opts), ctypes.c_void_p(sh))
    if st != KDA_OK:
        raise KdaError(st, "kda_bwd")
    grads["workspace"] = workspace
    return grads


def kda_get_device_status(workspace, stream=None) -> int:
    """Status word of the last kda_fwd that used `workspace` (synchronises)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(workspace.device)
    sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    out = ctypes.c_int(0)
    st = _lib.load().kda_get_device_status(_ptr(workspace), ctypes.byref(out), ctypes.c_void_p(sh))
    if st != KDA_OK:
        raise KdaError(st, "kda_get_device_status")
    return int(out.value)
