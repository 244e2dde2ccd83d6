"""ctypes loader for the in-tree libkda.so.  Fails loudly when it is missing:
there is no fallback implementation."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkda.so")

# Public symbols of include/kda.h.
EXPORTS = ("kda_status_string", "kda_get_workspace_size", "kda_fwd", "kda_get_device_status",
           "kda_fwd_static_scratch", "kda_static_scratch_device_status",
           "kda_fwd_transition", "kda_compose_states", "kda_bwd_get_workspace_size", "kda_bwd",
           "kda_get_chunk_states_size")

_lib = None


class kda_options(ctypes.Structure):
    _fields_ = [("cp_mode", ctypes.c_int32), ("seg_chunks", ctypes.c_int32),
                ("path", ctypes.c_int32), ("num_v_heads", ctypes.c_int32),
                ("g_dtype", ctypes.c_int32), ("debug_stall", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 2), ("chunk_states", ctypes.c_void_p),
                ("chunk_states_bytes", ctypes.c_size_t)]


def load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libkda.so not found at {LIB_PATH}; build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_get_workspace_size.restype = ctypes.c_int
    lib.kda_get_workspace_size.argtypes = [I64, I32, ctypes.POINTER(ctypes.c_size_t)]
    lib.kda_fwd.restype = ctypes.c_int
    lib.kda_fwd.argtypes = [P, P, P, P, P, F, P, P, P, F, P, P, P, I64, I64, I32, I32, I32, P,
                            ctypes.c_size_t, ctypes.POINTER(kda_options), P]
    lib.kda_fwd_static_scratch.restype = ctypes.c_int
    lib.kda_fwd_static_scratch.argtypes = [P, P, P, P, P, F, P, P, P, F, P, P, P, I64, I64, I32,
                                           I32, I32, ctypes.POINTER(kda_options), P]
    lib.kda_get_chunk_states_size.restype = ctypes.c_int
    lib.kda_get_chunk_states_size.argtypes = [I64, I32, I32, ctypes.POINTER(ctypes.c_size_t)]
    lib.kda_bwd_get_workspace_size.restype = ctypes.c_int
    lib.kda_bwd_get_workspace_size.argtypes = [I64, I32, I32, I32, ctypes.POINTER(ctypes.c_size_t)]
    lib.kda_bwd.restype = ctypes.c_int
    lib.kda_bwd.argtypes = ([P, P, P, P, P, F, P, P, F, P, P, P, P] + [P] * 8 +
                            [I64, I64, I32, I32, I32, P, ctypes.c_size_t,
                             ctypes.POINTER(kda_options), P])
    lib.kda_get_device_status.restype = ctypes.c_int
    lib.kda_get_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_int), P]
    lib.kda_fwd_transition.restype = ctypes.c_int
    lib.kda_fwd_transition.argtypes = [P, P, P, P, P, P, P, F, P, I64, I64, I32, I32, P, P, P,
                                       ctypes.c_size_t, ctypes.POINTER(kda_options), P]
    lib.kda_compose_states.restype = ctypes.c_int
    lib.kda_compose_states.argtypes = [P, P, I32, I64, P, P, P]
    lib.kda_static_scratch_device_status.restype = ctypes.c_int
    lib.kda_static_scratch_device_status.argtypes = [ctypes.POINTER(ctypes.c_int), P]
    _lib = lib
    return lib
