"""ctypes view of the C ABI in include/kda.h (argument marshalling only).

Loading fails loudly when libkda.so has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = range(5)
KDA_BF16, KDA_F32 = 0, 1
STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_CUDA",
                4: "KDA_ERR_TIMEOUT"}
ABI_VERSION = 5

# every symbol include/kda.h declares
EXPORTS = ("kda_fwd", "kda_fwd_workspace_size", "kda_saved_size", "kda_bwd", "kda_bwd_workspace_size",
           "kda_step", "kda_cp_combine", "kda_fwd_cp", "kda_fwd_cp_workspace_size", "kda_attnres_fwd", "kda_attnres_bwd", "kda_attnres_bwd_workspace_size",
           "kda_conv_fwd", "kda_conv_bwd", "kda_conv_bwd_workspace_size", "kda_conv_step",
           "kda_fwd_no_alloc", "kda_set_profile_events", "kda_last_error", "kda_abi_version")
ATTNRES_MAX_SOURCES = 9
CONV_MAX_WIDTH = 4
KDA_ACT_NONE, KDA_ACT_SILU = 0, 1
NO_ALLOC_SCRATCH_BYTES = 256 * 1024 * 1024


class FwdArgs(C.Structure):
    _fields_ = [
        ("n_seqs", C.c_int32), ("total_tokens", C.c_int64), ("heads", C.c_int32),
        ("dk", C.c_int32), ("dv", C.c_int32), ("chunk", C.c_int32), ("scale", C.c_float),
        ("io_dtype", C.c_int32), ("cu_seqlens", C.c_void_p),
        ("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p), ("beta", C.c_void_p), ("g", C.c_void_p),
        ("h0", C.c_void_p), ("o", C.c_void_p), ("hT", C.c_void_p), ("saved", C.c_void_p),
        ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t), ("dev_status", C.c_void_p),
        ("h0_identity", C.c_int32), ("skip_prep", C.c_int32),
        ("wait_limit_ns", C.c_int64), ("debug_starve", C.c_int32),
    ]


class FwdCpArgs(C.Structure):
    _fields_ = [("fwd", FwdArgs), ("n_segments", C.c_int32), ("workspace", C.c_void_p),
                ("workspace_bytes", C.c_size_t)]


class CpArgs(C.Structure):
    _fields_ = [
        ("n_seqs", C.c_int32), ("n_segments", C.c_int32), ("heads", C.c_int32), ("dk", C.c_int32), ("dv", C.c_int32),
        ("M", C.c_void_p), ("b", C.c_void_p), ("h0", C.c_void_p), ("s_in", C.c_void_p),
    ]


class AttnresFwdArgs(C.Structure):
    _fields_ = [
        ("n_sources", C.c_int32), ("tokens", C.c_int64), ("dim", C.c_int32), ("eps", C.c_float),
        ("io_dtype", C.c_int32), ("src", C.c_void_p * ATTNRES_MAX_SOURCES), ("w", C.c_void_p), ("out", C.c_void_p),
        ("alpha", C.c_void_p), ("rstd", C.c_void_p), ("logit", C.c_void_p),
    ]


class AttnresBwdArgs(C.Structure):
    _fields_ = [
        ("fwd", AttnresFwdArgs), ("d_out", C.c_void_p), ("d_src", C.c_void_p * ATTNRES_MAX_SOURCES),
        ("dw", C.c_void_p), ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
    ]


class ConvArgs(C.Structure):
    _fields_ = [
        ("n_seqs", C.c_int32), ("total_tokens", C.c_int64), ("channels", C.c_int32), ("width", C.c_int32),
        ("activation", C.c_int32), ("io_dtype", C.c_int32), ("cu_seqlens", C.c_void_p),
        ("x", C.c_void_p), ("weight", C.c_void_p), ("bias", C.c_void_p), ("state_in", C.c_void_p),
        ("y", C.c_void_p), ("state_out", C.c_void_p),
    ]


class ConvBwdArgs(C.Structure):
    _fields_ = [
        ("fwd", ConvArgs), ("dy", C.c_void_p), ("d_state_out", C.c_void_p), ("dx", C.c_void_p),
        ("dweight", C.c_void_p), ("dbias", C.c_void_p), ("d_state_in", C.c_void_p),
        ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
    ]


class ConvStepArgs(C.Structure):
    _fields_ = [
        ("n_seqs", C.c_int32), ("steps", C.c_int32), ("channels", C.c_int32), ("width", C.c_int32),
        ("activation", C.c_int32), ("io_dtype", C.c_int32),
        ("x", C.c_void_p), ("weight", C.c_void_p), ("bias", C.c_void_p), ("state", C.c_void_p),
        ("state_indices", C.c_void_p), ("n_slots", C.c_int32), ("accept_len", C.c_void_p),
        ("first_slot", C.c_void_p), ("y", C.c_void_p), ("dev_status", C.c_void_p),
    ]


class BwdArgs(C.Structure):
    _fields_ = [
        ("fwd", FwdArgs), ("dO", C.c_void_p), ("dhT", C.c_void_p),
        ("dq", C.c_void_p), ("dk", C.c_void_p), ("dv", C.c_void_p), ("dbeta", C.c_void_p), ("dg", C.c_void_p),
        ("dh0", C.c_void_p), ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
    ]


class StepArgs(C.Structure):
    _fields_ = [
        ("n_seqs", C.c_int32), ("steps", C.c_int32), ("heads", C.c_int32), ("dk", C.c_int32), ("dv", C.c_int32),
        ("scale", C.c_float), ("io_dtype", C.c_int32),
        ("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p), ("beta", C.c_void_p), ("g", C.c_void_p),
        ("state", C.c_void_p), ("accept_len", C.c_void_p), ("o", C.c_void_p),
        ("state_indices", C.c_void_p), ("n_slots", C.c_int32), ("first_slot", C.c_void_p),
        ("dev_status", C.c_void_p),
    ]


class KdaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH):
    """Load libkda.so (once). Raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                          "or `python gated_delta_rule_chunked_gb300/build.py` (no CPU fallback exists)")
    lib = C.CDLL(path)
    lib.kda_fwd.argtypes = [C.POINTER(FwdArgs), C.c_void_p]
    lib.kda_fwd.restype = C.c_int
    lib.kda_bwd.argtypes = [C.POINTER(BwdArgs), C.c_void_p]
    lib.kda_bwd.restype = C.c_int
    lib.kda_step.argtypes = [C.POINTER(StepArgs), C.c_void_p]
    lib.kda_step.restype = C.c_int
    lib.kda_cp_combine.argtypes = [C.POINTER(CpArgs), C.c_void_p]
    lib.kda_cp_combine.restype = C.c_int
    lib.kda_fwd_cp.argtypes = [C.POINTER(FwdCpArgs), C.c_void_p]
    lib.kda_fwd_cp.restype = C.c_int
    lib.kda_fwd_cp_workspace_size.argtypes = [C.POINTER(FwdCpArgs)]
    lib.kda_fwd_cp_workspace_size.restype = C.c_size_t
    lib.kda_attnres_fwd.argtypes = [C.POINTER(AttnresFwdArgs), C.c_void_p]
    lib.kda_attnres_fwd.restype = C.c_int
    lib.kda_attnres_bwd.argtypes = [C.POINTER(AttnresBwdArgs), C.c_void_p]
    lib.kda_attnres_bwd.restype = C.c_int
    lib.kda_attnres_bwd_workspace_size.argtypes = [C.POINTER(AttnresBwdArgs)]
    lib.kda_attnres_bwd_workspace_size.restype = C.c_size_t
    lib.kda_conv_fwd.argtypes = [C.POINTER(ConvArgs), C.c_void_p]
    lib.kda_conv_fwd.restype = C.c_int
    lib.kda_conv_bwd.argtypes = [C.POINTER(ConvBwdArgs), C.c_void_p]
    lib.kda_conv_bwd.restype = C.c_int
    lib.kda_conv_bwd_workspace_size.argtypes = [C.POINTER(ConvBwdArgs)]
    lib.kda_conv_bwd_workspace_size.restype = C.c_size_t
    lib.kda_conv_step.argtypes = [C.POINTER(ConvStepArgs), C.c_void_p]
    lib.kda_conv_step.restype = C.c_int
    lib.kda_fwd_workspace_size.argtypes = [C.POINTER(FwdArgs)]
    lib.kda_fwd_workspace_size.restype = C.c_size_t
    lib.kda_saved_size.argtypes = [C.POINTER(FwdArgs)]
    lib.kda_saved_size.restype = C.c_size_t
    lib.kda_bwd_workspace_size.argtypes = [C.POINTER(BwdArgs)]
    lib.kda_bwd_workspace_size.restype = C.c_size_t
    lib.kda_last_error.argtypes = []
    lib.kda_last_error.restype = C.c_char_p
    lib.kda_fwd_no_alloc.argtypes = [C.POINTER(FwdArgs), C.c_void_p]
    lib.kda_fwd_no_alloc.restype = C.c_int
    lib.kda_set_profile_events.argtypes = [C.c_void_p, C.c_int32]
    lib.kda_set_profile_events.restype = None
    lib.kda_abi_version.argtypes = []
    lib.kda_abi_version.restype = C.c_int32
    if lib.kda_abi_version() != ABI_VERSION:
        raise ImportError(f"libkda.so ABI {lib.kda_abi_version()} != binding ABI {ABI_VERSION}; rebuild")
    _lib = lib
    return lib


def check(status: int):
    if status != KDA_OK:
        raise KdaError(status, load().kda_last_error().decode())
