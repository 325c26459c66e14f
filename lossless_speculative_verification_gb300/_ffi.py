"""ctypes binding of liblsv.so (the C ABI in include/lsv.h).

Argument marshalling only.  If the compiled library is missing this module
raises; there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "liblsv.so")

STATUS = {
    0: "LSV_OK", 1: "LSV_ERR_INVALID_ARG", 2: "LSV_ERR_UNSUPPORTED", 3: "LSV_ERR_MISALIGNED",
    4: "LSV_ERR_WORKSPACE", 5: "LSV_ERR_CUDA", 6: "LSV_ERR_TIMEOUT", 7: "LSV_ERR_DEVICE_INDEX",
}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE_INDEX = range(8)

# Every function the header declares, with its ctypes signature.
P = ctypes.c_void_p
I32 = ctypes.c_int32
SZ = ctypes.c_size_t
U64 = ctypes.c_uint64


class MoeShape(ctypes.Structure):
    _fields_ = [("T", I32), ("H", I32), ("E", I32), ("k", I32), ("S", I32), ("I", I32)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("w_router", P), ("w_gate_up", P), ("w_down", P), ("ws_gate_up", P), ("ws_down", P)]


class DraftWeights(ctypes.Structure):
    _fields_ = [("emb", P), ("w_proj", P), ("w_q", P), ("w_k", P), ("w_v", P), ("w_o", P), ("w_gate_up", P),
                ("w_down", P), ("w_vocab", P)]


SHAPE_P = ctypes.POINTER(MoeShape)
WEIGHTS_P = ctypes.POINTER(MoeWeights)
DRAFT_P = ctypes.POINTER(DraftWeights)

SIGNATURES = {
    "lsv_workspace_size": (SZ, [SHAPE_P]),
    "moe_prefetch_weights": (I32, [WEIGHTS_P, SHAPE_P, SZ, P]),
    "moe_route": (I32, [P, P, SHAPE_P, P, P, P, P]),
    "moe_permute": (I32, [P, SHAPE_P, P, P, P, P, P, SZ, P]),
    "moe_grouped_ffn": (I32, [P, P, P, P, WEIGHTS_P, SHAPE_P, P, P, P, SZ, P]),
    "moe_combine": (I32, [P, P, P, P, SHAPE_P, P, P]),
    "moe_verify_layer": (I32, [P, WEIGHTS_P, SHAPE_P, P, P, P, P, SZ, P]),
    "spec_verify_workspace_size": (SZ, [I32, I32, I32]),
    "spec_verify_accept": (I32, [P, P, I32, I32, I32, P, P, P, P, SZ, P]),
    "spec_verify_accept_noalloc": (I32, [P, P, I32, I32, I32, P, P, P, P]),
    "spec_verify_lmhead_workspace_size": (SZ, [I32, I32, I32, I32]),
    "spec_verify_attention_workspace_size": (SZ, [I32, I32, I32, I32, I32]),
    "spec_k_policy": (I32, [P, I32, P, P, P, P]),
    "dense_matmul": (I32, [P, P, P, I32, I32, I32, P]),
    "spec_draft_workspace_size": (SZ, [I32, I32, I32, I32, I32, I32]),
    "dense_swiglu": (I32, [P, P, P, I32, I32, I32, P]),
    "lsv_gather_rows": (I32, [P, P, I32, I32, I32, P, P]),
    "spec_cache_append": (I32, [P, P, P, P, P, I32, I32, I32, I32, P]),
    "spec_draft_loop": (I32, [DRAFT_P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, I32, P, P, P, SZ, P]),
    "spec_accept_histogram": (I32, [P, I32, I32, P, P]),
    "spec_cond_accept_from_histogram": (I32, [P, I32, P]),
    "spec_verify_attention": (I32, [P, P, P, P, I32, I32, I32, I32, I32, ctypes.c_float, P, P, SZ, P]),
    "spec_verify_lmhead": (I32, [P, P, P, I32, I32, I32, I32, P, P, P, P, SZ, P]),
    "rmsnorm_residual": (I32, [P, P, P, I32, I32, ctypes.c_float, P]),
    "lsv_get_device_error": (I32, [ctypes.POINTER(I32), P]),
    "lsv_set_wait_limit_ns": (I32, [U64]),
    "lsv_selftest_wait_timeout": (I32, [U64, P]),
    "lsv_status_string": (ctypes.c_char_p, [I32]),
    "lsv_version": (I32, []),
}

_lock = threading.Lock()
_lib = None


class LsvError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__("%s returned %s (%d)" % (fn, STATUS.get(code, "?"), code))


def load() -> ctypes.CDLL:
    """Load liblsv.so; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("liblsv.so not built (%s); run __graft_entry__.build() first" % LIB_PATH)
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


def check(fn: str, code: int) -> None:
    if code != OK:
        raise LsvError(fn, code)
