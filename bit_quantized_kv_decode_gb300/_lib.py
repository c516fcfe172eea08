"""ctypes view of libkvq.so (the C-ABI declared in include/kvq.h)."""
from __future__ import annotations

import ctypes
import os

from . import build as _build

KVQ_OK = 0
STATUS_NAMES = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "workspace too small",
                4: "CUDA error", 5: "no sm_103 device"}

DEV_BAD_SEQ_LEN = 0x1
DEV_BAD_PAGE = 0x2
DEV_NONFINITE = 0x4
DEV_TIMEOUT = 0x8

TOKENWISE = 0
CHANNELWISE = 1
OPERANDS_FP8 = 0
OPERANDS_BF16 = 1
FLAG_TEST_STALL = 0x1
FLAG_TEST_STALL_MMA = 0x4
FLAG_E2M1_V = 0x2
PATH_SPECIALISED = 0
PATH_GENERAL = 1

# Every symbol include/kvq.h declares.
EXPORTS = ("kvq_status_string", "kvq_version", "kvq_cache_bytes", "kvq_pack", "kvq_append", "kvq_dequant",
           "kvq_decode_workspace_size", "kvq_decode_path", "kvq_decode_attn", "kvq_decode_attn_static", "kvq_merge")


class CacheDesc(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("k_scheme", ctypes.c_int32), ("v_scheme", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("group_size", ctypes.c_int32)]


class AttnDesc(ctypes.Structure):
    _fields_ = [("cache", CacheDesc), ("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("operand_mode", ctypes.c_int32), ("sm_scale", ctypes.c_float),
                ("num_ctas", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class KvqError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} (status {status})")
        self.status = status


_LIB = None


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libkvq.so; raise if it has not been built (there is no fallback)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or lib_path()
    if not os.path.exists(p):
        raise RuntimeError(f"libkvq.so not found at {p}; build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    P, I32, U32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
    lib.kvq_status_string.restype = ctypes.c_char_p
    lib.kvq_status_string.argtypes = [I32]
    lib.kvq_version.restype = I32
    lib.kvq_version.argtypes = []
    lib.kvq_cache_bytes.restype = I32
    lib.kvq_cache_bytes.argtypes = [ctypes.POINTER(CacheDesc), ctypes.POINTER(SZ), ctypes.POINTER(SZ)]
    lib.kvq_pack.restype = I32
    lib.kvq_pack.argtypes = [ctypes.POINTER(CacheDesc), I32, P, I32, I32, P, P, I32, P, P, P, P, P]
    lib.kvq_append.restype = I32
    lib.kvq_append.argtypes = [ctypes.POINTER(CacheDesc), I32, P, I32, P, P, I32, P, P, P, P, P, P]
    lib.kvq_dequant.restype = I32
    lib.kvq_dequant.argtypes = [ctypes.POINTER(CacheDesc), I32, P, P, P, I32, I32, P, P, I32, P, P, P]
    lib.kvq_decode_workspace_size.restype = I32
    lib.kvq_decode_workspace_size.argtypes = [ctypes.POINTER(AttnDesc), ctypes.POINTER(SZ)]
    lib.kvq_decode_path.restype = I32
    lib.kvq_decode_path.argtypes = [ctypes.POINTER(AttnDesc), ctypes.POINTER(I32)]
    lib.kvq_decode_attn.restype = I32
    lib.kvq_decode_attn.argtypes = [ctypes.POINTER(AttnDesc), P, P, P, P, P, P, P, P, P, P, P, P, SZ, P, P]
    lib.kvq_decode_attn_static.restype = I32
    lib.kvq_decode_attn_static.argtypes = [ctypes.POINTER(AttnDesc), P, P, P, P, P, P, P, P, P, P, P, P, P]
    lib.kvq_merge.restype = I32
    lib.kvq_merge.argtypes = [P, P, I32, I32, I32, P, P, P]
    _ = U32
    if path is None:
        _LIB = lib
    return lib


def check(status: int, what: str) -> None:
    if status != KVQ_OK:
        raise KvqError(status, what)
