"""ctypes binding of libkvq.so (the C ABI declared in include/kvq.h).

Argument marshalling only. The shared library is loaded from this package directory on first
use; if it is missing the import of a function raises, so no call can silently fall back to
anything else.
"""
from __future__ import annotations

import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvq.so")

KVQ_Q4_0, KVQ_Q6_0, KVQ_HAD_INT4, KVQ_ASYM4_G32, KVQ_Q8_0, KVQ_HAD_INT2 = 0, 1, 2, 3, 4, 5
KVQ_F32, KVQ_BF16, KVQ_F16 = 0, 1, 2
LAYOUT_IDS = {"q4_0": KVQ_Q4_0, "q6_0": KVQ_Q6_0, "had_int4": KVQ_HAD_INT4, "asym4_g32": KVQ_ASYM4_G32,
              "q8_0": KVQ_Q8_0, "had_int2": KVQ_HAD_INT2}
HADAMARD_IDS = (KVQ_HAD_INT4, KVQ_HAD_INT2)


def mixed(k: int, v: int) -> int:
    """KVQ_MIXED(k, v) of include/kvq.h: K plane in layout k, V plane in layout v."""
    return k | ((v + 1) << 8)


def plane_ids(layout: int):
    """(K layout, V layout) of a layout value (plain or mixed)."""
    k = layout & 0xFF
    return k, ((layout >> 8) - 1) if layout >> 8 else k
STATUS_NAMES = {0: "KVQ_OK", 1: "KVQ_EINVAL", 2: "KVQ_ESHAPE", 3: "KVQ_ECAPACITY", 4: "KVQ_EUNSUPPORTED",
                5: "KVQ_EALIGN", 6: "KVQ_ECUDA", 7: "KVQ_EWORKSPACE"}

# Every symbol the header declares (checked by the CPU test suite).
EXPORTS = ("kvq_row_bytes", "kvq_cache_bytes", "kvq_store_q4_0", "kvq_store_q6_0", "kvq_store_hadamard_int4",
           "kvq_store_asym4_g32", "kvq_attend_workspace_bytes", "kvq_decode_attend", "kvq_debug_scores_i32",
           "kvq_status_string", "kvq_last_error", "kvq_profile_phase1_events",
           "kvq_attend_chunk", "kvq_decode_attend_static", "kvq_append_decode_attend",
           "kvq_paged_cache_bytes", "kvq_paged_store", "kvq_paged_attend_workspace_bytes", "kvq_paged_attend_chunk",
           "kvq_paged_decode_attend", "kvq_paged_append_decode_attend", "kvq_store_q8_0", "kvq_store_hadamard_int2",
           "kvq_store", "kvq_paged_attend_plan_chunk", "kvq_append_decode_attend_host_workspace_bytes",
           "kvq_append_decode_attend_host", "kvq_paged_append_decode_attend_host_workspace_bytes",
           "kvq_paged_append_decode_attend_host", "kvq_debug_attend_scores_i32")
STATIC_SCRATCH_BYTES = 16 * 1024 * 1024   # KVQ_STATIC_SCRATCH_BYTES in include/kvq.h


class KvqCache(C.Structure):
    _fields_ = [("layout", C.c_int32), ("batch", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("capacity", C.c_int32), ("n_recent", C.c_int32),
                ("k_payload", C.c_void_p), ("v_payload", C.c_void_p),
                ("k_scale", C.c_void_p), ("v_scale", C.c_void_p),
                ("k_zero", C.c_void_p), ("v_zero", C.c_void_p),
                ("k_recent", C.c_void_p), ("v_recent", C.c_void_p)]


class KvqPagedCache(C.Structure):
    _fields_ = [("layout", C.c_int32), ("batch", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("page_size", C.c_int32), ("n_pages", C.c_int32), ("max_pages_per_seq", C.c_int32),
                ("n_recent", C.c_int32),
                ("k_payload", C.c_void_p), ("v_payload", C.c_void_p),
                ("k_scale", C.c_void_p), ("v_scale", C.c_void_p),
                ("k_zero", C.c_void_p), ("v_zero", C.c_void_p),
                ("k_recent", C.c_void_p), ("v_recent", C.c_void_p),
                ("block_table", C.c_void_p)]


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({detail})")


_lib = None


def lib() -> C.CDLL:
    """Load libkvq.so once and declare the prototypes."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    L = C.CDLL(LIB_PATH)
    P, I32, SZ = C.c_void_p, C.c_int32, C.c_size_t
    cache_p = C.POINTER(KvqCache)
    L.kvq_row_bytes.argtypes, L.kvq_row_bytes.restype = [I32, I32], SZ
    L.kvq_cache_bytes.argtypes, L.kvq_cache_bytes.restype = [I32, I32, I32, I32, I32, I32, C.POINTER(SZ)], I32
    for name in ("kvq_store_q4_0", "kvq_store_q6_0", "kvq_store_hadamard_int4", "kvq_store_asym4_g32",
                 "kvq_store_q8_0", "kvq_store_hadamard_int2", "kvq_store"):
        f = getattr(L, name)
        f.argtypes, f.restype = [cache_p, P, P, I32, I32, I32, P], I32
    L.kvq_attend_workspace_bytes.argtypes = [cache_p, I32, I32, I32, I32]
    L.kvq_attend_workspace_bytes.restype = SZ
    L.kvq_attend_chunk.argtypes, L.kvq_attend_chunk.restype = [cache_p, I32, I32, I32, I32], I32
    L.kvq_decode_attend.argtypes = [cache_p, P, I32, I32, I32, I32, I32, I32, C.c_float, I32, P, P, SZ, P]
    L.kvq_decode_attend.restype = I32
    L.kvq_append_decode_attend.argtypes = [cache_p, P, P, I32, I32, I32, P, I32, I32, I32, I32, I32, I32, C.c_float,
                                           I32, P, P, SZ, P]
    L.kvq_append_decode_attend.restype = I32
    L.kvq_decode_attend_static.argtypes = [cache_p, P, I32, I32, I32, I32, I32, I32, C.c_float, I32, P, P]
    L.kvq_decode_attend_static.restype = I32
    L.kvq_debug_scores_i32.argtypes = [cache_p, P, I32, I32, I32, I32, P, P, P]
    L.kvq_debug_scores_i32.restype = I32
    L.kvq_debug_attend_scores_i32.argtypes = [cache_p, P, I32, I32, I32, I32, I32, I32, C.c_float, I32, P, P, SZ, P, P,
                                              P]
    L.kvq_debug_attend_scores_i32.restype = I32
    paged_p = C.POINTER(KvqPagedCache)
    L.kvq_paged_cache_bytes.argtypes = [I32, I32, I32, I32, I32, I32, I32, C.POINTER(SZ)]
    L.kvq_paged_cache_bytes.restype = I32
    L.kvq_paged_store.argtypes, L.kvq_paged_store.restype = [paged_p, P, P, I32, I32, P, P], I32
    L.kvq_paged_attend_workspace_bytes.argtypes = [paged_p, I32, I32, I32, I32]
    L.kvq_paged_attend_workspace_bytes.restype = SZ
    L.kvq_paged_attend_chunk.argtypes = [paged_p, I32, I32, I32, C.c_int64, I32]
    L.kvq_paged_attend_chunk.restype = I32
    L.kvq_paged_attend_plan_chunk.argtypes = [paged_p, I32, I32, I32, P]
    L.kvq_paged_attend_plan_chunk.restype = I32
    L.kvq_paged_decode_attend.argtypes = [paged_p, P, I32, I32, I32, P, I32, I32, C.c_float, I32, P, P, SZ, P]
    L.kvq_paged_decode_attend.restype = I32
    L.kvq_paged_append_decode_attend.argtypes = [paged_p, P, P, I32, I32, P, I32, I32, I32, P, I32, I32, C.c_float,
                                                 I32, P, P, SZ, P]
    L.kvq_paged_append_decode_attend.restype = I32
    L.kvq_append_decode_attend_host_workspace_bytes.argtypes = [cache_p, I32, I32, I32, I32, I32, I32, I32]
    L.kvq_append_decode_attend_host_workspace_bytes.restype = SZ
    L.kvq_append_decode_attend_host.argtypes = L.kvq_append_decode_attend.argtypes
    L.kvq_append_decode_attend_host.restype = I32
    L.kvq_paged_append_decode_attend_host_workspace_bytes.argtypes = [paged_p, I32, I32, I32, I32, I32, I32, I32]
    L.kvq_paged_append_decode_attend_host_workspace_bytes.restype = SZ
    L.kvq_paged_append_decode_attend_host.argtypes = L.kvq_paged_append_decode_attend.argtypes
    L.kvq_paged_append_decode_attend_host.restype = I32
    L.kvq_status_string.argtypes, L.kvq_status_string.restype = [I32], C.c_char_p
    L.kvq_last_error.argtypes, L.kvq_last_error.restype = [], C.c_char_p
    L.kvq_profile_phase1_events.argtypes, L.kvq_profile_phase1_events.restype = [P, P], I32
    _lib = L
    return L


def check(status: int, where: str) -> None:
    if status != 0:
        raise KvqError(status, where, lib().kvq_last_error().decode())
