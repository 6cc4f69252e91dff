"""ctypes declarations of ``libap.so`` (the C ABI in ``include/ap.h``).

Loading fails loudly when the library has not been built: there is no other
implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libap.so")

P = ctypes.c_void_p
i32, i64, u32, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_uint64


class PoolConfig(ctypes.Structure):
    _fields_ = [("page_tokens", i32), ("num_slots", i32), ("page_bytes", i64), ("num_pages", i64),
                ("spill_pages", i64), ("max_records_per_slot", i32), ("max_segments", i32),
                ("max_pages_per_record", i64), ("max_ctas", i32), ("reserved", i32), ("max_num_pages", i64)]


class PoolState(ctypes.Structure):
    _fields_ = [("head", u64), ("tail", u64), ("spill_head", u64), ("spill_tail", u64), ("flags", u32),
                ("copy_done", u32), ("high_water", i64), ("spill_high_water", i64), ("held", i64),
                ("held_high_water", i64), ("num_pages", i64), ("pad", i64 * 6)]


class RecordInfo(ctypes.Structure):
    _fields_ = [("record_id", u64), ("slot", i32), ("nseg", i32), ("npages", i64), ("ndev", i64),
                ("nspill", i64), ("nlost", i64)]


# name -> (restype, argtypes); every ap_* symbol the header declares
SIGNATURES = {
    "ap_status_str": (ctypes.c_char_p, [i32]),
    "ap_last_error": (ctypes.c_char_p, []),
    "ap_version": (ctypes.c_char_p, []),
    "ap_launch_count": (ctypes.c_uint64, []),
    "ap_route_topk": (i32, [P, i64, i32, i32, P, P, P]),
    "ap_dispatch_scratch_bytes": (i32, [i64, i32, i32, P]),
    "ap_dispatch_permute": (i32, [P, i64, i32, P, i32, i32, i32, i32, i32, P, P, i64, P, P, P, P, P, P, i64, P, P]),
    "ap_dispatch_permute_noalloc": (i32, [P, i64, i32, P, i32, i32, i32, i32, i32, P, P, i64, P, P, P, P, P, P, P]),
    "ap_combine_unpermute": (i32, [P, i64, i32, P, P, i64, i32, P, P, P]),
    "ap_combine_backward": (i32, [P, P, i64, i32, P, P, i64, i32, P, P, P, P]),
    "ap_dispatch_backward": (i32, [P, i64, i32, P, i64, i32, P, P, P]),
    "ap_pool_required_bytes": (i32, [P, P, P, P]),
    "ap_pool_init": (i32, [P, P, P, P, P, P]),
    "ap_pool_reset": (i32, [P, P]),
    "ap_pool_grow": (i32, [P, i64, P, P]),
    "ap_pool_destroy": (i32, [P]),
    "ap_pool_max_ctas": (i32, [P, P]),
    "ap_pool_set_max_ctas": (i32, [P, i32]),
    "ap_stash_push": (i32, [P, i32, i32, P, P, i64, i32, P, P, P, P]),
    "ap_stash_pop": (i32, [P, i32, i32, P, i64, P, P]),
    "ap_dispatch_stash": (i32, [P, i32, P, i64, i32, P, i32, i32, i32, i32, i32, P, P, i64, P, P, P, P, P, P, i64, P,
                                P, P]),
    "ap_dispatch_stash_ranked": (i32, [P, i32, P, i64, i32, P, i32, i32, i32, i32, i32, P, P, i64, P, P, P, P, P, P,
                                       i64, P, P, i32, P]),
    "ap_count_rank": (i32, [P, P, P, i64, i32, i32, P, i64, P, P, i64, i32, i32, P, P, P, P, P]),
    "ap_pool_time_copies": (i32, [P, P, P]),
    "ap_route_dispatch_stash": (i32, [P, i32, P, P, P, i64, i32, P, i32, i32, i32, i32, i32, P, P, i64, P, P, P, P,
                                      P, P, i64, P, P, P]),
    "ap_pool_queue_len": (i32, [P, i32, P]),
    "ap_pool_flags_device_ptr": (i32, [P, P]),
    "ap_overflow_query": (i32, [P, P, i32]),
    "ap_pool_read_state": (i32, [P, P]),
    "ap_pool_stats": (i32, [P, P, P, P, i32]),
    "ap_pool_read_rings": (i32, [P, P, P]),
    "ap_pool_read_record": (i32, [P, i32, i32, P, P, P, P, i64]),
    "ap_cast_e4m3": (i32, [P, P, i64, P]),
    "ap_arena_create": (i32, [P, i64, i32]),
    "ap_arena_grow": (i32, [P, i64]),
    "ap_arena_info": (i32, [P, P, P, P]),
    "ap_arena_destroy": (i32, [P]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build the CUDA library first "
                           "(python -m activation_paging_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class APError(RuntimeError):
    def __init__(self, status: int, what: str):
        lib = load()
        name = lib.ap_status_str(status).decode()
        msg = lib.ap_last_error().decode()
        super().__init__(f"{what}: {name} ({status}): {msg}")
        self.status = status


def check(status: int, what: str) -> None:
    if status != 0:
        raise APError(status, what)
