"""CPU oracle for the MoE token-movement path with a paged activation stash.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package.  The
product library never calls it, and it shares no code with the CUDA sources.

The arithmetic lives in ``ap_oracle.c`` (plain single-threaded C compiled with
``-ffp-contract=off``); this module only compiles it and marshals numpy arrays.
Every function cites, in the C source, the page and section it follows:

* torchtitan pull 5541 (HybridEP eager scheduling with a paged stash),
  "AI-Generated Details" and "Verification";
* torchtitan pull 5542, "[graph_trainer] Overlap HybridEP and paging across
  combined PP graphs";
* Megatron-LM pull 7342, token-wise ChunkedEP for Qwen3 MoE;
* OpenPipe/ART pull 971, "Price HybridEP recompute outputs at the live
  communication extent".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ap_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libap_oracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, EEMPTY, EQFULL = 0, -1, -2, -3
FLAG_POOL_OVERFLOW = 0x1
FLAG_SPILL_OVERFLOW = 0x2
FLAG_RECORD_OVERFLOW = 0x4
FLAG_BAD_COUNT = 0x8
FLAG_BAD_INDEX = 0x10


def build(force: bool = False) -> str:
    """Compile the oracle into ``libap_oracle.so`` next to its source."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i32, i64, u8 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint8
        sig = {
            "or_route_topk": (i32, [P, i64, i32, i32, P, P]),
            "or_dispatch_plan": (i32, [P, i64, i32, i32, i32, i32, P, P, P, P, P, i64, P]),
            "or_permute_rows": (None, [P, i64, i64, P, i32, P]),
            "or_e4m3_encode": (u8, [ctypes.c_float]),
            "or_e4m3_decode": (ctypes.c_double, [u8]),
            "or_e4m3_encode_n": (None, [P, i64, P]),
            "or_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
            "or_quantize_rows_e4m3": (None, [P, i64, i32, P, P]),
            "or_permute_rows_fp8": (None, [P, P, i64, i32, P, i32, P, P]),
            "or_combine": (None, [P, i64, i32, P, P, i64, i32, P, P]),
            "or_combine_backward": (None, [P, P, i64, i32, P, P, i64, i32, P, P, P]),
            "or_dispatch_backward": (None, [P, i64, i32, P, i64, i32, P, P]),
            "or_pool_new": (P, [i32, i64, i64, i32, i32, i32, i64, i64, i32, u8, i64]),
            "or_pool_grow": (i32, [P, i64]),
            "or_pool_free": (None, [P]),
            "or_pool_reset": (None, [P]),
            "or_pool_push": (i32, [P, i32, i32, P, P, i64, i32, P, P, P]),
            "or_pool_pop": (i32, [P, i32, i32, P, i64, P]),
            "or_pool_state": (None, [P, P, P, P]),
            "or_pool_rings": (None, [P, P, P]),
            "or_pool_queue_len": (i32, [P, i32]),
            "or_pool_record": (i32, [P, i32, i32, P, P, P, P, i64]),
            "or_pool_bytes": (P, [P]),
            "or_pool_spill_bytes": (P, [P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _chk(rc: int, what: str):
    if rc != OK:
        raise OracleError(rc, what)


class OracleError(RuntimeError):
    def __init__(self, rc: int, what: str):
        super().__init__(f"oracle {what}: status {rc}")
        self.rc = rc


# --------------------------------------------------------------------------
# route / dispatch / combine
# --------------------------------------------------------------------------
def route_topk(logits: np.ndarray, k: int):
    """softmax -> top-k (ties to the lower expert) -> renormalised weights."""
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    _chk(_load().or_route_topk(_ptr(logits), T, E, k, _ptr(idx), _ptr(w)), "route_topk")
    return idx, w


def capacity_rows(cf: float, T: int, k: int, E: int) -> int:
    """Rows per expert for a capacity factor: ceil(cf * T * k / E)."""
    num = cf * T * k
    c = int(num // E)
    if c * E < num:
        c += 1
    return c


def dispatch_plan(idx: np.ndarray, E: int, capacity: int, padded: bool):
    """counts, live, seg_off, dest, src_tok (rows never written hold -1), status."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    live = np.empty(E, np.int32)
    seg_off = np.empty(E, np.int32)
    dest = np.empty((T, k), np.int32)
    rows = E * capacity if padded else T * k
    src_tok = np.full(max(rows, 1), -1, np.int32)
    status = np.zeros(1, np.uint32)
    _chk(_load().or_dispatch_plan(_ptr(idx), T, k, E, capacity, int(padded), _ptr(counts), _ptr(live),
                                  _ptr(seg_off), _ptr(dest), _ptr(src_tok), rows, _ptr(status)),
         "dispatch_plan")
    return dict(counts=counts, live=live, seg_off=seg_off, dest=dest, src_tok=src_tok[:rows],
                rows=rows, status=int(status[0]))


def permute_rows(x: np.ndarray, dest: np.ndarray, out: np.ndarray) -> np.ndarray:
    """out[dest[t, j]] = x[t] byte-for-byte for every kept pair (in place)."""
    x = np.ascontiguousarray(x)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    T, k = dest.shape
    rb = x.nbytes // max(T, 1) if T else 0
    assert out.flags["C_CONTIGUOUS"] and out.dtype == x.dtype
    _load().or_permute_rows(_ptr(x), T, rb, _ptr(dest), k, _ptr(out))
    return out


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32).ravel()
    out = np.empty(v.size, np.uint8)
    _load().or_e4m3_encode_n(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode_one(c: int) -> float:
    return _load().or_e4m3_decode(c)


def f32_to_bf16_one(f: float) -> int:
    return _load().or_f32_to_bf16(f)


def quantize_rows_e4m3(x_bf16: np.ndarray):
    """Per-row amax scaling to E4M3; returns (codes uint8 [T,H], scale f32 [T])."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T, H = x.shape
    q = np.empty((T, H), np.uint8)
    s = np.empty(T, np.float32)
    _load().or_quantize_rows_e4m3(_ptr(x), T, H, _ptr(q), _ptr(s))
    return q, s


def permute_rows_fp8(q, scale, dest, xd, xd_scale):
    T, H = q.shape
    k = dest.shape[1]
    _load().or_permute_rows_fp8(_ptr(q), _ptr(scale), T, H, _ptr(np.ascontiguousarray(dest, np.int32)), k,
                                _ptr(xd), _ptr(xd_scale))
    return xd, xd_scale


def combine(y_bf16: np.ndarray, dest: np.ndarray, w: np.ndarray):
    """out[t] = bf16(sum_j w[t,j] * y[dest[t,j]]) with single-precision mul/add, j ascending."""
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    T, k = dest.shape
    H = y.shape[1]
    out = np.empty((T, H), np.uint16)
    status = np.zeros(1, np.uint32)
    _load().or_combine(_ptr(y), y.shape[0], H, _ptr(dest), _ptr(w), T, k, _ptr(out), _ptr(status))
    return out, int(status[0])


def combine_backward(dout_bf16: np.ndarray, y_bf16: np.ndarray, dest: np.ndarray, w: np.ndarray,
                     dy_fill: int = 0xA5):
    """dy rows (BF16(w * dout), canary elsewhere), dw [T, k] f32 and status."""
    dout = np.ascontiguousarray(dout_bf16, dtype=np.uint16)
    y = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    T, k = dest.shape
    H = y.shape[1]
    dy = np.frombuffer(np.full(y.size * 2, dy_fill, np.uint8).tobytes(), np.uint16).reshape(y.shape).copy()
    dw = np.empty((T, k), np.float32)
    status = np.zeros(1, np.uint32)
    _load().or_combine_backward(_ptr(dout), _ptr(y), y.shape[0], H, _ptr(dest), _ptr(w), T, k, _ptr(dy), _ptr(dw),
                                _ptr(status))
    return dy, dw, int(status[0])


def dispatch_backward(dxd_bf16: np.ndarray, dest: np.ndarray):
    """dx[t] = BF16(sum_j dxd[dest[t, j]]) with single-precision accumulation."""
    dxd = np.ascontiguousarray(dxd_bf16, dtype=np.uint16)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    T, k = dest.shape
    H = dxd.shape[1]
    dx = np.empty((T, H), np.uint16)
    status = np.zeros(1, np.uint32)
    _load().or_dispatch_backward(_ptr(dxd), dxd.shape[0], H, _ptr(dest), T, k, _ptr(dx), _ptr(status))
    return dx, int(status[0])


def dispatch(x_bf16: np.ndarray, idx: np.ndarray, E: int, capacity: int, padded: bool,
             fp8: bool = False, fill: int = 0xA5):
    """Whole dispatch step: plan + permuted payload (BF16 bytes, or E4M3 + scale).

    Rows never written are pre-filled with the byte ``fill`` (a canary)."""
    plan = dispatch_plan(idx, E, capacity, padded)
    T, H = x_bf16.shape
    R = plan["rows"]
    if fp8:
        q, s = quantize_rows_e4m3(x_bf16)
        xd = np.full((R, H), fill, np.uint8)
        xs = np.frombuffer(np.full(R * 4, fill, np.uint8).tobytes(), np.float32).copy()
        permute_rows_fp8(q, s, plan["dest"], xd, xs)
        plan["xd"], plan["xd_scale"] = xd, xs
    else:
        xd = np.frombuffer(np.full(R * H * 2, fill, np.uint8).tobytes(), np.uint16).reshape(R, H).copy()
        permute_rows(np.ascontiguousarray(x_bf16, np.uint16), plan["dest"], xd)
        plan["xd"] = xd
    return plan


# --------------------------------------------------------------------------
# paged stash
# --------------------------------------------------------------------------
class Pool:
    """Byte-exact simulation of the page pool, free lists, records and flags.

    ``keep_bytes=False`` keeps metadata only (page tables, rings, flags), for
    sizes whose byte image would not fit the host.  ``max_num_pages``: the
    most device pages ``grow`` may reach (0: ``num_pages``, a pool that never
    grows); spill page ids start there.  ``num_pages`` may be 0 then (a
    calibration pool with no device pages yet)."""

    def __init__(self, page_tokens: int, page_bytes: int, num_pages: int, num_slots: int,
                 max_records_per_slot: int, max_segments: int, max_pages_per_record: int,
                 spill_pages: int = 0, keep_bytes: bool = True, fill: int = 0xA5, max_num_pages: int = 0):
        self.lib = _load()
        self.P, self.page_bytes, self.N = page_tokens, page_bytes, num_pages
        self.NMAX = max_num_pages or num_pages
        self.SP, self.S, self.R = spill_pages, num_slots, max_records_per_slot
        self.max_pages = max_pages_per_record
        self.keep_bytes = keep_bytes
        self.h = self.lib.or_pool_new(page_tokens, page_bytes, num_pages, num_slots, max_records_per_slot,
                                      max_segments, max_pages_per_record, spill_pages, int(keep_bytes), fill,
                                      max_num_pages)
        if not self.h:
            raise OracleError(EINVAL, "pool_new")

    def grow(self, num_pages: int):
        """Add device pages up to num_pages (see or_pool_grow)."""
        _chk(self.lib.or_pool_grow(self.h, num_pages), "grow")
        self.N = num_pages

    def close(self):
        if self.h:
            self.lib.or_pool_free(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self):
        self.lib.or_pool_reset(self.h)

    def push(self, slot: int, planes, src_rows: int, seg_off, live) -> int:
        """planes: list of 2-D C-contiguous numpy arrays (rows first)."""
        nplanes = len(planes)
        arrs = [np.ascontiguousarray(p) for p in planes]
        ptrs = (ctypes.c_void_p * 2)(*[a.ctypes.data for a in arrs] + [None] * (2 - nplanes))
        rb = np.zeros(2, np.int64)
        for i, a in enumerate(arrs):
            rb[i] = a.nbytes // a.shape[0] if a.shape[0] else a.dtype.itemsize * int(np.prod(a.shape[1:]))
        seg_off = np.ascontiguousarray(seg_off, np.int32)
        live = np.ascontiguousarray(live, np.int32)
        rid = ctypes.c_uint64(0)
        rc = self.lib.or_pool_push(self.h, slot, nplanes, ctypes.cast(ptrs, ctypes.c_void_p), _ptr(rb), src_rows,
                                   int(seg_off.size), _ptr(seg_off), _ptr(live), ctypes.byref(rid))
        _chk(rc, "push")
        return rid.value

    def push_rb(self, slot: int, row_bytes, src_rows: int, seg_off, live) -> int:
        """Metadata-only push (no source bytes): row_bytes per plane."""
        assert not self.keep_bytes
        rb = np.zeros(2, np.int64)
        rb[: len(row_bytes)] = row_bytes
        seg_off = np.ascontiguousarray(seg_off, np.int32)
        live = np.ascontiguousarray(live, np.int32)
        rid = ctypes.c_uint64(0)
        ptrs = (ctypes.c_void_p * 2)(None, None)
        rc = self.lib.or_pool_push(self.h, slot, len(row_bytes), ctypes.cast(ptrs, ctypes.c_void_p), _ptr(rb),
                                   src_rows, int(seg_off.size), _ptr(seg_off), _ptr(live), ctypes.byref(rid))
        _chk(rc, "push")
        return rid.value

    def pop(self, slot: int, planes=None, dst_rows: int = 0, nplanes: int | None = None) -> int:
        """planes: list of destination numpy arrays (modified in place), or None (metadata only)."""
        rid = ctypes.c_uint64(0)
        if planes is None:
            rc = self.lib.or_pool_pop(self.h, slot, nplanes or 1, None, dst_rows, ctypes.byref(rid))
        else:
            for a in planes:
                assert a.flags["C_CONTIGUOUS"]
            ptrs = (ctypes.c_void_p * 2)(*[a.ctypes.data for a in planes] + [None] * (2 - len(planes)))
            rc = self.lib.or_pool_pop(self.h, slot, len(planes), ctypes.cast(ptrs, ctypes.c_void_p), dst_rows,
                                      ctypes.byref(rid))
        _chk(rc, "pop")
        return rid.value

    def state(self):
        ctr = np.zeros(4, np.uint64)
        flags = np.zeros(1, np.uint32)
        hw = np.zeros(5, np.int64)
        self.lib.or_pool_state(self.h, _ptr(ctr), _ptr(flags), _ptr(hw))
        return dict(head=int(ctr[0]), tail=int(ctr[1]), spill_head=int(ctr[2]), spill_tail=int(ctr[3]),
                    flags=int(flags[0]), high_water=int(hw[0]), spill_high_water=int(hw[1]),
                    held=int(hw[2]), held_high_water=int(hw[3]), num_pages=int(hw[4]))

    def rings(self):
        ring = np.empty(self.N, np.int32)
        sring = np.empty(max(self.SP, 1), np.int32)
        self.lib.or_pool_rings(self.h, _ptr(ring), _ptr(sring))
        return ring, sring[: self.SP]

    def queue_len(self, slot: int) -> int:
        return self.lib.or_pool_queue_len(self.h, slot)

    def record(self, slot: int, qpos: int = 0):
        info = np.zeros(6, np.int64)
        pt = np.empty(self.max_pages, np.int32)
        r0 = np.empty(self.max_pages, np.int64)
        nr = np.empty(self.max_pages, np.int32)
        _chk(self.lib.or_pool_record(self.h, slot, qpos, _ptr(info), _ptr(pt), _ptr(r0), _ptr(nr), self.max_pages),
             "record")
        n = int(info[1])
        return dict(id=int(info[0]), npages=n, ndev=int(info[2]), nspill=int(info[3]), nlost=int(info[4]),
                    nseg=int(info[5]), page_table=pt[:n].copy(), row0=r0[:n].copy(), nrows=nr[:n].copy())

    def pool_bytes(self) -> np.ndarray:
        assert self.keep_bytes
        addr = self.lib.or_pool_bytes(self.h)
        return np.ctypeslib.as_array((ctypes.c_uint8 * (self.N * self.page_bytes)).from_address(addr))

    def spill_bytes(self) -> np.ndarray:
        assert self.keep_bytes
        if self.SP == 0:
            return np.zeros(0, np.uint8)
        addr = self.lib.or_pool_spill_bytes(self.h)
        return np.ctypeslib.as_array((ctypes.c_uint8 * (self.SP * self.page_bytes)).from_address(addr))


def page_plane_offset(page_tokens: int, row_bytes0: int) -> int:
    """Byte offset of plane 1 inside a page: plane 0 rounded up to 16 bytes."""
    return (page_tokens * row_bytes0 + 15) // 16 * 16
