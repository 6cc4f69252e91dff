"""GB300 token movement for a top-k MoE layer with a paged activation stash.

Thin Python binding of ``libap.so`` (C ABI in ``include/ap.h``).  Every step
runs in the library's CUDA kernels; this module only allocates tensors with
PyTorch (device memory, pinned host memory, streams) and passes their
addresses.  There is no CPU fallback: without the built library every call
raises.

    route_topk        softmax -> top-k -> renormalised weights
    dispatch_permute  expert-major, capacity-bounded permutation (BF16 / E4M3)
    Pool              paged stash: push / pop / reset / overflow read-out,
                      calibration and lazy growth (over an Arena)
    Arena             device memory that grows in place
    combine_unpermute top-k weighted un-permute to dense BF16 [T, H]
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import APError, PoolConfig, PoolState, RecordInfo, check

FLAG_POOL_OVERFLOW = 0x1
FLAG_SPILL_OVERFLOW = 0x2
FLAG_RECORD_OVERFLOW = 0x4
FLAG_BAD_COUNT = 0x8
FLAG_BAD_INDEX = 0x10
FLAG_CORRUPT = 0x20
DTYPE_BF16, DTYPE_E4M3 = 0, 1

__all__ = ["route_topk", "dispatch_permute", "dispatch_scratch_bytes", "combine_unpermute", "combine_backward",
           "dispatch_backward", "cast_e4m3", "Pool", "Arena", "APError", "lib", "launch_count"]


def lib():
    return _lib.load()


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _p(t):
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def route_topk(logits: torch.Tensor, k: int, idx: torch.Tensor | None = None, w: torch.Tensor | None = None,
               stream=None):
    """idx [T, k] int32 and w [T, k] float32 for float32 logits [T, E]."""
    _need(logits, torch.float32, "logits")
    T, E = logits.shape
    if idx is None:
        idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if w is None:
        w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    check(lib().ap_route_topk(_p(logits), T, E, k, _p(idx), _p(w), _stream(stream)), "route_topk")
    return idx, w


def launch_count() -> int:
    """Kernels the library has enqueued in this process (a graph replay adds none)."""
    return int(lib().ap_launch_count())


def dispatch_scratch_bytes(T: int, k: int, E: int) -> int:
    n = ctypes.c_int64(0)
    check(lib().ap_dispatch_scratch_bytes(T, k, E, ctypes.byref(n)), "dispatch_scratch_bytes")
    return n.value


def count_rank(E: int, idx: torch.Tensor | None = None, logits: torch.Tensor | None = None, k: int | None = None,
               x: torch.Tensor | None = None, out: dict | None = None, status: torch.Tensor | None = None,
               stream=None, scan: bool = False, capacity: int = 0, padded: bool = False) -> dict:
    """Count/rank alone (``ap_count_rank``) on ``stream`` (default: the
    current stream): ``dest`` ([T, k] int32 ranks inside blocks of 64 tokens)
    and ``scratch`` (the blocks' expert histograms), for a later
    ``Pool.dispatch_stash(..., ranked=True, out=...)`` ordered after it.  With
    ``logits`` ([T, E] float32) it routes first and adds ``idx`` and ``w``;
    else ``idx`` is read.  ``x``: the rows the copy will read (an L2
    prefetch hint).  ``scan``: also the dispatch's expert scan for
    ``capacity`` / ``padded`` (adds ``counts``, ``live``, ``seg_off``; the
    scratch then holds block bases, and the dict is marked ``scanned``)."""
    o = dict(out) if out is not None else {}
    if logits is not None:
        _need(logits, torch.float32, "logits")
        T = logits.shape[0]
        dev = logits.device
        if "idx" not in o:
            o["idx"] = torch.empty((T, k), dtype=torch.int32, device=dev)
        if "w" not in o:
            o["w"] = torch.empty((T, k), dtype=torch.float32, device=dev)
        idx = o["idx"]
    else:
        _need(idx, torch.int32, "idx")
        T, k = idx.shape
        dev = idx.device
        o["idx"] = idx
    if "dest" not in o:
        o["dest"] = torch.empty((T, k), dtype=torch.int32, device=dev)
    sb = dispatch_scratch_bytes(T, k, E)
    if "scratch" not in o or o["scratch"].numel() < sb:
        o["scratch"] = torch.empty(sb, dtype=torch.uint8, device=dev)
    if scan:
        for name in ("counts", "live", "seg_off"):
            if name not in o:
                o[name] = torch.empty(E, dtype=torch.int32, device=dev)
    rb = x.shape[1] * x.element_size() if x is not None else 0
    check(lib().ap_count_rank(_p(logits), _p(o.get("w") if logits is not None else None), _p(idx), T, k, E, _p(x), rb,
                              _p(o["dest"]), _p(o["scratch"]), o["scratch"].numel(), capacity, int(padded),
                              _p(o["counts"] if scan else None), _p(o["live"] if scan else None),
                              _p(o["seg_off"] if scan else None), _p(status), _stream(stream)), "count_rank")
    o["scanned"] = scan
    return o


def dispatch_permute(x: torch.Tensor, idx: torch.Tensor, E: int, capacity: int = 0, padded: bool = False,
                     fp8: bool = False, out: dict | None = None, status: torch.Tensor | None = None, stream=None):
    """Permute BF16 rows x [T, H] into expert-major rows.

    Returns a dict with xd ([rows, H] bf16, or uint8 codes), xd_scale (E4M3
    only), counts, live, seg_off ([E] int32), dest ([T, k] int32), src_tok
    ([rows] int32, -1 where never written) and scratch.  Pass ``out`` (such a
    dict) to reuse buffers."""
    _need(x, torch.bfloat16, "x")
    _need(idx, torch.int32, "idx")
    T, H = x.shape
    k = idx.shape[1]
    dev = x.device
    rows = E * capacity if padded else T * k
    o = dict(out) if out is not None else {}
    if "xd" not in o:
        o["xd"] = torch.empty((rows, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    if fp8 and "xd_scale" not in o:
        o["xd_scale"] = torch.empty(rows, dtype=torch.float32, device=dev)
    for name, shape in (("counts", (E,)), ("live", (E,)), ("seg_off", (E,)), ("dest", (T, k))):
        if name not in o:
            o[name] = torch.empty(shape, dtype=torch.int32, device=dev)
    if "src_tok" not in o:
        o["src_tok"] = torch.full((rows,), -1, dtype=torch.int32, device=dev)
    sb = dispatch_scratch_bytes(T, k, E)
    if "scratch" not in o or o["scratch"].numel() < sb:
        o["scratch"] = torch.empty(sb, dtype=torch.uint8, device=dev)
    xd = o["xd"]
    check(lib().ap_dispatch_permute(_p(x), T, H, _p(idx), k, E, capacity, int(padded),
                                    DTYPE_E4M3 if fp8 else DTYPE_BF16, _p(xd), _p(o.get("xd_scale")), xd.shape[0],
                                    _p(o["counts"]), _p(o["live"]), _p(o["seg_off"]), _p(o["dest"]),
                                    _p(o["src_tok"]), _p(o["scratch"]), o["scratch"].numel(), _p(status),
                                    _stream(stream)), "dispatch_permute")
    return o


def combine_unpermute(y: torch.Tensor, dest: torch.Tensor, w: torch.Tensor, out: torch.Tensor | None = None,
                      status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out [T, H] bf16 = sum_j w[t, j] * y[dest[t, j]] (FP32 accumulation)."""
    _need(y, torch.bfloat16, "y")
    _need(dest, torch.int32, "dest")
    _need(w, torch.float32, "w")
    T, k = dest.shape
    H = y.shape[1]
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=y.device)
    check(lib().ap_combine_unpermute(_p(y), y.shape[0], H, _p(dest), _p(w), T, k, _p(out), _p(status),
                                     _stream(stream)), "combine_unpermute")
    return out


def combine_backward(dout: torch.Tensor, y: torch.Tensor, dest: torch.Tensor, w: torch.Tensor,
                     dy: torch.Tensor | None = None, dw: torch.Tensor | None = None,
                     status: torch.Tensor | None = None, stream=None):
    """dy [rows, H] bf16 (rows no pair maps to are left as given) and dw [T, k] f32."""
    _need(dout, torch.bfloat16, "dout")
    _need(y, torch.bfloat16, "y")
    _need(dest, torch.int32, "dest")
    _need(w, torch.float32, "w")
    T, k = dest.shape
    H = y.shape[1]
    if dy is None:
        dy = torch.zeros_like(y)
    if dw is None:
        dw = torch.empty((T, k), dtype=torch.float32, device=y.device)
    check(lib().ap_combine_backward(_p(dout), _p(y), y.shape[0], H, _p(dest), _p(w), T, k, _p(dy), _p(dw),
                                    _p(status), _stream(stream)), "combine_backward")
    return dy, dw


def dispatch_backward(dxd: torch.Tensor, dest: torch.Tensor, dx: torch.Tensor | None = None,
                      status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """dx [T, H] bf16 = sum_j dxd[dest[t, j]] (FP32 accumulation)."""
    _need(dxd, torch.bfloat16, "dxd")
    _need(dest, torch.int32, "dest")
    T, k = dest.shape
    H = dxd.shape[1]
    if dx is None:
        dx = torch.empty((T, H), dtype=torch.bfloat16, device=dxd.device)
    check(lib().ap_dispatch_backward(_p(dxd), dxd.shape[0], H, _p(dest), T, k, _p(dx), _p(status),
                                     _stream(stream)), "dispatch_backward")
    return dx


def cast_e4m3(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _need(x, torch.float32, "x")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    check(lib().ap_cast_e4m3(_p(x), _p(out), x.numel(), _stream(stream)), "cast_e4m3")
    return out


def page_bytes_for(page_tokens: int, row_bytes) -> int:
    """Smallest page (multiple of 256 bytes) holding page_tokens rows of each plane."""
    need = page_tokens * row_bytes[0]
    if len(row_bytes) == 2:
        need = (need + 15) // 16 * 16 + page_tokens * row_bytes[1]
    return (need + 255) // 256 * 256


class Arena:
    """Device memory whose size grows in place (``ap_arena_*``: reserved
    addresses, physical memory mapped on demand).  ``view(n)`` is a uint8
    tensor over the first n bytes; views stay valid while the arena lives."""

    def __init__(self, max_bytes: int, device="cuda"):
        self.lib = lib()
        self.device = torch.device(device)
        self.handle = ctypes.c_void_p()
        check(self.lib.ap_arena_create(ctypes.byref(self.handle), int(max_bytes), self.device.index or 0),
              "arena_create")

    def grow(self, nbytes: int):
        check(self.lib.ap_arena_grow(self.handle, int(nbytes)), "arena_grow")

    def info(self):
        base, mapped, reserved = ctypes.c_void_p(), ctypes.c_int64(), ctypes.c_int64()
        check(self.lib.ap_arena_info(self.handle, ctypes.byref(base), ctypes.byref(mapped), ctypes.byref(reserved)),
              "arena_info")
        return base.value or 0, mapped.value, reserved.value

    def view(self, nbytes: int) -> torch.Tensor:
        base, mapped, _ = self.info()
        if nbytes > mapped:
            raise ValueError(f"{nbytes} bytes requested, {mapped} mapped")
        if nbytes == 0:  # nothing mapped yet: no address to view
            return torch.empty(0, dtype=torch.uint8, device=self.device)
        return torch.as_tensor(_DeviceSpan(base, nbytes, self), device=self.device)

    def close(self):
        if getattr(self, "handle", None) and self.handle.value:
            check(self.lib.ap_arena_destroy(self.handle), "arena_destroy")
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _DeviceSpan:
    """A device byte range in the CUDA array interface (keeps its owner alive)."""

    def __init__(self, ptr: int, nbytes: int, owner):
        self.owner = owner
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (ptr, False),
                                         "version": 3, "strides": None}


class Pool:
    """Paged activation stash over PyTorch-owned memory.

    The device pool, its metadata and the pinned host spill are torch tensors
    held by this object; the library keeps only their addresses.  Every push,
    pop and reset runs on ``self.stream`` (a high-priority stream by
    default).  Order work on other streams with ``stream.wait_stream`` /
    ``self.stream.wait_stream``.

    ``max_num_pages > num_pages`` makes a growable pool: its pages live in an
    :class:`Arena` reserved for ``max_num_pages`` pages and mapped as the pool
    grows (``grow``); ``num_pages`` may then be 0, a calibration pool whose
    pushes park their live prefixes in the spill pages (or lose them) while
    ``state()["held_high_water"]`` measures the device pages the schedule
    needs (``calibrated_pages``)."""

    def __init__(self, page_tokens: int, page_bytes: int, num_pages: int, num_slots: int = 1,
                 max_records_per_slot: int = 8, max_segments: int = 1024, max_pages_per_record: int | None = None,
                 spill_pages: int = 0, max_ctas: int = 0, device="cuda", stream: torch.cuda.Stream | None = None,
                 fill: int | None = None, max_num_pages: int = 0):
        self.lib = lib()
        nmax = max(max_num_pages, num_pages)
        if max_pages_per_record is None:
            max_pages_per_record = nmax + spill_pages
        self.cfg = PoolConfig(page_tokens, num_slots, page_bytes, num_pages, spill_pages, max_records_per_slot,
                              max_segments, max_pages_per_record, max_ctas, 0, max_num_pages)
        a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        check(self.lib.ap_pool_required_bytes(ctypes.byref(self.cfg), ctypes.byref(a), ctypes.byref(b),
                                              ctypes.byref(c)), "pool_required_bytes")
        self.device = torch.device(device)
        self.fill = fill
        self.arena = None
        if nmax > num_pages:
            self.arena = Arena(nmax * page_bytes, self.device)
            self.arena.grow(a.value)
            self.pool = self.arena.view(a.value)
        else:
            self.pool = torch.empty(a.value, dtype=torch.uint8, device=self.device)
        self.meta = torch.empty(b.value, dtype=torch.uint8, device=self.device)
        self.spill = torch.empty(c.value, dtype=torch.uint8, pin_memory=True) if c.value else None
        if fill is not None:
            self.pool.fill_(fill)
            if self.spill is not None:
                self.spill.fill_(fill)
            torch.cuda.synchronize(self.device)
        self.stream = stream if stream is not None else torch.cuda.Stream(device=self.device, priority=-1)
        self.handle = ctypes.c_void_p()
        check(self.lib.ap_pool_init(ctypes.byref(self.handle), ctypes.byref(self.cfg),
                                    _p(self.pool) if num_pages else None, _p(self.meta), _p(self.spill),
                                    self.stream.cuda_stream), "pool_init")
        self.N, self.SP, self.P, self.NMAX = num_pages, spill_pages, page_tokens, nmax
        self.page_bytes = page_bytes
        self.max_pages = max_pages_per_record

    def grow(self, num_pages: int):
        """Grow the device pool to ``num_pages`` in place, with records still
        queued (``ap_pool_grow``).  New pages are filled with ``fill`` when the
        pool was created with one.  Graphs captured before must be captured
        again (they hold the old page count)."""
        if num_pages == self.N:
            return
        if self.arena is None:
            raise ValueError("this pool was created without room to grow (max_num_pages)")
        nbytes = num_pages * self.page_bytes
        self.arena.grow(nbytes)
        pool = self.arena.view(nbytes)
        if self.fill is not None:
            with torch.cuda.stream(self.stream):
                pool[self.N * self.page_bytes:].fill_(self.fill)
        check(self.lib.ap_pool_grow(self.handle, num_pages, self.arena.info()[0], self.stream.cuda_stream),
              "pool_grow")
        self.pool, self.N = pool, num_pages

    def calibrated_pages(self, margin: float = 1.0) -> int:
        """Device pages for the schedule run so far: the most pages its queued
        records ever held, times ``margin`` (synchronises the paging stream)."""
        import math
        return int(math.ceil(self.state()["held_high_water"] * margin))

    # -- lifecycle --------------------------------------------------------
    def close(self):
        if getattr(self, "handle", None) and self.handle.value:
            self.lib.ap_pool_destroy(self.handle)
            self.handle = ctypes.c_void_p()
        if getattr(self, "arena", None) is not None:
            # the paging stream's work on the pages ends before the mapping can
            # go; the arena itself is released with its last tensor view
            self.stream.synchronize()
            self.arena = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self):
        check(self.lib.ap_pool_reset(self.handle, self.stream.cuda_stream), "pool_reset")

    @property
    def max_ctas(self) -> int:
        v = ctypes.c_int32()
        check(self.lib.ap_pool_max_ctas(self.handle, ctypes.byref(v)), "pool_max_ctas")
        return v.value

    @max_ctas.setter
    def max_ctas(self, value: int):
        check(self.lib.ap_pool_set_max_ctas(self.handle, int(value)), "pool_set_max_ctas")

    # -- data path ----------------------------------------------------------
    @staticmethod
    def _planes(planes):
        rows = planes[0].shape[0]
        ptrs = (ctypes.c_void_p * 2)()
        rb = (ctypes.c_int64 * 2)()
        for i, t in enumerate(planes):
            if not t.is_contiguous() or t.shape[0] != rows:
                raise ValueError("planes must be contiguous with the same number of rows")
            ptrs[i] = t.data_ptr()
            rb[i] = (t.numel() // rows) * t.element_size() if rows else t[0:0].element_size()
        return ptrs, rb, rows

    def _order_after_caller(self, tensors):
        """Make the paging stream wait for the caller's current stream, and tell
        the caching allocator that the tensors are used on the paging stream."""
        cur = torch.cuda.current_stream(self.device)
        if cur != self.stream:
            self.stream.wait_stream(cur)
            for t in tensors:
                if t is not None and t.is_cuda:
                    t.record_stream(self.stream)

    def push(self, slot: int, planes, seg_off: torch.Tensor, live: torch.Tensor) -> int:
        """Stash the live prefixes of every segment of ``planes`` (list of 1-2 tensors).

        The paging stream first waits for the caller's current stream."""
        self._order_after_caller(list(planes) + [seg_off, live])
        ptrs, rb, rows = self._planes(planes)
        rid = ctypes.c_uint64()
        nseg = seg_off.numel()
        check(self.lib.ap_stash_push(self.handle, slot, len(planes), ptrs, rb, rows, nseg, _p(seg_off), _p(live),
                                     ctypes.byref(rid), self.stream.cuda_stream), "stash_push")
        return rid.value

    def dispatch_stash(self, slot: int, x: torch.Tensor, idx: torch.Tensor, E: int, capacity: int = 0,
                       padded: bool = False, fp8: bool = False, out: dict | None = None,
                       status: torch.Tensor | None = None, ranked: bool = False):
        """Fused dispatch + push into ``slot`` (BF16 rows, or E4M3 codes and
        row scales as two planes): returns the dispatch dict (as
        ``dispatch_permute``) with the record id under ``record_id``.
        ``ranked``: ``out`` holds ``count_rank``'s ``dest`` and ``scratch``
        for this idx (``ap_dispatch_stash_ranked``: no count/rank launch), and
        its ``counts``, ``live`` and ``seg_off`` when it ran the scan
        (``out["scanned"]``, for the same capacity and padded); the paging
        stream must already be ordered after the stream that ran it (this
        call orders it after the caller's current stream)."""
        _need(idx, torch.int32, "idx")
        if ranked and (out is None or "dest" not in out or "scratch" not in out):
            raise ValueError("ranked dispatch_stash needs out['dest'] and out['scratch'] from count_rank")
        if ranked and out.get("scanned") and any(n not in out for n in ("counts", "live", "seg_off")):
            raise ValueError("a scanned count_rank's counts, live and seg_off belong in out")
        return self._dispatch_stash(slot, x, idx, idx.shape[1], E, capacity, padded, fp8, out, status, ranked=ranked)

    def route_dispatch_stash(self, slot: int, logits: torch.Tensor, x: torch.Tensor, k: int, E: int | None = None,
                             capacity: int = 0, padded: bool = False, fp8: bool = False, out: dict | None = None,
                             status: torch.Tensor | None = None):
        """Route (as ``route_topk``) and fused dispatch + push in one call:
        the routing runs inside the count/rank launch.  Returns the dispatch
        dict with ``idx``, ``w`` and ``record_id`` added (``out`` may supply
        ``idx`` and ``w`` too)."""
        _need(logits, torch.float32, "logits")
        T, E_l = logits.shape
        E = E_l if E is None else E
        o = dict(out) if out is not None else {}
        if "idx" not in o:
            o["idx"] = torch.empty((T, k), dtype=torch.int32, device=logits.device)
        if "w" not in o:
            o["w"] = torch.empty((T, k), dtype=torch.float32, device=logits.device)
        return self._dispatch_stash(slot, x, o["idx"], k, E, capacity, padded, fp8, o, status, logits=logits,
                                    w=o["w"])

    def _dispatch_stash(self, slot, x, idx, k, E, capacity, padded, fp8, out, status, logits=None, w=None,
                        ranked=False):
        _need(x, torch.bfloat16, "x")
        T, H = x.shape
        dev = x.device
        rows = E * capacity if padded else T * k
        o = dict(out) if out is not None else {}
        if "xd" not in o:
            o["xd"] = torch.empty((rows, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
        if fp8 and "xd_scale" not in o:
            o["xd_scale"] = torch.empty(rows, dtype=torch.float32, device=dev)
        for name, shape in (("counts", (E,)), ("live", (E,)), ("seg_off", (E,)), ("dest", (T, k))):
            if name not in o:
                o[name] = torch.empty(shape, dtype=torch.int32, device=dev)
        if "src_tok" not in o:
            o["src_tok"] = torch.full((rows,), -1, dtype=torch.int32, device=dev)
        sb = dispatch_scratch_bytes(T, k, E)
        if "scratch" not in o or o["scratch"].numel() < sb:
            o["scratch"] = torch.empty(sb, dtype=torch.uint8, device=dev)
        self._order_after_caller([x, idx, status, logits] + [v for v in o.values() if isinstance(v, torch.Tensor)])
        rid = ctypes.c_uint64()
        xd = o["xd"]
        tail = (DTYPE_E4M3 if fp8 else DTYPE_BF16, _p(xd), _p(o.get("xd_scale") if fp8 else None), xd.shape[0],
                _p(o["counts"]), _p(o["live"]), _p(o["seg_off"]), _p(o["dest"]), _p(o["src_tok"]), _p(o["scratch"]),
                o["scratch"].numel(), _p(status), ctypes.byref(rid), self.stream.cuda_stream)
        if ranked:
            scanned = int(bool(o.get("scanned", False)))
            check(self.lib.ap_dispatch_stash_ranked(self.handle, slot, _p(x), T, H, _p(idx), k, E, capacity,
                                                    int(padded), *tail[:-1], scanned, tail[-1]),
                  "dispatch_stash_ranked")
        elif logits is None:
            check(self.lib.ap_dispatch_stash(self.handle, slot, _p(x), T, H, _p(idx), k, E, capacity, int(padded),
                                             *tail), "dispatch_stash")
        else:
            check(self.lib.ap_route_dispatch_stash(self.handle, slot, _p(logits), _p(w), _p(x), T, H, _p(idx), k, E,
                                                   capacity, int(padded), *tail), "route_dispatch_stash")
        o["record_id"] = rid.value
        return o

    def pop(self, slot: int, planes) -> int:
        """Reload the slot's oldest record into ``planes`` (same rows as pushed).

        The paging stream first waits for the caller's current stream; the
        caller orders later reads after ``self.stream``."""
        self._order_after_caller(list(planes))
        ptrs, _, rows = self._planes(planes)
        rid = ctypes.c_uint64()
        check(self.lib.ap_stash_pop(self.handle, slot, len(planes), ptrs, rows, ctypes.byref(rid),
                                    self.stream.cuda_stream), "stash_pop")
        return rid.value

    def time_copies(self, before: torch.cuda.Event | None, after: torch.cuda.Event | None):
        """Record ``before`` / ``after`` (timing events) around the copy kernel
        of every following push, fused dispatch + push and pop; None, None
        stops it.  The events must stay alive while set."""
        for e in (before, after):
            if e is not None and e.cuda_event == 0:
                e.record(self.stream)  # torch creates the event on its first record
        self._timing = (before, after)  # keep them alive while the library holds them
        check(self.lib.ap_pool_time_copies(self.handle, before.cuda_event if before is not None else None,
                                           after.cuda_event if after is not None else None), "pool_time_copies")

    def queue_len(self, slot: int) -> int:
        v = ctypes.c_int32()
        check(self.lib.ap_pool_queue_len(self.handle, slot, ctypes.byref(v)), "pool_queue_len")
        return v.value

    # -- read-outs (synchronise the paging stream) -------------------------------
    def overflow(self, wait: bool = True) -> int:
        f = ctypes.c_uint32()
        check(self.lib.ap_overflow_query(self.handle, ctypes.byref(f), int(wait)), "overflow_query")
        return f.value

    def flags_device_ptr(self) -> int:
        p = ctypes.c_void_p()
        check(self.lib.ap_pool_flags_device_ptr(self.handle, ctypes.byref(p)), "pool_flags_device_ptr")
        return p.value

    def state(self) -> dict:
        s = PoolState()
        check(self.lib.ap_pool_read_state(self.handle, ctypes.byref(s)), "pool_read_state")
        return dict(head=s.head, tail=s.tail, spill_head=s.spill_head, spill_tail=s.spill_tail, flags=s.flags,
                    high_water=s.high_water, spill_high_water=s.spill_high_water, held=s.held,
                    held_high_water=s.held_high_water, num_pages=s.num_pages)

    def stats(self, wait: bool = True) -> dict:
        """Device pages in use, their high-water mark and spill pages in use
        (``ap_pool_stats``).  ``wait=False`` touches no GPU and returns the
        figures of the last synchronising read-out."""
        a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        check(self.lib.ap_pool_stats(self.handle, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), int(wait)),
              "pool_stats")
        return dict(pages_in_use=a.value, high_water=b.value, spill_in_use=c.value)

    def rings(self):
        import numpy as np
        ring = np.empty(self.N, np.int32)
        sring = np.empty(max(self.SP, 1), np.int32)
        check(self.lib.ap_pool_read_rings(self.handle, ring.ctypes.data, sring.ctypes.data if self.SP else None),
              "pool_read_rings")
        return ring, sring[: self.SP]

    def record(self, slot: int, qpos: int = 0) -> dict:
        import numpy as np
        info = RecordInfo()
        check(self.lib.ap_pool_read_record(self.handle, slot, qpos, ctypes.byref(info), None, None, None, 0),
              "pool_read_record")
        n = info.npages
        pt = np.empty(max(n, 1), np.int32)
        r0 = np.empty(max(n, 1), np.int64)
        nr = np.empty(max(n, 1), np.int32)
        check(self.lib.ap_pool_read_record(self.handle, slot, qpos, ctypes.byref(info), pt.ctypes.data,
                                           r0.ctypes.data, nr.ctypes.data, n), "pool_read_record")
        return dict(id=info.record_id, npages=n, ndev=info.ndev, nspill=info.nspill, nlost=info.nlost,
                    nseg=info.nseg, page_table=pt[:n], row0=r0[:n], nrows=nr[:n])
