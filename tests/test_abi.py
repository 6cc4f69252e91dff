"""The C ABI library: it loads without a GPU, exports every symbol the header
declares, and rejects bad arguments on the host before launching anything.
None of these tests touches a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from activation_paging_gb300 import build, _lib
    build.build()
    return _lib.load()


def header_symbols():
    text = open(os.path.join(ROOT, "include", "ap.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ap_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    from activation_paging_gb300 import _lib
    syms = header_symbols()
    assert len(syms) >= 20
    for s in syms:
        assert hasattr(lib, s), s
    assert sorted(_lib.SIGNATURES) == syms  # the binding declares exactly the header's calls


def test_status_strings(lib):
    assert lib.ap_status_str(0) == b"AP_OK"
    assert lib.ap_status_str(-1) == b"AP_EINVAL"
    assert lib.ap_status_str(-2) == b"AP_EEMPTY"
    assert lib.ap_status_str(-3) == b"AP_EQFULL"
    assert lib.ap_status_str(-5) == b"AP_ESTREAM"
    assert lib.ap_version().startswith(b"0.")


def test_required_bytes_host_only(lib):
    from activation_paging_gb300._lib import PoolConfig
    cfg = PoolConfig(64, 1, 64 * 4096, 2253, 0, 8, 128, 4096, 0, 0)
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    assert lib.ap_pool_required_bytes(ctypes.byref(cfg), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)) == 0
    assert a.value == 2253 * 64 * 4096
    assert c.value == 0
    # ring + state + one record: header, seg_off/live/pg_base, descriptors and page table
    assert b.value >= 256 + 4 * 2253 + 128 + 4 * 128 * 2 + 8 * 129 + 4096 * (16 + 4)
    assert b.value % 256 == 0
    bad = [
        PoolConfig(0, 1, 4096, 16, 0, 8, 8, 16, 0, 0),      # page_tokens 0
        PoolConfig(4, 1, 4100, 16, 0, 8, 8, 16, 0, 0),      # page_bytes not a multiple of 16
        PoolConfig(4, 0, 4096, 16, 0, 8, 8, 16, 0, 0),      # no slot
        PoolConfig(4, 1, 4096, 0, 0, 8, 8, 16, 0, 0),       # no page
        PoolConfig(4, 1, 4096, 2 ** 31, 0, 8, 8, 16, 0, 0),  # page ids beyond int32
        PoolConfig(4, 1, 4096, 16, 0, 8, 8, 16, -1, 0),     # negative grid bound
        PoolConfig(4, 1, 4096, 16, 0, 8, 8, 16, 0, 7),      # reserved != 0
        PoolConfig(4, 1, 4096, 17, 0, 8, 8, 16, 0, 0, 16),  # more pages than the growth limit
        PoolConfig(4, 1, 4096, 0, 0, 8, 8, 16, 0, 0, -1),   # negative growth limit
        PoolConfig(4, 1, 4096, 8, 2 ** 31 - 16, 8, 8, 16, 0, 0, 16),  # spill ids beyond int32
    ]
    for cfg in bad:
        assert lib.ap_pool_required_bytes(ctypes.byref(cfg), None, None, None) == -1
    # a calibration pool: no device pages yet, room for 100; the metadata
    # holds the ring for 100 pages and the grow work space
    cal = PoolConfig(4, 1, 4096, 0, 50, 8, 8, 16, 0, 0, 100)
    assert lib.ap_pool_required_bytes(ctypes.byref(cal), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)) == 0
    assert a.value == 0 and c.value == 50 * 4096
    assert b.value >= 256 + 4 * 100 + 4 * 50 + 4 * 100


def test_arena_without_a_gpu_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    a = ctypes.c_void_p(1)
    assert lib.ap_arena_create(ctypes.byref(a), 1 << 20, 0) in (-4, -6)  # AP_ECUDA or AP_ENOTSUP
    assert not a.value
    assert lib.ap_arena_destroy(None) == 0


def test_pool_calls_reject_a_null_pool(lib):
    assert lib.ap_pool_time_copies(None, None, None) == -1
    assert lib.ap_pool_grow(None, 8, None, None) == -1
    assert lib.ap_pool_reset(None, None) == -1


def test_route_rejects_bad_sizes(lib):
    p = ctypes.c_void_p(16)
    assert lib.ap_route_topk(p, 10, 0, 1, p, p, None) == -1       # E = 0
    assert lib.ap_route_topk(p, 10, 8, 9, p, p, None) == -1       # k > E
    assert lib.ap_route_topk(p, 10, 2048, 8, p, p, None) == -1    # E > 1024
    assert lib.ap_route_topk(p, 10, 64, 33, p, p, None) == -1     # k > 32
    assert lib.ap_route_topk(None, 10, 8, 2, p, p, None) == -1    # NULL logits
    assert lib.ap_route_topk(None, 0, 8, 2, None, None, None) == 0  # empty: nothing to do
    n0 = lib.ap_launch_count()
    assert lib.ap_route_topk(p, 10, 8, 9, p, p, None) == -1
    assert b"bad sizes" in lib.ap_last_error()
    assert lib.ap_launch_count() == n0  # a rejected call enqueues nothing


def test_dispatch_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    n = ctypes.c_int64()
    assert lib.ap_dispatch_scratch_bytes(1000, 8, 128, ctypes.byref(n)) == 0
    assert n.value >= 4 * 128 * 4 and n.value % 256 == 0
    args = dict(x=p, T=100, H=64, idx=p, k=2, E=8, cap=0, padded=0, dt=0, xd=p, xs=None, rows=200,
                counts=p, live=p, seg=p, dest=p, src=None, scratch=p, sb=n.value, st=None, stream=None)

    def call(**kw):
        a = dict(args, **kw)
        return lib.ap_dispatch_permute(a["x"], a["T"], a["H"], a["idx"], a["k"], a["E"], a["cap"], a["padded"],
                                       a["dt"], a["xd"], a["xs"], a["rows"], a["counts"], a["live"], a["seg"],
                                       a["dest"], a["src"], a["scratch"], a["sb"], a["st"], a["stream"])
    assert call(rows=199) == -1            # xd too small for T*k rows
    assert call(padded=1, cap=0) == -1     # padded needs a capacity
    assert call(padded=1, cap=30, rows=239) == -1
    assert call(dt=7) == -1                # unknown payload type
    assert call(dt=1) == -1                # E4M3 needs a scale plane
    assert call(sb=16) == -1               # scratch too small
    assert call(k=33) == -1
    assert call(E=2000) == -1


def test_count_rank_rejects_bad_arguments(lib):
    """ap_count_rank checks its sizes, work space and pointers before any
    launch (no GPU is touched), and ap_dispatch_stash_ranked a NULL pool."""
    p = ctypes.c_void_p(256)
    n = ctypes.c_int64()
    assert lib.ap_dispatch_scratch_bytes(1000, 8, 128, ctypes.byref(n)) == 0

    def call(logits=None, w=None, idx=p, T=1000, k=8, E=128, x=None, rb=0, dest=p, scratch=p, sb=n.value, cap=0,
             padded=0, counts=None, live=None, seg=None):
        return lib.ap_count_rank(logits, w, idx, T, k, E, x, rb, dest, scratch, sb, cap, padded, counts, live, seg,
                                 None, None)
    n0 = lib.ap_launch_count()
    assert call(k=0) == -1
    assert call(k=33) == -1
    assert call(E=2000) == -1
    assert call(logits=p, w=p, k=8, E=4) == -1   # routing needs k <= E
    assert call(logits=p, w=None) == -1          # routing writes w
    assert call(sb=n.value - 256) == -1          # work space too small
    assert call(dest=None) == -1
    assert call(rb=-1) == -1
    assert call(counts=p, live=p) == -1                # the scan needs all three outputs
    assert call(counts=p, live=p, seg=p, padded=1) == -1  # padded needs a capacity
    assert b"count_rank" in lib.ap_last_error()
    assert lib.ap_launch_count() == n0
    assert lib.ap_dispatch_stash_ranked(None, 0, p, 10, 64, p, 2, 8, 0, 0, 0, p, None, 20, p, p, p, p, None, p,
                                        n.value, None, None, 0, None) == -1


def test_combine_rejects_bad_arguments(lib):
    p = ctypes.c_void_p(256)
    assert lib.ap_combine_unpermute(p, 10, 0, p, p, 4, 2, p, None, None) == -1   # H = 0
    assert lib.ap_combine_unpermute(p, 10, 8, p, p, 4, 40, p, None, None) == -1  # k > 32
    assert lib.ap_combine_unpermute(p, 10, 8, None, p, 4, 2, p, None, None) == -1
    assert lib.ap_combine_unpermute(p, 10, 8, p, p, 0, 2, p, None, None) == 0     # no token


def test_pool_init_rejects_bad_buffers(lib):
    from activation_paging_gb300._lib import PoolConfig
    cfg = PoolConfig(4, 1, 4096, 16, 0, 8, 8, 16, 0, 0)
    h = ctypes.c_void_p()
    assert lib.ap_pool_init(ctypes.byref(h), ctypes.byref(cfg), None, ctypes.c_void_p(512), None, None) == -1
    assert lib.ap_pool_init(ctypes.byref(h), ctypes.byref(cfg), ctypes.c_void_p(512 + 16), ctypes.c_void_p(512),
                            None, None) == -1  # pool not 256-byte aligned
    assert lib.ap_pool_init(ctypes.byref(h), ctypes.byref(cfg), ctypes.c_void_p(512), ctypes.c_void_p(512),
                            ctypes.c_void_p(4096), None) == -1  # spill given with spill_pages = 0
    assert lib.ap_pool_init(None, ctypes.byref(cfg), None, None, None, None) == -1
    assert not h.value


def test_pool_calls_reject_null_pool(lib):
    assert lib.ap_stash_push(None, 0, 1, None, None, 0, 0, None, None, None, None) == -1
    assert lib.ap_stash_pop(None, 0, 1, None, 0, None, None) == -1
    assert lib.ap_pool_reset(None, None) == -1
    assert lib.ap_pool_destroy(None) == 0
    f = ctypes.c_uint32()
    assert lib.ap_overflow_query(None, ctypes.byref(f), 0) == -1
    n = ctypes.c_int64()
    assert lib.ap_pool_stats(None, ctypes.byref(n), None, None, 0) == -1
    assert lib.ap_pool_stats(None, None, None, None, 1) == -1


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "activation_paging_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "ap_oracle" not in text, f
