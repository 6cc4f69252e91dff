"""The allocation-free dispatch entry point gives the same results as the
ordinary one.

ap_dispatch_permute_noalloc serves callers that cannot allocate device memory
(for example code running where another allocator already holds the whole GPU,
or loops that must not enter cudaMalloc).  It keeps its work space in a fixed
array inside the library instead of taking caller scratch.  This test calls
it through the C ABI twice in a row, with different inputs and sizes, and
compares every output with ap_dispatch_permute on the same inputs: indices
and bytes must match exactly, as in the other dispatch tests.  It also checks
that a size needing more than the built-in work space is refused.  This file
is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

from activation_paging_gb300 import inputs
from gpu_util import bf16_to_dev, host, to_dev

pytestmark = pytest.mark.gpu

ap = pytest.importorskip("activation_paging_gb300")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(x, idx, E, capacity, padded, fp8):
    lib = ap.lib()
    T, H = x.shape
    k = idx.shape[1]
    rows = E * capacity if padded else T * k
    dev = x.device
    o = {"xd": torch.zeros((rows, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev),
         "xd_scale": torch.zeros(rows, dtype=torch.float32, device=dev) if fp8 else None,
         "counts": torch.empty(E, dtype=torch.int32, device=dev),
         "live": torch.empty(E, dtype=torch.int32, device=dev),
         "seg_off": torch.empty(E, dtype=torch.int32, device=dev),
         "dest": torch.empty((T, k), dtype=torch.int32, device=dev),
         "src_tok": torch.full((rows,), -1, dtype=torch.int32, device=dev)}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = lib.ap_dispatch_permute_noalloc(_p(x), T, H, _p(idx), k, E, capacity, int(padded), int(fp8), _p(o["xd"]),
                                         _p(o["xd_scale"]), rows, _p(o["counts"]), _p(o["live"]), _p(o["seg_off"]),
                                         _p(o["dest"]), _p(o["src_tok"]), _p(status),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.ap_last_error()
    return o, status


def call_ordinary(x, idx, E, capacity, padded, fp8):
    rows = E * capacity if padded else x.shape[0] * idx.shape[1]
    H = x.shape[1]
    out = {"xd": torch.zeros((rows, H), dtype=torch.uint8 if fp8 else torch.bfloat16, device=x.device)}
    if fp8:
        out["xd_scale"] = torch.zeros(rows, dtype=torch.float32, device=x.device)
    status = torch.zeros(1, dtype=torch.int32, device=x.device)
    return ap.dispatch_permute(x, idx, E, capacity, padded, fp8=fp8, out=out, status=status), status


@pytest.mark.parametrize("first,second", [
    # (T, H, E, k, capacity, padded, fp8): the second call is smaller, so a
    # stale work space from the first call would show
    ((8192, 2048, 128, 8, 0, False, False), (1000, 256, 64, 6, 120, True, False)),
    ((4096, 2056, 64, 6, 0, False, True), (333, 100, 8, 3, 0, False, True)),
])
def test_noalloc_matches_ordinary_dispatch_twice(first, second):
    for n, (T, H, E, k, C, padded, fp8) in enumerate((first, second)):
        logits = inputs.router_logits(50 + n, T, E)
        x = bf16_to_dev(inputs.normal_bf16(50 + n, inputs.X_STREAM, (T, H)))
        idx, _ = ap.route_topk(to_dev(logits), k)
        got, st_g = call_noalloc(x, idx, E, C, padded, fp8)
        exp, st_e = call_ordinary(x, idx, E, C, padded, fp8)
        torch.cuda.synchronize()
        for key in ("counts", "live", "seg_off", "dest", "src_tok"):
            assert torch.equal(got[key], exp[key]), key
        assert torch.equal(got["xd"].view(torch.uint8), exp["xd"].view(torch.uint8))
        if fp8:
            assert torch.equal(got["xd_scale"].view(torch.int32), exp["xd_scale"].view(torch.int32))
        assert int(host(st_g)[0]) == int(host(st_e)[0]) == 0


def test_noalloc_refuses_sizes_beyond_its_work_space():
    lib = ap.lib()
    dummy = torch.empty(16, dtype=torch.int32, device="cuda")
    p = _p(dummy)
    T, E, k = 1 << 20, 1024, 8  # (T/64)*E*4 bytes = 64 MiB > 1 MiB (count/rank blocks of 64 tokens)
    rc = lib.ap_dispatch_permute_noalloc(p, T, 64, p, k, E, 0, 0, 0, p, None, T * k, p, p, p, p, None, None, None)
    assert rc == -1
    assert b"work space" in lib.ap_last_error()
