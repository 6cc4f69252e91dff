"""Seeded synthetic inputs and workload shapes.

This module serves both the CUDA path and the CPU oracle: it holds the shapes
of the workloads and draws their random inputs, and nothing of the method's
arithmetic (no routing, counting, paging or combining).  Every tensor comes
from numpy's PCG64 generator seeded with ``[seed, stream]``:

* stream 0: token activations x, N(0, 1) in single precision rounded to BF16;
* stream 1: router logits, N(0, 1) single precision, plus an optional Zipf
  per-expert bias ``-beta * s * ln(rank_e)`` where ``rank_e = 1 + pi(e)`` for a
  seeded permutation pi (stream 4);
* stream 2: expert outputs y, N(0, 1) rounded to BF16;
* stream 3: opaque payload bytes (uniform 0..255).

A workload with several chunks, microbatches or layers draws each part with a
distinct seed (``seed + part``).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

X_STREAM, LOGIT_STREAM, Y_STREAM, BYTE_STREAM, PERM_STREAM = 0, 1, 2, 3, 4


def rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round single precision to BF16 bit patterns (nearest-even); inputs are finite."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, stream: int, shape) -> np.ndarray:
    """N(0, 1) values as BF16 bit patterns (uint16)."""
    g = rng(seed, stream)
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    step = 1 << 24
    for i in range(0, n, step):
        m = min(step, n - i)
        out[i:i + m] = f32_to_bf16_bits(g.standard_normal(m, dtype=np.float32))
    return out.reshape(shape)


def zipf_bias(E: int, s: float, beta: float, seed: int) -> np.ndarray:
    """Per-expert logit bias -beta*s*ln(rank) over a seeded rank permutation."""
    if s == 0.0 or beta == 0.0:
        return np.zeros(E, np.float32)
    perm = rng(seed, PERM_STREAM).permutation(E)
    rank = 1.0 + perm.astype(np.float64)
    return (-beta * s * np.log(rank)).astype(np.float32)


def router_logits(seed: int, T: int, E: int, zipf_s: float = 0.0, zipf_beta: float = 0.0) -> np.ndarray:
    g = rng(seed, LOGIT_STREAM)
    logits = g.standard_normal((T, E), dtype=np.float32)
    if zipf_s:
        logits += zipf_bias(E, zipf_s, zipf_beta, seed)[None, :]
    return logits


def payload_bytes(seed: int, shape) -> np.ndarray:
    return rng(seed, BYTE_STREAM).integers(0, 256, size=shape, dtype=np.uint8)


def round_up(v: int, m: int) -> int:
    return (v + m - 1) // m * m


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shapes of one synthetic workload.

    T is tokens per chunk (or per microbatch); ``chunks`` token chunks, or
    ``microbatches`` x ``layers`` records, make one step.  ``capacity_factor``
    0 means dropless.  ``num_pages`` and ``spill_pages`` size the page pool."""
    name: str
    T: int
    H: int
    E: int
    k: int
    chunks: int = 1
    capacity_factor: float = 0.0
    padded: bool = False
    fp8: bool = False
    page_tokens: int = 64
    num_pages: int = 0
    num_slots: int = 1
    spill_pages: int = 0
    zipf_s: float = 0.0
    zipf_beta: float = 0.0
    microbatches: int = 1
    layers: int = 1
    seed: int = 0

    @property
    def capacity(self) -> int:
        """ceil(cf * T * k / E) rows per expert, or 0 (dropless)."""
        if self.capacity_factor <= 0:
            return 0
        num = self.capacity_factor * self.T * self.k
        c = int(num // self.E)
        return c + 1 if c * self.E < num else c

    @property
    def rows(self) -> int:
        """Rows of the dispatch buffer: E*C padded, T*k compact."""
        return self.E * self.capacity if self.padded else self.T * self.k

    @property
    def row_bytes(self) -> tuple:
        """Bytes per row of each stash plane: BF16 row, or E4M3 row + FP32 scale."""
        return (self.H, 4) if self.fp8 else (self.H * 2,)

    @property
    def page_bytes(self) -> int:
        rb = self.row_bytes
        need = self.page_tokens * rb[0]
        if len(rb) == 2:
            need = round_up(need, 16) + self.page_tokens * rb[1]
        return round_up(need, 256)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# Zipf strength for the skewed workload: the bias scale beta at which the
# busiest expert receives ~8x the mean load (max/mean in [7.5, 8.5]) on the
# seed-0 logits, found by bisection with the CPU oracle's router
# (oracle/calibrate_zipf.py writes this value).
SKEWED_ZIPF_BETA = 0.375

WORKLOADS = {
    # T=256, H=128, E=8, top-2, capacity factor 1.25 (C = 80, padded
    # [8, 80, 128]); 16-token pages, 64 pages, 4 FIFO slots.
    "tiny": Workload("tiny", T=256, H=128, E=8, k=2, capacity_factor=1.25, padded=True,
                     page_tokens=16, num_pages=64, num_slots=4),
    # Qwen3-MoE-like layer: 16384 tokens in 2 chunks of 8192, H=2048, E=128,
    # top-8, dropless; 64-token pages, pool = ceil(1.1 * live rows / 64).
    "qwen3_moe": Workload("qwen3_moe", T=8192, H=2048, E=128, k=8, chunks=2, page_tokens=64,
                          num_pages=math.ceil(1.1 * 2 * 8192 * 8 / 64), num_slots=1),
    # Skewed routing: T=32768, Zipf(s=1.2) bias, capacity factor 1.0 (C=2048),
    # padded with drops; pool of E*ceil(C/64) = 4096 pages.
    "skewed": Workload("skewed", T=32768, H=2048, E=128, k=8, capacity_factor=1.0, padded=True,
                       page_tokens=64, num_pages=4096, zipf_s=1.2, zipf_beta=SKEWED_ZIPF_BETA),
    # DeepSeek-V2-Lite-like FP8 stack: 4096 tokens per microbatch, 8
    # microbatches, 27 layers (one slot each), E=64, top-6, E4M3 payload with
    # a per-row FP32 scale, 128-token pages.  Pool: no-overflow bound
    # records * (rows/P + E).
    "dsv2_lite_fp8": Workload("dsv2_lite_fp8", T=4096, H=2048, E=64, k=6, fp8=True, page_tokens=128,
                              num_pages=27 * 8 * (4096 * 6 // 128 + 64), num_slots=27,
                              microbatches=8, layers=27),
    # Overflow / spill: T=32768, H=7168, E=256, top-8, Zipf(s=1.5, beta=1);
    # pool = 60% of two live records' rows, spill = 50% of them.
    "spill": Workload("spill", T=32768, H=7168, E=256, k=8, page_tokens=64,
                      num_pages=math.ceil(0.6 * 2 * 32768 * 8 / 64),
                      spill_pages=math.ceil(0.5 * 2 * 32768 * 8 / 64), num_slots=2,
                      zipf_s=1.5, zipf_beta=1.0),
}
WORKLOADS["dsv2_lite_fp8_h2056"] = WORKLOADS["dsv2_lite_fp8"].replace(name="dsv2_lite_fp8_h2056", H=2056)
