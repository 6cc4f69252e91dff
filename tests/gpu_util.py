"""Helpers of the GPU tests: numpy <-> torch without changing a bit."""
import numpy as np
import torch

from activation_paging_gb300.inputs import bf16_bits_to_f32


def bf16_to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_to_host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().numpy()


def route_tolerance(logits: np.ndarray, idx: np.ndarray, w_or: np.ndarray) -> np.ndarray:
    """Per-weight bound of |w_gpu - w_oracle| for single-precision routing.

    The kernel computes d = l_j - m (one rounding, relative 2^-24 |d|), z = exp(d)
    (at most 2 ulp), the sum of k terms (k-1 roundings) and one division; the
    oracle's double result is rounded once to single.  Relative error of w is at
    most (2*|d|max + 4 + k + 1 + 1) * 2^-24 with the 2-ulp exponential counted
    twice (numerator and sum)."""
    l_sel = np.take_along_axis(logits.astype(np.float64), idx, 1)
    dmax = np.abs(l_sel - l_sel[:, :1]).max(1, keepdims=True)
    k = idx.shape[1]
    rel = (2 * dmax + 2 * 4 + k + 2) * 2.0 ** -24
    return rel * np.abs(w_or.astype(np.float64)) + 2.0 ** -149


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v.astype(np.float64))
    return np.where(a == 0, 2.0 ** -133, 2.0 ** (np.frexp(a)[1] - 8))


def combine_within(got: np.ndarray, exp: np.ndarray, y: np.ndarray, dest: np.ndarray, w: np.ndarray,
                   dw: np.ndarray) -> bool:
    """Combine outputs computed from weights that differ by at most dw per entry.

    Both sides round the same kind of single-precision sum of k products, so
    |got - exp| <= ulp + sum_j dw_j |y_j| + 2k 2^-24 sum_j |w_j y_j|, with ulp
    the BF16 unit of the larger output."""
    g = bf16_bits_to_f32(got).astype(np.float64)
    e = bf16_bits_to_f32(exp).astype(np.float64)
    yf = bf16_bits_to_f32(y).astype(np.float64)
    T, k = dest.shape
    spread = np.zeros_like(e)
    mag = np.zeros_like(e)
    for j in range(k):
        r = dest[:, j]
        ok = r >= 0
        spread[ok] += dw[ok, j:j + 1] * np.abs(yf[r[ok]])
        mag[ok] += np.abs(w[ok, j:j + 1].astype(np.float64) * yf[r[ok]])
    bound = np.maximum(bf16_ulp(g), bf16_ulp(e)) + spread + 2 * k * 2.0 ** -24 * mag
    return bool(np.all(np.abs(g - e) <= bound))
