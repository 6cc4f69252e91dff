"""Helpers of the GPU tests: numpy <-> torch without changing a bit."""
import numpy as np
import torch


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
