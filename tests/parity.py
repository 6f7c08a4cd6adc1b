"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare it element by element with the CPU oracle on the same seeded
inputs."""
from __future__ import annotations

import numpy as np
import torch

import bit_row_speculative_gb300 as q4
import oracle
import synth_inputs as si

TOL = 2e-3          # |y - exact| <= TOL * sum_k |x_k w_k| per output


def xbits(x: torch.Tensor) -> np.ndarray:
    return si.bf16_bits(x.cpu()).numpy().view(np.uint16)


def check_tolerance(y_gpu: np.ndarray, ref: np.ndarray, scale: np.ndarray, what: str = "") -> float:
    """Assert the tolerance; return the worst err/scale ratio seen."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - ref)
    zero = scale == 0
    assert np.all(y_gpu[zero] == 0.0), f"{what}: outputs with sum|x*w| = 0 must be exactly 0"
    bad = err > TOL * scale
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} outputs outside tolerance, e.g. {idx.tolist()} "
                             f"err {err[bad][:5]} scale {scale[bad][:5]}")
    nz = ~zero
    return float((err[nz] / scale[nz]).max()) if nz.any() else 0.0


def sample_columns(N: int, count: int, seed: int) -> np.ndarray:
    """Sorted unique columns: the first and last 16 plus a seeded random draw."""
    rng = np.random.default_rng(seed)
    edge = np.concatenate([np.arange(min(16, N)), np.arange(max(0, N - 16), N)])
    pick = rng.choice(N, size=min(count, N), replace=False)
    return np.unique(np.concatenate([edge, pick])).astype(np.int64)


def run_and_check(x: torch.Tensor, W: torch.Tensor, N: int, K: int, cols=None, what: str = ""):
    """x bf16 [M,K] (any device), W uint8 packed (any device)."""
    dev = torch.device("cuda")
    y = q4.matmul(x.to(dev).contiguous(), W.to(dev), N, K)
    q4.device_status()
    y = y.cpu().numpy()
    Wh = W.cpu().numpy()
    ref, scale = oracle.matmul(xbits(x), Wh, N, K, cols=cols)
    yc = y if cols is None else y[:, cols]
    return y, check_tolerance(yc, ref, scale, what)
