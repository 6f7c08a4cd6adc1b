"""q4_matmul_noalloc: the verify matmul for callers that may not allocate
device memory (a serving engine that gives all free HBM to its own pools at
start-up, a plug-in running inside an application that owns the allocator, a
loop that cannot take cudaMalloc's implicit synchronisation).  Its scratch is
a fixed array inside the library's device image.  These tests call it through
the C ABI and compare it with q4_matmul on the same inputs, two calls in a row,
so the second call runs on scratch that the first one left behind.

The file name keeps it last in collection order."""
import ctypes

import numpy as np
import pytest
import torch

import bit_row_speculative_gb300 as q4
import synth_inputs as si
from parity import TOL


def _abs_products(x: torch.Tensor, W: torch.Tensor, N: int, K: int) -> torch.Tensor:
    """sum_k |x[m,k] * w[n,k]| in fp64 on the GPU (plain PyTorch dequantisation)."""
    G = K // 64
    nib = W[: N * K // 2].view(N, K // 2)
    q = torch.stack([nib & 15, nib >> 4], dim=-1).reshape(N, K).to(torch.float64)
    sb = W[N * K // 2:].view(torch.bfloat16).to(torch.float64)
    s = sb[: N * G].view(N, G).repeat_interleave(64, dim=1)
    b = sb[N * G:].view(N, G).repeat_interleave(64, dim=1)
    w = (s * q + b).abs()
    return x.to(torch.float64).abs() @ w.t()


def _within(y, y_ref, scale, what):
    err = (y.to(torch.float64) - y_ref.to(torch.float64)).abs()
    bad = err > TOL * scale
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} outputs differ beyond the tolerance"


@pytest.mark.gpu
@pytest.mark.parametrize("name,M", [("attn_in", 16), ("attn_in", 1), ("down", 5), ("odd", 3)])
def test_noalloc_matches_q4_matmul_twice(name, M):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    N, K = (320, 576) if name == "odd" else si.SHAPES[name]     # "odd": K not a multiple of 512
    lib = q4.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        W = si.make_weights(N, K, 71 + call, device="cuda")
        x = si.make_x(M, K, 81 + call, device="cuda")
        y_ref = q4.matmul(x, W, N, K)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        rc = lib.q4_matmul_noalloc(x.data_ptr(), W.data_ptr(), M, N, K, y.data_ptr(), stream)
        assert rc == q4.Q4_OK, lib.q4_last_error().decode()
        q4.device_status()
        assert bool(torch.isfinite(y).all()), f"call {call}: output not fully written"
        _within(y, y_ref, _abs_products(x, W, N, K), f"{name} M={M} call {call}")


@pytest.mark.gpu
def test_noalloc_rejects_k_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    N, K = 8, 20480 + 512
    W = torch.zeros(q4.packed_bytes(N, K), dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((1, N), dtype=torch.float32, device="cuda")
    lib = q4.lib()
    rc = lib.q4_matmul_noalloc(x.data_ptr(), W.data_ptr(), 1, N, K, y.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)
    assert rc == q4.Q4_ERR_UNSUPPORTED_SHAPE
    assert b"20480" in lib.q4_last_error()
    assert np.all(y.cpu().numpy() == 0)


def test_noalloc_rejects_k_beyond_its_scratch_on_host():
    """The size check happens on the host before any device work."""
    lib = q4.lib()
    buf = ctypes.create_string_buffer(64)
    p = (ctypes.addressof(buf) + 15) & ~15
    rc = lib.q4_matmul_noalloc(p, p, 1, 8, 20480 + 64, p, None)
    assert rc == q4.Q4_ERR_UNSUPPORTED_SHAPE
