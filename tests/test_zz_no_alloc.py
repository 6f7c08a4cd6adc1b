"""q4_matmul_noalloc: the verify matmul for callers that may not allocate
device memory (a serving engine that gives all free HBM to its own pools at
start-up, a plug-in running inside an application that owns the allocator, a
loop that cannot take cudaMalloc's implicit synchronisation).  Its scratch is
a fixed array inside the library's device image.  These tests call it through
the C ABI and check it against the CPU oracle element by element on the same
seeded inputs, two calls in a row (the second runs on scratch the first left
behind), check that its rows do not depend on M, and that the calls and the
status query allocate no device memory.

The file name keeps it last in collection order."""
import ctypes

import numpy as np
import pytest
import torch

import bit_row_speculative_gb300 as q4
import oracle
import synth_inputs as si
from parity import check_tolerance, sample_columns, xbits


def _noalloc(lib, x, W, N, K, stream):
    M = x.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    rc = lib.q4_matmul_noalloc(x.data_ptr(), W.data_ptr(), M, N, K, y.data_ptr(), stream)
    assert rc == q4.Q4_OK, lib.q4_last_error().decode()
    return y


@pytest.mark.gpu
@pytest.mark.parametrize("name,M", [("attn_in", 16), ("attn_in", 1), ("down", 5), ("odd", 3)])
def test_noalloc_matches_oracle_twice(name, M):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    N, K = (320, 576) if name == "odd" else si.SHAPES[name]     # "odd": K not a multiple of 512
    lib = q4.lib()
    stream = torch.cuda.current_stream().cuda_stream
    cols = sample_columns(N, 256, seed=N + M) if N > 512 else None
    for call in range(2):
        W = si.make_weights(N, K, 71 + call, device="cuda")
        x = si.make_x(M, K, 81 + call, device="cuda")
        y = _noalloc(lib, x, W, N, K, stream)
        q4.device_status()
        y = y.cpu().numpy()
        assert np.isfinite(y).all(), f"call {call}: output not fully written"
        ref, scale = oracle.matmul(xbits(x), W.cpu().numpy(), N, K, cols=cols)
        check_tolerance(y if cols is None else y[:, cols], ref, scale, f"{name} M={M} call {call}")


@pytest.mark.gpu
def test_noalloc_rows_do_not_depend_on_M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    N, K = si.SHAPES["attn_in"]
    lib = q4.lib()
    stream = torch.cuda.current_stream().cuda_stream
    W = si.make_weights(N, K, 91, device="cuda")
    x16 = si.make_x(16, K, 92, device="cuda")
    y16 = _noalloc(lib, x16, W, N, K, stream).cpu().numpy()
    for M in range(1, 16):
        yM = _noalloc(lib, x16[:M].contiguous(), W, N, K, stream).cpu().numpy()
        assert np.array_equal(yM, y16[:M]), f"M={M}"
    q4.device_status()


@pytest.mark.gpu
def test_noalloc_allocates_nothing():
    """Device memory free before and after two calls and a status query is the
    same.  One call comes first: on a device where the library's device image
    is not loaded yet, the runtime loads it then (the static scratch array is
    part of that image)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    N, K, M = 4096, 5120, 8
    lib = q4.lib()
    stream = torch.cuda.current_stream().cuda_stream
    W = si.make_weights(N, K, 95, device="cuda")
    x = si.make_x(M, K, 96, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert lib.q4_matmul_noalloc(x.data_ptr(), W.data_ptr(), M, N, K, y.data_ptr(), stream) == q4.Q4_OK
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(2):
        rc = lib.q4_matmul_noalloc(x.data_ptr(), W.data_ptr(), M, N, K, y.data_ptr(), stream)
        assert rc == q4.Q4_OK, lib.q4_last_error().decode()
    assert lib.q4_device_status(stream) == q4.Q4_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


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
