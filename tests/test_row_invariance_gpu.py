"""Bit-identical batched verify ("Faster, with the same words" (goinfer.dev),
section "How it works": several rows in one pass with results identical to
single-row decode).  Row m of y must not depend on M, on its position among the
rows, or on the contents of the other rows; repeated calls give the same bits."""
import numpy as np
import pytest
import torch

import bit_row_speculative_gb300 as q4
import synth_inputs as si

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _y(x, W, N, K):
    return q4.matmul(x.contiguous(), W, N, K).cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "attn_in", "gate_up", "down", "gdn_in", "gdn_out", "lm_head"])
def test_rows_identical_across_M(name):
    N, K = si.SHAPES[name]
    W = si.make_weights(N, K, 5, device="cuda")
    # 32 rows: both record widths (16 rows for M <= 16, 32 rows above) must give the same bits
    x32 = si.make_x(32, K, 6, device="cuda")
    y32 = _y(x32, W, N, K)
    for M in range(1, 32):
        yM = _y(x32[:M], W, N, K)
        assert np.array_equal(yM, y32[:M]), f"M={M}"
    # each row alone, in every position, with other neighbours
    other = si.make_x(32, K, 9, device="cuda")
    for m in (0, 5, 15, 16, 31):
        alone = _y(x32[m:m + 1], W, N, K)
        assert np.array_equal(alone[0], y32[m])
        mixed = other.clone()
        mixed[31 - m] = x32[m]
        ym = _y(mixed, W, N, K)
        assert np.array_equal(ym[31 - m], y32[m])
        ym16 = _y(mixed[16:].contiguous(), W, N, K)          # the same row in a 16-row call
        if 31 - m >= 16:
            assert np.array_equal(ym16[15 - m], y32[m])


def test_run_to_run_determinism():
    N, K = si.SHAPES["attn_in"]
    W = si.make_weights(N, K, 12, device="cuda")
    x = si.make_x(16, K, 13, device="cuda")
    first = _y(x, W, N, K)
    for _ in range(5):
        assert np.array_equal(_y(x, W, N, K), first)
