"""q4_topk_probs on the GPU against the oracle (oracle/topk.py): indices bit-exact
(the order logit-descending, ties to the lower index, is unique), probabilities
within 2 float ulps of the double-precision oracle.  LM-head-sized rows
(248,320 logits) with planted ties across slice boundaries, every M, several
top_k / temperature / top_p, rows independent of the other rows, determinism,
and the epilogue chained after the LM-head matmul."""
import numpy as np
import pytest
import torch

import bit_row_speculative_gb300 as q4
import synth_inputs as si
from oracle import topk as T

pytestmark = pytest.mark.gpu

VOCAB = 248320


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _logits(M, N, seed, ties=True):
    g = torch.Generator().manual_seed(seed)
    y = (torch.randn((M, N), generator=g) * 3.0).to(torch.float32)
    if ties:
        # the row's maximum copied to other positions, some across 16K-slice boundaries
        for m in range(M):
            j = int(torch.argmax(y[m]))
            for t in (5, 16383, 16384, 70000, N - 1):
                if t < N:
                    y[m, t] = y[m, j]
            y[m, 3] = y[m, 16390] = -0.0
            y[m, 4] = 0.0
    return y


def _check(y, k, temp, p):
    idx, pr = q4.topk_probs(y.cuda(), k, temp, p)
    q4.device_status()
    # the library takes temperature and top_p as fp32: the oracle gets the same values
    ref_i, ref_p = T.topk_probs(y.numpy(), k, float(np.float32(temp)), float(np.float32(p)))
    assert np.array_equal(idx.cpu().numpy(), ref_i), "indices differ from the oracle"
    got = pr.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref_p) <= 2.0 * np.spacing(np.float32(np.maximum(ref_p, 1e-38))) + 1e-45)


@pytest.mark.parametrize("M", [1, 3, 16, 32])
@pytest.mark.parametrize("k,temp,p", [(32, 1.0, 1.0), (20, 0.7, 0.95), (1, 1.0, 1.0), (8, 2.5, 0.5)])
def test_lm_head_rows_against_oracle(M, k, temp, p):
    _check(_logits(M, VOCAB, 100 + M + k), k, temp, p)


@pytest.mark.parametrize("N", [7, 32, 100, 8192, 8193, 16384, 16385, 40000])
def test_small_and_ragged_rows(N):
    _check(_logits(4, N, N, ties=N > 20000), 32 if N >= 32 else N, 1.3, 0.9)


@pytest.mark.parametrize("pattern", ["ascending", "descending", "crowded_threads", "plateau"])
def test_adversarial_orders(pattern):
    """Orders that defeat a bound taken from per-thread maxima as far as it can
    be defeated: sorted rows, the largest logits crowded into few threads of a
    slice (every candidate of 32 threads passes), and a plateau of equal values
    just below a few larger ones."""
    M, N = 3, 50000
    g = torch.Generator().manual_seed(3)
    y = torch.randn((M, N), generator=g).to(torch.float32)
    if pattern == "ascending":
        y = torch.sort(y, dim=1).values
    elif pattern == "descending":
        y = torch.sort(y, dim=1, descending=True).values
    elif pattern == "crowded_threads":
        pos = torch.arange(N)
        y[:, (pos % 256) < 32] += 100.0          # thread-strided positions of the first 32 threads of each slice
    else:
        y[:, ::3] = 2.0
        y[:, 1000:1005] = 3.0
    _check(y, 32, 1.1, 0.97)


def test_all_equal_logits():
    y = torch.full((2, 50000), 1.25, dtype=torch.float32)
    idx, pr = q4.topk_probs(y.cuda(), 32, 1.0, 1.0)
    assert idx.cpu()[0].tolist() == list(range(32))
    assert torch.all(pr.cpu() == 1.0 / 32)


def test_rows_independent_and_deterministic():
    y = _logits(16, VOCAB, 7)
    idx, pr = q4.topk_probs(y.cuda(), 32, 0.8, 0.9)
    for m in (0, 9, 15):
        i1, p1 = q4.topk_probs(y[m:m + 1].contiguous().cuda(), 32, 0.8, 0.9)
        assert torch.equal(i1[0].cpu(), idx[m].cpu()) and torch.equal(p1[0].cpu(), pr[m].cpu())
    i2, p2 = q4.topk_probs(y.cuda(), 32, 0.8, 0.9)
    assert torch.equal(i2, idx) and torch.equal(p2, pr)


def test_after_lm_head_matmul():
    """The epilogue on the LM head's own output, chained on one stream."""
    N, K = si.SHAPES["lm_head"]
    W = si.make_weights(N, K, si.w_seed(4), device="cuda")
    x = si.make_x(16, K, si.x_seed(4), device="cuda")
    y = q4.matmul(x, W, N, K)
    idx, pr = q4.topk_probs(y, 32, 1.0, 0.95)
    q4.device_status()
    ref_i, ref_p = T.topk_probs(y.cpu().numpy(), 32, 1.0, 0.95)
    assert np.array_equal(idx.cpu().numpy(), ref_i)
    assert np.allclose(pr.cpu().numpy(), ref_p, rtol=3e-7, atol=1e-30)


@pytest.mark.parametrize("M", [1, 16, 32])
def test_fused_head_equals_matmul_then_epilogue(M):
    """q4_lm_head_topk (logits in the library's scratch, discarded from L2 after
    the epilogue reads them) gives the same bits as q4_matmul + q4_topk_probs,
    call after call (the scratch is rewritten each time)."""
    N, K = si.SHAPES["lm_head"]
    W = si.make_weights(N, K, si.w_seed(4), device="cuda")
    for seed in (1, 2):
        x = si.make_x(M, K, si.x_seed(4) + 10 * M + seed, device="cuda")
        i_f, p_f = q4.lm_head_topk(x, W, N, K, 32, 0.9, 0.95)
        y = q4.matmul(x, W, N, K)
        i_s, p_s = q4.topk_probs(y, 32, 0.9, 0.95)
        q4.device_status()
        assert torch.equal(i_f, i_s) and torch.equal(p_f, p_s)


def test_fused_head_ragged_rows():
    """A row length that is not a multiple of 32 floats: slices that do not end
    on a 128-byte line keep their boundary lines (only whole lines are dropped)."""
    N, K = 40009, 1024
    W = si.make_weights(N, K, 77, device="cuda")
    x = si.make_x(5, K, 78, device="cuda")
    i_f, p_f = q4.lm_head_topk(x, W, N, K, 20, 1.3, 0.8)
    y = q4.matmul(x, W, N, K)
    i_s, p_s = q4.topk_probs(y, 20, 1.3, 0.8)
    q4.device_status()
    assert torch.equal(i_f, i_s) and torch.equal(p_f, p_s)
    ref_i, _ = T.topk_probs(y.cpu().numpy(), 20, float(np.float32(1.3)), float(np.float32(0.8)))
    assert np.array_equal(i_f.cpu().numpy(), ref_i)
