"""GPU parity of q4_matmul against the CPU oracle (through the C ABI), on the
seeded synthetic inputs of every workload shape, plus hand-packed groups with
closed-form results and the degenerate cases."""
import numpy as np
import pytest
import torch

import bit_row_speculative_gb300 as q4
import oracle_pins as P
import synth_inputs as si
from parity import check_tolerance, run_and_check, sample_columns

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def test_tiny_workload_all_rows():
    """N=256, K=512, M=4, seed 0: every output against the oracle."""
    N, K, M = si.SHAPES["tiny"] + (4,)
    W = si.make_weights(N, K, si.w_seed(1))
    x = si.make_x(M, K, si.x_seed(1))
    run_and_check(x, W, N, K, what="tiny")


@pytest.mark.parametrize("M", list(range(1, 33)))
def test_tiny_shape_every_M(M):
    N, K = si.SHAPES["tiny"]
    W = si.make_weights(N, K, 7)
    x = si.make_x(M, K, 100 + M)
    run_and_check(x, W, N, K, what=f"tiny M={M}")


@pytest.mark.parametrize("N,K,M", [(1, 64, 1), (7, 64, 3), (33, 192, 16), (129, 576, 5), (1000, 1024, 16),
                                   (300, 2112, 2), (2, 4160, 9), (517, 5120, 16), (160, 4096, 8),
                                   (130, 17408, 16), (33, 192, 24), (517, 5120, 32), (130, 17408, 25),
                                   (1000, 1024, 17), (300, 2112, 31)])
def test_ragged_shapes(N, K, M):
    """Ragged N (tails of every tile size), small and odd K, and K spanning
    several shared-memory chunks."""
    W = si.make_weights(N, K, 31 + N)
    x = si.make_x(M, K, 77 + K)
    run_and_check(x, W, N, K, what=f"N={N} K={K} M={M}")


@pytest.mark.parametrize("name,Ms", [("attn_in", [1, 2, 4, 8, 16, 24, 32]), ("gate_up", [1, 16, 32]),
                                     ("down", [1, 16, 32]), ("gdn_in", [1, 16, 24]), ("gdn_out", [1, 16, 32])])
def test_model_shapes_sampled(name, Ms):
    """The 27B-shaped projections at full size; sampled columns against the oracle."""
    N, K = si.SHAPES[name]
    wl = 2 if name == "attn_in" else 3
    W = si.make_weights(N, K, si.w_seed(wl, list(si.SHAPES).index(name)), device="cuda")
    cols = sample_columns(N, 384, seed=N + K)
    for M in Ms:
        x = si.make_x(M, K, si.x_seed(wl) + M)
        run_and_check(x, W, N, K, cols=cols, what=f"{name} M={M}")


def test_lm_head_sampled():
    N, K = si.SHAPES["lm_head"]
    W = si.make_weights(N, K, si.w_seed(4), device="cuda")
    x = si.make_x(16, K, si.x_seed(4))
    run_and_check(x, W, N, K, cols=sample_columns(N, 256, seed=4), what="lm_head M=16")


def _gpu(x_np_f32, W_np, N, K):
    x = torch.from_numpy(np.ascontiguousarray(x_np_f32, dtype=np.float32)).to(torch.bfloat16)
    W = torch.from_numpy(np.ascontiguousarray(W_np))
    return q4.matmul(x.cuda(), W.cuda(), N, K).cpu().numpy().astype(np.float64)


def test_hand_packed_one_hot():
    """x = e_k returns w[n,k] = s*q_k + b exactly (nibble order, planes)."""
    rng = np.random.default_rng(11)
    N, K = 3, 128
    q = rng.integers(0, 16, size=(N, K))
    s = np.array([[0.5, 2.0], [0.25, 4.0], [1.0, 8.0]], dtype=np.float32)
    b = np.array([[-3.0, 0.75], [1.5, -0.125], [-64.0, 6.0]], dtype=np.float32)
    W = P.hand_pack(q, s, b)
    for M in (1, 16):
        xs = np.zeros((M, K), dtype=np.float32)
        ks = [(m * 37 + 5) % K for m in range(M)]
        for m, k in enumerate(ks):
            xs[m, k] = 1.0
        y = _gpu(xs, W, N, K)
        for m, k in enumerate(ks):
            want = s[:, k // 64].astype(np.float64) * q[:, k] + b[:, k // 64]
            assert np.array_equal(y[m], want), (M, m, k)


def test_hand_packed_closed_forms():
    K = 256
    ones = np.ones((2, K), dtype=np.float32)
    q = np.tile(np.arange(K) % 16, (2, 1))
    s = np.ones((2, K // 64), dtype=np.float32)
    y = _gpu(ones, P.hand_pack(q, s, np.full_like(s, -7.5)), 2, K)
    assert np.all(y == 0.0)
    y = _gpu(ones, P.hand_pack(np.full((2, K), 15), s, np.zeros_like(s)), 2, K)
    assert np.all(y == 15.0 * K)


def test_bf16_fold_detector():
    """Every w = 1 + 2^-8: a path that rounds w to bf16 fails the tolerance."""
    K = 5120
    q = np.ones((4, K), dtype=np.int64)
    s = np.full((4, K // 64), 2.0**-8, dtype=np.float32)
    b = np.ones((4, K // 64), dtype=np.float32)
    y = _gpu(np.ones((16, K), np.float32), P.hand_pack(q, s, b), 4, K)
    exact = K * (1 + 2.0**-8)
    check_tolerance(y, np.full_like(y, exact), np.full_like(y, exact), "fold detector")


def test_degenerate_zero_outputs():
    """x = 0 and w = 0 (q = c, b = -c*s) must give exactly zero."""
    rng = np.random.default_rng(3)
    N, K = 40, 1024
    s = np.full((N, K // 64), 0.0078125, dtype=np.float32)
    q = rng.integers(0, 16, size=(N, K))
    W = P.hand_pack(q, s, np.full_like(s, -0.0625))
    assert np.all(_gpu(np.zeros((5, K), np.float32), W, N, K) == 0.0)
    for c in (0, 3, 8, 15):
        Wc = P.hand_pack(np.full((N, K), c), s, np.full_like(s, -c * 0.0078125))
        xr = rng.standard_normal((16, K)).astype(np.float32)
        assert np.all(_gpu(xr, Wc, N, K) == 0.0), c


def test_wide_dynamic_range():
    """Scales and biases across many binades, x with mixed magnitudes."""
    rng = np.random.default_rng(17)
    N, K, M = 64, 2048, 16
    G = K // 64
    q = rng.integers(0, 16, size=(N, K))
    s = np.exp2(rng.integers(-20, 6, size=(N, G))).astype(np.float32)
    b = (-s * rng.integers(0, 16, size=(N, G)) * np.exp2(rng.integers(-3, 3, size=(N, G)))).astype(np.float32)
    b = (b.view(np.uint32) & 0xFFFF0000).view(np.float32)
    xr = (rng.standard_normal((M, K)) * np.exp2(rng.integers(-10, 10, size=(M, K)))).astype(np.float32)
    xr = (xr.view(np.uint32) & 0xFFFF0000).view(np.float32)
    W = P.hand_pack(q, s, b)
    x = torch.from_numpy(xr).to(torch.bfloat16)
    run_and_check(x, torch.from_numpy(W), N, K, what="dynamic range")


def _bf16_magnitudes(rng, shape, lo_exp, hi_exp):
    """Random signs, |x| uniform in binades [2^lo_exp, 2^hi_exp), as bf16-exact float32."""
    e = rng.integers(lo_exp, hi_exp, size=shape)
    v = rng.choice([-1.0, 1.0], size=shape) * (1.0 + rng.random(shape)) * np.exp2(e)
    return (v.astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)


def test_x_range_window_edges():
    """The activation range the header states, |x| in [2^-93, 2^28): rows drawn
    from the lowest binades (2^-93 .. 2^-90), from the highest (2^26 .. 2^27),
    and rows mixing both ends with normal values, against the oracle."""
    rng = np.random.default_rng(23)
    N, K, M = 200, 2048, 16
    W = si.make_weights(N, K, 29)
    xr = rng.standard_normal((M, K)).astype(np.float32)
    xr = (xr.view(np.uint32) & 0xFFFF0000).view(np.float32)
    xr[0] = _bf16_magnitudes(rng, K, -93, -90)
    xr[3] = _bf16_magnitudes(rng, K, 27, 28)                  # the top binade: |x| < 2^28
    xr[7] = _bf16_magnitudes(rng, K, -93, 27)                 # every binade of the window in one row
    xr[9, : K // 2] = _bf16_magnitudes(rng, K // 2, -93, -92)
    xr[9, K // 2:] = _bf16_magnitudes(rng, K // 2, 27, 28)
    xr[15] = 0.0
    xr[15, ::97] = _bf16_magnitudes(rng, xr[15, ::97].shape, -93, -92)   # a sparse row of tiny values
    x = torch.from_numpy(xr).to(torch.bfloat16)
    for rows in (slice(0, 16), slice(0, 1), slice(3, 4), slice(15, 16)):
        run_and_check(x[rows].contiguous(), W, N, K, what=f"x range rows {rows}")
