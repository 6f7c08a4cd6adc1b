"""Pins for the CPU oracle: checks against values that do not come from the
oracle itself.  Each pin takes an ``oracle.Oracle`` (the real one, or a
deliberately broken copy built by the mutation tests) and raises
AssertionError when the oracle disagrees with the pin.

Weight format under test ("Splash engine" page, section "The engine hard-codes
the model"): 32 bytes of unsigned nibbles plus a bf16 scale and a bf16 bias per
group of 64 inputs; w = scale*q + bias; low nibble = even input; planes laid
out [nibbles][scales][biases].
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

GROUP = 64
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- hand packing
def bf16_bits_exact(values) -> np.ndarray:
    """Bit patterns of values that are exactly representable in bf16."""
    f = np.asarray(values, dtype=np.float32)
    u = f.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("value not exactly representable in bf16")
    return (u >> 16).astype(np.uint16)


def hand_pack(q: np.ndarray, s: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Pack integer nibbles q [N,K] (0..15), exact-bf16 scales s and biases b
    [N, K/64] into the planar byte layout, written out directly from the
    format description (independent of any generator)."""
    q = np.asarray(q, dtype=np.int64)
    N, K = q.shape
    assert K % GROUP == 0 and q.min() >= 0 and q.max() <= 15
    nib = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)      # low nibble = even input
    sb = bf16_bits_exact(s).reshape(N, K // GROUP)
    bb = bf16_bits_exact(b).reshape(N, K // GROUP)
    s_bytes = np.stack([sb & 0xFF, sb >> 8], axis=-1).astype(np.uint8).reshape(-1)
    b_bytes = np.stack([bb & 0xFF, bb >> 8], axis=-1).astype(np.uint8).reshape(-1)
    return np.concatenate([nib.reshape(-1), s_bytes, b_bytes])


def x_bits(values) -> np.ndarray:
    return bf16_bits_exact(values)


def random_exact_case(rng: np.random.Generator, M: int, N: int, K: int):
    """Random q, bf16-exact s, b, x (values drawn as small-mantissa numbers)."""
    G = K // GROUP
    q = rng.integers(0, 16, size=(N, K))
    # bf16-exact values: 8-bit signed significand times a power of two
    def exact(shape, lo_exp, hi_exp):
        mant = rng.integers(-255, 256, size=shape).astype(np.float64)
        ex = rng.integers(lo_exp, hi_exp + 1, size=shape)
        v = (mant * np.exp2(ex - 7)).astype(np.float32)
        # round away any bits bf16 cannot hold (mantissa up to 255 needs 8 bits: fine)
        return v
    s = np.abs(exact((N, G), -10, -5))
    b = exact((N, G), -8, -3)
    x = exact((M, K), -3, 2)
    return q, s, b, x


# --------------------------------------------------------------------- pins
def pin_packed_bytes(o) -> None:
    """Closed form N*K/16*9 for every workload shape; 0 for bad shapes."""
    cases = {
        (256, 512): 73_728,
        (14336, 5120): 41_287_680,
        (34816, 5120): 100_270_080,
        (5120, 17408): 50_135_040,
        (16640, 5120): 47_923_200,
        (5120, 6144): 17_694_720,
        (248320, 5120): 715_161_600,
    }
    for (N, K), want in cases.items():
        assert o.packed_bytes(N, K) == want, (N, K)
    for N, K in [(0, 64), (1, 0), (1, 32), (3, 100), (1, 65)]:
        assert o.packed_bytes(N, K) == 0, (N, K)
    big = 1 << 40
    assert o.packed_bytes(big, big) == 0          # N*K overflows 64 bits
    assert o.packed_bytes(1, 64) == 36


def read_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split()
            out[k] = float(v)
    return out


def model_byte_accounting(o) -> dict:
    """Byte accounting of the 27B-class hybrid built from the page's model struct
    and the oracle's packed-size function.  The per-matrix decomposition is this
    project's reconstruction (the page prints only totals)."""
    L, H, V, I = 64, 5120, 248320, 17408
    n_attn = L // 4                       # every fourth layer is full attention
    n_gdn = L - n_attn
    mats = []                              # (N, K, count)
    mats += [(2 * I, H, L), (H, I, L)]     # MLP gate/up, down
    mats += [(14336, H, n_attn), (H, 24 * 256, n_attn)]          # attention in / out
    mats += [(16640, H, n_gdn), (H, 48 * 128, n_gdn)]             # GDN in / out
    mats += [(V, H, 1), (V, H, 1)]         # input embedding, LM head
    q4_params = sum(N * K * c for N, K, c in mats)
    q4_bytes = sum(o.packed_bytes(N, K) * c for N, K, c in mats)
    # non-Q4 bf16 parameters (reconstruction): GDN conv1d, RMSNorm weights,
    # A_log + dt_bias, GDN head norms, q/k norms
    extra = 48 * 10240 * 4 + (64 * 2 * 5120 + 5120) + 48 * 96 + 48 * 128 + 16 * 512
    embed_bytes = o.packed_bytes(V, H)
    return {"q4_params": q4_params, "q4_bytes": q4_bytes, "extra_params": extra,
            "params": q4_params + extra, "bytes": q4_bytes + 2 * extra,
            "embed_bytes": embed_bytes, "lm_head_bytes": o.packed_bytes(V, H)}


def pin_model_totals(o) -> None:
    g = read_golden("qwen38_27b_bytes.txt")
    acc = model_byte_accounting(o)
    assert acc["params"] == int(g["total_params"])
    assert round(acc["bytes"] / 1e9, 3) == g["total_gb"]
    assert round(acc["lm_head_bytes"] / 1e6) == g["lm_head_mb"]
    # draft-free step: every weight but the untied input embedding, plus the
    # recurrent state read and written back
    state = g["gdn_state_mib"] * 2**20
    step = acc["bytes"] - acc["embed_bytes"] + 2 * state
    assert round(307e9 / step, 1) == g["draft_free_bound_tok_s_at_307"]
    # arithmetic intensity: 2*M flops per weight over the bytes per weight
    bpw = o.packed_bytes(1, 64) / 64
    assert round(2 * 8 / bpw) == g["intensity_flop_per_byte_m8"]
    assert round(2 * 32 / bpw) == g["intensity_flop_per_byte_m32"]


def pin_one_hot(o) -> None:
    """x = e_k picks out w[n,k] = s*q_k + b: identifies the low/high nibble and
    which plane holds the scale and which the bias."""
    rng = np.random.default_rng(11)
    N, K = 3, 128
    q = rng.integers(0, 16, size=(N, K))
    s = np.array([[0.5, 2.0], [0.25, 4.0], [1.0, 8.0]], dtype=np.float32)
    b = np.array([[-3.0, 0.75], [1.5, -0.125], [-64.0, 6.0]], dtype=np.float32)
    W = hand_pack(q, s, b)
    for k in [0, 1, 2, 3, 30, 31, 62, 63, 64, 65, 100, 127]:
        xv = np.zeros((1, K), dtype=np.float32)
        xv[0, k] = 1.0
        y, a = o.matmul(x_bits(xv), W, N, K, threads=1)
        for n in range(N):
            want = float(s[n, k // 64]) * int(q[n, k]) + float(b[n, k // 64])
            assert y[0, n] == want, (n, k, y[0, n], want)
            assert a[0, n] == abs(want)


def pin_group_closed_forms(o) -> None:
    K = 256
    ones = x_bits(np.ones((1, K), dtype=np.float32))
    # q_k = k mod 16, s = 1, b = -7.5: every group sums to zero
    q = np.tile(np.arange(K) % 16, (2, 1))
    s = np.ones((2, K // 64), dtype=np.float32)
    b = np.full((2, K // 64), -7.5, dtype=np.float32)
    y, _ = o.matmul(ones, hand_pack(q, s, b), 2, K, threads=1)
    assert np.all(y == 0.0)
    # all q = 15, s = 1, b = 0: 15 * K
    q = np.full((2, K), 15)
    y, _ = o.matmul(ones, hand_pack(q, s, np.zeros_like(s)), 2, K, threads=1)
    assert np.all(y == 15.0 * K)
    # per-group scale 2^g and bias b_g with x = 1: sum_g (2^g * sum q + 64 b_g)
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, size=(1, K))
    s = np.exp2(np.arange(K // 64, dtype=np.float32))[None, :]
    b = np.array([[0.5, -1.0, 2.0, -0.25]], dtype=np.float32)
    y, _ = o.matmul(ones, hand_pack(q, s, b), 1, K, threads=1)
    want = sum(2.0**g * int(q[0, 64 * g:64 * g + 64].sum()) + 64 * float(b[0, g]) for g in range(K // 64))
    assert y[0, 0] == want


def pin_bf16_fold_detector(o) -> None:
    """x = 1, s = 2^-8, q = 1, b = 1: every w = 1 + 2^-8 exactly, y = K*(1 + 2^-8).
    A path that rounds w to bf16 gets 1.0 per weight (a tie to even) and misses
    the 2e-3 relative tolerance."""
    K = 512
    q = np.ones((1, K), dtype=np.int64)
    s = np.full((1, K // 64), 2.0**-8, dtype=np.float32)
    b = np.ones((1, K // 64), dtype=np.float32)
    y, a = o.matmul(x_bits(np.ones((1, K), np.float32)), hand_pack(q, s, b), 1, K, threads=1)
    assert y[0, 0] == K * (1 + 2.0**-8)
    assert a[0, 0] == K * (1 + 2.0**-8)
    folded = K * 1.0
    assert abs(folded - y[0, 0]) > 2e-3 * a[0, 0]


def exact_rational(q, s, b, x):
    """sum_g s_g * (sum_{k in g} q_k x_k) + b_g * (sum_{k in g} x_k), exactly."""
    M, K = x.shape
    N = q.shape[0]
    out = [[Fraction(0)] * N for _ in range(M)]
    absout = [[Fraction(0)] * N for _ in range(M)]
    xf = [[Fraction(float(v)) for v in row] for row in x]
    for n in range(N):
        for m in range(M):
            tot = Fraction(0)
            atot = Fraction(0)
            for g in range(K // GROUP):
                sg, bg = Fraction(float(s[n, g])), Fraction(float(b[n, g]))
                P = sum(int(q[n, k]) * xf[m][k] for k in range(g * GROUP, (g + 1) * GROUP))
                X = sum(xf[m][k] for k in range(g * GROUP, (g + 1) * GROUP))
                tot += sg * P + bg * X
                atot += sum(abs(xf[m][k] * (sg * int(q[n, k]) + bg))
                            for k in range(g * GROUP, (g + 1) * GROUP))
            out[m][n] = tot
            absout[m][n] = atot
    return out, absout


def pin_exact_rational(o, seeds=(1, 2, 3)) -> None:
    """Random tiny shapes against exact rational arithmetic: the fp64 result
    must lie within K * 2^-53 * sum|x*w| of the exact value."""
    for seed in seeds:
        rng = np.random.default_rng(seed)
        M, N, K = 3, 5, 128 if seed % 2 else 64
        q, s, b, x = random_exact_case(rng, M, N, K)
        W = hand_pack(q, s, b)
        y, a = o.matmul(x_bits(x), W, N, K, threads=2)
        ex, eabs = exact_rational(q, s, b, x)
        for m in range(M):
            for n in range(N):
                bound = K * 2.0**-53 * float(eabs[m][n]) * 1.01
                assert abs(Fraction(y[m, n]) - ex[m][n]) <= Fraction(bound), (m, n)
                assert abs(a[m, n] - float(eabs[m][n])) <= bound + 1e-300


def pin_zero_cases(o) -> None:
    rng = np.random.default_rng(9)
    N, K = 4, 192
    q = rng.integers(0, 16, size=(N, K))
    s = np.full((N, K // 64), 0.125, dtype=np.float32)
    b = np.full((N, K // 64), -1.0, dtype=np.float32)
    W = hand_pack(q, s, b)
    y, a = o.matmul(x_bits(np.zeros((2, K), np.float32)), W, N, K)
    assert np.all(y == 0.0) and np.all(a == 0.0)
    # w == 0 everywhere: q = c with b = -c*s
    c = 8
    qc = np.full((N, K), c)
    bc = np.full((N, K // 64), -c * 0.125, dtype=np.float32)
    xv = rng.standard_normal((2, K)).astype(np.float32)
    xv = (xv.view(np.uint32) & 0xFFFF0000).view(np.float32)
    y, a = o.matmul(x_bits(xv), hand_pack(qc, s, bc), N, K)
    assert np.all(y == 0.0) and np.all(a == 0.0)


def pin_scaling_invariants(o) -> None:
    """Exact invariants of a linear map in binary floating point: scaling x by 2
    scales y exactly; columns do not depend on which other columns are asked
    for; the thread count changes nothing."""
    rng = np.random.default_rng(21)
    M, N, K = 2, 9, 256
    q, s, b, x = random_exact_case(rng, M, N, K)
    W = hand_pack(q, s, b)
    y1, _ = o.matmul(x_bits(x), W, N, K, threads=1)
    y2, _ = o.matmul(x_bits(2 * x), W, N, K, threads=3)
    assert np.array_equal(y2, 2 * y1)
    cols = np.array([7, 0, 3], dtype=np.int64)
    yc, _ = o.matmul(x_bits(x), W, N, K, cols=cols, threads=2)
    assert np.array_equal(yc, y1[:, cols])


def pin_bf16_rounding(o) -> None:
    """Round-to-nearest-even to bf16, from the IEEE definition."""
    cases = [
        (1.0, 0x3F80),
        (1.0 + 2.0**-8, 0x3F80),                 # tie -> even (down)
        (1.0 + 3 * 2.0**-8, 0x3F82),             # tie -> even (up)
        (1.0 + 2.0**-8 + 2.0**-30, 0x3F81),      # just above the tie
        (-2.5, 0xC020),
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0**-133, 0x0001),                     # smallest subnormal
        (3.0 * 2.0**-134, 0x0002),               # subnormal tie -> even
        (3.3895313892515355e38, 0x7F7F),         # largest finite bf16
        (3.4e38, 0x7F80),                        # rounds past the largest: inf
        (float("inf"), 0x7F80),
    ]
    for v, want in cases:
        assert o.f64_to_bf16(v) == want, (v, hex(o.f64_to_bf16(v)), hex(want))
    assert o.bf16_to_f64(0x3F81) == 1.0 + 2.0**-7


def pin_glue(o) -> None:
    """Glue closed forms: RMS-normalising a constant row gives 1/sqrt(1+eps/c^2)
    (bf16 1.0 for |c| >> sqrt(eps)); silu(0) = 0; a 3-4 row normalises to
    3/sqrt(12.5) and 4/sqrt(12.5); silu(a) -> a for large a."""
    K = 64
    y = np.full((2, K), 3.0, dtype=np.float32)
    y[1] = -0.5
    x = o.glue(y, K, 1)
    assert np.all(x[0] == 0x3F80) and np.all(x[1] == 0xBF80)
    # RMSNORM reads only the first K columns of a wider y
    yw = np.concatenate([y, np.full((2, 32), 1e6, np.float32)], axis=1)
    assert np.array_equal(o.glue(yw, K, 1), x)
    # two-value row: [3, 4] repeated -> mean square 12.5
    y2 = np.tile(np.array([3.0, 4.0], np.float32), (1, K // 2))
    x2 = o.glue(y2, K, 1)
    r = 1.0 / math.sqrt(12.5 + 1e-6)
    assert x2[0, 0] == o.f64_to_bf16(3 * r) == 0x3F59   # 0.8485 -> 0.84765625
    assert x2[0, 1] == o.f64_to_bf16(4 * r) == 0x3F91   # 1.1314 -> 1.1328125
    # SwiGLU: gate 0 -> silu 0 -> all-zero row -> zeros
    g = np.zeros((1, 2 * K), np.float32)
    g[0, K:] = 5.0
    assert np.all(o.glue(g, K, 2) == 0)
    # gate 30 (silu(30) = 30 to within 3e-12), up 1: constant row -> 1.0
    g = np.concatenate([np.full((1, K), 30.0, np.float32), np.ones((1, K), np.float32)], axis=1)
    assert np.all(o.glue(g, K, 2) == 0x3F80)
    pin_swiglu_orientation(o)


def pin_swiglu_orientation(o) -> None:
    """Which half of y is the gate.  Row 0: gate = 30 on the first 32 inputs and
    0 on the last 32; up alternates 1, 2 (and 7 where the gate is 0).  Then
    v = silu(gate) * up = [30, 60, 30, 60, ..., 0, ..., 0] up to 1e-13 relative,
    mean square (16*900 + 16*3600) / 64 = 1125, so x = 30/sqrt(1125) = 2/sqrt(5)
    -> bf16 229/256 = 0x3F65 and 60/sqrt(1125) = 4/sqrt(5) -> 229/128 = 0x3FE5,
    and exactly 0 where the gate is 0.  Row 1 flips the sign of the odd ups:
    -2/sqrt(5) -> 0xBF65.  With the halves swapped, v = silu(up) * gate gives
    silu(1)*30 : silu(2)*30 = 0.731 : 1.762, not 1 : 2, and nonzero values where
    the gate is 0, so every output differs."""
    K = 64
    gate = np.zeros((2, K), np.float32)
    gate[:, :32] = 30.0
    up = np.zeros((2, K), np.float32)
    up[:, 0:32:2] = 1.0
    up[:, 1:32:2] = 2.0
    up[:, 32:] = 7.0
    up[1, 0:32:2] = -1.0
    x = o.glue(np.concatenate([gate, up], axis=1), K, 2)
    want0 = np.array([0x3F65, 0x3FE5] * 16 + [0] * 32, dtype=np.uint16)
    want1 = np.array([0xBF65, 0x3FE5] * 16 + [0] * 32, dtype=np.uint16)
    assert np.array_equal(x[0], want0), [hex(v) for v in x[0][:4]]
    assert np.array_equal(x[1], want1), [hex(v) for v in x[1][:4]]


ALL_PINS = [pin_packed_bytes, pin_model_totals, pin_one_hot, pin_group_closed_forms,
            pin_bf16_fold_detector, pin_exact_rational, pin_zero_cases,
            pin_scaling_invariants, pin_bf16_rounding, pin_glue]
