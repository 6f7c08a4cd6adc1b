"""Pins of the edge-score oracle (oracle/edges.py) against values that do not
come from the oracle: one-hot codebook rows whose scores are read off by hand,
exact integer brute force in Python integers, the special case hidden = 1 that
reduces the trilinear form to a dot product (numpy's), exact scaling, and the
last dimension of a full rank-256 row.  Every pin also runs against copies of
the oracle with one plausible mistake planted, and must catch each one."""
import math

import numpy as np
import pytest

from oracle import edges as E


def bf16_exact(values) -> np.ndarray:
    """bf16 bit patterns of values that bf16 holds exactly (small integers, powers of two)."""
    f = np.asarray(values, dtype=np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exact in bf16"
    return (u >> 16).astype(np.uint16)


def bf16_random(rng, shape) -> np.ndarray:
    """bf16 bit patterns of random values (truncated fp32: any bf16 is a valid input)."""
    f = (rng.standard_normal(shape) * 0.25).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def pin_one_hot(f):
    # predecessor rows 2 and 4 are unit vectors e_3 and e_7; successor rows 1 and 5 are e_3 and e_7
    V, R = 6, 16
    P = np.zeros((V, R), np.float32)
    S = np.zeros((V, R), np.float32)
    P[2, 3] = P[4, 7] = 1.0
    S[1, 3] = S[5, 7] = 1.0
    hidden = np.stack([np.arange(1, R + 1), 100 + np.arange(R)]).astype(np.float32)
    pred = np.array([[2] * 8 + [4] * 8, [4] * 16])
    cand = np.array([[1, 5] * 8, [5] * 8 + [1] * 8])
    got = f(bf16_exact(P), bf16_exact(S), hidden, pred, cand)
    want = np.zeros((2, 16, 16))
    for i in range(16):
        for j in range(16):
            if i < 8 and j % 2 == 0:
                want[0, i, j] = hidden[0, 3]          # 4
            if i >= 8 and j % 2 == 1:
                want[0, i, j] = hidden[0, 7]          # 8
            if j < 8:
                want[1, i, j] = hidden[1, 7]          # 107
    assert np.array_equal(got, want)


def pin_integer_brute_force(f):
    rng = np.random.default_rng(5)
    V, R, rows = 10, 32, 3
    Pi = rng.integers(-8, 9, size=(V, R))
    Si = rng.integers(-8, 9, size=(V, R))
    Hi = rng.integers(-16, 17, size=(rows, R))
    pred = rng.integers(0, V, size=(rows, 16))
    cand = rng.integers(0, V, size=(rows, 16))
    got = f(bf16_exact(Pi), bf16_exact(Si), Hi.astype(np.float32), pred, cand)
    for r in range(rows):
        for i in range(16):
            for j in range(16):
                exact = sum(int(Pi[pred[r, i], d]) * int(Hi[r, d]) * int(Si[cand[r, j], d]) for d in range(R))
                assert got[r, i, j] == exact


def pin_dot_product_case(f):
    # hidden = 1: the trilinear form is the dot product of the two codebook rows
    rng = np.random.default_rng(6)
    V, R = 50, 256
    P, S = bf16_random(rng, (V, R)), bf16_random(rng, (V, R))
    pred = rng.integers(0, V, size=(2, 16))
    cand = rng.integers(0, V, size=(2, 16))
    got = f(P, S, np.ones((2, R), np.float32), pred, cand)
    Pf, Sf = E.bf16_bits_to_f64(P), E.bf16_bits_to_f64(S)
    for r in range(2):
        want = Pf[pred[r]] @ Sf[cand[r]].T
        assert np.allclose(got[r], want, rtol=1e-12, atol=1e-12)


def pin_scaling(f):
    # hidden times 2^5: every score times 2^5, exactly
    rng = np.random.default_rng(8)
    V, R = 40, 64
    P, S = bf16_random(rng, (V, R)), bf16_random(rng, (V, R))
    h = rng.standard_normal((2, R)).astype(np.float32)
    pred = rng.integers(0, V, size=(2, 16))
    cand = rng.integers(0, V, size=(2, 16))
    a = f(P, S, h, pred, cand)
    b = f(P, S, h * np.float32(32.0), pred, cand)
    assert np.array_equal(b, a * 32.0)
    assert not np.array_equal(a, np.zeros_like(a))


def pin_last_dimension(f):
    # full rank 256: only the last dimension is nonzero in both codebooks
    V, R = 3, 256
    P = np.zeros((V, R), np.float32)
    S = np.zeros((V, R), np.float32)
    P[1, R - 1] = 2.0
    S[2, R - 1] = 0.5
    h = np.full((1, R), 3.0, np.float32)
    got = f(bf16_exact(P), bf16_exact(S), h, np.full((1, 16), 1), np.full((1, 16), 2))
    assert np.all(got == 3.0)


PINS = [pin_one_hot, pin_integer_brute_force, pin_dot_product_case, pin_scaling, pin_last_dimension]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(E.edge_scores)


def test_rejects_out_of_range_ids():
    P = np.zeros((4, 8), np.uint16)
    with pytest.raises(ValueError):
        E.edge_scores(P, P, np.zeros((1, 8), np.float32), np.full((1, 16), 4), np.zeros((1, 16), int))
    with pytest.raises(ValueError):
        E.edge_scores(P, P, np.zeros((1, 8), np.float32), np.zeros((1, 16), int), np.full((1, 16), -1))


def test_abs_terms_bounds_the_score():
    rng = np.random.default_rng(9)
    P, S = bf16_random(rng, (20, 64)), bf16_random(rng, (20, 64))
    h = rng.standard_normal((2, 64)).astype(np.float32)
    pred, cand = rng.integers(0, 20, size=(2, 16)), rng.integers(0, 20, size=(2, 16))
    assert np.all(np.abs(E.edge_scores(P, S, h, pred, cand)) <= E.abs_terms(P, S, h, pred, cand) * (1 + 1e-12))


# ------------------------------------------------------------ planted mistakes
def _mutant(transpose=False, no_hidden=False, next_row_hidden=False, succ_for_both=False, drop_last=False,
            low_half=False):
    def widen(bits):
        if low_half:
            return np.asarray(bits, np.uint16).astype(np.uint32).view(np.float32).astype(np.float64)
        return E.bf16_bits_to_f64(bits)

    def f(pred_cb, succ_cb, hidden, pred_ids, cand_ids):
        pred_cb = np.asarray(pred_cb, np.uint16)
        succ_cb = np.asarray(succ_cb, np.uint16)
        rows, R = hidden.shape
        out = np.zeros((rows, 16, 16))
        for r in range(rows):
            h = np.asarray(hidden[(r + 1) % rows if next_row_hidden else r], np.float64)
            if no_hidden:
                h = np.ones(R)
            for i in range(16):
                ctx = widen((succ_cb if succ_for_both else pred_cb)[pred_ids[r][i]]) * h
                for j in range(16):
                    t = ctx * widen(succ_cb[cand_ids[r][j]])
                    if drop_last:
                        t = t[:-1]
                    v = math.fsum(t.tolist())
                    if transpose:
                        out[r, j, i] = v
                    else:
                        out[r, i, j] = v
        return out
    return f


MUTANTS = {
    "output_transposed": _mutant(transpose=True),
    "hidden_ignored": _mutant(no_hidden=True),
    "hidden_of_next_row": _mutant(next_row_hidden=True),
    "successor_codebook_for_both": _mutant(succ_for_both=True),
    "last_dimension_dropped": _mutant(drop_last=True),
    "bf16_as_low_half": _mutant(low_half=True),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    caught = 0
    for pin in PINS:
        try:
            pin(MUTANTS[name])
        except (AssertionError, ArithmeticError):
            caught += 1
    assert caught > 0, f"no pin catches the planted mistake {name}"


def test_unmutated_copy_passes():
    for pin in PINS:
        pin(_mutant())
