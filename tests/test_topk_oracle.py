"""Pins of the sampling-epilogue oracle (oracle/topk.py) against values that do
not come from the oracle: hand-built rankings, probabilities that are exact in
binary (uniform logits), closed forms of a two-way softmax, exact invariances,
and a brute-force ranking by Python's sort.  Each pin also runs against copies
of the oracle with one plausible mistake planted, and must catch every one."""
import math

import numpy as np
import pytest

from oracle import topk as T


def pin_tie_order(f):
    # equal logits rank by lower index first; the largest logit first
    logits = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, -1.0]], dtype=np.float32)
    idx, _ = f(logits, 5, 1.0, 1.0)
    assert idx[0, :5].tolist() == [1, 2, 4, 3, 0]
    assert idx[0, 5:].tolist() == [-1] * 27


def pin_uniform_exact(f):
    # uniform logits: every exp is exactly 1, so the probabilities are exact
    logits = np.full((2, 40), 7.5, dtype=np.float32)
    idx, p = f(logits, 4, 0.7, 1.0)
    assert idx[0, :4].tolist() == [0, 1, 2, 3]
    assert p[0, :4].tolist() == [0.25] * 4 and p[0, 4:].sum() == 0.0
    _, p = f(logits, 4, 0.7, 0.5)            # 0.25 + 0.25 reaches 0.5: two kept
    assert p[0, :4].tolist() == [0.5, 0.5, 0.0, 0.0]
    _, p = f(logits, 4, 0.7, 0.51)           # the entry that crosses is kept
    assert p[0, :3].tolist() == pytest.approx([1 / 3] * 3, abs=1e-15) and p[0, 3] == 0.0
    _, p = f(logits, 4, 0.7, 0.2)            # one kept, renormalized to 1
    assert p[0, :4].tolist() == [1.0, 0.0, 0.0, 0.0]


def pin_two_way_closed_form(f):
    # k = 2: p0 = 1 / (1 + exp(-(a - b) / T)), the logistic function
    a, b, temp = 2.0, 0.5, 0.75
    logits = np.array([[b, a, -5.0]], dtype=np.float32)
    idx, p = f(logits, 2, temp, 1.0)
    assert idx[0, :2].tolist() == [1, 0]
    p0 = 1.0 / (1.0 + math.exp(-(a - b) / temp))
    assert p[0, 0] == pytest.approx(p0, rel=1e-15) and p[0, 1] == pytest.approx(1.0 - p0, rel=1e-14)


def pin_invariances(f):
    rng = np.random.default_rng(7)
    logits = rng.integers(-20, 20, size=(3, 200)).astype(np.float32)   # small integers: shifts are exact
    idx, p = f(logits, 32, 1.5, 0.9)
    idx2, p2 = f(logits + 64.0, 32, 1.5, 0.9)                           # shift by a constant
    assert np.array_equal(idx, idx2) and np.array_equal(p, p2)
    idx3, p3 = f(logits * 4.0, 32, 6.0, 0.9)                            # scale logits and T by 4
    assert np.array_equal(idx, idx3) and np.array_equal(p, p3)
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-15)
    assert np.all(np.diff(p[:, :32], axis=1) <= 0.0)                    # probabilities follow the ranking


def pin_brute_force_ranking(f):
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((4, 300)).astype(np.float32)
    logits[:, 10] = logits[:, 20]                                        # ties
    for k in (1, 7, 32):
        idx, _ = f(logits, k, 1.0, 1.0)
        for m in range(4):
            want = sorted(range(300), key=lambda i: (-float(logits[m, i]), i))[:k]
            assert idx[m, :k].tolist() == want


def pin_temperature_limit(f):
    # a very small temperature puts all mass on the largest logit
    logits = np.array([[0.0, 1.0, 0.9]], dtype=np.float32)
    idx, p = f(logits, 3, 1e-4, 1.0)                 # exp(-0.1 / 1e-4) underflows to 0
    assert idx[0, :3].tolist() == [1, 2, 0]
    assert p[0, 0] == 1.0 and p[0, 1] == 0.0 and p[0, 2] == 0.0


PINS = [pin_tie_order, pin_uniform_exact, pin_two_way_closed_form, pin_invariances, pin_brute_force_ranking,
        pin_temperature_limit]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(T.topk_probs)


# ------------------------------------------------------------ planted mistakes
def _mutant(order_key=None, cut_excludes_crossing=False, no_renorm=False, temp_multiplies=False):
    def f(logits, top_k, temperature, top_p):
        logits = np.asarray(logits, dtype=np.float32)
        M, N = logits.shape
        idx = np.full((M, 32), -1, dtype=np.int32)
        probs = np.zeros((M, 32))
        for m in range(M):
            row = logits[m].astype(np.float64)
            if order_key is None:
                order = np.lexsort((np.arange(N), -row))[:top_k]
            else:
                order = np.array(sorted(range(N), key=lambda i: order_key(row, i))[:top_k])
            idx[m, :top_k] = order
            l0 = row[order[0]]
            e = [math.exp((row[j] - l0) * temperature if temp_multiplies else (row[j] - l0) / temperature)
                 for j in order]
            p = [v / sum(e) for v in e]
            keep = top_k
            if top_p < 1.0:
                c = 0.0
                for n in range(top_k):
                    c += p[n]
                    if c >= top_p:
                        keep = n if (cut_excludes_crossing and n > 0) else n + 1
                        break
            s = 1.0 if no_renorm else sum(p[:keep])
            for n in range(keep):
                probs[m, n] = p[n] / s
        return idx, probs
    return f


MUTANTS = {
    "ties_higher_index_first": _mutant(order_key=lambda row, i: (-row[i], -i)),
    "ascending_logits": _mutant(order_key=lambda row, i: (row[i], i)),
    "cut_drops_crossing_entry": _mutant(cut_excludes_crossing=True),
    "no_renormalization": _mutant(no_renorm=True),
    "temperature_multiplies": _mutant(temp_multiplies=True),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    f = MUTANTS[name]
    caught = 0
    for pin in PINS:
        try:
            pin(f)
        except (AssertionError, ArithmeticError):
            caught += 1
    assert caught > 0, f"no pin catches the planted mistake {name}"


def test_unmutated_reference_copy_passes():
    # the mutant builder without a mistake must pass every pin (the mutants differ only by the mistake)
    for pin in PINS:
        pin(_mutant())
