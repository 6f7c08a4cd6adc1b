"""CPU oracle for the draft selector's edge scores -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module; the CUDA library never uses it.

What it computes ("Splash engine" analysis, section "The draft is a small model
with an unusual selector": the selector takes the top 16 candidates at each of
the 7 draft positions and scores every (predecessor, candidate) pair with a
trilinear form over a rank-256 embedding of the previous token, a rank-256
projection of the position's hidden state and a rank-256 embedding of the
candidate; the two codebooks are bf16, 248,320 x 256 each).  For every row r
(one draft position of one lane) and every pair (i, j) of its 16 predecessors
and 16 candidates:

    context[d]     = pred_cb[pred_ids[r, i], d] * hidden[r, d]
    score[r, i, j] = sum over d of context[d] * succ_cb[cand_ids[r, j], d]

Arithmetic: every bf16 widens exactly; a bf16 x fp32 product has at most 32
significant bits and times another bf16 at most 40, so each term is exact in
double, and the sum over d is rounded once (``math.fsum``, correctly rounded).
The result is the exact score to within half a double ulp.

Codebooks are passed as uint16 arrays of bf16 bit patterns [V, R]; hidden as
float32 [rows, R]; ids as integers [rows, 16].  Ids must lie in 0..V-1.
"""
from __future__ import annotations

import math

import numpy as np

PAIRS = 16      # predecessors and candidates per row


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly (a bf16 is the upper half of an IEEE fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def edge_scores(pred_cb, succ_cb, hidden, pred_ids, cand_ids) -> np.ndarray:
    pred_cb = np.asarray(pred_cb, dtype=np.uint16)
    succ_cb = np.asarray(succ_cb, dtype=np.uint16)
    hidden = np.asarray(hidden, dtype=np.float32)
    pred_ids = np.asarray(pred_ids, dtype=np.int64)
    cand_ids = np.asarray(cand_ids, dtype=np.int64)
    V, R = pred_cb.shape
    if succ_cb.shape != (V, R):
        raise ValueError("the two codebooks must have the same shape")
    rows = hidden.shape[0]
    if hidden.shape != (rows, R) or pred_ids.shape != (rows, PAIRS) or cand_ids.shape != (rows, PAIRS):
        raise ValueError("hidden [rows, R], pred_ids and cand_ids [rows, 16]")
    for ids in (pred_ids, cand_ids):
        if ids.size and (ids.min() < 0 or ids.max() >= V):
            raise ValueError("ids must lie in 0..V-1")
    out = np.zeros((rows, PAIRS, PAIRS), dtype=np.float64)
    for r in range(rows):
        h = hidden[r].astype(np.float64)
        for i in range(PAIRS):
            context = bf16_bits_to_f64(pred_cb[pred_ids[r, i]]) * h            # exact
            for j in range(PAIRS):
                terms = context * bf16_bits_to_f64(succ_cb[cand_ids[r, j]])    # exact
                out[r, i, j] = math.fsum(terms.tolist())
    return out


def abs_terms(pred_cb, succ_cb, hidden, pred_ids, cand_ids) -> np.ndarray:
    """sum over d of |context[d] * succ[d]| per score (the scale of the rounding error bound)."""
    pred_cb = np.asarray(pred_cb, dtype=np.uint16)
    succ_cb = np.asarray(succ_cb, dtype=np.uint16)
    out = np.zeros((hidden.shape[0], PAIRS, PAIRS), dtype=np.float64)
    for r in range(hidden.shape[0]):
        P = np.abs(bf16_bits_to_f64(pred_cb[np.asarray(pred_ids[r])]) * np.asarray(hidden[r], np.float64))
        S = np.abs(bf16_bits_to_f64(succ_cb[np.asarray(cand_ids[r])]))
        out[r] = P @ S.T
    return out
