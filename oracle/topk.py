"""CPU oracle for the LM-head sampling epilogue -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
import this module; the CUDA library never uses it.

What it computes ("Splash engine" analysis, section "Exact, up to top-32": the
target contributes 32 candidates per row, and their probabilities are
"temperature over its first top_k entries, truncated by top_p, renormalized";
MAX_TOP_K is 32 and top_k is mandatory, in [1, 32]), for each row of logits:

1. rank all N entries by logit, largest first; equal logits by lower index
   first (this project's reading: the page does not say how ties are ordered,
   and this order makes the result unique);
2. keep the first top_k of them;
3. p_j = exp((l_j - l_0) / T) / sum_{i < top_k} exp((l_i - l_0) / T) over those
   entries, in double, sums taken in rank order (l_0 is the largest logit, so
   every exponent is <= 0);
4. truncate by top_p: keep the shortest prefix whose cumulative probability
   reaches top_p (the entry that crosses top_p is kept; this project's reading
   of "truncated by top_p"); top_p >= 1 keeps all top_k entries;
5. renormalize the kept probabilities to sum to 1.

Output per row: ``idx[32]`` (int32; entries past top_k are -1) and
``probs[32]`` (float64; zero past the kept prefix).
"""
from __future__ import annotations

import math

import numpy as np

WIDTH = 32


def topk_probs(logits: np.ndarray, top_k: int, temperature: float, top_p: float):
    logits = np.asarray(logits, dtype=np.float32)
    if logits.ndim != 2:
        raise ValueError("logits must be [M, N]")
    M, N = logits.shape
    if not (1 <= top_k <= WIDTH) or top_k > N:
        raise ValueError("top_k must be in [1, 32] and at most N")
    if not (temperature > 0.0) or not (top_p > 0.0):
        raise ValueError("temperature and top_p must be positive")
    idx = np.full((M, WIDTH), -1, dtype=np.int32)
    probs = np.zeros((M, WIDTH), dtype=np.float64)
    for m in range(M):
        row = logits[m].astype(np.float64)
        # step 1-2: value descending, index ascending (lexsort sorts by the last key first)
        order = np.lexsort((np.arange(N), -row))[:top_k]
        idx[m, :top_k] = order
        # step 3: softmax at temperature T over the top_k entries, in rank order
        l0 = row[order[0]]
        e = [math.exp((row[j] - l0) / temperature) for j in order]
        total = 0.0
        for v in e:
            total += v
        p = [v / total for v in e]
        # step 4: shortest prefix reaching top_p
        keep = top_k
        if top_p < 1.0:
            c = 0.0
            for n in range(top_k):
                c += p[n]
                if c >= top_p:
                    keep = n + 1
                    break
        # step 5: renormalize the kept prefix
        kept = 0.0
        for n in range(keep):
            kept += p[n]
        for n in range(keep):
            probs[m, n] = p[n] / kept
    return idx, probs
