"""q4_draft_select_edges on the GPU against the oracle (oracle/edges.py).

Tolerance, from the kernel's arithmetic: each context value pred * hidden is
rounded once to fp32 (relative error <= u = 2^-24), each of the four
accumulators adds R/4 exact products with one rounding per fused multiply-add,
and two more additions combine them; so |score - exact| <= (R/4 + 2) u * S + O(u^2)
with S = sum over d of |term|.  The tests allow (R/4 + 3) u * S.

Cases: the full-size workload (two 248,320 x 256 codebooks, 4 lanes x 7
positions, predecessors chained from the previous position's candidates), small
vocabularies and every rank shape (R = 8 .. 256), ids 0 and V - 1 and repeated
ids, one-hot rows with exact scores, rows independent of the other rows and
deterministic, and out-of-range ids reported through the device status."""
import numpy as np
import pytest
import torch

import bit_row_speculative_gb300 as q4
import synth_inputs as si
from oracle import edges as E

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _bits(cb: torch.Tensor) -> np.ndarray:
    return cb.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _run(P, S, hidden, pred, cand):
    out = q4.draft_select_edges(P.cuda(), S.cuda(), hidden.cuda(), pred.cuda(), cand.cuda())
    q4.device_status()
    return out.cpu().numpy().astype(np.float64)


def _check(P, S, hidden, pred, cand, got=None):
    if got is None:
        got = _run(P, S, hidden, pred, cand)
    Pb, Sb = _bits(P), _bits(S)
    want = E.edge_scores(Pb, Sb, hidden.numpy(), pred.numpy(), cand.numpy())
    bound = E.abs_terms(Pb, Sb, hidden.numpy(), pred.numpy(), cand.numpy()) * (P.shape[1] / 4 + 3) * U
    err = np.abs(got - want)
    assert np.all(err <= bound), f"max excess {np.max(err - bound)}"
    return got


@pytest.fixture(scope="module")
def full_codebooks():
    V, R = si.VOCAB, si.EDGE_RANK
    return si.make_codebook(V, R, 6001), si.make_codebook(V, R, 6002)


def test_full_size_workload(full_codebooks):
    P, S = full_codebooks
    hidden, pred, cand = si.make_edge_inputs(4, si.VOCAB, si.EDGE_RANK, 6999)
    got = _check(P, S, hidden, pred, cand)
    # position 0 of each lane: every predecessor is the anchor, so the 16 rows of its scores agree
    for lane in range(4):
        r = lane * si.EDGE_POSITIONS
        assert np.all(got[r] == got[r][0:1])


@pytest.mark.parametrize("V,R,rows", [(37, 8, 1), (37, 64, 3), (1000, 200, 29), (5, 256, 2), (300, 128, 64)])
def test_small_shapes(V, R, rows):
    P, S = si.make_codebook(V, R, 11 + R), si.make_codebook(V, R, 12 + R)
    g = torch.Generator().manual_seed(V + R + rows)
    hidden = torch.randn((rows, R), generator=g)
    pred = torch.randint(0, V, (rows, 16), generator=g, dtype=torch.int32)
    cand = torch.randint(0, V, (rows, 16), generator=g, dtype=torch.int32)
    pred[0, 0], pred[0, 1], cand[0, 0], cand[0, 15] = 0, V - 1, V - 1, 0      # both ends of the codebook
    cand[-1, :] = cand[-1, 0]                                                    # repeated ids
    _check(P, S, hidden, pred, cand)


def test_one_hot_exact():
    V, R = 8, 256
    P = torch.zeros((V, R))
    S = torch.zeros((V, R))
    for t in range(V):
        P[t, (37 * t) % R] = 1.0 + t
        S[t, (37 * t) % R] = 0.5
    hidden = torch.arange(R, dtype=torch.float32)[None, :].repeat(2, 1)
    pred = torch.arange(16, dtype=torch.int32)[None, :].remainder(V).repeat(2, 1)
    cand = torch.tensor([[t % V for t in range(16)], [(t + 3) % V for t in range(16)]], dtype=torch.int32)
    got = _run(P.to(torch.bfloat16), S.to(torch.bfloat16), hidden, pred, cand)
    for r in range(2):
        for i in range(16):
            for j in range(16):
                a, b = int(pred[r, i]), int(cand[r, j])
                want = (1.0 + a) * float((37 * a) % R) * 0.5 if a == b else 0.0
                assert got[r, i, j] == want


def test_rows_independent_and_deterministic(full_codebooks):
    P, S = full_codebooks
    hidden, pred, cand = si.make_edge_inputs(2, si.VOCAB, si.EDGE_RANK, 6998)
    Pd, Sd = P.cuda(), S.cuda()
    all_rows = q4.draft_select_edges(Pd, Sd, hidden.cuda(), pred.cuda(), cand.cuda())
    again = q4.draft_select_edges(Pd, Sd, hidden.cuda(), pred.cuda(), cand.cuda())
    assert torch.equal(all_rows, again)
    for r in (0, 5, 13):
        one = q4.draft_select_edges(Pd, Sd, hidden[r:r + 1].contiguous().cuda(), pred[r:r + 1].contiguous().cuda(),
                                    cand[r:r + 1].contiguous().cuda())
        assert torch.equal(one[0], all_rows[r])
    q4.device_status()


def test_out_of_range_id_is_reported():
    V, R = 50, 64
    P, S = si.make_codebook(V, R, 21), si.make_codebook(V, R, 22)
    g = torch.Generator().manual_seed(5)
    hidden = torch.randn((2, R), generator=g)
    pred = torch.randint(0, V, (2, 16), generator=g, dtype=torch.int32)
    cand = torch.randint(0, V, (2, 16), generator=g, dtype=torch.int32)
    bad_pred, bad_cand = pred.clone(), cand.clone()
    bad_pred[1, 4] = V            # one past the end: not read
    bad_cand[0, 9] = -3
    out = q4.draft_select_edges(P.cuda(), S.cuda(), hidden.cuda(), bad_pred.cuda(), bad_cand.cuda())
    with pytest.raises(q4.Q4Error) as ei:
        q4.device_status()
    assert ei.value.status == q4.Q4_ERR_INVALID_INDEX
    got = out.cpu().numpy()
    assert np.all(got[1, 4, :] == 0.0) and np.all(got[0, :, 9] == 0.0)
    # the other scores are the valid ones
    ok = _run(P, S, hidden, pred, cand)
    mask = np.ones_like(got, dtype=bool)
    mask[1, 4, :] = False
    mask[0, :, 9] = False
    assert np.array_equal(got[mask], ok[mask].astype(np.float32))
    q4.device_status()            # the record was cleared
