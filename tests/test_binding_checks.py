"""The Python binding checks every tensor before its pointer reaches the
library, which cannot see sizes: a wrong dtype, shape, rank or layout, or a
tensor off the GPU, raises ValueError naming the argument, and no compute call
is made.  Runs without a GPU (host tensors stop at the device check)."""
import pytest
import torch

import bit_row_speculative_gb300 as q4

N, K, M = 256, 512, 4
HOST_ONLY = ("q4_packed_bytes", "q4_decode_step_workspace_bytes")


class _HostOnly:
    """The real library for size queries; any compute entry point fails the test."""

    def __init__(self, real):
        self._real = real

    def __getattr__(self, name):
        if name not in HOST_ONLY:
            raise AssertionError(f"{name} was called with unchecked arguments")
        return getattr(self._real, name)


@pytest.fixture(autouse=True)
def _no_compute_calls(monkeypatch):
    real = q4.lib()
    monkeypatch.setattr(q4, "lib", lambda: _HostOnly(real))


def _x(m=M, k=K, dtype=torch.bfloat16):
    return torch.zeros((m, k), dtype=dtype)


def _W(n=N, k=K):
    return torch.zeros(n * k // 16 * 9, dtype=torch.uint8)


def _raises(fn, *words):
    with pytest.raises(ValueError) as ei:
        fn()
    for w in words:
        assert w in str(ei.value), str(ei.value)


def test_matmul_checks():
    _raises(lambda: q4.matmul(_x(dtype=torch.float16), _W(), N, K), "x", "bfloat16")
    _raises(lambda: q4.matmul(_x()[0], _W(), N, K), "x", "2-D")
    _raises(lambda: q4.matmul(_x(k=2 * K)[:, ::2], _W(), N, K), "x", "contiguous")
    _raises(lambda: q4.matmul(_x(k=448), _W(), N, K), "columns")
    _raises(lambda: q4.matmul(_x(), _W()[:-1], N, K), "W", "bytes")
    _raises(lambda: q4.matmul(_x(), _W().view(torch.int8), N, K), "W", "uint8")
    _raises(lambda: q4.matmul(_x(), _W(), N, K, y=torch.zeros((M, N - 1))), "y", "shape")
    _raises(lambda: q4.matmul(_x(), _W(), N, K, y=torch.zeros((M, N), dtype=torch.float64)), "y", "float32")
    _raises(lambda: q4.matmul(_x(), _W(), N, K, y=torch.zeros((M, N))), "CUDA device")
    _raises(lambda: q4.matmul_noalloc(_x(), _W(), N, K, torch.zeros((M + 1, N))), "y", "shape")
    _raises(lambda: q4.matmul_noalloc(_x(), _W(), N, K, torch.zeros((M, N))), "CUDA device")


def test_glue_checks():
    _raises(lambda: q4.glue(torch.zeros((M, N), dtype=torch.bfloat16), K, q4.GLUE_RMSNORM), "y", "float32")
    _raises(lambda: q4.glue(torch.zeros((M, N)), K, q4.GLUE_RMSNORM, x_next=_x(k=K + 64)), "x_next", "shape")
    _raises(lambda: q4.glue(torch.zeros((M, N)), K, q4.GLUE_RMSNORM), "CUDA device")


def test_decode_step_checks():
    layers = [(_W(1024, 512), 1024, 512, q4.GLUE_RMSNORM), (_W(256, 1024), 256, 1024, q4.GLUE_NONE)]
    x0 = _x(k=512)
    _raises(lambda: q4.decode_step([], x0), "empty")
    _raises(lambda: q4.decode_step([(_W(1024, 512)[:-16], 1024, 512, 1)] + layers[1:], x0), "layers[0].W", "bytes")
    _raises(lambda: q4.decode_step(layers, _x(k=1024)), "x0", "first layer")
    _raises(lambda: q4.decode_step(layers, x0, y_last=torch.zeros((M, 255))), "y_last", "shape")
    _raises(lambda: q4.decode_step(layers, x0, workspace=torch.zeros(64, dtype=torch.float32)), "workspace", "uint8")
    _raises(lambda: q4.decode_step(layers, x0), "CUDA device")


def test_topk_checks():
    logits = torch.zeros((M, 1000))
    _raises(lambda: q4.topk_probs(logits.to(torch.bfloat16), 8, 1.0, 1.0), "logits", "float32")
    _raises(lambda: q4.topk_probs(logits[0], 8, 1.0, 1.0), "logits", "2-D")
    _raises(lambda: q4.topk_probs(logits, 8, 1.0, 1.0, idx=torch.zeros((M, 32), dtype=torch.int64)), "idx", "int32")
    _raises(lambda: q4.topk_probs(logits, 8, 1.0, 1.0, probs=torch.zeros((M, 16))), "probs", "shape")
    _raises(lambda: q4.topk_probs(logits, 8, 1.0, 1.0), "CUDA device")
    _raises(lambda: q4.lm_head_topk(_x(k=448), _W(), N, K, 8, 1.0, 1.0), "columns")
    _raises(lambda: q4.lm_head_topk(_x(), _W(N + 1, K), N, K, 8, 1.0, 1.0), "W", "bytes")
    _raises(lambda: q4.lm_head_topk(_x(), _W(), N, K, 8, 1.0, 1.0), "CUDA device")


def test_edges_checks():
    V, R, rows = 50, 64, 3
    P = torch.zeros((V, R), dtype=torch.bfloat16)
    h = torch.zeros((rows, R))
    ids = torch.zeros((rows, 16), dtype=torch.int32)
    _raises(lambda: q4.draft_select_edges(P.float(), P, h, ids, ids), "pred_cb", "bfloat16")
    _raises(lambda: q4.draft_select_edges(P, P[:-1], h, ids, ids), "succ_cb", "shape")
    _raises(lambda: q4.draft_select_edges(P, P, torch.zeros((rows, R + 8)), ids, ids), "rank")
    _raises(lambda: q4.draft_select_edges(P, P, h, ids.long(), ids), "pred_ids", "int32")
    _raises(lambda: q4.draft_select_edges(P, P, h, ids, ids[:, :8].contiguous()), "cand_ids", "shape")
    _raises(lambda: q4.draft_select_edges(P, P, h, ids, ids, score=torch.zeros((rows, 256))), "score", "shape")
    _raises(lambda: q4.draft_select_edges(P, P, h, ids, ids), "CUDA device")
