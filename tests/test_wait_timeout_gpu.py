"""Timeout reporting on the GPU without a fault: a bounded wait that nothing
satisfies runs out, the kernel records it and exits, q4_device_status reports
Q4_ERR_TIMEOUT once, and the context keeps working."""
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


def test_wait_that_runs_out_is_reported_once_and_context_survives():
    N, K, M = 640, 1024, 4
    W = si.make_weights(N, K, 31, device="cuda")
    x = si.make_x(M, K, 32, device="cuda")
    before = q4.matmul(x, W, N, K).cpu()
    q4.device_status()                                   # clean start
    q4.check_wait_timeout(200_000)                       # ~0.1 ms of SM clock
    with pytest.raises(q4.Q4Error) as ei:
        q4.device_status()
    assert ei.value.status == q4.Q4_ERR_TIMEOUT
    q4.device_status()                                   # the record was cleared
    after = q4.matmul(x, W, N, K).cpu()                  # the context still computes
    q4.device_status()
    assert torch.equal(before, after)


def test_wait_check_on_a_side_stream():
    s = torch.cuda.Stream()
    q4.check_wait_timeout(50_000, stream=s)
    with pytest.raises(q4.Q4Error) as ei:
        q4.device_status(stream=s)
    assert ei.value.status == q4.Q4_ERR_TIMEOUT
    q4.device_status(stream=s)
