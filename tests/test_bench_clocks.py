"""The bench's clock rule on the CPU: which clock records void a timed region,
and that such a region is measured exactly once more -- on every rank when any
rank's record is rejected (two gloo ranks)."""
import os
import socket
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _clocks(sm=2070.0, mx=2070.0, reasons=()):
    return {"sm_mhz": sm, "sm_max_mhz": mx, "reasons": list(reasons), "samples": 5}


def test_clock_rejection_rules():
    assert bench.clock_rejection(_clocks()) is None
    assert bench.clock_rejection(_clocks(sm=1800.0, reasons=["sw_power_cap"])) is None      # power cap: kept
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        why = bench.clock_rejection(_clocks(reasons=["sw_power_cap", r]))
        assert why is not None and r in why
    assert "no reason" in bench.clock_rejection(_clocks(sm=1200.0))                          # a clock lock
    assert bench.clock_rejection(_clocks(sm=1900.0)) is None                                 # within 15%
    assert bench.clock_rejection({"sm_mhz": None, "sm_max_mhz": None,
                                  "reasons": ["clock sampling unavailable"]}) is None


class _FakeSampler:
    """Returns queued clock records, one per timed region."""
    queue = []

    def __init__(self, gpu_id):
        pass

    def stop(self):
        return dict(_FakeSampler.queue.pop(0))


def _region(records, world=1, dev=None):
    _FakeSampler.queue = list(records)
    calls = []

    def run():
        calls.append(len(calls))
        return f"measurement {len(calls)}"

    result, clocks = bench.timed_region(run, None, world, dev, lambda: None, lambda: None,
                                        sampler_cls=_FakeSampler, settle=0.0)
    return calls, result, clocks


def test_clean_region_runs_once():
    calls, result, clocks = _region([_clocks()])
    assert calls == [0] and result == "measurement 1"
    assert clocks["remeasured"] is False and "rejected" not in clocks


def test_rejected_region_is_measured_once_more():
    calls, result, clocks = _region([_clocks(reasons=["hw_thermal_slowdown"]), _clocks()])
    assert calls == [0, 1] and result == "measurement 2"
    assert clocks["remeasured"] is True and "hw_thermal_slowdown" in clocks["first_rejected"]
    assert "rejected" not in clocks and clocks["reasons"] == []


def test_rejected_twice_is_reported_not_retried_again():
    calls, result, clocks = _region([_clocks(sm=900.0), _clocks(sm=905.0), _clocks()])
    assert calls == [0, 1] and result == "measurement 2"
    assert clocks["remeasured"] is True and "no reason" in clocks["rejected"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench as b
        # only rank 1 sees a slowdown in the first region; both ranks must measure again
        first = _clocks(reasons=["sw_thermal_slowdown"]) if rank == 1 else _clocks()
        _FakeSampler.queue = [first, _clocks(), _clocks()]
        n = []
        _, clocks = b.timed_region(lambda: n.append(1), None, world, None, lambda: None, lambda: None,
                                   sampler_cls=_FakeSampler, settle=0.0)
        out.put((rank, len(n), clocks["remeasured"], clocks.get("first_rejected")))
    finally:
        dist.destroy_process_group()


def test_any_rank_rejected_remeasures_every_rank_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2, 2]
    assert all(r[2] for r in res)
    assert res[0][3] == "rejected on another rank" and "sw_thermal_slowdown" in res[1][3]
