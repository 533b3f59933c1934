"""The step under CUDA-graph capture, on concurrent streams and host threads,
and the bounded waits' failure path (a wait that nothing completes)."""
import threading
import time

import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
from synth_inputs import workload

from gpu_cases import HP, DeviceCase, OracleCase, compare, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _bits(case):
    return [x.bits() for x in case.state + case.params]


def _step_args(case):
    return ([g.t for g in case.grads], [s.t for s in case.state], [p.t for p in case.params])


def test_bounded_wait_gives_up_and_reports():
    t0 = time.perf_counter()
    bits = fsp.selftest_bounded_wait(200)
    dt = time.perf_counter() - t0
    assert bits == 4
    assert 0.15 < dt < 10.0
    assert fsp.device_error() == 0            # read-and-clear
    # the device is still usable: a normal step afterwards completes cleanly
    w = workload(0)
    c = DeviceCase(w.shapes, w.n_d, w.mode, w.grad_dtype, w.data_seed)
    c.step(w.step, debug=False)
    torch.cuda.synchronize()
    assert fsp.device_error() == 0


@pytest.mark.parametrize("mode,n_d,n_rep", [("fsdp2", 4, 1), ("hsdp", 8, 2), ("fsdp2", 9, 1)])
def test_cuda_graph_replay_equals_eager(mode, n_d, n_rep):
    shapes = [(3001, 7), (12289,), (9, 5), (1,)]
    eager = DeviceCase(shapes, n_d, mode, "f32", 21, n_rep)
    graphed = DeviceCase(shapes, n_d, mode, "f32", 21, n_rep)
    fresh = DeviceCase(shapes, n_d, mode, "f32", 21, n_rep)
    # first call outside capture (uploads the tile table), then restore inputs
    graphed.step(1, debug=False)
    torch.cuda.synchronize()
    for dst, src in zip(graphed.state + graphed.params, fresh.state + fresh.params):
        dst.raw.copy_(src.raw)
    grads, state, params = _step_args(graphed)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        for t in (10, 11):
            fsp.sharded_step(graphed.plan, grads, *state, params, HP, t, stream=stream)
    g.replay()
    for t in (10, 11):
        eager.step(t, debug=False)
    torch.cuda.synchronize()
    for a, b in zip(_bits(eager), _bits(graphed)):
        assert np.array_equal(a, b)
    assert fsp.device_error() == 0


def test_two_plans_on_concurrent_streams():
    w0 = workload(0)
    cases = [DeviceCase(w0.shapes, w0.n_d, w0.mode, "f32", 31 + i) for i in range(2)]
    refs = [DeviceCase(w0.shapes, w0.n_d, w0.mode, "f32", 31 + i) for i in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for t in (10, 11, 12):
        for c, s in zip(cases, streams):
            grads, state, params = _step_args(c)
            fsp.sharded_step(c.plan, grads, *state, params, HP, t, stream=s)
    torch.cuda.synchronize()
    for r in refs:
        for t in (10, 11, 12):
            r.step(t, debug=False)
    torch.cuda.synchronize()
    for c, r in zip(cases, refs):
        for a, b in zip(_bits(c), _bits(r)):
            assert np.array_equal(a, b)


def test_first_use_of_a_plan_from_several_host_threads():
    shapes = [(4097, 3), (77,)]
    cases = [DeviceCase(shapes, 4, "fsdp2", "f32", 41) for _ in range(4)]
    plan = fsp.plan_layout(shapes, 4)          # fresh plan: no tile table on the device yet
    errors = []
    barrier = threading.Barrier(4)

    def run(c):
        try:
            s = torch.cuda.Stream()
            barrier.wait()
            grads, state, params = _step_args(c)
            fsp.sharded_step(plan, grads, *state, params, HP, 10, stream=s)
            s.synchronize()
        except Exception as e:   # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(c,)) for c in cases]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors
    first = _bits(cases[0])
    for c in cases[1:]:
        for a, b in zip(first, _bits(c)):
            assert np.array_equal(a, b)
    assert fsp.device_error() == 0


# --- tiles handed out in order from a per-launch counter (plans with many tiles per CTA) ---

BIG = ((3000, 4096), (4099,), (77, 3))   # ~12.3M elements: at least 16 tiles per CTA on 152 SMs


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


@pytest.mark.parametrize("n_d,mode,n_rep,gd", [(4, "fsdp2", 1, "f32"), (8, "hsdp", 2, "f32"), (6, "fsdp2", 1, "bf16")])
def test_ordered_tiles_match_the_oracle(n_d, mode, n_rep, gd):
    """A tile skipped or taken twice by the counter schedule shows up here: a
    sentinel left in place, or state updated twice."""
    dev = DeviceCase(BIG, n_d, mode, gd, 51, n_rep)
    assert dev.plan.n_tiles >= 16 * _sms()      # large enough for the counter schedule
    ora = OracleCase(BIG, n_d, mode, gd, 51, n_rep)
    dev.step(10)
    ora.step(10)
    torch.cuda.synchronize()
    compare(dev, ora)


def test_noalloc_counter_schedule_equals_the_step():
    ref = DeviceCase(BIG, 4, "fsdp2", "f32", 52)
    new = DeviceCase(BIG, 4, "fsdp2", "f32", 52)
    assert ref.plan.n_tiles >= 16 * _sms()
    stream = torch.cuda.current_stream()
    for t in (10, 11):
        ref.step(t, debug=False)
        grads, state, params = _step_args(new)
        fsp.sharded_step_noalloc(new.plan, grads, *state, params, HP, t, stream=stream)
    torch.cuda.synchronize()
    for a, b in zip(_bits(ref), _bits(new)):
        assert np.array_equal(a, b)
    assert new.all_guards_intact()
    assert fsp.device_error() == 0


@pytest.mark.parametrize("mode", ["relaxed", "global"])
def test_cuda_graph_of_ordered_steps(mode):
    eager = DeviceCase(BIG, 4, "fsdp2", "f32", 53)
    graphed = DeviceCase(BIG, 4, "fsdp2", "f32", 53)
    fresh = DeviceCase(BIG, 4, "fsdp2", "f32", 53)
    assert graphed.plan.n_tiles >= 16 * _sms()
    graphed.step(1, debug=False)      # first use outside capture (tile table, counter pool)
    torch.cuda.synchronize()
    for dst, src in zip(graphed.state + graphed.params, fresh.state + fresh.params):
        dst.raw.copy_(src.raw)
    del fresh
    grads, state, params = _step_args(graphed)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode=mode):
        for t in (10, 11):
            fsp.sharded_step(graphed.plan, grads, *state, params, HP, t, stream=stream)
    for _ in range(2):                # each replay zeroes its counters again
        g.replay()
        for t in (10, 11):
            eager.step(t, debug=False)
        torch.cuda.synchronize()
        for a, b in zip(_bits(eager), _bits(graphed)):
            assert np.array_equal(a, b)
    assert graphed.all_guards_intact()
    assert fsp.device_error() == 0


def test_one_plan_on_concurrent_streams_with_ordered_tiles():
    cases = [DeviceCase(BIG, 4, "fsdp2", "f32", 61 + i) for i in range(2)]
    refs = [DeviceCase(BIG, 4, "fsdp2", "f32", 61 + i) for i in range(2)]
    plan = cases[0].plan                       # one plan, two sets of buffers, in flight together
    streams = [torch.cuda.Stream() for _ in range(2)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for t in (10, 11, 12):
        for c, s in zip(cases, streams):
            grads, state, params = _step_args(c)
            fsp.sharded_step(plan, grads, *state, params, HP, t, stream=s)
    torch.cuda.synchronize()
    for r in refs:
        for t in (10, 11, 12):
            r.step(t, debug=False)
    torch.cuda.synchronize()
    for c, r in zip(cases, refs):
        for a, b in zip(_bits(c), _bits(r)):
            assert np.array_equal(a, b)
    assert fsp.device_error() == 0
