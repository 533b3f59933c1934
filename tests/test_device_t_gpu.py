"""The step with its update index in device memory: eager, advanced on the
device, and captured once in a CUDA graph and replayed."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp

from gpu_cases import HP, DeviceCase, ensure_built

pytestmark = pytest.mark.gpu

SHAPES = [(3001, 7), (12289,), (9, 5), (1,)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _bufs(c):
    return [g.t for g in c.grads], [s.t for s in c.state], [p.t for p in c.params]


def _same(a, b):
    for x, y in zip(a.state + a.params, b.state + b.params):
        assert np.array_equal(x.bits(), y.bits())


@pytest.mark.parametrize("mode,n_d,n_rep,dtype", [("fsdp2", 8, 1, "f32"), ("distopt", 4, 1, "bf16"),
                                                  ("hsdp", 8, 2, "f32"), ("fsdp2", 9, 1, "f32")])
def test_device_t_eager_equals_host_t(mode, n_d, n_rep, dtype):
    ref = DeviceCase(SHAPES, n_d, mode, dtype, 61, n_rep)
    dev = DeviceCase(SHAPES, n_d, mode, dtype, 61, n_rep)
    t = torch.tensor([10], dtype=torch.int64, device="cuda")
    g, s, p = _bufs(dev)
    for step in (10, 11):
        ref.step(step, debug=False)
        fsp.sharded_step_device_t(dev.plan, g, *s, p, HP, t, advance=True)
        torch.cuda.synchronize()
        _same(ref, dev)
    assert int(t.item()) == 12
    assert fsp.device_error() == 0


BIG = [(3000, 4096), (4099,), (77, 3)]   # enough tiles per CTA for the in-order (counter) schedule


@pytest.mark.parametrize("shapes", [SHAPES, BIG], ids=["small", "large"])
def test_graph_of_one_step_replayed(shapes):
    ref = DeviceCase(shapes, 8, "fsdp2", "f32", 62)
    dev = DeviceCase(shapes, 8, "fsdp2", "f32", 62)
    fresh = DeviceCase(shapes, 8, "fsdp2", "f32", 62)
    t = torch.tensor([1], dtype=torch.int64, device="cuda")
    g, s, p = _bufs(dev)
    fsp.sharded_step_device_t(dev.plan, g, *s, p, HP, t, advance=False)   # first call outside capture
    torch.cuda.synchronize()
    for dst, src in zip(dev.state + dev.params, fresh.state + fresh.params):
        dst.raw.copy_(src.raw)
    t.fill_(10)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        fsp.sharded_step_device_t(dev.plan, g, *s, p, HP, t, advance=True, stream=stream)
    for step in (10, 11, 12):
        graph.replay()
        ref.step(step, debug=False)
    torch.cuda.synchronize()
    _same(ref, dev)
    assert int(t.item()) == 13
    assert fsp.device_error() == 0


def test_index_below_one_is_reported_and_treated_as_one():
    ref = DeviceCase(SHAPES, 4, "fsdp2", "f32", 63)
    dev = DeviceCase(SHAPES, 4, "fsdp2", "f32", 63)
    t = torch.tensor([0], dtype=torch.int64, device="cuda")
    g, s, p = _bufs(dev)
    fsp.device_error()
    fsp.sharded_step_device_t(dev.plan, g, *s, p, HP, t, advance=False)
    ref.step(1, debug=False)
    torch.cuda.synchronize()
    assert fsp.device_error() == 8
    _same(ref, dev)
