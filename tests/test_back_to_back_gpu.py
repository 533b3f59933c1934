"""Steps launched back to back on one stream, with no host synchronisation
between them, give the same bits as the same steps with the host waiting for
each one.  The bulk step kernel may start while the launch before it on the
stream finishes (programmatic stream serialisation) and must still read that
launch's results: the state a previous step of the same plan wrote, and the
update index a kernel advanced in device memory."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
from gpu_cases import HP, DeviceCase, ensure_built

pytestmark = pytest.mark.gpu

# Small plans (a few tiles per CTA, so no tile counter is zeroed between the
# launches and consecutive launches overlap) of several meshes; the generic
# kernel (N_d = 9) sits between bulk launches as an ordinary predecessor.
LAYERS = [
    ([(1024, 1024), (512, 1024), (1024,), (333, 129)], 4, "fsdp2", "f32", 1),
    ([(2048, 512), (77, 1000), (4097,)], 8, "distopt", "f32", 1),
    ([(512, 1024), (1536, 256), (5, 4099)], 9, "fsdp2", "f32", 1),
    ([(1024, 768), (999, 17)], 16, "fsdp2", "bf16", 1),
    ([(1024, 1024), (3, 4097)], 8, "hsdp", "f32", 2),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _cases(seed0):
    return [DeviceCase(shapes, n_d, mode, gdt, seed0 + i, n_rep)
            for i, (shapes, n_d, mode, gdt, n_rep) in enumerate(LAYERS)]


def _bits(case):
    return [b.bits() for b in case.state + case.params]


def _assert_same(a, b, what):
    for k, (x, y) in enumerate(zip(_bits(a), _bits(b))):
        assert np.array_equal(x, y), f"{what}: buffer {k} differs from the synchronised run"
    assert a.all_guards_intact() and b.all_guards_intact(), f"{what}: guard band overwritten"


def test_layer_stack_back_to_back():
    """Five plans stepped in turn, three updates each, as a model stepped layer
    by layer: every launch directly after another on the stream."""
    ref, run = _cases(500), _cases(500)
    for t in (1, 2, 3):
        for c in ref:
            c.step(t, debug=False)
            torch.cuda.synchronize()
    for t in (1, 2, 3):
        for c in run:
            c.step(t, debug=False)
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(ref, run)):
        _assert_same(a, b, f"layer {i}")
    assert fsp.device_error() == 0


def test_device_resident_index_advanced_between_launches():
    """The update index in device memory: step, advance kernel, step, ... with
    no host wait; each step must read the index the advance kernel wrote."""
    shapes, n_d, mode, gdt, n_rep = LAYERS[0]
    ref = DeviceCase(shapes, n_d, mode, gdt, 77, n_rep)
    run = DeviceCase(shapes, n_d, mode, gdt, 77, n_rep)
    for t in (1, 2, 3, 4):
        ref.step(t, debug=False)
        torch.cuda.synchronize()
    t_dev = torch.ones(1, dtype=torch.int64, device="cuda")
    for _ in range(4):
        fsp.sharded_step_device_t(run.plan, [g.t for g in run.grads], *[s.t for s in run.state],
                                  [q.t for q in run.params], HP, t_dev)
    torch.cuda.synchronize()
    assert int(t_dev.item()) == 5
    _assert_same(ref, run, "device-resident t")
    assert fsp.device_error() == 0


def test_zero3_steps_then_unshard_back_to_back():
    """ZeRO-3 steps (no all-gather) each followed at once by the unshard of
    the new master (both kernels may start while the launch before them
    finishes): every parameter copy must come from the master the step just
    wrote, as with the host waiting after each launch."""
    cases = []
    for _ in range(2):
        row = []
        for i, (shapes, n_d, mode, gdt, n_rep) in enumerate(LAYERS):
            row.append(DeviceCase(shapes, n_d, mode, gdt, 900 + i, n_rep))
        cases.append(row)
    ref, run = cases

    def zero3_then_unshard(c, t, sync):
        st = [s.t for s in c.state]
        fsp.sharded_step(c.plan, [g.t for g in c.grads], *st, None, HP, t)
        if sync:
            torch.cuda.synchronize()
        fsp.unshard(c.plan, st[0], [q.t for q in c.params])
        if sync:
            torch.cuda.synchronize()

    for t in (1, 2, 3):
        for c in ref:
            zero3_then_unshard(c, t, True)
        for c in run:
            zero3_then_unshard(c, t, False)
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(ref, run)):
        _assert_same(a, b, f"layer {i}")
    assert fsp.device_error() == 0


def test_layer_stack_replayed_from_one_graph():
    """The five plans' steps with the update index in device memory, captured
    once in one CUDA graph (consecutive launches joined by programmatic
    edges) and replayed: equal to the steps with host waits."""
    ref, run = _cases(700), _cases(700)
    for t in (1, 2, 3):
        for c in ref:
            c.step(t, debug=False)
            torch.cuda.synchronize()
    t_devs = [torch.ones(1, dtype=torch.int64, device="cuda") for _ in run]

    def step_all(stream):
        for c, t_dev in zip(run, t_devs):
            fsp.sharded_step_device_t(c.plan, [g.t for g in c.grads], *[s.t for s in c.state],
                                      [q.t for q in c.params], HP, t_dev, stream=stream)

    side = torch.cuda.Stream()
    step_all(side)          # t = 1, eager: every device table is uploaded outside the capture
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side, capture_error_mode="relaxed"):
        step_all(side)
    graph.replay()          # t = 2
    graph.replay()          # t = 3
    torch.cuda.synchronize()
    assert [int(t.item()) for t in t_devs] == [4] * len(run)
    for i, (a, b) in enumerate(zip(ref, run)):
        _assert_same(a, b, f"layer {i}")
    assert fsp.device_error() == 0
