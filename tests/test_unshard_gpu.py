"""GPU parity of the FSDP2 unshard (fp32 shards -> bf16 -> every rank's full buffer)."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
from oracle import step as OS
from synth_inputs import workload

from gpu_cases import HP, PARAM_SENTINEL, DeviceCase, Guarded, OracleCase, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


CASES = [("fsdp2", 4, 1), ("fsdp2", 1, 1), ("fsdp2", 6, 1), ("fsdp2", 16, 1), ("fsdp2", 33, 1), ("distopt", 8, 1),
         ("distopt", 6, 1), ("hsdp", 8, 2), ("hsdp", 6, 3)]
SHAPES = [(3001, 7), (12289,), (9, 5), (1,), (5, 4099), (2, 3, 5)]


@pytest.mark.parametrize("mode,n_d,n_rep", CASES)
def test_unshard_matches_oracle(mode, n_d, n_rep):
    dev = DeviceCase(SHAPES, n_d, mode, "f32", 17, n_rep)
    ora = OracleCase(SHAPES, n_d, mode, "f32", 17, n_rep)
    fsp.unshard(dev.plan, dev.state[0].t, [p.t for p in dev.params])
    OS.unshard(ora.plan, ora.state[0], ora.params)
    torch.cuda.synchronize()
    for q in range(n_d):
        assert np.array_equal(dev.params[q].bits(), ora.params[q]), f"rank {q}"
    n = dev.plan.valid_elems
    assert all(np.all(p.bits()[n:] == PARAM_SENTINEL) for p in dev.params)
    assert dev.all_guards_intact()


@pytest.mark.parametrize("mode,n_d,n_rep", [("fsdp2", 8, 1), ("distopt", 8, 1), ("hsdp", 8, 2), ("fsdp2", 9, 1)])
def test_unshard_after_step_reproduces_its_params(mode, n_d, n_rep):
    dev = DeviceCase(SHAPES, n_d, mode, "f32", 18, n_rep)
    dev.step(10, debug=False)
    fresh = [Guarded(dev.plan.full_len_padded, torch.bfloat16, PARAM_SENTINEL) for _ in range(n_d)]
    fsp.unshard(dev.plan, dev.state[0].t, [p.t for p in fresh])
    torch.cuda.synchronize()
    for a, b in zip(dev.params, fresh):
        assert np.array_equal(a.bits(), b.bits())
        assert b.guards_intact()


def test_unshard_full_size_qwen3():
    w = workload(1)
    dev = DeviceCase(w.shapes, w.n_d, w.mode, "f32", w.data_seed)
    try:
        fsp.unshard(dev.plan, dev.state[0].t, [p.t for p in dev.params])
        torch.cuda.synchronize()
        p0 = dev.params[0].t.view(torch.int16)
        for q in range(1, w.n_d):
            assert torch.equal(dev.params[q].t.view(torch.int16), p0)
        master = dev.state[0].t
        for sg in dev.plan.segments:
            if sg.length:
                a, c = sg.full_off, sg.state_off
                assert torch.equal(p0[a:a + sg.length], master[c:c + sg.length].to(torch.bfloat16).view(torch.int16))
    finally:
        del dev
        torch.cuda.empty_cache()


@pytest.mark.parametrize("mode,n_d,n_rep", [("fsdp2", 8, 1), ("distopt", 6, 1), ("hsdp", 8, 2), ("fsdp2", 9, 1)])
def test_zero3_step_then_unshard_equals_the_gathering_step(mode, n_d, n_rep):
    """The step without all-gather leaves every param buffer alone and updates
    the state exactly like the full step; unsharding afterwards gives the full
    step's params."""
    full = DeviceCase(SHAPES, n_d, mode, "f32", 19, n_rep)
    z3 = DeviceCase(SHAPES, n_d, mode, "f32", 19, n_rep)
    before = [p.bits().copy() for p in z3.params]
    for t in (10, 11):
        full.step(t, debug=False)
        fsp.sharded_step(z3.plan, [g.t for g in z3.grads], *[s.t for s in z3.state], None, HP, t)
    torch.cuda.synchronize()
    for a, b in zip(full.state, z3.state):
        assert np.array_equal(a.bits(), b.bits())
    for p, b in zip(z3.params, before):
        assert np.array_equal(p.bits(), b)
    fsp.unshard(z3.plan, z3.state[0].t, [p.t for p in z3.params])
    torch.cuda.synchronize()
    for a, b in zip(full.params, z3.params):
        assert np.array_equal(a.bits(), b.bits())
    assert fsp.device_error() == 0


@pytest.mark.parametrize("mode,n_d,n_rep", CASES)
def test_shard_matches_oracle(mode, n_d, n_rep):
    """fsp_shard (full fp32 parameters -> every replica's master slots; m, v
    zeroed) against the oracle's shard, slot for slot."""
    from oracle import plan as OP
    from gpu_cases import STATE_SENTINEL
    shapes = SHAPES
    dev = DeviceCase(shapes, n_d, mode, "f32", 19, n_rep)
    oplan = OP.plan_layout(shapes, n_d, mode, n_rep=n_rep)
    rng = np.random.default_rng(n_d * 7 + n_rep)
    full_h = rng.standard_normal(dev.plan.full_len_padded).astype(np.float32)
    full = Guarded(dev.plan.full_len_padded, torch.float32, 0)
    full.t.copy_(torch.from_numpy(full_h))
    for s in dev.state:
        s.raw[s.g:s.g + s.n].view(torch.int32).fill_(int(np.array([STATE_SENTINEL], np.uint32).view(np.int32)[0]))
    fsp.shard(dev.plan, full.t, dev.state[0].t, dev.state[1].t, dev.state[2].t)
    want = np.full(oplan.state_len_total, STATE_SENTINEL, np.uint32).view(np.float32)
    OS.shard(oplan, full_h, want)
    torch.cuda.synchronize()
    assert np.array_equal(dev.state[0].bits(), want.view(np.uint32))
    for s in dev.state[1:]:
        assert not s.bits().any()                    # the Adam moments start at zero
    assert dev.all_guards_intact() and full.guards_intact()
    assert fsp.device_error() == 0
