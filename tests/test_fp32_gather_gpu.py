"""The step whose all-gather writes the fp32 master itself (a
MixedPrecisionPolicy that keeps parameters in fp32), and the fp32 unshard:
state equal to the bf16 step's, every rank's fp32 copy equal to the owner's
new master bit for bit, padding untouched."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp

from gpu_cases import HP, STATE_SENTINEL, DeviceCase, Guarded, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


SMALL = ((3001, 7), (77, 3), (4099,), (1,), (12289,), (9, 5), (0, 4))
BIG = ((3000, 4096), (4099,), (77, 3))


def _expected_copies(plan, master_bits, n_d):
    """Every rank's fp32 buffer: the owner's master at its full indices (the
    rank's own replica group for HSDP), the sentinel elsewhere."""
    want = [np.full(plan.full_len_padded, STATE_SENTINEL, np.uint32) for _ in range(n_d)]
    group = plan.n_shard
    for s in plan.segments:
        if not s.length:
            continue
        first = (s.rank // group) * group
        for q in range(first, first + group):
            want[q][s.full_off:s.full_off + s.length] = master_bits[s.state_off:s.state_off + s.length]
    return want


@pytest.mark.parametrize("shapes,n_d,mode,n_rep,gd", [
    (SMALL, 4, "fsdp2", 1, "f32"), (SMALL, 6, "fsdp2", 1, "bf16"), (SMALL, 3, "distopt", 1, "f32"),
    (SMALL, 8, "hsdp", 2, "f32"), (SMALL, 9, "fsdp2", 1, "f32"), (BIG, 4, "fsdp2", 1, "f32"),
])
def test_fp32_gather_step_and_unshard(shapes, n_d, mode, n_rep, gd):
    ref = DeviceCase(shapes, n_d, mode, gd, 103, n_rep)
    f32 = DeviceCase(shapes, n_d, mode, gd, 103, n_rep)
    z3 = DeviceCase(shapes, n_d, mode, gd, 103, n_rep)
    plan = f32.plan
    bufs = [Guarded(plan.full_len_padded, torch.float32, STATE_SENTINEL) for _ in range(n_d)]
    ref.step(10, debug=False)
    fsp.sharded_step_fp32_gather(plan, [g.t for g in f32.grads], *[s.t for s in f32.state], [b.t for b in bufs],
                                 HP, 10)
    fsp.sharded_step(z3.plan, [g.t for g in z3.grads], *[s.t for s in z3.state], None, HP, 10)
    torch.cuda.synchronize()
    for a, b in zip(ref.state, f32.state):
        assert np.array_equal(a.bits(), b.bits())
    want = _expected_copies(plan, f32.state[0].bits(), n_d)
    for q, b in enumerate(bufs):
        assert np.array_equal(b.bits(), want[q]), f"rank {q}"
    # the fp32 unshard of the ZeRO-3 state gives the same buffers
    out = [Guarded(plan.full_len_padded, torch.float32, STATE_SENTINEL) for _ in range(n_d)]
    fsp.unshard(z3.plan, z3.state[0].t, [b.t for b in out], fp32=True)
    torch.cuda.synchronize()
    for q, b in enumerate(out):
        assert np.array_equal(b.bits(), want[q]), f"unshard rank {q}"
    assert all(b.guards_intact() for b in bufs + out)
    assert fsp.device_error() == 0
