"""The step with the distributed optimizer's write-back: every element's
averaged gradient also lands in its owner's slice of the owner's own fp32 grad
buffer, in the same pass; state and parameters equal the plain step's."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp

from gpu_cases import HP, DeviceCase, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


SMALL = ((3001, 7), (77, 3), (4099,), (1,), (12289,), (9, 5), (0, 4))
BIG = ((3000, 4096), (4099,), (77, 3))


@pytest.mark.parametrize("shapes,n_d,mode", [
    (SMALL, 4, "fsdp2"), (SMALL, 8, "fsdp2"), (SMALL, 6, "fsdp2"), (SMALL, 3, "distopt"),
    (SMALL, 9, "fsdp2"),          # per-thread kernel
    (BIG, 4, "fsdp2"),            # tiles in order from the counter
])
def test_writeback_step(shapes, n_d, mode):
    ref = DeviceCase(shapes, n_d, mode, "f32", 101)
    wb = DeviceCase(shapes, n_d, mode, "f32", 101)
    before = [g.bits().copy() for g in wb.grads]
    ref.step(10, debug=True)                  # reduced gradient into ref.reduced (state layout)
    fsp.sharded_step_writeback(wb.plan, [g.t for g in wb.grads], *[s.t for s in wb.state],
                               [p.t for p in wb.params], HP, 10)
    torch.cuda.synchronize()
    for a, b in zip(ref.state + ref.params, wb.state + wb.params):
        assert np.array_equal(a.bits(), b.bits())
    reduced = ref.reduced.bits()
    want = [x.copy() for x in before]
    for s in wb.plan.segments:
        if s.length:
            want[s.rank][s.full_off:s.full_off + s.length] = reduced[s.state_off:s.state_off + s.length]
    for q, g in enumerate(wb.grads):
        assert np.array_equal(g.bits(), want[q]), f"grad buffer {q}"
    assert wb.all_guards_intact()
    assert fsp.device_error() == 0
