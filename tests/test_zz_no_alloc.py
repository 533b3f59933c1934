"""fsp_sharded_step_noalloc, called through the C ABI, gives the results of
fsp_sharded_step on two calls in a row.

The no-allocation entry point serves callers that cannot call cudaMalloc (a
framework's allocator owns the device, a fixed pool must not grow, or the
call sits where the CUDA allocator must not be reached): it keeps the tile
list in the library's fixed device array instead of a per-plan allocation.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
from fsdp_sharded_mixed_pass_gb300 import fsp as B
from synth_inputs import workload

from gpu_cases import HP, DeviceCase, ensure_built, ulp_dist, within_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _noalloc_call(case: DeviceCase, t: int):
    args = B._step_args(case.plan, [g.t for g in case.grads], *[s.t for s in case.state],
                        [p.t for p in case.params], HP, t, case.grad_dtype)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return B.lib().fsp_sharded_step_noalloc(*args, stream)


CASES = [
    (workload(0).shapes, 4, "fsdp2", "f32", workload(0).data_seed),
    (((3001, 7), (5, 4099), (1,), (12289,), (777, 64)), 6, "fsdp2", "bf16", 31),
    (((4097,), (64, 129), (2, 3, 5)), 3, "distopt", "f32", 7),
]


@pytest.mark.parametrize("shapes,n_d,mode,grad_dtype,seed", CASES)
def test_noalloc_matches_sharded_step_on_two_calls(shapes, n_d, mode, grad_dtype, seed):
    ref = DeviceCase(shapes, n_d, mode, grad_dtype, seed)
    new = DeviceCase(shapes, n_d, mode, grad_dtype, seed)
    for t in (10, 11):
        ref.step(t, debug=False)
        assert _noalloc_call(new, t) == B.FSP_OK, B.lib().fsp_last_error().decode()
        torch.cuda.synchronize()
        for a, b in zip(ref.state, new.state):
            ab, bb = a.bits(), b.bits()
            # identical bits (this covers the NaN sentinels in padding slots) or within tolerance
            ok = (ab == bb) | within_tol(bb.view(np.float32), ab.view(np.float32))
            assert ok.all()
        for a, b in zip(ref.params, new.params):
            assert ulp_dist(b.bits(), a.bits()).max(initial=0) <= 1
        assert new.all_guards_intact()


def test_noalloc_rejects_plans_beyond_its_array():
    # 262144 tiles of 4096 elements: one element more needs one tile more
    plan = fsp.plan_layout([(262144 * 4096 + 1,)], 1)
    assert plan.n_tiles == 262145
    fake = ctypes.c_void_p(1 << 40)
    ptrs = (ctypes.c_void_p * 1)(fake)
    hp = B._hp(HP)
    st = B.lib().fsp_sharded_step_noalloc(plan.handle, ptrs, 0, fake, fake, fake, ptrs, ctypes.byref(hp), 1,
                                          ctypes.c_void_p(0))
    assert st == B.FSP_EUNSUPPORTED
    assert "262144" in B.lib().fsp_last_error().decode()
