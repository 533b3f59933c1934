"""fsp_sharded_step_noalloc, called through the C ABI, gives the results of
fsp_sharded_step bit for bit, on two calls in a row, and allocates no device
memory.

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

from gpu_cases import HP, PARAM_SENTINEL, DeviceCase, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _noalloc_call(case: DeviceCase, t: int, plan=None, gather=True):
    plan = plan or case.plan
    params = [p.t for p in case.params] if gather else None
    args = B._step_args(plan, [g.t for g in case.grads], *[s.t for s in case.state], params, HP, t,
                        case.grad_dtype)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return B.lib().fsp_sharded_step_noalloc(*args, stream)


def _step(case: DeviceCase, t: int, gather=True):
    params = [p.t for p in case.params] if gather else None
    fsp.sharded_step(case.plan, [g.t for g in case.grads], *[s.t for s in case.state], params, HP, t)


def _assert_same_bits(ref: DeviceCase, new: DeviceCase):
    """State and params identical bit for bit (padding sentinels included)."""
    for a, b in zip(ref.state + ref.params, new.state + new.params):
        assert np.array_equal(a.bits(), b.bits())
    assert new.all_guards_intact()


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
        _step(ref, t)
        assert _noalloc_call(new, t) == B.FSP_OK, B.lib().fsp_last_error().decode()
        torch.cuda.synchronize()
        _assert_same_bits(ref, new)
    assert fsp.device_error() == 0


def test_noalloc_without_param_buffers_is_the_zero3_step():
    """param_bufs NULL: the update without the all-gather, as fsp_sharded_step."""
    shapes, n_d, mode, grad_dtype, seed = CASES[1]
    ref = DeviceCase(shapes, n_d, mode, grad_dtype, seed)
    new = DeviceCase(shapes, n_d, mode, grad_dtype, seed)
    for t in (10, 11):
        _step(ref, t, gather=False)
        assert _noalloc_call(new, t, gather=False) == B.FSP_OK, B.lib().fsp_last_error().decode()
        torch.cuda.synchronize()
        _assert_same_bits(ref, new)
    for p in new.params:
        assert (p.bits() == PARAM_SENTINEL).all()


def test_noalloc_switches_between_plans():
    """Calls with plan A, then B, then A again: each call runs on its own
    plan's tile list (the shared array is rewritten when the plan changes)."""
    a_shapes, b_shapes = CASES[0][0], ((4099, 3), (17,), (8192,))
    ref_a, new_a = (DeviceCase(a_shapes, 4, "fsdp2", "f32", 5) for _ in range(2))
    ref_b, new_b = (DeviceCase(b_shapes, 4, "fsdp2", "f32", 6) for _ in range(2))
    for t, (ref, new) in zip((10, 10, 11), ((ref_a, new_a), (ref_b, new_b), (ref_a, new_a))):
        _step(ref, t)
        assert _noalloc_call(new, t) == B.FSP_OK, B.lib().fsp_last_error().decode()
        torch.cuda.synchronize()
        _assert_same_bits(ref, new)


def test_noalloc_allocates_no_device_memory():
    """Free device memory is unchanged across calls with a fresh plan whose
    tile list (65536 tiles, 2 MiB) goes into the library's array; the same
    call through fsp_sharded_step, which allocates a tile table of that size,
    shows up in the same measurement."""
    shapes = [(65536 * 4096,)]
    n = shapes[0][0]
    grads = [torch.zeros(n, dtype=torch.float32, device="cuda")]
    state = [torch.zeros(n, dtype=torch.float32, device="cuda") for _ in range(3)]
    params = [torch.zeros(n, dtype=torch.bfloat16, device="cuda")]
    stream = torch.cuda.current_stream()
    # a first call loads the library's code and arrays on this device (that load is not the call's allocation)
    warm = fsp.plan_layout(shapes, 1)
    fsp.sharded_step_noalloc(warm, grads, *state, params, HP, 1, stream=stream)
    torch.cuda.synchronize()
    fresh = fsp.plan_layout(shapes, 1)
    assert fresh.n_tiles == 65536
    before = torch.cuda.mem_get_info()[0]
    for t in (2, 3):
        fsp.sharded_step_noalloc(fresh, grads, *state, params, HP, t, stream=stream)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == before
    control = fsp.plan_layout(shapes, 1)
    before = torch.cuda.mem_get_info()[0]
    fsp.sharded_step(control, grads, *state, params, HP, 4, stream=stream)
    torch.cuda.synchronize()
    assert before - torch.cuda.mem_get_info()[0] >= 2 * 2 ** 20
    assert fsp.device_error() == 0


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
