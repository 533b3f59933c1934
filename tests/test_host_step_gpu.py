"""fsp_sharded_step_host (gradients and bf16 params in host memory, state on
the device, chunked copy/compute pipeline) gives fsp_sharded_step's results."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
from synth_inputs import workload

from gpu_cases import HP, PARAM_SENTINEL, DeviceCase, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


CASES = [
    (workload(0).shapes, 4, "fsdp2", "f32", workload(0).data_seed, 8192),
    (workload(0).shapes, 4, "fsdp2", "f32", workload(0).data_seed, 0),
    (((3001, 7), (5, 4099), (1,), (12289,), (777, 64), (2, 3, 5)), 6, "fsdp2", "bf16", 31, 4096),
    (((4097,), (64, 129), (2, 3, 5), (9000,)), 3, "distopt", "f32", 7, 12288),
    (((40, 9), (7,)), 16, "fsdp2", "bf16", 5, 0),
    (((3 * 33 + 1, 17), (5,)), 33, "fsdp2", "f32", 6, 4096),
]


CASES += [
    (((3001, 7), (12289,), (9, 5)), 8, "hsdp", "f32", 11, 4096),   # 2 x 4 mesh
    (((3001, 7), (12289,), (9, 5)), 6, "hsdp", "bf16", 12, 8192),  # 2 x 3 mesh (generic kernel)
    (((3000, 4096), (4099,), (77, 3)), 4, "fsdp2", "f32", 13, 0),   # one chunk with tiles in order
]


@pytest.mark.parametrize("shapes,n_d,mode,grad_dtype,seed,chunk", CASES)
def test_host_step_matches_device_step(shapes, n_d, mode, grad_dtype, seed, chunk):
    n_rep = 2 if mode == "hsdp" else 1
    ref = DeviceCase(shapes, n_d, mode, grad_dtype, seed, n_rep)
    hst = DeviceCase(shapes, n_d, mode, grad_dtype, seed, n_rep)
    plan = hst.plan
    host_g = [g.t.cpu().pin_memory() for g in hst.grads]
    host_p = [torch.full((plan.full_len_padded,), PARAM_SENTINEL - 65536, dtype=torch.int16).view(torch.bfloat16)
              .pin_memory() for _ in range(n_d)]
    ws = torch.empty(fsp.host_step_workspace_bytes(plan, grad_dtype, chunk), dtype=torch.uint8, device="cuda")
    for t in (10, 11):
        ref.step(t, debug=False)
        fsp.sharded_step_host(plan, host_g, *[s.t for s in hst.state], host_p, HP, t, ws, chunk_elems=chunk,
                              grad_dtype=grad_dtype)
        torch.cuda.synchronize()
        for a, b in zip(ref.state, hst.state):
            assert np.array_equal(a.bits(), b.bits())
        for q in range(n_d):
            got = host_p[q].view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(got, ref.params[q].bits())
    assert fsp.device_error() == 0


def test_host_step_rejects_bad_workspace_and_device_buffers():
    shapes, n_d = workload(0).shapes, 4
    c = DeviceCase(shapes, n_d, "fsdp2", "f32", 1)
    host_g = [g.t.cpu().pin_memory() for g in c.grads]
    host_p = [p.t.cpu().pin_memory() for p in c.params]
    need = fsp.host_step_workspace_bytes(c.plan, "f32", 8192)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fsp.FspError, match="workspace too small"):
        fsp.sharded_step_host(c.plan, host_g, *[s.t for s in c.state], host_p, HP, 1, small, chunk_elems=8192)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(fsp.FspError, match="host memory"):
        fsp.sharded_step_host(c.plan, [g.t for g in c.grads], *[s.t for s in c.state], host_p, HP, 1, ws,
                              chunk_elems=8192)
    torch.cuda.synchronize()
