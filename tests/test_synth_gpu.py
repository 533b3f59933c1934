"""The device generator reproduces the host generator bit for bit."""
import numpy as np
import pytest
import torch

import synth_inputs as S
from synth_inputs import device as D

from gpu_cases import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


@pytest.mark.parametrize("start", [0, 12345, 2 ** 33 + 7])
def test_device_matches_host(start):
    n = 300_001
    idx = np.arange(start, start + n, dtype=np.int64)
    for rank in (0, 5):
        t = torch.empty(n, dtype=torch.float32, device="cuda")
        D.fill_grad(t, 77, rank, "f32", start=start)
        assert np.array_equal(t.cpu().numpy().view(np.uint32), S.grad_f32(77, rank, idx).view(np.uint32))
        b = torch.empty(n, dtype=torch.bfloat16, device="cuda")
        D.fill_grad(b, 77, rank, "bf16", start=start)
        assert np.array_equal(b.view(torch.int16).cpu().numpy().view(np.uint16), S.grad_bf16_bits(77, rank, idx))
    m = torch.empty(n, device="cuda")
    a = torch.empty(n, device="cuda")
    v = torch.empty(n, device="cuda")
    D.fill_state_segments(m, a, v, 9, [(start, 0, n)])
    assert np.array_equal(m.cpu().numpy(), S.master_f32(9, idx))
    assert np.array_equal(a.cpu().numpy(), S.adam_m_f32(9, idx))
    assert np.array_equal(v.cpu().numpy(), S.adam_v_f32(9, idx))
