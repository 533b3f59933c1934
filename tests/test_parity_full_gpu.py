"""GPU parity at the workloads' full sizes, in the launch configuration the
bench times (the production entry, one step): sampled elements against the
oracle one by one, plus properties checked over every element on the device."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
import synth_inputs as S
from oracle import plan as OP
from oracle import step as OS
from synth_inputs import device as D
from synth_inputs import workload

from gpu_cases import (HP, PARAM_SENTINEL, SCALED_BOUND, STATE_SENTINEL, Guarded, ensure_built,
                       PARAM_ULP_BAR, state_errors, ulp_dist, within_tol)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _sample_indices(oplan, rng, n_random):
    """Random full indices plus every segment's first/last elements and the
    elements around its 4096-element tile boundaries."""
    P = oplan.valid_elems
    picks = [rng.integers(0, P, size=min(n_random, P))] if P else []
    for s in oplan.segments:
        if s.length == 0:
            continue
        a, b = s.full_off, s.full_off + s.length
        edge = [a, a + 1, a + 2, a + 3, b - 4, b - 3, b - 2, b - 1]
        t = (a // 4096 + 1) * 4096
        if t < b:
            edge += [t - 1, t, t + 1]
        picks.append(np.clip(np.array(edge, np.int64), a, b - 1))
    return np.unique(np.concatenate(picks)) if picks else np.zeros(0, np.int64)


def _state_index(oplan, f):
    """Replica 0's state slot of each full index."""
    segs = sorted((s for s in oplan.segments if s.length and s.rank < oplan.n_shard), key=lambda s: s.full_off)
    starts = np.array([s.full_off for s in segs], np.int64)
    k = np.searchsorted(starts, f, side="right") - 1
    offs = np.array([s.state_off - s.full_off for s in segs], np.int64)
    return f + offs[k]


def _full_size_case(shapes, n_d, mode, grad_dtype, seed, t, n_random=200_000, n_rep=1):
    plan = fsp.plan_layout(shapes, n_d, mode, n_replicate=n_rep)
    oplan = OP.plan_layout(shapes, n_d, mode, n_rep=n_rep)
    gdt = torch.float32 if grad_dtype == "f32" else torch.bfloat16
    grads = [Guarded(plan.full_len_padded, gdt, 0) for _ in range(n_d)]
    for q, g in enumerate(grads):
        D.fill_grad(g.t, seed, q, grad_dtype)
    state = [Guarded(plan.state_len_total, torch.float32, STATE_SENTINEL) for _ in range(3)]
    D.fill_state_segments(state[0].t, state[1].t, state[2].t, seed,
                          [(s.full_off, s.state_off, s.length) for s in plan.segments])
    params = [Guarded(plan.full_len_padded, torch.bfloat16, PARAM_SENTINEL) for _ in range(n_d)]
    torch.cuda.synchronize()

    fsp.sharded_step(plan, [g.t for g in grads], *[s.t for s in state], [p.t for p in params], HP, t)
    torch.cuda.synchronize()

    # --- sampled elements against the oracle ---------------------------------
    rng = np.random.default_rng(seed)
    f = _sample_indices(oplan, rng, n_random)
    s = _state_index(oplan, f)
    fd = torch.from_numpy(f).cuda()
    sd = torch.from_numpy(s).cuda()
    got = [st.t[sd].cpu().numpy() for st in state]
    for r in range(1, n_rep):   # every replica group's copy of the state is the same
        for st in state:
            assert np.array_equal(st.t[sd + r * (plan.state_len_total // n_rep)].cpu().numpy().view(np.uint32),
                                  got[state.index(st)].view(np.uint32))
    got_p = [p.t.view(torch.int16)[fd].cpu().numpy().view(np.uint16) for p in params]
    if grad_dtype == "f32":
        cols = [S.grad_f32(seed, q, f) for q in range(n_d)]
    else:
        cols = [S.grad_bf16_bits(seed, q, f) for q in range(n_d)]
    olds = (S.master_f32(seed, f), S.adam_m_f32(seed, f), S.adam_v_f32(seed, f))
    th, mm, vv, b, _ = OS.elementwise_step(cols, grad_dtype, *olds, HP, t, n_rep=n_rep)
    errs = state_errors(got, (th, mm, vv), olds)
    for name, g_, r_, se in zip(("master", "exp_avg", "exp_avg_sq"), got, (th, mm, vv), errs):
        ok = within_tol(g_, r_)
        assert ok.all(), f"{name}: {int((~ok).sum())} of {ok.size} sampled elements out of tolerance"
        assert np.all(se <= SCALED_BOUND * 2 ** 24), f"{name}: error {se.max():.1f} x 2^-24 of the terms' scale"
    for q in range(n_d):
        assert np.array_equal(got_p[q], OS.bf16_rne(got[0])), f"param copy {q} != bf16_rne(device master)"
        assert (ulp_dist(got_p[q], b) <= PARAM_ULP_BAR).all(), f"param copy {q} more than 1 bf16 ulp from the oracle"

    # --- properties over every element ---------------------------------------
    p0 = params[0].t.view(torch.int16)
    for q in range(1, n_d):
        assert torch.equal(params[q].t.view(torch.int16), p0), f"param copy {q} differs from copy 0"
    master = state[0].t
    if mode == "distopt":
        n = plan.valid_elems
        assert torch.equal(p0[:n], master[:n].to(torch.bfloat16).view(torch.int16))
        assert bool((p0[n:] == -1).all()), "DistOpt padding of a param buffer was written"
    else:
        for sg in plan.segments:
            if sg.length:
                a, c = sg.full_off, sg.state_off
                assert torch.equal(p0[a:a + sg.length],
                                   master[c:c + sg.length].to(torch.bfloat16).view(torch.int16))
    padding = plan.state_len_total - plan.valid_elems * n_rep
    for st in state:
        n_sent = int((st.t.view(torch.int32) == int(np.uint32(STATE_SENTINEL).view(np.int32))).sum())
        assert n_sent == padding, "a padding slot of the state was written (or an owned one was not)"
    assert all(x.guards_intact() for x in grads + state + params), "guard band overwritten"
    assert fsp.device_error() == 0, "a bounded wait in the step kernel ran out"


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4, 5], ids=lambda i: workload(i).name)
def test_workload_full_size(idx):
    w = workload(idx)
    try:
        _full_size_case(w.shapes, w.n_d, w.mode, w.grad_dtype, w.data_seed, w.step, n_rep=w.n_rep)
    finally:
        torch.cuda.empty_cache()


def test_more_than_2_31_elements():
    """A 1-D parameter of 2^31 + 4099 elements on 2 ranks: full and state
    indices beyond 32 bits."""
    try:
        _full_size_case([(2 ** 31 + 4099,)], 2, "fsdp2", "f32", seed=44, t=3, n_random=50_000)
    finally:
        torch.cuda.empty_cache()
