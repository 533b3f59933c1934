"""GPU parity of the distributed-optimizer flow with clipping: reduce-scatter
written back into the owners' grad slices, global norm, clipped AdamW."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
import synth_inputs as S
from oracle import plan as OP
from oracle import step as OS
from synth_inputs import workload

from gpu_cases import (HP, SCALED_BOUND, DeviceCase, OracleCase, check_params, ensure_built, PARAM_ULP_BAR,
                       state_errors, ulp_dist, within_tol)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


def _clipped(dev: DeviceCase, t, max_norm):
    out = torch.zeros(4, dtype=torch.float32, device="cuda")
    fsp.sharded_step_clipped(dev.plan, [g.t for g in dev.grads], *[s.t for s in dev.state],
                             [p.t for p in dev.params], HP, t, max_norm, out)
    torch.cuda.synchronize()
    return float(out[0]), np.float32(out[1].item())


def _check(dev, ora, norm, coef, o_norm, o_coef):
    assert abs(norm - o_norm) <= 1e-6 * o_norm + 1e-30
    assert ulp_dist(np.array([coef]).view(np.uint32), np.array([o_coef], np.float32).view(np.uint32))[0] <= 1
    # write-back: owner slices bit-exact, the rest of every grad buffer unchanged
    for q, (g, og) in enumerate(zip(dev.grads, ora.grads)):
        assert np.array_equal(g.bits(), og.view(np.uint32)), f"grad buffer {q}"
    si = ora.si
    gots = [d.bits()[si].view(np.float32) for d in dev.state]
    errs = state_errors(gots, [o[si] for o in ora.state], [o[si] for o in ora.prev])
    for name, g_, o_, e in zip(("master", "m", "v"), gots, ora.state, errs):
        assert within_tol(g_, o_[si]).all(), name
        assert (e <= SCALED_BOUND * 2 ** 24).all(), f"{name}: {e.max():.1f}"
    p0 = dev.params[0].bits()
    assert np.array_equal(p0[ora.fi], OS.bf16_rne(gots[0])), "params != bf16_rne(device master)"
    for q in range(len(dev.params)):
        assert np.array_equal(dev.params[q].bits(), p0)
        check_params(dev.params[q].bits(), ora.params[q], ora.fi, f"param copy {q}")
    assert dev.all_guards_intact() and fsp.device_error() == 0


@pytest.mark.parametrize("mode", ["fsdp2", "distopt"])
@pytest.mark.parametrize("n_d", [1, 2, 3, 4, 6, 8, 9, 16])
@pytest.mark.parametrize("max_norm", [1e-4, 1e30])
def test_clipped_step_matches_oracle(mode, n_d, max_norm):
    rng = np.random.default_rng(n_d * 7 + (mode == "distopt"))
    shapes = [(int(rng.integers(1, 3 * n_d + 5)), int(rng.choice([1, 3, 64]))) for _ in range(6)] + [(4097,)]
    dev = DeviceCase(shapes, n_d, mode, "f32", 500 + n_d)
    ora = OracleCase(shapes, n_d, mode, "f32", 500 + n_d)
    for t in (10, 11):
        norm, coef = _clipped(dev, t, max_norm)
        ora.prev = [a.copy() for a in ora.state]
        ora.hp = HP
        o_norm, o_coef = OS.sharded_step_clipped(ora.plan, ora.grads, *ora.state, ora.params, HP, t, max_norm)
        _check(dev, ora, norm, coef, o_norm, o_coef)
        if max_norm > 1e20:
            assert coef == 1.0
        else:
            assert coef < 1.0


def test_unclipped_flow_equals_the_fused_step():
    w = workload(0)
    a = DeviceCase(w.shapes, w.n_d, w.mode, "f32", w.data_seed)
    b = DeviceCase(w.shapes, w.n_d, w.mode, "f32", w.data_seed)
    _clipped(a, w.step, 1e30)
    b.step(w.step, debug=False)
    torch.cuda.synchronize()
    for x, y in zip(a.state + a.params, b.state + b.params):
        assert np.array_equal(x.bits(), y.bits())


@pytest.mark.parametrize("idx", [1, 2], ids=lambda i: workload(i).name)
def test_clipped_full_size(idx):
    """Full-size workload: the norm against an fp64 torch sum of the rank-ordered
    fold, write-back against that fold, sampled elements against the oracle."""
    w = workload(idx)
    dev = DeviceCase(w.shapes, w.n_d, w.mode, "f32", w.data_seed)
    try:
        # the reduced gradient, folded in rank order in fp32 with torch, before the step
        G = torch.zeros(dev.plan.full_len_padded, dtype=torch.float32, device="cuda")
        for g in dev.grads:
            G += g.t
        G /= float(w.n_d)
        ref_norm = float(torch.sqrt(torch.sum(G[:dev.plan.valid_elems].double() ** 2)))
        norm, coef = _clipped(dev, w.step, 0.05)
        assert abs(norm - ref_norm) <= 1e-6 * ref_norm
        assert coef == OS.clip_coefficient(ref_norm, 0.05) or \
            ulp_dist(np.array([coef]).view(np.uint32),
                     np.array([OS.clip_coefficient(ref_norm, 0.05)]).view(np.uint32))[0] <= 1
        assert coef < 1.0
        for sg in dev.plan.segments:   # write-back into every owner's slice
            if sg.length:
                a, n = sg.full_off, sg.length
                assert torch.equal(dev.grads[sg.rank].t[a:a + n], G[a:a + n])
        # sampled elements: oracle step with the GPU's coefficient
        oplan = OP.plan_layout(w.shapes, w.n_d, w.mode)
        rng = np.random.default_rng(5)
        f = np.unique(rng.integers(0, oplan.valid_elems, 100_000))
        segs = sorted((s for s in oplan.segments if s.length), key=lambda s: s.full_off)
        starts = np.array([s.full_off for s in segs])
        k = np.searchsorted(starts, f, side="right") - 1
        sidx = f + np.array([s.state_off - s.full_off for s in segs])[k]
        Gf = OS.average(OS.rank_ordered_sum([S.grad_f32(w.data_seed, q, f) for q in range(w.n_d)]), w.n_d)
        olds = (S.master_f32(w.data_seed, f), S.adam_m_f32(w.data_seed, f), S.adam_v_f32(w.data_seed, f))
        th, mm, vv = OS.adamw(*olds, (Gf * coef).astype(np.float32), HP, w.step)
        sd = torch.from_numpy(sidx).cuda()
        got = [st.t[sd].cpu().numpy() for st in dev.state]
        for name, g_, r_, e in zip(("master", "m", "v"), got, (th, mm, vv), state_errors(got, (th, mm, vv), olds)):
            assert within_tol(g_, r_).all() and (e <= SCALED_BOUND * 2 ** 24).all(), name
        p0 = dev.params[0].t.view(torch.int16)[torch.from_numpy(f).cuda()].cpu().numpy().view(np.uint16)
        assert np.array_equal(p0, OS.bf16_rne(got[0])), "params != bf16_rne(device master)"
        assert (ulp_dist(p0, OS.bf16_rne(th)) <= PARAM_ULP_BAR).all()
        assert fsp.device_error() == 0
    finally:
        del dev
        torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", ["fsdp2", "distopt"])
def test_norm_is_accurate_far_beyond_the_bar(mode):
    """The norm's squares are summed per thread in an fp32 pair (Dot2), then in
    fp64, and the result is handed out as fp32: on 12.3 M elements it is the
    fp32 rounding of an fp64 torch norm of the same reduced gradient (1 ulp at
    most, for a norm that falls next to a rounding boundary), where the stated
    bar would allow 1e-6 relative (~17 ulps)."""
    shapes = [(3000, 4096), (4099,), (77, 3)]
    dev = DeviceCase(shapes, 8, mode, "f32", 77)
    try:
        G = torch.zeros(dev.plan.full_len_padded, dtype=torch.float32, device="cuda")
        for g in dev.grads:
            G += g.t
        G /= 8.0
        ref = float(torch.sqrt(torch.sum(G[:dev.plan.valid_elems].double() ** 2)))
        norm, _ = _clipped(dev, 3, 1.0)
        got = np.array([norm], np.float32).view(np.uint32)
        want = np.array([ref], np.float32).view(np.uint32)
        assert ulp_dist(got, want)[0] <= 1, (norm, ref)
        assert fsp.device_error() == 0
    finally:
        del dev
        torch.cuda.empty_cache()


@pytest.mark.parametrize("n_rep,n_shard", [(2, 2), (2, 4), (3, 3), (4, 2)])
@pytest.mark.parametrize("max_norm", [1e-4, 1e30])
def test_hsdp_clipped_step_matches_oracle(n_rep, n_shard, max_norm):
    """HSDP meshes: the grouped reduction written back to the owner in every
    replica group, the norm over each element once, every group's state copy
    updated with the clipped gradient and gathered within its group."""
    rng = np.random.default_rng(n_rep * 13 + n_shard)
    shapes = [(int(rng.integers(1, 3 * n_shard + 5)), int(rng.choice([1, 3, 64]))) for _ in range(5)] + [(4097,)]
    n_d = n_rep * n_shard
    dev = DeviceCase(shapes, n_d, "hsdp", "f32", 700 + n_d, n_rep)
    ora = OracleCase(shapes, n_d, "hsdp", "f32", 700 + n_d, n_rep)
    for t in (10, 11):
        norm, coef = _clipped(dev, t, max_norm)
        ora.prev = [a.copy() for a in ora.state]
        ora.hp = HP
        o_norm, o_coef = OS.sharded_step_clipped(ora.plan, ora.grads, *ora.state, ora.params, HP, t, max_norm)
        _check(dev, ora, norm, coef, o_norm, o_coef)
        assert (coef < 1.0) == (max_norm < 1e20)
