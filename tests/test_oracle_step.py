"""Pins of the oracle's step (CPU only).

Each stage is tied to something other than the oracle itself: the pages' worked
all-reduce = reduce-scatter + all-gather example, hand-worked AdamW cases with
exactly representable numbers, torch.optim.AdamW for the update's form, a
library routine for the bf16 cast, exact
rational arithmetic for the averaging, and brute-force agreement between the
sharded step and the unsharded all-reduce definition.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import synth_inputs as S
from oracle import plan as P
from oracle import step as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Stage 1: reduce-scatter
# --------------------------------------------------------------------------

def test_zero1_toy_rs_ag_equals_half_all_reduce():
    g = _golden("zero1_toy.json")
    n = g["n_ranks"]
    grads = [np.float32(10 * r) + np.arange(8, dtype=np.float32) for r in range(n)]
    plan = P.plan_fsdp2([(8,)], n)
    assert O.all_reduce(grads, mean=False).tolist() == g["all_reduce"]
    sums = O.reduce_scatter(plan, grads, mean=False)
    rank0 = [s for s, seg in zip(sums, plan.segments) if seg.rank == 0][0]
    assert rank0.tolist() == g["reduce_scatter_rank0"]
    gathered = O.rs_update_ag(plan, grads, lambda s: np.float32(0.5) * s)
    for buf in gathered:
        assert buf.tolist() == g["all_gather_of_half_sum"]
        assert (buf.tolist() == (0.5 * np.array(g["all_reduce"])).tolist()) == g["rs_ag_equals_half_ar"]
    # the step averages: every owner sees the all-reduce divided by N
    avg = np.concatenate(O.reduce_scatter(plan, grads, mean=True))
    assert avg.tolist() == [x / n for x in g["all_reduce"]] == [15.0, 16.0, 17.0, 18.0, 19.0, 20.0, 21.0, 22.0]


def test_sum_is_left_fold_in_rank_order():
    # fp32: 1e8 + 1 rounds back to 1e8, so only the left fold 0..3 gives 1.
    grads = [np.array([v], np.float32) for v in (1e8, 1.0, -1e8, 1.0)]
    assert O.rank_ordered_sum(grads).tolist() == [1.0]
    grads = [np.array([v], np.float32) for v in (1.0, 1e8, 1.0, -1e8)]
    assert O.rank_ordered_sum(grads).tolist() == [0.0]


def _correctly_rounded_f32(exact: Fraction) -> set:
    """The fp32 value(s) nearest to ``exact`` (two on an exact tie)."""
    approx = np.float32(float(exact))
    cands = [np.nextafter(approx, np.float32(-np.inf)), approx, np.nextafter(approx, np.float32(np.inf))]
    dist = [abs(Fraction(float(c)) - exact) for c in cands]
    best = min(dist)
    return {float(c) for c, d in zip(cands, dist) if d == best}


def test_average_is_correctly_rounded_division():
    """x / 6 rounded once - not x * fl(1/6), which differs for some x."""
    rng = np.random.default_rng(3)
    xs = rng.standard_normal(20000).astype(np.float32)
    inv = np.float32(1) / np.float32(6)
    differing = [x for x in xs if np.float32(x * inv) != np.float32(x / np.float32(6))]
    assert len(differing) > 10
    for x in differing[:200]:
        got = O.average(np.array([x], np.float32), 6)[0]
        assert float(got) in _correctly_rounded_f32(Fraction(float(x)) / 6)


def test_bf16_grads_widen_exactly():
    bits = np.array([0x3F80, 0xBF80, 0x3A83, 0x0001, 0x7F7F], np.uint16)
    got = O.bf16_bits_to_f32(bits)
    want = torch.tensor(bits.astype(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# --------------------------------------------------------------------------
# Stage 2: AdamW, hand-worked with exactly representable numbers
# --------------------------------------------------------------------------

def _hp(**kw):
    h = dict(lr=0.0, beta1=0.9, beta2=0.95, eps=0.0, weight_decay=0.0)
    h.update(kw)
    return h


def _one(theta, m, v, g, hp, t):
    th, mm, vv = O.adamw(np.array([theta], np.float32), np.array([m], np.float32),
                         np.array([v], np.float32), np.array([g], np.float32), hp, t)
    return float(th[0]), float(mm[0]), float(vv[0])


def test_adamw_worked_case():
    # m' = .5*.25 + .5*.5 = .375; v' = .75*.0625 + .25*.25 = .109375
    # bias corrections at t=2: 1-.25 = .75 and 1-.5625 = .4375 -> m_hat .5, v_hat .25
    # theta' = 1 - .125 * .5 / sqrt(.25) = .875
    assert _one(1.0, 0.25, 0.0625, 0.5, _hp(lr=0.125, beta1=0.5, beta2=0.75), 2) == (0.875, 0.375, 0.109375)


def test_adamw_weight_decay_is_decoupled_on_old_theta():
    # as above with wd = .5: 1 - .125*.5*1 - .125*1 = .8125
    # (decaying after the step would give .875 * .9375 = .8203125)
    th, _, _ = _one(1.0, 0.25, 0.0625, 0.5, _hp(lr=0.125, beta1=0.5, beta2=0.75, weight_decay=0.5), 2)
    assert th == 0.8125


def test_adamw_ema_operands():
    # lr = 0: theta unchanged; m' = .75*.25 + .25*.5 = .3125, v' = .5*.125 + .5*.25 = .1875
    assert _one(2.0, 0.25, 0.125, 0.5, _hp(beta1=0.75, beta2=0.5), 7) == (2.0, 0.3125, 0.1875)


def test_adamw_first_step_moves_by_lr_times_normalised_grad():
    # t=1, m=v=0: m_hat = G, v_hat = G^2, so theta' = theta - lr G / (|G| + eps).
    # G = 2^-10, eps = 2^-12: G / (|G| + eps) = 4/5 ; lr = 1/8 -> step 0.1
    G, eps, lr = 2.0 ** -10, 2.0 ** -12, 0.125
    th, mm, vv = _one(1.0, 0.0, 0.0, G, _hp(lr=lr, eps=eps), 1)
    assert th == pytest.approx(1.0 - 0.1, rel=0, abs=2 ** -23)
    th_neg, _, _ = _one(1.0, 0.0, 0.0, -G, _hp(lr=lr, eps=eps), 1)
    assert th_neg == pytest.approx(1.0 + 0.1, rel=0, abs=2 ** -23)


def test_adamw_zero_grad_only_decays():
    # G = 0, m = v = 0: theta' = theta (1 - lr wd) = 1 - .5*.25 = .875
    assert _one(1.0, 0.0, 0.0, 0.0, _hp(lr=0.5, weight_decay=0.25, eps=1e-8), 3) == (0.875, 0.0, 0.0)


def test_adamw_zero_betas():
    # b1 = b2 = 0: m' = G, v' = G^2, no bias correction; G = .25, lr = .5, eps = .25
    # theta' = 3 - .5 * .25 / (.25 + .25) = 2.75
    assert _one(3.0, 9.0, 9.0, 0.25, _hp(lr=0.5, beta1=0.0, beta2=0.0, eps=0.25), 5) == (2.75, 0.25, 0.0625)


# --------------------------------------------------------------------------
# Stage 3: bf16 cast
# --------------------------------------------------------------------------

@pytest.mark.parametrize("t", [1, 10, 1000])
def test_adamw_matches_torch_optim_adamw(t):
    """The reading 'PyTorch-style decoupled AdamW' checked against an
    implementation that is not the oracle's: torch.optim.AdamW in fp64, from
    the same m, v and step count t - 1, one step.  Both round to fp32 at the
    end; they agree bit for bit except where the two fp64 evaluations straddle
    an fp32 rounding boundary (then by one ulp)."""
    n = 100_000
    idx = np.arange(n)
    g = S.grad_f32(77, 0, idx)
    th, m, v = S.master_f32(77, idx), S.adam_m_f32(77, idx), S.adam_v_f32(77, idx)
    want = O.adamw(th, m, v, g, HP, t)
    h = O.hparams_f32(HP)
    p = torch.nn.Parameter(torch.from_numpy(th.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=h["lr"], betas=(h["beta1"], h["beta2"]), eps=h["eps"],
                            weight_decay=h["weight_decay"], foreach=False)
    p.grad = torch.from_numpy(g.astype(np.float64))
    opt.state[p] = {"step": torch.tensor(float(t - 1), dtype=torch.float64),
                    "exp_avg": torch.from_numpy(m.astype(np.float64)),
                    "exp_avg_sq": torch.from_numpy(v.astype(np.float64))}
    opt.step()
    got = (p.detach().numpy().astype(np.float32), opt.state[p]["exp_avg"].numpy().astype(np.float32),
           opt.state[p]["exp_avg_sq"].numpy().astype(np.float32))
    for a, b in zip(got, want):
        ai = a.view(np.int32).astype(np.int64)
        bi = b.view(np.int32).astype(np.int64)
        assert np.abs(ai - bi).max() <= 1
        assert (ai == bi).mean() > 0.999


def test_bf16_rne_hand_cases():
    one = 1.0
    cases = {
        one: 0x3F80,
        one + 2 ** -8: 0x3F80,                 # halfway, kept part even -> down
        one + 3 * 2 ** -8: 0x3F82,             # halfway, kept part odd -> up
        one + 2 ** -8 + 2 ** -20: 0x3F81,      # just above halfway -> up
        one + 2 ** -8 - 2 ** -20: 0x3F80,      # just below halfway -> down
        -1.5: 0xBFC0,
        0.0: 0x0000,
    }
    xs = np.array(list(cases), np.float32)
    assert O.bf16_rne(xs).tolist() == list(cases.values())


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32) * 0.02,
                        rng.standard_normal(1000).astype(np.float32) * 1e30,
                        rng.standard_normal(1000).astype(np.float32) * 1e-38])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_rne(x), want)


# --------------------------------------------------------------------------
# The whole step: sharded == unsharded (all-reduce) definition, bit for bit
# --------------------------------------------------------------------------

SENTINEL_STATE = np.uint32(0x7FC0DEAD)
SENTINEL_PARAM = np.uint16(0xFFFF)


def _inputs(plan, grad_dtype, seed):
    full = plan.full_len_padded
    idx = np.arange(full)
    if grad_dtype == "f32":
        grads = [S.grad_f32(seed, q, idx) for q in range(plan.n_d)]
    else:
        grads = [S.grad_bf16_bits(seed, q, idx) for q in range(plan.n_d)]
    fi, si = P.owned_indices(plan)
    states = []
    for fn in (S.master_f32, S.adam_m_f32, S.adam_v_f32):
        buf = np.full(plan.state_len_total, SENTINEL_STATE, np.uint32).view(np.float32)
        buf[si] = fn(seed, fi)
        states.append(buf)
    params = [np.full(full, SENTINEL_PARAM, np.uint16) for _ in range(plan.n_d)]
    return grads, states, params


def _tiny_shapes(rng, n_d):
    shapes = []
    for _ in range(int(rng.integers(1, 9))):
        rows = int(rng.integers(1, 2 * n_d + 4))
        cols = int(rng.choice([1, 3, 64]))
        shapes.append((rows,) if cols == 1 else (rows, cols))
    return shapes


@pytest.mark.parametrize("grad_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", ["fsdp2", "distopt"])
@pytest.mark.parametrize("n_d", [1, 2, 3, 4, 5, 6, 7, 8, 16])
def test_sharded_equals_unsharded(n_d, mode, grad_dtype):
    rng = np.random.default_rng(1000 * n_d + (mode == "distopt") * 10 + (grad_dtype == "bf16"))
    shapes = _tiny_shapes(rng, n_d)
    plan = P.plan_layout(shapes, n_d, mode)
    seed = 77 + n_d
    grads, (master, m, v), params = _inputs(plan, grad_dtype, seed)
    fi, si = P.owned_indices(plan)
    theta0, m0, v0 = master[si].copy(), m[si].copy(), v[si].copy()
    master_bits = master.view(np.uint32).copy()
    reduced = np.zeros(plan.state_len_total, np.float32)
    O.sharded_step(plan, grads, grad_dtype, master, m, v, params, HP, 10, reduced_out=reduced)

    # unsharded definition over the logical (full-index) order
    order = np.argsort(fi)
    n = plan.valid_elems
    th_f = np.empty(n, np.float32); m_f = np.empty(n, np.float32); v_f = np.empty(n, np.float32)
    th_f[fi] = theta0; m_f[fi] = m0; v_f[fi] = v0
    th_u, m_u, v_u, b_u = O.unsharded_step(grads, grad_dtype, th_f, m_f, v_f, n, HP, 10)
    assert np.array_equal(master[si][order].view(np.uint32), th_u.view(np.uint32))
    assert np.array_equal(m[si][order].view(np.uint32), m_u.view(np.uint32))
    assert np.array_equal(v[si][order].view(np.uint32), v_u.view(np.uint32))
    g_u = O.all_reduce(grads, grad_dtype, n)
    assert np.array_equal(reduced[si][order].view(np.uint32), g_u.view(np.uint32))
    for q in range(n_d):   # every rank's gathered copy is the same bf16 of the new master
        assert np.array_equal(params[q][:n], b_u)
        assert np.all(params[q][n:] == SENTINEL_PARAM)
    # state slots that no element owns keep their sentinel
    untouched = np.ones(plan.state_len_total, bool)
    untouched[si] = False
    assert np.array_equal(master.view(np.uint32)[untouched], master_bits[untouched])
    assert np.all(master.view(np.uint32)[untouched] == SENTINEL_STATE)


def test_fsdp2_and_distopt_agree_per_logical_element():
    shapes = [(9, 4), (3,), (17,), (2, 2, 2), (40, 3)]
    out = {}
    for mode in ("fsdp2", "distopt"):
        plan = P.plan_layout(shapes, 4, mode)
        grads, (master, m, v), params = _inputs(plan, "f32", 5)
        O.sharded_step(plan, grads, "f32", master, m, v, params, HP, 10)
        fi, si = P.owned_indices(plan)
        o = np.argsort(fi)
        out[mode] = (master[si][o], m[si][o], v[si][o], params[0][:plan.valid_elems])
    for a, b in zip(out["fsdp2"], out["distopt"]):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_step_index_must_be_positive():
    plan = P.plan_fsdp2([(4,)], 2)
    grads, (master, m, v), params = _inputs(plan, "f32", 1)
    with pytest.raises(ValueError):
        O.sharded_step(plan, grads, "f32", master, m, v, params, HP, 0)


def test_elementwise_step_matches_sharded_step():
    plan = P.plan_fsdp2([(13, 5), (7,)], 3)
    grads, (master, m, v), params = _inputs(plan, "f32", 9)
    fi, si = P.owned_indices(plan)
    th0, m0, v0 = master[si].copy(), m[si].copy(), v[si].copy()
    O.sharded_step(plan, grads, "f32", master, m, v, params, HP, 4)
    th, mm, vv, b, _ = O.elementwise_step([g[fi] for g in grads], "f32", th0, m0, v0, HP, 4)
    assert np.array_equal(th, master[si]) and np.array_equal(mm, m[si]) and np.array_equal(vv, v[si])
    assert np.array_equal(b, params[1][fi])


# --------------------------------------------------------------------------
# The pins are sensitive: plant a mistake in the oracle, watch a pin fail
# --------------------------------------------------------------------------

def _adamw_eps_inside_sqrt(theta, m, v, g, hp, t):
    h = O.hparams_f32(hp)
    th = np.asarray(theta, np.float64); mm = np.asarray(m, np.float64)
    vv = np.asarray(v, np.float64); gg = np.asarray(g, np.float64)
    m1 = h["beta1"] * mm + (1 - h["beta1"]) * gg
    v1 = h["beta2"] * vv + (1 - h["beta2"]) * gg * gg
    mh = m1 / (1 - h["beta1"] ** t); vh = v1 / (1 - h["beta2"] ** t)
    out = th - h["lr"] * h["weight_decay"] * th - h["lr"] * mh / np.sqrt(vh + h["eps"])
    return out.astype(np.float32), m1.astype(np.float32), v1.astype(np.float32)


def _adamw_no_bias_correction(theta, m, v, g, hp, t):
    return _adamw_with(theta, m, v, g, hp, t, bias=False)


def _adamw_with(theta, m, v, g, hp, t, bias=True):
    h = O.hparams_f32(hp)
    th = np.asarray(theta, np.float64); mm = np.asarray(m, np.float64)
    vv = np.asarray(v, np.float64); gg = np.asarray(g, np.float64)
    m1 = h["beta1"] * mm + (1 - h["beta1"]) * gg
    v1 = h["beta2"] * vv + (1 - h["beta2"]) * gg * gg
    mh = m1 / (1 - h["beta1"] ** t) if bias else m1
    vh = v1 / (1 - h["beta2"] ** t) if bias else v1
    out = th - h["lr"] * h["weight_decay"] * th - h["lr"] * mh / (np.sqrt(vh) + h["eps"])
    return out.astype(np.float32), m1.astype(np.float32), v1.astype(np.float32)


@pytest.mark.parametrize("planted", [_adamw_eps_inside_sqrt, _adamw_no_bias_correction])
def test_planted_adamw_mistake_is_caught(monkeypatch, planted):
    monkeypatch.setattr(O, "adamw", planted)
    with pytest.raises(AssertionError):
        test_adamw_first_step_moves_by_lr_times_normalised_grad()
        test_adamw_worked_case()


def test_planted_reduction_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(O, "average", lambda s, n: (s * (np.float32(1) / np.float32(n))).astype(np.float32))
    with pytest.raises(AssertionError):
        test_average_is_correctly_rounded_division()
