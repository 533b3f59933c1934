"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in the oracle - a floor instead of a ceiling, a
wrong padding unit, a reversed fold, a truncating cast, a gather that misses
ranks, a wrong byte-ledger or collective-volume formula, ... - and requires
that at least one of the pins written against the pages, closed forms or
library routines then fails.  The mistakes are planted with monkeypatch, in
the oracle only, and undone after each case."""
from fractions import Fraction

import numpy as np
import pytest

import test_oracle_clip as TC
import test_oracle_hsdp as TH
import test_oracle_ledger as TL
import test_oracle_plan as TP
import test_oracle_step as TS
import test_oracle_unshard as TU
from oracle import ledger as L
from oracle import plan as P
from oracle import step as O


def _params_of(test, name):
    """The argument tuples a parametrised pin runs with."""
    for mark in getattr(test, "pytestmark", []):
        if mark.name == "parametrize" and mark.args[0].replace(" ", "") == name:
            return [a if isinstance(a, tuple) else (a,) for a in mark.args[1]]
    raise LookupError(name)


def _fails(pins) -> bool:
    for pin, args in pins:
        try:
            pin(*args)
        except Exception:   # an assertion, or the mistake breaking the code outright
            return True
    return False


# ---- planner mistakes ------------------------------------------------------

def _floor_chunk(mp):
    mp.setattr(P, "shard_rows", lambda rows, n_d: max(1, rows // n_d))


def _lcm_64(mp):
    mp.setattr(P, "DISTOPT_ALIGN", 64)


def _state_align_8(mp):
    mp.setattr(P, "STATE_ALIGN", 8)


def _ignore_param_align(mp):
    orig = P._offsets
    mp.setattr(P, "_offsets", lambda shapes, align=1: orig(shapes, 1))


def _hsdp_shard_major(mp):
    def plan_hsdp(shapes, n_rep, n_shard, param_align=1):
        inner = P.plan_fsdp2(shapes, n_shard, param_align)
        copy = n_shard * inner.state_len_per_rank
        segs = tuple(P.Segment(s.param, s.rank * n_rep + r, s.full_off, r * copy + s.state_off, s.length,
                               s.padded_len) for r in range(n_rep) for s in inner.segments)
        return P.Plan("hsdp", n_rep * n_shard, inner.shapes, inner.param_offsets, inner.valid_elems,
                      inner.full_len_padded, inner.state_len_per_rank, segs, n_rep)
    mp.setattr(P, "plan_hsdp", plan_hsdp)


# ---- step mistakes ---------------------------------------------------------

def _reversed_fold(mp):
    orig = O.rank_ordered_sum
    mp.setattr(O, "rank_ordered_sum", lambda slices: orig(list(slices)[::-1]))


def _groups_last(mp):
    # HSDP: fold across replica groups first, then inside the group
    def hybrid_sum(slices, n_rep):
        n_s = len(slices) // n_rep
        partials = [O.rank_ordered_sum(slices[j::n_s]) for j in range(n_s)]
        return O.rank_ordered_sum(partials)
    mp.setattr(O, "hybrid_sum", hybrid_sum)


def _truncating_cast(mp):
    mp.setattr(O, "bf16_rne", lambda x: (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16))


def _bf16_as_integers(mp):
    mp.setattr(O, "bf16_bits_to_f32", lambda bits: np.asarray(bits, np.uint16).astype(np.float32))


def _gather_to_owner_only(mp):
    def all_gather(plan, per_segment_values, params):
        for seg, vals in zip(plan.segments, per_segment_values):
            params[seg.rank][seg.full_off:seg.full_off + seg.length] = vals
    mp.setattr(O, "all_gather", all_gather)


def _decay_on_new_theta(mp):
    def adamw(theta, m, v, g, hp, t):
        h = O.hparams_f32(hp)
        th = np.asarray(theta, np.float32).astype(np.float64)
        mm = np.asarray(m, np.float32).astype(np.float64)
        vv = np.asarray(v, np.float32).astype(np.float64)
        gg = np.asarray(g, np.float32).astype(np.float64)
        m1 = h["beta1"] * mm + (1 - h["beta1"]) * gg
        v1 = h["beta2"] * vv + (1 - h["beta2"]) * gg * gg
        u = h["lr"] * (m1 / (1 - h["beta1"] ** t)) / (np.sqrt(v1 / (1 - h["beta2"] ** t)) + h["eps"])
        out = (th - u) * (1 - h["lr"] * h["weight_decay"])
        return out.astype(np.float32), m1.astype(np.float32), v1.astype(np.float32)
    mp.setattr(O, "adamw", adamw)


def _clip_without_epsilon(mp):
    mp.setattr(O, "clip_coefficient", lambda norm, max_norm: np.float32(min(1.0, float(np.float32(max_norm)) / norm)))


def _shard_first_group_only(mp):
    def shard(plan, full, master):
        full = np.asarray(full, dtype=np.float32)
        for seg in plan.segments:
            if seg.rank < plan.n_shard:
                master[seg.state_off:seg.state_off + seg.length] = full[seg.full_off:seg.full_off + seg.length]
    mp.setattr(O, "shard", shard)


# ---- ledger mistakes ---------------------------------------------------------

def _zero2_as_fsdp(mp):
    orig = L.bytes_per_param
    mp.setattr(L, "bytes_per_param",
               lambda scheme, n_d, grad_bytes=4: orig("fsdp" if scheme == "zero2" else scheme, n_d, grad_bytes))


def _all_reduce_once(mp):
    orig = L.coll_bytes
    mp.setattr(L, "coll_bytes", lambda kind, n, size: orig("all_gather" if kind == "all_reduce" else kind, n, size))


def _whole_payload(mp):
    orig = L.coll_bytes
    mp.setattr(L, "coll_bytes", lambda kind, n, size: Fraction(size) * (2 if kind == "all_reduce" else 1)
               if n > 1 and kind != "send_recv" else orig(kind, n, size))


def _no_gqa(mp):
    orig = L.dense_param_count
    mp.setattr(L, "dense_param_count", lambda h, layers, heads, kv_heads, *a, **k: orig(h, layers, heads, heads, *a, **k))


def _state_moved_once(mp):
    mp.setattr(L, "sharded_step_bytes", lambda n_d, grad_bytes, n_rep=1: n_d * grad_bytes + 12 * n_rep + 2 * n_d)


MUTANTS = {
    "floor_chunk": (_floor_chunk, [(TP.test_fsdp2_shards_equal_torch_chunk, (4,)),
                                   (TP.test_qwen3_layer_shard_table_matches_walkthrough, ())]),
    "lcm_64": (_lcm_64, [(TP.test_distopt_lcm_padding, a)
                         for a in _params_of(TP.test_distopt_lcm_padding, "total,n_d,padded")]),
    "state_align_8": (_state_align_8, [(TP.test_fsdp2_state_alignment_and_rank_major_order, ())]),
    "ignore_param_align": (_ignore_param_align, [(TP.test_per_param_layout_worked_by_hand, ())]),
    "hsdp_shard_major": (_hsdp_shard_major, [(TH.test_hsdp_plan_is_replicated_fsdp2, ())]),
    "reversed_fold": (_reversed_fold, [(TS.test_sum_is_left_fold_in_rank_order, ())]),
    "groups_last": (_groups_last, [(TH.test_hybrid_sum_is_group_then_across_groups, ())]),
    "truncating_cast": (_truncating_cast, [(TS.test_bf16_rne_hand_cases, ()), (TS.test_bf16_rne_matches_torch, ())]),
    "bf16_as_integers": (_bf16_as_integers, [(TS.test_bf16_grads_widen_exactly, ())]),
    "gather_to_owner_only": (_gather_to_owner_only, [(TS.test_sharded_equals_unsharded, (4, "fsdp2", "f32")),
                                                     (TS.test_zero1_toy_rs_ag_equals_half_all_reduce, ())]),
    "decay_on_new_theta": (_decay_on_new_theta, [(TS.test_adamw_weight_decay_is_decoupled_on_old_theta, ()),
                                                 (TS.test_adamw_matches_torch_optim_adamw, (10,))]),
    "clip_without_epsilon": (_clip_without_epsilon, [(TC.test_global_norm_and_coefficient_by_hand, ())]),
    "shard_first_group_only": (_shard_first_group_only,
                               [(TU.test_shard_then_unshard_gives_the_cast_of_every_element, ("hsdp", 8, 2))]),
    "ledger_zero2_as_fsdp": (_zero2_as_fsdp, [(TL.test_bytes_per_param_tables, (8,))]),
    "all_reduce_counted_once": (_all_reduce_once, [(TL.test_all_reduce_is_reduce_scatter_plus_all_gather_in_volume, ())]),
    "collectives_send_the_whole_payload": (_whole_payload, [(TL.test_qwen3_layer_comm_volume, ())]),
    "param_count_without_gqa": (_no_gqa, [(TL.test_workload_param_counts_follow_the_formula, ()),
                                          (TL.test_7b_parameter_count_and_ledger, ())]),
    "state_moved_once": (_state_moved_once, [(TL.test_algorithmic_bytes_per_element, (1, 72))]),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(monkeypatch, name):
    plant, pins = MUTANTS[name]
    assert not _fails(pins), "a pin fails on the unmodified oracle"
    plant(monkeypatch)
    assert _fails(pins), f"no pin caught the planted mistake {name!r}"
