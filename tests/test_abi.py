"""C-ABI library on the host: loads, exports what include/fsp.h declares, plans
bit-exactly like the oracle, and rejects bad arguments before any launch."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import fsdp_sharded_mixed_pass_gb300 as fsp
from fsdp_sharded_mixed_pass_gb300 import fsp as B
from oracle import ledger as OL
from oracle import plan as OP
from synth_inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HP = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


@pytest.fixture(scope="module", autouse=True)
def built():
    if not os.path.exists(B.LIB_PATH):
        from fsdp_sharded_mixed_pass_gb300 import build
        build.build()
    return B.lib()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fsp_\w+)\s*\(", text))
    return names


def test_header_declares_exactly_the_binding_exports():
    assert _declared() == set(fsp.EXPORTS)


def test_library_exports_every_declared_symbol():
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\b[TW] (fsp_\w+)$", out, flags=re.M))
    missing = _declared() - exported
    assert not missing, missing
    for name in _declared():
        assert getattr(B.lib(), name) is not None


def _compare_plans(lib_plan, o):
    assert lib_plan.n_d == o.n_d
    assert lib_plan.valid_elems == o.valid_elems
    assert lib_plan.full_len_padded == o.full_len_padded
    assert lib_plan.state_len_per_rank == o.state_len_per_rank
    assert lib_plan.state_len_total == o.state_len_total
    # the library lists segments rank-major (its state order); the oracle by parameter
    got = [(s.rank, s.param, s.full_off, s.state_off, s.length, s.padded_len) for s in lib_plan.segments]
    want = sorted((s.rank, s.param, s.full_off, s.state_off, s.length, s.padded_len) for s in o.segments)
    assert got == want
    # tiles: one per started 4096-block of each non-empty segment of one replica
    tiles = 0
    for s in o.segments:
        if s.length and s.rank < o.n_shard:
            tiles += (s.full_off + s.length - 1) // 4096 - s.full_off // 4096 + 1
    assert lib_plan.n_tiles == tiles


@pytest.mark.parametrize("w", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_planner_matches_oracle_on_workloads(w):
    lib_plan = fsp.plan_layout(w.shapes, w.n_d, w.mode, n_replicate=w.n_rep)
    _compare_plans(lib_plan, OP.plan_layout(w.shapes, w.n_d, w.mode, n_rep=w.n_rep))
    assert (lib_plan.n_replicate, lib_plan.n_shard) == (w.n_rep, w.n_d // w.n_rep)


@pytest.mark.parametrize("n_rep,n_shard", [(1, 1), (1, 5), (2, 1), (2, 2), (2, 3), (4, 4), (3, 7), (8, 8), (16, 4)])
def test_hsdp_planner_matches_oracle(n_rep, n_shard):
    rng = np.random.default_rng(n_rep * 100 + n_shard)
    shapes = [(int(rng.integers(0, 3 * n_shard + 5)), int(rng.choice([1, 3, 64]))) for _ in range(int(rng.integers(0, 25)))]
    _compare_plans(fsp.plan_layout(shapes, n_rep * n_shard, "hsdp", n_replicate=n_rep),
                   OP.plan_layout(shapes, n_rep * n_shard, "hsdp", n_rep=n_rep))


@pytest.mark.parametrize("mode", ["fsdp2", "distopt"])
@pytest.mark.parametrize("n_d", [1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 33, 64])
def test_planner_matches_oracle_on_random_shapes(mode, n_d):
    rng = np.random.default_rng(n_d * 31 + len(mode))
    shapes = []
    for _ in range(int(rng.integers(0, 40))):
        nd = int(rng.integers(1, 4))
        shape = [int(rng.integers(0, 3 * n_d + 5))] + [int(rng.choice([1, 2, 3, 7, 64])) for _ in range(nd - 1)]
        shapes.append(tuple(shape))
    _compare_plans(fsp.plan_layout(shapes, n_d, mode), OP.plan_layout(shapes, n_d, mode))


def test_empty_plan():
    p = fsp.plan_layout([], 4, "fsdp2")
    assert (p.valid_elems, p.state_len_total, p.n_segments, p.n_tiles) == (0, 0, 0, 0)
    p = fsp.plan_layout([], 4, "distopt")
    assert (p.valid_elems, p.full_len_padded, p.n_tiles) == (0, 0, 0)


@pytest.mark.parametrize("w", WORKLOADS, ids=[w.name for w in WORKLOADS])
def test_ledger_matches_oracle(w):
    led = fsp.plan_layout(w.shapes, w.n_d, w.mode, n_replicate=w.n_rep).ledger(w.grad_dtype)
    P, n, g, nr = w.numel, w.n_d, w.grad_bytes, w.n_rep
    ns = n // nr
    sent = OL.hsdp_step_sent(nr, ns, g * P, 2 * P)
    want = {
        "resident_ddp": OL.resident_bytes("ddp", P, n, g),
        "resident_distopt": OL.resident_bytes("distopt", P, n, g),
        "resident_zero2": OL.resident_bytes("zero2", P, n, g),
        "resident_fsdp": OL.resident_bytes("fsdp", P, n, g),
        "reduce_scatter_sent": sent["reduce_scatter"],
        "all_gather_sent": sent["all_gather"],
        "step_hbm_bytes": OL.sharded_step_bytes(n, g, nr) * P,
        "resident_hsdp": OL.hsdp_bytes_per_param(ns, g) * P,
        "cross_group_all_reduce_sent": sent["cross_group_all_reduce"],
    }
    for k, v in want.items():
        assert led[k] == pytest.approx(float(v), rel=1e-12), k


# ---- argument errors, all detected on the host before any CUDA call ----------

def _raw_layout(dims, ndims, n_params, n_d, mode):
    L = B.lib()
    out = ctypes.c_void_p()
    d = (ctypes.c_int64 * max(1, len(dims)))(*dims)
    nd = (ctypes.c_int32 * max(1, len(ndims)))(*ndims)
    st = L.fsp_plan_layout(d, nd, n_params, n_d, mode, ctypes.byref(out))
    if out.value:
        L.fsp_plan_destroy(out)
    return st


def test_hsdp_layout_rejects():
    L = B.lib()
    d = (ctypes.c_int64 * 1)(4)
    nd = (ctypes.c_int32 * 1)(1)
    out = ctypes.c_void_p()
    for nr, ns in ((0, 4), (2, 0), (8, 9), (-1, 2)):
        assert L.fsp_plan_layout_hsdp(d, nd, 1, nr, ns, ctypes.byref(out)) == B.FSP_EINVAL
    assert L.fsp_plan_layout_hsdp(d, nd, 1, 2, 2, None) == B.FSP_EINVAL


@pytest.mark.parametrize("dims,ndims,n_params,n_d,mode", [
    ([4], [1], 1, 0, 0),        # n_d < 1
    ([4], [1], 1, 65, 0),       # n_d > 64
    ([4], [1], 1, 2, 7),        # unknown mode
    ([-1], [1], 1, 2, 0),       # negative dim
    ([4], [0], 1, 2, 0),        # ndims < 1
    ([4] * 9, [9], 1, 2, 0),    # ndims > 8
    ([4], [1], -1, 2, 0),       # n_params < 0
    ([1 << 40, 1 << 20], [2], 1, 2, 0),   # too many elements
])
def test_plan_layout_rejects(dims, ndims, n_params, n_d, mode):
    assert _raw_layout(dims, ndims, n_params, n_d, mode) == B.FSP_EINVAL
    assert B.lib().fsp_last_error().decode() != ""


def test_plan_layout_null_out():
    L = B.lib()
    d = (ctypes.c_int64 * 1)(4)
    nd = (ctypes.c_int32 * 1)(1)
    assert L.fsp_plan_layout(d, nd, 1, 2, 0, None) == B.FSP_EINVAL


def test_segment_index_out_of_range():
    p = fsp.plan_layout([(8,)], 2)
    seg = B._Segment()
    assert B.lib().fsp_plan_segment(p.handle, 2, ctypes.byref(seg)) == B.FSP_EINVAL
    assert B.lib().fsp_plan_segment(p.handle, -1, ctypes.byref(seg)) == B.FSP_EINVAL


class _Fake:
    """A stand-in buffer with a chosen address; never dereferenced."""

    def __init__(self, addr):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def _fakes(plan, base=1 << 40, align=0):
    gstride = plan.full_len_padded * 4 + 4096
    grads = [_Fake(base + q * gstride + align) for q in range(plan.n_d)]
    pbase = base + plan.n_d * gstride
    params = [_Fake(pbase + q * gstride) for q in range(plan.n_d)]
    sbase = pbase + plan.n_d * gstride
    sstride = plan.state_len_total * 4 + 4096
    return grads, [_Fake(sbase + i * sstride) for i in range(3)], params


def _step_status(plan, grads, state, params, hp=HP, step=1, dtype="f32"):
    try:
        fsp.sharded_step(plan, grads, *state, params, hp, step, stream=0, grad_dtype=dtype)
    except fsp.FspError as e:
        return e.status, str(e)
    return B.FSP_OK, ""


def test_step_rejects_bad_arguments_on_host():
    plan = fsp.plan_layout([(64, 8)], 4)
    grads, state, params = _fakes(plan)
    assert _step_status(plan, grads, state, params, step=0)[0] == B.FSP_EINVAL
    assert _step_status(plan, grads, state, params, step=-3)[0] == B.FSP_EINVAL
    for bad in (dict(HP, beta1=1.0), dict(HP, beta2=-0.1), dict(HP, lr=-1.0), dict(HP, eps=float("nan")),
                dict(HP, weight_decay=float("inf"))):
        assert _step_status(plan, grads, state, params, hp=bad)[0] == B.FSP_EINVAL
    g2, s2, p2 = _fakes(plan, align=4)
    st, msg = _step_status(plan, g2, s2, p2)
    assert st == B.FSP_EINVAL and "aligned" in msg
    # overlapping buffers: param 1 inside grad 0
    g3, s3, p3 = _fakes(plan)
    p3[1] = _Fake(g3[0].addr + 64)
    st, msg = _step_status(plan, g3, s3, p3)
    assert st == B.FSP_EINVAL and "overlaps" in msg
    # null state pointer
    g4, s4, p4 = _fakes(plan)
    s4[1] = _Fake(0)
    assert _step_status(plan, g4, s4, p4)[0] == B.FSP_EINVAL
    g5, s5, p5 = _fakes(plan)
    p5[2] = _Fake(0)
    assert _step_status(plan, g5, s5, p5)[0] == B.FSP_EINVAL


def test_step_rejects_wrong_buffer_count_and_dtype():
    plan = fsp.plan_layout([(64, 8)], 4)
    grads, state, params = _fakes(plan)
    with pytest.raises(ValueError):
        fsp.sharded_step(plan, grads[:3], *state, params, HP, 1, stream=0, grad_dtype="f32")
    L = B.lib()
    args = B._step_args(plan, grads, *state, params, HP, 1, "f32")
    args[2] = 9   # unknown dtype
    assert L.fsp_sharded_step(*args, ctypes.c_void_p(0)) == B.FSP_EINVAL
    assert L.fsp_sharded_step(None, *args[1:], ctypes.c_void_p(0)) == B.FSP_EINVAL


def test_empty_plan_step_is_a_noop():
    plan = fsp.plan_layout([(0, 5)], 3)
    grads, state, params = _fakes(plan)
    assert _step_status(plan, grads, state, params)[0] == B.FSP_OK


def test_status_strings():
    L = B.lib()
    for s in range(5):
        assert L.fsp_status_string(s)
    assert L.fsp_status_string(99) == b"unknown status"


def test_clipped_step_rejects_on_host():
    L = B.lib()
    hsdp = fsp.plan_layout([(64, 8)], 4, "hsdp", n_replicate=2)
    fsdp = fsp.plan_layout([(64, 8)], 4)
    for plan, dtype, max_norm, want in ((hsdp, "bf16", 1.0, B.FSP_EUNSUPPORTED),
                                        (hsdp, "f32", -1.0, B.FSP_EINVAL),
                                        (fsdp, "bf16", 1.0, B.FSP_EUNSUPPORTED),
                                        (fsdp, "f32", 0.0, B.FSP_EINVAL),
                                        (fsdp, "f32", float("inf"), B.FSP_EINVAL)):
        grads, state, params = _fakes(plan)
        args = B._step_args(plan, grads, *state, params, HP, 1, dtype)
        assert L.fsp_sharded_step_clipped(*args, max_norm, ctypes.c_void_p(1 << 44), ctypes.c_void_p(0)) == want


def test_build_is_free_of_compiler_warnings():
    log = B.LIB_PATH + ".ptxas.txt"
    if not os.path.exists(log):
        pytest.skip("library built without a log")
    text = open(log).read()
    assert "warning" not in text.lower(), [l for l in text.splitlines() if "warning" in l.lower()][:5]


# ---- per-parameter plans and tensor tables ---------------------------------------

@pytest.mark.parametrize("n_rep,n_shard", [(1, 1), (1, 3), (1, 8), (2, 2), (2, 4), (1, 16)])
def test_per_param_planner_matches_oracle(n_rep, n_shard):
    rng = np.random.default_rng(n_rep * 17 + n_shard)
    shapes = [tuple([int(rng.integers(0, 3 * n_shard + 40))] + [int(rng.choice([1, 3, 7, 64]))
                                                                 for _ in range(int(rng.integers(0, 3)))])
              for _ in range(int(rng.integers(1, 30)))]
    n_d = n_rep * n_shard
    lib_plan = fsp.plan_layout_params(shapes, n_d, n_replicate=n_rep)
    o = OP.plan_layout(shapes, n_d, "hsdp" if n_rep > 1 else "fsdp2", n_rep=n_rep, param_align=16)
    _compare_plans(lib_plan, o)
    assert lib_plan.param_offsets == o.param_offsets
    assert lib_plan.param_align == 16
    assert fsp.plan_layout(shapes, n_d, "fsdp2").param_align == 1


def test_per_param_worked_example_through_the_abi():
    p = fsp.plan_layout_params([(3,), (5, 2), (17,)], 2)
    assert p.param_offsets == (0, 16, 32) and (p.valid_elems, p.full_len_padded) == (30, 49)
    assert sorted((s.param, s.rank, s.full_off, s.state_off, s.length) for s in p.segments) == [
        (0, 0, 0, 0, 2), (0, 1, 2, 50, 1), (1, 0, 16, 16, 6), (1, 1, 22, 54, 4), (2, 0, 32, 32, 9), (2, 1, 41, 73, 8)]


def test_param_table_rejects_on_host():
    L = B.lib()
    flat = fsp.plan_layout([(64, 8), (5,)], 2)
    pp = fsp.plan_layout_params([(64, 8), (5,)], 2)
    base = 1 << 40

    def ptrs(plan, shift=0, stride=1 << 20, nulls=()):
        vals = [0 if k in nulls else base + k * stride + shift for k in range(plan.n_d * plan.n_params)]
        return (ctypes.c_void_p * len(vals))(*vals)

    out = ctypes.c_void_p()
    st = L.fsp_param_table_create(flat.handle, ptrs(flat), 0, None, 1, ctypes.byref(out))
    assert st == B.FSP_EINVAL and "per-parameter" in L.fsp_last_error().decode()
    assert L.fsp_param_table_create(pp.handle, None, 0, None, 1, ctypes.byref(out)) == B.FSP_EINVAL
    assert L.fsp_param_table_create(pp.handle, ptrs(pp), 7, None, 1, ctypes.byref(out)) == B.FSP_EINVAL
    assert L.fsp_param_table_create(pp.handle, ptrs(pp, shift=4), 0, None, 1, ctypes.byref(out)) == B.FSP_EINVAL
    assert "aligned" in L.fsp_last_error().decode()
    assert L.fsp_param_table_create(pp.handle, ptrs(pp, nulls=(1,)), 0, None, 1, ctypes.byref(out)) == B.FSP_EINVAL
    # 64 x 8 fp32 = 2 KiB tensors 1 KiB apart overlap
    assert L.fsp_param_table_create(pp.handle, ptrs(pp, stride=1024), 0, None, 1, ctypes.byref(out)) == B.FSP_EINVAL
    assert "overlaps" in L.fsp_last_error().decode()
    # a param tensor on top of a grad tensor
    g = ptrs(pp)
    prm = (ctypes.c_void_p * 4)(*[g[k] for k in range(4)])
    assert L.fsp_param_table_create(pp.handle, g, 0, prm, 1, ctypes.byref(out)) == B.FSP_EINVAL
    assert L.fsp_param_table_create(pp.handle, g, 0, None, 1, None) == B.FSP_EINVAL
    assert L.fsp_param_table_create(pp.handle, g, 0, None, 5, ctypes.byref(out)) == B.FSP_EINVAL   # param dtype
    assert L.fsp_sharded_step_params(None, None, None, None, None, None, 1, None) == B.FSP_EINVAL
    assert L.fsp_unshard_params(pp.handle, None, None, None) == B.FSP_EINVAL
    L.fsp_param_table_destroy(None)


def test_per_param_layout_rejects():
    L = B.lib()
    d = (ctypes.c_int64 * 1)(4)
    nd = (ctypes.c_int32 * 1)(1)
    out = ctypes.c_void_p()
    for nr, ns in ((0, 4), (2, 0), (8, 9)):
        assert L.fsp_plan_layout_params(d, nd, 1, nr, ns, ctypes.byref(out)) == B.FSP_EINVAL
    p = fsp.plan_layout_params([(4,)], 2)
    a, b = ctypes.c_int64(), ctypes.c_int64()
    assert L.fsp_plan_param(p.handle, 1, ctypes.byref(a), ctypes.byref(b)) == B.FSP_EINVAL
    assert L.fsp_plan_param(p.handle, 0, ctypes.byref(a), ctypes.byref(b)) == B.FSP_OK and (a.value, b.value) == (0, 4)


def test_writeback_step_rejects_on_host():
    L = B.lib()
    hsdp = fsp.plan_layout([(64, 8)], 4, "hsdp", n_replicate=2)
    fsdp = fsp.plan_layout([(64, 8)], 4)
    for plan, dtype in ((hsdp, "f32"), (fsdp, "bf16")):
        grads, state, params = _fakes(plan)
        args = B._step_args(plan, grads, *state, params, HP, 1, dtype)
        assert L.fsp_sharded_step_writeback(*args, ctypes.c_void_p(0)) == B.FSP_EUNSUPPORTED
    grads, state, params = _fakes(fsdp)
    args = B._step_args(fsdp, grads, *state, params, HP, 0, "f32")
    assert L.fsp_sharded_step_writeback(*args, ctypes.c_void_p(0)) == B.FSP_EINVAL


def test_fp32_gather_checks_fp32_buffer_sizes_on_host():
    L = B.lib()
    plan = fsp.plan_layout([(64, 8)], 4)
    grads, state, params = _fakes(plan)
    args = B._step_args(plan, grads, *state, params, HP, 1, "f32")
    args[6] = None            # param_bufs NULL is not allowed here
    assert L.fsp_sharded_step_fp32_gather(*args, ctypes.c_void_p(0)) == B.FSP_EINVAL
    # fp32 buffers are twice the bf16 size: adjacent fakes laid out for bf16 now overlap
    g, s, p = _fakes(plan)
    p = [_Fake(p[0].addr + q * plan.full_len_padded * 2) for q in range(plan.n_d)]
    args = B._step_args(plan, g, *s, p, HP, 1, "f32")
    assert L.fsp_sharded_step_fp32_gather(*args, ctypes.c_void_p(0)) == B.FSP_EINVAL
    assert "overlaps" in L.fsp_last_error().decode()


def test_param_table_wrapper_checks_counts():
    pp = fsp.plan_layout_params([(64, 8), (5,)], 2)
    one = [_Fake(1 << 40), _Fake((1 << 40) + 4096)]
    with pytest.raises(ValueError):
        fsp.ParamTable(pp, [one], grad_dtype="f32")                       # one rank of two
    with pytest.raises(ValueError):
        fsp.ParamTable(pp, [one, one[:1]], grad_dtype="f32")              # a missing tensor
    with pytest.raises(ValueError):
        fsp.ParamTable(pp, [one, one], params=[one], grad_dtype="f32", param_dtype="bf16")


def test_noalloc_step_checks_like_the_step_on_host():
    """The no-allocation entry runs fsp_sharded_step's host checks: the same
    statuses and the same named messages, before any device call."""
    L = B.lib()
    plan = fsp.plan_layout([(64, 8)], 4)
    g, s, p = _fakes(plan)
    p = [_Fake(p[0].addr + q * 512) for q in range(plan.n_d)]        # param_bufs[0] overlaps param_bufs[1]
    for fn in (L.fsp_sharded_step, L.fsp_sharded_step_noalloc):
        args = B._step_args(plan, g, *s, p, HP, 1, "f32")
        assert fn(*args, ctypes.c_void_p(0)) == B.FSP_EINVAL
        assert L.fsp_last_error().decode() == "param_bufs[0] overlaps param_bufs[1]"
        args = B._step_args(plan, g, *s, p, HP, 0, "f32")
        assert fn(*args, ctypes.c_void_p(0)) == B.FSP_EINVAL
        assert "step must be >= 1" in L.fsp_last_error().decode()


@pytest.mark.parametrize("shapes,n_d,mode,n_rep", [
    (None, 4, "fsdp2", 1),                                            # the one-layer Qwen3 workload
    (((3001, 7), (5, 4099), (1,), (12289,), (777, 64)), 6, "fsdp2", 1),
    (((4097,), (64, 129), (2, 3, 5)), 3, "distopt", 1),
    (((9,), (1,), (3,), (8193, 2)), 8, "hsdp", 2),
])
def test_work_tiles_cover_the_owned_elements_once(shapes, n_d, mode, n_rep):
    """The kernels' work tiles, against the oracle planner: every owned element
    of replica group 0 exactly once, at the oracle's state slot, with its
    owner; tiles in full-index order, none crossing a multiple of 4096."""
    import numpy as np
    from oracle import plan as OP
    from synth_inputs import workload
    shapes = shapes or workload(0).shapes
    plan = fsp.plan_layout(shapes, n_d, mode, n_replicate=n_rep)
    tiles = plan.tiles()
    assert len(tiles) == plan.n_tiles
    op = OP.plan_layout(shapes, n_d, mode, n_rep=n_rep)
    fi, si = OP.owned_indices(op)
    want = {}
    for seg in op.segments:
        if seg.rank < n_d // n_rep:                     # replica group 0 (HSDP); every rank otherwise
            for x in range(seg.length):
                want[seg.full_off + x] = (seg.state_off + x, seg.rank)
    got = {}
    prev_end = -1
    for fb, sb, ln, r, pm in tiles:
        assert ln > 0 and fb >= prev_end and fb // 4096 == (fb + ln - 1) // 4096
        prev_end = fb + ln
        for x in range(ln):
            assert fb + x not in got
            got[fb + x] = (sb + x, r)
    assert got == want
    assert set(want) <= set(fi.tolist())


def test_plan_tiles_checks_its_arguments():
    L = B.lib()
    plan = fsp.plan_layout([(4099,)], 2)
    n = ctypes.c_int64()
    assert L.fsp_plan_tiles(None, 0, None, 0, ctypes.byref(n)) == B.FSP_EINVAL
    assert L.fsp_plan_tiles(plan.handle, 0, None, 0, None) == B.FSP_EINVAL
    assert L.fsp_plan_tiles(plan.handle, 0, None, 1, ctypes.byref(n)) == B.FSP_EINVAL      # cap > 0 needs out
    assert L.fsp_plan_tiles(plan.handle, 0, None, -1, ctypes.byref(n)) == B.FSP_EINVAL
    for unit in (-8, 12, 24):                                                              # not 8k dividing 4096
        assert L.fsp_plan_tiles(plan.handle, unit, None, 0, ctypes.byref(n)) == B.FSP_EINVAL
    assert L.fsp_plan_tiles(plan.handle, 0, None, 0, ctypes.byref(n)) == B.FSP_OK and n.value == plan.n_tiles
    buf = (B._Tile * 1)()                                                             # a short buffer: the first tiles only
    assert L.fsp_plan_tiles(plan.handle, 0, buf, 1, ctypes.byref(n)) == B.FSP_OK and n.value == plan.n_tiles
    first = plan.tiles()[0]
    assert (buf[0].full_begin, buf[0].state_begin, buf[0].len) == first[:3]
    # the round order: same conventions, grid >= 1
    assert L.fsp_plan_round_order(None, 152, None, 0, ctypes.byref(n)) == B.FSP_EINVAL
    assert L.fsp_plan_round_order(plan.handle, 152, None, 0, None) == B.FSP_EINVAL
    assert L.fsp_plan_round_order(plan.handle, 152, None, 1, ctypes.byref(n)) == B.FSP_EINVAL
    for grid in (0, -1):
        assert L.fsp_plan_round_order(plan.handle, grid, None, 0, ctypes.byref(n)) == B.FSP_EINVAL
    assert L.fsp_plan_round_order(plan.handle, 1, None, 0, ctypes.byref(n)) == B.FSP_OK and n.value == plan.n_tiles
    assert L.fsp_plan_round_order(plan.handle, 2 ** 31 - 1, None, 0, ctypes.byref(n)) == B.FSP_OK   # one round
    empty = fsp.plan_layout([], 2)
    assert L.fsp_plan_round_order(empty.handle, 152, None, 0, ctypes.byref(n)) == B.FSP_OK and n.value == 0


def _busiest_cta_chunks(tiles, grid):
    """Most 1024-element chunks (a partial one counting as one) any CTA takes
    when CTA b takes entries b, b + grid, ... of `tiles`."""
    load = [0] * grid
    for i, t in enumerate(tiles):
        load[i % grid] += -(-t[2] // 1024)
    return max(load)


@pytest.mark.parametrize("n_d,mode,grid", [(4, "fsdp2", 152), (8, "fsdp2", 152), (2, "fsdp2", 152),
                                           (4, "distopt", 152), (6, "fsdp2", 100), (4, "fsdp2", 7),
                                           (4, "fsdp2", 1), (4, "fsdp2", 5000)])
def test_round_order_balances_the_stride(n_d, mode, grid):
    """The order small plans are strided over: each round of `grid` entries
    holds exactly the plan's tiles of that round (so the CTAs' window of the
    buffers is the plan order's), and the busiest CTA's chunk count is below
    the plain stride's, or the plan's own order is returned.  On the one-layer
    Qwen3 workload (N_d = 4, 152 CTAs) the busiest CTA goes from 20 chunks to
    17 against a mean of 15.4."""
    from synth_inputs import workload
    plan = fsp.plan_layout(workload(0).shapes, n_d, mode)
    base = plan.tiles(0)
    order = plan.round_order(grid)
    assert len(order) == len(base)
    for k in range(0, len(base), grid):
        assert sorted(order[k:k + grid]) == sorted(base[k:k + grid])
    b, o = _busiest_cta_chunks(base, grid), _busiest_cta_chunks(order, grid)
    assert o < b or order == base
    if (n_d, mode, grid) == (4, "fsdp2", 152):
        assert (o, b) == (17, 20)
    if grid == 1 or grid >= len(base):      # one CTA, or one partial round: nothing to balance
        assert order == base


def test_round_order_on_random_plans():
    """Random ragged plans and grids: the round order is a permutation of the
    plan's tiles within every round (so the last, partial round only ever
    holds the plan's last tiles, at CTAs 0 .. n - 1), and never leaves a CTA
    busier than the plain stride does."""
    rng = np.random.default_rng(20261202)
    for _ in range(40):
        n_d = int(rng.integers(1, 17))
        shapes = [(int(rng.integers(1, 9000)),) if rng.random() < 0.4 else
                  (int(rng.integers(1, 3000)), int(rng.integers(1, 700))) for _ in range(int(rng.integers(1, 30)))]
        plan = fsp.plan_layout(shapes, n_d, "fsdp2" if rng.random() < 0.7 else "distopt")
        base = plan.tiles(0)
        grid = int(rng.integers(1, max(2, len(base))))
        order = plan.round_order(grid)
        for k in range(0, len(base), grid):
            assert sorted(order[k:k + grid]) == sorted(base[k:k + grid])
        assert _busiest_cta_chunks(order, grid) <= _busiest_cta_chunks(base, grid)


@pytest.mark.parametrize("shapes,n_d,mode,unit", [
    (None, 4, "fsdp2", 2048),                                         # the one-layer Qwen3 workload
    (((3001, 7), (5, 4099), (1,), (12289,), (777, 64)), 6, "fsdp2", 2048),
    (((4097,), (64, 129), (2, 3, 5)), 3, "distopt", 1024),
    (((9,), (1,), (3,)), 2, "fsdp2", 8),
])
def test_step_tiles_split_the_plan_tiles(shapes, n_d, mode, unit):
    """The step kernels' schedule on full-size buffers: the plan's tiles split
    at multiples of `unit` of the full index, in the same order, every element
    exactly once with the same owner, parameter and state offset."""
    from synth_inputs import workload
    shapes = shapes or workload(0).shapes
    plan = fsp.plan_layout(shapes, n_d, mode)
    base = plan.tiles(0)
    cut = plan.tiles(unit)
    assert len(cut) >= len(base)
    it = iter(cut)
    for fb, sb, ln, r, pm in base:
        f = fb
        while f < fb + ln:
            cf, cs, cl, cr, cp = next(it)
            assert (cf, cs, cr, cp) == (f, sb + (f - fb), r, pm)
            assert 0 < cl <= unit and cf // unit == (cf + cl - 1) // unit     # inside one unit
            assert cf + cl == fb + ln or (cf + cl) % unit == 0                 # cut only at unit multiples
            f += cl
        assert f == fb + ln
    assert next(it, None) is None
