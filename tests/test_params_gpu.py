"""Per-parameter tensors: the step reads every rank's per-parameter gradient
tensors and writes every rank's per-parameter bf16 tensors in place (FSDP2's
copy-in / copy-out folded into the step), with results bit-identical to the
step on full-size buffers holding the same values, which the other GPU tests
compare with the oracle."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
from synth_inputs import device as D

from gpu_cases import HP, PARAM_SENTINEL, STATE_SENTINEL, DeviceCase, Guarded, ensure_built, ulp_dist

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


SHAPES = ((3001, 7), (77, 3), (4099,), (1,), (12289,), (9, 5), (0, 4), (640, 64))


def _numel(s):
    n = 1
    for d in s:
        n *= d
    return n


class ParamCase:
    """The inputs of a flat DeviceCase, copied into per-parameter tensors of a
    per-parameter plan (state keyed by the logical element, like the flat case)."""

    def __init__(self, flat: DeviceCase, n_rep=1, with_params=True, param_dtype=torch.bfloat16):
        self.flat = flat
        shapes, n_d = flat.shapes, flat.n_d
        self.shapes = shapes
        self.plan = fsp.plan_layout_params(shapes, n_d, n_replicate=n_rep)
        gdt = torch.float32 if flat.grad_dtype == "f32" else torch.bfloat16
        self.flat_off = flat.plan.param_offsets
        self.grads = [[Guarded(_numel(s), gdt, 0) for s in shapes] for _ in range(n_d)]
        for q in range(n_d):
            for i, s in enumerate(shapes):
                n = _numel(s)
                self.grads[q][i].t.copy_(flat.grads[q].t[self.flat_off[i]:self.flat_off[i] + n])
        sentinel = PARAM_SENTINEL if param_dtype == torch.bfloat16 else STATE_SENTINEL
        self.params = [[Guarded(_numel(s), param_dtype, sentinel) for s in shapes] for _ in range(n_d)] \
            if with_params else None
        p = self.plan
        self.state = [Guarded(p.state_len_total, torch.float32, STATE_SENTINEL) for _ in range(3)]
        # segment (virtual full_off) -> the logical element index the flat case keys its values by
        segs = [(s.full_off - p.param_offsets[s.param] + self.flat_off[s.param], s.state_off, s.length)
                for s in p.segments]
        D.fill_state_segments(self.state[0].t, self.state[1].t, self.state[2].t, flat.seed, segs)
        self.table = fsp.ParamTable(p, [[g.t for g in row] for row in self.grads],
                                    None if self.params is None else [[x.t for x in row] for row in self.params])
        torch.cuda.synchronize()

    def step(self, t, stream=None):
        fsp.sharded_step_params(self.plan, self.table, *[s.t for s in self.state], HP, t, stream=stream)

    def state_matches_flat(self):
        """Every owned state slot equals the flat case's slot of the same (param, rank) element."""
        fl = {(s.param, s.rank): s for s in self.flat.plan.segments}
        got = [x.bits() for x in self.state]
        want = [x.bits() for x in self.flat.state]
        owned = np.zeros(self.plan.state_len_total, bool)
        for s in self.plan.segments:
            f = fl[(s.param, s.rank)]
            assert f.length == s.length
            for a, b in zip(got, want):
                assert np.array_equal(a[s.state_off:s.state_off + s.length], b[f.state_off:f.state_off + f.length])
            owned[s.state_off:s.state_off + s.length] = True
        for a in got:
            assert np.all(a[~owned] == STATE_SENTINEL)

    def params_match_flat(self):
        for q in range(self.flat.n_d):
            flat_bits = self.flat.params[q].bits()
            for i, s in enumerate(self.shapes):
                n = _numel(s)
                assert np.array_equal(self.params[q][i].bits(), flat_bits[self.flat_off[i]:self.flat_off[i] + n]), \
                    f"rank {q} param {i}"

    def guards_intact(self):
        bufs = [g for row in self.grads for g in row] + self.state
        if self.params is not None:
            bufs += [x for row in self.params for x in row]
        return all(b.guards_intact() for b in bufs)


# bulk-copy kernel meshes, then meshes that run the per-thread kernel (9, 24, HSDP 3 x 3)
CASES = [(4, "fsdp2", 1, "f32"), (8, "fsdp2", 1, "f32"), (3, "fsdp2", 1, "f32"), (6, "fsdp2", 1, "bf16"),
         (8, "hsdp", 2, "f32"), (16, "fsdp2", 1, "bf16"), (9, "fsdp2", 1, "f32"), (24, "fsdp2", 1, "bf16"),
         (9, "hsdp", 3, "f32")]


@pytest.mark.parametrize("n_d,mode,n_rep,gd", CASES)
def test_per_param_step_equals_flat_step(n_d, mode, n_rep, gd):
    flat = DeviceCase(SHAPES, n_d, mode, gd, 71, n_rep)
    pc = ParamCase(flat, n_rep)
    for t in (10, 11):
        flat.step(t, debug=False)
        pc.step(t)
    torch.cuda.synchronize()
    pc.state_matches_flat()
    pc.params_match_flat()
    for q in range(n_d):   # the gradients are only read
        for i, s in enumerate(SHAPES):
            n = _numel(s)
            assert torch.equal(pc.grads[q][i].t.view(torch.int16 if gd == "bf16" else torch.int32),
                               flat.grads[q].t[pc.flat_off[i]:pc.flat_off[i] + n].view(
                                   torch.int16 if gd == "bf16" else torch.int32))
    assert pc.guards_intact() and flat.all_guards_intact()
    assert fsp.device_error() == 0


@pytest.mark.parametrize("n_d,n_rep", [(4, 1), (8, 2)])
def test_per_param_unshard_and_reduce_only_table(n_d, n_rep):
    mode = "hsdp" if n_rep > 1 else "fsdp2"
    flat = DeviceCase(SHAPES, n_d, mode, "f32", 73, n_rep)
    full = ParamCase(flat, n_rep)
    reduce_only = ParamCase(flat, n_rep, with_params=False)
    flat.step(10, debug=False)
    full.step(10)
    reduce_only.step(10)                      # ZeRO-3: state only, parameters left sharded
    torch.cuda.synchronize()
    for a, b in zip(full.state, reduce_only.state):
        assert np.array_equal(a.bits(), b.bits())
    # unshard from reduce_only's master into full's tensors, after wiping them
    for row in full.params:
        for x in row:
            x.t.view(torch.int16).fill_(np.int16(-1))
    fsp.unshard_params(full.plan, full.table, reduce_only.state[0].t)
    torch.cuda.synchronize()
    full.params_match_flat()
    assert full.guards_intact() and reduce_only.guards_intact()
    with pytest.raises(fsp.FspError):
        fsp.unshard_params(reduce_only.plan, reduce_only.table, reduce_only.state[0].t)
    with pytest.raises(fsp.FspError):        # a table belongs to its own plan
        fsp.sharded_step_params(full.plan, reduce_only.table, *[s.t for s in full.state], HP, 11)
    assert fsp.device_error() == 0


def test_per_param_step_in_a_cuda_graph():
    flat = DeviceCase(SHAPES, 4, "fsdp2", "f32", 79)
    pc = ParamCase(flat)
    pc.step(10)                               # first use outside capture (uploads the tile table)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        pc.step(11, stream=stream)
    g.replay()
    flat.step(10, debug=False)
    flat.step(11, debug=False)
    torch.cuda.synchronize()
    pc.state_matches_flat()
    pc.params_match_flat()
    assert fsp.device_error() == 0


BIG = ((3000, 4096), (4099,), (77, 3))   # enough tiles per CTA for the in-order (counter) schedule


@pytest.mark.parametrize("n_d,mode,n_rep,gd", [(4, "fsdp2", 1, "f32"), (8, "hsdp", 2, "f32"), (16, "fsdp2", 1, "bf16")])
def test_per_param_step_equals_flat_step_on_a_large_plan(n_d, mode, n_rep, gd):
    flat = DeviceCase(BIG, n_d, mode, gd, 83, n_rep)
    pc = ParamCase(flat, n_rep)
    assert pc.plan.n_tiles >= 16 * torch.cuda.get_device_properties(0).multi_processor_count
    flat.step(10, debug=False)
    pc.step(10)
    torch.cuda.synchronize()
    pc.state_matches_flat()
    pc.params_match_flat()
    assert pc.guards_intact()
    assert fsp.device_error() == 0


@pytest.mark.parametrize("max_norm", [1e-4, 1e30])
@pytest.mark.parametrize("shapes,n_d,n_rep", [(SHAPES, 4, 1), (BIG, 4, 1), (SHAPES, 8, 2)],
                         ids=["small", "large", "hsdp_2x4"])
def test_per_param_clipped_flow_equals_flat(max_norm, shapes, n_d, n_rep):
    """The distributed-optimizer flow with clipping on per-parameter tensors:
    the write-back lands in the owner's slice of the owner's gradient tensor
    (HSDP: in every replica group), and norm, coefficient, state and
    parameters are the flat flow's."""
    flat = DeviceCase(shapes, n_d, "hsdp" if n_rep > 1 else "fsdp2", "f32", 89, n_rep)
    pc = ParamCase(flat, n_rep)
    out_f = torch.zeros(4, dtype=torch.float32, device="cuda")
    out_p = torch.zeros(4, dtype=torch.float32, device="cuda")
    fsp.sharded_step_clipped(flat.plan, [g.t for g in flat.grads], *[s.t for s in flat.state],
                             [p.t for p in flat.params], HP, 10, max_norm, out_f)
    fsp.sharded_step_clipped_params(pc.plan, pc.table, *[s.t for s in pc.state], HP, 10, max_norm, out_p)
    torch.cuda.synchronize()
    nf, cf = out_f[:2].tolist()
    n_p, c_p = out_p[:2].tolist()
    # the norm's partial sums group by tile, and the tiles differ (virtual offsets):
    # two fp64-accurate norms, each rounded to the fp32 output, at most 1 ulp apart
    assert ulp_dist(np.array([nf], np.float32).view(np.uint32), np.array([n_p], np.float32).view(np.uint32))[0] <= 1
    # in general the coefficients could be one ulp apart too (two norms that straddle a rounding
    # boundary); these fixed inputs give equal ones, so state and parameters compare bit for bit
    assert cf == c_p
    assert (cf == 1.0) == (max_norm > 1e20)
    pc.state_matches_flat()
    pc.params_match_flat()
    for q in range(flat.n_d):       # write-back: each gradient tensor equals the flat buffer's slice
        fb = flat.grads[q].bits()
        for i, s in enumerate(shapes):
            n = _numel(s)
            assert np.array_equal(pc.grads[q][i].bits(), fb[pc.flat_off[i]:pc.flat_off[i] + n]), f"rank {q} grad {i}"
    assert pc.guards_intact()
    assert fsp.device_error() == 0


def test_per_param_device_t_replayed_in_a_cuda_graph():
    """One captured per-parameter step with t in device memory, replayed twice,
    equals the flat step at t = 10 and 11."""
    flat = DeviceCase(SHAPES, 8, "fsdp2", "f32", 97)
    pc = ParamCase(flat)
    t_dev = torch.tensor([10], dtype=torch.int64, device="cuda")
    # first use of the plan outside capture, on scratch copies of the state (the
    # parameter tensors it writes are rewritten by every later step)
    scratch = [s.t.clone() for s in pc.state]
    fsp.sharded_step_params_device_t(pc.plan, pc.table, *scratch, HP, torch.ones(1, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fsp.sharded_step_params_device_t(pc.plan, pc.table, *[s.t for s in pc.state], HP, t_dev, stream=stream)
    g.replay()
    g.replay()
    flat.step(10, debug=False)
    flat.step(11, debug=False)
    torch.cuda.synchronize()
    assert int(t_dev.item()) == 12
    pc.state_matches_flat()
    pc.params_match_flat()
    assert fsp.device_error() == 0


@pytest.mark.parametrize("shapes", [SHAPES, BIG], ids=["small", "large"])
def test_per_param_writeback_equals_flat(shapes):
    flat = DeviceCase(shapes, 4, "fsdp2", "f32", 107)
    pc = ParamCase(flat)
    fsp.sharded_step_writeback(flat.plan, [g.t for g in flat.grads], *[s.t for s in flat.state],
                               [p.t for p in flat.params], HP, 10)
    fsp.sharded_step_writeback_params(pc.plan, pc.table, *[s.t for s in pc.state], HP, 10)
    torch.cuda.synchronize()
    pc.state_matches_flat()
    pc.params_match_flat()
    for q in range(flat.n_d):
        fb = flat.grads[q].bits()
        for i, s in enumerate(shapes):
            n = _numel(s)
            assert np.array_equal(pc.grads[q][i].bits(), fb[pc.flat_off[i]:pc.flat_off[i] + n]), f"rank {q} grad {i}"
    assert pc.guards_intact()
    assert fsp.device_error() == 0


@pytest.mark.parametrize("shapes,n_d,n_rep", [(SHAPES, 4, 1), (SHAPES, 8, 2), (SHAPES, 9, 1), (BIG, 4, 1)],
                         ids=["fsdp2", "hsdp", "per-thread", "large"])
def test_per_param_fp32_parameters_equal_flat_fp32_gather(shapes, n_d, n_rep):
    mode = "hsdp" if n_rep > 1 else "fsdp2"
    flat = DeviceCase(shapes, n_d, mode, "f32", 109, n_rep)
    pc = ParamCase(flat, n_rep, param_dtype=torch.float32)
    assert pc.table.param_dtype == "f32"
    fbufs = [Guarded(flat.plan.full_len_padded, torch.float32, STATE_SENTINEL) for _ in range(n_d)]
    fsp.sharded_step_fp32_gather(flat.plan, [g.t for g in flat.grads], *[s.t for s in flat.state],
                                 [b.t for b in fbufs], HP, 10)
    pc.step(10)
    torch.cuda.synchronize()
    pc.state_matches_flat()
    for q in range(n_d):
        fb = fbufs[q].bits()
        for i, s in enumerate(shapes):
            n = _numel(s)
            assert np.array_equal(pc.params[q][i].bits(), fb[pc.flat_off[i]:pc.flat_off[i] + n]), f"rank {q} param {i}"
    # and the fp32 unshard into the same tensors after wiping them
    for row in pc.params:
        for x in row:
            x.t.view(torch.int32).fill_(-1)
    fsp.unshard_params(pc.plan, pc.table, pc.state[0].t)
    torch.cuda.synchronize()
    for q in range(n_d):
        fb = fbufs[q].bits()
        for i, s in enumerate(shapes):
            n = _numel(s)
            assert np.array_equal(pc.params[q][i].bits(), fb[pc.flat_off[i]:pc.flat_off[i] + n])
    assert pc.guards_intact()
    assert fsp.device_error() == 0
