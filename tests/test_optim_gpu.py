"""ShardedAdamW - plan, state and update index behind an optimizer-shaped
handle - against the oracle: shard full parameters, two steps, unshard."""
import numpy as np
import pytest
import torch

import fsdp_sharded_mixed_pass_gb300 as fsp
import synth_inputs as S
from oracle import plan as OP
from oracle import step as OS

from gpu_cases import HP, PARAM_ULP_BAR, ensure_built, state_errors, ulp_dist, within_tol, SCALED_BOUND

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ensure_built()


SHAPES = [(3001, 7), (12289,), (9, 5), (1,), (5, 4099)]


@pytest.mark.parametrize("mode,n_d,n_rep", [("fsdp2", 4, 1), ("distopt", 8, 1), ("hsdp", 8, 2)])
def test_sharded_adamw_matches_oracle(mode, n_d, n_rep):
    opt = fsp.ShardedAdamW(SHAPES, n_d, mode, n_replicate=n_rep, lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]),
                           eps=HP["eps"], weight_decay=HP["weight_decay"])
    plan = opt.plan
    n = opt.full_len
    idx = np.arange(n)
    full = S.master_f32(23, idx)
    grads_h = [S.grad_f32(23, q, idx) for q in range(n_d)]
    opt.load_full(torch.from_numpy(full).cuda())
    grads = [torch.from_numpy(g).cuda() for g in grads_h]
    params = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(n_d)]
    oplan = OP.plan_layout(SHAPES, n_d, mode, n_rep=n_rep)
    om = np.zeros(oplan.state_len_total, np.float32)
    OS.shard(oplan, full, om)
    o_state = [om, np.zeros_like(om), np.zeros_like(om)]
    o_params = [np.zeros(n, np.uint16) for _ in range(n_d)]
    for t in (1, 2):
        prev = [x.copy() for x in o_state]
        opt.step(grads, params)
        OS.sharded_step(oplan, grads_h, "f32", *o_state, o_params, HP, t)
    torch.cuda.synchronize()
    assert opt.t == 2
    _, si = OP.owned_indices(oplan)
    got = [x.cpu().numpy()[si] for x in (opt.master, opt.exp_avg, opt.exp_avg_sq)]
    want = [x[si] for x in o_state]
    errs = state_errors(got, want, [x[si] for x in prev])
    for g, w, e in zip(got, want, errs):
        assert within_tol(g, w).all() and (e <= SCALED_BOUND * 2 ** 24).all()
    fi, _ = OP.owned_indices(oplan)
    for q in range(n_d):
        pb = params[q].view(torch.int16).cpu().numpy().view(np.uint16)
        assert (ulp_dist(pb[fi], o_params[q][fi]) <= PARAM_ULP_BAR).all()
    # unshard of the current master reproduces the step's gathered parameters
    again = [torch.full((n,), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16) for _ in range(n_d)]
    opt.unshard(again)
    torch.cuda.synchronize()
    for q in range(n_d):
        a = again[q].view(torch.int16).cpu().numpy()
        b = params[q].view(torch.int16).cpu().numpy()
        assert np.array_equal(a[fi], b[fi])
    assert fsp.device_error() == 0


def test_capturable_steps_replay_in_a_graph_bit_for_bit():
    """capturable=True: t lives on the device; one eager step, then a captured
    step replayed twice equals three eager steps of the host-t handle."""
    kw = dict(lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"], weight_decay=HP["weight_decay"])
    eager = fsp.ShardedAdamW(SHAPES, 4, "fsdp2", **kw)
    cap = fsp.ShardedAdamW(SHAPES, 4, "fsdp2", capturable=True, **kw)
    assert cap.capturable and not eager.capturable and cap.t == 0
    n = eager.full_len
    idx = np.arange(n)
    full = torch.from_numpy(S.master_f32(31, idx)).cuda()
    grads = [torch.from_numpy(S.grad_f32(31, q, idx)).cuda() for q in range(4)]
    pe = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    pc = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    eager.load_full(full)
    cap.load_full(full)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    cap.step(grads, pc, stream=stream)                 # eager first step (t = 1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        cap.step(grads, pc, stream=stream)
    for _ in range(2):
        graph.replay()                                   # t = 2, 3
    for _ in range(3):
        eager.step(grads, pe)
    torch.cuda.synchronize()
    assert cap.t == 3 and eager.t == 3
    for a, b in zip((cap.master, cap.exp_avg, cap.exp_avg_sq), (eager.master, eager.exp_avg, eager.exp_avg_sq)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    for a, b in zip(pc, pe):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    cap.t = 0                                            # resume index, set on the device
    cap.load_full(full)
    torch.cuda.synchronize()
    assert cap.t == 0
    assert fsp.device_error() == 0


@pytest.mark.parametrize("capturable", [False, True])
@pytest.mark.parametrize("n_d,n_rep", [(4, 1), (8, 2)])
def test_optimizer_on_per_parameter_tensors_equals_the_flat_one(n_d, n_rep, capturable):
    """on_tensors: the same parameters loaded per tensor, the same gradients in
    per-parameter tensors; after two steps every parameter tensor equals the
    flat optimizer's buffer slice, bit for bit, and so does the unshard."""
    kw = dict(lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"], weight_decay=HP["weight_decay"])
    mode = "hsdp" if n_rep > 1 else "fsdp2"
    flat = fsp.ShardedAdamW(SHAPES, n_d, mode, n_replicate=n_rep, **kw)
    numel = [int(np.prod(s)) for s in SHAPES]
    offs = flat.plan.param_offsets
    n = flat.full_len
    idx = np.arange(n)
    full = torch.from_numpy(S.master_f32(41, idx)).cuda()
    gflat = [torch.from_numpy(S.grad_f32(41, q, idx)).cuda() for q in range(n_d)]
    pflat = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(n_d)]
    gt = [[gflat[q][o:o + k].clone().view(s) for o, k, s in zip(offs, numel, SHAPES)] for q in range(n_d)]
    pt = [[torch.zeros(s, dtype=torch.bfloat16, device="cuda") for s in SHAPES] for _ in range(n_d)]
    per = fsp.ShardedAdamW.on_tensors(SHAPES, n_d, gt, pt, n_replicate=n_rep, capturable=capturable, **kw)
    flat.load_params([full[o:o + k].view(s) for o, k, s in zip(offs, numel, SHAPES)])
    per.load_params([full[o:o + k].view(s) for o, k, s in zip(offs, numel, SHAPES)])
    for _ in range(2):
        flat.step(gflat, pflat)
        per.step()
    torch.cuda.synchronize()
    assert per.t == flat.t == 2
    def same():
        for q in range(n_d):
            for i, (o, k) in enumerate(zip(offs, numel)):
                assert torch.equal(pt[q][i].reshape(-1).view(torch.int16), pflat[q][o:o + k].view(torch.int16)), (q, i)
    same()
    for q in range(n_d):
        for x in pt[q]:
            x.zero_()
    per.unshard()
    torch.cuda.synchronize()
    same()
    with pytest.raises(ValueError):
        per.step(gflat, pflat)
    assert fsp.device_error() == 0
