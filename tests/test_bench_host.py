"""bench.py's host logic on CPU: the gloo control plane of the replica path
(world size 2), the reference arm's JSON line, and the clock check."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    d = bench.Dist(world)
    d.barrier()
    m = d.max(10.0 * rank + 0.5)
    d.barrier()
    d.close()
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(f"{d.rank} {d.world} {m}")


def test_replica_control_plane_two_ranks(tmp_path):
    mp.start_processes(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, start_method="spawn")
    got = sorted(open(tmp_path / f"r{r}.txt").read().split() for r in range(2))
    assert got == [["0", "2", "10.5"], ["1", "2", "10.5"]]


def test_single_process_dist_is_a_noop():
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    d = bench.Dist(1)
    d.barrier()
    assert (d.rank, d.world, d.max(3.0)) == (0, 1, 3.0)


def _run_bench(args, env_extra=None):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True,
                          text=True, env=env, cwd=ROOT, timeout=600)


def test_reference_arm_prints_one_json_line():
    r = _run_bench(["--impl", "reference", "--workload", "0", "--param-slice", "0:4", "--steps", "2",
                    "--warmup", "1"])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["value"] > 0 and line["unit"] == "params/s"
    # the workload's own config, as the GPU arm reports it; the timed sample beside it
    w, shapes, label = bench.resolve_workload("0", "0:4", None)
    full_p = sum(bench.math.prod(sh) for sh in shapes)
    flush = 2 * bench.L2_BYTES
    assert line["config"] == bench.step_config(w, label, type("P", (), {"valid_elems": full_p}), flush)
    assert line["ms_per_step"] == pytest.approx(full_p / line["value"] * 1e3)
    assert line["sample"]["params_per_step"] > 0 and line["sample"]["ms_per_step"] > 0


def test_reference_arm_other_ranks_print_nothing():
    r = _run_bench(["--impl", "reference", "--workload", "0", "--steps", "1", "--warmup", "0"],
                   {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_fsp_arm_fails_loudly_without_a_gpu():
    r = _run_bench(["--workload", "0", "--steps", "1", "--warmup", "0"])
    assert r.returncode != 0


@pytest.mark.parametrize("clocks,bad", [
    ({"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": []}, False),
    ({"sm_mhz": 1900, "sm_max_mhz": 2070, "reasons": ["sw_power_cap"]}, False),
    ({"sm_mhz": 1500, "sm_max_mhz": 2070, "reasons": ["hw_slowdown"]}, True),
    ({"sm_mhz": 1500, "sm_max_mhz": 2070, "reasons": ["sw_thermal_slowdown"]}, True),
    ({"sm_mhz": 600, "sm_max_mhz": 2070, "reasons": []}, True),
    ({"error": "no nvidia-smi"}, False),
])
def test_clock_rejection_rule(clocks, bad):
    assert bench.clocks_bad(clocks) == bad


def test_cpu_sample_cuts_oversized_params_into_row_blocks():
    from synth_inputs import workload
    shapes, n = bench.cpu_sample_shapes(workload(1).shapes)
    # the 151936 x 1024 embedding comes first: blocks of 15625 whole rows (16,000,000 elements)
    assert shapes == ((15625, 1024),) and n == 16_000_000


def test_rank_count_override_and_param_slice():
    w, shapes, label = bench.resolve_workload("qwen3_0p6b_fsdp2", "1:45", 24)
    assert w.n_d == 24 and w.mode == "fsdp2" and len(shapes) == 44
    assert label == "qwen3_0p6b_fsdp2@N_d=24[1:45]"
    w, _, label = bench.resolve_workload("5", None, 6)          # HSDP: 2 groups of 3
    assert (w.n_d, w.n_rep, label) == (6, 2, "qwen3_0p6b_hsdp_2x4@N_d=6")
    w, _, label = bench.resolve_workload("1", None, 8)          # its own N_d: unchanged
    assert label == "qwen3_0p6b_fsdp2"
    for bad in (7, 0, 65):
        with pytest.raises(SystemExit):
            bench.resolve_workload("5" if bad == 7 else "1", None, bad)


def test_param_runs_keep_the_params_in_order():
    from synth_inputs import workload
    shapes = workload(1).shapes
    runs = bench._param_runs(shapes, 4_000_000)
    flat = [s for r, _ in runs for s in r]
    # every param in order, an oversized one as consecutive blocks of its rows
    it = iter(flat)
    for s in shapes:
        rows = 0
        while rows < s[0]:
            piece = next(it)
            assert piece[1:] == s[1:]
            rows += piece[0]
        assert rows == s[0]
    assert next(it, None) is None
    assert sum(n for _, n in runs) == workload(1).numel
    for r, n in runs:
        assert n == sum(bench.math.prod(s) for s in r)
        assert n <= 4_000_000 or len(r) == 1
    assert bench.cpu_sample_shapes(shapes, 4_000_000) == runs[0]
    # fewer runs than cores: reused from the start; more: spread over the workload
    assert bench.cpu_sample_runs(shapes, 4_000_000, len(runs) + 2)[-2:] == [runs[0][0], runs[1][0]]
    spread = bench.cpu_sample_runs(shapes, 4_000_000, 4)
    assert spread == [runs[k * len(runs) // 4][0] for k in range(4)]
    assert spread[0][0] == (3906, 1024) and spread[-1] != spread[0]   # embedding rows and later layers


def test_oracle_pool_times_every_process():
    w, shapes, _ = bench.resolve_workload("0", "0:4", None)
    done, secs, sizes = bench.time_oracle_pool(w, shapes, 2, 1_000_000, warmup=1, steps=3)
    assert len(sizes) == 2 and done == 3 * sum(sizes) and secs > 0
    assert sizes[0] == sum(bench.math.prod(s) for s in bench.cpu_sample_runs(shapes, 1_000_000, 1)[0])


def test_oracle_pool_reports_a_failing_process():
    import dataclasses
    w, shapes, _ = bench.resolve_workload("0", "0:2", None)
    with pytest.raises(RuntimeError, match="oracle pool"):
        bench.time_oracle_pool(dataclasses.replace(w, grad_dtype="f8"), shapes, 2, 1_000_000, steps=1,
                               limit_s=300)


def test_pool_size_respects_host_memory(monkeypatch):
    w, _, _ = bench.resolve_workload("1", None, None)
    monkeypatch.setattr(bench, "host_cores", lambda: 16)
    monkeypatch.setattr(bench, "host_memory_available", lambda: 0)
    assert bench.pool_size(w, 4_000_000) == 16
    per = 4_000_000 * (8 * 6 + 12 + 160)
    monkeypatch.setattr(bench, "host_memory_available", lambda: 6 * per)
    assert bench.pool_size(w, 4_000_000) == 3
    monkeypatch.setattr(bench, "host_memory_available", lambda: per)
    assert bench.pool_size(w, 4_000_000) == 1


def test_traffic_record_matches_the_current_kernel_source():
    """The committed ncu traffic record is found and still belongs to the
    step kernel's current source (else the bench line reports traffic null)."""
    from synth_inputs import workload
    assert os.path.exists(bench.TRAFFIC_FILE)
    for name in ("qwen3_0p6b_fsdp2", "ragged_500", "dense_1p5b_bf16grad", "qwen3_0p6b_hsdp_2x4"):
        w = workload(name)
        algorithmic = w.n_d * w.grad_bytes + 24 * w.n_rep + 2 * w.n_d
        tpe = bench.traffic_per_elem(name)
        assert tpe is not None and 0.95 < tpe / algorithmic < 1.05, name
    # the headline workload's figure is a capture of its whole launch
    P = 596049920
    assert bench.traffic_basis("qwen3_0p6b_fsdp2", P).endswith(f"of this size ({P} elements)")
    assert "scaled to" in bench.traffic_basis("ragged_500", 1407887633)


def test_roofline_kernel_label_follows_the_mesh():
    for name, n_d, want in (("1", None, "sharded_step_kernel"), ("1", 9, "sharded_step_generic_kernel"),
                            ("5", None, "sharded_step_kernel"), ("5", 6, "sharded_step_generic_kernel"),
                            ("4", None, "sharded_step_kernel"), ("1", 24, "sharded_step_generic_kernel")):
        w, _, _ = bench.resolve_workload(name, None, n_d)
        assert bench.step_kernel_name(w) == want, (name, n_d)


def test_bulk_mesh_set_mirrors_the_library_table():
    import re
    src = open(os.path.join(ROOT, "fsdp_sharded_mixed_pass_gb300", "csrc", "fsp_step.cu")).read()
    decl = re.search(r"using Kernels = KernelTable<GradT,(.*?)>;", src, re.S).group(1)
    meshes = {(int(a), int(b)) for a, b in re.findall(r"Mesh<(\d+),\s*(\d+)>", decl)}
    assert meshes == set(bench.BULK_MESHES)
