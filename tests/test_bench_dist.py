"""The benchmark's multi-process host logic on CPU: two gloo ranks, max of
the per-rank times and sum of the per-rank work (no GPU, no data path)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        bench.barrier(world)
        ms, units = bench.aggregate(10.0 + rank * 5.0, 100.0 * (rank + 1), world)
        q.put((rank, ms, units))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, units in got:
        assert ms == 15.0          # slowest rank's time
        assert units == 300.0      # work of all ranks


def test_single_process_identity():
    assert bench.aggregate(3.5, 7.0, 1) == (3.5, 7.0)


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        steps, warmup, ref_rows = 1, 0, 8
    w = bench.WORKLOADS["b8h32n512d64_bf16"]
    assert bench.run_reference(A, w, 2, 1) is None
    line = bench.run_reference(A, w, 2, 0)
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_kernel_hash_is_stable():
    assert bench.kernel_source_hash() == bench.kernel_source_hash()
    assert len(bench.kernel_source_hash()) == 16


def test_code_digest_ignores_comments_only():
    src = "int f(int x) {\n  return x + 1;   // one more\n}\n"
    assert bench.code_digest([src]) == bench.code_digest(
        ["// header\nint f(int x) {\n\n  return x + 1;   // one more, reworded\n}\n"])
    assert bench.code_digest([src]) != bench.code_digest([src.replace("x + 1", "x + 2")])
    assert bench.code_digest([src, ""]) != bench.code_digest(["", src + "int g;"])


def test_reference_cli_prints_one_contract_line():
    # the whole command line, as the harness launches it: one JSON line on
    # stdout with the contract's keys (the reference arm runs on CPU)
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--workload", "b8h32n512d64_bf16", "--steps", "1", "--warmup", "0"],
                         cwd=root, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "b8h32n512d64_bf16"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_clock_summary_reads_reasons_and_loaded_clock(tmp_path):
    # nvidia-smi rows as the sampler writes them (csv, noheader, nounits):
    # index, sm MHz, max sm MHz, power W, active mask, then four reasons
    rows = ["0, 1980, 2070, 120.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 2055, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2040, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 980.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "garbage line"]
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(rows) + "\n")
    s = bench.ClockSampler(0)
    s.proc, s.path = object(), str(path)
    out = s.summary()
    assert out["reasons"] == ["sw_power_cap"]
    assert out["sm_max_mhz"] == 2070.0 and out["samples"] == 4
    # median over the samples drawing at least half the peak power (the idle
    # 120 W sample is left out)
    assert out["sm_mhz"] == 2055.0 and out["power_w_max"] == 980.0
    assert not path.exists()          # the sampler's file is removed once read


def test_clock_summary_flags_throttling_and_missing_samples(tmp_path):
    path = tmp_path / "clocks.csv"
    path.write_text("0, 1500, 2070, 800.0, 0x8, Active, Not Active, Active, Not Active\n")
    s = bench.ClockSampler(0)
    s.proc, s.path = object(), str(path)
    assert s.summary()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    empty = bench.ClockSampler(0)
    assert empty.summary()["reasons"] == ["unsampled"]


def test_l2_note_names_the_flush_rule():
    assert "no flush" in bench.l2_note(bench.WORKLOADS["b8h32n8192d64_bf16"])
    assert "> 129 MB L2" in bench.l2_note(bench.WORKLOADS["b8h32n8192d64_bf16"])
    assert "sets rotated" in bench.l2_note(bench.WORKLOADS["b8h32n512d64_fp16"])


@pytest.mark.parametrize("name", sorted(bench.WORKLOADS))
def test_input_sets_keep_every_step_out_of_l2(name):
    # between two uses of one input set more than twice the L2's bytes pass
    # (or one set alone is that large), so no timed step reads inputs the
    # previous steps left in the 129 MB L2
    w = bench.WORKLOADS[name]
    n = bench.input_sets(w)
    assert n >= 1 and n * bench.set_bytes(w) >= 2 * bench.L2_BYTES
    if bench.set_bytes(w) >= 2 * bench.L2_BYTES:
        assert n == 1
    # the headline shape needs no rotation
    assert bench.input_sets(bench.WORKLOADS["b8h32n8192d64_bf16"]) == 1
    assert bench.set_bytes(bench.WORKLOADS["b8h32n8192d64_bf16"]) == \
        bench.WORKLOADS["b8h32n8192d64_bf16"].hbm_bytes()


def test_split_plan_modes():
    w = bench.WORKLOADS["b8h32n8192d64_bf16"]
    assert bench.split_plan(w, 1, 0, "heads") == (w, 0, 256, "weak")
    g, h0, h1, sc = bench.split_plan(w, 4, 2, "heads")
    assert g.B == 32 and (h0, h1) == (512, 768) and sc == "weak"
    g, h0, h1, sc = bench.split_plan(w, 3, 2, "strong")
    assert g is w and (h0, h1) == (171, 256) and sc == "strong"
    assert bench.split_plan(w, 8, 5, "replicate") == (w, 0, 256, "weak")
    with pytest.raises(ValueError):
        bench.split_plan(w, 2, 0, "rows")


def _split_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.WORKLOADS["b8h32n8192d64_bf16"]
        for mode in ("heads", "strong"):
            g, h0, h1, _ = bench.split_plan(w, world, rank, mode)
            mine = torch.tensor([h0, h1, g.B * g.H], dtype=torch.int64)
            every = [torch.zeros(3, dtype=torch.int64) for _ in range(world)]
            dist.all_gather(every, mine)
            q.put((rank, mode, [tuple(t.tolist()) for t in every]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_the_timed_problems():
    # the (batch, head) ranges the two ranks of the split modes time: they
    # tile the global problems exactly once; "heads" keeps B*H per rank
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_split_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = [q.get(timeout=10) for _ in range(2 * world)]
    for rank, mode, every in got:
        total = every[0][2]
        assert every[0][0] == 0 and every[-1][1] == total
        assert all(a[1] == b[0] for a, b in zip(every, every[1:]))
        if mode == "heads":
            assert total == 2 * 256 and all(h1 - h0 == 256 for h0, h1, _ in every)
        else:
            assert total == 256 and all(h1 - h0 == 128 for h0, h1, _ in every)


@pytest.mark.parametrize("dtype,tol", [("bf16", (2e-2, 2e-3)), ("fp16", (5e-3, 5e-4))])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq,nk", [(96, 96), (40, 96)])
def test_standard_comparator_computes_attention_on_cpu(dtype, tol, causal, nq, nk):
    # the unfused comparator (materialised S in the dtype, fp32 softmax)
    # against the oracle, on CPU tensors: checks its arithmetic and its
    # bottom-right causal mask
    import numpy as np
    import oracle
    from exact_attention_39_gb300 import workloads as W
    w = W.Workload("std", 1, 2, nq, 64, dtype, causal, seed=3, Nk=nk)
    q, k, v = W.make_inputs(w)
    o = bench.standard_attention(q, k, v, causal, w.scale)
    o_ref, _ = oracle.attention_fwd(q.double().numpy(), k.double().numpy(),
                                    v.double().numpy(), w.scale, causal)
    err = np.abs(o.double().numpy() - o_ref)
    assert err.max() <= tol[0] and err.mean() <= tol[1], (err.max(), err.mean())


def test_peaks_fall_back_when_the_measured_file_is_absent(tmp_path, monkeypatch):
    import json
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1234.5}))
    peaks, src = bench.load_peaks()
    assert src == "measured" and peaks["bf16_tflops"] == 1234.5


def test_cpu_baseline_leg_counts_whole_heads():
    w = bench.WORKLOADS["tiny_b1h2n128d64_fp16"]
    secs, flops, heads, threads, one = bench.time_oracle(w, budget_s=0.0, max_heads=2,
                                                         rows_1t=16)
    # a zero budget still times one whole head, then stops
    assert heads == 1 and secs > 0 and threads >= 1 and one > 0
    assert flops == w.with_(B=1, H=1).flops()


def test_shape_option_names_the_workload():
    w = bench.parse_shape("2,32,8192,64,bf16")
    assert (w.B, w.H, w.N, w.d, w.dtype, w.causal) == (2, 32, 8192, 64, "bf16", False)
    assert w.name == "b2h32n8192d64_bf16"
    w = bench.parse_shape("1,4,1024,128,fp16,causal")
    assert w.causal and w.name == "b1h4n1024d128_fp16_causal" and w.in_mult == 0.5
    with pytest.raises(SystemExit):
        bench.parse_shape("1,2,3")
