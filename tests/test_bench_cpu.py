"""CPU checks of the measurement side: the byte account of the workloads, the
reference arm's JSON line, and the multi-rank helpers of bench.py (max over
ranks, barrier) on world_size 2 with the gloo backend."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

import workloads
from sparse_kv_decode_gb300 import byte_account as ba

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_of_the_llama_32k_layer():
    w = workloads.WORKLOADS[2]
    dense = ba.dense_verify_bytes(w.batch, w.hq, w.hkv, w.d, w.n - 1, 1)
    sparse = ba.sparse_decode_bytes(w.batch, w.hq, w.d, w.batch * w.hkv * w.keep[0])
    assert dense == 8 * 32768 * 512 + 32 * 512              # full K/V + q in / o out
    assert round(dense / 1e6, 1) == 134.2
    assert round(sparse / 1e6, 1) == 40.6                    # 8 x 9830 rows x (512 B + int32 index)
    # the byte bound of 30% selection over dense (ByteCross ideal speedup, attention only)
    assert 3.2 < dense / sparse < 3.4


def test_keep_lengths_of_the_workloads():
    assert workloads.WORKLOADS[2].keep == (9830,)
    assert workloads.WORKLOADS[4].keep == (13107, 39321, 65536)
    w3 = workloads.WORKLOADS[3]
    assert w3.frames * w3.frame_tokens + w3.text_tokens == w3.n == 12800


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny", "--steps", "2", "--warmup", "0"], capture_output=True, text=True, env=env,
                       timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference"
    assert rec["unit"] == "us/step" and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["warmup"] >= 3
    # whole steps are timed (the tiny workload has 4 units), so the line's time fits its own run
    assert rec["units_timed_per_step"] == rec["units_per_step"] == 4 and not rec["extrapolated"]
    assert rec["ms_per_step"] * rec["steps"] / 1e3 <= rec["run_wall_s"]
    # the same config as the GPU arm prints
    import bench
    assert rec["config"] == bench.workload_config(workloads.by_name("tiny"), 0)


def test_cpu_baseline_on_worker_processes():
    import bench
    rec = bench.cpu_baseline(workloads.by_name("tiny"), 0, timed_rounds=1)
    assert rec["kind"] == "oracle" and rec["value"] > 0
    assert rec["cores"] == min(bench.host_cores(), 4) and "worker processes" in rec["sample"]
    assert not rec["extrapolated"]


def test_cpu_baseline_falls_back_to_one_process(monkeypatch):
    import bench

    def no_workers(*args, **kwargs):
        raise RuntimeError("no workers here")

    monkeypatch.setattr(bench, "oracle_decode_rounds", no_workers)
    rec = bench.cpu_baseline(workloads.by_name("tiny"), 0, timed_rounds=1)
    assert rec["cores"] == 1 and rec["value"] > 0 and "no workers here" in rec["sample"]


def test_oracle_step_plan_samples_large_steps_evenly():
    import bench
    w = workloads.by_name("sparsemm")
    units, sampled = bench.oracle_step_plan(w, 512)
    assert sampled and len(units) == 512 and len(set(units)) == 512
    assert units[0] == (0, 0, 0) and units[-1][0] == w.layers - 1
    units, sampled = bench.oracle_step_plan(workloads.by_name("llama8b_32k"), 512)
    assert not sampled and len(units) == 32 * 8


def test_traffic_figures_only_for_their_sources_and_workload(tmp_path, monkeypatch):
    import bench
    for rel in bench.ATTN_SOURCES:
        f = tmp_path / rel
        f.parent.mkdir(parents=True, exist_ok=True)
        f.write_text("// " + rel + "\n")
    other = tmp_path / "sparse_kv_decode_gb300" / "csrc" / "other_kernel.cu"
    other.write_text("// another kernel\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash()
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# phase  bytes_per_call  csrc_hash  workload\n"
        "sparse  4.0e+07   %s   llama8b_32k\n"
        "dense   1.3e+08   0123456789abcdef   llama8b_32k\n" % h)
    assert bench.traffic_from_profiles("sparse", "llama8b_32k") == 4.0e7
    assert bench.traffic_from_profiles("sparse", "llama8b_128k") is None   # another workload
    assert bench.traffic_from_profiles("dense", "llama8b_32k") is None     # stale sources
    other.write_text("// another kernel, changed\n")                       # not an attention source
    assert bench.traffic_from_profiles("sparse", "llama8b_32k") == 4.0e7
    (tmp_path / bench.ATTN_SOURCES[0]).write_text("// attention kernel, changed\n")
    assert bench.traffic_from_profiles("sparse", "llama8b_32k") is None


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_init()
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + 5.0 * r, w)
    q.put((r, w, m))
    torch.distributed.destroy_process_group()


def test_bench_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 15.0), (1, 2, 15.0)]


def test_std_io_model_of_the_video_workload():
    # StD 3.3: I/O_sparse = gamma (K + m_t), I/O_dense = m_v + m_t, average over alpha gamma
    # accepted tokens; video workload: gamma 5, K = 768 visual, m_t = 256 text, m_v = 12 544
    assert ba.std_io_sparse(5, 768, 256) == 5 * 1024
    assert ba.std_io_dense(12544, 256) == 12800
    assert ba.std_io_total(5, 768, 256, 12544) == 17920
    # every draft accepted: 17 920 / 5 entries per token against 12 800 for vanilla decoding
    assert ba.std_io_average(5, 768, 256, 12544, 1.0) == 3584.0
    a = ba.std_alpha_threshold(5, 768, 256, 12544)
    assert abs(a - (1024 / 12800 + 0.2)) < 1e-15
    # at the threshold the average equals the vanilla per-token I/O, below it StD reads more
    assert abs(ba.std_io_average(5, 768, 256, 12544, a) - 12800) < 1e-9
    assert ba.std_io_average(5, 768, 256, 12544, 0.9 * a) > 12800


def test_sd_speedup_model():
    # SpecVLM: Speedup = tau / (gamma T_d/T_t + T_t^gamma/T_t); a free draft and a verify as
    # cheap as one decode give the accept length itself
    assert ba.sd_speedup(3.0, 4, 0.0, 1.0) == 3.0
    assert abs(ba.sd_speedup(4.0, 4, 0.25, 1.0) - 2.0) < 1e-15
