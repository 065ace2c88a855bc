#!/usr/bin/env python
"""Benchmark of the sparse-KV decode hot path on one GB300 (or N replicas).

One step = one pass of the whole path over one batch of synthetic input:
  a1 head budgets (host)           -> per-head list lengths, copied to the device
  a2 window scoring, every layer   -> fp32 scores
  a3 top-K selection, every layer  -> per-head index lists
  a4 sparse decode, every layer    -> o over the selected rows
  a5 dense decode (split-K), every layer -> o over the full cache
Each of a2..a5 is one CUDA graph of the per-layer library calls; CUDA events
between the phases give each kernel's share of the step.

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
instead (the reference arm: a deliberately slow program, on a bounded sample).
"""
import os

# The oracle's CPU timing runs one single-threaded BLAS per worker process.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import dataclasses  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402
from sparse_kv_decode_gb300 import byte_account as ba  # noqa: E402

METRIC = "µs/decode-step and achieved HBM GB/s (% of GB300 peak), sparse vs dense attn"
UNIT = "us/step"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="sdkv", choices=["sdkv", "reference"])
    ap.add_argument("--workload", default="llama8b_32k")
    ap.add_argument("--keep-index", type=int, default=0, help="which keep ratio of the workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (small profiling cases only; reported in config)")
    ap.add_argument("--no-next", action="store_true", help="skip the timings of the next rows (f1..f4)")
    ap.add_argument("--clocks-log", default="",
                    help="file for the raw nvidia-smi samples of the timed region (default: a temporary file)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------- distributed
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, path=""):
        self.proc = None
        self.keep = bool(path)
        self.path = path or os.path.join(tempfile.gettempdir(), "sdkv_clocks_%d.csv" % os.getpid())
        try:
            os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0, t1, uuid=None):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                except Exception:
                    ts = None
                if uuid and parts[1] and uuid not in parts[1]:
                    continue
                rows.append((ts, parts))
        if not self.keep:
            os.remove(self.path)
        win = [p for ts, p in rows if ts is None or (t0 - 0.3 <= ts <= t1 + 0.3)] or [p for _, p in rows]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(p[2]) for p in win if p[2].replace(".", "").isdigit()]
        smax = [float(p[3]) for p in win if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for p in win:
            for nm, val in zip(names, p[6:10]):
                if val.strip().lower() in ("active", "1", "yes"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(win)}


# ----------------------------------------------------------------------------- the path
class Path:
    """Device buffers and CUDA graphs of one step of the whole hot path."""

    PHASES = ("score", "select", "sparse", "dense")

    def __init__(self, w, keep_index, dev):
        import sparse_kv_decode_gb300 as sk
        self.sk = sk
        self.w = w
        self.dev = dev
        L, B, Hq, Hkv, d, n = w.layers, w.batch, w.hq, w.hkv, w.d, w.n
        self.L, self.B, self.Hq, self.Hkv, self.d, self.n = L, B, Hq, Hkv, d, n
        self.BH = B * Hkv
        self.scale = 1.0 / math.sqrt(d)
        self.layers = [workloads.make_layer(w, l, device=dev) for l in range(L)]
        # a1 inputs: head scores over the L x Hkv heads of one sequence
        self.s_heads = workloads.head_scores(w).numpy()
        if w.keep:
            k_h = w.keep[keep_index]
            self.budget_args = (L * Hkv * k_h, w.n_recent, 0.1, n)
        else:
            self.budget_args = (w.avg_budget * L * Hkv, w.w_local, w.rho, n)
        # two pinned staging buffers for the a1 output, so the host never writes
        # one that a copy still reads
        self.offs_pinned = [torch.zeros((L, self.BH + 1), dtype=torch.int32).pin_memory() for _ in range(2)]
        self.offs_done = [None, None]
        self.flip = 0
        self.offs_host = self.offs_pinned[0]
        self.offs_dev = torch.zeros((L, self.BH + 1), dtype=torch.int32, device=dev)
        self.budgets()
        self.totals = [int(x) for x in self.offs_host[:, -1]]
        self.offs_dev.copy_(self.offs_host)
        self.scores = torch.empty((L, B, Hkv, n), dtype=torch.float32, device=dev)
        self.idx = torch.empty((L, max(max(self.totals), 1)), dtype=torch.int32, device=dev)
        self.o_sp = torch.empty((L, B, Hq, d), dtype=torch.bfloat16, device=dev)
        self.l_sp = torch.empty((L, B, Hq), dtype=torch.float32, device=dev)
        self.o_de = torch.empty((L, B, Hq, 1, d), dtype=torch.bfloat16, device=dev)
        self.l_de = torch.empty((L, B, Hq, 1), dtype=torch.float32, device=dev)
        self.q_de = [lay["q"][:, :, None, :].contiguous() for lay in self.layers]
        self.ws_score = sk.new_workspace(sk.workspace_size(sk.OP_SCORE, B, Hq, Hkv, d, n, w.window), dev)
        self.ws_sel = sk.new_workspace(sk.workspace_size(sk.OP_SELECT, B, 0, Hkv, 0, n, 0), dev)
        self.ws_sp = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), dev)
        self.ws_de = sk.new_workspace(sk.workspace_size(sk.OP_DENSE_VERIFY, B, Hq, Hkv, d, n, 1), dev)
        self.graphs = {}

    def budgets(self):
        """a1 on the host: budgets of all L x Hkv heads; every sequence of the
        batch gets lists of the same lengths."""
        total_B, w_loc, rho, cap = self.budget_args
        b = self.sk.head_budgets(self.s_heads, total_B, w_loc, rho, cap).reshape(self.L, self.Hkv)
        per = np.tile(b, (1, self.B))                      # [L][B*Hkv], sequence-major
        offs = self.offs_host.numpy()
        offs[:, 0] = 0
        np.cumsum(per, axis=1, out=offs[:, 1:])
        return b

    def phase_score(self):
        w = self.w
        for l, lay in enumerate(self.layers):
            self.sk.score_obs_window(lay["q_obs"], lay["k"], self.n, w.q_pos0, self.scale,
                                     scores=self.scores[l], ws=self.ws_score)

    def phase_select(self):
        w = self.w
        for l in range(self.L):
            self.sk.select_topk(self.scores[l], self.n, w.cand_lo, w.cand_hi, w.n_sink, w.n_recent,
                                self.offs_dev[l], self.totals[l], indices=self.idx[l], ws=self.ws_sel)

    def phase_sparse(self):
        for l, lay in enumerate(self.layers):
            self.sk.sparse_decode_attn(lay["q"], lay["k"], lay["v"], self.offs_dev[l], self.idx[l], self.scale,
                                       o=self.o_sp[l], lse=self.l_sp[l], ws=self.ws_sp)

    def phase_dense(self):
        for l, lay in enumerate(self.layers):
            self.sk.dense_verify_attn(self.q_de[l], lay["k"], lay["v"], self.n - 1, self.scale,
                                      o=self.o_de[l], lse=self.l_de[l], ws=self.ws_de)

    def capture(self):
        # eager pass first (sets kernel attributes, checks everything runs)
        for ph in self.PHASES:
            getattr(self, "phase_" + ph)()
        torch.cuda.synchronize()
        for ph in self.PHASES:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                getattr(self, "phase_" + ph)()
            self.graphs[ph] = g
        torch.cuda.synchronize()

    def step_budgets(self):
        """a1 on the host and the copy of its lists' offsets to the device."""
        self.flip ^= 1
        if self.offs_done[self.flip] is not None:
            self.offs_done[self.flip].synchronize()
        self.offs_host = self.offs_pinned[self.flip]
        self.budgets()
        self.offs_dev.copy_(self.offs_host, non_blocking=True)
        ev = torch.cuda.Event()
        ev.record()
        self.offs_done[self.flip] = ev

    def layer_ops(self, l):
        """a2..a5 of layer l through the public API (eager, current stream)."""
        w, lay = self.w, self.layers[l]
        self.sk.score_obs_window(lay["q_obs"], lay["k"], self.n, w.q_pos0, self.scale, scores=self.scores[l],
                                 ws=self.ws_score)
        self.sk.select_topk(self.scores[l], self.n, w.cand_lo, w.cand_hi, w.n_sink, w.n_recent, self.offs_dev[l],
                            self.totals[l], indices=self.idx[l], ws=self.ws_sel)
        self.sk.sparse_decode_attn(lay["q"], lay["k"], lay["v"], self.offs_dev[l], self.idx[l], self.scale,
                                   o=self.o_sp[l], lse=self.l_sp[l], ws=self.ws_sp)
        self.sk.dense_verify_attn(self.q_de[l], lay["k"], lay["v"], self.n - 1, self.scale, o=self.o_de[l],
                                  lse=self.l_de[l], ws=self.ws_de)

    def step(self, evs=None):
        self.step_budgets()
        for i, ph in enumerate(self.PHASES):
            if evs is not None:
                evs[i].record()
            self.graphs[ph].replay()
        if evs is not None:
            evs[len(self.PHASES)].record()

    def launches_per_step(self):
        return self.L * (2 + 1 + 1 + 1)   # score = 2 kernels, select, sparse, dense

    def alg_bytes_per_layer(self):
        mean_total = float(np.mean(self.totals))
        return {
            "score": ba.score_bytes(self.B, self.Hq, self.Hkv, self.d, self.n, self.w.window),
            "select": ba.select_bytes(self.B, self.Hkv, self.n, int(mean_total)),
            "sparse": ba.sparse_decode_bytes(self.B, self.Hq, self.d, int(mean_total)),
            "dense": ba.dense_verify_bytes(self.B, self.Hq, self.Hkv, self.d, self.n - 1, 1),
        }


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_kv_decode_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        path = os.path.join(csrc, name)
        if not os.path.isfile(path):
            continue
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(phase, workload):
    """DRAM bytes per launch from profiles/dram_traffic.txt, if they were taken
    with the current kernel sources (same source hash) on this workload's
    full-size launch, else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if (len(parts) >= 4 and not line.startswith("#") and parts[0] == phase and parts[2] == cur
                    and parts[3] == workload):
                return float(parts[1])
    return None


# ----------------------------------------------------------------------------- CPU oracle timing
def _oracle_unit(w, kk, vv, qo, qq):
    """The whole path of one KV head through the oracle: its window scores, its
    top-K list, and the sparse and dense decode of its G query heads."""
    import oracle
    kh = w.keep[0] if w.keep else w.avg_budget
    sc = oracle.score_obs_window(qo, kk, w.n, w.q_pos0)
    offs = np.array([0, kh])
    idx = oracle.select_topk(sc, w.n, w.cand_lo, w.cand_hi, w.n_sink, w.n_recent, offs)
    oracle.sparse_decode(qq, kk, vv, offs, idx)
    oracle.dense_verify(qq[:, :, None, :], kk, vv, w.n - 1)


def _unit_inputs(w, lay, b, h):
    G = w.hq // w.hkv
    return (lay["k"][b:b + 1, h:h + 1].cpu(), lay["v"][b:b + 1, h:h + 1].cpu(),
            lay["q_obs"][b:b + 1, h * G:(h + 1) * G].cpu(), lay["q"][b:b + 1, h * G:(h + 1) * G].cpu())


def oracle_units(w, layer_fn, n_units, rng_seed=0):
    """Seconds per unit of the oracle in this process on `n_units` sampled
    (layer, sequence, KV head) units."""
    rng = np.random.default_rng(rng_seed)
    units = [(int(rng.integers(w.layers)), int(rng.integers(w.batch)), int(rng.integers(w.hkv)))
             for _ in range(n_units)]
    total = 0.0
    for (l, b, h) in units:
        args = _unit_inputs(w, layer_fn(l), b, h)
        t0 = time.perf_counter()
        _oracle_unit(w, *args)
        total += time.perf_counter() - t0
    return total / n_units


def host_cores():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _oracle_worker(name, layer, units, rounds, start_bar, out_q):
    """One host core (one process, one BLAS thread): its units of one layer,
    timed `rounds` times; every round starts at a barrier of all workers."""
    try:
        w = workloads.by_name(name)
        lay = workloads.make_layer(w, layer, device="cpu")
        data = [_unit_inputs(w, lay, b, h) for (b, h) in units]
        del lay
        res = []
        for _ in range(rounds):
            start_bar.wait(timeout=300)
            t0 = time.time()
            for args in data:
                _oracle_unit(w, *args)
            res.append((t0, time.time(), len(data)))
        out_q.put((res, None))
    except Exception as e:
        start_bar.abort()   # release the other workers at once
        out_q.put((None, repr(e)))


def oracle_parallel(w, cores, per_worker, rounds, timeout=900.0):
    """Seconds per unit, per round, of the oracle run by `cores` worker
    processes at once (started with spawn), each on `per_worker` sampled
    (sequence, KV head) units of its own layer: the wall time of the round over
    the units all workers processed."""
    import multiprocessing as mp
    import queue
    ctx = mp.get_context("spawn")
    start_bar = ctx.Barrier(cores)
    out_q = ctx.Queue()
    rng = np.random.default_rng(7)
    procs = []
    for i in range(cores):
        units = [(int(rng.integers(w.batch)), int(rng.integers(w.hkv))) for _ in range(per_worker)]
        p = ctx.Process(target=_oracle_worker, args=(w.name, (7 * i) % w.layers, units, rounds, start_bar, out_q),
                        daemon=True)
        p.start()
        procs.append(p)
    results, deadline = [], time.time() + timeout
    try:
        while len(results) < cores:
            try:
                res, err = out_q.get(timeout=5)
            except queue.Empty:
                if time.time() > deadline or any(p.exitcode not in (None, 0) for p in procs):
                    raise RuntimeError("an oracle worker died or timed out")
                continue
            if err is not None:
                raise RuntimeError("oracle worker: " + err)
            results.append(res)
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()
    per_round = []
    for r in range(rounds):
        t0 = min(res[r][0] for res in results)
        t1 = max(res[r][1] for res in results)
        per_round.append((t1 - t0) / sum(res[r][2] for res in results))
    return per_round


def cpu_baseline(w, layer_fn, seconds):
    """The oracle on all host cores: one worker process per core, each timing
    a bounded sample of whole-path units; scaled to one step of the workload.
    Falls back to one core (and says so) if worker processes cannot run."""
    per_unit = oracle_units(w, layer_fn, 1)
    per_worker = max(1, min(8, int(seconds / max(per_unit, 1e-3))))
    units_per_step = w.layers * w.batch * w.hkv
    what = ("whole path for one KV head (scores, top-K list, sparse and dense decode of its %d query heads), "
            "fp64 numpy" % (w.hq // w.hkv))
    cores = host_cores()
    try:
        per_unit = oracle_parallel(w, cores, per_worker, 1)[0]
        sample = ("%d (sequence, KV head) units of the %s workload on each of %d worker processes (one per host "
                  "core, one BLAS thread each, one layer each), timed together; a unit is the %s; wall time "
                  "over units, scaled by %d units per step" % (per_worker, w.name, cores, what, units_per_step))
    except Exception as e:   # no worker processes: this process alone
        cores = 1
        per_worker = max(1, min(64, int(seconds / max(per_unit, 1e-3))))
        per_unit = oracle_units(w, layer_fn, per_worker, rng_seed=1)
        sample = ("%d (layer, sequence, KV head) units of the %s workload in one process (worker processes "
                  "failed: %s); a unit is the %s; scaled by %d units per step"
                  % (per_worker, w.name, e, what, units_per_step))
    return {"value": per_unit * units_per_step * 1e6, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": sample}


# ----------------------------------------------------------------------------- arms
def run_reference(args, world, rank):
    if rank != 0:
        return
    w = workloads.by_name(args.workload)
    warm = max(args.warmup, 3)
    units_per_step = w.layers * w.batch * w.hkv
    cores = host_cores()
    try:
        # every step: one whole-path unit on each host core, all cores at once
        per_round = oracle_parallel(w, cores, 1, warm + args.steps)
        note = ("fp64 CPU oracle on %d worker processes (one per host core, one BLAS thread each); each step "
                "times one sampled (sequence, KV head) unit of the whole path per worker, all at once, and "
                "scales the wall time per unit to the full step" % cores)
    except Exception as e:
        cores = 1
        cache = {}

        def layer_fn(l):
            if l not in cache:
                cache.clear()
                cache[l] = workloads.make_layer(w, l, device="cpu")
            return cache[l]

        per_round = [oracle_units(w, layer_fn, 2, rng_seed=100 + i) for i in range(warm + args.steps)]
        note = ("fp64 CPU oracle in one process (worker processes failed: %s); each step times 2 sampled "
                "(layer, sequence, KV head) units of the whole path and scales to the full step" % e)
    us = float(np.mean(per_round[warm:])) * units_per_step * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": warm, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "note": note},
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d unit(s) per step on %d core(s), scaled by %d units per step"
                                   % (cores, cores, units_per_step)},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_e2e(path, K, world):
    """The same step through the public API with the inputs in pinned host
    memory: every step copies all layers' K, V, window queries and decode
    queries to the device and reads the decode outputs back.  Layer l's inputs
    go over on a copy stream while layer l - 1 computes (the host link, about
    0.2 TB/s here, is the bound; the compute hides behind it)."""
    host = []
    h2d = 0
    for lay in path.layers:
        hl = {}
        for name in ("k", "v", "q_obs", "q"):
            t = torch.empty(lay[name].shape, dtype=lay[name].dtype, pin_memory=True)
            t.copy_(lay[name])
            hl[name] = t
            h2d += t.numel() * t.element_size()
        host.append(hl)
    outs = [path.o_sp, path.l_sp, path.o_de, path.l_de]
    out_host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
    d2h = sum(o.numel() * o.element_size() for o in outs)

    comp = torch.cuda.current_stream()
    copy_st = torch.cuda.Stream()
    arrived = [torch.cuda.Event() for _ in path.layers]
    done = torch.cuda.Event()
    done.record(comp)

    def step():
        path.step_budgets()
        copy_st.wait_event(done)          # the previous step no longer reads the inputs
        for l, (lay, hl) in enumerate(zip(path.layers, host)):
            with torch.cuda.stream(copy_st):
                for name in ("k", "v", "q_obs", "q"):
                    lay[name].copy_(hl[name], non_blocking=True)
                arrived[l].record(copy_st)
            comp.wait_event(arrived[l])
            path.q_de[l].copy_(lay["q"][:, :, None, :], non_blocking=True)
            path.layer_ops(l)
        for o, oh in zip(outs, out_host):
            oh.copy_(o, non_blocking=True)
        done.record(comp)

    step()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    barrier(world)
    s.record()
    for _ in range(K):
        step()
    e.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(s.elapsed_time(e), world)
    return {"value": ms / K * 1e3, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": K}


def time_graph_us(fn, reps: int = 10, flush: torch.Tensor | None = None) -> float:
    """Median device time (µs) of one CUDA-graph replay of `fn`'s launches,
    with an L2 flush (a write larger than L2) before every replay."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    ts = []
    for r in range(reps + 3):
        if flush is not None:
            flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        if r >= 3:
            ts.append(a.elapsed_time(b) * 1e3)
    return float(np.median(ts))


def next_rows_timings(path, hbm_peak, dev):
    """Timings of the rows beyond the hot path (each a separate measurement,
    outside the step):
      f1  compaction of the selected rows (once per selection) and the decode
          over the compacted rows, on this workload's lists, every layer;
      f2  decode over sink + recent lists (4 + 64), every layer;
      f3  SpecVLM selection for one request of the video workload (28 layers x
          4 KV heads of window scores over 12,800 tokens, 12,544 of them video);
      f4  one StD round of the video workload per layer: 5 draft steps (list
          append on the device + sparse decode over the 1,024 kept + drafted
          rows) and the verify of the 5 drafts, in one graph."""
    sk = path.sk
    L, B, Hq, Hkv, d, n = path.L, path.B, path.Hq, path.Hkv, path.d, path.n
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    # f1
    kc, vc = [], []
    for l, lay in enumerate(path.layers):
        tot = path.totals[l]
        kc.append(torch.empty((max(tot, 1), d), dtype=torch.bfloat16, device=dev))
        vc.append(torch.empty((max(tot, 1), d), dtype=torch.bfloat16, device=dev))
    ws_c = sk.new_workspace(sk.workspace_size(sk.OP_COMPACT, B, 0, Hkv, d, 0, 0), dev)

    def compact():
        for l, lay in enumerate(path.layers):
            sk.compact_kv(lay["k"], lay["v"], path.offs_dev[l], path.idx[l], path.totals[l], k_out=kc[l],
                          v_out=vc[l], ws=ws_c)

    def contig():
        for l, lay in enumerate(path.layers):
            sk.sparse_decode_compact(lay["q"], kc[l], vc[l], path.offs_dev[l], Hkv, path.scale, o=path.o_sp[l],
                                     lse=path.l_sp[l], ws=path.ws_sp)
    t_comp = time_graph_us(compact, flush=flush) / L
    t_contig = time_graph_us(contig, flush=flush) / L
    mean_total = float(np.mean(path.totals))
    b_comp = 2 * mean_total * 4 * d                                  # read and write K and V rows
    b_contig = mean_total * 4 * d + B * Hq * 4 * d                   # K/V rows + q in / o out
    out["f1_compaction"] = {"us_per_layer": t_comp, "alg_bytes_per_layer": b_comp,
                            "gbs": b_comp / t_comp / 1e3, "frac_of_measured_hbm": b_comp / t_comp / 1e3 / hbm_peak}
    out["f1_contiguous_decode"] = {"us_per_layer": t_contig, "alg_bytes_per_layer": b_contig,
                                   "gbs": b_contig / t_contig / 1e3,
                                   "frac_of_measured_hbm": b_contig / t_contig / 1e3 / hbm_peak}
    assert sk.workspace_status(ws_c) == 0 and sk.workspace_status(path.ws_sp) == 0
    del kc, vc
    # f2
    w_offs, w_idx = sk.window_lists(B, Hkv, n, 4, 64, dev)

    def window():
        for l, lay in enumerate(path.layers):
            sk.sparse_decode_attn(lay["q"], lay["k"], lay["v"], w_offs, w_idx, path.scale, o=path.o_sp[l],
                                  lse=path.l_sp[l], ws=path.ws_sp)
    t_win = time_graph_us(window, flush=flush) / L
    b_win = B * Hkv * 68 * (4 * d + 4) + B * Hq * 4 * d
    out["f2_window_decode"] = {"us_per_layer": t_win, "alg_bytes_per_layer": b_win, "lists": "4 sinks + 64 recent"}
    # f3 and f4 on the video workload
    vw = workloads.by_name("video")
    g = torch.Generator(device=dev).manual_seed(7)
    units = vw.layers * vw.hkv
    scores = torch.rand((1, units, vw.n), generator=g, device=dev) ** 4
    v_hi = vw.frames * vw.frame_tokens
    ws_s = sk.new_workspace(sk.workspace_size(sk.OP_SPECVLM, 1, 0, 0, 0, v_hi, 0), dev)
    imp = torch.empty((1, vw.n), dtype=torch.float32, device=dev)
    sidx = torch.empty((1, vw.n), dtype=torch.int32, device=dev)
    cnt = torch.empty(1, dtype=torch.int32, device=dev)

    def spec():
        sk.specvlm_select(scores, 0, v_hi, 0.5, 0.9, v_hi, vw.n, importance=imp, indices=sidx, counts=cnt, ws=ws_s)
    t_spec = time_graph_us(spec, flush=flush)
    out["f3_specvlm_select"] = {"us_per_request": t_spec, "units": units, "tokens": vw.n, "video_tokens": v_hi,
                                "lam_r": 0.5, "r": 0.9, "kept": int(cnt.item())}
    gam = vw.gamma
    lay = workloads.make_layer(vw, 0, device=dev, n=vw.n + gam)
    vs = 1.0 / math.sqrt(vw.d)
    BHv = vw.batch * vw.hkv
    kh = vw.text_tokens + 768
    base_o = torch.arange(BHv + 1, dtype=torch.int32, device=dev) * kh
    sc = sk.score_obs_window(lay["q_obs"][:, :, : vw.text_tokens].contiguous(), lay["k"], vw.n, vw.q_pos0, vs)
    base_i = sk.select_topk(sc, vw.n, vw.cand_lo, vw.cand_hi, vw.n_sink, vw.n_recent, base_o, BHv * kh)
    d_offs = torch.empty((gam, BHv + 1), dtype=torch.int32, device=dev)
    d_idx = torch.empty((gam, BHv * (kh + gam)), dtype=torch.int32, device=dev)
    o_d = torch.empty((vw.batch, vw.hq, vw.d), dtype=torch.bfloat16, device=dev)
    o_v = torch.empty((vw.batch, vw.hq, gam, vw.d), dtype=torch.bfloat16, device=dev)
    ws_sp = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, vw.batch, vw.hq, vw.hkv, vw.d, 0, 0), dev)
    ws_de = sk.new_workspace(sk.workspace_size(sk.OP_DENSE_VERIFY, vw.batch, vw.hq, vw.hkv, vw.d, vw.n + gam, gam),
                             dev)

    q_step = [lay["q_ver"][:, :, t].contiguous() for t in range(gam)]   # each draft step's query

    def round_():
        # every draft step's list (base + the drafted positions so far) in one launch
        sk.draft_lists(base_o, base_i, BHv * kh, vw.n, gam, offsets=d_offs, indices=d_idx)
        for t in range(gam):
            sk.sparse_decode_attn(q_step[t], lay["k"], lay["v"], d_offs[t], d_idx[t], vs, o=o_d, ws=ws_sp,
                                  want_lse=False)
        sk.dense_verify_attn(lay["q_ver"], lay["k"], lay["v"], vw.n, vs, o=o_v, ws=ws_de, want_lse=False)
    t_round = time_graph_us(round_, flush=flush)
    out["f4_std_round"] = {"us_per_layer": t_round, "us_per_step_all_layers": t_round * vw.layers, "gamma": gam,
                           "kept_per_head": kh, "launches_per_layer": gam + 2}
    return out


def run_sdkv(args, world, rank, local):
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl sdkv")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workloads.by_name(args.workload)
    if args.layers:
        w = dataclasses.replace(w, layers=args.layers)
    hbm_peak, peak_kind = peaks()
    path = Path(w, args.keep_index, dev)
    path.capture()
    warm = max(args.warmup, 3)
    K = args.steps
    for _ in range(warm):
        path.step()
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(args.clocks_log)
    time.sleep(0.25)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(Path.PHASES) + 1)] for _ in range(K)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    start.record()
    for i in range(K):
        path.step(evs[i])
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    clocks = sampler.stop(t0, t1, uuid)
    total_ms = max_over_ranks(start.elapsed_time(end), world)
    phase_ms = {ph: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)) / K
                for j, ph in enumerate(Path.PHASES)}
    us_step = total_ms / K * 1e3

    # device-side status words must be clean
    for wsb in (path.ws_score, path.ws_sel, path.ws_sp, path.ws_de):
        st = path.sk.workspace_status(wsb)
        if st != 0:
            raise SystemExit("device status %d raised during the bench" % st)

    alg = path.alg_bytes_per_layer()
    L = path.L
    breakdown = {}
    for ph in Path.PHASES:
        per_layer_us = phase_ms[ph] * 1e3 / L
        gbs = alg[ph] / (per_layer_us * 1e-6) / 1e9
        breakdown[ph] = {"us_per_step": phase_ms[ph] * 1e3, "us_per_layer": per_layer_us,
                         "alg_bytes_per_layer": alg[ph], "gbs": gbs,
                         "frac_of_measured_hbm": gbs / hbm_peak, "frac_of_8tbs_nominal": gbs / NOMINAL_HBM_GBS}
    dominant = max(Path.PHASES, key=lambda ph: phase_ms[ph])
    dom = breakdown[dominant]
    kernel_names = {"score": "sdkv_score_obs_window (score_kernel pass 1 + pass 2)",
                    "select": "sdkv_select_topk (select_topk_kernel)",
                    "sparse": "sdkv_sparse_decode_attn (attn_splitk_kernel, gathered)",
                    "dense": "sdkv_dense_verify_attn (attn_splitk_kernel, dense)"}
    roofline = {"bound": "hbm", "achieved": dom["gbs"], "peak": hbm_peak, "unit": "GB/s",
                "frac": dom["gbs"] / hbm_peak, "traffic": traffic_from_profiles(dominant, w.name),
                "kernel": kernel_names[dominant], "peak_kind": peak_kind,
                "alg_bytes_per_launch": dom["alg_bytes_per_layer"], "us_per_launch": dom["us_per_layer"]}
    keep = ("%d" % w.keep[args.keep_index]) if w.keep else "ragged SparseMM budgets"
    line = {
        "metric": METRIC, "value": us_step, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": warm,
        "ms_per_step": us_step / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s: %d layers x (%d q / %d KV heads, d=%d), batch %d, context %d, window %d, "
                               "keep %s per head (%d sinks + %d recent + top-K)" % (
                                   w.name, w.layers, w.hq, w.hkv, w.d, w.batch, w.n, w.window, keep,
                                   w.n_sink, w.n_recent),
                   "l2": "inputs larger than L2: %d distinct layers, %.2f GB of K/V per step" % (
                       L, L * 2 * w.batch * w.hkv * w.n * w.d * 2 / 1e9),
                   "step": "a1 budgets (host) + a2 score + a3 select + a4 sparse decode + a5 dense decode, "
                           "all layers; a2..a5 one CUDA graph each"},
        "sparse_vs_dense": {
            "sparse_us_per_step": breakdown["sparse"]["us_per_step"],
            "dense_us_per_step": breakdown["dense"]["us_per_step"],
            "speedup": breakdown["dense"]["us_per_step"] / breakdown["sparse"]["us_per_step"],
            "byte_bound": alg["dense"] / alg["sparse"],
            "sparse_frac_of_measured_hbm": breakdown["sparse"]["frac_of_measured_hbm"],
            "dense_frac_of_measured_hbm": breakdown["dense"]["frac_of_measured_hbm"],
            "sparse_frac_of_8tbs": breakdown["sparse"]["frac_of_8tbs_nominal"],
            "dense_frac_of_8tbs": breakdown["dense"]["frac_of_8tbs_nominal"],
        },
        "breakdown": breakdown,
        "roofline": roofline,
        "gpu_launches": path.launches_per_step() * K,
        "clocks": clocks,
    }
    if not args.no_e2e:
        line["e2e"] = run_e2e(path, min(K, 5), world)
    if rank == 0 and not args.no_next:
        line["next_rows"] = next_rows_timings(path, hbm_peak, dev)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, lambda l: path.layers[l], args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))


def main():
    args = parse()
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_sdkv(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
