#!/usr/bin/env python
"""Benchmark of the sparse-KV decode hot path on one GB300 (or N replicas).

Headline (`value`): one decode step of the Llama-3.1-8B-shaped 32K workload,
i.e. the gathered sparse decode (a4) of every layer over per-head lists that
were fixed after selection, in one CUDA graph of the per-layer library calls.
Before it, once per sequence (the prefill), the step's lists come from the
library itself:
  a1 head budgets (host)           -> per-head list lengths
  a2 window scoring, every layer   -> fp32 scores
  a3 top-K selection, every layer  -> per-head index lists
Measured beside the headline, in the same run:
  a5 dense decode (split-K) of every layer, the comparison of the pages;
  a2 + a3 of every layer (`prefill_select`, once per sequence);
  the 128K workload (keep 10/30/50%, dense, gamma=8 verify), the video workload
  (StD draft decode, dense, gamma=5 verify; the StD I/O model and the measured
  verify-over-dense ratio), and the SparseMM ragged-budget workload;
  the rows around the hot path (compaction, window lists, SpecVLM, StD round).

Prints ONE JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
instead (the reference arm: a deliberately slow program) on whole decode steps.
"""
import os

# The oracle's CPU timing runs one single-threaded BLAS per worker process.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import ctypes  # noqa: E402
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


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="sdkv", choices=["sdkv", "reference"])
    ap.add_argument("--workload", default="llama8b_32k")
    ap.add_argument("--keep-index", type=int, default=0, help="which keep ratio of the workload")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the 128K, video and SparseMM blocks")
    ap.add_argument("--no-next", action="store_true", help="skip the timings of the next rows (f1..f4)")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (small profiling cases only; reported in config)")
    ap.add_argument("--clocks-log", default="",
                    help="file for the raw nvidia-smi samples of the timed region (default: a temporary file)")
    return ap.parse_args(argv)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def workload_config(w, keep_index=0):
    """The `config` of both arms' JSON lines (identical strings in both)."""
    if w.keep:
        keep = "%d per head (%d sinks + %d recent + top-K)" % (w.keep[keep_index], w.n_sink, w.n_recent)
    else:
        keep = ("ragged SparseMM budgets, average %d per head (w=%d, rho=%.1f; %d recent + top-K)"
                % (w.avg_budget, w.w_local, w.rho, w.n_recent))
    return {
        "workload": "%s: %d layers x (%d q / %d KV heads, d=%d), batch %d, context %d, keep %s; one decode step "
                    "= the sparse decode of every layer over lists fixed after selection" % (
                        w.name, w.layers, w.hq, w.hkv, w.d, w.batch, w.n, keep),
        "l2": "inputs larger than L2: %d distinct layers of K/V (%.2f GB)" % (
            w.layers, w.layers * 2 * w.batch * w.hkv * w.n * w.d * 2 / 1e9),
    }


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


# ----------------------------------------------------------------------------- device state
class Decode:
    """Device state of one workload after its prefill: K/V caches and queries
    of `distinct` layers (cycled when fewer than the workload's layers), the
    per-head lists of each keep ratio from the library's own a1..a3, and the
    per-layer library calls of each phase."""

    def __init__(self, w, dev, distinct=0, verify=False):
        import sparse_kv_decode_gb300 as sk
        self.sk, self.w, self.dev = sk, w, dev
        L, B, Hq, Hkv, d, n = w.layers, w.batch, w.hq, w.hkv, w.d, w.n
        self.L, self.B, self.Hq, self.Hkv, self.d, self.n = L, B, Hq, Hkv, d, n
        self.BH = B * Hkv
        self.scale = 1.0 / math.sqrt(d)
        nd = min(L, distinct) if distinct else L
        self.lays = [workloads.make_layer(w, l, device=dev) for l in range(nd)]
        self.q_de = [lay["q"][:, :, None, :].contiguous() for lay in self.lays]
        self.s_heads = workloads.head_scores(w).numpy()
        self.scores = torch.empty((L, B, Hkv, n), dtype=torch.float32, device=dev)
        self.o_sp = torch.empty((L, B, Hq, d), dtype=torch.bfloat16, device=dev)
        self.l_sp = torch.empty((L, B, Hq), dtype=torch.float32, device=dev)
        self.o_de = torch.empty((L, B, Hq, 1, d), dtype=torch.bfloat16, device=dev)
        self.l_de = torch.empty((L, B, Hq, 1), dtype=torch.float32, device=dev)
        self.ws_score = sk.new_workspace(sk.workspace_size(sk.OP_SCORE, B, Hq, Hkv, d, n, w.window), dev)
        self.ws_sel = sk.new_workspace(sk.workspace_size(sk.OP_SELECT, B, 0, Hkv, 0, n, 0), dev)
        self.ws_sp = sk.new_workspace(sk.workspace_size(sk.OP_SPARSE_DECODE, B, Hq, Hkv, d, 0, 0), dev)
        self.ws_de = sk.new_workspace(sk.workspace_size(sk.OP_DENSE_VERIFY, B, Hq, Hkv, d, n, 1), dev)
        self.verify = verify
        if verify:
            self.o_v = torch.empty((L, B, Hq, w.gamma, d), dtype=torch.bfloat16, device=dev)
            self.ws_v = sk.new_workspace(sk.workspace_size(sk.OP_DENSE_VERIFY, B, Hq, Hkv, d, n, w.gamma), dev)
        self.lists = {}          # keep index -> (offsets [L][BH+1] int32 device, indices [L][max] int32, totals)

    def lay(self, l):
        return self.lays[l % len(self.lays)]

    def workspaces(self):
        out = [self.ws_score, self.ws_sel, self.ws_sp, self.ws_de]
        return out + ([self.ws_v] if self.verify else [])

    # a1 on the host: budgets of all L x Hkv heads; every sequence of the batch gets lists of the same lengths
    def budgets(self, ki):
        w = self.w
        if w.keep:
            args = (self.L * self.Hkv * w.keep[ki], w.n_recent, 0.1, self.n)
        else:
            args = (w.avg_budget * self.L * self.Hkv, w.w_local, w.rho, self.n)
        b = self.sk.head_budgets(self.s_heads, *args).reshape(self.L, self.Hkv)
        per = np.tile(b, (1, self.B))                      # [L][B*Hkv], sequence-major
        offs = np.zeros((self.L, self.BH + 1), dtype=np.int32)
        np.cumsum(per, axis=1, out=offs[:, 1:])
        return offs

    def score_all(self):
        w = self.w
        for l in range(self.L):
            lay = self.lay(l)
            self.sk.score_obs_window(lay["q_obs"], lay["k"], self.n, w.q_pos0, self.scale, scores=self.scores[l],
                                     ws=self.ws_score)

    def select_all(self, ki):
        w = self.w
        offs, idx, totals = self.lists[ki]
        for l in range(self.L):
            self.sk.select_topk(self.scores[l], self.n, w.cand_lo, w.cand_hi, w.n_sink, w.n_recent, offs[l],
                                totals[l], indices=idx[l], ws=self.ws_sel)

    def prefill(self, keep_indices=(0,)):
        """a1 (host) for every keep ratio, a2 once, a3 per keep ratio."""
        for ki in keep_indices:
            offs = self.budgets(ki)
            totals = [int(x) for x in offs[:, -1]]
            idx = torch.empty((self.L, max(max(totals), 1)), dtype=torch.int32, device=self.dev)
            self.lists[ki] = (torch.from_numpy(offs).to(self.dev), idx, totals)
        self.score_all()
        for ki in keep_indices:
            self.select_all(ki)
        torch.cuda.synchronize()

    def sparse_step(self, ki):
        offs, idx, _ = self.lists[ki]
        for l in range(self.L):
            lay = self.lay(l)
            self.sk.sparse_decode_attn(lay["q"], lay["k"], lay["v"], offs[l], idx[l], self.scale, o=self.o_sp[l],
                                       lse=self.l_sp[l], ws=self.ws_sp)

    def dense_step(self):
        for l in range(self.L):
            lay = self.lay(l)
            self.sk.dense_verify_attn(self.q_de[l % len(self.lays)], lay["k"], lay["v"], self.n - 1, self.scale,
                                      o=self.o_de[l], lse=self.l_de[l], ws=self.ws_de)

    def verify_step(self):
        g = self.w.gamma
        for l in range(self.L):
            lay = self.lay(l)
            self.sk.dense_verify_attn(lay["q_ver"], lay["k"], lay["v"], self.n - g, self.scale, o=self.o_v[l],
                                      ws=self.ws_v, want_lse=False)

    def prefill_step(self, ki):
        self.score_all()
        self.select_all(ki)

    def mean_total(self, ki):
        return float(np.mean(self.lists[ki][2]))

    def alg_bytes(self, phase, ki=0):
        """Algorithmic bytes of one layer's launch of a phase."""
        w, B, Hq, Hkv, d, n = self.w, self.B, self.Hq, self.Hkv, self.d, self.n
        if phase == "sparse":
            return ba.sparse_decode_bytes(B, Hq, d, int(self.mean_total(ki)))
        if phase == "dense":
            return ba.dense_verify_bytes(B, Hq, Hkv, d, n - 1, 1)
        if phase == "verify":
            return ba.dense_verify_bytes(B, Hq, Hkv, d, n - w.gamma, w.gamma)
        if phase == "score":
            return ba.score_bytes(B, Hq, Hkv, d, n, w.window)
        if phase == "select":
            return ba.select_bytes(B, Hkv, n, int(self.mean_total(ki)))
        raise KeyError(phase)


def capture(fn):
    """One eager run of `fn` (sets kernel attributes, checks it runs), then a
    CUDA graph of its launches."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(g, reps, flush=None):
    """Median device time (µs) of one replay of `g` over `reps` replays after 3
    untimed ones; with `flush`, an L2-sized write before every replay."""
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


def phase_record(us_step, layers, alg_bytes_per_layer, hbm_peak):
    per_layer = us_step / layers
    gbs = alg_bytes_per_layer / (per_layer * 1e-6) / 1e9
    return {"us_per_step": us_step, "us_per_layer": per_layer, "alg_bytes_per_layer": alg_bytes_per_layer,
            "gbs": gbs, "frac_of_measured_hbm": gbs / hbm_peak, "frac_of_8tbs_nominal": gbs / NOMINAL_HBM_GBS}


# The files the split-K attention kernels (the gathered, contiguous and dense
# decodes whose traffic profiles/dram_traffic.txt records) are compiled from.
ATTN_SOURCES = ("sparse_kv_decode_gb300/csrc/attn_splitk.cu", "sparse_kv_decode_gb300/csrc/sdkv_common.cuh",
                "sparse_kv_decode_gb300/csrc/sdkv_internal.h", "include/sdkv.h")


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in ATTN_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
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
def host_cores():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def step_units(w):
    """The (layer, sequence, KV head) units of one decode step."""
    return [(l, b, h) for l in range(w.layers) for b in range(w.batch) for h in range(w.hkv)]


def _unit_lists_budgets(w, keep_index):
    """Per-(layer, KV head) list lengths: the oracle's own head budgets (a1)."""
    import oracle
    s = workloads.head_scores(w).numpy()
    if w.keep:
        b = oracle.head_budgets(s, w.layers * w.hkv * w.keep[keep_index], w.n_recent, 0.1, w.n)
    else:
        b = oracle.head_budgets(s, w.avg_budget * w.layers * w.hkv, w.w_local, w.rho, w.n)
    return np.asarray(b).reshape(w.layers, w.hkv)


def _decode_worker(name, keep_index, units, rounds, start_bar, out_q):
    """One host core (one process, one BLAS thread).  Set-up, untimed: its
    units' inputs and their lists from the oracle's own budgets, window scores
    and top-K selection (once per sequence, as on the GPU).  Then `rounds`
    timed rounds, each the oracle's sparse decode of every unit; every round
    starts at a barrier of all workers."""
    try:
        import oracle
        w = workloads.by_name(name)
        budgets = _unit_lists_budgets(w, keep_index)
        G = w.group
        data, cache = [], {}
        for (l, b, h) in units:
            if l not in cache:
                cache.clear()
                cache[l] = workloads.make_layer(w, l, device="cpu")
            lay = cache[l]
            kk = lay["k"][b:b + 1, h:h + 1].clone()
            vv = lay["v"][b:b + 1, h:h + 1].clone()
            qo = lay["q_obs"][b:b + 1, h * G:(h + 1) * G]
            qq = lay["q"][b:b + 1, h * G:(h + 1) * G].clone()
            sc = oracle.score_obs_window(qo, kk, w.n, w.q_pos0)
            offs = np.array([0, int(budgets[l, h])])
            idx = oracle.select_topk(sc, w.n, w.cand_lo, w.cand_hi, w.n_sink, w.n_recent, offs)
            data.append((qq, kk, vv, offs, idx))
        cache.clear()
        res = []
        for _ in range(rounds):
            start_bar.wait(timeout=900)
            t0 = time.time()
            for (qq, kk, vv, offs, idx) in data:
                oracle.sparse_decode(qq, kk, vv, offs, idx)
            res.append((t0, time.time(), len(data)))
        out_q.put((res, None))
    except Exception as e:
        start_bar.abort()   # release the other workers at once
        out_q.put((None, repr(e)))


def oracle_decode_rounds(w, keep_index, units, cores, rounds, timeout=1800.0):
    """Wall seconds of each round of the oracle's sparse decode of `units`, run
    by `cores` worker processes at once (started with spawn; worker i takes a
    contiguous block of the units, so it draws few layers)."""
    import multiprocessing as mp
    import queue
    ctx = mp.get_context("spawn")
    cores = max(1, min(cores, len(units)))
    start_bar = ctx.Barrier(cores)
    out_q = ctx.Queue()
    per = (len(units) + cores - 1) // cores
    procs = []
    for i in range(cores):
        p = ctx.Process(target=_decode_worker,
                        args=(w.name, keep_index, units[i * per:(i + 1) * per], rounds, start_bar, out_q),
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
    out = []
    for r in range(rounds):
        t0 = min(res[r][0] for res in results)
        t1 = max(res[r][1] for res in results)
        out.append(t1 - t0)
    return out, cores


def oracle_step_plan(w, max_units):
    """Units timed per step: the whole step when it has at most `max_units`
    units, else an evenly spaced sample (the value is then scaled to the step
    and the line says so)."""
    units = step_units(w)
    if len(units) <= max_units:
        return units, False
    stride = len(units) / max_units
    return [units[int(i * stride)] for i in range(max_units)], True


def oracle_decode_inline(w, keep_index, units, rounds):
    """The same rounds in this process (one core), for when worker processes
    cannot start."""
    import queue

    class _Bar:
        def wait(self, timeout=None):
            pass

        def abort(self):
            pass
    q = queue.Queue()
    _decode_worker(w.name, keep_index, units, rounds, _Bar(), q)
    res, err = q.get()
    if err is not None:
        raise RuntimeError("oracle: " + err)
    return [t1 - t0 for (t0, t1, _) in res]


def cpu_baseline(w, keep_index, timed_rounds=2, max_units=512):
    """The oracle's decode step on all host cores (one worker process per core),
    whole steps timed (1 untimed round, then `timed_rounds`).  Falls back to
    this process alone (and says so) if worker processes cannot run."""
    units, sampled = oracle_step_plan(w, max_units)
    total = len(step_units(w))
    where = ""
    try:
        rounds, used = oracle_decode_rounds(w, keep_index, units, host_cores(), 1 + timed_rounds)
        where = "%d worker processes (one per host core, one BLAS thread each)" % used
    except Exception as e:
        units, sampled = oracle_step_plan(w, 16)
        rounds, used = oracle_decode_inline(w, keep_index, units, 1 + timed_rounds), 1
        where = "this process alone (worker processes failed: %s)" % e
    per_step = float(np.mean(rounds[1:])) * (total / len(units))
    sample = ("the oracle's sparse decode (fp64 numpy) of %s%d (layer, sequence, KV head) units of the %s workload, "
              "on %s, lists from the oracle's own budgets, window scores and top-K selection; mean of %d timed "
              "rounds after 1 untimed"
              % ("" if not sampled else "a sample of ", len(units), w.name, where, timed_rounds)
              + ("" if not sampled else "; scaled by %d / %d units per step" % (total, len(units))))
    return {"value": per_step * 1e6, "unit": UNIT, "cores": used, "kind": "oracle", "sample": sample,
            "units_timed_per_step": len(units), "units_per_step": total, "extrapolated": sampled}


# ----------------------------------------------------------------------------- arms
def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle's decode step on the host cores."""
    if rank != 0:
        return
    w = workloads.by_name(args.workload)
    if args.layers:
        w = dataclasses.replace(w, layers=args.layers)
    warm = max(args.warmup, 3)
    units, sampled = oracle_step_plan(w, 512)
    total = len(step_units(w))
    t_start = time.time()
    rounds, cores = oracle_decode_rounds(w, args.keep_index, units, host_cores(), warm + args.steps)
    scale = total / len(units)
    us = float(np.mean(rounds[warm:])) * scale * 1e6
    sample = ("the oracle's sparse decode (fp64 numpy) of %s%d (layer, sequence, KV head) units per step on %d "
              "worker processes (one per host core, one BLAS thread each), lists from the oracle's own budgets, "
              "window scores and top-K selection (set-up, untimed)"
              % ("a sample of " if sampled else "all ", len(units), cores)
              + ("; scaled by %d / %d units per step" % (total, len(units)) if sampled else ""))
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": warm, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.keep_index),
        "units_timed_per_step": len(units), "units_per_step": total, "extrapolated": sampled,
        "timed_wall_s": float(np.sum(rounds[warm:])), "run_wall_s": time.time() - t_start,
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def run_e2e(D, ki, K, world):
    """The decode step end to end through the C ABI (sdkv_sparse_decode_attn once
    per layer, arguments marshalled once): every step copies all layers' decode
    queries from pinned host memory to the device and reads o and lse back.
    The caches and lists are device state from the prefill, not step inputs."""
    sk = D.sk
    L = sk.lib()
    offs, idx, _ = D.lists[ki]
    q_dev = torch.stack([D.lay(l)["q"] for l in range(D.L)]).contiguous()
    q_host = torch.empty(q_dev.shape, dtype=q_dev.dtype, pin_memory=True)
    q_host.copy_(q_dev)
    o_host = torch.empty(D.o_sp.shape, dtype=D.o_sp.dtype, pin_memory=True)
    l_host = torch.empty(D.l_sp.shape, dtype=D.l_sp.dtype, pin_memory=True)
    st = torch.cuda.current_stream().cuda_stream
    keep_alive, calls = [], []
    for l in range(D.L):
        lay = D.lay(l)
        strides = (ctypes.c_int64 * 3)(*lay["k"].stride()[:3])
        keep_alive.append(strides)
        calls.append((q_dev[l].data_ptr(), lay["k"].data_ptr(), lay["v"].data_ptr(), strides, lay["k"].shape[2],
                      offs[l].data_ptr(), idx[l].data_ptr(), idx[l].numel(), D.B, D.Hq, D.Hkv, D.d,
                      ctypes.c_float(D.scale), D.o_sp[l].data_ptr(), D.l_sp[l].data_ptr(), D.ws_sp.data_ptr(),
                      D.ws_sp.numel(), st))

    def step():
        q_dev.copy_(q_host, non_blocking=True)
        for c in calls:
            rc = L.sdkv_sparse_decode_attn(*c)
            if rc != 0:
                raise RuntimeError("sdkv_sparse_decode_attn: %s" % L.sdkv_last_error().decode())
        o_host.copy_(D.o_sp, non_blocking=True)
        l_host.copy_(D.l_sp, non_blocking=True)

    step()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    s.record()
    for _ in range(K):
        step()
    e.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(s.elapsed_time(e), world)
    return {"value": ms / K * 1e3, "unit": UNIT, "h2d_bytes_per_step": q_host.numel() * q_host.element_size(),
            "d2h_bytes_per_step": o_host.numel() * o_host.element_size() + l_host.numel() * l_host.element_size(),
            "steps": K, "path": "C ABI: sdkv_sparse_decode_attn per layer; decode queries copied from pinned "
                                "host memory and o, lse read back every step"}


def sparse_dense_block(D, kis, hbm_peak, reps, with_verify=False, with_select=False, flush=None):
    """Per-layer times of the sparse decode at each keep ratio, the dense decode
    and (optionally) the gamma verify and the prefill selection of workload D.
    `flush`: an L2-sized write before every replay (for steps whose inputs fit
    in L2)."""
    out = {}
    for ki in kis:
        g = capture(lambda: D.sparse_step(ki))
        us = time_graph(g, reps, flush)
        tag = ("keep_%dpct" % round(100 * D.w.keep[ki] / D.n)) if D.w.keep else "ragged"
        out[tag] = phase_record(us, D.L, D.alg_bytes("sparse", ki), hbm_peak)
        out[tag]["kept_per_head_mean"] = D.mean_total(ki) / D.BH
        del g
    g = capture(D.dense_step)
    out["dense"] = phase_record(time_graph(g, reps, flush), D.L, D.alg_bytes("dense"), hbm_peak)
    del g
    if with_verify:
        g = capture(D.verify_step)
        out["verify_gamma%d" % D.w.gamma] = phase_record(time_graph(g, reps, flush), D.L, D.alg_bytes("verify"),
                                                         hbm_peak)
        del g
    if with_select:
        g = capture(lambda: D.prefill_step(kis[0]))
        us = time_graph(g, reps, flush)
        out["prefill_select"] = {"us_per_sequence": us, "us_per_layer": us / D.L}
        del g
    for ws in D.workspaces():
        st = D.sk.workspace_status(ws)
        if st != 0:
            raise SystemExit("device status %d raised during the bench" % st)
    return out


def config_blocks(hbm_peak, dev, reps):
    """The other single-GPU workloads, each a separate measurement."""
    out = {}
    # Llama-3.1-8B shape at 128K: keep 10 / 30 / 50%, dense, gamma = 8 verify
    w = workloads.by_name("llama8b_128k")
    D = Decode(w, dev, verify=True)
    D.prefill((0, 1, 2))
    blk = sparse_dense_block(D, (0, 1, 2), hbm_peak, reps, with_verify=True, with_select=True)
    blk["sparse_vs_dense"] = {k: blk["dense"]["us_per_layer"] / v["us_per_layer"] for k, v in blk.items()
                              if k.startswith("keep_")}
    blk["byte_bound"] = {k: blk["dense"]["alg_bytes_per_layer"] / v["alg_bytes_per_layer"] for k, v in blk.items()
                         if k.startswith("keep_")}
    out["llama8b_128k"] = blk
    del D
    torch.cuda.empty_cache()
    # SparseMM: ragged head budgets, batch 8, 32 MHA heads; 8 distinct layers (4.3 GB of K/V each) cycled
    w = workloads.by_name("sparsemm")
    D = Decode(w, dev, distinct=8)
    D.prefill((0,))
    blk = sparse_dense_block(D, (0,), hbm_peak, max(3, reps // 4))
    blk["note"] = "8 distinct layers cycled over the 32 launches of a step; each layer's K/V (4.3 GB) exceeds L2"
    out["sparsemm"] = blk
    del D
    torch.cuda.empty_cache()
    # video (Qwen2-7B shape): the StD draft decode over 256 text + 768 visual, dense decode, gamma = 5 verify
    w = workloads.by_name("video")
    D = Decode(w, dev, verify=True)
    D.prefill((0,))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)   # the step's 59 MB of kept rows fit in L2
    blk = sparse_dense_block(D, (0,), hbm_peak, reps, with_verify=True, with_select=True, flush=flush)
    blk["note"] = "L2 flushed (256 MB write) before every replay"
    out["video"] = blk
    del flush
    del D
    torch.cuda.empty_cache()
    return out


def io_model(video, llama128):
    """The StD I/O model (3.3) for the video workload, and the measured
    counterparts: verify over dense decode (SpecVLM's T_t^gamma / T_t) and
    draft over dense decode (T_d / T_t), attention kernels only."""
    w = workloads.by_name("video")
    gamma, m_t, m_v = w.gamma, w.text_tokens, w.frames * w.frame_tokens
    K = w.keep[0] - m_t
    t_draft = next(v["us_per_layer"] for k, v in video.items() if k.startswith("keep_"))
    t_dense = video["dense"]["us_per_layer"]
    t_ver = video["verify_gamma%d" % gamma]["us_per_layer"]
    round_us = gamma * t_draft + t_ver
    res = {
        "io_model": {
            "workload": "video", "gamma": gamma, "K_visual": K, "m_t": m_t, "m_v": m_v,
            "io_sparse_entries": ba.std_io_sparse(gamma, K, m_t),
            "io_dense_entries": ba.std_io_dense(m_v, m_t),
            "io_total_entries": ba.std_io_total(gamma, K, m_t, m_v),
            "io_average_entries_alpha_1": ba.std_io_average(gamma, K, m_t, m_v, 1.0),
            "io_vanilla_entries_per_token": m_v + m_t,
            "alpha_threshold_io": ba.std_alpha_threshold(gamma, K, m_t, m_v),
            "measured_us_per_layer": {"draft_decode": t_draft, "verify": t_ver, "dense_decode": t_dense,
                                      "round": round_us},
            "alpha_threshold_time": round_us / (gamma * t_dense),
            "note": "alpha_threshold_time: the accepted fraction of the gamma drafts above which a round "
                    "(gamma draft decodes + one verify) costs less attention time per accepted token than "
                    "dense decoding; alpha_threshold_io is the page's entry-count condition",
        },
        "verify_over_dense": {
            "video_gamma5": t_ver / t_dense,
            "llama8b_128k_gamma8": llama128["verify_gamma8"]["us_per_layer"] / llama128["dense"]["us_per_layer"],
        },
        "draft_over_dense": {"video": t_draft / t_dense},
    }
    td, ttg = t_draft / t_dense, t_ver / t_dense
    res["sd_speedup_model_video"] = {"gamma": gamma, "td_over_tt": td, "ttg_over_tt": ttg,
                                     "by_accept_length": {str(tau): ba.sd_speedup(tau, gamma, td, ttg)
                                                          for tau in range(1, gamma + 2)},
                                     "note": "SpecVLM's speed-up model with the measured attention kernel times; "
                                             "the accept length needs a model and is not measured"}
    return res


def next_rows_timings(D, hbm_peak, dev):
    """Timings of the rows beyond the hot path (each a separate measurement):
      f1  compaction of the selected rows (once per selection) and the decode
          over the compacted rows, on the headline lists, every layer;
      f2  decode over sink + recent lists (4 + 64), every layer;
      f3  SpecVLM selection for one request of the video workload (28 layers x
          4 KV heads of window scores over 12,800 tokens, 12,544 of them video);
      f4  one StD round of the video workload per layer: 5 draft steps (list
          append on the device + sparse decode over the 1,024 kept + drafted
          rows) and the verify of the 5 drafts, in one graph."""
    sk = D.sk
    L, B, Hq, Hkv, d, n = D.L, D.B, D.Hq, D.Hkv, D.d, D.n
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    offs, idx, totals = D.lists[0]
    kc = [torch.empty((max(t, 1), d), dtype=torch.bfloat16, device=dev) for t in totals]
    vc = [torch.empty((max(t, 1), d), dtype=torch.bfloat16, device=dev) for t in totals]
    ws_c = sk.new_workspace(sk.workspace_size(sk.OP_COMPACT, B, 0, Hkv, d, 0, 0), dev)

    def compact():
        for l in range(L):
            lay = D.lay(l)
            sk.compact_kv(lay["k"], lay["v"], offs[l], idx[l], totals[l], k_out=kc[l], v_out=vc[l], ws=ws_c)

    def contig():
        for l in range(L):
            sk.sparse_decode_compact(D.lay(l)["q"], kc[l], vc[l], offs[l], Hkv, D.scale, o=D.o_sp[l],
                                     lse=D.l_sp[l], ws=D.ws_sp)
    t_comp = time_graph(capture(compact), 10, flush) / L
    t_contig = time_graph(capture(contig), 10, flush) / L
    mean_total = float(np.mean(totals))
    b_comp = 2 * mean_total * 4 * d                                  # read and write K and V rows
    b_contig = mean_total * 4 * d + B * Hq * 4 * d                   # K/V rows + q in / o out
    out["f1_compaction"] = {"us_per_layer": t_comp, "alg_bytes_per_layer": b_comp,
                            "gbs": b_comp / t_comp / 1e3, "frac_of_measured_hbm": b_comp / t_comp / 1e3 / hbm_peak}
    out["f1_contiguous_decode"] = {"us_per_layer": t_contig, "alg_bytes_per_layer": b_contig,
                                   "gbs": b_contig / t_contig / 1e3,
                                   "frac_of_measured_hbm": b_contig / t_contig / 1e3 / hbm_peak}
    assert sk.workspace_status(ws_c) == 0 and sk.workspace_status(D.ws_sp) == 0
    del kc, vc
    # f2
    w_offs, w_idx = sk.window_lists(B, Hkv, n, 4, 64, dev)

    def window():
        for l in range(L):
            lay = D.lay(l)
            sk.sparse_decode_attn(lay["q"], lay["k"], lay["v"], w_offs, w_idx, D.scale, o=D.o_sp[l],
                                  lse=D.l_sp[l], ws=D.ws_sp)
    t_win = time_graph(capture(window), 10, flush) / L
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
    t_spec = time_graph(capture(spec), 10, flush)
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
    t_round = time_graph(capture(round_), 10, flush)
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
    ki = args.keep_index
    D = Decode(w, dev)
    D.prefill((ki,))
    step_graph = capture(lambda: D.sparse_step(ki))          # the decode step: a4 of every layer
    warm = max(args.warmup, 3)
    K = args.steps
    for _ in range(warm):
        step_graph.replay()
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(args.clocks_log)
    time.sleep(0.25)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    start.record()
    for _ in range(K):
        step_graph.replay()
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    clocks = sampler.stop(t0, t1, uuid)
    us_step = max_over_ranks(start.elapsed_time(end), world) / K * 1e3
    for ws in D.workspaces():
        st = D.sk.workspace_status(ws)
        if st != 0:
            raise SystemExit("device status %d raised during the bench" % st)

    L = D.L
    reps = max(10, min(K, 50))
    breakdown = {"sparse": phase_record(us_step, L, D.alg_bytes("sparse", ki), hbm_peak)}
    breakdown["sparse"]["kept_per_head_mean"] = D.mean_total(ki) / D.BH
    g = capture(D.dense_step)
    breakdown["dense"] = phase_record(time_graph(g, reps), L, D.alg_bytes("dense"), hbm_peak)
    del g
    g = capture(D.score_all)
    breakdown["score"] = phase_record(time_graph(g, reps), L, D.alg_bytes("score"), hbm_peak)
    del g
    g = capture(lambda: D.select_all(ki))
    breakdown["select"] = phase_record(time_graph(g, reps), L, D.alg_bytes("select", ki), hbm_peak)
    del g
    prefill_us = breakdown["score"]["us_per_step"] + breakdown["select"]["us_per_step"]
    sp = breakdown["sparse"]
    roofline = {"bound": "hbm", "achieved": sp["gbs"], "peak": hbm_peak, "unit": "GB/s",
                "frac": sp["gbs"] / hbm_peak, "traffic": traffic_from_profiles("sparse", w.name),
                "kernel": "sdkv_sparse_decode_attn (gathered decode: attn_splitk_kernel, or packed_decode_kernel "
                          "for many lists)", "peak_kind": peak_kind,
                "alg_bytes_per_launch": sp["alg_bytes_per_layer"], "us_per_launch": sp["us_per_layer"]}
    line = {
        "metric": METRIC, "value": us_step, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": warm,
        "ms_per_step": us_step / 1e3, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, ki),
        "dense_decode_us_per_step": breakdown["dense"]["us_per_step"],
        "prefill_select": {"us_per_sequence": prefill_us, "us_per_layer": prefill_us / L,
                           "what": "a2 window scoring + a3 top-K selection of every layer, once per sequence"},
        "sparse_vs_dense": {
            "sparse_us_per_step": us_step,
            "dense_us_per_step": breakdown["dense"]["us_per_step"],
            "speedup": breakdown["dense"]["us_per_step"] / us_step,
            "byte_bound": D.alg_bytes("dense") / D.alg_bytes("sparse", ki),
            "sparse_frac_of_measured_hbm": sp["frac_of_measured_hbm"],
            "dense_frac_of_measured_hbm": breakdown["dense"]["frac_of_measured_hbm"],
            "sparse_frac_of_8tbs": sp["frac_of_8tbs_nominal"],
            "dense_frac_of_8tbs": breakdown["dense"]["frac_of_8tbs_nominal"],
        },
        "breakdown": breakdown,
        "roofline": roofline,
        "gpu_launches": L * K,
        "clocks": clocks,
    }
    if not args.no_e2e:
        line["e2e"] = run_e2e(D, ki, max(3, min(K, 20)), world)
    if rank == 0 and not args.no_next:
        line["next_rows"] = next_rows_timings(D, hbm_peak, dev)
    del D, step_graph
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_configs:
        cfg = config_blocks(hbm_peak, dev, 20)
        line["configs"] = cfg
        line.update(io_model(cfg["video"], cfg["llama8b_128k"]))
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, ki)
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
