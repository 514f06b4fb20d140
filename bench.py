#!/usr/bin/env python3
"""Throughput of the batched verify-and-commit step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference] [--config 3]

One step = one pass of the whole hot path over one batch: row statistics, acceptance, first
rejection, residual/bonus draw, emit and the KV commit -- one spec_verify_sample_commit launch
(spec_verify_greedy_commit for greedy batches; trees and truncated sampling are followed by a
separate spec_commit_kv_lengths launch).
The default workload is sampling with B=128 sequences, gamma=4 drafts, V=128256, bf16 logits,
T=0.8 (295.5 MB of logits per step).  Prints one JSON line (rank 0).

Metric: verified draft rows per second (sum of gamma_b over the batch, per step) and the
achieved HBM bandwidth of the verify kernel: algorithmic bytes (every valid logit row read
once) divided by its CUDA-event duration, against the measured HBM copy bandwidth.

--impl reference times the float64 CPU oracle on all host cores instead, on a bounded sample
of the same workload per step (rank 0 only).  The native line's cpu_baseline times the same
oracle on one core and on all cores; its parity field compares one call's outputs with the
oracle on every sequence of the batch.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft rows/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "verify_sample_B128_g4_V128256_bf16_dram.txt")
KERNEL_SRC = os.path.join(ROOT, "speculative_decoding_verification_34_gb300", "csrc", "verify.cu")
# the verify kernel's sources: the kernel and the draw placement it compiles in
KERNEL_SRCS = (KERNEL_SRC, os.path.join(ROOT, "speculative_decoding_verification_34_gb300", "csrc", "schedule.h"))


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5, 6],
                    help="1-5: the sampling/greedy workloads; 6: 63-node draft trees (greedy tree verify)")
    ap.add_argument("--copies", type=int, default=4, help="resident input copies rotated per step")
    ap.add_argument("--top-k", type=int, default=0, help="truncated sampling: top-k on every sequence (0: off)")
    ap.add_argument("--top-p", type=float, default=1.0, help="truncated sampling: top-p on every sequence (1: off)")
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    return ap.parse_args()


def is_tree(wl):
    return hasattr(wl, "node_parents")


def workload_config(wl, l2_note):
    if is_tree(wl):
        return {"workload": wl.name, "B": wl.B, "tree_nodes": wl.nmax, "V": wl.V, "logits": wl.dtype,
                "temperature": 0.0, "algorithmic_bytes_per_step": wl.algorithmic_bytes(),
                "verified_rows_per_step": wl.verified_rows(), "l2": l2_note}
    c = {"workload": wl.name, "B": wl.B, "gamma": wl.gmax, "V": wl.V, "logits": wl.dtype,
         "temperature": float(wl.temperature.max()), "algorithmic_bytes_per_step": wl.algorithmic_bytes(),
         "verified_rows_per_step": wl.verified_rows(), "l2": l2_note}
    if getattr(wl, "top_k", None) is not None:
        c["top_k"], c["top_p"] = int(wl.top_k[0]), float(wl.top_p[0])
    return c


def oracle_one(wl, b):
    """The oracle on sequence b alone; returns the draft rows (or tree nodes) it judged."""
    from oracle import specverify_oracle as O
    if is_tree(wl):
        O.verify_tree_batch(wl.target, wl.dtype, wl.node_tokens, wl.node_parents, wl.num_nodes, seqs=[b])
        return int(wl.num_nodes[b])
    O.verify_batch(wl.target, wl.draft, wl.dtype, wl.draft_tokens, wl.num_draft,
                   None if wl.greedy_only else wl.temperature, wl.u_accept, wl.u_sample, seqs=[b],
                   top_k=getattr(wl, "top_k", None), top_p=getattr(wl, "top_p", None),
                   nan_masked=getattr(wl, "top_k", None) is not None)
    return int(wl.num_draft[b])


def apply_truncation(wl, args):
    """--top-k / --top-p: the same truncation for every sequence of a sampling workload."""
    import numpy as np
    if is_tree(wl) or wl.greedy_only or (args.top_k <= 0 and not (0.0 < args.top_p < 1.0)):
        return False
    wl.top_k = np.full(wl.B, args.top_k, dtype=np.int32)
    wl.top_p = np.full(wl.B, args.top_p, dtype=np.float32)
    wl.name = f"{wl.name}-topk{args.top_k}-topp{args.top_p:g}"
    return True


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if d.get("hbm_gbs"):
            return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy)"
    return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def code_sha256(*paths):
    """sha256 of C/CUDA sources (in order) with their comments removed and their whitespace
    collapsed, so that an edit of comments alone keeps a recorded measurement of the compiled
    code valid."""
    text = "\n".join(open(p, encoding="utf-8").read() for p in paths)
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":                       # string or character literal, escapes kept
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    code = " ".join("".join(out).split())
    return hashlib.sha256(code.encode("utf-8")).hexdigest()


def recorded_traffic(units_per_launch):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this exact
    kernel source; else None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    kv = {}
    for line in open(TRAFFIC_FILE, encoding="utf-8"):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("code_sha256") != code_sha256(*KERNEL_SRCS):
        return None
    try:
        return int(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None, period_ms=50):
        self.rows, self.proc, self.err = [], None, None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               f"-lms", str(period_ms)]
        if gpu_id is not None:
            cmd += ["-i", str(gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError as e:
            self.err = str(e)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.err or not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": self.err or "no nvidia-smi samples"}
        win = [r for t, r in self.rows if t0 <= t <= t1 + 0.05] or [r for _, r in self.rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, reasons = [], set()
        smax = None
        for r in win:
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def smi_gpu_id(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",")]
        if local_rank < len(ids):
            return ids[local_rank]
    return local_rank


def all_reduce_max(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_workload(config, rank):
    """Weak scaling: sequences are independent, so every rank verifies its own batch of the
    same shape (seeded by its rank); nothing is exchanged on the data path."""
    from speculative_decoding_verification_34_gb300 import workloads as W
    return W.WORKLOADS[config](seed=rank)


def aggregate_rate(world, rows_per_step, steps, max_elapsed_ms):
    """Whole-job rows/s: the rows all ranks verified over the slowest rank's time."""
    return world * rows_per_step * steps / (max_elapsed_ms / 1e3)


def cpu_oracle_rate(wl, seconds, seqs_cap=None):
    """Oracle throughput on one core over a bounded sample of the batch: rows/s, sequences used."""
    t0 = time.perf_counter()
    n = rows = 0
    order = list(range(wl.B))
    while True:
        b = order[n % wl.B]
        rows += oracle_one(wl, b)
        n += 1
        el = time.perf_counter() - t0
        if (el >= seconds and n >= 2) or (seqs_cap and n >= seqs_cap):
            return rows / el, n, rows, el


# ---- the oracle on all host cores: one spawned process per core, the logits shared ----------

_POOL_STATE = {}
_BIG = ("target", "draft")


def _pool_init(root, meta, shm_specs):
    if root not in sys.path:
        sys.path.insert(0, root)
    import types
    from multiprocessing import shared_memory

    import numpy as np
    arrays = {}
    for name, (shm_name, shape, dt) in shm_specs.items():
        shm = shared_memory.SharedMemory(name=shm_name)   # the parent unlinks it
        _POOL_STATE["shm_" + name] = shm
        arrays[name] = np.ndarray(shape, dtype=np.dtype(dt), buffer=shm.buf)
    _POOL_STATE["wl"] = types.SimpleNamespace(**meta, **arrays)


def _pool_task(seqs):
    wl = _POOL_STATE["wl"]
    return sum(oracle_one(wl, b) for b in seqs)


class OraclePool:
    """A spawn-context process pool over the host cores with the workload's logits in shared
    memory (spawn, not fork: the parent has already initialised CUDA)."""

    def __init__(self, wl, procs=None):
        import multiprocessing as mp
        from multiprocessing import shared_memory

        import numpy as np
        self.procs = procs or len(os.sched_getaffinity(0))
        self.shms, specs, meta = [], {}, {}
        for k, v in vars(wl).items():
            if k in _BIG and isinstance(v, np.ndarray):
                shm = shared_memory.SharedMemory(create=True, size=max(1, v.nbytes))
                np.ndarray(v.shape, dtype=v.dtype, buffer=shm.buf)[...] = v
                self.shms.append(shm)
                specs[k] = (shm.name, v.shape, v.dtype.str)
            else:
                meta[k] = v
        from concurrent.futures import ProcessPoolExecutor
        # an executor, not multiprocessing.Pool: a worker that dies raises here instead of being
        # replaced forever
        self.pool = ProcessPoolExecutor(self.procs, mp_context=mp.get_context("spawn"),
                                        initializer=_pool_init, initargs=(ROOT, meta, specs))
        list(self.pool.map(_pool_task, [[] for _ in range(self.procs)]))   # every worker started

    def run(self, seqs):
        """Verify the listed sequences over all workers; returns (rows, seconds)."""
        chunks = [seqs[i::self.procs] for i in range(self.procs)]
        t0 = time.perf_counter()
        rows = sum(self.pool.map(_pool_task, chunks))
        return rows, time.perf_counter() - t0

    def close(self):
        self.pool.shutdown(wait=True, cancel_futures=True)
        for shm in self.shms:
            shm.close()
            shm.unlink()


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(wl, seconds, runs=3):
    """The oracle timed on one core and on all cores (processes over sequences), each as the
    median of `runs` runs over a bounded sample of the batch, about `seconds` in total."""
    per = max(0.2, seconds / (2 * runs))
    single = [cpu_oracle_rate(wl, per)[0] for _ in range(runs)]
    r1 = statistics.median(single)
    rows_per_seq = max(1.0, wl.verified_rows() / wl.B)
    pool = OraclePool(wl)
    try:
        n = max(pool.procs, int(round(per * r1 * pool.procs / rows_per_seq)))
        seqs = [i % wl.B for i in range(n)]
        allc = []
        for _ in range(runs):
            rows, el = pool.run(seqs)
            allc.append(rows / el)
    finally:
        pool.close()
    return {"value": r1, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "value_all": statistics.median(allc), "cores_all": pool.procs, "runs": runs,
            "runs_single": single, "runs_all": allc, "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "sample": f"median of {runs} runs per leg: one core cycling over the batch's {wl.B} sequences "
                      f"for {per:.1f} s a run; {pool.procs} processes over {n} sequence verifications a run; "
                      f"float64 numpy oracle"}


def parity_record(wl, gpu, tol=1e-5):
    """The GPU outputs of one call against the oracle on every sequence of the batch: decisions
    whose oracle margin is below tol are flagged (either branch is correct there) and counted;
    every other sequence must match exactly.  Also alpha = sum min(p, q) per draft row (the
    acceptance rate of that row) and the closed-form expected emit 1 + sum_j prod_{i<j} alpha_i
    beside the measured mean emit."""
    import math

    import numpy as np
    from oracle import specverify_oracle as O
    flagged = differ = mismatch = 0
    perr = 0.0
    if is_tree(wl):
        res = O.verify_tree_batch(wl.target, wl.dtype, wl.node_tokens, wl.node_parents, wl.num_nodes)
    else:
        res = O.verify_batch(wl.target, wl.draft, wl.dtype, wl.draft_tokens, wl.num_draft,
                             None if wl.greedy_only else wl.temperature, wl.u_accept, wl.u_sample,
                             top_k=getattr(wl, "top_k", None), top_p=getattr(wl, "top_p", None),
                             nan_masked=getattr(wl, "top_k", None) is not None)
    g_all = gpu["out"].shape[1] - 1
    for b, r in enumerate(res):
        want = np.full(g_all + 1, -1)
        want[: len(r.tokens)] = r.tokens
        same = (int(gpu["m"][b]) == r.m and np.array_equal(gpu["out"][b], want)
                and int(gpu["status"][b]) == r.status)
        fl = (not is_tree(wl)) and r.flagged(tol)
        flagged += fl
        differ += fl and not same
        mismatch += (not fl) and not same
        if not is_tree(wl) and not r.greedy and gpu.get("diag") is not None:
            for i in range(r.gamma):
                if not math.isnan(r.p_draft[i]):
                    perr = max(perr, abs(float(gpu["diag"][b][2 * i]) - r.p_draft[i]),
                               abs(float(gpu["diag"][b][2 * i + 1]) - r.q_draft[i]))
    rec = {"checked": len(res), "flagged": flagged, "differ": differ, "mismatch": mismatch,
           "margin": tol, "prob_max_abs_err": perr,
           "sample": f"every sequence of one call ({len(res)}), float64 oracle"}
    if not is_tree(wl) and not wl.greedy_only:
        alphas, expect = [], []
        for b in range(wl.B):
            T = float(wl.temperature[b])
            g = min(max(int(wl.num_draft[b]), 0), wl.gmax)
            if not T > 0:
                continue
            run, e = 1.0, 1.0
            for i in range(g):
                P = O.widen(wl.target[b, i], wl.dtype)
                Q = O.widen(wl.draft[b, i], wl.dtype)
                tk = int(wl.top_k[b]) if getattr(wl, "top_k", None) is not None else 0
                tp = float(wl.top_p[b]) if getattr(wl, "top_p", None) is not None else 1.0
                p = O.truncated_distribution(P, T, tk, tp)[0]
                q = O.truncated_distribution(Q, T, tk, tp)[0]
                a = float(np.minimum(p, q).sum())
                alphas.append(a)
                run *= a
                e += run
            expect.append(e)
        m = gpu["m"][np.asarray(wl.temperature) > 0]
        rec["alpha_mean"] = statistics.fmean(alphas) if alphas else None
        rec["expected_emitted_per_sampling_sequence"] = statistics.fmean(expect) if expect else None
        rec["measured_emitted_per_sampling_sequence"] = float(m.mean()) + 1.0 if len(m) else None
    return rec


# ------------------------------------------------------------------------------------------

def run_reference(args):
    """The float64 oracle as it stands, on all host cores (one spawned process per core, over
    sequences), each step a bounded sample of the workload's sequences."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from speculative_decoding_verification_34_gb300 import workloads as W
    wl = W.WORKLOADS[args.config](seed=0)
    apply_truncation(wl, args)
    pool = OraclePool(wl)
    try:
        # size each step so that the whole run stays within ~150 s: whole sequences, at least
        # one per process
        t0 = time.perf_counter()
        oracle_one(wl, 0)
        t_seq = time.perf_counter() - t0
        per_step = int(150.0 / max(1, args.steps + args.warmup) / max(t_seq, 1e-6) * pool.procs)
        per_step = max(pool.procs, min(per_step, wl.B * pool.procs))
        nxt = [0]

        def step():
            seqs = [(nxt[0] + i) % wl.B for i in range(per_step)]
            nxt[0] += per_step
            return pool.run(seqs)[0]

        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        rows = sum(step() for _ in range(args.steps))
        el = time.perf_counter() - t0
    finally:
        pool.close()
    value = rows / el
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, "CPU oracle: host memory"),
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": pool.procs, "kind": "oracle",
                             "cpu_model": cpu_model(), "nproc": os.cpu_count(),
                             "sample": f"{per_step} sequence verifications per step cycling over the batch's "
                                       f"{wl.B} sequences, {pool.procs} processes, float64 numpy oracle"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_native(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_34_gb300 import build
    from speculative_decoding_verification_34_gb300 import specverify as sv
    from speculative_decoding_verification_34_gb300 import workloads as W

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    sv.load_library()

    wl = shard_workload(args.config, rank)
    tree = is_tree(wl)
    trunc = apply_truncation(wl, args)
    B, g, V = wl.B, (wl.nmax if tree else wl.gmax), wl.V

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(np.ascontiguousarray(a)).to(device)

    ncopies = max(1, args.copies)
    tgt = [to_dev(wl.target) for _ in range(ncopies)]
    if tree:
        drf, temp, ua, us = None, None, None, None
        toks, nd, pars = to_dev(wl.node_tokens), to_dev(wl.num_nodes), to_dev(wl.node_parents)
        path = torch.empty((B, g), dtype=torch.int32, device=device)
    else:
        drf = [to_dev(wl.draft) for _ in range(ncopies)] if not wl.greedy_only else None
        toks, nd = to_dev(wl.draft_tokens), to_dev(wl.num_draft)
        temp, ua, us = to_dev(wl.temperature), to_dev(wl.u_accept), to_dev(wl.u_sample)
    kv0 = to_dev(wl.kv_len)
    out = torch.empty((B, g + 1), dtype=torch.int32, device=device)
    macc = torch.empty(B, dtype=torch.int32, device=device)
    st = torch.empty(B, dtype=torch.int32, device=device)
    dg = torch.empty((B, 2 * g + 1), dtype=torch.float32, device=device)
    kv = kv0.clone()
    dkv = kv0.clone()
    stream = torch.cuda.current_stream(device)
    ws = sv.alloc_workspace(B, g, V, sv.SPEC_BF16 if wl.dtype == "bf16" else sv.SPEC_F32, device)
    if tree:
        # tree verification and the commit of the round in one launch
        verify = [sv.prepare_verify_tree_greedy_commit(tgt[c], toks, pars, nd, out, macc, kv, dkv, True,
                                                       path_nodes=path, status=st, workspace=ws, stream=stream)
                  for c in range(ncopies)]
    elif wl.greedy_only:
        # verification and the commit of the round in one launch
        verify = [sv.prepare_verify_greedy_commit(tgt[c], toks, nd, out, macc, kv, dkv, True, status=st,
                                                  workspace=ws, stream=stream) for c in range(ncopies)]
    elif trunc:
        # truncated verification and the commit of the round: its two launches
        tk, tp = to_dev(wl.top_k), to_dev(wl.top_p)
        verify = [sv.prepare_verify_sample_truncated_commit(tgt[c], drf[c], toks, nd, temp, tk, tp, ua, us, out, macc,
                                                            kv, dkv, True, diag=dg, status=st, workspace=ws,
                                                            stream=stream) for c in range(ncopies)]
    else:
        verify = [sv.prepare_verify_sample_commit(tgt[c], drf[c], toks, nd, temp, ua, us, out, macc, kv, dkv, True,
                                                  diag=dg, status=st, workspace=ws, stream=stream)
                  for c in range(ncopies)]
    # every path has a fused call: a step is one verify call (a separate commit launch would
    # only be timed where none existed)
    fused = True
    commit = sv.prepare_commit_kv_lengths(macc, kv, dkv, True, stream=stream, gmax=g)
    step_commit = None if fused else commit

    for i in range(args.warmup):
        verify[i % ncopies]()
        if step_commit:
            step_commit()
    torch.cuda.synchronize(device)
    mean_emit = float(macc.float().mean().item()) + 1.0

    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(smi_gpu_id(local))
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(device)
    n0 = sv.spec_launch_count()
    w0 = time.time()
    # the steps alone, bracketed by one pair of events: ms_per_step and the headline value
    start.record(stream)
    for i in range(K):
        verify[i % ncopies]()
        if step_commit:
            step_commit()
    end.record(stream)
    torch.cuda.synchronize(device)
    launches = sv.spec_launch_count() - n0
    if world > 1:
        dist.barrier()
    # the same K steps again with an event pair around each verify launch: the kernel's own
    # duration for the roofline (these events are kept out of the step timing above)
    for i in range(K):
        ev0[i].record(stream)
        verify[i % ncopies]()
        ev1[i].record(stream)
        if step_commit:
            step_commit()
    torch.cuda.synchronize(device)
    w1 = time.time()
    if world > 1:
        dist.barrier()
    sampler.stop()
    clocks = sampler.summary(w0, w1)

    elapsed_ms = start.elapsed_time(end)
    kern_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    kern_mean_ms = statistics.fmean(kern_ms)
    kern_med_ms = statistics.median(kern_ms)
    ks = sorted(kern_ms)
    kern_p10, kern_p90 = ks[len(ks) // 10], ks[(9 * len(ks)) // 10]
    outliers = sum(1 for x in ks if x > 1.05 * kern_med_ms)
    elapsed_ms = all_reduce_max(elapsed_ms, world, device)
    kern_mean_ms = all_reduce_max(kern_mean_ms, world, device)

    rows_step = wl.verified_rows()
    value = aggregate_rate(world, rows_step, K, elapsed_ms)
    abytes = wl.algorithmic_bytes()
    peak, peak_src = measured_peak()
    # The verify call's average duration.  Where a step is exactly one verify call and nothing
    # else (the fused calls: one launch, or the truncated call's two), the timed region's length
    # over K is that average, the gap to the next call included.  Otherwise (a separate commit
    # launch in the step: trees) the per-launch event pairs give it.  An event pair around a
    # launch adds its own time, measured here on an empty pair.
    one_launch_per_step = fused and launches == K * (2 if trunc else 1)
    region_ms = elapsed_ms / K
    kern_avg_ms = region_ms if one_launch_per_step else kern_mean_ms
    achieved = abytes / (kern_avg_ms / 1e3) / 1e9
    torch.cuda.synchronize(device)
    ee = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(200)]
    torch.cuda._sleep(int(2e6))
    for a_, b_ in ee:
        a_.record(stream)
        b_.record(stream)
    torch.cuda.synchronize(device)
    empty_pair_us = statistics.median(a_.elapsed_time(b_) for a_, b_ in ee) * 1e3

    # ---- the post-verify kernels alone (stops, commit), per launch, on the same stream ----
    # Each batch of launches is queued behind a verify call, so the GPU runs them back to back
    # and the events around each one measure device time, not the host's launch gaps.
    budgets = torch.full((B,), 3, dtype=torch.int32, device=device)
    stops = sv.prepare_apply_stops(out, macc, 0, budgets, st, stream=stream)

    def per_launch_us(fn, batches=25, per=8):
        for _ in range(10):
            fn()
        times = []
        for _ in range(batches):
            e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(per)]
            verify[0]()
            for a, b_ in e:
                a.record(stream)
                fn()
                b_.record(stream)
            torch.cuda.synchronize(device)
            times += [a.elapsed_time(b_) for a, b_ in e]
        return statistics.median(times) * 1e3
    post = {"spec_apply_stops_us": per_launch_us(stops), "spec_commit_kv_lengths_us": per_launch_us(commit),
            "statistic": "median of 200 launches queued behind a verify call"}

    # ---- end to end through the public binding, host buffers, copies inside the region ----
    pin = lambda a: (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16
                     else torch.from_numpy(np.ascontiguousarray(a))).pin_memory()
    if tree:
        h_in = [pin(wl.target), pin(wl.node_tokens), pin(wl.node_parents), pin(wl.num_nodes), pin(wl.kv_len)]
        d_in = [tgt[0], toks, pars, nd, kv]
    elif wl.greedy_only:
        h_in = [pin(wl.target), pin(wl.draft_tokens), pin(wl.num_draft), pin(wl.kv_len)]
        d_in = [tgt[0], toks, nd, kv]
    else:
        h_in = [pin(wl.target), pin(wl.draft), pin(wl.draft_tokens), pin(wl.num_draft),
                pin(wl.temperature), pin(wl.u_accept), pin(wl.u_sample), pin(wl.kv_len)]
        d_in = [tgt[0], drf[0], toks, nd, temp, ua, us, kv]
    h_out = [torch.empty_like(out, device="cpu").pin_memory(), torch.empty_like(macc, device="cpu").pin_memory(),
             torch.empty_like(kv, device="cpu").pin_memory()]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out)

    def e2e_step():
        for h, d in zip(h_in, d_in):
            d.copy_(h, non_blocking=True)
        if tree:
            sv.spec_verify_tree_greedy_commit(d_in[0], d_in[1], d_in[2], d_in[3], out, macc, kv, None, True,
                                              path_nodes=path, status=st, workspace=ws)
        elif wl.greedy_only:
            sv.spec_verify_greedy_commit(d_in[0], d_in[1], d_in[2], out, macc, kv, None, True, status=st,
                                         workspace=ws)
        elif trunc:
            sv.spec_verify_sample_truncated_commit(d_in[0], d_in[1], d_in[2], d_in[3], d_in[4], tk, tp, d_in[5],
                                                   d_in[6], out, macc, kv, None, True, diag=dg, status=st,
                                                   workspace=ws)
        else:
            sv.spec_verify_sample_commit(d_in[0], d_in[1], d_in[2], d_in[3], d_in[4], d_in[5], d_in[6],
                                         out, macc, kv, None, True, diag=dg, status=st, workspace=ws)
        if not fused:
            sv.spec_commit_kv_lengths(macc, kv, None, True, gmax=g)
        h_out[0].copy_(out, non_blocking=True)
        h_out[1].copy_(macc, non_blocking=True)
        h_out[2].copy_(kv, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(device)
    if world > 1:
        dist.barrier()
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    ee.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms = all_reduce_max(es.elapsed_time(ee), world, device)
    e2e_value = aggregate_rate(world, rows_step, args.e2e_steps, e2e_ms)

    # ---- the outputs of one call (every input copy holds the same data) against the oracle ----
    verify[0]()
    torch.cuda.synchronize(device)
    gpu_out = {"out": out.cpu().numpy(), "m": macc.cpu().numpy(), "status": st.cpu().numpy(),
               "diag": None if (tree or wl.greedy_only) else dg.cpu().numpy()}

    cpu = parity = None
    if rank == 0:
        parity = parity_record(wl, gpu_out)
    if rank == 0 and world == 1:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    if rank == 0:
        traffic = recorded_traffic(1)
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
            "data": "synthetic",
            "config": workload_config(wl, f"inputs larger than L2 ({abytes / 1e6:.1f} MB of logits per step), "
                                          f"rotated over {ncopies} resident copies"),
            "hbm_gbs": achieved, "hbm_frac_of_measured_peak": achieved / peak,
            "sequences_per_s": world * B * K / (elapsed_ms / 1e3), "mean_emitted_per_sequence": mean_emit,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": ("verify_kernel<bf16, vec, greedy> with the commit (spec_verify_tree_greedy_commit)" if tree
                                    else "trunc_rows + trunc_draw kernels with the commit (spec_verify_sample_truncated_commit)"
                                    if trunc
                                    else "verify_kernel<bf16, vec, greedy> with the commit (spec_verify_greedy_commit)"
                                    if wl.greedy_only
                                    else "verify_kernel<bf16, vec, mixed> with the commit (spec_verify_sample_commit)"),
                         "kernel_ms": kern_avg_ms,
                         "kernel_ms_source": ("timed region / launches: one verify launch per step, back to back"
                                              if one_launch_per_step and not trunc
                                              else "timed region / steps: one truncated call (two launches) per step"
                                              if one_launch_per_step else "mean of per-launch event pairs"),
                         "kernel_ms_mean": kern_mean_ms, "kernel_ms_median": kern_med_ms,
                         "kernel_ms_p10": kern_p10, "kernel_ms_p90": kern_p90, "kernel_ms_max": ks[-1],
                         "frac_per_launch_events_mean": abytes / (kern_mean_ms / 1e3) / 1e9 / peak,
                         "frac_of_median": abytes / (kern_med_ms / 1e3) / 1e9 / peak,
                         "empty_event_pair_us": empty_pair_us,
                         "launches_timed": len(ks), "launches_above_1p05_median": outliers,
                         "slowest_launches_ms": ks[-3:],
                         "kernel_timing": "kernel_ms_mean/median/p10/p90/max: a second pass of the K steps with an "
                                          "event pair around each verify launch (each pair adds its own time: "
                                          "empty_event_pair_us)",
                         "algorithmic_bytes_per_launch": abytes, "peak_source": peak_src},
            "step_minus_kernel_median_ms": elapsed_ms / K - kern_med_ms,
            "step_minus_kernel_mean_ms": elapsed_ms / K - kern_mean_ms,
            "cpu_baseline": cpu, "parity": parity,
            "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": args.e2e_steps},
            "gpu_launches": launches, "clocks": clocks, "post_kernels": post,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
