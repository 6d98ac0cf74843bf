"""Benchmark of the DCOCO per-cycle hot path (corrected draft blocks per second).

One step = one whole correction cycle over one batch of synthetic drafter output:
top-K over the B x V logits of every stream, candidate representations, pair states, all
(B-1)K^2 transition scores, the prefix-first walk and greedy verification.  Default workload:
32 concurrent streams, B=16, K=16, V=151936, d=E=4096, r=256, H=512, bf16 inputs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica on its own streams (no collective on
the data path); the time is the max over ranks.  `--impl reference` times the float64 CPU
oracle on the host cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "corrected draft blocks/sec (B=16,K=16,32 streams) + % of HBM/tensor roofline"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, 1900.0, "fallback"


# ----------------------------------------------------------------------------- replicas (N ranks)


def rank_workload(cfg, rank: int):
    """Rank r runs its own replica on its own N streams: the input seeds are offset by r * N
    (the weights and the embedding table are the same on every rank)."""
    return cfg.replace(base_seed=cfg.base_seed + rank * cfg.N) if rank else cfg


def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The job's time for a region that every rank timed: the slowest rank's.  A collective
    (every rank calls it); with one rank, ms itself."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, n_streams: int, steps: int, ms: float) -> float:
    """Corrected draft blocks per second of the whole job: every rank's streams over the job's time."""
    return world * n_streams * steps / (ms / 1e3)


# ----------------------------------------------------------------------------- CPU oracle arm

ORACLE_SNIPPET = r"""
import json, os, sys, time
sys.path.insert(0, {root!r})
import numpy as np
import oracle, workloads as wl
cfg = wl.CONFIGS[{cfg!r}].replace(N=1)
n_streams, reps, budget, stream0, emb_path = {n_streams}, {reps}, {budget}, {stream0}, {emb_path!r}
emb = np.load(emb_path, mmap_mode="r") if emb_path else wl.embedding(cfg)
w = wl.weights(cfg)
f = lambda a: wl.to_f64(a, cfg.dtype)
W = {{k: f(v) for k, v in w.items()}}
streams = []
for n in range(stream0, stream0 + n_streams):
    c = cfg.replace(base_seed=cfg.base_seed + n)
    streams.append((wl.logits(c), wl.hidden(c)))
if {sync}:  # the processes of one run start their timed loops together, on the parent's word
    print("ready", flush=True)
    sys.stdin.readline()
times = []
while len(times) < reps and (budget <= 0 or sum(times) < budget):
    t0 = time.perf_counter()
    for lg, h in streams:
        vals, ids = oracle.topk(f(lg), cfg.K)
        uniq, inv = np.unique(ids, return_inverse=True)
        rep = oracle.candidate_repr(inv.reshape(ids.shape), f(emb[uniq]), f(h), W)
        s = oracle.pair_state(f(h), W)
        S = oracle.transition_scores(rep["z"], s, vals, W)
        k, tok = oracle.select(S, vals, ids)
        t = wl.verifier_tokens(cfg, tok)
        oracle.verify_greedy(tok, t)
    times.append(time.perf_counter() - t0)
print(json.dumps({{"times": times, "streams": n_streams}}))
"""


def _oracle_env():
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    return env


def run_oracle(cfg_name: str, n_streams: int, reps: int, budget_s: float = 0.0, emb_path: str = ""):
    """Times the oracle in a fresh single-threaded process (no CUDA context, no fork):
    `reps` repetitions, or fewer once `budget_s` seconds of timed work are done."""
    code = ORACLE_SNIPPET.format(root=ROOT, cfg=cfg_name, n_streams=n_streams, reps=reps, budget=budget_s, stream0=0,
                                 emb_path=emb_path, sync=False)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=_oracle_env())
    if res.returncode != 0:
        raise RuntimeError(f"oracle run failed:\n{res.stderr[-2000:]}")
    return json.loads(res.stdout.strip().splitlines()[-1])


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def run_oracle_all_cores(cfg_name: str, streams_per_proc: int, reps: int, budget_s: float, emb_path: str = "",
                         procs: int = 0, skip: int = 0):
    """The oracle on every host core: one single-threaded process per core, each on its own
    streams (process p owns streams p*s .. p*s+s-1), all starting their timed loops together.
    Returns the whole host's rate in blocks/s (the first `skip` repetitions of each process
    left out) and the process count."""
    procs = procs or host_cores()
    running = []
    for p in range(procs):
        code = ORACLE_SNIPPET.format(root=ROOT, cfg=cfg_name, n_streams=streams_per_proc, reps=reps, budget=budget_s,
                                     stream0=p * streams_per_proc, emb_path=emb_path, sync=True)
        running.append(subprocess.Popen([sys.executable, "-c", code], stdin=subprocess.PIPE, stdout=subprocess.PIPE,
                                        stderr=subprocess.PIPE, text=True, env=_oracle_env()))
    for pr in running:  # every process has built its inputs
        if pr.stdout.readline().strip() != "ready":
            pr.wait()
    for pr in running:
        if pr.poll() is None:
            pr.stdin.write("go\n")
            pr.stdin.flush()
    results = []
    for pr in running:
        out, err = pr.communicate()
        if pr.returncode != 0:
            raise RuntimeError(f"oracle run failed:\n{err[-2000:]}")
        results.append(json.loads(out.strip().splitlines()[-1]))
    # each process's timed loop runs concurrently with the others'; the host's rate is every
    # process's blocks over the longest loop
    blocks = sum(r["streams"] * len(r["times"][skip:]) for r in results)
    wall = max(sum(r["times"][skip:]) for r in results)
    return blocks / wall, procs


class EmbeddingFile:
    """The workload's embedding table written once to a temporary .npy file that every oracle
    process maps read-only, instead of each process drawing its own 1.2 GB copy."""

    def __init__(self, cfg, table=None):
        self.cfg, self.table, self.path = cfg, table, ""

    def __enter__(self):
        import tempfile
        d = "/dev/shm" if os.path.isdir("/dev/shm") and os.access("/dev/shm", os.W_OK) else tempfile.gettempdir()
        fd, self.path = tempfile.mkstemp(suffix=".npy", prefix="dcoco_emb_", dir=d)
        os.close(fd)
        np.save(self.path, wl.embedding(self.cfg) if self.table is None else self.table)
        return self.path

    def __exit__(self, *exc):
        if self.path and os.path.exists(self.path):
            os.unlink(self.path)


def reference_arm(args, cfg):
    """The oracle on every host core: one single-threaded process per core, one stream each;
    a step is every process's full cycle over its stream, so each step is a bounded sample of
    the workload (host cores x 1 of its streams)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    with EmbeddingFile(cfg) as emb_path:
        procs = min(host_cores(), cfg.N)
        reps = args.warmup + args.steps
        # warm-up repetitions are timed inside each process but left out of the rate below
        rate_all, procs = run_oracle_all_cores(cfg.name, 1, reps, 0.0, emb_path, procs=procs, skip=args.warmup)
    value = rate_all
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "blocks/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * procs / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(cfg),
            "cpu_baseline": {"value": value, "unit": "blocks/s", "cores": procs, "kind": "oracle",
                             "sample": f"{procs} of {cfg.N} streams per step (one full block each, one "
                                       f"single-threaded process per host core), same shapes and distributions"},
            "e2e": {"value": value, "unit": "blocks/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm


def captured_traffic(kernel: str):
    """DRAM bytes per launch (read + write) from the committed ncu capture of `kernel`, or
    None when the kernel's source has changed since that capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        with open(os.path.join(ROOT, "draft_correction_gb300", "csrc", rec["source"]), "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
        return rec["dram_bytes_per_launch"] if digest == rec["source_sha256"] else None
    except (OSError, KeyError, ValueError):
        return None



def cycle_work(cfg, w_h):
    """Algorithmic HBM bytes and tensor flops of one whole cycle (a1..a6, greedy verify).

    Bytes: the logits once, each candidate's embedding row once, the hidden states once, every
    weight once, the verifier tokens in and the committed tokens, accept lengths and commit
    counts out.  Flops: 2 x rows x in x out of every projection (W_e on the gathered rows, W_h on
    the slots, both halves of W_f, U and V on the candidates, W_pair on the slots' two halves,
    W on the pairs).  The transition MLP (SFU) and the walk are not counted."""
    esz = 2 if cfg.dtype == "bf16" else 4
    N, B, K, V, d, E, r, H = cfg.N, cfg.B, cfg.K, cfg.V, cfg.d, cfg.E, cfg.r, cfg.H
    weights = sum(int(np.asarray(v).size) for v in w_h.values()) * esz
    nbytes = (N * B * V * esz + N * B * K * E * esz + N * B * d * esz + weights
              + N * (B + 1) * 4 + N * (B + 1) * 4 + 2 * N * 4)
    M, NB, NP = N * B * K, N * B, N * (B - 1)
    flops = 2.0 * (M * E * r + NB * d * r + M * r * r + NB * r * r + 2 * M * r * H + NB * 2 * d * r + NP * r * H)
    return nbytes, flops


def cycle_roofline(cfg, ms_per_step, w_h):
    """The cycle's roofline: whichever of the HBM time and the tensor time of its algorithmic
    work is longer binds; achieved = that work over the measured step time."""
    hbm, bf16, kind = peaks()
    nbytes, flops = cycle_work(cfg, w_h)
    t_hbm, t_tensor = nbytes / (hbm * 1e9), flops / (bf16 * 1e12)
    sec = ms_per_step * 1e-3
    if t_hbm >= t_tensor:
        out = {"bound": "hbm", "achieved": round(nbytes / sec / 1e9, 1), "peak": hbm, "unit": "GB/s",
               "frac": round(t_hbm / sec, 4), "peak_source": f"{kind} hbm_gbs (burst)"}
    else:
        out = {"bound": "tensor", "achieved": round(flops / sec / 1e12, 1), "peak": bf16, "unit": "TFLOP/s",
               "frac": round(t_tensor / sec, 4), "peak_source": f"{kind} bf16_tflops (burst)"}
    out.update({"kernel": "whole cycle (one CUDA graph, a1..a6)", "traffic": None,
                "algorithmic_bytes_per_step": nbytes, "algorithmic_tensor_flops_per_step": flops,
                "hbm_time_us_at_peak": round(t_hbm * 1e6, 2), "tensor_time_us_at_peak": round(t_tensor * 1e6, 2),
                "measured_us_per_step": round(ms_per_step * 1e3, 2)})
    return out


def arithmetic(cfg):
    """The precision each part of the path computes in (the line's dtype names the inputs)."""
    if cfg.dtype == "bf16":
        return {"inputs": "bf16 logits, embeddings, hidden states and weights",
                "topk": "exact comparison of the bf16 values (64-bit value/index keys)",
                "projections": "bf16 operands on tcgen05, fp32 accumulation in tensor memory; LayerNorm and "
                               "SiLU epilogues in fp32; b, z, U z / V z stored in bf16",
                "scorer": "pre-activations, tanh.approx.f16x2 and 8-term partial sums in f16; per-output "
                          "totals in fp32 (stages_us.score_transitions_fp32 times the all-fp32 path)",
                "walk_verify": "fp32 comparisons; residual draws in exact 62-bit fixed point"}
    return {"inputs": "f32", "projections": "tf32 operands on tcgen05, fp32 accumulation",
            "scorer": "fp32 with tanh.approx.f32", "walk_verify": "fp32; residual draws in exact 62-bit fixed point"}


def config_dict(cfg):
    return {"workload": cfg.name, "streams": cfg.N, "B": cfg.B, "K": cfg.K, "V": cfg.V, "d": cfg.d, "E": cfg.E,
            "r": cfg.r, "H": cfg.H, "verify": "greedy", "parallelism": "replicas (streams sharded, no collective)",
            "l2": "flushed before every timed step: 256 MB written, then another 256 MB read, so the step "
                  "starts with no reusable and no dirty lines in L2"}


class ClockSampler:
    """nvidia-smi samples during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks = getattr(self, "marks", []) + [time.time()]

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        marks = getattr(self, "marks", [])
        lines = [ln for _, ln in self.lines]
        window = "whole measurement"
        if len(marks) >= 2:
            inside = [ln for t, ln in self.lines if marks[0] <= t <= marks[-1] + 0.2]
            if len(inside) >= 3:
                lines, window = inside, "timed loop"
            else:
                lines, window = [ln for t, ln in self.lines if t <= marks[-1] + 0.2], \
                    "timed loop and the 1 s of identical steps before it"
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, flag in zip(names, parts[3:7]):
                if flag.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "window": window}


def gpu_arm(args, cfg):
    import torch
    import torch.distributed as dist

    import draft_correction_gb300 as dc
    from draft_correction_gb300 import build as dcb

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        dcb.build()
    if world > 1:
        dist.barrier()
    dc.lib()

    # Inputs: every rank owns its own N streams (seeds offset by rank); table and weights shared.
    rcfg = rank_workload(cfg, rank)
    logits_h = wl.logits(rcfg)
    hidden_h = wl.hidden(rcfg)
    emb_h = wl.embedding(cfg)
    emb = dc.to_device(emb_h, cfg.dtype, dev)
    w_h = wl.weights(cfg)
    w = dc.CorrectorWeights.from_numpy(w_h, cfg.dtype, dev)
    logits = dc.to_device(logits_h, cfg.dtype, dev)
    hidden = dc.to_device(hidden_h, cfg.dtype, dev)
    cyc = dc.Cycle(w, cfg.N, cfg.B, cfg.K, cfg.V, device=dev, keep_intermediates=True)

    # Greedy verifier tokens drawn against this stream's own corrected draft.
    t_zero = torch.zeros((cfg.N, cfg.B + 1), dtype=torch.int32, device=dev)
    out = cyc.run(logits, emb, hidden, t=t_zero)
    torch.cuda.synchronize()
    t_host = wl.verifier_tokens(rcfg, out["tokens"].cpu().numpy())
    t_dev = dc.to_device(t_host, "i32", dev)

    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    flush_clean = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)  # float: no widening copy

    def flush_l2():
        # Writing a buffer larger than L2 evicts everything useful; reading a second one then
        # writes those dirty lines back before the timed region instead of inside it.
        flush.fill_(1)
        flush_clean.sum()

    # One cycle captured as a CUDA graph (11 kernels, no host work between them).
    for _ in range(2):
        cyc.run(logits, emb, hidden, t=t_dev)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cyc.run(logits, emb, hidden, t=t_dev)
    torch.cuda.synchronize()

    def timed_loop(fn, steps, warmup):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        for _ in range(warmup):
            flush_l2()
            fn()
        torch.cuda.synchronize()
        for s, e in ev:
            flush_l2()
            s.record(stream)
            fn()
            e.record(stream)
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in ev]

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # nvidia-smi samples every 200 ms: keep identical steps running for ~1 s before the
        # timed loop (untimed, part of the warm-up) so that the clock record is not empty
        t_end = time.time() + 1.0
        while time.time() < t_end:
            for _ in range(50):
                flush_l2()
                graph.replay()
            torch.cuda.synchronize()
        clk.mark()
        ms = timed_loop(graph.replay, args.steps, args.warmup)
        clk.mark()
    torch.cuda.synchronize()
    total_ms = max_over_ranks(sum(ms), world, dev)
    value = whole_job_rate(world, cfg.N, args.steps, total_ms)
    assert dc.device_status() == 0, "device status word reports a fault"

    # Variant: the per-vocabulary candidate table (LN(W_e Emb) computed once, outside the timed
    # region, as a weight preprocessing step); the same cycle otherwise.  Reported beside the
    # headline, which keeps the per-cycle projection of the gathered embedding rows.
    variants = {}
    if world == 1 and cfg.dtype == "bf16":
        table = dc.embedding_table(emb, w)
        for _ in range(2):
            cyc.run(logits, emb, hidden, t=t_dev, table=table)
        torch.cuda.synchronize()
        graph_t = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_t):
            cyc.run(logits, emb, hidden, t=t_dev, table=table)
        torch.cuda.synchronize()
        ms_t = timed_loop(graph_t.replay, args.steps, args.warmup)
        variants["precomputed_embedding_table"] = {
            "value": round(cfg.N * len(ms_t) / (sum(ms_t) / 1e3), 1), "unit": "blocks/s",
            "ms_per_step": round(sum(ms_t) / len(ms_t), 4),
            "note": "dcoco_cycle_table: rows of LN(W_e Emb), computed once per weights, gathered per cycle"}
        del table

        # Variant: the cycle from the drafter's hidden state.  Top-K is the fused output
        # projection (h [N,B,d] x W_lm [V,d]^T) and selection, so the logits never reach HBM;
        # the same hidden states feed the corrector.  W_lm is synthetic, ~N(0, (3/sqrt(d))^2).
        W_lm = dc.to_device(wl.lm_head(cfg), cfg.dtype, dev)
        for _ in range(2):
            cyc.run(None, emb, hidden, t=t_dev, W_lm=W_lm)
        torch.cuda.synchronize()
        graph_l = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_l):
            cyc.run(None, emb, hidden, t=t_dev, W_lm=W_lm)
        torch.cuda.synchronize()
        ms_l = timed_loop(graph_l.replay, args.steps, args.warmup)
        # the fused kernel pair alone (projection + per-range lists, then the merge)
        lm_vals = torch.empty((cfg.N, cfg.B, cfg.K), dtype=torch.float32, device=dev)
        lm_ids = torch.empty((cfg.N, cfg.B, cfg.K), dtype=torch.int32, device=dev)
        lm_ws = torch.empty((max(16, dc.lib().dcoco_lm_head_topk_workspace_size(1, cfg.N, cfg.B, cfg.V, cfg.K)),),
                            dtype=torch.uint8, device=dev)
        lm_steps = max(5, min(args.steps, 20))
        lm_ms = timed_loop(lambda: dc.lm_head_topk(hidden, W_lm, cfg.K, lm_vals, lm_ids, lm_ws), lm_steps, 2)
        lm_us = 1e3 * statistics.mean(lm_ms)
        lm_flops = 2.0 * cfg.N * cfg.B * cfg.V * cfg.d
        _, bf16_peak, peak_kind_t = peaks()
        lm_tf = lm_flops / (lm_us * 1e-6) / 1e12
        # for comparison: the unfused path, a cuBLAS projection writing bf16 logits, then top-K
        h2 = hidden.reshape(cfg.N * cfg.B, cfg.d)
        lg = torch.empty((cfg.N * cfg.B, cfg.V), dtype=hidden.dtype, device=dev)

        def unfused():
            torch.matmul(h2, W_lm.t(), out=lg)
            dc.topk(lg.view(cfg.N, cfg.B, cfg.V), cfg.K, vals=lm_vals, ids=lm_ids)

        un_us = 1e3 * statistics.mean(timed_loop(unfused, lm_steps, 2))
        # for comparison: the same fused kernel with one-CTA MMAs instead of CTA pairs
        prev_pair = dc.set_lm_pair(-1)
        try:
            ws1 = torch.empty((max(16, dc.lib().dcoco_lm_head_topk_workspace_size(1, cfg.N, cfg.B, cfg.V, cfg.K)),),
                              dtype=torch.uint8, device=dev)
            one_us = 1e3 * statistics.mean(
                timed_loop(lambda: dc.lm_head_topk(hidden, W_lm, cfg.K, lm_vals, lm_ids, ws1), lm_steps, 2))
        finally:
            dc.set_lm_pair(prev_pair)
        del ws1
        # the binding roof: W_lm streams once (HBM), the projection is a dense contraction (tensor)
        lm_bytes = cfg.V * cfg.d * (2 if cfg.dtype == "bf16" else 4) + cfg.N * cfg.B * cfg.d * 2
        hbm_peak, _, _ = peaks()
        if lm_flops / (bf16_peak * 1e12) >= lm_bytes / (hbm_peak * 1e9):
            lm_roof = {"bound": "tensor", "achieved": round(lm_tf, 1), "peak": bf16_peak, "unit": "TFLOP/s",
                       "frac": round(lm_tf / bf16_peak, 4), "peak_source": f"{peak_kind_t} bf16_tflops (burst)",
                       "algorithmic_flops_per_launch": lm_flops}
        else:
            lm_gbs = lm_bytes / (lm_us * 1e-6) / 1e9
            lm_roof = {"bound": "hbm", "achieved": round(lm_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                       "frac": round(lm_gbs / hbm_peak, 4), "peak_source": f"{peak_kind_t} hbm_gbs (burst)",
                       "algorithmic_bytes_per_launch": lm_bytes}
        lm_roof.update({"kernel": "lm_topk_kernel + lm_merge_kernel", "traffic": None})
        variants["fused_lm_head_topk"] = {
            "value": round(cfg.N * len(ms_l) / (sum(ms_l) / 1e3), 1), "unit": "blocks/s",
            "ms_per_step": round(sum(ms_l) / len(ms_l), 4),
            "kernel_us": round(lm_us, 1),
            "roofline": lm_roof,
            "unfused_cublas_projection_then_topk_us": round(un_us, 1),
            "one_cta_mma_kernel_us": round(one_us, 1),
            "note": "dcoco_cycle_lm: the cycle from the drafter's hidden state; W_lm [V, d] synthetic"}
        del W_lm, lg, lm_ws

    # Per-stage device times (same inputs, same launch configuration, L2 flushed).
    ids, vals = cyc.out["ids"], cyc.out["vals"]
    uz = torch.empty((cfg.N, cfg.B, cfg.K, cfg.H), dtype=w.act_dtype, device=dev)
    stage_steps = max(5, min(args.steps, 30))
    stages = {
        "topk": lambda: dc.topk(logits, cfg.K, vals=vals, ids=ids),
        "pair_state": lambda: dc.pair_state(hidden, w),
        "candidate_repr": lambda: dc.candidate_repr(ids, emb, hidden, w),
    }
    uzv = dc.candidate_repr(ids, emb, hidden, w)
    wsp = dc.pair_state(hidden, w)
    S = dc.score_transitions(uzv[0], uzv[1], wsp, vals, w)
    stages["score_transitions"] = lambda: dc.score_transitions(uzv[0], uzv[1], wsp, vals, w)
    stages["select"] = lambda: dc.select(S, vals, ids)
    if cfg.dtype == "bf16":
        # the same scores with float32 operands and arithmetic throughout (tanh.approx.f32), for
        # comparison with the half-precision transition MLP the bf16 path uses
        w32 = dc.CorrectorWeights.from_numpy({k: wl.bf16_to_f32(v) for k, v in w_h.items()}, "f32", dev)
        uz32, vz32 = uzv[0].float(), uzv[1].float()
        stages["score_transitions_fp32"] = lambda: dc.score_transitions(uz32, vz32, wsp, vals, w32)
    stages["verify"] = lambda: dc.verify(cyc.out["tokens"], t=t_dev)
    # the scope table's next rows at the same shape: whole-path rules and speculative sampling
    stages["select_path_global_sum"] = lambda: dc.select_path(S, vals, ids, "global_sum")
    stages["select_path_geometric"] = lambda: dc.select_path(S, vals, ids, "geometric", 0.75)
    if rank == 0:
        prng = np.random.default_rng(11)
        spec_V = cfg.V
        p_d = torch.softmax(torch.randn((cfg.N, cfg.B, spec_V), device=dev) * 2, dim=-1)
        q_d = torch.softmax(torch.randn((cfg.N, cfg.B + 1, spec_V), device=dev) * 2, dim=-1)
        u_d = torch.from_numpy(prng.random((cfg.N, cfg.B + 1, 2), dtype=np.float32)).to(dev)
        draft_d = torch.multinomial(p_d.reshape(-1, spec_V), 1).reshape(cfg.N, cfg.B).to(torch.int32)
        stages["verify_speculative"] = lambda: dc.verify_speculative(draft_d, p_d, q_d, u_d)
        stages["verify_stochastic"] = lambda: dc.verify(draft_d, q=q_d, u=u_d, mode=dc.VERIFY_STOCHASTIC)
    del uz
    stage_us = {k: 1e3 * statistics.mean(timed_loop(fn, stage_steps, 2)) for k, fn in stages.items()}

    # Roofline of the dominant kernel (top-K, HBM-bound): algorithmic bytes per launch.
    hbm, _, peak_kind = peaks()
    topk_bytes = cfg.N * cfg.B * cfg.V * (2 if cfg.dtype == "bf16" else 4) + cfg.N * cfg.B * cfg.K * 8
    topk_s = stage_us["topk"] * 1e-6
    achieved = topk_bytes / topk_s / 1e9
    roofline = {"bound": "hbm", "kernel": "topk_kernel", "achieved": round(achieved, 1), "peak": hbm,
                "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": captured_traffic("topk"),
                "peak_source": f"{peak_kind} hbm_gbs (burst)", "algorithmic_bytes_per_launch": topk_bytes}
    # The whole cycle (what the metric measures) against its own binding roof.
    roofline["cycle"] = cycle_roofline(cfg, total_ms / args.steps, w_h)

    # End to end through the public API: pinned host inputs -> device, cycle, results -> host.
    def pinned(a):
        if cfg.dtype == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).pin_memory()

    logits_pin = pinned(logits_h)
    hidden_pin = pinned(hidden_h)
    t_pin = torch.from_numpy(t_host).pin_memory()
    com_pin = torch.empty((cfg.N, cfg.B + 1), dtype=torch.int32).pin_memory()
    acc_pin = torch.empty((cfg.N,), dtype=torch.int32).pin_memory()

    # Double-buffered like a serving loop: while the cycle of step i runs on the compute stream,
    # step i+1's inputs are copied into the other buffer set on a copy stream.  Every step's
    # host-to-device copy and result read-back lies inside the timed region (the whole loop is
    # timed once, from before the first copy to after the last read-back); each step's 156 MB
    # of fresh logits is larger than L2, so no flush is needed between steps.
    in_sets = [(logits, hidden, t_dev), (torch.empty_like(logits), torch.empty_like(hidden), torch.empty_like(t_dev))]
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    used = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(b):
        lg_b, hd_b, t_b = in_sets[b]
        copy_stream.wait_event(used[b])
        with torch.cuda.stream(copy_stream):
            lg_b.copy_(logits_pin, non_blocking=True)
            hd_b.copy_(hidden_pin, non_blocking=True)
            t_b.copy_(t_pin, non_blocking=True)
            copied[b].record(copy_stream)

    def e2e_run(steps):
        for b in range(2):
            used[b].record(stream)
        copy_in(0)
        for i in range(steps):
            b = i & 1
            if i + 1 < steps:
                copy_in(1 - b)
            stream.wait_event(copied[b])
            lg_b, hd_b, t_b = in_sets[b]
            o = cyc.run(lg_b, emb, hd_b, t=t_b)
            com_pin.copy_(o["committed"], non_blocking=True)
            acc_pin.copy_(o["accept_len"], non_blocking=True)
            used[b].record(stream)

    e2e_steps = max(5, min(args.steps, 30))
    e2e_run(3)  # warm-up
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_val = whole_job_rate(world, cfg.N, e2e_steps, max_over_ranks(e0.elapsed_time(e1), world, dev))
    h2d = logits_h.nbytes + hidden_h.nbytes + t_host.nbytes
    d2h = com_pin.numel() * 4 + acc_pin.numel() * 4

    cpu = cpu_all = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        with EmbeddingFile(cfg, emb_h) as emb_path:
            # a bounded sample of about 10 s of host work: a few streams, repeated
            n_streams = min(2, cfg.N)
            r = run_oracle(cfg.name, n_streams, 200, budget_s=10.0, emb_path=emb_path)
            reps = len(r["times"])
            sec = statistics.mean(r["times"])
            cpu = {"value": n_streams / sec, "unit": "blocks/s", "cores": 1, "kind": "oracle",
                   "sample": f"{n_streams} of {cfg.N} streams, full cycle each, {reps} repetitions, "
                             f"single host thread"}
            # every host core: one single-threaded process per core, its own stream each, ~10 s
            procs = min(host_cores(), cfg.N)
            rate, procs = run_oracle_all_cores(cfg.name, 1, 200, 10.0, emb_path, procs=procs)
            cpu_all = {"value": rate, "unit": "blocks/s", "cores": procs, "kind": "oracle",
                       "sample": f"{procs} of {cfg.N} streams, one single-threaded process per host core "
                                 f"(of {host_cores()}), full cycle each, repeated for about 10 s"}
    del emb_h

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "blocks/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic",
                "config": config_dict(cfg), "roofline": roofline, "cpu_baseline": cpu,
                "cpu_baseline_all_cores": cpu_all, "arithmetic": arithmetic(cfg),
                "e2e": {"value": round(e2e_val, 1), "unit": "blocks/s", "h2d_bytes_per_step": h2d,
                        "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                        "pipeline": "inputs double-buffered: step i+1 copied while step i computes"},
                "gpu_launches": 11 * args.steps, "clocks": clk.summary(),
                "stages_us": {k: round(v, 2) for k, v in stage_us.items()},
                "step_ms_p10_p50_p90": [round(float(np.percentile(ms, q)), 4) for q in (10, 50, 90)],
                "variants": variants}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def sweep_arm(args):
    """The 42-point draft-correct-verify sweep on the headline shapes: corrected draft blocks/s of
    the whole cycle with greedy and with stochastic verification at every (N, B, K), one CUDA
    graph per point, L2 flushed before every step.  Prints one JSON line with every point."""
    import torch

    import draft_correction_gb300 as dc
    from draft_correction_gb300 import build as dcb

    dcb.build()
    dc.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    base = wl.HEADLINE
    emb = dc.to_device(wl.embedding(base), base.dtype, dev)
    w = dc.CorrectorWeights.from_numpy(wl.weights(base), base.dtype, dev)
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    flush_clean = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def timed(fn, steps, warmup):
        for _ in range(warmup):
            flush.fill_(1)
            flush_clean.sum()
            fn()
        torch.cuda.synchronize()
        ms = []
        for _ in range(steps):
            flush.fill_(1)
            flush_clean.sum()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return ms

    points = []
    hbm, _, _ = peaks()
    for n in wl.SWEEP_STREAMS:
        for b in wl.SWEEP_B:
            cfg_nb = base.replace(N=n, B=b)
            logits = dc.to_device(wl.logits(cfg_nb), base.dtype, dev)
            hidden = dc.to_device(wl.hidden(cfg_nb), base.dtype, dev)
            q = dc.to_device(wl.verifier_probs(cfg_nb), "f32", dev)
            u = dc.to_device(wl.uniforms(cfg_nb), "f32", dev)
            for k in wl.SWEEP_K:
                cfg = cfg_nb.replace(name=f"sweep_n{n}_b{b}_k{k}", K=k)
                cyc = dc.Cycle(w, n, b, k, cfg.V, device=dev, keep_intermediates=False)
                out = cyc.run(logits, emb, hidden, t=torch.zeros((n, b + 1), dtype=torch.int32, device=dev))
                torch.cuda.synchronize()
                t = dc.to_device(wl.verifier_tokens(cfg, out["tokens"].cpu().numpy()), "i32", dev)
                pt = {"workload": cfg.name, "streams": n, "B": b, "K": k}
                for mode, name, kw in ((dc.VERIFY_GREEDY, "greedy", {"t": t}),
                                       (dc.VERIFY_STOCHASTIC, "stochastic", {"q": q, "u": u})):
                    for _ in range(2):
                        cyc.run(logits, emb, hidden, mode=mode, **kw)
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        cyc.run(logits, emb, hidden, mode=mode, **kw)
                    torch.cuda.synchronize()
                    ms = timed(g.replay, args.steps, args.warmup)
                    pt[f"{name}_blocks_per_s"] = round(n * len(ms) / (sum(ms) / 1e3), 1)
                    pt[f"{name}_ms_per_cycle"] = round(sum(ms) / len(ms), 4)
                    del g
                # top-K share of the HBM roofline at this point (bf16 logits)
                pt["logits_mb"] = round(n * b * cfg.V * 2 / 1e6, 1)
                points.append(pt)
                del cyc
            del logits, hidden, q, u
    assert dc.device_status() == 0, "device status word reports a fault"
    print(json.dumps({"metric": METRIC, "sweep": points, "unit": "blocks/s", "n_gpus": 1, "steps": args.steps,
                      "warmup": args.warmup, "dtype": base.dtype, "data": "synthetic",
                      "l2": "flushed before every timed step", "hbm_peak_gbs": hbm}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=wl.HEADLINE.name, choices=sorted(wl.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="the 42-point (streams, B, K) sweep instead of one workload")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.sweep and args.impl == "ours":
        return sweep_arm(args)
    cfg = wl.CONFIGS[args.config]
    if args.impl == "reference":
        return reference_arm(args, cfg)
    return gpu_arm(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
