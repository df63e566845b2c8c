"""Benchmark of the CSA indexer hot path (fused score + per-row top-k).

Default workload: long-context prefill, B=2, S=16384, compress_rate 4
(W=4096), H=64, D=128, top_k=2048, seeded N(0,1) bf16 inputs; one step is one
``csa_index_fused`` call over the whole batch (scores never written to HBM).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  ``value`` is useful causal TFLOP/s,
2*H*D*(visible (s,t) pairs) / time, with inputs resident in HBM; ``e2e`` is
the same metric through the host-buffer entry point (csa_index_fused_host:
pinned host inputs in, indices back in pinned host memory), with every
step's host<->device copies inside the timed region.  Under torchrun every rank runs its own
replica of the workload by default (rows and batches are independent; no
collective on the data path), so scaling is weak and ``value`` sums all
ranks' work over the slowest rank's time; with ``--shard rows`` the ranks
split the query rows of one problem instead (strong scaling; the shards'
indices are gathered and checked against one full call after the timed
region).  ``--impl reference`` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from csa_inputs import WORKLOADS, Inputs, make_inputs  # noqa: E402

METRIC = "indexer useful TFLOP/s and query rows/s at S=16K; % of bf16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + write) per timed unit come from the ncu launch lists
# summarised in profiles/: each summary carries a line
#     bench-traffic: <workload> <bytes> sources=<hash>
# (prefill_16k: per launch of the fused kernel; decode_32k: per step, the
# score launch plus the selection launch, the span its roofline is timed
# over).  <hash> is forward_sources_hash() of the build that was profiled; a
# figure whose hash differs from the current sources is stale and reported
# as null.
FORWARD_SOURCES = ("csa_ptx.cuh", "csa_select.cuh", "csa_score_kernel.cuh", "csa_prefill.cu", "csa_topk.cu",
                   "csa_api.cu", "csa_internal.h")


def forward_sources_hash() -> str:
    """Hash of the sources of the forward kernels and their launch code."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_indexer_csa_gb300", "csrc")
    for name in FORWARD_SOURCES:
        h.update(name.encode())
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def measured_traffic(workload: str):
    """DRAM bytes per timed unit of `workload` from profiles/, or None."""
    pat = re.compile(r"^bench-traffic:\s+(\S+)\s+([0-9.eE+]+)\s+sources=(\w+)")
    cur = forward_sources_hash()
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                m = pat.match(line.strip())
                if m and m.group(1) == workload and m.group(3) == cur:
                    return float(m.group(2))
    return None

# ----------------------------------------------------------------------------- work accounting
def visible_counts(inp: Inputs) -> np.ndarray:
    """v[b,s]: visible entries per row (future mask and segment ids), counted
    from the inputs with plain integer arithmetic."""
    wl = inp.wl
    start = np.zeros(wl.B, dtype=np.int64) if inp.q_start is None else inp.q_start.numpy()
    pos = start[:, None] + np.arange(wl.S)[None, :]
    thr = np.clip((pos + 1) // wl.compress_rate, 0, wl.W)
    if inp.q_seg is None:
        return thr
    v = np.zeros((wl.B, wl.S), dtype=np.int64)
    kv = inp.kv_seg.numpy()
    qs = inp.q_seg.numpy()
    for b in range(wl.B):
        for seg in np.unique(qs[b]):
            match = np.cumsum(kv[b] == seg)  # entries of this segment among t < n
            rows = qs[b] == seg
            tb = thr[b, rows]
            v[b, rows] = np.where(tb > 0, match[np.maximum(tb - 1, 0)], 0)
    return v


def work(inp: Inputs):
    wl = inp.wl
    v = visible_counts(inp)
    pairs = int(v.sum())
    nontrivial = int(v[v > wl.top_k].sum())
    per_pair = 2.0 * wl.H * wl.D
    return dict(pairs=pairs, flops=per_pair * pairs, flops_nontrivial=per_pair * nontrivial,
                rows=wl.B * wl.S, nontrivial_rows=int((v > wl.top_k).sum()))


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                return json.load(f), "measured"
        except Exception:
            pass
    return FALLBACK_PEAKS, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed plumbing
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return rank, world, local, dist
    return 0, 1, 0, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------------- CPU oracle timing
def oracle_sample(inp: Inputs, budget_s: float, block: int = 256, seed: int = 0):
    """Time the CPU oracle (fp64 scores + full-sort selection) on random row
    blocks of batch 0 until `budget_s` seconds pass; returns rate figures."""
    from oracle import csa_oracle as O

    wl = inp.wl
    q = inp.q[0:1].double().numpy()
    k = inp.k[0:1].double().numpy()
    w = inp.w[0:1].double().numpy()
    q_start = None if inp.q_start is None else inp.q_start[0:1].numpy()
    q_seg = None if inp.q_seg is None else inp.q_seg[0:1].numpy()
    kv_seg = None if inp.kv_seg is None else inp.kv_seg[0:1].numpy()
    v = visible_counts(inp)[0]
    rng = np.random.default_rng(seed)
    t0 = time.perf_counter()
    rows_done, pairs_done = 0, 0
    while True:
        rows = np.sort(rng.choice(wl.S, size=min(block, wl.S), replace=False))
        sc = O.index_scores(q, k, w, wl.scale, wl.compress_rate, q_start, q_seg, kv_seg, rows=rows)
        O.select_topk(sc, wl.top_k)
        rows_done += len(rows)
        pairs_done += int(v[rows].sum())
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    flops = 2.0 * wl.H * wl.D * pairs_done
    return dict(seconds=el, rows=rows_done, pairs=pairs_done, tflops=flops / el / 1e12, rows_per_s=rows_done / el)


def run_reference(args, wl, inp):
    budget = max(0.5, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(inp, budget * 0.25, block=64)
    res = [oracle_sample(inp, budget, block=64, seed=i) for i in range(args.steps)]
    secs = sum(r["seconds"] for r in res)
    flops = sum(2.0 * wl.H * wl.D * r["pairs"] for r in res)
    rows = sum(r["rows"] for r in res)
    value = flops / secs / 1e12
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(wl, args.gpus),
        "rows_per_s": rows / secs,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows} random query rows of batch 0 ({args.steps} steps of about "
                                   f"{budget:.1f} s), fp64 scores + full-sort selection"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(wl, n_gpus, shard="replicas"):
    if n_gpus <= 1:
        par = "single GPU"
    elif shard == "rows":
        par = f"row shards x{n_gpus} (one problem, rows balanced by visible entries)"
    else:
        par = f"replicas x{n_gpus}"
    return {"workload": wl.name, "B": wl.B, "S": wl.S, "W": wl.W, "H": wl.H, "D": wl.D,
            "compress_rate": wl.compress_rate, "top_k": wl.top_k, "w_dtype": wl.w_dtype,
            "q_start": wl.q_start, "docs": list(wl.docs) if wl.docs else None,
            "global_batch": wl.B * n_gpus, "seq_len": wl.S,
            "parallelism": par,
            "l2": (("no flush: inputs larger than L2 ({:.0f} MiB)" if not needs_l2_flush(wl) else
                    "flushed: a {} MiB buffer written between timed steps, outside the steps' own events "
                    "(inputs {{:.0f}} MiB)".format(L2_FLUSH_BYTES >> 20)).format(input_bytes(wl) / 2**20))}


L2_BYTES = 129 * 10**6  # GB300
L2_FLUSH_BYTES = 256 << 20


def input_bytes(wl) -> int:
    """Bytes of q, k and w (and segment ids) one step reads."""
    wsz = 2 if wl.w_dtype == "bf16" else 4
    n = wl.B * wl.H * wl.S * wl.D * 2 + wl.B * wl.W * wl.D * 2 + wl.B * wl.S * wl.H * wsz
    if wl.docs:
        n += wl.B * (wl.S + wl.W) * 4
    return n


def needs_l2_flush(wl) -> bool:
    """Inputs that fit in L2 would stay resident from one timed step to the
    next: such workloads flush L2 between steps instead."""
    return input_bytes(wl) < L2_BYTES


# ----------------------------------------------------------------------------- GPU arm
def run_ours(args, wl, inp):
    import sparse_attention_indexer_csa_gb300 as csa

    rank, world, local, dist = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU for the library arm")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    csa.load()
    stream = torch.cuda.current_stream(dev)
    wk = work(inp)
    full_inp = inp
    rows_mode = args.shard == "rows"
    s0 = s1 = 0
    if rows_mode:
        # this rank's query rows of the one shared problem, positioned by q_start
        from sparse_attention_indexer_csa_gb300.shard import row_shards

        s0, s1 = row_shards(wl.S, wl.W, wl.compress_rate, world, wl.q_start or 0)[rank]
        base = inp.q_start if inp.q_start is not None else torch.zeros(wl.B, dtype=torch.int64)
        inp = Inputs(wl, inp.q[:, :, s0:s1].contiguous(), inp.k, inp.w[:, s0:s1].contiguous(),
                     None if inp.q_seg is None else inp.q_seg[:, s0:s1].contiguous(), inp.kv_seg, base + s0)

    q, k, w = inp.q.to(dev), inp.k.to(dev), inp.w.to(dev)
    q_seg = None if inp.q_seg is None else inp.q_seg.to(dev)
    kv_seg = None if inp.kv_seg is None else inp.kv_seg.to(dev)
    q_start = None if inp.q_start is None else inp.q_start.to(dev)
    S_local = q.shape[2]
    p = csa.make_problem(q, k, w, wl.scale, wl.compress_rate, wl.top_k)
    idx = torch.empty(wl.B, S_local, wl.top_k, dtype=torch.int32, device=dev)
    ws_bytes = csa.workspace_size(p, 1)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev) if ws_bytes else None
    # decode-style single rows and rows longer than 16384 take two kernels;
    # segment ids add the summary pre-pass
    launches_per_step = (2 if (wl.S <= 2 or wl.W > 16384 or args.two_pass) else 1) + \
        (1 if (inp.q_seg is not None and wl.S > 2 and wl.W <= 16384 and not args.two_pass) else 0)

    two_pass = args.two_pass
    if two_pass:  # the scores through HBM, then the selection kernel: for comparison only
        sc_buf = torch.empty(wl.B, S_local, wl.W, dtype=torch.float32, device=dev)
        pt = csa.Problem(wl.B, 1, S_local, 1, wl.W, 1, 1.0, wl.top_k, csa.CSA_F32, csa.CSA_Q_HEAD_MAJOR)

    def step():
        if S_local == 0:  # an empty row shard
            return
        if two_pass:
            st = csa.index_score_raw(p, q, k, w, q_seg, kv_seg, q_start, sc_buf, stream)
            if st == csa.CSA_OK:
                st = csa.index_topk_raw(pt, sc_buf, idx, None, stream)
        else:
            st = csa.index_fused_raw(p, q, k, w, q_seg, kv_seg, q_start, idx, None, ws, stream)
        if st != csa.CSA_OK:
            raise RuntimeError(f"csa_index_fused returned {st}")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if csa.device_status(stream) != csa.CSA_OK:
        raise RuntimeError("device status word reports an error after warm-up")

    # ---- device-resident timing (K steps, per-step events on the launch stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ
                          else local)
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.25)  # let the sampler take its first reading
    flush = needs_l2_flush(wl)
    fbuf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    for i in range(args.steps):
        if flush:
            fbuf.fill_(i & 0xFF)  # on `stream` (the current stream): evicts the previous step's inputs
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(dist)
    total_ms = t_all0.elapsed_time(t_all1)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    if flush:  # the flushes are not the workload's: time the steps alone
        total_ms = sum(launch_ms)
    del fbuf
    total_ms = max_over_ranks(total_ms, dist)
    ms_step = total_ms / args.steps
    if csa.device_status(stream) != csa.CSA_OK:
        raise RuntimeError("device status word reports an error after the timed region")

    # ---- end to end: pinned host inputs -> the library's host entry point
    # (csa_index_fused_host), result back in pinned host memory
    pin = (lambda t: t) if args.no_e2e else (lambda t: t.pin_memory())
    hq, hk, hw = pin(inp.q), pin(inp.k), pin(inp.w)
    hqs = None if inp.q_seg is None else pin(inp.q_seg)
    hks = None if inp.kv_seg is None else pin(inp.kv_seg)
    hst = None if inp.q_start is None else pin(inp.q_start)
    ph = csa.make_problem(hq, hk, hw, wl.scale, wl.compress_rate, wl.top_k)
    h2d, d2h = csa.fused_host_bytes(ph, hst, hqs is not None)

    # Each step is one call: it enqueues the copies of its inputs (only the
    # q rows that can need scores), the computation and the copy of its
    # indices back on its own stream.  Three calls are in flight, as a
    # serving loop would keep them, each with its own device workspace and
    # host result buffer, so one step's copies overlap another's compute.
    e2e_ms = float("nan")
    if not args.no_e2e:
        n_sets = 3
        sets = [dict(ws=torch.empty(csa.workspace_size(ph, 3), dtype=torch.uint8, device=dev),
                     host=torch.empty(idx.shape, dtype=idx.dtype).pin_memory(), stream=torch.cuda.Stream(dev))
                for _ in range(n_sets)]

        def e2e_steps_run(n):
            for i in range(n):
                bs = sets[i % n_sets]
                st = csa.index_fused_host_raw(ph, hq, hk, hw, hqs, hks, hst, bs["host"], bs["ws"], bs["stream"])
                if st != csa.CSA_OK:
                    raise RuntimeError(f"csa_index_fused_host returned {st}")

        e2e_steps = max(3 * n_sets, min(args.steps, 12))
        e2e_steps_run(n_sets)
        torch.cuda.synchronize()
        barrier(dist)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for bs in sets:
            bs["stream"].wait_event(e0)
        e2e_steps_run(e2e_steps)
        for bs in sets:
            stream.wait_stream(bs["stream"])
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dist)
        ref = idx.cpu()
        for bs in sets:
            if not torch.equal(bs["host"], ref):
                raise RuntimeError("end-to-end result differs from the device-resident result")
        del sets

    shard_check = None
    if rows_mode and world > 1:
        # every rank's rows (padded to the longest shard), compared on rank 0
        # with one call over all rows, outside the timed region
        from sparse_attention_indexer_csa_gb300.shard import row_shards

        maxr = int(max_over_ranks(float(S_local), dist))
        pad = torch.full((wl.B, maxr, wl.top_k), -2, dtype=torch.int32, device=dev)
        pad[:, :S_local] = idx
        parts = [torch.empty_like(pad) for _ in range(world)]
        dist.all_gather(parts, pad)
        if rank == 0:
            shards = row_shards(wl.S, wl.W, wl.compress_rate, world, wl.q_start or 0)
            got = torch.cat([parts[r][:, :e - b] for r, (b, e) in enumerate(shards)], dim=1)
            g = lambda t: None if t is None else t.to(dev)  # noqa: E731
            full = csa.index_fused(g(full_inp.q), g(full_inp.k), g(full_inp.w), wl.scale, wl.compress_rate,
                                   wl.top_k, g(full_inp.q_seg), g(full_inp.kv_seg), g(full_inp.q_start))
            if not torch.equal(got, full):
                raise RuntimeError("row shards differ from one call over all rows")
            shard_check = f"bit-identical to one call over all rows (shards {shards})"
    if rows_mode:  # one problem split over the ranks: its work, once
        total_flops, total_rows = wk["flops"], wk["rows"]
    else:
        total_flops = sum_over_ranks(wk["flops"], dist)
        total_rows = sum_over_ranks(wk["rows"], dist)
    value = total_flops / (ms_step * 1e-3) / 1e12
    peaks, peak_src = read_peaks()
    avg_launch_ms = sum(launch_ms) / len(launch_ms)
    achieved = wk["flops_nontrivial"] / (avg_launch_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    bound, unit = "tensor", "TFLOP/s"
    traffic = measured_traffic(wl.name) if (args.batch is None and args.seed is None) else None
    if wl.name.startswith("decode"):
        # k streaming bound: algorithmic bytes = k + q + w + scores write/read + idx
        bytes_alg = decode_bytes(wl)
        achieved = bytes_alg / (avg_launch_ms * 1e-3) / 1e9
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        bound, unit = "hbm", "GB/s"

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "strong" if rows_mode else "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_dict(wl, world, "rows" if rows_mode else "replicas"),
        "rows_per_s": total_rows / (ms_step * 1e-3),
        "useful_pairs": wk["pairs"], "nontrivial_rows": wk["nontrivial_rows"],
        "tflops_nontrivial_rows": wk["flops_nontrivial"] / (ms_step * 1e-3) / 1e12,
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})",
                     "achieved_counts": "2*H*D per visible pair of rows with visible > top_k (rows at or below "
                                        "top_k are emitted without scores)" if bound == "tensor" else
                                        "k + q + w bytes read, scores written and re-read, indices written"},
        "e2e": None if args.no_e2e else {
            "value": total_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
            "api": "csa_index_fused_host (host inputs and indices; the library enqueues the copies, sending "
                   "only the q rows that can need scores)",
            "overlap": "three calls in flight on three streams, each with its own device workspace"},
        "gpu_launches": (launches_per_step if S_local > 0 else 0) * args.steps,
        "clocks": clk,
    }
    if shard_check is not None:
        line["shard_check"] = shard_check
    if args.two_pass:
        line["mode"] = "two-pass comparison: scores [B,S,W] fp32 through HBM, then the selection kernel"
    if args.gather:  # gather of the selected rows, timed on its own over the same selection
        gout = torch.empty(wl.B, wl.S, wl.top_k, wl.D, dtype=torch.bfloat16, device=dev)
        for _ in range(3):
            csa.index_gather(k, idx, out=gout, stream=stream)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        n_g = 50
        g0.record(stream)
        for _ in range(n_g):
            csa.index_gather(k, idx, out=gout, stream=stream)
        g1.record(stream)
        torch.cuda.synchronize()
        g_ms = g0.elapsed_time(g1) / n_g
        n_sel = int((idx >= 0).sum().item())
        g_bytes = gout.numel() * 2 + idx.numel() * 4 + n_sel * wl.D * 2
        line["gather"] = {"ms": g_ms, "bytes": g_bytes, "GB/s": g_bytes / (g_ms * 1e-3) / 1e9,
                          "frac_of_hbm": g_bytes / (g_ms * 1e-3) / 1e9 / float(peaks.get("hbm_gbs", 6800.0))}
    if rank == 0 and world == 1 and not args.no_backward and wl.H == 64 and wl.D == 128 and wl.S > 2:
        # the backward of the same scores, reported beside the forward (not in its step)
        try:
            b_ms, b_tf = backward_leg(wl, wk, q, k, w, q_seg, kv_seg, q_start, dev, stream, steps=20)
            line["backward"] = {"ms_per_step": b_ms, "value": b_tf, "unit": "TFLOP/s",
                                "frac_of_bf16_peak": b_tf / float(peaks.get("bf16_tflops",
                                                                            FALLBACK_PEAKS["bf16_tflops"])),
                                "steps": 20,
                                "counts": "3 x 2*H*D per visible pair (logits recomputed, dq, dk)"}
        except Exception as ex:  # reported, never hides the forward line
            line["backward"] = {"error": str(ex)[:300]}
    if rank == 0 and world == 1 and not args.no_side and args.batch is None and wl.name == "prefill_16k":
        # the other two targets, each timed on its own beside the headline
        # workload: decode (HBM-bound) and packed documents at a seed whose
        # rows include some above top_k (seed 0 has none)
        for key, side in (("decode", WORKLOADS["decode_32k"]), ("packed", WORKLOADS["packed_8k"].with_(seed=1))):
            try:
                line[key] = side_leg(side, dev, stream)
            except Exception as ex:  # reported, never hides the headline line
                line[key] = {"error": str(ex)[:300]}
        if args.packed_seeds > 0:
            try:
                line["packed_seeds"] = packed_seeds_leg(args.packed_seeds, dev, stream)
            except Exception as ex:
                line["packed_seeds"] = {"error": str(ex)[:300]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = oracle_sample(inp, args.cpu_seconds)
        line["cpu_baseline"] = {"value": cb["tflops"], "unit": "TFLOP/s", "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"{cb['rows']} random query rows of batch 0 in {cb['seconds']:.1f} s, "
                                          f"fp64 scores + full-sort selection ({cb['rows_per_s']:.1f} rows/s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def side_leg(wl, dev, stream, steps=50, warmup=5):
    """Times csa_index_fused on another workload with CUDA events on `stream`
    (inputs resident; each is larger than L2, so no flush is needed) and
    returns its figures for a sub-object of the bench line."""
    import sparse_attention_indexer_csa_gb300 as csa

    inp = make_inputs(wl)
    wk = work(inp)
    g = lambda t: None if t is None else t.to(dev)  # noqa: E731
    q, k, w, qs, ks, st = g(inp.q), g(inp.k), g(inp.w), g(inp.q_seg), g(inp.kv_seg), g(inp.q_start)
    p = csa.make_problem(q, k, w, wl.scale, wl.compress_rate, wl.top_k)
    idx = torch.empty(wl.B, wl.S, wl.top_k, dtype=torch.int32, device=dev)
    nb = csa.workspace_size(p, 1)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev) if nb else None

    def step():
        r = csa.index_fused_raw(p, q, k, w, qs, ks, st, idx, None, ws, stream)
        if r != csa.CSA_OK:
            raise RuntimeError(f"csa_index_fused returned {r}")

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.25)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if csa.device_status(stream) != csa.CSA_OK:
        raise RuntimeError(f"device status word reports an error after {wl.name}")
    ms = e0.elapsed_time(e1) / steps
    peaks, peak_src = read_peaks()
    out = {"workload": wl.name, "seed": wl.seed, "B": wl.B, "S": wl.S, "W": wl.W, "top_k": wl.top_k,
           "steps": steps, "ms_per_step": ms, "value": wk["flops"] / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "rows_per_s": wk["rows"] / (ms * 1e-3), "nontrivial_rows": wk["nontrivial_rows"],
           "tflops_nontrivial_rows": wk["flops_nontrivial"] / (ms * 1e-3) / 1e12, "clocks": clk}
    if wl.name.startswith("decode"):
        bytes_alg = decode_bytes(wl)
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        out["roofline"] = {"bound": "hbm", "achieved": bytes_alg / (ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s",
                           "frac": bytes_alg / (ms * 1e-3) / 1e9 / hbm, "traffic": measured_traffic(wl.name),
                           "peak_source": f"{peak_src} hbm_gbs",
                           "achieved_counts": "k + q + w bytes read, scores written and re-read, indices written "
                                              "(score kernel + selection kernel per step)"}
    else:
        bf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        a = wk["flops_nontrivial"] / (ms * 1e-3) / 1e12
        out["roofline"] = {"bound": "tensor", "achieved": a, "peak": bf, "unit": "TFLOP/s", "frac": a / bf,
                           "traffic": measured_traffic(f"{wl.name}_seed{wl.seed}"),
                           "peak_source": f"{peak_src} bf16_tflops",
                           "achieved_counts": "2*H*D per visible pair of rows with visible > top_k"}
    del q, k, w, qs, ks, st, idx, ws
    return out


def packed_seeds_leg(n, dev, stream):
    """The packed-document workload over generator seeds 0 .. n-1 (documents
    and so the work differ by seed): each seed timed on its own, then the
    average over the seeds -- total useful work over total time."""
    per = []
    for seed in range(n):
        r = side_leg(WORKLOADS["packed_8k"].with_(seed=seed), dev, stream, steps=20, warmup=3)
        per.append(r)
    t = sum(r["ms_per_step"] for r in per)
    fl = sum(r["tflops_nontrivial_rows"] * r["ms_per_step"] for r in per)  # TFLOP/s x ms
    peaks, peak_src = read_peaks()
    bf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    return {"workload": "packed_8k", "seeds": n, "ms_per_step_mean": t / n,
            "tflops_nontrivial_rows": fl / t, "frac_of_bf16_peak": fl / t / bf,
            "nontrivial_rows_mean": sum(r["nontrivial_rows"] for r in per) / n,
            "per_seed_ms": [round(r["ms_per_step"], 5) for r in per],
            "per_seed_nontrivial_rows": [r["nontrivial_rows"] for r in per],
            "peak_source": f"{peak_src} bf16_tflops"}


def decode_bytes(wl):
    """Algorithmic bytes of one decode step: k, q and w read, the fp32 scores
    written and read back by the selection, the indices written."""
    return (wl.B * wl.W * wl.D * 2 + wl.B * wl.H * wl.S * wl.D * 2 + wl.B * wl.S * wl.H * 2
            + 2 * wl.B * wl.S * wl.W * 4 + wl.B * wl.S * wl.top_k * 4)


def backward_leg(wl, wk, q, k, w, q_seg, kv_seg, q_start, dev, stream, steps, warmup=3):
    """Times csa_index_backward (dq, dk, dw for a fixed seeded cotangent of
    the scores) with CUDA events on `stream`; returns (ms per step, useful
    TFLOP/s): 3 x 2*H*D per visible pair (logits recomputed, dq, dk)."""
    import sparse_attention_indexer_csa_gb300 as csa

    gen = torch.Generator().manual_seed(wl.seed + 1000)
    g = torch.randn(wl.B, wl.S, wl.W, generator=gen, dtype=torch.float32).to(dev)
    p = csa.make_problem(q, k, w, wl.scale, wl.compress_rate, 1)
    dq = torch.empty(wl.B, wl.H, wl.S, wl.D, dtype=torch.float32, device=dev)
    dk = torch.empty(wl.B, wl.W, wl.D, dtype=torch.float32, device=dev)
    dw = torch.empty(wl.B, wl.S, wl.H, dtype=torch.float32, device=dev)
    ws = torch.empty(csa.workspace_size(p, 2), dtype=torch.uint8, device=dev)

    def step():
        st = csa.abi.index_backward_raw(p, q, k, w, q_seg, kv_seg, q_start, g, dq, dk, dw, ws, stream)
        if st != csa.CSA_OK:
            raise RuntimeError(f"csa_index_backward returned {st}")

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if csa.device_status(stream) != csa.CSA_OK:
        raise RuntimeError("device status word reports an error after the backward")
    ms = e0.elapsed_time(e1) / steps
    return ms, 3.0 * wk["flops"] / (ms * 1e-3) / 1e12


def run_backward(args, wl, inp):
    """One line for the backward of the score step (csa_index_backward):
    dq, dk, dw for a fixed seeded cotangent of the scores; per step a memset
    of dk, the dq/dw kernel and the dk kernel."""
    import sparse_attention_indexer_csa_gb300 as csa

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU for the library arm")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    csa.load()
    stream = torch.cuda.current_stream(dev)
    wk = work(inp)
    q, k, w = inp.q.to(dev), inp.k.to(dev), inp.w.to(dev)
    q_seg = None if inp.q_seg is None else inp.q_seg.to(dev)
    kv_seg = None if inp.kv_seg is None else inp.kv_seg.to(dev)
    q_start = None if inp.q_start is None else inp.q_start.to(dev)
    clocks = ClockSampler(0)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.25)
    ms, achieved = backward_leg(wl, wk, q, k, w, q_seg, kv_seg, q_start, dev, stream, args.steps, args.warmup)
    clk = clocks.stop()
    peaks, peak_src = read_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    line = {
        "metric": "indexer backward useful TFLOP/s (dq, dk, dw of the visible scores)", "value": achieved,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "mode": "backward", "config": config_dict(wl, 1),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})",
                     "achieved_counts": "3 x 2*H*D per visible pair (logits recomputed, dq, dk); the whole step: "
                                        "the dq/dw kernel and the dk kernel (each recomputes the logits)"},
        "e2e": None, "gpu_launches": None, "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="prefill_16k", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--batch", type=int, default=None, help="override B (smaller profiling case)")
    ap.add_argument("--seed", type=int, default=None, help="override the workload's input seed")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward of the score step instead (its own JSON line)")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the backward measurement reported beside the forward")
    ap.add_argument("--shard", default="replicas", choices=["replicas", "rows"],
                    help="under torchrun: independent replicas per rank (weak scaling) or one problem whose "
                         "query rows are split over the ranks (strong scaling)")
    ap.add_argument("--two-pass", action="store_true",
                    help="time the score kernel then the selection kernel over stored scores instead of the "
                         "fused path (comparison only)")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the decode and packed-document legs reported beside the headline")
    ap.add_argument("--packed-seeds", type=int, default=0,
                    help="also time the packed-document workload over seeds 0..N-1 and report the average "
                         "(about 3 s of input generation per seed)")
    ap.add_argument("--gather", action="store_true",
                    help="also time the gather of the selected compressed rows (reported, not in the step)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    wl = WORKLOADS[args.workload]
    if args.batch is not None:
        wl = wl.with_(B=args.batch)
    if args.seed is not None:
        wl = wl.with_(seed=args.seed)
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        inp = make_inputs(wl.with_(seed=wl.seed + rank))
        run_reference(args, wl, inp)
        return
    # replicas draw their own inputs; row shards all cut the same problem
    inp = make_inputs(wl.with_(seed=wl.seed + (rank if args.shard == "replicas" else 0)))
    if args.backward:
        run_backward(args, wl, inp)
        return
    run_ours(args, wl, inp)


if __name__ == "__main__":
    main()
