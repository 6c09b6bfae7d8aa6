#!/usr/bin/env python3
"""Benchmark: vision tokens scored + selected per second on one GB300.

One step = the whole hot path over one batch: importance scores (schedule,
row-LSE pass, column pass), pooled top-B, compaction of hidden rows and
position ids. Inputs are resident in HBM before the timed region; L2 is
flushed (a 512 MiB write) between steps and the flush is not timed.

Prints ONE JSON line (rank 0). ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload instead (the reference arm).
Replicas only: under torchrun every rank runs its own copy of the workload on
its own GPU with no data exchange; value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "vision tokens scored+selected/sec at 1 GB300; importance % of roofline"
DEFAULT_WORKLOAD = "thirty_images"
L2_NOTE = "flushed (512 MiB write) between GPU steps, untimed"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
_CSRC = "attention_score_vision_gb300/csrc/"
# Sources each kernel is built from (a traffic figure taken on other sources reads as null).
KERNEL_SOURCES = {
    "imp_pass_kernel": [_CSRC + f for f in ("imp_pass.cuh", "imp_pass1.cu", "imp_pass2.cu",
                                            "ptx.cuh", "common.cuh", "launch_util.cuh")],
    "topk_cluster_kernel": [_CSRC + f for f in ("topk.cu", "common.cuh", "launch_util.cuh")],
    "gather_kernel": [_CSRC + f for f in ("gather.cu", "common.cuh", "launch_util.cuh")],
}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["tsel", "reference"], default="tsel")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--images", type=int, default=0,
                    help="only the first N images of the workload, as one 60%% request "
                         "(a smaller case of the same shapes, e.g. for counter captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-small", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--cpu-child", nargs=3, metavar=("WORKLOAD", "PAIRS", "IMAGES"),
                    help=argparse.SUPPRESS)
    ap.add_argument("--cpu-small", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args(argv)


def src_hash(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# CPU oracle legs (run in a child process; segments spread over a pool of
# host processes with one BLAS thread each)
# ---------------------------------------------------------------------------

def oracle_sample(w, pair_budget: float):
    """Images of the workload, in order, that fit in ~pair_budget attended pairs
    (at least one image; every image when the budget covers the workload).
    Returns the list of image indices and their pairs."""
    import numpy as np
    nq = np.diff(w.cu_seqlens_q).astype(np.int64)
    nk = np.diff(w.cu_seqlens_k).astype(np.int64)
    cost = w.num_heads * nq * nk
    chosen, pairs = [], 0
    for g in range(w.num_seg):
        if pairs + cost[g] <= pair_budget:
            chosen.append(g)
            pairs += int(cost[g])
    if not chosen:
        g = int(np.argmin(cost))
        chosen, pairs = [g], int(cost[g])
    return chosen, pairs


def _oracle_segment(args):
    """One image through oracle.importance (a pool task)."""
    import oracle
    qb, kb, nq, nk = args
    return oracle.importance(qb, kb, [0, nq], [0, nk])


def oracle_step(w, chosen, pool) -> dict:
    """The oracle over the chosen images as one request: importance image by
    image across the pool (attention is block-diagonal), then the pooled top-B
    (60% keep, or the workload's own budgets when every image is chosen) and
    the compaction, once. Returns the wall time and the sizes."""
    import numpy as np
    import oracle
    import workloads as W
    cq, ck = w.cu_seqlens_q, w.cu_seqlens_k
    tasks = [(w.q_bits[cq[g]:cq[g + 1]], w.k_bits[ck[g]:ck[g + 1]], int(cq[g + 1] - cq[g]),
              int(ck[g + 1] - ck[g])) for g in chosen]
    order = sorted(range(len(chosen)), key=lambda i: -tasks[i][2] * tasks[i][3])
    full = len(chosen) == w.num_seg
    cu_k = np.concatenate([[0], np.cumsum([tasks[i][3] for i in range(len(chosen))])]).astype(np.int64)
    n = int(cu_k[-1])
    if full:
        req_off, keep = w.req_tok_offsets, w.keep_per_req
    else:
        req_off, keep = np.array([0, n], np.int32), np.array([W.keep_floor(n, 600)], np.int32)
    hidden = np.concatenate([w.hidden_bits[ck[g]:ck[g + 1]] for g in chosen])
    pos = np.concatenate([w.pos[ck[g]:ck[g + 1]] for g in chosen])
    t0 = time.perf_counter()
    parts = dict(zip(order, pool.map(_oracle_segment, [tasks[i] for i in order])))
    scores = np.concatenate([parts[i][1] for i in range(len(chosen))])
    keep_idx, _ = oracle.select_topk(scores, req_off, keep)
    oracle.gather_compact(hidden, pos, cu_k, keep_idx)
    dt = time.perf_counter() - t0
    pairs = int(sum(w.num_heads * t[2] * t[3] for t in tasks))
    return {"seconds": dt, "images": len(chosen), "tokens": n, "pairs": pairs,
            "full_pairs": w.attended_pairs(), "full_tokens": w.total_k, "full": full}


def oracle_pool(workers: int):
    import concurrent.futures as cf
    import multiprocessing as mp
    return cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn"))


def cpu_child(workload: str, pair_budget: float, images: int = 0) -> dict:
    """The oracle over the workload (every image when pair_budget covers it)."""
    import workloads as W
    w = W.make(workload)
    if images > 0:
        w = W.first_images(w, images)
    chosen, _ = oracle_sample(w, pair_budget)
    workers = host_cores()
    with oracle_pool(workers) as pool:
        pool.submit(int, 0).result()          # workers up before the clock starts
        res = oracle_step(w, chosen, pool)
    res["cores"] = workers
    return res


SMALL_REQUESTS = ("single_image_256", "six_views_1536", "text_query_3072")


def cpu_small_child() -> dict:
    """The oracle on each small request in one process with one BLAS thread:
    importance, pooled top-B and compaction; input generation not timed."""
    import oracle
    import workloads as W
    out = {}
    for name in SMALL_REQUESTS:
        w = W.make(name)
        t0 = time.perf_counter()
        _, s = oracle.importance(w.q_bits, w.k_bits, w.cu_seqlens_q, w.cu_seqlens_k,
                                 w.softmax_scale)
        keep_idx, _ = oracle.select_topk(s, w.req_tok_offsets, w.keep_per_req)
        oracle.gather_compact(w.hidden_bits, w.pos, w.cu_seqlens_k, keep_idx)
        dt = time.perf_counter() - t0
        out[name] = {"seconds": dt, "tokens_per_s": w.total_k / dt, "cores": 1}
    return out


def run_cpu_small_child() -> dict:
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = "1"
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-small"],
                       capture_output=True, text=True, env=env, timeout=600)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_cpu_child(workload: str, pair_budget: float, images: int = 0) -> dict:
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[v] = "1"
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-child", workload,
                        str(pair_budget), str(images)], capture_output=True, text=True, env=env,
                       timeout=900)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_rate(res: dict) -> float:
    """Tokens/s of the full workload (measured on it, or scaled from the sample's
    images by attended pairs when only a sample was run)."""
    t_full = res["seconds"] * res["full_pairs"] / max(res["pairs"], 1)
    return res["full_tokens"] / t_full


def make_workload(args):
    import workloads as W
    w = W.make(args.workload)
    return W.first_images(w, args.images) if args.images > 0 else w


def workload_config(w, workload: str, world: int, l2: str) -> dict:
    """The `config` object both arms report for one workload."""
    return {"workload": workload, "images": w.num_seg, "visual_tokens": w.total_k,
            "query_tokens": w.total_q, "heads": w.num_heads, "kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "hidden": int(w.hidden_bits.shape[1]),
            "pos_dim": int(w.pos.shape[1]), "keep_total": w.total_keep,
            "requests": int(w.keep_per_req.size), "attended_pairs": w.attended_pairs(),
            "l2": l2, "parallelism": "replicas" if world > 1 else "single GPU"}


def reference_arm(args) -> None:
    """The fp64 oracle, as it stands, on every host core (one process per core,
    one BLAS thread each): each step the whole workload when the run fits in
    about two minutes, else the same first images every step."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = make_workload(args)
    workers = host_cores()
    budget = REFERENCE_PAIRS_PER_S * workers * 120.0 / max(1, args.steps + args.warmup)
    chosen, pairs = oracle_sample(w, budget)
    res = []
    with oracle_pool(workers) as pool:
        pool.submit(int, 0).result()
        for i in range(args.warmup + args.steps):
            r = oracle_step(w, chosen, pool)
            if i >= args.warmup:
                res.append(r)
    r0 = res[0]
    rate = statistics.median(cpu_rate(r) for r in res)
    if r0["full"]:
        sample = (f"full workload per step ({args.workload}: {r0['tokens']} tokens, "
                  f"{r0['pairs']:.3g} attended head-query-key pairs): importance image by image "
                  f"over {workers} processes (fp64 numpy, 1 BLAS thread each), then top-B and "
                  f"compaction once")
    else:
        sample = (f"images {chosen} ({r0['tokens']} tokens, {r0['pairs']:.3g} attended pairs) of "
                  f"the {args.workload} workload per step over {workers} processes (fp64 numpy, "
                  f"1 BLAS thread each); tokens/s scaled to the full workload by attended pairs")
    line = {"metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.median(r["seconds"] for r in res),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            # the GPU arm's config, so both lines describe the same workload
            "config": workload_config(w, args.workload, args.gpus, L2_NOTE),
            "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": workers, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((num(r[2]) or 0.0) for r in rows)}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("src_hash") != src_hash(KERNEL_SOURCES[kernel.split("<")[0]]):
        return None
    return e.get("bytes_per_launch")


def gather_dram_rate(workload: str, t_ms: float, algo_bytes: int, hbm_peak: float) -> dict:
    """The compaction's DRAM-only rate: bytes that reached DRAM during the kernel
    (one ncu capture on the current sources) over the event-timed duration.
    The rest of the written rows are still dirty in L2 when the kernel ends
    and reach DRAM during the next kernel."""
    dram = load_traffic("gather_kernel", workload)
    if dram is None:
        return {"dram_bytes_per_launch": None}
    return {"dram_bytes_per_launch": dram,
            "dram_GB/s": dram / (t_ms * 1e-3) / 1e9,
            "dram_hbm_frac": dram / (t_ms * 1e-3) / hbm_peak,
            "l2_resident_bytes_at_end": max(0, algo_bytes - dram)}


def reduce_max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank value over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(tokens_per_replica: int, world: int, ms_max: float) -> float:
    """Whole-job tokens/s: every rank processed its own replica of the workload."""
    return world * tokens_per_replica / (ms_max * 1e-3)


def workload_throughput(tsel, w, dev, flush, stream, ex2_peak, bf16_peak, steps: int = 20,
                        warmup: int = 3) -> dict:
    """Whole-path throughput of one workload (events around each step, L2 flushed
    in between, untimed) and its importance time against the importance roofline."""
    import numpy as np
    import torch

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    q, k, hidden = bf16(w.q_bits), bf16(w.k_bits), bf16(w.hidden_bits)
    cq, ck, ro, kp, pos = (i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), i32(w.req_tok_offsets),
                           i32(w.keep_per_req), i32(w.pos))
    G, Tq, Tk, H, K = w.num_seg, w.total_q, w.total_k, w.num_heads, w.total_keep
    R = w.keep_per_req.size
    ws = torch.zeros(tsel.tsel_score_select_workspace_size(G, Tq, Tk, H, R), dtype=torch.uint8,
                     device=dev)
    scores = torch.empty(Tk, device=dev)
    lse = torch.empty((H, Tq), device=dev)
    keep_idx = torch.empty(K, dtype=torch.int32, device=dev)
    cu_keep = torch.empty(R + 1, dtype=torch.int32, device=dev)
    oh = torch.empty((K, hidden.shape[1]), dtype=torch.bfloat16, device=dev)
    op = torch.empty((K, w.pos.shape[1]), dtype=torch.int32, device=dev)
    oi = torch.empty(K, dtype=torch.int32, device=dev)
    oc = torch.empty(G + 1, dtype=torch.int32, device=dev)
    IMP = tsel.TSEL_IMP_STAGE_PREP | tsel.TSEL_IMP_STAGE_PASS1 | tsel.TSEL_IMP_STAGE_PASS2

    def score_select(flags):
        tsel.tsel_score_select(q, k, cq, ck, w.max_seqlen_q, w.max_seqlen_k, ro, kp, K, flags=flags,
                               lse=lse, scores=scores, keep_idx=keep_idx, cu_keep=cu_keep,
                               workspace=ws, stream=stream)

    def gather():
        tsel.tsel_gather_compact(hidden, pos, ck, keep_idx, out_hidden=oh, out_pos=op, out_img_id=oi,
                                 out_cu_seqlens=oc, workspace=ws, stream=stream)

    one_launch = tsel.tsel_importance_one_launch(G, Tq, Tk, w.max_seqlen_q, w.max_seqlen_k, H,
                                                 w.head_dim) == 1

    def importance_alone():
        if one_launch:   # the one-launch kernel (the stage bits would select the two-pass form)
            tsel.tsel_importance(q, k, cq, ck, w.max_seqlen_q, w.max_seqlen_k, lse=lse,
                                 scores=scores, workspace=ws, stream=stream)
        else:
            score_select(IMP)

    whole, stage = [], []
    for i in range(warmup + steps):       # the path as it runs: one fused call + compaction
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        score_select(0)
        gather()
        b.record(stream)
        if i >= warmup:
            whole.append((a, b))
    for i in range(warmup + steps):       # importance stages apart, for its roofline
        flush.fill_(i & 0xFF)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ev[0].record(stream)
        importance_alone()
        ev[1].record(stream)
        score_select(tsel.TSEL_SEL_STAGE_TOPK)
        gather()
        if i >= warmup:
            stage.append(ev)
    torch.cuda.synchronize()
    if tsel.tsel_read_device_status(ws) != 0:
        raise RuntimeError(f"device status set for {w.name}")
    t_step = sum(a.elapsed_time(b) for a, b in whole) / len(whole)
    t_imp = sum(e[0].elapsed_time(e[1]) for e in stage) / len(stage)
    E = w.attended_pairs()
    roof = max(4 * w.head_dim * E / bf16_peak, 2 * E / ex2_peak)
    return {"tokens": Tk, "ms_per_step": t_step, "tokens_per_s": Tk / (t_step * 1e-3),
            "importance_ms": t_imp, "importance_roofline_frac": roof / (t_imp * 1e-3),
            "topk_paths": tsel.tsel_select_path_counts(ws),
            "importance_launches": "one" if one_launch else "schedule + two passes",
            "note": f"{steps} steps of the fused score + select call and the compaction; "
                    "importance timed apart (the one-launch kernel, or the schedule and the "
                    "two passes, then an event)"}


def small_request_latency(tsel, w, dev, flush, stream, reps: int = 20) -> dict:
    """Device time of the whole path (importance, top-B, compaction) for one small
    request, launched eagerly and replayed from a CUDA graph; L2 flushed (untimed)
    before every timed run."""
    import numpy as np
    import torch

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    q, k, hidden = bf16(w.q_bits), bf16(w.k_bits), bf16(w.hidden_bits)
    cq, ck, ro, kp, pos = (i32(w.cu_seqlens_q), i32(w.cu_seqlens_k), i32(w.req_tok_offsets),
                           i32(w.keep_per_req), i32(w.pos))
    G, Tq, Tk, H, K = w.num_seg, w.total_q, w.total_k, w.num_heads, w.total_keep
    R = w.keep_per_req.size
    ws = torch.zeros(tsel.tsel_score_select_workspace_size(G, Tq, Tk, H, R), dtype=torch.uint8,
                     device=dev)
    scores = torch.empty(Tk, device=dev)
    lse = torch.empty((H, Tq), device=dev)
    keep_idx = torch.empty(K, dtype=torch.int32, device=dev)
    cu_keep = torch.empty(R + 1, dtype=torch.int32, device=dev)
    oh = torch.empty((K, hidden.shape[1]), dtype=torch.bfloat16, device=dev)
    op = torch.empty((K, w.pos.shape[1]), dtype=torch.int32, device=dev)
    oi = torch.empty(K, dtype=torch.int32, device=dev)
    oc = torch.empty(G + 1, dtype=torch.int32, device=dev)

    def path(st):
        tsel.tsel_score_select(q, k, cq, ck, w.max_seqlen_q, w.max_seqlen_k, ro, kp, K, lse=lse,
                               scores=scores, keep_idx=keep_idx, cu_keep=cu_keep, workspace=ws,
                               stream=st)
        tsel.tsel_gather_compact(hidden, pos, ck, keep_idx, out_hidden=oh, out_pos=op, out_img_id=oi,
                                 out_cu_seqlens=oc, workspace=ws, stream=st)

    def timed(fn):
        out = []
        for i in range(reps + 3):
            flush.fill_(i & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            if i >= 3:
                out.append(a.elapsed_time(b) * 1e3)
        return float(np.median(out))

    eager_us = timed(lambda: path(stream))
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        path(side)
    stream.wait_stream(side)
    graph_us = timed(g.replay)
    if tsel.tsel_read_device_status(ws) != 0:
        raise RuntimeError(f"device status set for {w.name}")
    return {"tokens": Tk, "keep": K, "eager_us": eager_us, "graph_us": graph_us,
            "note": "median of 20 runs, L2 flushed before each (untimed)"}


def gpu_arm(args) -> None:
    import numpy as np
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    # CPU baseline first (a child process, before this process touches the GPU).
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        try:
            cpu = run_cpu_child(args.workload, float("inf"), args.images)
        except Exception as exc:  # reported, never fatal
            cpu = {"error": str(exc)[-300:]}
    cpu_small = {}
    if rank == 0 and not args.no_cpu_baseline and not args.no_small:
        try:
            cpu_small = run_cpu_small_child()
        except Exception as exc:  # reported, never fatal
            cpu_small = {"error": str(exc)[-300:]}

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import attention_score_vision_gb300 as tsel
    import workloads as W
    tsel.build()
    tsel.load_library()

    w = make_workload(args)
    dev = torch.device("cuda", local)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32))

    host = {"q": bf16(w.q_bits), "k": bf16(w.k_bits), "cu_q": i32(w.cu_seqlens_q),
            "cu_k": i32(w.cu_seqlens_k), "req_off": i32(w.req_tok_offsets),
            "keep": i32(w.keep_per_req), "hidden": bf16(w.hidden_bits), "pos": i32(w.pos)}
    d = {k: v.to(dev) for k, v in host.items()}
    G, Tq, Tk, H, Hkv, hd = w.num_seg, w.total_q, w.total_k, w.num_heads, w.num_kv_heads, w.head_dim
    K = w.total_keep
    D = w.hidden_bits.shape[1]
    P = w.pos.shape[1]
    R = w.keep_per_req.size
    ws = torch.zeros(tsel.tsel_score_select_workspace_size(G, Tq, Tk, H, R), dtype=torch.uint8,
                     device=dev)
    scores = torch.empty(Tk, dtype=torch.float32, device=dev)
    lse = torch.empty((H, Tq), dtype=torch.float32, device=dev)
    keep_idx = torch.empty(K, dtype=torch.int32, device=dev)
    cu_keep = torch.empty(R + 1, dtype=torch.int32, device=dev)
    out_h = torch.empty((K, D), dtype=torch.bfloat16, device=dev)
    out_p = torch.empty((K, P), dtype=torch.int32, device=dev)
    out_i = torch.empty(K, dtype=torch.int32, device=dev)
    out_c = torch.empty(G + 1, dtype=torch.int32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    S1, S2, S3 = tsel.TSEL_IMP_STAGE_PREP, tsel.TSEL_IMP_STAGE_PASS1, tsel.TSEL_IMP_STAGE_PASS2
    S4 = tsel.TSEL_SEL_STAGE_TOPK

    def score_select(flags, q=None, k=None, cu_q=None, cu_k=None, req_off=None, keep=None):
        # importance and the pooled top-B in one call (the product path)
        tsel.tsel_score_select(q if q is not None else d["q"], k if k is not None else d["k"],
                               cu_q if cu_q is not None else d["cu_q"],
                               cu_k if cu_k is not None else d["cu_k"],
                               w.max_seqlen_q, w.max_seqlen_k,
                               req_off if req_off is not None else d["req_off"],
                               keep if keep is not None else d["keep"], K, flags=flags, lse=lse,
                               scores=scores, keep_idx=keep_idx, cu_keep=cu_keep, workspace=ws,
                               stream=stream)

    def importance(flags, q=None, k=None, cu_q=None, cu_k=None):
        tsel.tsel_importance(q if q is not None else d["q"], k if k is not None else d["k"],
                             cu_q if cu_q is not None else d["cu_q"],
                             cu_k if cu_k is not None else d["cu_k"],
                             w.max_seqlen_q, w.max_seqlen_k, flags=flags, lse=lse, scores=scores,
                             workspace=ws, stream=stream)

    def topk(req_off=None, keep=None):
        tsel.tsel_select_topk(scores, req_off if req_off is not None else d["req_off"],
                              keep if keep is not None else d["keep"], K, keep_idx=keep_idx,
                              cu_keep=cu_keep, workspace=ws, stream=stream)

    def gather(hidden=None, pos=None, cu_k=None):
        tsel.tsel_gather_compact(hidden if hidden is not None else d["hidden"],
                                 pos if pos is not None else d["pos"],
                                 cu_k if cu_k is not None else d["cu_k"], keep_idx, out_hidden=out_h,
                                 out_pos=out_p, out_img_id=out_i, out_cu_seqlens=out_c,
                                 workspace=ws, stream=stream)

    # --- MUFU ex2 peak (probe kernel, best of 3) --------------------------
    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    pblocks, piters = sms * 4, 2048
    sink = torch.empty(pblocks * 512 + 4, dtype=torch.float32, device=dev)
    tsel.tsel_probe_ex2(pblocks, piters, sink)
    best = None
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        tsel.tsel_probe_ex2(pblocks, piters, sink)
        b.record(stream)
        b.synchronize()
        t = a.elapsed_time(b) * 1e-3
        best = t if best is None else min(best, t)
    ex2_peak = pblocks * 512 * piters * 8 / best        # exp2 / s
    # the SM clock during the last probe launch: block 0's cycles over its ns
    p_cyc, p_ns = (int(x) for x in sink[pblocks * 512:].view(torch.int64).cpu().tolist())
    probe_mhz = p_cyc / p_ns * 1e3 if p_ns > 0 else None

    # --- warm-up -----------------------------------------------------------
    for _ in range(args.warmup):
        flush.fill_(1)
        score_select(0)
        gather()
    torch.cuda.synchronize()
    if tsel.tsel_read_device_status(ws) != 0:
        raise RuntimeError("device status set during warm-up")

    # --- timed (device-resident inputs): the whole path per step, events only
    # around it, so consecutive kernels overlap launch and drain (PDL) as in use
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        evs[i][0].record(stream)
        score_select(0)
        gather()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    status = tsel.tsel_read_device_status(ws)
    if status != 0:
        raise RuntimeError(f"device status 0x{status:x} after the timed loop")
    ms_local = sum(step_ms) / len(step_ms)
    ms = reduce_max_over_ranks(ms_local, dev)
    value = replica_throughput(Tk, world, ms)

    # --- per-kernel times: the same steps with an event between the stages
    # (events break the launch overlap, so these are each kernel alone) -------
    # topk: the histogram-started top-B of the fused call; topk_plain: the
    # plain top-B (tsel_select_topk) on the same scores, for comparison
    names = ["prep", "pass1", "pass2", "topk", "gather", "topk_plain"]
    n_stage = max(5, min(args.steps, 50))
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(n_stage)]
    for i in range(n_stage):
        flush.fill_(i & 0xFF)
        e = sevs[i]
        e[0].record(stream)
        score_select(S1)
        e[1].record(stream)
        score_select(S2)
        e[2].record(stream)
        score_select(S3)
        e[3].record(stream)
        score_select(S4)
        e[4].record(stream)
        gather()
        e[5].record(stream)
        topk()
        e[6].record(stream)
    torch.cuda.synchronize()
    per = {n: [] for n in names}
    for e in sevs:
        for j, n in enumerate(names):
            per[n].append(e[j].elapsed_time(e[j + 1]))
    if tsel.tsel_read_device_status(ws) != 0:
        raise RuntimeError("device status set in the per-kernel loop")
    redo_pairs = tsel.tsel_importance_redo_pairs(ws)
    topk_paths = tsel.tsel_select_path_counts(ws)

    # --- top-B + compaction back to back inside the step, as the path runs
    # them (the compaction launches while the top-B runs and waits for it on
    # the device); events only around those two launches. Directly after the
    # flush, the compaction would also pay for writing back the flush's dirty
    # L2 lines, which the importance passes absorb in a real step -------------
    sel_evs = []
    for i in range(n_stage):
        flush.fill_(i & 0xFF)
        score_select(S1 | S2 | S3)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        score_select(S4)
        gather()
        b.record(stream)
        sel_evs.append((a, b))
    torch.cuda.synchronize()
    sel_span = [a.elapsed_time(b) for a, b in sel_evs]
    if tsel.tsel_read_device_status(ws) != 0:
        raise RuntimeError("device status set in the selection loop")

    # --- what top-B + compaction add to the step: the whole step against the
    # same importance chain alone (schedule and both passes in one call), each
    # with events only around it and interleaved, so the top-B's launch
    # overlaps the column pass's drain as it does in the step ----------------
    chain_evs, fused_evs, whole_evs = [], [], []
    for i in range(n_stage):
        for j, evl in enumerate((chain_evs, fused_evs, whole_evs)):
            flush.fill_((i + j) & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if j == 0:
                score_select(S1 | S2 | S3)   # schedule and both passes
            elif j == 1:
                score_select(0)              # ... and the top-B
            else:
                score_select(0)              # ... and the compaction
                gather()
            b.record(stream)
            evl.append((a, b))
    torch.cuda.synchronize()
    chain_ms = sum(a.elapsed_time(b) for a, b in chain_evs) / len(chain_evs)
    fused_ms = sum(a.elapsed_time(b) for a, b in fused_evs) / len(fused_evs)
    whole_ms = sum(a.elapsed_time(b) for a, b in whole_evs) / len(whole_evs)
    # the differences mean what they say only when the fused call scores with
    # the same launches as the chain (not the one-launch kernel of small problems)
    same_chain = tsel.tsel_importance_one_launch(G, Tq, Tk, w.max_seqlen_q, w.max_seqlen_k, H,
                                                 hd) == 0
    if tsel.tsel_read_device_status(ws) != 0:
        raise RuntimeError("device status set in the step-difference loop")

    # --- the same path as three separate calls (importance, plain top-B,
    # compaction), for comparison with the fused call ------------------------
    sep = []
    for i in range(args.warmup + args.steps):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        importance(0)
        topk()
        gather()
        b.record(stream)
        if i >= args.warmup:
            sep.append((a, b))
    torch.cuda.synchronize()
    sep_ms = reduce_max_over_ranks(sum(x.elapsed_time(y) for x, y in sep) / len(sep), dev)
    separate_calls = {"ms_per_step": sep_ms, "value": replica_throughput(Tk, world, sep_ms),
                      "unit": "tokens/s",
                      "note": "tsel_importance + tsel_select_topk (radix rounds over the scores) "
                              "+ tsel_gather_compact"}

    # --- LSE-provided mode: the attention kernel's LSE reused, column pass only ---
    lse_given = lse.clone()
    lp_ms = []
    LP = tsel.TSEL_IMP_LSE_PROVIDED
    for i in range(args.warmup + args.steps):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        tsel.tsel_importance(d["q"], d["k"], d["cu_q"], d["cu_k"], w.max_seqlen_q, w.max_seqlen_k,
                             flags=LP, lse=lse_given, scores=scores, workspace=ws, stream=stream)
        topk()
        gather()
        b.record(stream)
        if i >= args.warmup:
            lp_ms.append((a, b))
    torch.cuda.synchronize()
    lp = reduce_max_over_ranks(sum(x.elapsed_time(y) for x, y in lp_ms) / len(lp_ms), dev)
    lse_provided = {"ms_per_step": lp, "value": replica_throughput(Tk, world, lp), "unit": "tokens/s",
                    "note": "LSE supplied by the caller (as the attention kernel's LSE would be); "
                            "prep + LSE import + column pass + top-B + compaction"}

    # --- dynamic keep budget: importance -> budget -> top-B -> compaction, with
    # the kept count staying on the device (no host round trip) ----------------
    dyn_keep = torch.empty(R, dtype=torch.int32, device=dev)
    dyn_total = torch.empty(1, dtype=torch.int32, device=dev)
    dyn_idx = torch.empty(Tk, dtype=torch.int32, device=dev)
    dyn_cu = torch.empty(R + 1, dtype=torch.int32, device=dev)
    dyn_h = torch.empty((Tk, D), dtype=torch.bfloat16, device=dev)
    dyn_p = torch.empty((Tk, P), dtype=torch.int32, device=dev)
    dyn_i = torch.empty(Tk, dtype=torch.int32, device=dev)
    DYN = (900, 100, 900)   # tau: 90% of the score mass; keep between 10% and 90%
    dy_ms = []
    for i in range(args.warmup + args.steps):
        flush.fill_(i & 0xFF)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(stream)
        importance(0)
        ev[1].record(stream)
        tsel.tsel_dynamic_budget(scores, d["req_off"], *DYN, keep_per_req=dyn_keep,
                                 total_keep=dyn_total, workspace=ws, stream=stream)
        tsel.tsel_select_topk(scores, d["req_off"], dyn_keep, tsel.TSEL_KEEP_FROM_DEVICE,
                              keep_idx=dyn_idx, cu_keep=dyn_cu, workspace=ws, stream=stream)
        tsel.tsel_gather_compact_counted(d["hidden"], d["pos"], d["cu_k"], dyn_idx, dyn_cu[R:], Tk,
                                         out_hidden=dyn_h, out_pos=dyn_p, out_img_id=dyn_i,
                                         out_cu_seqlens=out_c, workspace=ws, stream=stream)
        ev[2].record(stream)
        if i >= args.warmup:
            dy_ms.append(ev)
    torch.cuda.synchronize()
    if tsel.tsel_read_device_status(ws) != 0:
        raise RuntimeError("device status set in the dynamic-budget run")
    dy = reduce_max_over_ranks(sum(e[0].elapsed_time(e[2]) for e in dy_ms) / len(dy_ms), dev)
    dy_sel = sum(e[1].elapsed_time(e[2]) for e in dy_ms) / len(dy_ms)
    dynamic = {"ms_per_step": dy, "value": replica_throughput(Tk, world, dy), "unit": "tokens/s",
               "selection_ms": dy_sel, "kept": int(dyn_total.item()), "tokens": Tk,
               "mass_permille": DYN[0], "min_permille": DYN[1], "max_permille": DYN[2],
               "note": "per-request budget from the scores (fewest top tokens holding 90% of the "
                       "score quanta, kept between 10% and 90%); budget + top-B + compaction "
                       "read the kept count on the device"}

    # --- FP8 E4M3 Q/K (one scale per tensor folded into the softmax scale) ----
    fp8 = None
    if not args.no_fp8:
        w8 = W.to_e4m3(w)
        q8 = torch.from_numpy(w8.q_bits).to(dev)
        k8 = torch.from_numpy(w8.k_bits).to(dev)
        f_ms, f_imp = [], []
        for i in range(args.warmup + args.steps):
            flush.fill_(i & 0xFF)
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            ev[0].record(stream)
            tsel.tsel_importance(q8, k8, d["cu_q"], d["cu_k"], w.max_seqlen_q, w.max_seqlen_k,
                                 softmax_scale=w8.softmax_scale, lse=lse, scores=scores,
                                 workspace=ws, stream=stream)
            ev[1].record(stream)
            topk()
            gather()
            ev[2].record(stream)
            if i >= args.warmup:
                f_ms.append(ev)
        torch.cuda.synchronize()
        if tsel.tsel_read_device_status(ws) != 0:
            raise RuntimeError("device status set in the FP8 run")
        step = reduce_max_over_ranks(sum(e[0].elapsed_time(e[2]) for e in f_ms) / len(f_ms), dev)
        imp = sum(e[0].elapsed_time(e[1]) for e in f_ms) / len(f_ms)
        fp8 = {"ms_per_step": step, "value": replica_throughput(Tk, world, step),
               "unit": "tokens/s", "importance_ms": imp,
               "note": "Q and K in FP8 E4M3 (kind::f8f6f4 MMAs, K padded to a multiple of "
                       "32), everything else as the bf16 line"}

    # --- end to end through the API with host buffers ------------------------
    e2e = None
    if not args.no_e2e:
        pin = {k: v.pin_memory() for k, v in host.items()}
        # two sets of device inputs: the next request crosses the host link
        # while this one is computed, as a serving loop overlaps them
        dbufs = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
        h_keep = torch.empty(K, dtype=torch.int32).pin_memory()
        h_cu = torch.empty(cu_keep.numel(), dtype=torch.int32).pin_memory()
        h_img = torch.empty(K, dtype=torch.int32).pin_memory()
        h_pos = torch.empty((K, P), dtype=torch.int32).pin_memory()
        h_cuk = torch.empty(G + 1, dtype=torch.int32).pin_memory()
        h2d = sum(v.numel() * v.element_size() for v in pin.values())
        d2h = sum(t.numel() * t.element_size() for t in (h_keep, h_cu, h_img, h_pos, h_cuk))

        copy_stream = torch.cuda.Stream(dev)
        late = ("hidden", "pos")     # needed only by the compaction
        released = [None, None]      # per input set: event after the last kernel that read it

        def e2e_step(i):
            # Every input of request i crosses the link on the copy stream, Q, K
            # and metadata first (one link: copies in parallel would only share
            # its bandwidth); the hidden rows and positions follow while the
            # importance passes run. The copy stream reuses an input set only
            # after the kernels of the request before last have read it.
            db = dbufs[i % 2]
            with torch.cuda.stream(copy_stream):
                if released[i % 2] is not None:
                    copy_stream.wait_event(released[i % 2])
                for k2, v in pin.items():
                    if k2 not in late:
                        db[k2].copy_(v, non_blocking=True)
                ev_first = torch.cuda.Event()
                ev_first.record(copy_stream)
                for k2 in late:
                    db[k2].copy_(pin[k2], non_blocking=True)
                ev_late = torch.cuda.Event()
                ev_late.record(copy_stream)
            stream.wait_event(ev_first)
            score_select(0, db["q"], db["k"], db["cu_q"], db["cu_k"], db["req_off"], db["keep"])
            stream.wait_event(ev_late)
            gather(db["hidden"], db["pos"], db["cu_k"])
            done = torch.cuda.Event()
            done.record(stream)
            released[i % 2] = done
            h_keep.copy_(keep_idx, non_blocking=True)
            h_cu.copy_(cu_keep, non_blocking=True)
            h_img.copy_(out_i, non_blocking=True)
            h_pos.copy_(out_p, non_blocking=True)
            h_cuk.copy_(out_c, non_blocking=True)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        n_e2e = max(5, min(args.steps, 50))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        copy_stream.wait_event(a)   # no copy of the timed steps starts before the clock
        for i in range(n_e2e):
            e2e_step(i)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max_over_ranks(a.elapsed_time(b) / n_e2e, dev)
        # the host link alone: the same input bytes copied in, nothing else
        link = []
        for i in range(4):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(copy_stream)
            with torch.cuda.stream(copy_stream):
                for k2, v in pin.items():
                    dbufs[0][k2].copy_(v, non_blocking=True)
            c1.record(copy_stream)
            link.append((c0, c1))
        torch.cuda.synchronize()
        copy_ms = min(x.elapsed_time(y) for x, y in link[1:])
        e2e = {"value": replica_throughput(Tk, world, e2e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms,
               "h2d_copy_ms": copy_ms, "h2d_GB/s": h2d / (copy_ms * 1e-3) / 1e9,
               "note": "every step copies its request's inputs in from pinned host memory "
                       "(Q, K and metadata, then hidden rows and positions during the importance "
                       "passes; two input sets, so the next request's copy overlaps this one's "
                       "kernels), runs importance+top-B+compaction and copies the selection "
                       "metadata out; compacted hidden rows stay on the device. h2d_copy_ms: "
                       "the same input bytes copied in alone (the step's floor when the "
                       "host link is slower than the kernels)"}

    # --- small requests: whole path replayed from one CUDA graph -------------
    small = {}
    if not args.no_small:
        for name in SMALL_REQUESTS:
            small[name] = small_request_latency(tsel, W.make(name), dev, flush, stream)
            if name in cpu_small:   # the oracle on one host core, same request
                small[name]["cpu_oracle_1core"] = cpu_small[name]

    # --- the other seeded workloads: throughput and importance roofline -------
    sweep = {}
    if not args.no_sweep:
        peaks_s, _ = load_peaks()
        for name in W.WORKLOADS:
            if name == args.workload:
                continue
            sweep[name] = workload_throughput(tsel, W.make(name), dev, flush, stream, ex2_peak,
                                              peaks_s["bf16_tflops"] * 1e12)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # --- roofline ------------------------------------------------------------
    peaks, peak_src = load_peaks()
    bf16_peak = peaks["bf16_tflops"] * 1e12
    hbm_peak = peaks["hbm_gbs"] * 1e9
    E = w.attended_pairs()
    med = {n: statistics.median(v) for n, v in per.items()}
    mean = {n: sum(v) / len(v) for n, v in per.items()}
    sel_mean = sum(sel_span) / len(sel_span)

    def pass_roof(t_ms):
        t_tensor = 2 * hd * E / bf16_peak
        t_exp = E / ex2_peak
        return {"t_tensor_ms": 1e3 * t_tensor, "t_exp_ms": 1e3 * t_exp,
                "bound": "alu" if t_exp >= t_tensor else "tensor",
                "frac": max(t_tensor, t_exp) / (t_ms * 1e-3)}

    roof1, roof2 = pass_roof(mean["pass1"]), pass_roof(mean["pass2"])
    dom = "pass2" if mean["pass2"] >= mean["pass1"] else "pass1"
    t_dom = mean[dom] * 1e-3
    if (roof2 if dom == "pass2" else roof1)["bound"] == "alu":
        roofline = {"kernel": f"imp_pass_kernel<{dom[-1]},{hd}>", "bound": "alu",
                    "achieved": E / t_dom / 1e9, "peak": ex2_peak / 1e9, "unit": "Gex2/s",
                    "frac": (E / t_dom) / ex2_peak}
    else:
        roofline = {"kernel": f"imp_pass_kernel<{dom[-1]},{hd}>", "bound": "tensor",
                    "achieved": 2 * hd * E / t_dom / 1e12, "peak": bf16_peak / 1e12,
                    "unit": "TFLOP/s", "frac": (2 * hd * E / t_dom) / bf16_peak}
    roofline["traffic"] = load_traffic(roofline["kernel"], args.workload)
    roofline["peak_source"] = f"{peak_src}; ex2 peak measured by the probe kernel in this run"
    t_imp = (mean["prep"] + mean["pass1"] + mean["pass2"]) * 1e-3
    imp_roof = max(4 * hd * E / bf16_peak, 2 * E / ex2_peak)
    R = w.keep_per_req.size
    topk_bytes = 4 * Tk + 4 * K + 4 * (R + 1) + 4 * R
    gather_bytes = K * (2 * 2 * D + 2 * 4 * P + 4 + 4) + 4 * 2 * (G + 1)
    kernels = {
        "prep": {"ms": mean["prep"]},
        # the row-LSE pass and its redo launch (which exits at once when no
        # row overflowed the fixed reference: redo_pairs = 0)
        "pass1": {"ms": mean["pass1"], **roof1, "redo_pairs": redo_pairs},
        "pass2": {"ms": mean["pass2"], **roof2},
        # the fused call's top-B, started from the column pass's histograms
        "topk": {"ms": mean["topk"], "GB/s": topk_bytes / (mean["topk"] * 1e-3) / 1e9,
                 "hbm_frac": topk_bytes / (mean["topk"] * 1e-3) / hbm_peak,
                 "in_step_ms": fused_ms - chain_ms if same_chain else None,
                 "in_step_note": f"the fused call {fused_ms:.4f} ms minus the importance chain "
                                 f"alone {chain_ms:.4f} ms (interleaved runs, events only around "
                                 "each): what the top-B adds to the call, its launch overlapping "
                                 "the column pass's drain; `ms` times it alone between events",
                 "paths": dict(zip(["radix", "hist_rounds", "hist_candidates", "rejected",
                                    "in_importance_launch"], topk_paths))},
        "topk_plain": {"ms": mean["topk_plain"],
                       "GB/s": topk_bytes / (mean["topk_plain"] * 1e-3) / 1e9,
                       "note": "tsel_select_topk on the same scores (three radix rounds)"},
        "gather": {"ms": mean["gather"], "GB/s": gather_bytes / (mean["gather"] * 1e-3) / 1e9,
                   "hbm_frac": gather_bytes / (mean["gather"] * 1e-3) / hbm_peak,
                   **gather_dram_rate(args.workload, mean["gather"], gather_bytes, hbm_peak)},
        # top-B + compaction as one selection step: events around the two
        # launches back to back (the path as it runs); "ms_isolated_sum" adds
        # the two kernels timed alone above, each with its own launch latency
        "selection": {"ms": sel_mean,
                      "GB/s": (topk_bytes + gather_bytes) / (sel_mean * 1e-3) / 1e9,
                      "hbm_frac": (topk_bytes + gather_bytes) / (sel_mean * 1e-3) / hbm_peak,
                      "ms_isolated_sum": mean["topk"] + mean["gather"],
                      "hbm_frac_isolated_sum": (topk_bytes + gather_bytes)
                                               / ((mean["topk"] + mean["gather"]) * 1e-3) / hbm_peak,
                      "in_step_ms": whole_ms - chain_ms if same_chain else None,
                      "in_step_GB/s": (topk_bytes + gather_bytes) / ((whole_ms - chain_ms) * 1e-3)
                                      / 1e9 if same_chain else None,
                      "in_step_hbm_frac": (topk_bytes + gather_bytes)
                                          / ((whole_ms - chain_ms) * 1e-3) / hbm_peak
                                          if same_chain else None,
                      "in_step_note": f"whole step {whole_ms:.4f} ms minus the importance chain "
                                      f"alone {chain_ms:.4f} ms (interleaved runs, events only "
                                      "around each): the time top-B and compaction add to the "
                                      "step. `ms` has an event between the column pass and the "
                                      "top-B, which keeps the top-B's launch off the pass's drain"},
    }

    if fp8 is not None:
        kd = (hd + 31) // 32 * 32          # K padded to the f8f6f4 K-step
        t_tensor8 = 2 * 2 * kd * E / (2 * bf16_peak)   # two passes; FP8 peak = 2 x bf16 (nominal ratio)
        t_exp8 = 2 * E / ex2_peak
        fp8["importance_roofline_frac"] = max(t_tensor8, t_exp8) / (fp8["importance_ms"] * 1e-3)

    cpu_baseline = None
    if cpu is not None and "error" not in cpu:
        cpu_baseline = {"value": cpu_rate(cpu), "unit": "tokens/s", "cores": cpu["cores"],
                        "kind": "oracle",
                        "sample": (f"full workload ({args.workload}: {cpu['tokens']} tokens, "
                                   f"{cpu['pairs']:.3g} attended pairs, {cpu['seconds']:.1f} s): "
                                   f"importance image by image over {cpu['cores']} processes "
                                   f"(fp64 numpy, 1 BLAS thread each), then top-B and compaction "
                                   f"once; input generation not timed")}
    elif cpu is not None:
        cpu_baseline = {"value": None, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
                        "sample": "failed: " + cpu["error"]}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(w, args.workload, world, L2_NOTE),
        "importance_roofline_frac": imp_roof / t_imp,
        "roofline": roofline,
        "kernels": kernels,
        "kernel_timing": (f"per-kernel times from {n_stage} further steps with an event between "
                          "the stages (each kernel alone, no launch overlap); the headline step "
                          "(tsel_score_select + tsel_gather_compact) has events only around the "
                          "whole path"),
        "cpu_baseline": cpu_baseline,
        "e2e": e2e,
        "separate_calls": separate_calls,
        "lse_provided": lse_provided,
        "dynamic_budget": dynamic,
        "fp8": fp8,
        "small_requests": small,
        "workloads": sweep,
        # per step: schedule, row-LSE pass, its redo launch, column pass, top-B, gather
        "gpu_launches": 6 * args.steps,
        "clocks": clocks,
        "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"],
                  "ex2_per_s": ex2_peak, "ex2_per_clk_per_sm_at_max":
                      ex2_peak / sms / (clocks["sm_max_mhz"] * 1e6) if clocks.get("sm_max_mhz") else None,
                  "ex2_probe_sm_mhz": probe_mhz,
                  "ex2_per_clk_per_sm_at_probe_clock":
                      ex2_peak / sms / (probe_mhz * 1e6) if probe_mhz else None,
                  "source": peak_src},
        "wall_s_timed": wall,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


REFERENCE_PAIRS_PER_S = 1.0e7   # rough oracle speed per core, all cores busy; only sizes the samples


def _single_thread_blas():
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        os.environ[v] = "1"


def main():
    args = parse_args()
    if args.cpu_child or args.impl == "reference":
        _single_thread_blas()   # before numpy is imported
    if args.cpu_child:
        print(json.dumps(cpu_child(args.cpu_child[0], float(args.cpu_child[1]),
                                   int(args.cpu_child[2]))))
        return
    if args.cpu_small:
        _single_thread_blas()
        print(json.dumps(cpu_small_child()))
        return
    if args.impl == "reference":
        reference_arm(args)
        return
    gpu_arm(args)


if __name__ == "__main__":
    main()
