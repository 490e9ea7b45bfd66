#!/usr/bin/env python
"""Benchmark of the sparse decode step on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl pks|reference]

One step = the whole hot path over one batch: int8 indexer scan of every
cached token, exact top-k, paged sparse attention (plus the residency update
for the workload with an HBM slot table).  Default workload: 16 requests x
131072 tokens, 64-token pages, GQA 64/8, head dim 128, 4-head int8 indexer,
top-2048.  Inputs are seeded synthetic tensors resident in HBM; L2 is flushed
(256 MB write, then 256 MB read of another buffer) between timed steps,
outside the timed intervals.

Prints one JSON line (rank 0).  Under torchrun every rank runs its own
replica batch (weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np
import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from top_sparse_attention_pks_gb300 import build as pkg_build  # noqa: E402
from top_sparse_attention_pks_gb300 import pks  # noqa: E402
from top_sparse_attention_pks_gb300.decoder import MlaDecodeStep, SparseDecodeStep  # noqa: E402
from top_sparse_attention_pks_gb300.workloads import (HISPARSE_WORKLOADS,  # noqa: E402
                                                      MLA_LATENT, MLA_WORKLOADS,
                                                      WORKLOADS, draw_float_weights,
                                                      draw_fp8_indexer, draw_host,
                                                      draw_mla_tensors, draw_tensors)

METRIC = "sparse decode steps/s"
UNIT = "steps/s"
NOMINAL_HBM_GBS = 8000.0  # the roofline denominator the target is stated against
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Evicts L2 between timed steps: a 256 MB write (twice the 129 MB L2),
    then a 256 MB read of a second buffer.  The read writes back the dirty
    lines the write leaves, so the next step starts with an L2 that holds
    none of its inputs and nothing to write back (a write alone leaves up to
    129 MB of dirty lines whose write-back lands inside the next step)."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def repo_libraries():
    """Shared objects of this repository mapped into this process."""
    try:
        maps = Path("/proc/self/maps").read_text().splitlines()
    except OSError:
        return []
    root = str(ROOT)
    return sorted({Path(ln.split()[-1]).name for ln in maps
                   if ln.split()[-1].startswith(root) and ln.split()[-1].endswith(".so")})


def measured_peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------ setup --

def block_table(wl, h, reference=False):
    """The batch's block table: from the library's page pool, or, for the
    oracle's arm (which loads nothing of the library), from the oracle's own
    allocator (the two are checked equal by the host tests)."""
    if reference:
        import oracle
        bt, _ = oracle.build_block_table(h["seq_lens"], wl.page_size, wl.max_pages,
                                         wl.num_pages, h["prefix_group"], wl.prefix_len,
                                         h["free_order"])
        return bt
    pool = pks.Pool(wl.num_pages, wl.page_size, h["free_order"])
    bt, _ = pool.build_block_table(h["seq_lens"], wl.max_pages, h["prefix_group"], wl.prefix_len)
    pool.close()
    return bt


def setup(wl, device, seed_offset=0, reference=False):
    h = draw_host(wl)
    bt = block_table(wl, h, reference)
    t = draw_tensors(wl, device, seed_offset)
    t["seq_lens"] = h["seq_lens"].to(device)
    t["block_table"] = torch.from_numpy(bt).to(device)
    return t, h, bt


def algorithmic_bytes(wl, lens, bt, topk):
    """Unique physical bytes of one step: indexer keys scanned, K/V rows
    gathered, outputs written (aliased prefix pages counted once).  With
    several query tokens per request (topk [B, Nq, k]) every query's gather
    counts: rows are unique within a query's selections, summed over queries."""
    P = wl.page_size
    topk = np.asarray(topk)
    if topk.ndim == 2:
        topk = topk[:, None, :]
    nq = topk.shape[1]
    scan_rows, kv_rows = [], [[] for _ in range(nq)]
    for b, n in enumerate(lens):
        n = int(n)
        if n == 0:
            continue
        t = np.arange(n, dtype=np.int64)
        scan_rows.append(bt[b, t // P].astype(np.int64) * P + t % P)
        for q in range(nq):
            sel = topk[b, q][topk[b, q] >= 0].astype(np.int64)
            kv_rows[q].append(bt[b, sel // P].astype(np.int64) * P + sel % P)
    n_scan = np.unique(np.concatenate(scan_rows)).size if scan_rows else 0
    n_kv = sum(np.unique(np.concatenate(r)).size for r in kv_rows if r)
    scan = n_scan * wl.Di
    kv = n_kv * wl.Hkv * wl.D * 2 * 2
    out = wl.B * nq * wl.Hq * wl.D * 2
    attended = nq * int(sum(min(int(n), wl.k) for n in lens))
    return dict(scan=scan, kv=kv, out=out, total=scan + kv + out, attended=attended)


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = Path(os.environ.get("TMPDIR", "/tmp")) / f"pks_clocks_{os.getpid()}.csv"

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in self.path.read_text().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), sm_max=float(parts[2]),
                                 reasons=parts[5:9]))
            except ValueError:
                continue
        self.path.unlink(missing_ok=True)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        active = sorted({names[i] for r in rows for i, v in enumerate(r["reasons"])
                         if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["sm_max"] for r in rows),
                "reasons": active, "samples": len(rows)}


# ------------------------------------------------------------ oracle arm --

def oracle_request_step(wl, t_host, b, n_tokens):
    """The oracle's whole step for request b truncated to n_tokens tokens."""
    import oracle
    P = wl.page_size
    lens = np.array([n_tokens], np.int32)
    if t_host.get("fp8"):  # FP8 e4m3 indexer: exact scores, selection on their fp32 values
        scores = oracle.indexer_scores_fp8(lens, t_host["bt"][b: b + 1], P,
                                           t_host["q_idx"][b: b + 1], t_host["w_f"][b: b + 1],
                                           t_host["idx_k"])
        idx = oracle.topk_f(lens, scores.astype(np.float32), wl.k)
    elif t_host.get("w_f") is not None:  # real-valued head weights
        scores = oracle.indexer_scores_f(lens, t_host["bt"][b: b + 1], P,
                                         t_host["q_idx"][b: b + 1], t_host["w_f"][b: b + 1],
                                         t_host["idx_k"])
        idx = oracle.topk_f(lens, scores, wl.k)
    else:
        scores = oracle.indexer_scores(lens, t_host["bt"][b: b + 1], P,
                                       t_host["q_idx"][b: b + 1], t_host["w_idx"],
                                       t_host["idx_k"])
        idx = oracle.topk(lens, scores, wl.k)
    oracle.sparse_attention(t_host["bt"][b: b + 1], P, idx, t_host["q"][b: b + 1],
                            t_host["kv_k"], t_host["kv_v"])


def oracle_inputs(wl, t, b):
    """Host copies of request b's pages, remapped to a compact pool."""
    lens = t["seq_lens"].cpu().numpy()
    bt = t["block_table"].cpu().numpy()
    n_pages = -(-int(lens[b]) // wl.page_size)
    pages = torch.from_numpy(bt[b, :n_pages].astype(np.int64)).to(t["kv_k"].device)
    cbt = np.full((wl.B, wl.max_pages), -1, np.int32)
    cbt[b, :n_pages] = np.arange(n_pages)
    return dict(bt=cbt, q_idx=t["q_idx"].cpu().numpy(), w_idx=t["w_idx"].cpu().numpy(),
                q=t["q"].cpu(), idx_k=t["idx_k"].index_select(0, pages).cpu().numpy(),
                kv_k=t["kv_k"].index_select(0, pages).cpu(),
                kv_v=t["kv_v"].index_select(0, pages).cpu(), len=int(lens[b]),
                w_f=t["w_idx_f"].cpu().numpy() if "w_idx_f" in t else None,
                fp8=bool(t.get("idx_fp8", False)))


def time_oracle(wl, t, budget_s, min_reps=1, steps=None, warmup=0):
    """Time the oracle on request 0 (longest-context request of the batch)."""
    import oracle
    cores = oracle.set_threads(0)
    lens = t["seq_lens"].cpu().numpy()
    b = int(np.argmax(lens))
    hi = oracle_inputs(wl, t, b)
    full = hi["len"]
    # calibrate on a slice, then choose the slice each timed step covers
    n0 = min(full, max(4 * wl.k, 8192))
    t0 = time.perf_counter()
    oracle_request_step(wl, hi, b, n0)
    c = (time.perf_counter() - t0) / n0
    n_steps = steps if steps is not None else None
    if n_steps is None:
        n_tok = full
    else:
        per_step = budget_s / max(1, n_steps + warmup)
        n_tok = int(min(full, max(min(full, 4 * wl.k), per_step / max(c, 1e-12))))
    for _ in range(warmup):
        oracle_request_step(wl, hi, b, n_tok)
    times = []
    t_start = time.perf_counter()
    while True:
        s = time.perf_counter()
        oracle_request_step(wl, hi, b, n_tok)
        times.append(time.perf_counter() - s)
        if n_steps is not None:
            if len(times) >= n_steps:
                break
        elif len(times) >= min_reps and time.perf_counter() - t_start >= budget_s:
            break
    mean = sum(times) / len(times)
    total_tokens = float(lens.sum())
    step_time = mean * total_tokens / n_tok  # scaled to the whole batch
    sample = (f"request {b} ({full} tokens) truncated to {n_tok} tokens per timed step, "
              f"{len(times)} steps; time scaled by tokens to the {wl.B}-request batch "
              f"({int(total_tokens)} tokens)")
    return dict(value=1.0 / step_time, unit=UNIT, cores=cores, kind="oracle", sample=sample,
                step_seconds=step_time, reps=len(times))


# ------------------------------------------------------------------ main --

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="b16_128k",
                    choices=sorted(WORKLOADS) + sorted(MLA_WORKLOADS) + sorted(HISPARSE_WORKLOADS))
    ap.add_argument("--impl", default="pks", choices=["pks", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stage-steps", type=int, default=200)
    ap.add_argument("--e2e-steps", type=int, default=500)
    ap.add_argument("--requests", type=int, default=0,
                    help="keep only the first N requests (smaller profiling case)")
    ap.add_argument("--topk", type=int, default=0, help="override the workload's k")
    ap.add_argument("--queries", type=int, default=1,
                    help="query tokens per request (each scores, selects and attends alone)")
    ap.add_argument("--layers", type=int, default=1,
                    help="with --hisparse: layers, each with its own pools and table")
    ap.add_argument("--hisparse", action="store_true",
                    help="workloads with a slot table: K/V in pinned host memory, HBM slots, "
                         "misses fetched every step (select, update, fetch, attention)")
    ap.add_argument("--float-weights", action="store_true",
                    help="real-valued indexer head weights, float [B, Hi] (fp32 scores), "
                         "uniform in [0.25, 2)")
    ap.add_argument("--signed-weights", action="store_true",
                    help="with --float-weights: weights uniform in [-2, 2)")
    ap.add_argument("--fp8-indexer", action="store_true",
                    help="FP8 e4m3 indexer queries and keys (implies --float-weights)")
    ap.add_argument("--mla", action="store_true",
                    help="the DSA step with sparse MLA attention (MQA mode, tcgen05): "
                         "indexer scan, top-k, MLA over the selection; default workload "
                         "mla_b16_128k")
    args = ap.parse_args()
    if args.mla and args.workload == "b16_128k":
        args.workload = "mla_b16_128k"
    if (args.workload in MLA_WORKLOADS) != args.mla:
        ap.error("MLA workloads run with --mla (and --mla only with MLA workloads)")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "pks" else "gloo")
    if args.impl == "reference" and rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        if args.impl == "reference":
            import oracle  # the reference arm runs the oracle alone: libpks is not built
            oracle.build()
        else:
            pkg_build.build_library()
    if dist:
        dist.barrier()
    if args.mla:
        mla_bench(MLA_WORKLOADS[args.workload], args, dev, rank, world, dist)
        if dist:
            dist.destroy_process_group()
        return
    if (args.workload in HISPARSE_WORKLOADS) and not args.hisparse:
        ap.error("HBM-residency workloads run with --hisparse")
    wl = {**WORKLOADS, **HISPARSE_WORKLOADS}[args.workload]
    if args.requests:
        wl = shrink(wl, args.requests)
    if args.topk:
        wl = wl.replace(k=args.topk)
    t, h, bt = setup(wl, dev, seed_offset=rank, reference=args.impl == "reference")
    if args.queries > 1:
        # Nq query tokens per request: seeded queries of shape [B, Nq, ...]
        gen = torch.Generator(device=dev)
        gen.manual_seed(2000 + rank)
        t["q"] = torch.randn((wl.B, args.queries, wl.Hq, wl.D), device=dev,
                             generator=gen).to(torch.bfloat16)
        t["q_idx"] = torch.randint(-127, 128, (wl.B, args.queries, wl.Hi, wl.Di),
                                   dtype=torch.int8, device=dev, generator=gen)
        args.no_cpu_baseline = True
    if args.fp8_indexer:
        args.float_weights = True
        t["q_idx"], t["idx_k"] = draw_fp8_indexer(wl, dev, seed_offset=rank)
        t["idx_fp8"] = True
    if args.float_weights:
        t["w_idx_f"] = draw_float_weights(wl, dev, seed_offset=rank, signed=args.signed_weights)

    if args.impl == "reference":
        ref = time_oracle(wl, t, budget_s=120.0, steps=args.steps, warmup=args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": ref["value"], "unit": UNIT,
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ref["step_seconds"] * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "int64+f64",
                "data": "synthetic", "config": config_dict(wl, args),
                "cpu_baseline": {k: ref[k] for k in ("value", "unit", "cores", "kind",
                                                     "sample")},
                "e2e": {"value": ref["value"], "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "loaded_libraries": repo_libraries()}
        print(json.dumps(line), flush=True)
        if dist:
            dist.destroy_process_group()
        return

    if args.hisparse:
        if wl.capacity <= 0:
            ap.error("--hisparse needs a workload with a slot table")
        hisparse_bench(wl, t, h, args, dev, rank)
        if dist:
            dist.destroy_process_group()
        return

    step = SparseDecodeStep(t, wl.k)
    res = None
    miss = n_miss = None
    if wl.capacity > 0:
        res = pks.ResidencyTable(wl.num_pages, wl.capacity, h["initial_resident"].numpy(),
                                 device=dev)
        miss = torch.empty(wl.num_pages, dtype=torch.int32, device=dev)
        n_miss = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())

    if res is not None:
        # the residency update (one CTA) needs only the selection: it runs on a
        # side stream beside the attention, whose grid leaves one SM free for it
        side = torch.cuda.Stream(device=dev)
        ev_fork = torch.cuda.Event()
        ev_join = torch.cuda.Event()
        attn_args = pks.pks_decode_args.from_buffer_copy(step.args)
        attn_args.attn_splits = torch.cuda.get_device_properties(dev).multi_processor_count - 1

    def one_step(stream):
        if res is None:
            step(stream)
            return
        pks.pks_decode_select(step.args, stream)
        ev_fork.record(stream)
        side.wait_event(ev_fork)
        res.update(step.topk_idx, t["block_table"], wl.page_size, miss, n_miss, side)
        pks.pks_sparse_attention(attn_args, stream)
        ev_join.record(side)
        stream.wait_event(ev_join)

    with torch.cuda.stream(s):
        for _ in range(3):
            one_step(s)
    torch.cuda.synchronize()
    if step.device_error(s) != 0:
        raise RuntimeError("device-side check fired during warm-up")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        one_step(s)
    # scan, top-k, attention + merge as the library reports them (+ residency
    # mark and update)
    launches_per_step = step.launches() + (2 if res is not None else 0)

    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            flush()
            g.replay()
    torch.cuda.synchronize()
    topk_host = step.topk_idx.cpu().numpy()
    ab = algorithmic_bytes(wl, h["seq_lens"].numpy(), bt, topk_host)

    # ---- timed region: K graph replays, each bracketed by events; L2 flushed
    # between steps outside the intervals
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the work
    with torch.cuda.stream(s):
        for i in range(args.steps):
            flush()
            starts[i].record(s)
            g.replay()
            ends[i].record(s)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    value, total_s = job_throughput(sum(step_ms) / 1e3, args.steps, world, dist, dev)
    ms_per_step = total_s * 1e3 / args.steps

    # ---- with an HBM slot table: the same step without the residency update
    # (graph of the decode step alone), reported beside the full step
    no_residency = None
    if res is not None:
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=s):
            step(s)
        n2 = min(args.steps, 500)
        st2 = [torch.cuda.Event(enable_timing=True) for _ in range(n2)]
        en2 = [torch.cuda.Event(enable_timing=True) for _ in range(n2)]
        with torch.cuda.stream(s):
            for _ in range(args.warmup):
                flush()
                g2.replay()
            for i in range(n2):
                flush()
                st2[i].record(s)
                g2.replay()
                en2[i].record(s)
        torch.cuda.synchronize()
        ms2 = statistics.median(a.elapsed_time(b) for a, b in zip(st2, en2))
        no_residency = {"ms_per_step": ms2, "value": 1e3 / ms2, "steps": n2,
                        "residency_update_ms": ms_per_step - ms2}

    # ---- per-stage times inside the real step (events between the stages)
    stage = {"scan": [], "topk": [], "attention": []}
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
           for _ in range(args.stage_steps)]
    with torch.cuda.stream(s):
        for row in evs:  # torch creates the CUDA events on first record
            for e in row:
                e.record(s)
        for i in range(args.stage_steps):
            flush()
            step.timed(evs[i], s)
    torch.cuda.synchronize()
    for e in evs:
        stage["scan"].append(e[0].elapsed_time(e[1]))
        stage["topk"].append(e[1].elapsed_time(e[2]))
        stage["attention"].append(e[2].elapsed_time(e[3]))
    stage_ms = {k: sum(v) / len(v) for k, v in stage.items()}
    peak, peak_kind = measured_peaks()
    kern_bytes = {"scan": ab["scan"], "attention": ab["kv"] + ab["out"]}
    dominant = max(("scan", "attention"), key=lambda k: stage_ms[k])
    achieved = kern_bytes[dominant] / (stage_ms[dominant] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": {"scan": "k_indexer_scan",
                                           "attention": "k_sparse_attention"}[dominant],
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy test)",
                "traffic": profiled_traffic(dominant, wl.name),
                "algorithmic_bytes_per_launch": kern_bytes[dominant],
                "launch_ms": stage_ms[dominant]}
    step_gbs = ab["total"] / (ms_per_step * 1e-3) / 1e9

    # ---- end to end through the public call with host buffers
    e2e = end_to_end(step, t, wl, args, s, flush, res, miss, n_miss)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = time_oracle(wl, t, budget_s=15.0)
        cpu = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "config": config_dict(wl, args),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "clocks": clk,
            "step_hbm": {"algorithmic_bytes": ab["total"], "scan_bytes": ab["scan"],
                         "kv_bytes": ab["kv"], "out_bytes": ab["out"],
                         "achieved_gbs": step_gbs,
                         "frac_of_8tbs": step_gbs / NOMINAL_HBM_GBS,
                         "frac_of_measured": step_gbs / peak},
            "tokens_attended_per_s": ab["attended"] * value,
            "stages_ms": stage_ms,
            "step_ms_p10_p50_p90": [float(np.percentile(step_ms, q)) for q in (10, 50, 90)],
        }
        if no_residency is not None:
            line["without_residency_update"] = no_residency
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def mla_setup(wl, device, seed_offset=0, reference=False):
    h = draw_host(wl)
    bt = block_table(wl, h, reference)
    t = draw_mla_tensors(wl, device, seed_offset)
    t["seq_lens"] = h["seq_lens"].to(device)
    t["block_table"] = torch.from_numpy(bt).to(device)
    return t, h, bt


def mla_algorithmic(wl, lens, bt, topk):
    """One MLA step's algorithmic bytes and FLOPs: indexer keys scanned, the
    unique selected latent rows (d + r bf16 values), queries and outputs; the
    pages' MQA-mode FLOP count 2 H (d + r) + 2 H d per attended token."""
    P = wl.page_size
    scan_rows, kv_rows, attended = [], [], 0
    for b, n in enumerate(lens):
        n = int(n)
        if n == 0:
            continue
        t = np.arange(n, dtype=np.int64)
        scan_rows.append(bt[b, t // P].astype(np.int64) * P + t % P)
        sel = topk[b][topk[b] >= 0].astype(np.int64)
        kv_rows.append(bt[b, sel // P].astype(np.int64) * P + sel % P)
        attended += sel.size
    n_scan = np.unique(np.concatenate(scan_rows)).size if scan_rows else 0
    n_kv = np.unique(np.concatenate(kv_rows)).size if kv_rows else 0
    scan = n_scan * wl.Di
    kv = n_kv * wl.D * 2
    q = wl.B * wl.Hq * wl.D * 2
    out = wl.B * wl.Hq * MLA_LATENT * 2
    flops = attended * 2 * wl.Hq * (wl.D + MLA_LATENT)
    return dict(scan=scan, kv=kv, q=q, out=out, attention=kv + q + out,
                total=scan + kv + q + out, flops=flops, attended=attended)


def time_mla_oracle(wl, t, budget_s, steps=None, warmup=0):
    """The oracle's MLA step (indexer scores, top-k, MLA attention) on the
    longest request, truncated so that a timed step fits the budget; the time
    is scaled by tokens to the whole batch."""
    import oracle
    cores = oracle.set_threads(0)
    lens = t["seq_lens"].cpu().numpy()
    b = int(np.argmax(lens))
    full = int(lens[b])
    n_pages = -(-full // wl.page_size)
    bt = t["block_table"].cpu().numpy()
    pages = torch.from_numpy(bt[b, :n_pages].astype(np.int64)).to(t["kv"].device)
    cbt = np.arange(n_pages, dtype=np.int32)[None]
    q_idx = t["q_idx"].cpu().numpy()[b: b + 1]
    w_idx = t["w_idx"].cpu().numpy()
    q = t["q"].cpu()[b: b + 1]
    idx_k = t["idx_k"].index_select(0, pages).cpu().numpy()
    kv = t["kv"].index_select(0, pages).cpu()

    fp8 = bool(t.get("idx_fp8", False))
    w_f = t["w_idx_f"].cpu().numpy()[b: b + 1] if "w_idx_f" in t else None

    def one(n_tok):
        ln = np.array([n_tok], np.int32)
        if fp8:
            sc = oracle.indexer_scores_fp8(ln, cbt, wl.page_size, q_idx, w_f, idx_k)
            idx = oracle.topk_f(ln, sc.astype(np.float32), wl.k)
        elif w_f is not None:
            sc = oracle.indexer_scores_f(ln, cbt, wl.page_size, q_idx, w_f, idx_k)
            idx = oracle.topk_f(ln, sc, wl.k)
        else:
            sc = oracle.indexer_scores(ln, cbt, wl.page_size, q_idx, w_idx, idx_k)
            idx = oracle.topk(ln, sc, wl.k)
        oracle.mla_sparse_attention(cbt, wl.page_size, idx, q, kv, MLA_LATENT)

    n0 = min(full, max(4 * wl.k, 8192))
    t0 = time.perf_counter()
    one(n0)
    c = (time.perf_counter() - t0) / n0
    per_step = budget_s / max(1, (steps or 3) + warmup)
    n_tok = int(min(full, max(min(full, 2 * wl.k), per_step / max(c, 1e-12))))
    for _ in range(warmup):
        one(n_tok)
    times = []
    for _ in range(steps or 3):
        s0 = time.perf_counter()
        one(n_tok)
        times.append(time.perf_counter() - s0)
    mean = sum(times) / len(times)
    step_time = mean * float(lens.sum()) / n_tok
    sample = (f"request {b} ({full} tokens) truncated to {n_tok} tokens per timed step, "
              f"{len(times)} steps; time scaled by tokens to the {wl.B}-request batch")
    return dict(value=1.0 / step_time, unit=UNIT, cores=cores, kind="oracle", sample=sample,
                step_seconds=step_time)


def mla_bench(wl, args, dev, rank, world, dist):
    """The DSA decode step with sparse MLA: pks_decode_select (scan + top-k)
    and pks_mla_sparse_attention, captured in one CUDA graph."""
    if args.requests:
        wl = shrink(wl, args.requests)
    if args.topk:
        wl = wl.replace(k=args.topk)
    t, h, bt = mla_setup(wl, dev, seed_offset=rank, reference=args.impl == "reference")
    if args.fp8_indexer:  # DSA's indexer: FP8 e4m3 queries and keys, real head weights
        args.float_weights = True
        t["q_idx"], t["idx_k"] = draw_fp8_indexer(wl, dev, seed_offset=rank)
        t["idx_fp8"] = True
    if args.float_weights:
        t["w_idx_f"] = draw_float_weights(wl, dev, seed_offset=rank, signed=args.signed_weights)
    cfg = config_dict(wl, args)
    cfg.update({"attention": "sparse MLA, MQA mode (tcgen05)", "mla_heads": wl.Hq,
                "latent_rope": [MLA_LATENT, wl.D - MLA_LATENT], "heads_q_kv": None,
                "head_dim": None})
    if args.impl == "reference":
        ref = time_mla_oracle(wl, t, budget_s=120.0, steps=args.steps, warmup=args.warmup)
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": ref["value"],
                          "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
                          "warmup": args.warmup, "ms_per_step": ref["step_seconds"] * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "int64+f64", "data": "synthetic", "config": cfg,
                          "cpu_baseline": {k: ref[k] for k in ("value", "unit", "cores",
                                                               "kind", "sample")},
                          "e2e": {"value": ref["value"], "unit": UNIT,
                                  "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                          "loaded_libraries": repo_libraries()}),
              flush=True)
        return
    step = MlaDecodeStep(t, wl.k)
    flush = L2Flush(dev)
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(3):
            step(s)
    torch.cuda.synchronize()
    if step.attention.device_error(s) != 0:
        raise RuntimeError("device-side check fired during warm-up")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    sel_launches = pks.pks_decode_launches(step.select_args) - 2  # scan + top-k only
    # the MLA kernel, plus the merge when the workspace holds split partials
    mla_launches = 1 + (1 if pks.pks_mla_workspace_size(step.attention.args) > 256 else 0)
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            flush()
            g.replay()
    torch.cuda.synchronize()
    ab = mla_algorithmic(wl, h["seq_lens"].numpy(), bt, step.topk_idx.cpu().numpy())

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(dev.index or 0)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    with torch.cuda.stream(s):
        for i in range(args.steps):
            flush()
            starts[i].record(s)
            g.replay()
            ends[i].record(s)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if dist:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    value, total_s = job_throughput(sum(step_ms) / 1e3, args.steps, world, dist, dev)
    ms_per_step = total_s * 1e3 / args.steps

    # stages: select (scan + top-k) and the MLA attention (+ merge), events on s
    n_st = max(1, args.stage_steps)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_st)]
    with torch.cuda.stream(s):
        for row in evs:
            for e in row:
                e.record(s)
        for i in range(n_st):
            flush()
            evs[i][0].record(s)
            step.select(s)
            evs[i][1].record(s)
            pks.pks_mla_sparse_attention(step.attention.args, s)
            evs[i][2].record(s)
    torch.cuda.synchronize()
    sel_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / n_st
    mla_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / n_st
    peak, peak_kind = measured_peaks()
    peaks = json.loads((ROOT / "MEASURED_PEAKS.json").read_text()) if peak_kind == "measured" \
        else {"bf16_tflops": 1900.0}
    mla_gbs = ab["attention"] / (mla_ms * 1e-3) / 1e9
    mla_tfs = ab["flops"] / (mla_ms * 1e-3) / 1e12
    tf_peak = float(peaks["bf16_tflops"])
    mla_roof = {"kernel": "k_mla_attention (+ k_mla_merge)", "launch_ms": mla_ms,
                "algorithmic_bytes_per_launch": ab["attention"], "achieved_gbs": mla_gbs,
                "frac_hbm": mla_gbs / peak, "flops_per_launch": ab["flops"],
                "achieved_tflops": mla_tfs, "frac_bf16": mla_tfs / tf_peak,
                "intensity_flop_per_byte": ab["flops"] / max(1, ab["attention"])}
    mla_roof["traffic"] = profiled_traffic("mla", wl.name)
    if sel_ms >= mla_ms:
        roofline = {"bound": "hbm", "kernel": "k_indexer_scan (+ top-k)",
                    "achieved": ab["scan"] / (sel_ms * 1e-3) / 1e9, "peak": peak,
                    "unit": "GB/s", "traffic": None, "algorithmic_bytes_per_launch": ab["scan"],
                    "launch_ms": sel_ms}
    else:
        tensor = mla_roof["frac_bf16"] > mla_roof["frac_hbm"]
        roofline = {"bound": "tensor" if tensor else "hbm", "kernel": "k_mla_attention",
                    "achieved": mla_tfs if tensor else mla_gbs,
                    "peak": tf_peak if tensor else peak,
                    "unit": "TFLOP/s" if tensor else "GB/s",
                    "traffic": profiled_traffic("mla", wl.name),
                    "algorithmic_bytes_per_launch": ab["attention"], "launch_ms": mla_ms}
    roofline["frac"] = roofline["achieved"] / roofline["peak"]
    roofline["peak_kind"] = f"{peak_kind} (MEASURED_PEAKS.json)"

    # end to end: queries and lengths/tables in from pinned host memory, the
    # public calls, output and top-k back to pinned host memory
    names = ["q", "q_idx", "seq_lens", "block_table"]
    host_in = {n: t[n].cpu().pin_memory() for n in names}
    out_h = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    idx_h = torch.empty(step.topk_idx.shape, dtype=torch.int32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = out_h.numel() * out_h.element_size() + idx_h.numel() * idx_h.element_size()
    n = max(1, min(args.steps, args.e2e_steps))

    def call():  # the calls a user makes for one step
        pks.pks_stage_copy([(t[nm], host_in[nm]) for nm in names], s)
        pks.pks_decode_select(step.select_args, s)
        pks.pks_mla_sparse_attention(step.attention.args, s)
        pks.pks_stage_copy([(out_h, step.out), (idx_h, step.topk_idx)], s)

    with torch.cuda.stream(s):
        call()
    s.synchronize()
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge, stream=s):
        call()
    tot = 0.0
    with torch.cuda.stream(s):
        for i in range(n + 3):
            flush()
            s.synchronize()
            t0 = time.perf_counter()
            ge.replay()
            s.synchronize()
            if i >= 3:
                tot += time.perf_counter() - t0
    e2e = {"value": n / tot, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": n, "timing": "host wall clock per step: one CUDA-graph replay of the step's "
                                 "calls (pks_stage_copy in from pinned memory, select, MLA, "
                                 "pks_stage_copy out) and a stream synchronise"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = time_mla_oracle(wl, t, budget_s=15.0)
        cpu = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    if rank == 0:
        step_gbs = ab["total"] / (ms_per_step * 1e-3) / 1e9
        print(json.dumps({
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": cfg, "roofline": roofline, "mla_attention": mla_roof,
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": (sel_launches + mla_launches) * args.steps, "clocks": clk,
            "step_hbm": {"algorithmic_bytes": ab["total"], "achieved_gbs": step_gbs,
                         "frac_of_8tbs": step_gbs / NOMINAL_HBM_GBS,
                         "frac_of_measured": step_gbs / peak},
            "tokens_attended_per_s": ab["attended"] * value,
            "stages_ms": {"select": sel_ms, "mla_attention": mla_ms},
            "step_ms_p10_p50_p90": [float(np.percentile(step_ms, q)) for q in (10, 50, 90)],
        }), flush=True)


def hisparse_bench(wl, t, h, args, dev, rank):
    """The decode step with the KV cache in pinned host memory and an LRU cache
    of its pages in HBM, over ``--layers`` layers (each its own pools, table and
    queries): select, residency update, miss fetch, attention through the
    table.  Timed twice on separate tables: every call of every layer one after
    another, and with each layer's fetch on a side stream under the
    neighbouring layers' selection and attention.  Prints one JSON line."""
    from top_sparse_attention_pks_gb300.decoder import ResidentLayers
    n_layers = max(1, args.layers)
    layers, q_var = [], []
    for l in range(n_layers):
        tl = dict(t) if l == 0 else setup(wl, dev, seed_offset=rank * 100 + l)[0]
        hk = tl["kv_k"].cpu().pin_memory()
        hv = tl["kv_v"].cpu().pin_memory()
        tl = dict(tl)
        del tl["kv_k"], tl["kv_v"]  # the pools live in host memory only
        layers.append(dict(tensors=tl, host_k=hk, host_v=hv,
                           init_pages=h["initial_resident"].numpy()))
        # a decode step brings a new indexer query: 8 seeded ones in rotation
        gen = torch.Generator(device=dev)
        gen.manual_seed(1000 + 100 * rank + l)
        q_var.append([torch.randint(-127, 128, tl["q_idx"].shape, dtype=torch.int8, device=dev,
                                    generator=gen) for _ in range(8)])
    torch.cuda.empty_cache()
    runs = {"serial": ResidentLayers(layers, wl.k, wl.capacity),
            "overlapped": ResidentLayers(layers, wl.k, wl.capacity)}
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    flush = L2Flush(dev)
    page_bytes = layers[0]["host_k"][0].numel() * layers[0]["host_k"].element_size()

    def set_queries(i):
        for l, L in enumerate(layers):
            L["tensors"]["q_idx"].copy_(q_var[l][i % 8])

    n = max(1, min(args.steps, 100))
    res = {}
    for name, run in runs.items():
        with torch.cuda.stream(s):
            for i in range(args.warmup):
                set_queries(i)
                run(s, overlap=name == "overlapped")
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        fetched = []
        for i in range(n):
            with torch.cuda.stream(s):
                set_queries(args.warmup + i)
                flush()
                ev[i][0].record(s)
                run(s, overlap=name == "overlapped")
                ev[i][1].record(s)
            if i < 10:  # admitted misses of this step, all layers
                torch.cuda.synchronize()
                k = 0
                for lay in run.layers:
                    nm = int(lay.n_miss.item())
                    ps = lay.table.page_slot()[lay.miss[:nm].long()]
                    k += int((ps >= 0).sum().item())
                fetched.append(k)
        torch.cuda.synchronize()
        res[name] = (float(np.median([e[0].elapsed_time(e[1]) for e in ev])),
                     float(np.mean(fetched)))
    # the four calls of layer 0, one after another, timed alone
    lay = runs["serial"].layers[0]
    st = []
    for i in range(min(n, 20)):
        with torch.cuda.stream(s):
            set_queries(i)
            flush()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
            e[0].record(s)
            lay.select(s)
            e[1].record(s)
            lay.update(s)
            e[2].record(s)
            lay.fetch(s)
            e[3].record(s)
            lay.attend(s)
            e[4].record(s)
        torch.cuda.synchronize()
        st.append([e[j].elapsed_time(e[j + 1]) for j in range(4)])
    med = np.median(np.array(st), axis=0)
    step_ms, fetch_pages = res["overlapped"]
    fetch_bytes = 2 * fetch_pages * page_bytes / n_layers
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": 1e3 / step_ms, "unit": UNIT, "n_gpus": 1,
            "steps": n, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": dict(config_dict(wl, args), kv_pools="pinned host memory",
                           hbm_slots=wl.capacity, layers=n_layers),
            "step_ms": {"overlapped": step_ms, "serial": res["serial"][0]},
            "layer0_stages_ms": {"select": med[0], "residency_update": med[1],
                                 "fetch": med[2], "attention": med[3]},
            "fetch": {"pages_per_layer_step": fetch_pages / n_layers,
                      "bytes_per_layer_step": fetch_bytes,
                      "gbs_alone": fetch_bytes / (med[2] * 1e-3) / 1e9 if med[2] > 0 else None},
            "timing": "CUDA events around each step (all layers), L2 flushed (256 MB write + "
                      "256 MB read) before each step; median over the steps",
            "queries": "a new seeded indexer query each step (8 in rotation per layer)",
        }), flush=True)


def job_throughput(local_s, steps, world, dist=None, device="cpu"):
    """Whole-job steps/s: every rank ran `steps` replica steps; the job took
    as long as its slowest rank (max over ranks).  Returns (value, max_s)."""
    total_s = float(local_s)
    if dist is not None and world > 1:
        tt = torch.tensor([total_s], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_s = float(tt.item())
    return world * steps / total_s, total_s


def shrink(wl, n):
    """The first n requests of a workload, with the pool cut to match."""
    if n >= wl.B:
        return wl
    kw = dict(B=n, num_pages=max(1, wl.num_pages * n // wl.B))
    if wl.seq_lens:
        kw["seq_lens"] = tuple(wl.seq_lens[:n])
    if wl.capacity:
        kw["capacity"] = max(1, wl.capacity * n // wl.B)
        kw["initial_resident"] = max(0, wl.initial_resident * n // wl.B)
    return wl.replace(**kw)


def config_dict(wl, args):
    return {"workload": wl.name, "requests": wl.B,
            "seq_len": list(wl.seq_lens) if wl.seq_lens and len(set(wl.seq_lens)) > 1
            else (wl.seq_lens[0] if wl.seq_lens else f"U[{wl.len_lo},{wl.len_hi}]"),
            "page_size": wl.page_size, "heads_q_kv": [wl.Hq, wl.Hkv], "head_dim": wl.D,
            "indexer_heads_dim": [wl.Hi, wl.Di],
            "indexer_dtype": "fp8 e4m3" if getattr(args, "fp8_indexer", False) else "int8",
            "top_k": wl.k,
            "kv_dtype": "bf16", "prefix": [wl.prefix_len, wl.group_size],
            "query_tokens": getattr(args, "queries", 1),
            "indexer_weights": ("float32 [B, Hi] U[-2,2)" if getattr(args, "signed_weights", False)
                                else "float32 [B, Hi] U[0.25,2)")
            if getattr(args, "float_weights", False) else "int32 [Hi] (ones)",
            "residency_slots": wl.capacity, "parallelism": f"replicas x{args.gpus}",
            "l2": "flushed between timed steps (256 MB write, then 256 MB read of another buffer; outside the timed intervals)",
            "timing": "CUDA events around each CUDA-graph replay of the step"}


PROFILED = {"scan": ("k_indexer.cu", "k_indexer_scan"),
            "attention": ("k_attention.cu", "k_sparse_attention"),
            "mla": ("k_mla.cu", "k_mla_attention")}


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    import hashlib
    src_name, prof_name = PROFILED[kernel]
    src = ROOT / "top_sparse_attention_pks_gb300" / "csrc" / src_name
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    prof = ROOT / "profiles" / f"{prof_name}_{workload}.md"
    if not prof.exists():
        return None
    kv = {}
    for line in prof.read_text().splitlines():
        if line.startswith("- ") and ":" in line:
            key, _, val = line[2:].partition(":")
            kv[key.strip()] = val.strip().strip("`")
    if kv.get("source_sha256_16") != sha:
        return None
    try:
        return int(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def end_to_end(step, t, wl, args, s, flush, res, miss, n_miss):
    """Per step: pinned host -> device copy of the step's inputs (queries,
    lengths, block table; one pks_stage_copy), the public pks_decode_step
    call, device -> pinned host copy of the outputs (attention output, top-k;
    one pks_stage_copy), host synchronise."""
    names = ["q", "q_idx", "seq_lens", "block_table"]
    host_in = {n: t[n].cpu().pin_memory() for n in names}
    out_h = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    idx_h = torch.empty(step.topk_idx.shape, dtype=torch.int32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = out_h.numel() * out_h.element_size() + idx_h.numel() * idx_h.element_size()
    extra = []
    if res is not None:
        extra = [torch.empty(1, dtype=torch.int32).pin_memory()]
        d2h += 4
    n = max(1, min(args.steps, args.e2e_steps))

    def call():  # the calls a user makes for one step
        # inputs in and outputs out with one staging launch each (SM loads and
        # stores over the CPU-GPU link)
        pks.pks_stage_copy([(t[nm], host_in[nm]) for nm in names], s)
        pks.pks_decode_step(step.args, s)
        outs = [(out_h, step.out), (idx_h, step.topk_idx)]
        if res is not None:
            res.update(step.topk_idx, t["block_table"], wl.page_size, miss, n_miss, s)
            outs.append((extra[0], n_miss))
        pks.pks_stage_copy(outs, s)

    # captured once (copies from and to the pinned host buffers included),
    # replayed per step: one launch from the host instead of ten calls
    with torch.cuda.stream(s):
        call()
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    total = 0.0
    with torch.cuda.stream(s):
        for i in range(n + 3):
            flush()
            s.synchronize()
            t0 = time.perf_counter()
            g.replay()
            s.synchronize()
            if i >= 3:
                total += time.perf_counter() - t0
    return {"value": n / total, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n,
            "timing": "host wall clock per step: one CUDA-graph replay of the step's calls "
                      "(pks_stage_copy of the inputs from pinned memory, pks_decode_step, "
                      "pks_stage_copy of output and top-k to pinned memory) and a stream "
                      "synchronise"}


if __name__ == "__main__":
    main()
