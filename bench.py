#!/usr/bin/env python
"""Decode benchmark: sparse-MLP decode tokens/s on the Llama-2-7B ReLU shape
(32 layers, dense layer 0, d_model 4096, d_ff 11008, fp16, K_max 2048, 1024
centroids per projection at 10% density, persistence 0.83, gate|up union),
with per-kernel GB/s against the measured GB300 HBM and host-link peaks.

One step = one decoded token through the whole path: dense layer 0,
predictor, active sets + delta + slot assignment, host-link gather and
deinterleave-scatter of the incoming rows, 31 sparse FFNs.

  python bench.py [--gpus N --steps K --warmup W] [--impl cuda|reference]

Under torchrun each rank decodes its own independent sequence (replicas: the
path has no exchange step); value = tokens of all ranks / max rank time.
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

METRIC = "sparse-MLP decode tok/s + delta-scatter GB/s, % of GB300 HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}

# dram__bytes_read.sum + dram__bytes_write.sum per launch from one ncu capture
# (profiles/*.md), keyed by (kind, workload); valid only while the kernel's
# source file still has the recorded hash.
NCU_TRAFFIC = {
    ("gather", "llama2-7b-relu"): {"src": "np_scatter.cu", "src_hash": "92078b0e6f793061", "bytes_per_launch": 113408},
    ("ffn", "llama2-7b-relu"): {"src": "np_ffn.cu", "src_hash": "6f6a8b516ec3344b", "bytes_per_launch": 50404000},
    ("dense", "llama2-7b-relu"): {"src": "np_ffn.cu", "src_hash": "6f6a8b516ec3344b", "bytes_per_launch": 273740000},
    # one persistent launch over the 31 sparse layers, per layer
    ("ffn_chain", "llama2-7b-relu"): {"src": "np_ffn.cu", "src_hash": "6f6a8b516ec3344b",
                                      "bytes_per_launch": 50480000},
    # the per-token pipeline's persistent launch (layers 1..39), scaled from a
    # 12-layer capture by the sparse layers it covers
    ("token_pipeline", "llama2-13b-relu"): {"src": "np_ffn.cu", "src_hash": "6f6a8b516ec3344b",
                                           "bytes_per_launch": 3384000000},
    # mean of the two standalone sparse launches of the capture; dense layer 0
    ("ffn", "llama2-7b-batch8"): {"src": "np_mma.cu", "src_hash": "c5045b62f412d001", "bytes_per_launch": 84082560},
    ("dense", "llama2-7b-batch8"): {"src": "np_mma.cu", "src_hash": "c5045b62f412d001", "bytes_per_launch": 278717440},
}
SRC_DIR = os.path.join(ROOT, "sparse_activation_decode_gb300", "csrc")


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=256)
    p.add_argument("--warmup", type=int, default=128)
    p.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    p.add_argument("--config", default="llama2-7b-relu")
    p.add_argument("--persistence", type=float, default=None,
                   help="override the workload's token-to-token mask persistence (batched sweep)")
    p.add_argument("--h2d-mode", default="fused", choices=["staged", "fused"])
    p.add_argument("--slots", default=None, choices=["reuse", "compact"],
                   help="placement of resident rows (default: the workload's)")
    p.add_argument("--residency", default=None, choices=["slotmap", "window", "frequency"],
                   help="residency policy (default: the workload's)")
    p.add_argument("--lookahead", type=int, default=None,
                   help="per-layer predictor: predict layer l from the input of layer l - k")
    p.add_argument("--cpu-sample-tokens", type=int, default=16,
                   help="oracle tokens timed for cpu_baseline (after a cold-start token; capped at ~30 s)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--profile-case", action="store_true",
                   help="run the small capture case used for ncu (8-token workload of --config, 3 decode steps, "
                        "then standalone calls) and exit")
    p.add_argument("--layers", type=int, default=None,
                   help="with --profile-case: keep only this many layers (same shapes per layer)")
    return p.parse_args(argv)


def parse_args(argv):
    return parse(argv)


def replica_seed(seed: int, rank: int) -> int:
    """Each rank decodes its own independent sequence (its own inputs)."""
    return seed + 7919 * rank


def job_throughput(ms_local: float, steps: int, batch: int, world: int, device: str):
    """The timed region's length as the maximum over ranks (barrier, then an
    all-reduce MAX; one rank: its own) and the whole job's tokens per second:
    every rank decodes `steps` tokens of `batch` sequences."""
    import torch
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    return ms_max, world * steps * batch / (ms_max * 1e-3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def h2d_peak_gbs(torch):
    """Best contiguous pinned-host -> device copy bandwidth (GB/s)."""
    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(n, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(4):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        b.synchronize()
        best = max(best, n / (a.elapsed_time(b) * 1e-3) / 1e9)
    del src, dst
    return best


def file_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def kernel_table(prof, peaks, h2d_peak):
    """Per kind: launches, time, algorithmic GB/s and fraction of its peak."""
    out = {}
    for kind, d in prof.items():
        if d["launches"] == 0:
            continue
        ms = d["ms"]
        gbs = d["bytes"] / (ms * 1e-3) / 1e9 if ms > 0 and d["bytes"] > 0 else None
        # the set kernel moves ~100 KB per launch: latency-bound, no roofline
        bound = {"gather": "host_link", "set": "latency"}.get(kind, "hbm")
        peak = {"host_link": h2d_peak, "hbm": peaks["hbm_gbs"]}.get(bound)
        out[kind] = {"launches": d["launches"], "ms_total": round(ms, 4),
                     "us_per_launch": round(1e3 * ms / d["launches"], 3),
                     "bytes_per_launch": d["bytes"] // d["launches"] if d["bytes"] else 0,
                     "gbs": round(gbs, 1) if gbs else None, "bound": bound,
                     "frac": round(gbs / peak, 4) if gbs and peak else None}
    return out


def traffic_for(kind, workload):
    ent = NCU_TRAFFIC.get((kind, workload))
    if not ent or ent["src_hash"] != file_hash(os.path.join(SRC_DIR, ent["src"])):
        return None
    return ent["bytes_per_launch"]


def link_busy_ms(timeline):
    """Union of the gather launches' intervals (two gather streams overlap)."""
    iv = sorted((a, b) for k, a, b in timeline if k == "gather")
    busy, cs, ce = 0.0, None, None
    for a, b in iv:
        if cs is None or a > ce:
            if cs is not None:
                busy += ce - cs
            cs, ce = a, b
        else:
            ce = max(ce, b)
    if cs is not None:
        busy += ce - cs
    return busy


COMPUTE_KINDS = ("dense", "predictor", "set", "ffn", "finish")


def _union(iv):
    """Sorted disjoint union of intervals [(a, b)]."""
    out = []
    for a, b in sorted(iv):
        if out and a <= out[-1][1]:
            out[-1][1] = max(out[-1][1], b)
        else:
            out.append([a, b])
    return out


def _measure(iv):
    return sum(b - a for a, b in iv)


def _intersect(u, v):
    """Total length of the intersection of two disjoint unions."""
    i = j = 0
    tot = 0.0
    while i < len(u) and j < len(v):
        a, b = max(u[i][0], v[j][0]), min(u[i][1], v[j][1])
        if b > a:
            tot += b - a
        if u[i][1] < v[j][1]:
            i += 1
        else:
            j += 1
    return tot


def link_overlap(timeline):
    """Host-link time against compute time over a profiled run (ms, totals):
    busy = union of the gather launches; exposed = link busy while no
    compute kernel (dense, predictor, set, FFN, final add) runs; idle =
    compute running while the link is idle (the windows a per-token pipeline
    cannot fill with reads); span = first start to last end."""
    link = _union([(a, b) for k, a, b in timeline if k == "gather"])
    comp = _union([(a, b) for k, a, b in timeline if k in COMPUTE_KINDS])
    both = _intersect(link, comp)
    busy, cbusy = _measure(link), _measure(comp)
    span = (max(b for _, _, b in timeline) - min(a for _, a, _ in timeline)) if timeline else 0.0
    return {"busy": busy, "exposed": busy - both, "overlapped": both, "idle_while_compute": cbusy - both,
            "span": span}


def isolated_kernels(dec, torch, cfg, reps=5):
    """Standalone launches (no concurrent host-link traffic), events on the
    launching stream: sparse FFN over every sparse layer, dense layer 0, and
    the predictor, each with its algorithmic bytes."""
    h = torch.randn(cfg.batch * cfg.d_model, device="cuda")
    out = {}
    st = dec.main_stream
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    counts = dec.counts()
    rec = cfg.n_proj * cfg.d_model * cfg.elem_bytes

    def timed(fn, n):
        fn()
        torch.cuda.synchronize()
        ev0.record(st)
        for _ in range(n):
            fn()
        ev1.record(st)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / n

    layers = range(cfg.n_dense, cfg.n_layers)
    rows = sum(c[0] for c in counts) / max(len(counts), 1)
    # the sparse FFNs chained over all sparse layers on the resident rows
    # (np_ffn_layers: for batch 1 one persistent launch), per layer
    hc = h.clone()
    ms = timed(lambda: dec.ffn_layers(cfg.n_dense, cfg.n_sparse, hc), reps) / len(layers)
    out["ffn_chain"] = {"us_per_layer": round(1e3 * ms, 3), "bytes_per_layer": int(rows * rec),
                        "gbs": round(rows * rec / (ms * 1e-3) / 1e9, 1)}
    # one standalone launch per layer (np_sparse_mlp)
    ms = timed(lambda: [dec.sparse_mlp(l, h) for l in layers], reps) / len(layers)
    out["ffn"] = {"us_per_launch": round(1e3 * ms, 3), "bytes_per_launch": int(rows * rec),
                  "gbs": round(rows * rec / (ms * 1e-3) / 1e9, 1)}
    if cfg.n_dense > 0:
        ms = timed(lambda: dec.dense_mlp(0, h), reps)
        byt = 3 * cfg.d_ff * cfg.d_model * cfg.elem_bytes
        out["dense"] = {"us_per_launch": round(1e3 * ms, 3), "bytes_per_launch": byt,
                        "gbs": round(byt / (ms * 1e-3) / 1e9, 1)}
    ms = timed(lambda: dec.predict(h), reps)
    if cfg.pred_kind == "shared_argmax":  # W1, then every head's centroid rows
        byt = (cfg.pred_hidden * cfg.d_model + cfg.n_heads * cfg.n_centroids * cfg.pred_hidden) * cfg.elem_bytes
    else:  # one layer's W1, W2 and output bias
        byt = (cfg.pred_hidden * cfg.d_model + cfg.d_ff * cfg.pred_hidden + cfg.d_ff) * cfg.elem_bytes
    out["predictor"] = {"us_per_call": round(1e3 * ms, 3), "bytes_per_call": byt,
                        "gbs": round(byt / (ms * 1e-3) / 1e9, 1)}
    return out


def scatter_isolated(wl, torch, xs, decoder_for):
    """The deinterleave-scatter kernel of the staged host-link mode (staging
    -> projection buffers, device memory only), timed by the library's
    per-launch events with one layer per np_scatter call so that nothing runs
    beside it: a cold start (every layer's full set) and a steady-state token.
    Algorithmic bytes: 2 x records x record bytes (read staging, write the
    buffers).  Shared-predictor workloads only (the per-layer predictor has
    no all-layer delta)."""
    cfg = wl.cfg
    if cfg.pred_kind != "shared_argmax" or cfg.n_sparse == 0:
        return None
    dec = decoder_for(wl, h2d_mode="staged")
    rec = cfg.n_proj * cfg.d_model * cfg.elem_bytes
    out = {}

    def one(t, label):
        h = xs[t].reshape(-1).clone()
        y = dec.dense_mlp(0, h)
        ids = dec.predict(h + y)
        dec.delta(ids, -1)
        torch.cuda.synchronize()
        rows = sum(c[1] for c in dec.counts())
        dec.profile()
        dec.set_profiling(True, exact=True)
        for l in range(cfg.n_dense, cfg.n_layers):
            dec.scatter(l)
            torch.cuda.synchronize()
        p = dec.profile()["scatter"]
        dec.set_profiling(False)
        byt = 2 * rows * rec / max(p["launches"], 1)
        us = 1e3 * p["ms"] / max(p["launches"], 1)
        g = byt / (us * 1e-6) / 1e9
        out[label] = {"us_per_launch": round(us, 3), "bytes_per_launch": int(byt), "gbs": round(g, 1)}

    one(0, "full_set")
    for t in range(1, 8):
        dec.decode_token(xs[t].clone())
    one(8, "steady")
    dec.check_error()
    dec.close()
    return out


def profile_case(args):
    """Small capture case for ncu: 8-step workload of --config (optionally
    cut to --layers layers, host-link mode --h2d-mode), 3 decoded steps,
    then standalone calls of every kernel kind: two sparse FFNs, dense layer
    0, the chained sparse FFNs, predictor, delta, scatter."""
    import torch
    from sparse_activation_decode_gb300 import decoder_for
    from sparse_activation_decode_gb300.build import build
    from workloads import CONFIGS, make_workload
    build()
    cfg = CONFIGS[args.config].replace(n_warm=0, n_decode=8)
    if args.layers:
        cfg = cfg.replace(n_layers=args.layers)
    wl = make_workload(cfg, device="cuda")
    dec = decoder_for(wl, h2d_mode=args.h2d_mode)
    xs = wl.x.cuda()
    for t in range(3):
        dec.decode_token(xs[t].clone())
    torch.cuda.synchronize()
    h = xs[4].reshape(-1).clone()
    l1, l2 = (7, 8) if cfg.n_layers > 8 else (cfg.n_dense + 1, cfg.n_dense + 2)
    dec.sparse_mlp(l1, h)
    dec.sparse_mlp(l2, h)
    if cfg.n_dense > 0:
        dec.dense_mlp(0, h)
    dec.ffn_layers(cfg.n_dense, cfg.n_sparse, h.clone())  # chained sparse FFNs
    if cfg.pred_kind == "shared_argmax":
        ids = dec.predict(h)
        dec.delta(ids, -1)
        dec.scatter(-1)
    else:  # per-layer predictor: one layer's prediction, delta and reads
        fire = dec.predict(h, cfg.n_dense)
        dec.delta(fire, cfg.n_dense)
        dec.scatter(cfg.n_dense)
    torch.cuda.synchronize()
    dec.check_error()
    dec.close()
    print("profile case done")


def config_dict(cfg, args, world):
    """The workload the line is quoted on (shared by both arms)."""
    return {"workload": cfg.name, "layers": cfg.n_layers, "dense_prefix": cfg.n_dense,
            "d_model": cfg.d_model, "d_ff": cfg.d_ff, "k_max": cfg.k_max, "centroids": cfg.n_centroids,
            "combine": cfg.combine, "persistence": cfg.persistence, "batch": cfg.batch,
            "density": cfg.density, "warm_fill_tokens": cfg.n_warm,
            "ffn": "tcgen05 tensor cores" if cfg.batch > 1 else "CUDA cores",
            "h2d_mode": args.h2d_mode, "slots": cfg.slots, "residency": cfg.residency,
            "lookahead": cfg.lookahead, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (per-token weights ~2 GB > 129 MB)"}


def workload_config(args):
    """CONFIGS[--config] with the command line's overrides."""
    from workloads import CONFIGS
    base = CONFIGS[args.config]
    if args.persistence is not None:
        base = base.replace(persistence=args.persistence)
    if args.slots is not None:
        base = base.replace(slots=args.slots)
    if args.residency is not None:
        base = base.replace(residency=args.residency)
    if args.lookahead is not None:
        base = base.replace(lookahead=args.lookahead)
    return base


def run_cuda(args):
    import torch
    import torch.distributed as dist
    from sparse_activation_decode_gb300 import decoder_for
    from sparse_activation_decode_gb300.build import build
    from workloads import CONFIGS, make_workload

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0:
        build()
    if world > 1:
        dist.barrier()
    build()
    peaks = load_peaks()
    W, K = args.warmup, args.steps
    base = workload_config(args)
    # token positions: the workload's prompt warm fill, W warm-up steps, K
    # timed steps, then the profiled, statistics and end-to-end passes, each
    # continuing the sequence
    n_fill = base.n_warm
    KP, NST = min(K, 64), 16
    span = (base.batch - 1) * base.phase_step + 24
    T = min(n_fill + W + 2 * K + KP + NST, base.n_centroids - span if base.n_centroids else 10 ** 9)
    cfg = base.replace(n_warm=0, n_decode=T, seed=replica_seed(base.seed, rank))
    B = cfg.batch
    t0 = time.time()
    # the host weight store in page-locked memory from the start
    store = torch.empty((cfg.n_sparse, cfg.d_ff, cfg.n_proj, cfg.d_model), dtype=cfg.torch_dtype, pin_memory=True)
    wl = make_workload(cfg, device="cuda", store_out=store)
    gen_s = time.time() - t0
    dec = decoder_for(wl, h2d_mode=args.h2d_mode)
    xs = wl.x.to("cuda")                                  # [T][B][D], resident before timing

    def tok(i):
        return xs[i % T].clone()

    h2d_peak = h2d_peak_gbs(torch) if rank == 0 else None
    # the prompt warm fill (the cold start is its first token), then warm-up
    pos = 0
    for i in range(n_fill + W):
        dec.decode_token(tok(pos))
        pos += 1
    torch.cuda.synchronize()
    hs = [tok(pos + k) for k in range(K)]
    pos += K
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    main = dec.main_stream
    n0 = dec.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(main)
        for k in range(K):
            dec.decode_token(hs[k])
        ev1.record(main)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    launches = dec.launch_count() - n0
    # the host link is shared with other tenants of the machine: measure it
    # again right after the timed region
    h2d_after = h2d_peak_gbs(torch) if rank == 0 else None
    ms_max, value = job_throughput(ms, K, B, world, "cuda")

    # end to end through host buffers (pinned), copies inside the timed
    # region: the K tokens right after the timed ones, before the profiled
    # passes, so that both figures come from the same stretch of the decode
    e2e = None
    if not args.no_e2e:
        D, B = cfg.d_model, cfg.batch
        hin = torch.stack([xs[(pos + k) % T] for k in range(K)]).cpu().pin_memory()
        pos += K
        hout = torch.empty_like(hin).pin_memory()
        hdev = torch.empty((B, D), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        ev0.record(main)
        for k in range(K):
            hdev.copy_(hin[k], non_blocking=True)
            dec.decode_token(hdev)
            hout[k].copy_(hdev, non_blocking=True)
        ev1.record(main)
        torch.cuda.synchronize()
        ms_e = ev0.elapsed_time(ev1)
        e2e = {"value": round(world * K * B / (ms_e * 1e-3), 2), "unit": "tok/s",
               "h2d_bytes_per_step": B * D * 4, "d2h_bytes_per_step": B * D * 4}

    # live per-kernel durations (events on each kernel's own stream); few
    # enough tokens that the library keeps every launch in its timeline
    dec.profile()
    dec.set_profiling(True)
    hs2 = [tok(pos + k) for k in range(KP)]
    pos += KP
    for k in range(KP):
        dec.decode_token(hs2[k])
    timeline = dec.timeline()
    counts = dec.counts()
    union_density = float(sum(c[0] for c in counts)) / (len(counts) * cfg.d_ff) if counts else None
    prof = dec.profile()
    dec.set_profiling(False)
    table = kernel_table(prof, peaks, h2d_peak or 0.0)
    link_ms = link_busy_ms(timeline)
    iso = isolated_kernels(dec, torch, cfg)
    # rows read over the host link and rows moved inside HBM per token
    # (synchronising stats calls, after every timed region of the decode)
    n_st, din_rows, moved_rows, act_rows = NST, 0, 0, 0
    for k in range(n_st):
        st = dec.decode_token(tok(pos), stats=True)
        pos += 1
        din_rows += st["din_rows"]
        moved_rows += st["moved_rows"]
        act_rows += st["active_rows"]
    rec_b = cfg.n_proj * cfg.d_model * cfg.elem_bytes
    movement = {"tokens": n_st, "h2d_records_per_token": round(din_rows / n_st, 1),
                "h2d_bytes_per_token": int(din_rows * rec_b / n_st),
                "hbm_moved_records_per_token": round(moved_rows / n_st, 1),
                "hbm_move_bytes_per_token": int(2 * moved_rows * rec_b / n_st),
                # rows reused from the previous token: 1 - |D_in| / |A| (the pages' persistence)
                "measured_persistence": round(1.0 - din_rows / act_rows, 4) if act_rows else None}

    dec.close()
    scat = scatter_isolated(wl, torch, xs, decoder_for) if rank == 0 else None

    if rank != 0:
        return None
    # the per-token pipeline reads the records inside its persistent FFN
    # launch (one per token): that launch is the host-link-bound kernel
    token_pipeline = "gather" not in table and "ffn" in table and movement["h2d_bytes_per_token"] > 0
    if token_pipeline:
        table["ffn"]["bound"] = "host_link"
        table["ffn"]["bytes_per_launch"] = movement["h2d_bytes_per_token"]
        g = movement["h2d_bytes_per_token"] / (table["ffn"]["us_per_launch"] * 1e-6) / 1e9
        table["ffn"]["gbs"] = round(g, 1)
        table["ffn"]["frac"] = round(g / h2d_peak, 4) if h2d_peak else None
    dom = max(((k, v) for k, v in table.items() if k != "finish"), key=lambda kv: kv[1]["ms_total"])
    dk, dv = dom
    ov = link_overlap(timeline)
    if token_pipeline and dk == "ffn":
        achieved, peak = table["ffn"]["gbs"], h2d_peak
        peak_src = "measured live in this run: contiguous pinned host->device copy"
        dk = "token_pipeline"
    elif dv["bound"] == "host_link":
        # concurrent gather launches share the link: rate over the union of
        # their intervals, per launch = bytes per launch / (busy / launches)
        gather_bytes = prof["gather"]["bytes"]
        n_tl = sum(1 for k, _, _ in timeline if k == "gather")
        ok = link_ms > 0 and n_tl == prof["gather"]["launches"]
        achieved = gather_bytes / (link_ms * 1e-3) / 1e9 if ok else None
        peak = h2d_peak
        peak_src = "measured live in this run: contiguous pinned host->device copy"
    else:
        achieved, peak = dv["gbs"], peaks["hbm_gbs"]
        peak_src = f"MEASURED_PEAKS.json hbm_gbs ({peaks['source']})"
    roofline = {"kernel": dk, "bound": dv["bound"], "achieved": round(achieved, 1) if achieved else None,
                "peak": round(peak, 1), "unit": "GB/s", "frac": round(achieved / peak, 4) if achieved else None,
                "traffic": traffic_for(dk, cfg.name), "peak_source": peak_src,
                "note": ("per-token pipeline: one persistent launch per token reads the incoming records over the "
                         "host link and runs layers 1..L-1; achieved = incoming record bytes per token / that "
                         "launch's duration" if dk == "token_pipeline" else
                         "host-link bound: records come from page-locked host memory; achieved = gathered bytes "
                         "/ union of the gather launches' event intervals over the profiled region; traffic "
                         "counts HBM bytes only (the link's bytes are not DRAM traffic and the written rows "
                         "are still in L2 when the launch ends)")
                        if dv["bound"] == "host_link" else None}
    hbm_kernels = {}
    for k in ("ffn", "dense"):
        if k in iso:
            g = iso[k]["gbs"]
            hbm_kernels[k] = {"isolated_gbs": g, "isolated_us_per_launch": iso[k]["us_per_launch"],
                              "frac_of_measured_hbm": round(g / peaks["hbm_gbs"], 4),
                              "frac_of_nominal_8tbs": round(g / 8000.0, 4),
                              "in_pipeline_gbs": None if token_pipeline and k == "ffn" else table.get(k, {}).get("gbs"),
                              "traffic": traffic_for(k, cfg.name)}
    if "ffn_chain" in iso:
        g = iso["ffn_chain"]["gbs"]
        hbm_kernels["ffn_chain"] = {"gbs": g, "us_per_layer": iso["ffn_chain"]["us_per_layer"],
                                    "frac_of_measured_hbm": round(g / peaks["hbm_gbs"], 4),
                                    "frac_of_nominal_8tbs": round(g / 8000.0, 4),
                                    "traffic_per_layer": traffic_for("ffn_chain", cfg.name)}
    if scat:
        for lab, v in scat.items():
            hbm_kernels["scatter_" + lab] = {"isolated_gbs": v["gbs"], "isolated_us_per_launch": v["us_per_launch"],
                                             "bytes_per_launch": v["bytes_per_launch"],
                                             "frac_of_measured_hbm": round(v["gbs"] / peaks["hbm_gbs"], 4),
                                             "note": "staged host-link mode (not the default fused path)"}
    if "predictor" in iso:
        g = iso["predictor"]["gbs"]
        hbm_kernels["predictor"] = {"isolated_gbs": g, "frac_of_measured_hbm": round(g / peaks["hbm_gbs"], 4),
                                    "isolated_us_per_call": iso["predictor"]["us_per_call"]}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms_max / K, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": f"{cfg.dtype} weights, f32 accumulate", "data": "synthetic (seeded; shapes of the pages' workloads)",
        "config": config_dict(base, args, world),
        "pipeline": "per-token persistent launch" if token_pipeline else "streams, graph replay",
        "roofline": roofline, "hbm_kernels": hbm_kernels, "kernels": table,
        "h2d_peak_gbs": round(h2d_peak, 1), "h2d_peak_after_gbs": round(h2d_after, 1),
        "host_link_busy_ms_per_token": round(link_ms / KP, 4),
        # Budgeting Bytes' exposed-I/O view of the profiled tokens: link time
        # no compute kernel overlaps, and compute time with the link idle
        "host_link_per_token_ms": {"busy": round(ov["busy"] / KP, 4), "exposed": round(ov["exposed"] / KP, 4),
                                   "overlapped_by_compute": round(ov["overlapped"] / KP, 4),
                                   "idle_while_compute": round(ov["idle_while_compute"] / KP, 4),
                                   "profiled_span": round(ov["span"] / KP, 4),
                                   "note": "profiled pass (events per launch on its stream; upper bounds for "
                                           "launches that wait on another stream)"},
        "profiled_tokens": KP, "movement": movement,
        "gpu_launches": launches, "active_density_last_step": round(union_density, 4) if union_density else None,
        "clocks": clk.summary(), "e2e": e2e, "workload_gen_s": round(gen_s, 1),
    }
    return line, wl


def run_oracle_tokens(wl, n_tokens, budget_s=None):
    """Decode tokens with the fp64 oracle from a cold start; returns
    (tokens timed, seconds) excluding the first (cold-start) token."""
    import numpy as np
    from oracle import OracleDecoder
    orc = OracleDecoder(wl, materialize_buffers=False)
    orc.step(wl.x[0].cpu().numpy())
    t0 = time.time()
    n = 0
    for t in range(1, 1 + n_tokens):
        orc.step(wl.x[t % wl.x.shape[0]].cpu().numpy())
        n += 1
        if budget_s and time.time() - t0 > budget_s:
            break
    return n, time.time() - t0


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def main():
    args = parse()
    if args.profile_case:
        return profile_case(args)
    if args.impl == "reference":
        return run_reference(args)
    res = run_cuda(args)
    if res is None:
        return
    line, wl = res
    if not args.no_cpu_baseline and args.gpus == 1 and int(os.environ.get("WORLD_SIZE", "1")) == 1:
        n, sec = run_oracle_tokens(wl, args.cpu_sample_tokens, budget_s=30)
        nb = wl.cfg.batch
        line["cpu_baseline"] = {"value": round(n * nb / sec, 4), "unit": "tok/s", "cores": cores_used(),
                                "kind": "oracle",
                                "sample": f"{n} steps x {nb} sequences of {wl.cfg.name} after a cold-start step, "
                                          "fp64 numpy"}
    print(json.dumps(line), flush=True)


def run_reference(args):
    """The reference arm is the fp64 oracle on the host cores, on the same
    workload, metric and config as the CUDA arm: W untimed warm-up tokens
    (the first is the cold start), then K timed tokens.  The oracle's work
    per token does not depend on the warm fill, which it skips."""
    import torch  # noqa: F401
    from workloads import make_workload
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    base = workload_config(args)
    W, K = max(args.warmup, 0), max(args.steps, 1)
    cfg = base.replace(n_warm=0, n_decode=W + K)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = make_workload(cfg, device=dev)
    wl.dense_w = wl.dense_w.cpu() if wl.dense_w is not None else None
    wl.pred_w1, wl.pred_w2 = wl.pred_w1.cpu(), wl.pred_w2.cpu()
    wl.pred_b2 = wl.pred_b2.cpu() if wl.pred_b2 is not None else None
    wl.x = wl.x.cpu()
    from oracle import OracleDecoder
    orc = OracleDecoder(wl, materialize_buffers=False)
    for t in range(W):
        orc.step(wl.x[t].numpy())
    t0 = time.time()
    for t in range(W, W + K):
        orc.step(wl.x[t].numpy())
    sec = time.time() - t0
    v = K * cfg.batch / sec
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tok/s", "n_gpus": args.gpus,
            "steps": K, "warmup": W, "ms_per_step": round(1e3 * sec / K, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; shapes of the "
            "pages' workloads)", "config": config_dict(base, args, args.gpus),
            "cpu_baseline": {"value": round(v, 4), "unit": "tok/s", "cores": cores_used(), "kind": "oracle",
                             "sample": f"{K} steps x {cfg.batch} sequences of {cfg.name} after {W} warm-up "
                                       "steps (the first a cold start); fp64 numpy"},
            "e2e": {"value": round(v, 4), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
