"""W12 skinny-GEMM benchmark: weight-GB/s and fraction of the HBM roofline.

Workload (default): the M = 1 single-row decode projections of one dense layer
with hidden 5120 / intermediate 17408 / 8 KV heads of 128 -- q 5120x5120,
k 1024x5120, v 1024x5120, o 5120x5120, gate 17408x5120, up 17408x5120,
down 5120x17408 -- with W ~ N(0, 0.02^2) x per-row U(0.5, 2) and 1e-4
Student-t(2) x 0.5 outliers, x ~ N(0, 1).  One step = the 7 W12 GEMMs of one
layer, launched as a decode step would: q/k/v read one activation vector and
gate/up another, so k, v and up are launched input-ready (they may overlap the
tail of the GEMM before them); q, o, gate and down wait for the kernel before
them.  Steps rotate over several independently drawn layers, each ~0.5 GB of
W12 data, so every step streams its weights from HBM (inputs > L2).

Prints one JSON line (rank 0).  `--impl reference` times the scalar CPU oracle
on a bounded sample of the same workload instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as WL  # noqa: E402

METRIC = "W12 GEMM weight-GB/s and % of GB300 HBM roofline at M=1/32/64; µs per layer"
WORKLOAD = ("single-row decode projections, M=1: q/o 5120x5120, k/v 1024x5120, gate/up "
            "17408x5120, down 5120x17408 (one dense layer; N(0,0.02^2) x U(0.5,2) rows, "
            "1e-4 Student-t(2)x0.5 outliers)")
FALLBACK_HBM_GBS = 6800.0

# Activations of one dense layer's projections: q, k and v read one vector,
# gate and up another; o and down read the outputs of attention and of the MLP
# activation.  In a decode step, the launches of k, v and up therefore find
# their input complete before the preceding GEMM starts (input-ready launch);
# q, o, gate and down wait for the kernel before them.
ACT_GROUPS = {"qkv": 5120, "o": 5120, "gate_up": 5120, "down": 17408}
PROJ_GROUP = {"q": "qkv", "k": "qkv", "v": "qkv", "o": "o", "gate": "gate_up", "up": "gate_up", "down": "down"}
READY_IN_LAYER = {"k", "v", "up"}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _kernel_hash():
    h = hashlib.sha256()
    for f in ("gemm_fma.cu", "kernels.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "lossless_bit_weight_skinny_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(name, alg_bytes_per_launch):
    """DRAM bytes per launch, from a committed ncu capture of one large launch
    of the same kernel: its DRAM/algorithmic byte ratio times this run's
    algorithmic bytes per launch (traffic grows in proportion to the weights
    streamed).  None if the kernel source changed since the capture."""
    p = os.path.join(ROOT, "profiles", f"{name}.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_sha") != _kernel_hash():
        return None
    return int(d["traffic_over_algorithmic"] * alg_bytes_per_launch)


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        pass

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:7], float(parts[7])))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[3] > 0] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(loaded), "reasons": reasons}


# ---------------------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------------------

def _make_layers(w12, torch, n_layers, seed0=1000):
    """Draw, encode and upload `n_layers` layers; returns [[(name, Dev, stats)]]."""
    layers = []
    for li in range(n_layers):
        projs = []
        for pi, (name, N, K) in enumerate(WL.LAYER_PROJECTIONS):
            wb = WL.projection_weights_torch(N, K, seed=seed0 + 16 * li + pi)
            host = wb.cpu().numpy().view(np.uint16)
            del wb
            h = w12.w12_encode(host)
            st = h.stats()
            d = w12.w12_upload(h)
            torch.cuda.synchronize()
            projs.append((name, d, st))
        layers.append(projs)
    return layers


def _step_bytes(layer, M):
    """Algorithmic bytes of one step: W12 arrays (incl. metadata) + x + y."""
    tot = 0
    for name, d, st in layer:
        tot += st["bytes_total"] - 40 + 2 * M * d.K + 4 * M * d.N
    return tot


def replica_aggregate(ms, rank_bytes, dist=None, device="cpu"):
    """Whole-job throughput of independent replicas: every rank streamed
    `rank_bytes` in its own `ms` of timed region; the job's time is the slowest
    rank's (max over ranks), its bytes the sum over ranks.  Returns
    (max ms, GB/s of the whole job)."""
    import torch

    world = 1
    if dist is not None:
        world = dist.get_world_size()
        t = torch.tensor([float(ms), float(rank_bytes)], dtype=torch.float64, device=device)
        tm = t[:1].clone()
        dist.all_reduce(tm, op=dist.ReduceOp.MAX)
        tb = t[1:].clone()
        dist.all_reduce(tb, op=dist.ReduceOp.SUM)
        ms, total = float(tm.item()), float(tb.item())
    else:
        total = float(rank_bytes)
    return ms, total / (ms * 1e-3) / 1e9


def run_w12(args):
    import torch

    import __graft_entry__

    __graft_entry__._load_builder().build()
    import lossless_bit_weight_skinny_gb300 as w12

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")

    layers = _make_layers(w12, torch, args.layers)
    M = 1

    def acts(Mx, seed):
        """One activation vector per group (q/k/v share one, gate/up another)."""
        return {g: torch.from_numpy(WL.activations(Mx, K, seed=seed + gi).view(np.int16)).cuda()
                .view(torch.bfloat16) for gi, (g, K) in enumerate(ACT_GROUPS.items())}

    xs = acts(M, 7)
    ys = {name: torch.empty((M, N), dtype=torch.float32, device="cuda") for name, N, K in WL.LAYER_PROJECTIONS}
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    n_proj = len(WL.LAYER_PROJECTIONS)

    def launch(mode, name, d, x, y):
        ready = mode == "independent" or (mode == "layer" and name in READY_IN_LAYER)
        w12.w12_gemm_ex(x, d, y, stream, input_ready=ready)

    def step(i, ev=None, mode="layer"):
        layer = layers[i % len(layers)]
        for j, (name, d, st) in enumerate(layer):
            if ev is not None:
                ev[j][0].record(stream)
            launch(mode, name, d, xs[PROJ_GROUP[name]], ys[name])
            if ev is not None:
                ev[j][1].record(stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    for layer in layers:
        for _, d, _ in layer:
            assert w12.w12_dev_status(d) == 0

    # The timed region replays one CUDA graph of G steps (rotating over the
    # layers), with nothing between the GEMM launches so that each may overlap
    # the previous one's tail (programmatic dependent launch).  Right after it,
    # still on the same warm state, a second graph with an event pair around
    # every launch gives each kernel's own duration (without that overlap).
    G = args.graph_steps
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(G):
            step(i)
    graph.replay()
    torch.cuda.synchronize()
    try:
        evs = [[[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
                for _ in range(n_proj)] for _ in range(G)]
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev, stream=stream):
            for i in range(G):
                step(i, evs[i], mode="none")
        graph_ev.replay()
        torch.cuda.synchronize()
    except TypeError:
        evs, graph_ev = None, None
    reps = max(1, args.steps // G)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    with sampler:
        time.sleep(0.25)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0.record(stream)
        for _ in range(reps):
            graph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        if graph_ev is not None:
            graph_ev.replay()
            torch.cuda.synchronize()
    clocks = sampler.stop()
    # per-replay spread of the same graph (after the timed region): each
    # replay between its own event pair, so median and minimum per step
    n_rep = min(reps, 50)
    rev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_rep)]
    for e0, e1 in rev:
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    per_step = sorted(1e3 * e0.elapsed_time(e1) / G for e0, e1 in rev)
    step_stats = {"median_us": round(per_step[len(per_step) // 2], 2), "min_us": round(per_step[0], 2),
                  "max_us": round(per_step[-1], 2), "replays": n_rep, "steps_per_replay": G}
    args.steps = reps * G
    step_bytes = _step_bytes(layers[0], M)
    ms, value = replica_aggregate(t0.elapsed_time(t1), step_bytes * args.steps, dist, "cuda")
    for layer in layers:
        for _, d, _ in layer:
            assert w12.w12_dev_status(d) == 0, "device status after timing"

    # per-launch durations of the dominant kernel (the M = 1 CUDA-core GEMM),
    # from the event pairs of the measurement replay
    kern_ms = 0.0
    kern_bytes = 0
    per_proj = {}
    for i in range(G):
        layer = layers[i % len(layers)]
        for j, (name, d, st) in enumerate(layer):
            bts = st["bytes_total"] - 40 + 2 * M * d.K + 4 * M * d.N
            dt = evs[i][j][0].elapsed_time(evs[i][j][1]) if evs else None
            if dt is None:
                continue
            kern_ms += dt
            kern_bytes += bts
            p = per_proj.setdefault(name, [0.0, 0, bts])
            p[0] += dt
            p[1] += 1
    if not evs:  # no timing events in graphs: bound the kernel time by the step time
        kern_ms, kern_bytes = ms, step_bytes * args.steps
    peak, peak_kind = _peaks()
    # The timed region launches nothing but the dominant kernel, back to back:
    # its average launch duration is the timed region over the launch count.
    n_launch = args.steps * n_proj
    achieved = step_bytes * args.steps / (ms * 1e-3) / 1e9
    achieved_isolated = kern_bytes / (kern_ms * 1e-3) / 1e9 if kern_ms else None
    traffic = _traffic("gemm_fma_m1", step_bytes / n_proj)

    def time_graph(Mx, xs_, ys_, mode, greps):
        """Replay a G-step graph of the layer at Mx rows in launch mode `mode`;
        returns ms per step."""
        def stepm(i):
            for name, d, st in layers[i % len(layers)]:
                launch(mode, name, d, xs_[PROJ_GROUP[name]], ys_[name])

        for i in range(max(3, args.warmup // 4)):
            stepm(i)
        torch.cuda.synchronize()
        gm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gm, stream=stream):
            for i in range(G):
                stepm(i)
        gm.replay()
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(greps):
            gm.replay()
        s1.record(stream)
        torch.cuda.synchronize()
        for layer in layers:
            for _, d, _ in layer:
                assert w12.w12_dev_status(d) == 0
        return s0.elapsed_time(s1) / (greps * G)

    # the same step with every launch waiting for the previous kernel, and with
    # every launch input-ready (the synthetic activations are all independent)
    short = max(2, args.steps // (4 * G))
    modes_us = {"layer": round(1e3 * ms / args.steps, 2),
                "no_overlap": round(1e3 * time_graph(M, xs, ys, "none", short), 2),
                "independent_inputs": round(1e3 * time_graph(M, xs, ys, "independent", short), 2)}

    # the same layer at M = 32, 64, 128 (tensor-core path, one launch per
    # projection) and 256 (two launches of 128 rows), shorter runs; GB/s counts
    # the W12 bytes once
    by_m = {"1": {"weight_GBps": round(value / world, 1), "us_per_layer": round(1e3 * ms / args.steps, 2)}}
    for Mx in (32, 64, 128, 256):
        xm = acts(Mx, 9)
        ym = {n: torch.empty((Mx, N), dtype=torch.float32, device="cuda") for n, N, K in WL.LAYER_PROJECTIONS}
        msm = time_graph(Mx, xm, ym, "layer", short)
        bm = _step_bytes(layers[0], Mx)
        by_m[str(Mx)] = {"weight_GBps": round(bm / (msm * 1e-3) / 1e9, 1), "us_per_layer": round(1e3 * msm, 2)}

    # Two-level-verification pair on a 17408x5120 matrix: the Q pass over the
    # 8-bit view at M = 64 (draft-tree nodes), then the exact pass at M = 16, for
    # the projection draw (the gate projection of the first layer) and for a
    # heavy-tailed draw (Student-t 1.5, ~1e-2 escapes), the latter also with
    # count-maximising windows (~2e-3 escapes; the top outliers escape instead).
    tlv = {}
    heavy_w = WL.heavy_weights(17408, 5120, seed=31)
    hheavy = w12.w12_encode(heavy_w)
    wheavy = w12.w12_upload(hheavy)
    hheavy_cm = w12.w12_encode(heavy_w, count_max=True)
    wheavy_cm = w12.w12_upload(hheavy_cm)
    del heavy_w
    x64 = torch.from_numpy(WL.activations(64, 5120, seed=41).view(np.int16)).cuda().view(torch.bfloat16)
    x16 = torch.from_numpy(WL.activations(16, 5120, seed=42).view(np.int16)).cuda().view(torch.bfloat16)
    y64 = torch.empty((64, 17408), dtype=torch.float32, device="cuda")
    y16 = torch.empty((16, 17408), dtype=torch.float32, device="cuda")
    for dist_name, dm in (("projection", layers[0][4][1]), ("heavy_tail", wheavy),
                          ("heavy_tail_count_max_windows", wheavy_cm)):
        def run(kind, dm=dm):
            if kind in ("q8", "pair"):
                w12.w12_gemm_ex(x64, dm, y64, stream, q8view=True)
            if kind in ("exact", "pair"):
                w12.w12_gemm_ex(x16, dm, y16, stream)

        res = {}
        for kind in ("q8", "exact", "pair"):
            for _ in range(3):
                run(kind)
            torch.cuda.synchronize()
            gt = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gt, stream=stream):
                for _ in range(G):
                    run(kind)
            gt.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(short):
                gt.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            res[kind + "_us"] = round(1e3 * e0.elapsed_time(e1) / (short * G), 2)
        assert w12.w12_dev_status(dm) == 0
        res["q8_view_GBps"] = round((17408 * 5120 + 2 * 64 * 5120 + 4 * 64 * 17408) / (res["q8_us"] * 1e3), 1)
        tlv[dist_name] = res
    # the Q pass over a separate INT8 copy of the projection draw, at M = 64
    q8c = w12.w12_i8_from_dev(layers[0][4][1], stream)
    for _ in range(3):
        w12.w12_gemm_i8(x64, q8c, y64, stream)
    torch.cuda.synchronize()
    gq = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gq, stream=stream):
        for _ in range(G):
            w12.w12_gemm_i8(x64, q8c, y64, stream)
    gq.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(short):
        gq.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    assert w12.w12_i8_status(q8c) == 0
    q_us = 1e3 * e0.elapsed_time(e1) / (short * G)
    tlv["projection"]["q_int8_copy_us"] = round(q_us, 2)
    tlv["projection"]["q_int8_copy_GBps"] = round((17408 * 5120 + 4 * 17408 + 2 * 64 * 5120 + 4 * 64 * 17408)
                                                  / (q_us * 1e3), 1)
    q8c.free()
    tlv["escape_fraction_heavy_tail"] = round(hheavy.stats()["escape_fraction"], 5)
    tlv["escape_fraction_heavy_tail_count_max_windows"] = round(hheavy_cm.stats()["escape_fraction"], 5)
    del hheavy, hheavy_cm
    wheavy.free()
    wheavy_cm.free()

    # Fused projections (the same bytes, merged at encode time): q/k/v stacked
    # into one 7168x5120 matrix and gate/up interleaved by rows into one
    # 34816x5120 matrix (every W12 row carries its own window, and the escape
    # tiles are 128 rows high, so merging rows is just a bigger matrix).  One
    # step = qkv (BF16 out), o (BF16 out), gate_up with the SiLU*mul epilogue
    # writing BF16 h[M][17408], and down reading h: each launch waits for the
    # kernel before it, and down consumes gate_up's output, as in a decode step.
    def fused_layer(li):
        out = []
        for gname, parts in (("qkv", ("q", "k", "v")), ("o", ("o",)), ("gate_up", ("gate", "up")), ("down", ("down",))):
            ws = [WL.projection_weights_torch(N, K, seed=1000 + 16 * li + pi)
                  for pi, (name, N, K) in enumerate(WL.LAYER_PROJECTIONS) if name in parts]
            if gname == "gate_up":  # row 2i = gate row i, row 2i+1 = up row i
                wcat = torch.stack(ws, 1).reshape(-1, ws[0].shape[1])
            else:
                wcat = torch.cat(ws, 0) if len(ws) > 1 else ws[0]
            out.append((gname, w12.w12_encode_device(wcat, stream)))
            del ws, wcat
        return out

    flayers = [fused_layer(li) for li in range(len(layers))]
    f_out = {"qkv": (7168, torch.bfloat16), "o": (5120, torch.bfloat16), "gate_up": (17408, torch.bfloat16),
             "down": (5120, torch.float32)}
    fy = {g: torch.empty((M, n), dtype=dt, device="cuda") for g, (n, dt) in f_out.items()}
    fx = {"qkv": xs["qkv"], "o": xs["o"], "gate_up": xs["gate_up"], "down": fy["gate_up"]}

    def stepf(i):
        for g, d in flayers[i % len(flayers)]:
            w12.w12_gemm_ex(fx[g], d, fy[g], stream, out_bf16=(g != "down"), silu_mul=(g == "gate_up"))

    for i in range(3):
        stepf(i)
    torch.cuda.synchronize()
    gf = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gf, stream=stream):
        for i in range(G):
            stepf(i)
    gf.replay()
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(short):
        gf.replay()
    f1.record(stream)
    torch.cuda.synchronize()
    f_us = 1e3 * f0.elapsed_time(f1) / (short * G)
    fused = {"us_per_layer": round(f_us, 2), "weight_GBps": round(step_bytes / (f_us * 1e3), 1),
             "step": "4 GEMMs: qkv 7168x5120 (BF16 out), o 5120x5120 (BF16 out), gate_up 34816x5120 "
                     "(gate/up rows interleaved; SiLU*mul epilogue, BF16 h[1][17408] out), down "
                     "5120x17408 reading h (FP32 out); merged at encode time, encoded on the device; "
                     "GB/s counts the unfused layer's bytes"}
    for fl in flayers:
        for _, d in fl:
            assert w12.w12_dev_status(d) == 0
            d.free()
    del flayers

    # Context, not the target: the same layers as dense BF16 weights through
    # torch.matmul (cuBLAS), graph-timed the same way (the pages compare the
    # W12 GEMM with cuBLAS at 1 and 32 rows).
    dense = None
    if not args.no_dense:
        dlayers = [[(name, WL.projection_weights_torch(N, K, seed=1000 + 16 * li + pi).view(torch.bfloat16))
                    for pi, (name, N, K) in enumerate(WL.LAYER_PROJECTIONS)] for li in range(len(layers))]
        dense = {"us_per_layer": {}, "w12_speedup": {}}
        for Mx, w12_us in ((1, modes_us["layer"]), (32, by_m["32"]["us_per_layer"]),
                           (128, by_m["128"]["us_per_layer"])):
            xdn = {g: v for g, v in acts(Mx, 9 if Mx > 1 else 7).items()}

            def stepd(i):
                for name, Wd in dlayers[i % len(dlayers)]:
                    torch.matmul(xdn[PROJ_GROUP[name]], Wd.t())

            for i in range(3):
                stepd(i)
            torch.cuda.synchronize()
            gd = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gd, stream=stream):
                for i in range(G):
                    stepd(i)
            gd.replay()
            torch.cuda.synchronize()
            d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            d0.record(stream)
            for _ in range(short):
                gd.replay()
            d1.record(stream)
            torch.cuda.synchronize()
            us = 1e3 * d0.elapsed_time(d1) / (short * G)
            dense["us_per_layer"][str(Mx)] = round(us, 2)
            dense["w12_speedup"][str(Mx)] = round(us / w12_us, 3)
        dense["weight_bytes_per_layer"] = sum(2 * N * K for _, N, K in WL.LAYER_PROJECTIONS)
        dense["note"] = "torch.matmul(x, W.t()) with BF16 W of the same seeds, BF16 out, one CUDA graph of G steps"
        del dlayers
        torch.cuda.empty_cache()

    # Conversion speed: one 17408x5120 BF16 matrix (178 MB) to W12, on the
    # device (weights already there) and with the host encoder (all cores).
    wconv = WL.projection_weights_torch(17408, 5120, seed=77)
    t_dev = []
    for _ in range(3):
        torch.cuda.synchronize()
        tc0 = time.perf_counter()
        dconv = w12.w12_encode_device(wconv, stream)
        t_dev.append(time.perf_counter() - tc0)
        dconv.free()
    whost = wconv.cpu().numpy().view(np.uint16)
    tc0 = time.perf_counter()
    hconv = w12.w12_encode(whost)
    t_host = time.perf_counter() - tc0
    del hconv, whost, wconv
    convert = {"device_ms": round(1e3 * min(t_dev), 2), "host_ms": round(1e3 * t_host, 1),
               "device_GBps_bf16_in": round(2 * 17408 * 5120 / min(t_dev) / 1e9, 1),
               "host_cores": len(os.sched_getaffinity(0))}

    # End to end: every step copies its activations from pinned host memory
    # (one transfer: the four activation vectors of the layer, packed), runs
    # the seven GEMMs through the public entry point, and copies the seven
    # results back (one transfer), inside the timed loop.  The calls of G
    # steps are captured once in a CUDA graph, as a serving loop would issue
    # them, and replayed; wall-clock time on the host.
    groups = list(ACT_GROUPS.items())
    x_off, off = {}, 0
    for g, K in groups:
        x_off[g] = off
        off += M * K
    hx = torch.from_numpy(np.concatenate([WL.activations(M, K, seed=7 + gi).view(np.int16).ravel()
                                          for gi, (g, K) in enumerate(groups)])).pin_memory()
    dx = torch.empty(off, dtype=torch.int16, device="cuda")
    dxv = {g: dx[x_off[g]:x_off[g] + M * K].view(torch.bfloat16).view(M, K) for g, K in groups}
    y_off, off = {}, 0
    for name, N, K in WL.LAYER_PROJECTIONS:
        y_off[name] = off
        off += M * N
    hy = torch.empty(off, dtype=torch.float32).pin_memory()
    dy = torch.empty(off, dtype=torch.float32, device="cuda")
    dyv = {name: dy[y_off[name]:y_off[name] + M * N].view(M, N) for name, N, K in WL.LAYER_PROJECTIONS}

    def step_e2e(i):
        dx.copy_(hx, non_blocking=True)
        for name, d, st in layers[i % len(layers)]:
            launch("layer", name, d, dxv[PROJ_GROUP[name]], dyv[name])
        hy.copy_(dy, non_blocking=True)

    for i in range(args.warmup):
        step_e2e(i)
    torch.cuda.synchronize()
    graph_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_e2e, stream=stream):
        for i in range(G):
            step_e2e(i)
    graph_e2e.replay()
    torch.cuda.synchronize()
    e_reps = max(2, args.steps // (2 * G))
    e_steps = e_reps * G
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    tw = time.perf_counter()
    for _ in range(e_reps):
        graph_e2e.replay()
    torch.cuda.synchronize()
    e_s = time.perf_counter() - tw
    # the job's time is the slowest rank's, its bytes the sum over ranks
    e_ms, e_gbs = replica_aggregate(1e3 * e_s, step_bytes * e_steps, dist, "cuda")
    h2d = int(hx.numel() * 2)
    d2h = int(hy.numel() * 4)
    e2e = {"value": round(e_gbs, 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "us_per_layer": round(1e3 * e_ms / e_steps, 2),
           "method": "per step: one H2D copy of the layer's activations from pinned memory, the 7 "
                     "w12_gemm_ex calls, one D2H copy of the 7 results; the calls of "
                     f"{G} steps captured in a CUDA graph and replayed; host wall clock"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)

    if rank == 0:
        st_all = [st for _, _, st in layers[0]]
        line = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms / args.steps, 5),
            "us_per_layer": round(1e3 * ms / args.steps, 2),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16 weights (W12) x bf16 activations, fp32 accumulate",
            "data": "synthetic",
            "config": {
                "workload": WORKLOAD,
                "M": M,
                "layers_rotated": args.layers,
                "step": "7 GEMMs (q,k,v,o,gate,up,down) of one layer; q/k/v share one activation "
                        "vector and gate/up another; k, v and up launch input-ready (their input "
                        "exists before the preceding GEMM starts), the others wait for the kernel "
                        "before them",
                "bytes_per_step": step_bytes,
                "l2": "inputs larger than L2: each step streams ~0.5 GB of W12 weights",
                "escape_fraction": round(sum(s["n_escapes"] for s in st_all)
                                         / sum(s["N"] * s["K"] for s in st_all), 7),
                "bits_per_weight": round(8 * sum(s["bytes_total"] for s in st_all)
                                         / sum(s["N"] * s["K"] for s in st_all), 4),
                "parallelism": f"replicas x{world}",
            },
            "by_M": by_m,
            "us_per_layer_by_launch_mode": modes_us,
            "two_level_verification_17408x5120": tlv,
            "dense_bf16_cublas": dense,
            "encode_17408x5120": convert,
            "fused_projections_m1": fused,
            "per_projection_us_event_bracketed": {k: round(1e3 * v[0] / v[1], 2) for k, v in per_proj.items()},
            "roofline": {
                "bound": "hbm",
                "kernel": "gemm_fma_kernel<1,false> (M=1)",
                "achieved": round(achieved, 1),
                "peak": peak,
                "peak_kind": f"{peak_kind} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": traffic,
                "frac_of_8TBps": round(achieved / 8000.0, 4),
                "launch_us": round(1e3 * ms / n_launch, 3),
                "bytes_per_launch": step_bytes // n_proj,
                "achieved_event_bracketed": round(achieved_isolated, 1) if achieved_isolated else None,
            },
            "e2e": e2e,
            "gpu_launches": n_launch,
            "clocks": clocks,
            "us_per_layer_spread": step_stats,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------------------
# the scalar CPU oracle (reference arm and CPU baseline)
# ---------------------------------------------------------------------------------------

def _oracle_sample(rows_frac: int, seed0=1000):
    """Per projection: the first N/rows_frac rows, encoded by the oracle."""
    import oracle as O

    out = []
    for pi, (name, N, K) in enumerate(WL.LAYER_PROJECTIONS):
        R = max(1, N // rows_frac)
        W = WL.projection_weights(R, K, seed=seed0 + pi)
        blob = O.encode(W)
        x = WL.activations(1, K, seed=7)
        out.append((name, R, K, blob, x, len(blob) - 40 + 2 * K + 4 * R))
    return out


def _oracle_pass(sample, threads):
    """Decode + float64 GEMM of every sampled projection, rows split over threads."""
    import concurrent.futures as cf

    import oracle as O

    def job(item):
        name, R, K, blob, x, _ = item
        W = O.decode(blob)
        return O.gemm(x, W)

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(job, sample))


def _cpu_model() -> str:
    import platform

    info = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    info.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    if "model name" in info:
        return info["model name"]
    if "cpu part" in info:  # Arm: implementer and part number
        return f"{platform.machine()} (CPU implementer {info.get('cpu implementer', '?')}, part {info['cpu part']})"
    return f"{platform.machine()} {platform.processor()}".strip()


def cpu_baseline(seconds_budget: float):
    """The oracle as it stands, timed on this host's cores on a bounded sample."""
    import oracle as O

    O.build()
    cores = len(os.sched_getaffinity(0))
    threads = min(cores, len(WL.LAYER_PROJECTIONS))
    frac = 16
    sample = _oracle_sample(frac)
    t = time.perf_counter()
    _oracle_pass(sample, threads)
    dt = time.perf_counter() - t
    reps = max(1, int(seconds_budget / max(dt, 1e-3)))
    reps = min(reps, 20)
    t = time.perf_counter()
    for _ in range(reps):
        _oracle_pass(sample, threads)
    dt = (time.perf_counter() - t) / reps
    nbytes = sum(s[5] for s in sample)
    t = time.perf_counter()
    _oracle_pass(sample, 1)
    dt1 = time.perf_counter() - t
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "value_1_thread": round(nbytes / dt1 / 1e9, 4), "cpu_model": _cpu_model(),
            "kind": "oracle",
            "sample": f"first 1/{frac} of the rows of each of the 7 projections of one layer, "
                      f"M=1: oracle decode + float64 GEMM, projections in parallel threads, "
                      f"{reps} reps; host has {cores} cores"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle as O

    O.build()
    cores = len(os.sched_getaffinity(0))
    threads = min(cores, len(WL.LAYER_PROJECTIONS))
    # each step is a bounded sample (the first 1/frac of every projection's
    # rows), sized so that warm-up + steps take about 150 s in all
    frac = 64
    sample = _oracle_sample(frac)
    t = time.perf_counter()
    _oracle_pass(sample, threads)
    probe = time.perf_counter() - t
    per_step = min(0.25, 150.0 / max(1, args.steps + args.warmup))
    while frac < 8192 and probe * 64 / frac > per_step:
        frac *= 2
    if frac != 64:
        sample = _oracle_sample(frac)
    for _ in range(args.warmup):
        _oracle_pass(sample, threads)
    t = time.perf_counter()
    for _ in range(args.steps):
        _oracle_pass(sample, threads)
    dt = time.perf_counter() - t
    nbytes = sum(s[5] for s in sample) * args.steps
    value = nbytes / dt / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * dt / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 weights (W12) x bf16 activations, fp64 accumulate",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1,
                   "sample": f"first 1/{frac} of the rows of each projection per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"first 1/{frac} of the rows of each of the 7 projections, "
                                   "oracle decode + float64 GEMM per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_case(cases):
    """Small profiling cases: one 17408x5120 W12 matrix (134 MB, larger than
    L2) and three launches of each named case's kernel, in order (for ncu
    captures); `cases` is a comma-separated list."""
    import torch

    import __graft_entry__

    __graft_entry__._load_builder().build()
    import lossless_bit_weight_skinny_gb300 as w12

    N, K = 17408, 5120
    wb = WL.projection_weights_torch(N, K, seed=5)
    d = w12.w12_upload(w12.w12_encode(wb.cpu().numpy().view(np.uint16)))
    rows = {"fma": 1, "fma2": 2, "fma4": 4, "tc16": 16, "tc32": 32, "tc": 64, "tc128": 128, "q8": 64, "q8m1": 1}
    for case in cases.split(","):
        M = rows[case]
        x = torch.from_numpy(WL.activations(M, K, seed=1).view(np.int16)).cuda().view(torch.bfloat16)
        fn = w12.w12_gemm_q8view if case.startswith("q8") else w12.w12_gemm
        for _ in range(3):
            y = fn(x, d)
        torch.cuda.synchronize()
        assert w12.w12_dev_status(d) == 0
        print(case, "ok", float(y.abs().sum()))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="w12", choices=["w12", "reference"])
    ap.add_argument("--layers", type=int, default=3)
    ap.add_argument("--graph-steps", type=int, default=12)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dense", action="store_true", help="skip the dense BF16 (cuBLAS) comparison")
    ap.add_argument("--case", default=None,
                    help="profiling cases, comma-separated: fma, fma2, fma4, tc16, tc32, tc (M=64), tc128, q8, q8m1")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.case:
        run_case(args.case)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_w12(args)


if __name__ == "__main__":
    main()
