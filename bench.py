#!/usr/bin/env python
"""Benchmark of the activation-sparse MoE decode path on GB300.

Workload (one step): batch-1 decode through 23 distinct MoE layers (hidden
2688, 128 routed experts of 1856 neurons, top-6, a 3712-neuron shared expert,
4-bit affine group-64 weights, 16.8 GB of weights in total), routed live
fraction 0.1, shared live fraction U(0.05, 0.15) per layer.  One step is 23
calls of hs_moe_layer_decode, captured in one CUDA graph.  The weights are far
larger than L2, so no L2 flush is needed between steps.

Metric: MoE-layer decode time in microseconds per layer per token (lower is
better), with the achieved HBM bandwidth on the bytes the method must move.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl hs|reference]

--impl reference times the CPU fp64 oracle on the host cores on the same
workload (a bounded sample of layers per step).  Under torchrun each rank
runs an independent replica (the path has no cross-GPU exchange).
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
# fp32 FMA peak of the GPU: 152 SMs x 128 lanes x 2 flops per FMA x 2.07 GHz (maximum SM clock)
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
sys.path.insert(0, ROOT)

METRIC = "MoE-layer decode us/token (batch 1, per layer) and achieved HBM GB/s at live frac 0.1"
UNIT = "us/layer"
LAYERS = 23
WORKLOAD = "moe_decode_b1_23layers_p0.1"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["hs", "reference"], default="hs")
    ap.add_argument("--p", type=float, default=0.1)
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cpu-all-cores", action="store_true", help="skip the all-cores oracle timing")
    ap.add_argument("--batch-sizes", type=str, default="2,3,8,32,64",
                    help="batch decode leg (one MoE layer, 30%% dead neurons); empty to skip")
    ap.add_argument("--no-prefill", action="store_true", help="skip the 2048-token prefill leg")
    ap.add_argument("--no-sweep", action="store_true", help="skip the live-fraction sweep")
    ap.add_argument("--no-router", action="store_true", help="skip the router projection leg")
    ap.add_argument("--no-row-scales", action="store_true",
                    help="skip the leg with the down projections re-quantised with row scales")
    ap.add_argument("--no-expert-down", action="store_true",
                    help="skip the single-expert sparse down leg (512 distinct experts)")
    ap.add_argument("--profile", action="store_true",
                    help="minimal run for profilers: no clock soak, dense, end-to-end or CPU legs")
    return ap.parse_args()


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (all ranks call it; any backend whose
    tensors live on `device`)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _config(args, extra=None):
    c = {"workload": WORKLOAD if args.p == 0.1 and args.layers == LAYERS else
         f"moe_decode_b1_{args.layers}layers_p{args.p}",
         "layers": args.layers, "batch": 1, "hidden": 2688, "routed_experts": 128, "top_k": 6,
         "routed_neurons": 1856, "shared_neurons": 3712, "weights": "W4 affine group-64, fp16 scale+bias",
         "p_routed": args.p, "p_shared": "U(0.05,0.15) per layer",
         "l2": "weights 16.8 GB > L2, no flush", "parallelism": "replicas" if _dist()[0] > 1 else "single"}
    if extra:
        c.update(extra)
    return c


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------- ncu traffic
def _sources_sha256(srcs) -> str:
    """One hash over the kernel's source files (the .cu and the headers it includes)."""
    h = hashlib.sha256()
    for src in srcs:
        h.update(open(src, "rb").read())
    return h.hexdigest()


def _recorded_traffic(kernel: str, srcs):
    """DRAM bytes per launch recorded under profiles/ for `kernel`, if the
    recorded source hash still matches the kernel's sources (None otherwise:
    the counters describe an older kernel)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}.txt")
    if not os.path.exists(path):
        return None
    rec = {}
    for ln in open(path):
        if ":" in ln and not ln.startswith("#"):
            k, v = ln.split(":", 1)
            rec[k.strip()] = v.strip()
    if rec.get("source_sha256") != _sources_sha256(srcs):
        return None
    try:
        return float(rec["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------- workload
def build_layers(n_layers, p, device, down_row_scales=False):
    import synth
    from activation_sparse_moe_gb300.layer import DeviceLayer, from_synth_expert, from_synth_stack
    layers = []
    for l in range(n_layers):
        L = synth.layer_inputs(0, "decode-23layers", l, p=p, p_shared=synth.shared_live_fraction(0, l), device=device)
        dl = DeviceLayer(from_synth_stack(L.up, L.down, L.offsets, device, down_row_scales=down_row_scales),
                         from_synth_expert(L.shared, device, down_row_scales=down_row_scales), top_k=6)
        layers.append(dl)
        del L
    return layers


def oracle_layer_expert_source(l, p):
    """Checkpoint-layout experts of layer l regenerated on the CPU (for the oracle)."""
    import synth
    cache = {}

    def routed(e):
        if e not in cache:
            cache[e] = synth.gen_expert((0, "decode-23layers", l, "routed"), synth.N_ROUTED, p=p, index=e)
        return cache[e]

    shared = synth.gen_expert((0, "decode-23layers", l, "shared"), synth.N_SHARED, p=synth.shared_live_fraction(0, l))
    return routed, shared


def time_oracle(n_layers_max, p, budget_s, steps=None):
    """Times the oracle on the host, one layer decode at a time over the first
    n_layers_max layers; returns the seconds of each decode."""
    import oracle
    import synth
    prepared = []
    for l in range(n_layers_max):
        x, lg = synth.tokens(0, "decode-23layers", l, 1)
        routed, shared = oracle_layer_expert_source(l, p)
        idx, _ = oracle.router_topk(lg[0], 6)
        for e in idx:
            routed(int(e))  # generate outside the timed region
        prepared.append((x[0], lg[0], routed, shared))
    times = []
    t_all = time.perf_counter()
    i = 0
    while True:
        x, lg, routed, shared = prepared[i % len(prepared)]
        t0 = time.perf_counter()
        oracle.moe_layer(x, lg, routed, shared, k=6)
        times.append(time.perf_counter() - t0)
        i += 1
        if steps is not None:
            if i >= steps:
                break
        elif time.perf_counter() - t_all > budget_s:
            break
    return times


def _oracle_all_cores_worker(i, p, n_layers, reps, barrier, queue):
    """One process of the all-cores oracle timing: prepares layers
    0..n_layers-1, waits for every process, then runs `reps` layer decodes
    (single-threaded BLAS) and reports its start and end (system-wide
    monotonic clock)."""
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    try:
        import oracle
        import synth
        prepared = []
        for l in range(n_layers):
            x, lg = synth.tokens(0, "decode-23layers", l, 1)
            routed, shared = oracle_layer_expert_source(l, p)
            idx, _ = oracle.router_topk(lg[0], 6)
            for e in idx:
                routed(int(e))
            prepared.append((x[0], lg[0], routed, shared))
        barrier.wait(timeout=300)
        t0 = time.monotonic()
        for r in range(reps):
            x, lg, routed, shared = prepared[(i + r) % n_layers]
            oracle.moe_layer(x, lg, routed, shared, k=6)
        queue.put((i, t0, time.monotonic(), None))
    except Exception as e:  # reported to the parent, which gives up on the leg
        queue.put((i, None, None, repr(e)))


def time_oracle_all_cores(p, reps=6, n_layers=2, timeout_s=600):
    """Oracle throughput on every host core the process may use: one process
    per core (spawned: the parent has a CUDA context), each decoding layers of
    the same workload independently (the 23 layers of a step are independent).
    Returns (seconds per layer decode, processes, layer decodes timed)."""
    import multiprocessing as mp
    n = len(os.sched_getaffinity(0))
    ctx = mp.get_context("spawn")
    barrier, queue = ctx.Barrier(n), ctx.Queue()
    procs = [ctx.Process(target=_oracle_all_cores_worker, args=(i, p, n_layers, reps, barrier, queue), daemon=True)
             for i in range(n)]
    for pr in procs:
        pr.start()
    res = []
    try:
        for _ in range(n):
            res.append(queue.get(timeout=timeout_s))
    finally:
        for pr in procs:
            pr.join(timeout=10)
            if pr.is_alive():
                pr.kill()
                pr.join()
    errs = [r[3] for r in res if r[3]]
    if errs:
        raise RuntimeError(errs[0])
    wall = max(r[2] for r in res) - min(r[1] for r in res)
    return wall / (n * reps), n, n * reps


def bench_batch(args, dev, stream, timed, bytemodel, hs, hbm_peak_gbs):
    """Batch decode through one MoE layer: 8 distinct layers with 30% of every
    expert's neurons permanently dead and p = 0.1 on the rest, cycled so that
    the weights a call reads are not left in L2 by the previous call.  B = 3
    stands for the verify step of speculative decoding (three rows through the
    same weights, sharing the permanently dead neurons)."""
    import numpy as np
    import torch
    import synth
    from activation_sparse_moe_gb300.layer import DeviceLayer, from_synth_expert, from_synth_stack
    n_layers = 8
    layers = []
    for l in range(n_layers):
        L = synth.layer_inputs(0, "batch-dead0.3", l, p=0.1, p_shared=0.1, dead_frac=0.3, device=dev)
        layers.append(DeviceLayer(from_synth_stack(L.up, L.down, L.offsets, dev), from_synth_expert(L.shared, dev), 6))
        del L
    out = {"workload": "moe_decode_batch_1layer_dead0.3_p0.1 (8 distinct layers cycled)", "unit": "us/layer"}
    for B in [int(b) for b in args.batch_sizes.split(",") if b]:
        xs, lgs = zip(*[synth.tokens(0, "batch-dead0.3", 100 * B + l, B) for l in range(n_layers)])
        X = torch.stack(xs).to(dev)
        LG = torch.stack(lgs).to(dev)
        Y = torch.empty((n_layers, B, 2688), dtype=torch.bfloat16, device=dev)
        WS = torch.zeros(max(d.workspace_size(B) for d in layers), dtype=torch.uint8, device=dev)
        req = 0
        token_live = 0   # sum over (token, slot) of the token's own live neurons
        with torch.cuda.stream(stream):
            for l, dl in enumerate(layers):
                dbg = {"topk_idx": torch.empty((B, 6), dtype=torch.int32, device=dev),
                       "topk_w": torch.empty((B, 6), dtype=torch.float32, device=dev),
                       "live_rows": torch.empty(1, dtype=torch.int32, device=dev),
                       "live_groups": torch.empty(1, dtype=torch.int32, device=dev),
                       "live_mask": torch.empty((B, 3712 // 64 + 6 * 1856 // 64), dtype=torch.int64, device=dev)}
                hs.hs_moe_layer_decode(dl.c, X[l], LG[l], B, Y[l], None, 0, dbg, WS, stream=stream)
                stream.synchronize()
                touched = len(set(dbg["topk_idx"].cpu().numpy().ravel().tolist()))
                req += bytemodel.decode_layer_bytes(2688, [3712] + [1856] * touched, int(dbg["live_rows"].item()),
                                                    int(dbg["live_groups"].item()), 128, batch=B)
                token_live += int(np.unpackbits(dbg["live_mask"].cpu().numpy().view(np.uint8)).sum())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l, dl in enumerate(layers):
                hs.hs_moe_layer_decode(dl.c, X[l], LG[l], B, Y[l], None, 0, None, WS, stream=stream)
        K = max(10, args.steps // 4)
        ms, _ = timed(g, K, 3, repeats=3)
        us = ms * 1e3 / (K * n_layers)
        # the same calls with every expert reading the union of all its tokens' live rows once
        gu = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gu, stream=stream):
            for l, dl in enumerate(layers):
                hs.hs_moe_layer_decode(dl.c, X[l], LG[l], B, Y[l], None, hs.HS_BATCH_EXPERT_UNION, None, WS,
                                       stream=stream)
        ms_u, _ = timed(gu, K, 3, repeats=3)
        us_u = ms_u * 1e3 / (K * n_layers)
        # algorithmic work: the dense up product of every (token, expert) pair and the down product over
        # each token's own live rows; floors at the measured HBM peak and at the fp32 FMA peak
        # (152 SMs x 128 lanes x 2 flops x 2.07 GHz = 80.5 TFLOP/s), and which one binds
        flop = 2 * 2688 * (B * (3712 + 6 * 1856) + token_live / n_layers)
        hbm_floor = req / n_layers / (hbm_peak_gbs * 1e3)
        alu_floor = flop / (FP32_PEAK_TFLOPS * 1e6)
        out[f"B{B}"] = {"us_per_layer": round(us, 3), "us_per_token_layer": round(us / B, 4),
                        "required_MB_per_layer": round(req / n_layers / 1e6, 2),
                        "achieved_GBs": round(req / n_layers / (us * 1e-6) / 1e9, 1),
                        "gflop_per_layer": round(flop / 1e9, 3),
                        "hbm_floor_us": round(hbm_floor, 2), "fp32_alu_floor_us": round(alu_floor, 2),
                        "binds": "hbm" if hbm_floor >= alu_floor else "fp32 alu",
                        "expert_union_path_us_per_layer": round(us_u, 3)}
        del g, gu, WS
    del layers
    torch.cuda.empty_cache()
    return out


def bench_expert_down(args, dev, stream, timed, bytemodel, hs, peak):
    """Single-expert sparse down: hs_expert_down_sparse of one token's h (relu(z)^2 with
    z ~ N(Phi^-1(0.1), 1), its own draw per copy) through 512 distinct routed
    experts' 2688 x 1856 down projections (1.44 GB of weights, far above L2),
    called back to back in one CUDA graph; per-call time and the bandwidth on
    the bytes each call must move (live rows, live groups' scale slabs, h, y)."""
    import numpy as np
    import torch
    import synth
    n_copies, N, H = 512, 1856, 2688
    codes = torch.empty((n_copies, N, H // 2), dtype=torch.uint8, device=dev)
    sb = torch.empty((n_copies, N // 64, H), dtype=torch.int32, device=dev)
    for l in range(n_copies // 128):
        _, down = synth.gen_routed_stack((0, "expert-down", l), 128, N, H, device=dev)
        ds, db = down.scale.view(torch.int16), down.bias.view(torch.int16)
        for e in range(128):
            i = 128 * l + e
            hs.hs_repack_down_nm(down.codes[e], ds[e], db[e], H, N, codes[i], sb[i])
        del down
    Hs = torch.stack([synth.expert_down_h(i, N, 0.1) for i in range(n_copies)]).to(dev)
    Y = torch.empty((n_copies, H), dtype=torch.bfloat16, device=dev)
    cnt = torch.zeros(n_copies, dtype=torch.int32, device=dev)
    WS = torch.zeros(hs.hs_expert_down_sparse_workspace_size(N, H), dtype=torch.uint8, device=dev)  # counters start at 0
    with torch.cuda.stream(stream):
        for i in range(n_copies):
            hs.hs_expert_down_sparse(Hs[i], codes[i], sb[i], N, H, Y[i], None, cnt[i:i + 1], 0, WS, stream=stream)
    stream.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    h_cpu = Hs.cpu().numpy()
    live_rows = cnt.cpu().numpy()
    assert np.array_equal(live_rows, (h_cpu > 0).sum(axis=1))
    live_groups = (h_cpu.reshape(n_copies, -1, 64) > 0).any(axis=2).sum(axis=1)
    req = sum(bytemodel.down_sparse_bytes(int(r), int(g), H) + N * 4 + H * 2 for r, g in zip(live_rows, live_groups))
    dense = n_copies * (bytemodel.down_sparse_bytes(N, N // 64, H) + N * 4 + H * 2)

    def capture(flags):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_copies):
                hs.hs_expert_down_sparse(Hs[i], codes[i], sb[i], N, H, Y[i], None, None, flags, WS, stream=stream)
        return g
    K = max(5, args.steps // 20)
    ms, _ = timed(capture(0), K, 3, repeats=3)
    ms_d, _ = timed(capture(hs.HS_FORCE_DENSE), K, 3, repeats=3)
    us, us_d = ms * 1e3 / (K * n_copies), ms_d * 1e3 / (K * n_copies)
    gbs = req / n_copies / (us * 1e-6) / 1e9
    return {"workload": "expert_down_sparse_1tok_512copies_p0.1 (2688x1856 W4 neuron-major)",
            "unit": "us/call", "us_per_call": round(us, 3), "required_KB_per_call": round(req / n_copies / 1e3, 1),
            "live_rows_per_call": round(float(live_rows.mean()), 1),
            "live_groups_per_call": round(float(live_groups.mean()), 2),
            "achieved_GBs": round(gbs, 1), "frac": round(gbs / peak, 4),
            "dense_flag_us_per_call": round(us_d, 3),
            "dense_flag_GBs": round(dense / n_copies / (us_d * 1e-6) / 1e9, 1),
            "kernels_per_call": 1}


def bench_router(args, layers, X, dev, stream, timed, hs, peak):
    """The router projection ahead of each of the 23 resident layers: logits =
    W_router x (bf16 [128][2688] per layer, 688 KB), alone and chained into
    the layer decode on one stream (the decode then routes on these logits)."""
    import torch
    import synth
    n, H, E = len(layers), 2688, 128
    W = torch.stack([synth.router_weights(0, "decode-23layers-router", l) for l in range(n)]).to(dev)
    LGr = torch.empty((n, E), dtype=torch.float32, device=dev)
    Y = torch.empty((n, H), dtype=torch.bfloat16, device=dev)
    WS = torch.zeros(max(dl.workspace_size(1) for dl in layers), dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        for l, dl in enumerate(layers):
            hs.hs_router_logits(X[l], W[l], 1, H, E, LGr[l], stream=stream)
            hs.hs_moe_layer_decode(dl.c, X[l], LGr[l], 1, Y[l], None, 0, None, WS, stream=stream)
    stream.synchronize()
    assert hs.hs_device_status() == hs.HS_OK

    def capture(with_layer):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l, dl in enumerate(layers):
                hs.hs_router_logits(X[l], W[l], 1, H, E, LGr[l], stream=stream)
                if with_layer:
                    hs.hs_moe_layer_decode(dl.c, X[l], LGr[l], 1, Y[l], None, 0, None, WS, stream=stream)
        return g
    K = max(10, args.steps // 4)
    ms_r, _ = timed(capture(False), K, 3, repeats=3)
    ms_rl, _ = timed(capture(True), K, 3, repeats=3)
    us_r, us_rl = ms_r * 1e3 / (K * n), ms_rl * 1e3 / (K * n)
    wbytes = E * H * 2 + H * 2 + E * 4
    return {"workload": "router projection bf16 128x2688 per layer, 23 layers, batch 1", "unit": "us/layer",
            "router_us_per_call": round(us_r, 3), "router_GBs": round(wbytes / (us_r * 1e-6) / 1e9, 1),
            "router_frac": round(wbytes / (us_r * 1e-6) / 1e9 / peak, 4),
            "router_and_layer_us_per_layer": round(us_rl, 3)}


def bench_row_scales(args, X, LG, dev, stream, timed, bytemodel, hs, peak):
    """The same 23 layers with every down projection re-quantised along the
    neuron axis (one (scale, bias) per neuron row and 64 outputs, section "The
    whole decode step"), decoded with HS_DOWN_ROW_SCALES: a live row brings
    its own 176 bytes of scales and no group slab is read."""
    import torch
    n, H = X.shape[0], 2688
    layers = build_layers(n, args.p, dev, down_row_scales=True)
    Y = torch.empty((n, H), dtype=torch.bfloat16, device=dev)
    WS = torch.zeros(max(dl.workspace_size(1) for dl in layers), dtype=torch.uint8, device=dev)
    flags = hs.HS_DOWN_ROW_SCALES
    rows = []
    with torch.cuda.stream(stream):
        for l, dl in enumerate(layers):
            dbg = {"live_rows": torch.empty(1, dtype=torch.int32, device=dev),
                   "live_groups": torch.empty(1, dtype=torch.int32, device=dev)}
            hs.hs_moe_layer_decode(dl.c, X[l], LG[l], 1, Y[l], None, flags, dbg, WS, stream=stream)
            stream.synchronize()
            rows.append(int(dbg["live_rows"].item()))
    assert hs.hs_device_status() == hs.HS_OK
    row_bytes = H // 2 + 4 * hs.hs_row_sb_words(H)
    req = sum(bytemodel.decode_layer_bytes(H, [3712] + [1856] * 6, 0, 0, 128) + r * row_bytes for r in rows)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for l, dl in enumerate(layers):
            hs.hs_moe_layer_decode(dl.c, X[l], LG[l], 1, Y[l], None, flags, None, WS, stream=stream)
    K = max(20, args.steps // 2)
    ms, _ = timed(g, K, 3, repeats=3)
    us = ms * 1e3 / (K * n)
    gbs = req / n / (us * 1e-6) / 1e9
    del layers, g
    torch.cuda.empty_cache()
    return {"workload": "moe_decode_b1_23layers_p0.1, down projections re-quantised with row scales",
            "unit": "us/layer", "us_per_layer": round(us, 3), "required_MB_per_layer": round(req / n / 1e6, 2),
            "live_rows_per_layer": round(sum(rows) / n, 1), "bytes_per_live_row": row_bytes,
            "achieved_GBs": round(gbs, 1), "frac": round(gbs / peak, 4), "flag": "HS_DOWN_ROW_SCALES"}


def bench_p_sweep(args, layers, X, LG, dev, stream, timed, bytemodel, hs, peak):
    """The live-fraction sweep on the same 23 resident layers: the
    routed experts' offsets for live fraction p are the p = 0.1 offsets scaled by
    Phi^-1(p) / Phi^-1(0.1) (the calibration off = Phi^-1(p) * ||w|| is linear
    in Phi^-1(p)); the shared expert keeps its own per-layer fraction; p = 1.0 is
    the dense path on the p = 0.1 inputs (reported as dense_path)."""
    import numpy as np
    import torch
    from scipy.special import ndtri
    from activation_sparse_moe_gb300.layer import DeviceLayer
    n = len(layers)
    Y = torch.empty((n, 2688), dtype=torch.bfloat16, device=dev)
    WS = torch.zeros(max(d.workspace_size(1) for d in layers), dtype=torch.uint8, device=dev)
    out = {}
    for p in (0.02, 0.05, 0.2, 0.5):
        ratio = float(ndtri(p) / ndtri(0.1))
        lp = [DeviceLayer(dl.routed.with_offsets((dl.routed.offsets.double() * ratio).float()), dl.shared, 6)
              for dl in layers]
        rows, groups = [], []
        with torch.cuda.stream(stream):
            for l, dl in enumerate(lp):
                dbg = {"live_rows": torch.empty(1, dtype=torch.int32, device=dev),
                       "live_groups": torch.empty(1, dtype=torch.int32, device=dev)}
                hs.hs_moe_layer_decode(dl.c, X[l], LG[l], 1, Y[l], None, 0, dbg, WS, stream=stream)
                stream.synchronize()
                rows.append(int(dbg["live_rows"].item()))
                groups.append(int(dbg["live_groups"].item()))
        step_bytes = sum(bytemodel.decode_layer_bytes(2688, [3712] + [1856] * 6, r, g, 128) for r, g in zip(rows, groups))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l, dl in enumerate(lp):
                hs.hs_moe_layer_decode(dl.c, X[l], LG[l], 1, Y[l], None, 0, None, WS, stream=stream)
        K = max(20, args.steps // 4)
        ms, _ = timed(g, K, 3, repeats=3)
        us = ms * 1e3 / (K * n)
        gbs = step_bytes / (ms * 1e-3 / K) / 1e9
        out[str(p)] = {"us_per_layer": round(us, 3), "required_MB_per_layer": round(step_bytes / n / 1e6, 2),
                       "achieved_GBs": round(gbs, 1), "frac": round(gbs / peak, 4),
                       "live_rows_per_layer": round(float(np.mean(rows)), 1)}
        del g, lp
    return out


def union_fractions(idx, words, NS, NR, tiles=(32, 128)):
    """Mean over token tiles of the fraction of an expert's neurons that are
    live for some token of the tile (the union), from the kernel's own
    (token, slot) live masks: each routed expert's tokens in token order cut
    into tiles of 32 and 128, the shared expert's likewise."""
    import numpy as np
    T, K = idx.shape
    w = words.view(np.uint64)
    gs, gr = NS // 64, NR // 64
    bits = lambda a: np.unpackbits(a.view(np.uint8), axis=-1).sum(axis=-1)
    out = {}
    for tt in tiles:
        fr = []
        for e in range(int(idx.max()) + 1):
            toks, slots = np.nonzero(idx == e)
            rows = np.stack([w[b, gs + j * gr:gs + (j + 1) * gr] for b, j in zip(toks, slots)]) if len(toks) else None
            for r in range(0, len(toks), tt):
                fr.append(bits(np.bitwise_or.reduce(rows[r:r + tt], axis=0)).sum() / NR)
        fs = [bits(np.bitwise_or.reduce(w[r:r + tt, :gs], axis=0)).sum() / NS for r in range(0, T, tt)]
        out[f"tile{tt}"] = {"routed": round(float(np.mean(fr)), 4), "shared": round(float(np.mean(fs)), 4)}
    out["note"] = ("synthetic activations are independent per token (p = 0.1 on the 70% of neurons not dead), "
                   "so a tile's union approaches the live 70%; real prompts' activations are correlated")
    return out


def bench_prefill(args, dev, stream, timed, hs, peaks):
    """Prefill of a 2048-token chunk through one MoE layer (30% of every
    expert's neurons permanently dead, p = 0.1 on the rest).  Roofline: the
    tensor cores (fp16 operands, fp32 accumulation) against the measured dense
    bf16 GEMM peak (same rate for fp16); the weights (0.73 GB) exceed L2."""
    import numpy as np
    import torch
    import synth
    from activation_sparse_moe_gb300.layer import DeviceLayer, from_synth_expert, from_synth_stack
    T, H, NR, NS = 2048, 2688, 1856, 3712
    L = synth.layer_inputs(0, "prefill-2048", 0, p=0.1, p_shared=0.1, dead_frac=0.3, device=dev)
    dl = DeviceLayer(from_synth_stack(L.up, L.down, L.offsets, dev), from_synth_expert(L.shared, dev), 6)
    del L
    x, lg = synth.tokens(0, "prefill-2048", 0, T)
    X, LG = x.to(dev), lg.to(dev)
    Y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    WS = torch.zeros(dl.prefill_workspace_size(T), dtype=torch.uint8, device=dev)
    dbg = {"tiles": torch.zeros(2, dtype=torch.int32, device=dev),
           "work": torch.zeros(3, dtype=torch.int64, device=dev)}
    # the first call also returns the routing and every (token, slot) live mask, for the union statistic
    dbg0 = dict(dbg, topk_idx=torch.zeros((T, 6), dtype=torch.int32, device=dev),
                topk_w=torch.zeros((T, 6), dtype=torch.float32, device=dev),
                live_mask=torch.zeros((T, NS // 64 + 6 * NR // 64), dtype=torch.int64, device=dev))
    with torch.cuda.stream(stream):
        hs.hs_moe_prefill(dl.c, X, LG, T, Y, None, 0, dbg0, WS, stream=stream)
    stream.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    tiles = [int(v) for v in dbg["tiles"].cpu()]
    work = [int(v) for v in dbg["work"].cpu()]
    union = union_fractions(dbg0["topk_idx"].cpu().numpy(), dbg0["live_mask"].cpu().numpy(), NS, NR)
    up_flops = 2 * H * (T * 6 * NR + T * NS)
    down_alg = 2 * H * work[0]      # union-live rows per (expert, token tile)
    down_exec = 2 * H * work[1]     # rows of the 64-neuron tiles not skipped
    down_dense = 2 * H * work[2]

    def graph(flags):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            hs.hs_moe_prefill(dl.c, X, LG, T, Y, None, flags, None, WS, stream=stream)
        return g

    g_sparse, g_dense = graph(0), graph(hs.HS_FORCE_DENSE)
    K = max(10, args.steps // 10)
    ms, runs = timed(g_sparse, K, 3, repeats=3)
    ms_dense = timed(g_dense, K, 3, repeats=3)[0]
    us = ms * 1e3 / K
    # the row gather (HS_PREFILL_ROW_GATHER): k-steps over each tile's union-live rows
    with torch.cuda.stream(stream):
        hs.hs_moe_prefill(dl.c, X, LG, T, Y, None, hs.HS_PREFILL_ROW_GATHER, dbg, WS, stream=stream)
    stream.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    tiles_g = [int(v) for v in dbg["tiles"].cpu()]
    work_g = [int(v) for v in dbg["work"].cpu()]
    g_gather = graph(hs.HS_PREFILL_ROW_GATHER)
    us_g = timed(g_gather, K, 3, repeats=3)[0] * 1e3 / K
    del g_gather
    alg = up_flops + down_alg
    achieved = alg / (us * 1e-6) / 1e12
    peak = float(peaks.get("bf16_tflops", 1900.0)) if peaks else 1900.0
    out = {"workload": "moe_prefill_2048tok_1layer_dead0.3_p0.1", "unit": "us/chunk",
           "us_per_chunk": round(us, 2), "tokens_per_s": round(T / (us * 1e-6), 1),
           "us_per_chunk_dense_flag": round(ms_dense * 1e3 / K, 2),
           "repeats_us": [round(r * 1e3 / K, 2) for r in runs],
           "skipped_tiles": tiles[0], "considered_tiles": tiles[1],
           "gflop": {"up": round(up_flops / 1e9, 2), "down_union_live": round(down_alg / 1e9, 2),
                     "down_executed": round(down_exec / 1e9, 2), "down_dense": round(down_dense / 1e9, 2)},
           "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                        "frac": round(achieved / peak, 4),
                        "peak_source": "measured" if peaks else "fallback",
                        "flops": "up dense + down over union-live rows per (expert, token tile)",
                        "executed_TFLOPs": round((up_flops + down_exec) / (us * 1e-6) / 1e12, 1)},
           "operands": "fp16 x fp16 -> fp32 (tcgen05.mma kind::f16, accumulators in TMEM)",
           "row_gather": {"flag": "HS_PREFILL_ROW_GATHER", "us_per_chunk": round(us_g, 2),
                          "skipped_ksteps": tiles_g[0], "ksteps_without_skip": tiles_g[1],
                          "gflop_down_executed": round(2 * H * work_g[1] / 1e9, 2),
                          "achieved_TFLOPs": round(alg / (us_g * 1e-6) / 1e12, 1)},
           "union_live_fraction": union}
    del g_sparse, g_dense, dl
    # our sub-configuration: the same 30% dead, but as whole 64-neuron groups (seeded choice per
    # expert, shared included), so that the tile skip has whole tiles to skip
    L = synth.layer_inputs(0, "prefill-2048", 0, p=0.1, p_shared=0.1, dead_frac=0.0, device=dev)
    rng = np.random.default_rng(5)
    for offs in [L.offsets[e] for e in range(L.offsets.shape[0])] + [L.shared.offset]:
        ng = offs.shape[0] // 64
        for gi in rng.choice(ng, size=int(round(0.3 * ng)), replace=False):
            offs[64 * int(gi):64 * (int(gi) + 1)] = float("-inf")
    dl = DeviceLayer(from_synth_stack(L.up, L.down, L.offsets, dev), from_synth_expert(L.shared, dev), 6)
    del L
    with torch.cuda.stream(stream):
        hs.hs_moe_prefill(dl.c, X, LG, T, Y, None, 0, dbg, WS, stream=stream)
    stream.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    tiles_c = [int(v) for v in dbg["tiles"].cpu()]
    work_c = [int(v) for v in dbg["work"].cpu()]
    g_c, g_cd = graph(0), graph(hs.HS_FORCE_DENSE)
    ms_c = timed(g_c, K, 3, repeats=3)[0]
    ms_cd = timed(g_cd, K, 3, repeats=3)[0]
    us_c = ms_c * 1e3 / K
    alg_c = up_flops + 2 * H * work_c[0]
    out["clustered_dead"] = {
        "note": "ours: the 30% dead neurons as whole 64-neuron groups (the tile skip's best case)",
        "us_per_chunk": round(us_c, 2), "us_per_chunk_dense_flag": round(ms_cd * 1e3 / K, 2),
        "skipped_tiles": tiles_c[0], "considered_tiles": tiles_c[1],
        "gflop_down_union_live": round(2 * H * work_c[0] / 1e9, 2),
        "gflop_down_executed": round(2 * H * work_c[1] / 1e9, 2),
        "achieved_TFLOPs": round(alg_c / (us_c * 1e-6) / 1e12, 1),
        "frac": round(alg_c / (us_c * 1e-6) / 1e12 / peak, 4)}
    del g_c, g_cd, WS, dl
    torch.cuda.empty_cache()
    return out


def main():
    args = _args()
    ws, rank, local = _dist()
    if args.impl == "reference":
        return run_reference(args, ws, rank)

    import numpy as np
    import torch
    from activation_sparse_moe_gb300 import build as hsbuild
    from activation_sparse_moe_gb300 import bytemodel, hs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    hsbuild.build()
    hs.lib()
    dev = torch.device("cuda", local)

    import synth
    n = args.layers
    layers = build_layers(n, args.p, dev)
    xs, lgs = [], []
    for l in range(n):
        x, lg = synth.tokens(0, "decode-23layers", l, 1)
        xs.append(x[0])
        lgs.append(lg[0])
    X = torch.stack(xs).to(dev)
    LG = torch.stack(lgs).to(dev)
    Y = torch.empty((n, 2688), dtype=torch.bfloat16, device=dev)
    wsz = max(dl.workspace_size(1) for dl in layers)
    WS = torch.zeros(wsz, dtype=torch.uint8, device=dev)  # zero before first use (control words)
    stream = torch.cuda.Stream(device=dev)

    # untimed pass with debug outputs: live rows and live groups per layer
    live_rows, live_groups = [], []
    NS, NR = 3712, 1856
    with torch.cuda.stream(stream):
        for l, dl in enumerate(layers):
            dbg = {"h": torch.empty(NS + 6 * NR, dtype=torch.float32, device=dev),
                   "live_rows": torch.empty(1, dtype=torch.int32, device=dev),
                   "live_groups": torch.empty(1, dtype=torch.int32, device=dev)}
            hs.hs_moe_layer_decode(dl.c, X[l], LG[l], 1, Y[l], None, 0, dbg, WS, stream=stream)
            stream.synchronize()
            h = dbg["h"].cpu().numpy()
            live_rows.append(int(dbg["live_rows"].item()))
            live_groups.append(int(dbg["live_groups"].item()))
            assert live_rows[-1] == int((h > 0).sum())
            assert live_groups[-1] == int((h.reshape(-1, 64) > 0).any(axis=1).sum())
    assert hs.hs_device_status() == hs.HS_OK
    req_bytes = [bytemodel.decode_layer_bytes(2688, [NS] + [NR] * 6, r, g, 128)
                 for r, g in zip(live_rows, live_groups)]
    dense_bytes = bytemodel.decode_layer_bytes(2688, [NS] + [NR] * 6, NS + 6 * NR, (NS + 6 * NR) // 64, 128)
    step_bytes = sum(req_bytes)

    def capture(flags):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l, dl in enumerate(layers):
                hs.hs_moe_layer_decode(dl.c, X[l], LG[l], 1, Y[l], None, flags, None, WS, stream=stream)
        return g

    # eager warm call (sets kernel attributes outside capture)
    with torch.cuda.stream(stream):
        for l, dl in enumerate(layers):
            hs.hs_moe_layer_decode(dl.c, X[l], LG[l], 1, Y[l], None, 0, None, WS, stream=stream)
    stream.synchronize()
    g_sparse = capture(0)
    g_dense = capture(hs.HS_FORCE_DENSE)

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    def timed(graph, K, W, repeats=1):
        """Median over `repeats` timed regions of K steps (each bracketed by a
        barrier and device synchronisation); returns (median ms, all ms)."""
        for _ in range(W):
            graph.replay()
        stream.synchronize()
        runs = []
        for _ in range(repeats):
            barrier()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(K):
                    graph.replay()
                e1.record(stream)
            stream.synchronize()
            torch.cuda.synchronize()
            barrier()
            ms = e0.elapsed_time(e1)
            if ws > 1:
                ms = max_over_ranks(ms, dev)
            runs.append(ms)
        return statistics.median(runs), runs

    K, W = args.steps, max(3, args.warmup)
    props = torch.cuda.get_device_properties(dev)
    gpu_id = getattr(props, "uuid", None)
    gpu_id = f"GPU-{gpu_id}" if gpu_id is not None and not str(gpu_id).startswith("GPU-") else str(gpu_id or local)
    with ClockSampler(gpu_id) as clk:
        # keep the GPU under this load long enough for the sampler (~1.5 s)
        t_end = time.time() + (0.0 if args.profile else 1.5)
        while time.time() < t_end:
            g_sparse.replay()
        stream.synchronize()
        ms, ms_runs = timed(g_sparse, K, W, repeats=1 if args.profile else 5)
    clocks = clk.summary()
    ms_dense = ms if args.profile else timed(g_dense, K, W, repeats=3)[0]

    us_layer = ms * 1e3 / (K * n)
    us_layer_dense = ms_dense * 1e3 / (K * n)
    achieved = step_bytes / (ms * 1e-3 / K) / 1e9  # GB/s on required bytes
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        peak = float(json.load(open(peaks_path))["hbm_gbs"])
        peak_src = "measured"
    else:
        peak, peak_src = 6800.0, "fallback"

    # end to end through the C ABI: pinned host inputs in, result out, every step
    Xh = X.cpu().pin_memory()
    LGh = LG.cpu().pin_memory()
    Yh = torch.empty((n, 2688), dtype=torch.bfloat16).pin_memory()
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        X.copy_(Xh, non_blocking=True)
        LG.copy_(LGh, non_blocking=True)
        for l, dl in enumerate(layers):
            hs.hs_moe_layer_decode(dl.c, X[l], LG[l], 1, Y[l], None, 0, None, WS, stream=stream)
        Yh.copy_(Y, non_blocking=True)
    ms_e2e = ms if args.profile else timed(g_e2e, K, W, repeats=3)[0]
    us_e2e = ms_e2e * 1e3 / (K * n)
    h2d = X.numel() * X.element_size() + LG.numel() * LG.element_size()
    d2h = Y.numel() * Y.element_size()

    sweep = None
    if not args.profile and not args.no_sweep:
        sweep = bench_p_sweep(args, layers, X, LG, dev, stream, timed, bytemodel, hs, peak)
        sweep["0.1"] = {"us_per_layer": round(us_layer, 3), "required_MB_per_layer": round(step_bytes / n / 1e6, 2),
                        "achieved_GBs": round(achieved, 1), "frac": round(achieved / peak, 4)}
        sweep["1.0"] = {"us_per_layer": round(us_layer_dense, 3), "note": "HS_FORCE_DENSE on the p = 0.1 inputs",
                        "required_MB_per_layer": round(dense_bytes / 1e6, 2),
                        "achieved_GBs": round(dense_bytes / (us_layer_dense * 1e-6) / 1e9, 1)}
    row_scales = None
    if not args.profile and not args.no_row_scales:
        row_scales = bench_row_scales(args, X, LG, dev, stream, timed, bytemodel, hs, peak)
    router = None
    if not args.profile and not args.no_router:
        router = bench_router(args, layers, X, dev, stream, timed, hs, peak)
    expert_down = None
    if not args.profile and not args.no_expert_down:
        expert_down = bench_expert_down(args, dev, stream, timed, bytemodel, hs, peak)
    batch = None
    if not args.profile and args.batch_sizes:
        batch = bench_batch(args, dev, stream, timed, bytemodel, hs, peak)
    prefill = None
    if not args.profile and not args.no_prefill:
        prefill = bench_prefill(args, dev, stream, timed, hs,
                                json.load(open(peaks_path)) if os.path.exists(peaks_path) else None)

    cpu = None
    if rank == 0 and ws == 1 and not (args.no_cpu_baseline or args.profile):
        times = time_oracle(3, args.p, budget_s=12.0)
        cpu = {"value": statistics.median(times) * 1e6, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{len(times)} layer decodes of layers 0-2 of the same workload (fp64 numpy, "
                         "single-threaded BLAS), median per layer"}
        if not args.no_cpu_all_cores:
            try:
                s_all, n_proc, n_dec = time_oracle_all_cores(args.p)
                cpu["all_cores"] = {"value": round(s_all * 1e6, 1), "unit": UNIT, "cores": n_proc,
                                    "sample": f"{n_proc} processes (one per host core), each {n_dec // n_proc} "
                                              "layer decodes of layers 0-1; wall time of all of them / decodes"}
            except Exception as e:  # the single-core figure above stands on its own
                cpu["all_cores"] = {"error": repr(e)[:200]}

    if rank == 0:
        csrc = os.path.join(ROOT, "activation_sparse_moe_gb300", "csrc")
        src = [os.path.join(csrc, f) for f in ("hs_decode.cu", "hs_kernels.cuh", "hs_common.cuh", "hs_host.h")]
        out = {
            "metric": METRIC, "value": round(us_layer, 4), "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": W,
            "ms_per_step": round(ms / K, 6), "repeats_us_per_layer": [round(r * 1e3 / (K * n), 3) for r in ms_runs],
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded; random W4 weights of the page's shapes)",
            "config": _config(args, {"operands": "W4 weights, bf16 activations, fp32 accumulate, bf16 out"}),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "peak_source": peak_src,
                         "kernel": "hs_moe_layer_decode (moe_decode_b1_kernel + reduce_partials_kernel)",
                         "bytes_per_launch": round(step_bytes / n),
                         "traffic": _recorded_traffic("moe_decode_b1_kernel", src),
                         "frac_of_8TBs": round(achieved / 8000.0, 4),
                         # the time the required bytes take at the peak, beside the measured us_per_layer
                         "byte_floor_us_per_layer": round(step_bytes / n / (peak * 1e3), 3)},
            "e2e": {"value": round(us_e2e, 4), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": 2 * n * K,  # the timed region of the headline metric
            "clocks": clocks,
            "dense_path": {"value": round(us_layer_dense, 4), "unit": UNIT, "flag": "HS_FORCE_DENSE",
                           "speedup_sparse_vs_dense": round(us_layer_dense / us_layer, 3),
                           "bytes_per_layer": dense_bytes},
            "live": {"rows_per_layer": round(float(np.mean(live_rows)), 1),
                     "groups_per_layer": round(float(np.mean(live_groups)), 1),
                     "required_MB_per_step": round(step_bytes / 1e6, 2)},
            "p_sweep": sweep,
            "row_scales": row_scales,
            "router": router,
            "expert_down": expert_down,
            "batch_decode": batch,
            "prefill": prefill,
            "cpu_baseline": cpu,
        }
        print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_reference(args, ws, rank):
    """The reference arm: the CPU oracle on the host cores, same workload."""
    if rank != 0:
        return
    K, W = args.steps, max(3, args.warmup)
    # bound the run: the oracle takes about a second per layer
    K_eff = min(K, 20)
    W_eff = min(W, 3)
    times = time_oracle(min(4, args.layers), args.p, budget_s=None, steps=K_eff + W_eff)
    t = times[W_eff:]
    v = statistics.median(t) * 1e6
    out = {"metric": METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": ws, "steps": len(t), "warmup": W_eff,
           "ms_per_step": round(statistics.median(t) * 1e3, 3), "higher_is_better": False, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
           "config": _config(args),
           "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
                            "sample": f"one layer decode per step cycling over layers 0-3, {len(t)} timed steps "
                                      f"(requested {K}), fp64 numpy"},
           "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(v, "1")
    main()
