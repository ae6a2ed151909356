"""Benchmark of the activation-sparse FFN hot path on GB300.

Workload: the Llama3.2-1B FFN stack -- 16 SwiGLU layers, d=2048, d_ff=8192,
bf16 weights ~N(0,0.02) with per-neuron LogNormal(0,1) gate-row scales,
gamma=0.7 loaded, delta=0.2 static, phi=0.4 computed, alpha=1024, a prompt of
T=512 tokens and 256 decode tokens at batch 1, on synthetic seeded data.

One step = one request through the online path:
  prefill  for every layer: |A| on the tensor cores (si_prefill_absact),
           per-token top-alpha + counts + top-beta union (si_select_from_absact);
  decode   256 tokens x 16 layers of si_sparse_ffn_decode_residual (y += FFN(x))
           on the selected set, with the decode plan built after prefill.
Both halves are CUDA graphs replayed on one stream; CUDA events bracket each.
The offline steps (profiler scores over 4096 calibration tokens, selective
loading) run once before the timed region and are reported on their own; the
SpAx three-tier decode of the Llama-3.1-8B stack is reported in "spax".

metric: sparse-FFN decode tokens/s at batch 1 (value), with the achieved HBM
GB/s of the selected-weight stream and the prefill select ms in the line.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       (N > 1: launched by torch.distributed.run, one independent replica per GPU)
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "sparse-FFN decode tokens/s (bs1) + achieved HBM GB/s; prefill select ms"
WL = synth.WORKLOADS["llama3.2-1b"]
SPAX_WL = synth.WORKLOADS["llama3.1-8b-spax"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# ------------------------------------------------------------------ distributed


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the timing rule: the slowest replica)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_path=None):
        self.gpu = gpu_index
        self.proc = None
        self.log_path = log_path

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        else:
            self.out = ""
        if self.log_path:
            with open(self.log_path, "w") as f:
                f.write(self.out)

    def summary(self):
        rows = [r.split(",") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if "Active" in r[5 + k] and "Not" not in r[5 + k]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ GPU arm


def gpu_weights(torch, seed, layer, d, N, sigma, dev):
    g = torch.Generator(device=dev)
    g.manual_seed(seed * 1000003 + layer)
    scale = torch.exp(sigma * torch.randn(N, 1, generator=g, device=dev, dtype=torch.float32))
    Wg = (torch.randn(N, d, generator=g, device=dev, dtype=torch.float32) * 0.02 * scale).to(torch.bfloat16)
    Wu = (torch.randn(N, d, generator=g, device=dev, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    Wd = (torch.randn(d, N, generator=g, device=dev, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    return Wg, Wu, Wd


def gpu_tokens(torch, seed, tag, rows, d, dev):
    g = torch.Generator(device=dev)
    g.manual_seed(seed * 7919 + tag)
    return torch.randn(rows, d, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)


def build_selectinfer(si, torch, dev, seed):
    """Weights, offline profile + pack (timed once), prompt and decode inputs."""
    w = WL
    layers, Ws = [], []
    t_prof = t_pack = 0.0
    for l in range(w.L):
        Wg, Wu, Wd = gpu_weights(torch, seed, l, w.d, w.N, w.sigma, dev)
        Xc = gpu_tokens(torch, seed, 100 + l, w.calib_tokens, w.d, dev)
        s = torch.zeros(w.N, dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        si.si_profile_scores(Wg, Wu, Xc, s)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        layer = si.si_pack_loaded(Wg, Wu, Wd, s, s, w.gamma, w.delta)
        torch.cuda.synchronize()
        t2 = time.perf_counter()
        t_prof += t1 - t0
        t_pack += t2 - t1
        layers.append(layer)
        Ws.append((Wg, Wu, Wd))
        del Xc
    return layers, Ws, t_prof, t_pack


def time_graph(torch, g, stream):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    return e0, e1


def run_gpu(args, world, rank, local):
    import torch
    import activation_sparse_gb300 as si

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        init_dist(world, "nccl")
    hbm_peak, tf_peak, tf_sus, peak_kind = peaks()
    w = WL
    seed = 1234 + rank
    n_loaded, n_static, n_sel, beta = si.si_counts(w.N, w.gamma, w.delta, w.phi)

    layers, Ws, t_prof, t_pack = build_selectinfer(si, torch, dev, seed)
    n_pad = layers[0].n_pad
    M = w.T * w.B
    X = [gpu_tokens(torch, seed, 200 + l, M, w.d, dev) for l in range(w.L)]
    xdec = gpu_tokens(torch, seed, 300, w.decode_tokens * w.L, w.d, dev).view(w.decode_tokens, w.L, w.d)
    A = torch.empty((M, n_pad), dtype=torch.float32, device=dev)
    S = [torch.empty((w.B, n_sel), dtype=torch.int32, device=dev) for _ in range(w.L)]
    y = torch.zeros((w.decode_tokens, w.L, w.d), dtype=torch.float32, device=dev)

    stream = torch.cuda.Stream(device=dev)

    def prefill_gemm_only():
        for l in range(w.L):
            si.si_prefill_absact(layers[l], X[l], w.T, w.B, A)

    def prefill():
        for l in range(w.L):
            si.si_prefill_absact(layers[l], X[l], w.T, w.B, A)
            si.si_select_from_absact(layers[l], A, w.T, w.B, w.alpha, w.phi, S[l])
            si.si_decode_plan(layers[l], S[l], n_sel, w.B)

    # decode in the residual form (y += FFN(x)), the way a transformer adds the
    # FFN output to its residual stream; y holds one residual row per (token, layer)
    def decode():
        for t in range(w.decode_tokens):
            for l in range(w.L):
                si.si_sparse_ffn_decode_residual(layers[l], S[l], n_sel, w.B, xdec[t, l], y[t, l])

    def decode_one_pass():
        for l in range(w.L):
            si.si_sparse_ffn_decode_residual(layers[l], S[l], n_sel, w.B, xdec[0, l], y[0, l])

    with torch.cuda.stream(stream):
        prefill()
        decode_one_pass()
        stream.synchronize()
        g_pre, g_dec, g_gemm = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_pre, stream=stream):
            prefill()
        with torch.cuda.graph(g_dec, stream=stream):
            decode()
        with torch.cuda.graph(g_gemm, stream=stream):
            prefill_gemm_only()
    assert si.si_device_error() == 0

    # warm-up
    for _ in range(args.warmup):
        g_pre.replay()
        g_dec.replay()
        g_gemm.replay()
    stream.synchronize()

    # our kernels per step: GEMM, top-alpha, top-beta per layer (the counts
    # are zeroed by a memset and the batch-1 plan is a device copy, neither a
    # kernel of ours; the B > 1 plan is), then one decode launch per layer-token
    launches_per_step = w.L * (3 + (1 if w.B > 1 else 0)) + w.decode_tokens * w.L
    pre_ms, dec_ms = [], []
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local, os.path.join(args.out_dir, "clocks_rank%d.csv" % rank) if args.out_dir else None) as clk:
        t_wall0 = time.perf_counter()
        ev = []
        for _ in range(args.steps):
            with torch.cuda.stream(stream):
                ev.append((time_graph(torch, g_pre, stream), time_graph(torch, g_dec, stream)))
        stream.synchronize()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
        barrier(world)
    for (p0, p1), (d0, d1) in ev:
        pre_ms.append(p0.elapsed_time(p1))
        dec_ms.append(d0.elapsed_time(d1))
    # the prefill GEMM alone (tensor-core roofline), also with events on its stream
    gemm_ms = []
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.steps)):
            e0, e1 = time_graph(torch, g_gemm, stream)
            stream.synchronize()
            gemm_ms.append(e0.elapsed_time(e1))
    assert si.si_device_error() == 0, "device error during the timed region"

    dec_total_s = max_over_ranks(sum(dec_ms) / 1e3, world, dev)
    step_total_s = max_over_ranks((sum(dec_ms) + sum(pre_ms)) / 1e3, world, dev)
    tokens_all = sum_over_ranks(w.decode_tokens * w.B * args.steps, world, dev)
    value = tokens_all / dec_total_s
    ms_per_token = dec_total_s * 1e3 / (w.decode_tokens * args.steps)
    sel_bytes_token = w.L * (n_sel * 6 * w.d + n_sel * 4 + 2 * w.d + 4 * w.d)
    launch_bytes = n_sel * 6 * w.d + n_sel * 4 + 2 * w.d + 4 * w.d
    launch_s = dec_total_s / (w.decode_tokens * w.L * args.steps)
    achieved_gbs = launch_bytes / launch_s / 1e9
    gemm_flop = w.L * 4.0 * M * w.d * n_loaded
    gemm_s = statistics.median(gemm_ms) / 1e3
    gemm_tfs = gemm_flop / gemm_s / 1e12

    # e2e: host buffers through the same C-ABI calls, copies inside the timed region
    e2e = run_e2e(si, torch, dev, stream, layers, S, n_sel, args)

    # Table 1's layer range on the same stack: the first five and the last two
    # layers keep the dense FFN (packed at gamma = 1, decoded on S = every position)
    layer_range = run_layer_range(si, torch, dev, stream, layers, Ws, S, n_sel, xdec, y)

    spax = None
    if not args.no_spax and rank == 0:
        del Ws
        torch.cuda.empty_cache()
        spax = run_spax(si, torch, dev, stream, args)

    clocks = clk.summary()
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_total_s * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded torch generator; shapes and distributions of the Llama3.2-1B FFN stack)",
        "config": {"workload": WL.name, "layers": w.L, "d": w.d, "d_ff": w.N, "gamma": w.gamma, "delta": w.delta,
                   "phi": w.phi, "alpha": w.alpha, "prompt_tokens": w.T, "batch": w.B,
                   "decode_tokens": w.decode_tokens, "n_loaded": n_loaded, "n_sel": n_sel,
                   "parallelism": "replicas x%d" % world,
                   "l2": "inputs larger than L2: 644 MB of selected weights per decode token, 1.1 GB packed"},
        "hbm_gbs": round(sel_bytes_token / (ms_per_token / 1e3) / 1e9, 1),
        "decode_ms_per_token": round(ms_per_token, 5),
        "prefill_select_ms": round(statistics.mean(pre_ms), 4),
        "prefill_gemm_ms": round(gemm_s * 1e3, 4),
        "offline_ms": {"profile_16_layers_4096_tokens": round(t_prof * 1e3, 3), "pack_16_layers": round(t_pack * 1e3, 3)},
        "roofline": {"kernel": "k_sparse_decode_b1", "bound": "hbm", "achieved": round(achieved_gbs, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved_gbs / hbm_peak, 4),
                     "peak_source": peak_kind, "traffic": args.traffic,
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch"
                     if args.traffic is not None else None,
                     "bytes_per_launch": launch_bytes, "launch_us": round(launch_s * 1e6, 3)},
        "prefill_roofline": {"kernel": "k_act_gemm", "bound": "tensor", "achieved": round(gemm_tfs, 1),
                             "peak": tf_peak, "unit": "TFLOP/s", "frac": round(gemm_tfs / tf_peak, 4),
                             "peak_source": peak_kind, "flop_per_stack": gemm_flop},
        "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"], "reasons": clocks["reasons"]},
        "wall_s_timed": round(t_wall, 4),
    }
    out["layer_range"] = layer_range
    if spax is not None:
        out["spax"] = spax
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_layer_range(si, torch, dev, stream, layers, Ws, S, n_sel, xdec, y, toks=64):
    """Decode tokens/s of the stack with SelectInfer's layer range (Table 1: first
    layer 5, skip the last 2): layers outside it run the dense FFN through the
    same decode, packed at gamma = 1 with S = every position."""
    w = WL
    mask = si.si_sparse_layers(w.L, 5, -2)
    full = torch.arange(w.N, dtype=torch.int32, device=dev).view(1, -1).contiguous()
    ones = torch.ones(w.N, dtype=torch.float32, device=dev)
    dense = {}
    for l in range(w.L):
        if not mask[l]:
            Wg, Wu, Wd = Ws[l]
            dense[l] = si.si_pack_loaded(Wg, Wu, Wd, ones, ones, 1.0, 0.0)

    def run():
        for t in range(toks):
            for l in range(w.L):
                if mask[l]:
                    si.si_sparse_ffn_decode_residual(layers[l], S[l], n_sel, 1, xdec[t, l], y[t, l])
                else:
                    si.si_sparse_ffn_decode_residual(dense[l], full, w.N, 1, xdec[t, l], y[t, l])

    with torch.cuda.stream(stream):
        for l in dense:
            si.si_decode_plan(dense[l], full, w.N, 1)
        run()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run()
        g.replay()
        e0, e1 = time_graph(torch, g, stream)
        stream.synchronize()
    assert si.si_device_error() == 0
    s_tok = e0.elapsed_time(e1) / 1e3 / toks
    n_sp = int(mask.sum())
    per = lambda n: n * 6 * w.d + n * 4 + 2 * w.d + 4 * w.d
    byts = n_sp * per(n_sel) + (w.L - n_sp) * per(w.N)
    for l in dense:
        dense[l].close()
    return {"first_layer": 5, "last_layer": -2, "sparse_layers": n_sp, "dense_layers": w.L - n_sp,
            "tokens": toks, "tokens_per_s": round(1.0 / s_tok, 2), "ms_per_token": round(s_tok * 1e3, 4),
            "bytes_per_token": byts, "hbm_gbs": round(byts / s_tok / 1e9, 1)}


def run_e2e(si, torch, dev, stream, layers, S, n_sel, args):
    """Same request through the C ABI with pinned HOST buffers: prompt and decode
    inputs copied in, S and outputs copied out, all inside the timed region."""
    w = WL
    M = w.T * w.B
    hX = [torch.empty((M, w.d), dtype=torch.bfloat16).pin_memory() for _ in range(w.L)]
    hx = torch.empty((w.decode_tokens, w.L, w.d), dtype=torch.bfloat16).pin_memory()
    hy = torch.empty((w.decode_tokens, w.L, w.d), dtype=torch.float32).pin_memory()
    hS = torch.empty((w.L, w.B, n_sel), dtype=torch.int32).pin_memory()
    for t in hX:
        t.copy_(torch.randn(M, w.d).to(torch.bfloat16))
    hx.copy_(torch.randn(w.decode_tokens, w.L, w.d).to(torch.bfloat16))
    dX = [torch.empty((M, w.d), dtype=torch.bfloat16, device=dev) for _ in range(w.L)]
    dx = torch.empty_like(hx, device=dev)
    dy = torch.empty_like(hy, device=dev)
    A = torch.empty((M, layers[0].n_pad), dtype=torch.float32, device=dev)

    def request():
        for l in range(w.L):
            dX[l].copy_(hX[l], non_blocking=True)
        dx.copy_(hx, non_blocking=True)
        for l in range(w.L):
            si.si_prefill_absact(layers[l], dX[l], w.T, w.B, A)
            si.si_select_from_absact(layers[l], A, w.T, w.B, w.alpha, w.phi, S[l])
            si.si_decode_plan(layers[l], S[l], n_sel, w.B)
            hS[l].copy_(S[l], non_blocking=True)
        dy.zero_()
        for t in range(w.decode_tokens):
            for l in range(w.L):
                si.si_sparse_ffn_decode_residual(layers[l], S[l], n_sel, w.B, dx[t, l], dy[t, l])
        hy.copy_(dy, non_blocking=True)

    with torch.cuda.stream(stream):
        request()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            request()
        for _ in range(max(1, args.warmup)):
            g.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
        stream.synchronize()
    s = e0.elapsed_time(e1) / 1e3
    h2d = sum(t.numel() * 2 for t in hX) + hx.numel() * 2
    d2h = hy.numel() * 4 + hS.numel() * 4
    return {"value": round(w.decode_tokens * w.B * args.steps / s, 2), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(s * 1e3 / args.steps, 4)}


def run_spax(si, torch, dev, stream, args):
    """SpAx three-tier decode on the Llama-3.1-8B FFN stack (32 x d=4096, d_ff=14336):
    per token and layer a dense gate/up pass, the tier choice and the tiered down-projection."""
    w = SPAX_WL
    seed = 99
    W, enc = [], []
    for l in range(w.L):
        Wg, Wu, Wd = gpu_weights(torch, seed, l, w.d, w.N, w.sigma, dev)
        enc.append(si.spax_encode(Wd, w.bits, w.group))
        del Wd
        W.append((Wg, Wu))
    toks = 64
    x = gpu_tokens(torch, seed, 400, toks * w.L, w.d, dev).view(toks, w.L, w.d)
    y = torch.empty((toks, w.L, w.d), dtype=torch.float32, device=dev)
    a = torch.empty((w.L, w.N), dtype=torch.float32, device=dev)

    def run():
        for t in range(toks):
            for l in range(w.L):
                si.spax_ffn_decode(enc[l], W[l][0], W[l][1], x[t, l], w.top_frac, w.mid_frac, y[t, l], a[l])

    def dense_only():
        for t in range(toks):
            for l in range(w.L):
                si.spax_dense_act(W[l][0], W[l][1], x[t, l], a[l])

    with torch.cuda.stream(stream):
        run()
        stream.synchronize()
        g, gd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run()
        with torch.cuda.graph(gd, stream=stream):
            dense_only()
        for _ in range(2):
            g.replay()
            gd.replay()
        stream.synchronize()
        e0, e1 = time_graph(torch, g, stream)
        f0, f1 = time_graph(torch, gd, stream)
        stream.synchronize()
    assert si.si_device_error() == 0
    ms = e0.elapsed_time(e1)
    dense_ms = f0.elapsed_time(f1)
    k_top, k_mid = si.si_count(w.top_frac, w.N), si.si_count(w.mid_frac, w.N)
    byts = w.L * (2 * w.N * w.d * 2 + k_top * 2 * w.d + k_mid * (w.d // 2 + 8 * (w.d // w.group)))
    per_tok = ms / 1e3 / toks
    dense_bytes = w.L * 2 * w.N * w.d * 2
    dense_s = dense_ms / 1e3 / (toks * w.L)
    hbm_peak, _, _, kind = peaks()
    select = spax_in_selected_set(si, torch, dev, stream, W, enc, seed)
    widths = spax_code_widths(si, torch, dev, stream, W, seed)
    return {"workload": w.name, "tokens": toks, "tokens_per_s": round(1.0 / per_tok, 2),
            "ms_per_token": round(per_tok * 1e3, 4), "hbm_gbs": round(byts / per_tok / 1e9, 1),
            "bytes_per_token": byts, "top_frac": w.top_frac, "mid_frac": w.mid_frac,
            "dense_act_roofline": {"kernel": "k_dense_act", "bound": "hbm",
                                   "achieved": round(dense_bytes / w.L / dense_s / 1e9, 1), "peak": hbm_peak,
                                   "unit": "GB/s", "frac": round(dense_bytes / w.L / dense_s / 1e9 / hbm_peak, 4),
                                   "peak_source": kind},
            "code_widths": widths, "in_selected_set": select}


def spax_in_selected_set(si, torch, dev, stream, W, enc, seed, layers=4, toks=64, phi=0.4):
    """SelectInfer x SpAx on the first `layers` layers: gate/up only on a selected
    set of phi*N neurons, then the top/middle tiers as fractions of that set."""
    w = SPAX_WL
    n_rows = si.si_count(phi, w.N)
    gen = torch.Generator(device="cpu").manual_seed(seed + 7)
    rows = [torch.sort(torch.randperm(w.N, generator=gen)[:n_rows])[0].to(torch.int32).to(dev) for _ in range(layers)]
    x = gpu_tokens(torch, seed, 402, toks * layers, w.d, dev).view(toks, layers, w.d)
    y = torch.empty((toks, layers, w.d), dtype=torch.float32, device=dev)
    a = torch.empty((layers, w.N), dtype=torch.float32, device=dev)

    def run():
        for t in range(toks):
            for l in range(layers):
                si.spax_select_decode(enc[l], W[l][0], W[l][1], rows[l], x[t, l], w.top_frac, w.mid_frac, y[t, l], a[l])

    with torch.cuda.stream(stream):
        run()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run()
        g.replay()
        e0, e1 = time_graph(torch, g, stream)
        stream.synchronize()
    assert si.si_device_error() == 0
    us = e0.elapsed_time(e1) * 1e3 / (toks * layers)
    k_top, k_mid = si.si_count(w.top_frac, n_rows), si.si_count(w.mid_frac, n_rows)
    ngp = -(-(w.d // w.group) // 2) * 2
    byts = n_rows * 2 * w.d * 2 + k_top * 2 * w.d + k_mid * (w.d * w.bits // 8 + 8 * ngp)
    return {"phi": phi, "selected": n_rows, "k_top": k_top, "k_mid": k_mid, "us_per_layer_token": round(us, 2),
            "bytes_per_layer_token": byts, "hbm_gbs": round(byts / us / 1e3, 1)}


def spax_code_widths(si, torch, dev, stream, W, seed, layers=4, toks=64):
    """The same SpAx layer-token with 2-, 4- and 8-bit middle-tier codes, on the
    first `layers` layers of the stack: microseconds per layer-token and the
    selected bytes (dense gate/up + bf16 top + b-bit records) per second."""
    w = SPAX_WL
    k_top, k_mid = si.si_count(w.top_frac, w.N), si.si_count(w.mid_frac, w.N)
    ngp = -(-(w.d // w.group) // 2) * 2
    x = gpu_tokens(torch, seed, 401, toks * layers, w.d, dev).view(toks, layers, w.d)
    y = torch.empty((toks, layers, w.d), dtype=torch.float32, device=dev)
    a = torch.empty((layers, w.N), dtype=torch.float32, device=dev)
    out = {}
    for bits in (2, 4, 8):
        enc = []
        for l in range(layers):
            _, _, Wd = gpu_weights(torch, seed, l, w.d, w.N, w.sigma, dev)
            enc.append(si.spax_encode(Wd, bits, w.group))
            del Wd

        def run():
            for t in range(toks):
                for l in range(layers):
                    si.spax_ffn_decode(enc[l], W[l][0], W[l][1], x[t, l], w.top_frac, w.mid_frac, y[t, l], a[l])

        with torch.cuda.stream(stream):
            run()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run()
            g.replay()
            e0, e1 = time_graph(torch, g, stream)
            stream.synchronize()
        assert si.si_device_error() == 0
        us = e0.elapsed_time(e1) * 1e3 / (toks * layers)
        byts = 2 * w.N * w.d * 2 + k_top * 2 * w.d + k_mid * (w.d * bits // 8 + 8 * ngp)
        out[str(bits)] = {"us_per_layer_token": round(us, 2), "hbm_gbs": round(byts / us / 1e3, 1),
                          "bytes_per_layer_token": byts}
        for e in enc:
            e.close()
    return out


# ------------------------------------------------------------------ CPU oracle


def cpu_sample(seconds_budget: float):
    """Times the oracle on a bounded sample of the workload: one full-size
    layer's sparse decode for a few tokens (the decode metric), plus the
    selection of one layer's prompt. Returns (decode tokens/s for the 16-layer
    stack, description, threads)."""
    import oracle
    w = WL
    Wg, Wu, Wd = synth.layer_weights(5, 0, w.d, w.N, w.sigma)
    sc = synth.lognormal_absact(5, 1, w.N)[0]
    loaded, st = oracle.rank_loaded(sc, sc, w.gamma, w.delta)
    n_sel = oracle.cnt(w.phi, w.N)
    A = synth.lognormal_absact(6, w.T, len(loaded))
    t0 = time.perf_counter()
    S = oracle.select(A, w.T, w.B, len(loaded), st, w.alpha, n_sel)
    t_sel = time.perf_counter() - t0
    xs = synth.tokens(7, 0, synth.T_DECODE, 64, w.d)
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle.sparse_ffn(Wg, Wu, Wd, loaded, S[0], xs[n % 64])
        n += 1
        el = time.perf_counter() - t0
        if el > seconds_budget or n >= 2000:
            break
    per_layer_token = el / n
    tps = 1.0 / (w.L * per_layer_token)
    desc = ("oracle sparse_ffn on %d layer-tokens of one full-size layer (d=2048, |S|=%d), "
            "scaled to the 16-layer stack; top-alpha/top-beta selection of one 512-token prompt took %.3f s"
            % (n, n_sel, t_sel))
    return tps, desc, oracle.num_threads(), n


def cpu_baseline(seconds_budget: float):
    tps, desc, cores, _ = cpu_sample(seconds_budget)
    return {"value": round(tps, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores."""
    if rank != 0:
        return
    t_all = time.perf_counter()
    vals = []
    for _ in range(args.warmup):
        cpu_sample(min(2.0, args.cpu_seconds))
    for _ in range(args.steps):
        tps, desc, cores, n = cpu_sample(args.cpu_seconds / max(1, args.steps))
        vals.append(tps)
    value = statistics.median(vals)
    w = WL
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * w.decode_tokens / value, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded counter-based generator)",
           "config": {"workload": WL.name, "layers": w.L, "d": w.d, "d_ff": w.N, "gamma": w.gamma,
                      "delta": w.delta, "phi": w.phi, "alpha": w.alpha, "prompt_tokens": w.T, "batch": w.B,
                      "decode_tokens": w.decode_tokens, "parallelism": "cpu"},
           "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": desc},
           "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "wall_s": round(time.perf_counter() - t_all, 2)}
    print(json.dumps(out), flush=True)


def run_profile_case(args):
    """A few launches of one kernel on one full-size layer, for ncu captures:
    decode (k_sparse_decode_b1 in the residual form with a decode plan, as
    the timed step runs it, Llama3.2-1B layer), prefill (k_act_gemm,
    512-token prompt), dense (k_dense_act) and tiered (k_tiered_down) on a
    Llama-3.1-8B layer. Prints one JSON line with the CUDA-event time."""
    import torch
    import activation_sparse_gb300 as si
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    case = args.profile_case
    if case in ("decode", "prefill"):
        w = WL
        Wg, Wu, Wd = gpu_weights(torch, 7, 0, w.d, w.N, w.sigma, dev)
        s = torch.rand(w.N, device=dev)
        layer = si.si_pack_loaded(Wg, Wu, Wd, s, s, w.gamma, w.delta)
        X = gpu_tokens(torch, 7, 1, w.T, w.d, dev)
        n_sel = si.si_count(w.phi, w.N)
        S = torch.empty((1, n_sel), dtype=torch.int32, device=dev)
        A = torch.empty((w.T, layer.n_pad), dtype=torch.float32, device=dev)
        si.si_select_dynamic(layer, X, w.T, 1, w.alpha, w.phi, S, A)
        x = gpu_tokens(torch, 7, 2, 1, w.d, dev)
        y = torch.empty((1, w.d), dtype=torch.float32, device=dev)
        si.si_decode_plan(layer, S, n_sel, 1)
        y.zero_()
        fn = (lambda: si.si_sparse_ffn_decode_residual(layer, S, n_sel, 1, x, y)) if case == "decode" else \
             (lambda: si.si_prefill_absact(layer, X, w.T, 1, A))
    else:
        w = SPAX_WL
        Wg, Wu, Wd = gpu_weights(torch, 7, 0, w.d, w.N, w.sigma, dev)
        enc = si.spax_encode(Wd, w.bits, w.group)
        x = gpu_tokens(torch, 7, 2, 1, w.d, dev)[0]
        a = torch.empty(w.N, dtype=torch.float32, device=dev)
        y = torch.empty(w.d, dtype=torch.float32, device=dev)
        si.spax_dense_act(Wg, Wu, x, a)
        fn = (lambda: si.spax_dense_act(Wg, Wu, x, a)) if case == "dense" else \
             (lambda: si.spax_tiered_down(enc, a, w.top_frac, w.mid_frac, y))
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    assert si.si_device_error() == 0
    print(json.dumps({"profile_case": case, "launches": args.steps, "ms_per_launch": e0.elapsed_time(e1) / args.steps}))


# DRAM bytes (read + write) of one k_sparse_decode_b1 launch on one
# Llama3.2-1B layer, from the ncu capture summarised in
# profiles/k_sparse_decode_b1_llama3.2-1b_layer.md (40.3226 MB read, 1.0 KB
# written). Set to None whenever that kernel changes until it is re-captured.
DECODE_TRAFFIC_BYTES = 40322560 + 1024


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-spax", action="store_true", help="skip the SpAx Llama-3.1-8B measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU oracle time budget")
    ap.add_argument("--traffic", type=float, default=DECODE_TRAFFIC_BYTES,
                    help="DRAM bytes per k_sparse_decode_b1 launch from an ncu capture (null when unknown)")
    ap.add_argument("--out-dir", default=None, help="directory for the clock samples (optional)")
    ap.add_argument("--profile-case", choices=["decode", "prefill", "dense", "tiered"], default=None,
                    help="run only a few launches of one kernel (for ncu captures)")
    args = ap.parse_args(argv)
    if args.profile_case:
        run_profile_case(args)
        return 0
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return 0
    run_gpu(args, world, rank, local)
    return 0


if __name__ == "__main__":
    sys.exit(main())
