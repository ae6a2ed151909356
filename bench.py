"""Benchmark of the activation-sparse FFN hot path on GB300.

Headline workload: the Llama3.2-3B FFN stack -- 28 SwiGLU layers, d=3072,
d_ff=8192, bf16 weights ~N(0,0.02) with per-neuron LogNormal(0,1) gate-row
scales, gamma=0.7 loaded, delta=0.25 static, phi=0.5 computed, alpha=1024, a
prompt of T=1024 tokens and 512 decode tokens at batch 1, on synthetic seeded
data (SelectInfer's headline model, section 6.7).

One step = one request through the online path:
  prefill  for every layer: |A| on the tensor cores (si_prefill_absact),
           per-token top-alpha + counts + top-beta union (si_select_from_absact),
           then the decode plan (si_decode_plan);
  decode   512 tokens x 28 layers of si_sparse_ffn_decode_residual (y += FFN(x))
           on the selected set, one launch per layer in stream order.
Both halves are CUDA graphs replayed on one stream; CUDA events bracket each.
The offline steps (profiler scores over 4096 calibration tokens, selective
loading) run once before the timed region and are reported on their own.

The line also carries, for the same stack: the decode stack (one cooperative
launch per token over all layers on an RMS-normalised residual stream,
si_sparse_ffn_decode_stack), the overwrite decode call (si_sparse_ffn_decode)
and Table 1's layer range; and one object per other workload (the single
d=256 layer, Llama3.2-1B, Qwen2.5-3B with 8 prompts, the Llama-3.1-8B SpAx
stack), each with its own roofline, prefill roofline, end-to-end figure and
CPU-oracle baseline.

metric: sparse-FFN decode tokens/s at batch 1 (value), with the achieved HBM
GB/s of the selected-weight stream and the prefill select ms in the line.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       (N > 1: launched by torch.distributed.run, one independent replica per GPU)
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "sparse-FFN decode tokens/s (bs1) + achieved HBM GB/s; prefill select ms"
HEAD = synth.WORKLOADS["llama3.2-3b"]
SUB_WORKLOADS = ["tiny-d256", "llama3.2-1b", "qwen2.5-3b", "llama3.1-8b-spax"]


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
    """nvidia-smi samples of SM clock and throttle reasons during a region (read-only queries)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, log_path=None):
        self.gpu = gpu_index
        self.proc = None
        self.log_path = log_path
        self.out = ""

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


# ------------------------------------------------------------------ traffic record


def kernel_source_hash():
    """Hash of the sources of the batch-1 decode kernel and the dense pass;
    a DRAM-traffic figure taken with other sources is not reported."""
    h = hashlib.sha256()
    for f in ("decode.cu", "ring.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "activation_sparse_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key):
    """(bytes per launch, source) of the ncu capture recorded for this kernel and
    workload, or (None, reason) when none was taken with the current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None, "no capture recorded"
    rec = json.load(open(p)).get(kernel_key)
    if not rec:
        return None, "no capture recorded for this kernel"
    if rec.get("source_hash") != kernel_source_hash():
        return None, "kernel changed since the capture"
    return int(rec["dram_bytes_per_launch"]), rec.get("capture", "ncu")


# ------------------------------------------------------------------ GPU helpers


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


def time_graph(torch, g, stream):
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    return e0, e1


def graph_of(torch, stream, fn):
    with torch.cuda.stream(stream):
        fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
    return g


def replay_ms(torch, g, stream, reps=1):
    """Mean ms of `reps` back-to-back replays (CUDA events on the launching stream)."""
    with torch.cuda.stream(stream):
        g.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        stream.synchronize()
    return e0.elapsed_time(e1) / reps


def decode_launch_bytes(w, n_union, n_sel):
    """Algorithmic bytes of one decode launch: the selected records (gate row,
    up row, down column; the union over the B sequences), their positions (and
    sequence masks for B > 1), x in and y out."""
    if w.B == 1:
        return n_sel * 6 * w.d + 4 * n_sel + 2 * w.d + 4 * w.d
    return n_union * 6 * w.d + 8 * n_union + w.B * (2 * w.d + 4 * w.d)


# ------------------------------------------------------------------ SelectInfer stacks


class SIStack:
    """Packed layers of one workload with their computed sets."""

    def __init__(self, si, torch, dev, w, seed, keep_weights=False):
        self.w, self.layers, self.Ws = w, [], []
        self.t_prof = self.t_pack = 0.0
        for l in range(w.L):
            Wg, Wu, Wd = gpu_weights(torch, seed, l, w.d, w.N, w.sigma, dev)
            Xc = gpu_tokens(torch, seed, 100 + l, w.calib_tokens, w.d, dev)
            s = torch.zeros(w.N, dtype=torch.float32, device=dev)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            si.si_profile_scores(Wg, Wu, Xc, s)
            torch.cuda.synchronize()
            t1 = time.perf_counter()
            self.layers.append(si.si_pack_loaded(Wg, Wu, Wd, s, s, w.gamma, w.delta))
            torch.cuda.synchronize()
            self.t_prof += t1 - t0
            self.t_pack += time.perf_counter() - t1
            if keep_weights:
                self.Ws.append((Wg, Wu, Wd))
            del Xc
        self.n_loaded, self.n_static, self.n_sel, self.beta = si.si_counts(w.N, w.gamma, w.delta, w.phi)
        self.n_pad = self.layers[0].n_pad
        self.M = w.T * w.B
        self.X = [gpu_tokens(torch, seed, 200 + l, self.M, w.d, dev) for l in range(w.L)]
        self.A = torch.empty((self.M, self.n_pad), dtype=torch.float32, device=dev)
        self.S = [torch.empty((w.B, self.n_sel), dtype=torch.int32, device=dev) for _ in range(w.L)]

    def prefill(self, si, gemm_only=False):
        w = self.w
        for l in range(w.L):
            si.si_prefill_absact(self.layers[l], self.X[l], w.T, w.B, self.A)
            if not gemm_only:
                si.si_select_from_absact(self.layers[l], self.A, w.T, w.B, w.alpha, w.phi, self.S[l])
                si.si_decode_plan(self.layers[l], self.S[l], self.n_sel, w.B)

    def union_sizes(self):
        return [int(np.unique(S.cpu().numpy()).size) for S in self.S]

    def close(self):
        for layer in self.layers:
            layer.close()


def run_selectinfer(si, torch, dev, stream, w, args, seed, *, steps, warmup, dec_tokens, world=1, rank=0,
                    local=0, headline=False):
    """Prefill selection + decode of one SelectInfer workload; returns the result object."""
    hbm_peak, tf_peak, tf_sus, peak_kind = peaks()
    st = SIStack(si, torch, dev, w, seed, keep_weights=headline)
    xdec = gpu_tokens(torch, seed, 300, dec_tokens * w.L * w.B, w.d, dev).view(dec_tokens, w.L, w.B, w.d)
    y = torch.zeros((dec_tokens, w.L, w.B, w.d), dtype=torch.float32, device=dev)
    residual = w.B == 1

    def decode():
        for t in range(dec_tokens):
            for l in range(w.L):
                if residual:
                    si.si_sparse_ffn_decode_residual(st.layers[l], st.S[l], st.n_sel, 1, xdec[t, l], y[t, l])
                else:
                    si.si_sparse_ffn_decode(st.layers[l], st.S[l], st.n_sel, w.B, xdec[t, l], y[t, l])

    with torch.cuda.stream(stream):
        st.prefill(si)
        stream.synchronize()
    g_pre = graph_of(torch, stream, lambda: st.prefill(si))
    g_dec = graph_of(torch, stream, decode)
    g_gemm = graph_of(torch, stream, lambda: st.prefill(si, gemm_only=True))
    assert si.si_device_error() == 0
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g_pre.replay()
            g_dec.replay()
            g_gemm.replay()
        stream.synchronize()

    pre_ms, dec_ms = [], []
    clk = None
    barrier(world)
    torch.cuda.synchronize()
    sampler = ClockSampler(local, os.path.join(args.out_dir, "clocks_rank%d.csv" % rank) if args.out_dir else None) \
        if headline else None
    if sampler:
        sampler.__enter__()
    t_wall0 = time.perf_counter()
    ev = []
    with torch.cuda.stream(stream):
        for _ in range(steps):
            ev.append((time_graph(torch, g_pre, stream), time_graph(torch, g_dec, stream)))
    stream.synchronize()
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    barrier(world)
    if sampler:
        sampler.__exit__(None, None, None)
        clk = sampler.summary()
    for (p0, p1), (d0, d1) in ev:
        pre_ms.append(p0.elapsed_time(p1))
        dec_ms.append(d0.elapsed_time(d1))
    gemm_ms = statistics.median(replay_ms(torch, g_gemm, stream) for _ in range(max(3, min(steps, 10))))
    assert si.si_device_error() == 0, "device error during the timed region"

    dec_total_s = max_over_ranks(sum(dec_ms) / 1e3, world, dev)
    step_total_s = max_over_ranks((sum(dec_ms) + sum(pre_ms)) / 1e3, world, dev)
    tokens_all = sum_over_ranks(dec_tokens * w.B * steps, world, dev)
    value = tokens_all / dec_total_s
    ms_per_token = dec_total_s * 1e3 / (dec_tokens * steps)
    unions = st.union_sizes() if w.B > 1 else [st.n_sel] * w.L
    launch_bytes = [decode_launch_bytes(w, u, st.n_sel) for u in unions]
    token_bytes = sum(launch_bytes)
    launch_s = dec_total_s / (dec_tokens * w.L * steps)
    achieved = (token_bytes / w.L) / launch_s / 1e9
    gemm_flop = w.L * 4.0 * st.M * w.d * st.n_loaded
    gemm_tfs = gemm_flop / (gemm_ms / 1e3) / 1e12
    # batches at d = 1024 / 2048 run on the tensor-core kernel (template: d / 128)
    if w.B == 1:
        kern = "k_sparse_decode_b1"
    elif w.d in (1024, 2048):
        kern = "k_sparse_decode_mma<%d>" % (w.d // 128)
    else:
        kern = "k_sparse_decode<%d>" % w.B
    traffic, traffic_src = recorded_traffic("%s@%s" % (kern, w.name))
    out = {
        "workload": w.name, "value": round(value, 2), "unit": "tokens/s",
        "ms_per_token": round(ms_per_token, 5), "decode_tokens": dec_tokens, "steps": steps,
        "hbm_gbs": round(token_bytes / (ms_per_token / 1e3) / 1e9, 1),
        "bytes_per_token": token_bytes,
        "decode_call": "si_sparse_ffn_decode_residual" if residual else "si_sparse_ffn_decode (B=%d)" % w.B,
        "prefill_select_ms": round(statistics.mean(pre_ms), 4),
        "prefill_gemm_ms": round(gemm_ms, 4),
        "offline_ms": {"profile": round(st.t_prof * 1e3, 3), "pack": round(st.t_pack * 1e3, 3)},
        "roofline": {"kernel": kern, "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "peak_source": peak_kind,
                     "traffic": traffic, "traffic_source": traffic_src,
                     "bytes_per_launch": int(round(token_bytes / w.L)), "launch_us": round(launch_s * 1e6, 3),
                     "launch_us_note": "decode time / launches: includes the gaps between dependent launches"},
        "prefill_roofline": {"kernel": "k_act_gemm", "bound": "tensor", "achieved": round(gemm_tfs, 1),
                             "peak": tf_peak, "unit": "TFLOP/s", "frac": round(gemm_tfs / tf_peak, 4),
                             "peak_source": peak_kind + " burst", "flop_per_stack": gemm_flop,
                             "tokens": st.M, "neurons": st.n_loaded},
        "gpu_launches_per_step": w.L * (3 + (1 if w.B > 1 else 0)) + dec_tokens * w.L,
    }
    if w.B > 1:
        out["union_per_layer"] = {"min": min(unions), "max": max(unions), "mean": round(float(np.mean(unions)), 1)}
    if w.d * w.N * 6 * w.L < 128e6:
        out["roofline"]["l2_resident"] = True
        out["roofline"]["note"] = "the selected weights fit in L2: a latency figure, not an HBM roofline"
    out["e2e"] = run_e2e(si, torch, dev, stream, st, w, args, min(dec_tokens, 64 if not headline else dec_tokens),
                         steps if headline else 2)
    if headline:
        out["_step_total_s"] = step_total_s
        out["_wall_s"] = t_wall
        out["_clocks"] = clk
        out["stack"] = run_stack(si, torch, dev, stream, st, w, seed)
        out["overwrite_form"] = run_overwrite(si, torch, dev, stream, st, w, seed, xdec)
        out["layer_range"] = run_layer_range(si, torch, dev, stream, st, w, xdec, y)
    st.close()
    del st, xdec, y
    torch.cuda.empty_cache()
    return out


def run_e2e(si, torch, dev, stream, st, w, args, toks, reps):
    """The request through the C ABI with pinned HOST buffers: prompt and decode
    inputs copied in, S and the decode outputs copied out, inside the timed
    region. The copies run on a second stream of the same graph, each tied by
    events to the work that needs it (a layer's prompt before its prefill, a
    token's inputs before its decode, its outputs after it), so they overlap
    the compute as copy engines allow; the step ends when every copy has
    landed."""
    hX = [torch.empty((st.M, w.d), dtype=torch.bfloat16).pin_memory() for _ in range(w.L)]
    hx = torch.empty((toks, w.L, w.B, w.d), dtype=torch.bfloat16).pin_memory()
    hy = torch.empty((toks, w.L, w.B, w.d), dtype=torch.float32).pin_memory()
    hS = torch.empty((w.L, w.B, st.n_sel), dtype=torch.int32).pin_memory()
    for t in hX:
        t.copy_(torch.randn(st.M, w.d).to(torch.bfloat16))
    hx.copy_(torch.randn(toks, w.L, w.B, w.d).to(torch.bfloat16))
    dX = [torch.empty((st.M, w.d), dtype=torch.bfloat16, device=dev) for _ in range(w.L)]
    dx = torch.empty_like(hx, device=dev)
    dy = torch.empty_like(hy, device=dev)
    cs = torch.cuda.Stream(device=dev)  # the copies

    def request():
        cur = torch.cuda.current_stream()
        cs.wait_stream(cur)  # the copies follow the previous work
        ev_X = [torch.cuda.Event() for _ in range(w.L)]
        ev_x = [torch.cuda.Event() for _ in range(toks)]
        with torch.cuda.stream(cs):
            for l in range(w.L):
                dX[l].copy_(hX[l], non_blocking=True)
                ev_X[l].record(cs)
            for t in range(toks):
                dx[t].copy_(hx[t], non_blocking=True)
                ev_x[t].record(cs)
        for l in range(w.L):
            cur.wait_event(ev_X[l])
            si.si_prefill_absact(st.layers[l], dX[l], w.T, w.B, st.A)
            si.si_select_from_absact(st.layers[l], st.A, w.T, w.B, w.alpha, w.phi, st.S[l])
            si.si_decode_plan(st.layers[l], st.S[l], st.n_sel, w.B)
            done = torch.cuda.Event()
            done.record(cur)
            cs.wait_event(done)
            with torch.cuda.stream(cs):
                hS[l].copy_(st.S[l], non_blocking=True)
        dy.zero_()
        for t in range(toks):
            cur.wait_event(ev_x[t])
            for l in range(w.L):
                if w.B == 1:
                    si.si_sparse_ffn_decode_residual(st.layers[l], st.S[l], st.n_sel, 1, dx[t, l], dy[t, l])
                else:
                    si.si_sparse_ffn_decode(st.layers[l], st.S[l], st.n_sel, w.B, dx[t, l], dy[t, l])
            done = torch.cuda.Event()
            done.record(cur)
            cs.wait_event(done)
            with torch.cuda.stream(cs):
                hy[t].copy_(dy[t], non_blocking=True)
        cur.wait_stream(cs)  # the step ends when every copy has landed

    g = graph_of(torch, stream, request)
    with torch.cuda.stream(stream):
        for _ in range(max(1, args.warmup)):
            g.replay()
        stream.synchronize()
    ms = replay_ms(torch, g, stream, reps)
    assert si.si_device_error() == 0
    h2d = sum(t.numel() * 2 for t in hX) + hx.numel() * 2
    d2h = hy.numel() * 4 + hS.numel() * 4
    return {"value": round(toks * w.B / (ms / 1e3), 2), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 4),
            "decode_tokens_per_step": toks,
            "note": "one request per step: prompt + decode inputs in from pinned host memory, sets and outputs "
                    "back, prefill selection and decode through the C ABI, one CUDA graph; the copies run on a "
                    "second stream of the graph, each tied by events to the work that needs it"}


def run_stack(si, torch, dev, stream, st, w, seed, toks=64):
    """The same layers and sets through the decode stack: one cooperative launch
    per token, x_l = bf16(RMSnorm(h)), h += FFN_l(x_l) (a dependent chain)."""
    hbm_peak, _, _, kind = peaks()
    stack = si.si_stack_create(st.layers)
    si.si_stack_plan(stack, [S.view(-1) for S in st.S], [st.n_sel] * w.L)
    h = gpu_tokens(torch, seed, 500, toks, w.d, dev).float().contiguous()

    def run():
        for t in range(toks):
            si.si_sparse_ffn_decode_stack(stack, h[t])

    g = graph_of(torch, stream, run)
    ms = statistics.median(replay_ms(torch, g, stream) for _ in range(3))
    assert si.si_device_error() == 0
    stack.close()
    us = ms * 1e3 / toks
    byts = w.L * decode_launch_bytes(w, st.n_sel, st.n_sel)
    return {"call": "si_sparse_ffn_decode_stack", "tokens": toks, "tokens_per_s": round(1e6 / us, 2),
            "us_per_token": round(us, 3),
            "roofline": {"kernel": "k_sparse_decode_stack", "bound": "hbm", "achieved": round(byts / us / 1e3, 1),
                         "peak": hbm_peak, "unit": "GB/s", "frac": round(byts / us / 1e3 / hbm_peak, 4),
                         "peak_source": kind, "bytes_per_token": byts},
            "note": "one launch per token; the layers form a real dependent chain (each layer reads the "
                    "RMS-normalised residual stream the previous one wrote)"}


def run_overwrite(si, torch, dev, stream, st, w, seed, xdec, toks=64):
    """The overwrite call (si_sparse_ffn_decode, deterministic 64-bit fixed-point sum) per layer."""
    hbm_peak, _, _, kind = peaks()
    y = torch.empty((toks, w.L, w.B, w.d), dtype=torch.float32, device=dev)

    def run():
        for t in range(toks):
            for l in range(w.L):
                si.si_sparse_ffn_decode(st.layers[l], st.S[l], st.n_sel, w.B, xdec[t, l], y[t, l])

    g = graph_of(torch, stream, run)
    ms = statistics.median(replay_ms(torch, g, stream) for _ in range(3))
    assert si.si_device_error() == 0
    us = ms * 1e3 / toks
    byts = w.L * decode_launch_bytes(w, st.n_sel, st.n_sel)
    return {"call": "si_sparse_ffn_decode", "tokens": toks, "tokens_per_s": round(1e6 / us, 2),
            "us_per_token": round(us, 3),
            "roofline": {"kernel": "k_sparse_decode_b1 (overwrite)", "bound": "hbm",
                         "achieved": round(byts / us / 1e3, 1), "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(byts / us / 1e3 / hbm_peak, 4), "peak_source": kind}}


def run_layer_range(si, torch, dev, stream, st, w, xdec, y, toks=64):
    """Decode tokens/s of the stack with SelectInfer's layer range (Table 1: first
    layer 5, skip the last 2): layers outside it run the dense FFN through the
    same decode, packed at gamma = 1 with S = every position."""
    mask = si.si_sparse_layers(w.L, 5, -2)
    full = torch.arange(w.N, dtype=torch.int32, device=dev).view(1, -1).contiguous()
    ones = torch.ones(w.N, dtype=torch.float32, device=dev)
    dense = {}
    for l in range(w.L):
        if not mask[l]:
            Wg, Wu, Wd = st.Ws[l]
            dense[l] = si.si_pack_loaded(Wg, Wu, Wd, ones, ones, 1.0, 0.0)

    def run():
        for t in range(toks):
            for l in range(w.L):
                if mask[l]:
                    si.si_sparse_ffn_decode_residual(st.layers[l], st.S[l], st.n_sel, 1, xdec[t, l], y[t, l])
                else:
                    si.si_sparse_ffn_decode_residual(dense[l], full, w.N, 1, xdec[t, l], y[t, l])

    with torch.cuda.stream(stream):
        for l in dense:
            si.si_decode_plan(dense[l], full, w.N, 1)
    g = graph_of(torch, stream, run)
    ms = statistics.median(replay_ms(torch, g, stream) for _ in range(3))
    assert si.si_device_error() == 0
    s_tok = ms / 1e3 / toks
    n_sp = int(mask.sum())
    byts = n_sp * decode_launch_bytes(w, st.n_sel, st.n_sel) + (w.L - n_sp) * decode_launch_bytes(w, w.N, w.N)
    for l in dense:
        dense[l].close()
    return {"first_layer": 5, "last_layer": -2, "sparse_layers": n_sp, "dense_layers": w.L - n_sp,
            "tokens": toks, "tokens_per_s": round(1.0 / s_tok, 2), "ms_per_token": round(s_tok * 1e3, 4),
            "bytes_per_token": byts, "hbm_gbs": round(byts / s_tok / 1e9, 1)}


# ------------------------------------------------------------------ SpAx


def run_spax(si, torch, dev, stream, args, toks=64):
    """SpAx three-tier decode on the Llama-3.1-8B FFN stack (32 x d=4096, d_ff=14336):
    per token and layer a dense gate/up pass, the tier choice and the tiered down-projection."""
    w = synth.WORKLOADS["llama3.1-8b-spax"]
    seed = 99
    hbm_peak, _, _, kind = peaks()
    W, enc = [], []
    for l in range(w.L):
        Wg, Wu, Wd = gpu_weights(torch, seed, l, w.d, w.N, w.sigma, dev)
        enc.append(si.spax_encode(Wd, w.bits, w.group))
        del Wd
        W.append((Wg, Wu))
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

    g, gd = graph_of(torch, stream, run), graph_of(torch, stream, dense_only)
    ms = statistics.median(replay_ms(torch, g, stream) for _ in range(3))
    dense_ms = statistics.median(replay_ms(torch, gd, stream) for _ in range(3))
    assert si.si_device_error() == 0
    k_top, k_mid = si.si_count(w.top_frac, w.N), si.si_count(w.mid_frac, w.N)
    ngp = -(-(w.d // w.group) // 2) * 2
    tier_bytes = k_top * 2 * w.d + k_mid * (w.d * w.bits // 8 + 8 * ngp)
    dense_bytes = 2 * w.N * w.d * 2
    byts = w.L * (dense_bytes + tier_bytes)
    per_tok = ms / 1e3 / toks
    dense_s = dense_ms / 1e3 / (toks * w.L)
    tier_s = max(per_tok / w.L - dense_s, 1e-9)
    traffic, tsrc = recorded_traffic("k_dense_act@" + w.name)
    out = {"workload": w.name, "value": round(1.0 / per_tok, 2), "unit": "tokens/s", "tokens": toks,
           "ms_per_token": round(per_tok * 1e3, 4), "hbm_gbs": round(byts / per_tok / 1e9, 1),
           "bytes_per_token": byts, "top_frac": w.top_frac, "mid_frac": w.mid_frac, "bits": w.bits,
           "roofline": {"kernel": "k_dense_act", "bound": "hbm", "achieved": round(dense_bytes / dense_s / 1e9, 1),
                        "peak": hbm_peak, "unit": "GB/s", "frac": round(dense_bytes / dense_s / 1e9 / hbm_peak, 4),
                        "peak_source": kind, "traffic": traffic, "traffic_source": tsrc,
                        "bytes_per_launch": dense_bytes, "launch_us": round(dense_s * 1e6, 3)},
           "tiered_roofline": {"kernel": "k_tiered_down", "bound": "hbm",
                               "achieved": round(tier_bytes / tier_s / 1e9, 1), "peak": hbm_peak, "unit": "GB/s",
                               "frac": round(tier_bytes / tier_s / 1e9 / hbm_peak, 4), "peak_source": kind,
                               "bytes_per_launch": tier_bytes, "launch_us": round(tier_s * 1e6, 3),
                               "note": "token time per layer minus the dense pass's time per layer"},
           "token_roofline_frac": round(byts / per_tok / 1e9 / hbm_peak, 4)}
    out["e2e"] = spax_e2e(si, torch, dev, stream, enc, W, w, args)
    out["all"] = spax_all(si, torch, dev, stream, W, enc, seed)
    out["in_selected_set"] = spax_in_selected_set(si, torch, dev, stream, W, enc, seed)
    out["code_widths"] = spax_code_widths(si, torch, dev, stream, W, seed)
    for e in enc:
        e.close()
    del W, enc, x, y, a
    torch.cuda.empty_cache()
    return out


def spax_all(si, torch, dev, stream, W, enc, seed, layers=8, toks=64, in_top=0.3, in_mid=0.3):
    """SpAx-ALL for the FFN on the first `layers` layers: tiers on the gate/up
    projections by |x| (input channels, 30 % bf16 / 30 % 4-bit codes) then the
    down tiers by |a|; k_spax_gate_up's own roofline from a gate/up-only graph."""
    w = synth.WORKLOADS["llama3.1-8b-spax"]
    hbm_peak, _, _, kind = peaks()
    gates, ups = [], []
    for l in range(layers):
        gates.append(si.spax_encode_rows(W[l][0], w.bits, w.group))
        ups.append(si.spax_encode_rows(W[l][1], w.bits, w.group))
    x = gpu_tokens(torch, seed, 403, toks * layers, w.d, dev).view(toks, layers, w.d)
    y = torch.empty((toks, layers, w.d), dtype=torch.float32, device=dev)
    a = torch.empty((layers, w.N), dtype=torch.float32, device=dev)

    def run():
        for t in range(toks):
            for l in range(layers):
                si.spax_all_decode(enc[l], gates[l], ups[l], x[t, l], in_top, in_mid, w.top_frac, w.mid_frac,
                                   y[t, l], a[l])

    def gate_up_only():
        for t in range(toks):
            for l in range(layers):
                si.spax_gate_up(gates[l], ups[l], x[t, l], in_top, in_mid, a[l])

    g, gg = graph_of(torch, stream, run), graph_of(torch, stream, gate_up_only)
    ms = statistics.median(replay_ms(torch, g, stream) for _ in range(3))
    gu_ms = statistics.median(replay_ms(torch, gg, stream) for _ in range(3))
    assert si.si_device_error() == 0
    for e in gates + ups:
        e.close()
    kt, km = si.si_count(in_top, w.d), si.si_count(in_mid, w.d)
    ngp_n = -(-(w.N // w.group) // 2) * 2
    gu_bytes = kt * w.N * 2 * 2 + km * 2 * (w.N * w.bits // 8 + 8 * (w.N // w.group))
    k_top, k_mid = si.si_count(w.top_frac, w.N), si.si_count(w.mid_frac, w.N)
    ngp = -(-(w.d // w.group) // 2) * 2
    down_bytes = k_top * 2 * w.d + k_mid * (w.d * w.bits // 8 + 8 * ngp)
    us = ms * 1e3 / (toks * layers)
    gu_us = gu_ms * 1e3 / (toks * layers)
    del ngp_n
    return {"layers": layers, "tokens": toks, "in_top_frac": in_top, "in_mid_frac": in_mid,
            "us_per_layer_token": round(us, 2), "bytes_per_layer_token": gu_bytes + down_bytes,
            "hbm_gbs": round((gu_bytes + down_bytes) / us / 1e3, 1),
            "frac": round((gu_bytes + down_bytes) / us / 1e3 / hbm_peak, 4),
            "tokens_per_s_32_layers": round(1e6 / (us * w.L), 2),
            "gate_up_roofline": {"kernel": "k_spax_gate_up", "bound": "hbm", "achieved": round(gu_bytes / gu_us / 1e3, 1),
                                 "peak": hbm_peak, "unit": "GB/s", "frac": round(gu_bytes / gu_us / 1e3 / hbm_peak, 4),
                                 "peak_source": kind, "bytes_per_launch": gu_bytes, "launch_us": round(gu_us, 3)}}


def spax_e2e(si, torch, dev, stream, enc, W, w, args, toks=16):
    """SpAx decode tokens through the C ABI with the token inputs copied in from
    pinned host memory and the outputs read back, inside the timed region."""
    hx = torch.randn(toks, w.L, w.d).to(torch.bfloat16).pin_memory()
    hy = torch.empty((toks, w.L, w.d), dtype=torch.float32).pin_memory()
    dx = torch.empty_like(hx, device=dev)
    dy = torch.empty_like(hy, device=dev)
    a = torch.empty((w.L, w.N), dtype=torch.float32, device=dev)

    def run():
        dx.copy_(hx, non_blocking=True)
        for t in range(toks):
            for l in range(w.L):
                si.spax_ffn_decode(enc[l], W[l][0], W[l][1], dx[t, l], w.top_frac, w.mid_frac, dy[t, l], a[l])
        hy.copy_(dy, non_blocking=True)

    g = graph_of(torch, stream, run)
    ms = statistics.median(replay_ms(torch, g, stream) for _ in range(3))
    assert si.si_device_error() == 0
    return {"value": round(toks / (ms / 1e3), 2), "unit": "tokens/s", "h2d_bytes_per_step": int(hx.numel() * 2),
            "d2h_bytes_per_step": int(hy.numel() * 4), "ms_per_step": round(ms, 4), "decode_tokens_per_step": toks}


def spax_in_selected_set(si, torch, dev, stream, W, enc, seed, layers=4, toks=64, phi=0.4):
    """SelectInfer x SpAx on the first `layers` layers: gate/up only on a selected
    set of phi*N neurons, then the top/middle tiers as fractions of that set."""
    w = synth.WORKLOADS["llama3.1-8b-spax"]
    hbm_peak, _, _, kind = peaks()
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

    g = graph_of(torch, stream, run)
    ms = statistics.median(replay_ms(torch, g, stream) for _ in range(3))
    assert si.si_device_error() == 0
    us = ms * 1e3 / (toks * layers)
    k_top, k_mid = si.si_count(w.top_frac, n_rows), si.si_count(w.mid_frac, n_rows)
    ngp = -(-(w.d // w.group) // 2) * 2
    byts = n_rows * 2 * w.d * 2 + k_top * 2 * w.d + k_mid * (w.d * w.bits // 8 + 8 * ngp)
    return {"phi": phi, "selected": n_rows, "k_top": k_top, "k_mid": k_mid, "us_per_layer_token": round(us, 2),
            "bytes_per_layer_token": byts, "hbm_gbs": round(byts / us / 1e3, 1),
            "frac": round(byts / us / 1e3 / hbm_peak, 4), "peak_source": kind}


def spax_code_widths(si, torch, dev, stream, W, seed, layers=4, toks=64):
    """The same SpAx layer-token with 2-, 3-, 4- and 8-bit middle-tier codes, on the
    first `layers` layers of the stack: microseconds per layer-token and the
    selected bytes (dense gate/up + bf16 top + b-bit records) per second."""
    w = synth.WORKLOADS["llama3.1-8b-spax"]
    k_top, k_mid = si.si_count(w.top_frac, w.N), si.si_count(w.mid_frac, w.N)
    ngp = -(-(w.d // w.group) // 2) * 2
    x = gpu_tokens(torch, seed, 401, toks * layers, w.d, dev).view(toks, layers, w.d)
    y = torch.empty((toks, layers, w.d), dtype=torch.float32, device=dev)
    a = torch.empty((layers, w.N), dtype=torch.float32, device=dev)
    out = {}
    for bits in (2, 3, 4, 8):
        enc = []
        for l in range(layers):
            _, _, Wd = gpu_weights(torch, seed, l, w.d, w.N, w.sigma, dev)
            enc.append(si.spax_encode(Wd, bits, w.group))
            del Wd

        def run():
            for t in range(toks):
                for l in range(layers):
                    si.spax_ffn_decode(enc[l], W[l][0], W[l][1], x[t, l], w.top_frac, w.mid_frac, y[t, l], a[l])

        g = graph_of(torch, stream, run)
        ms = statistics.median(replay_ms(torch, g, stream) for _ in range(3))
        assert si.si_device_error() == 0
        us = ms * 1e3 / (toks * layers)
        byts = 2 * w.N * w.d * 2 + k_top * 2 * w.d + k_mid * (w.d * bits // 8 + 8 * ngp)
        out[str(bits)] = {"us_per_layer_token": round(us, 2), "hbm_gbs": round(byts / us / 1e3, 1),
                          "bytes_per_layer_token": byts}
        for e in enc:
            e.close()
    return out


# ------------------------------------------------------------------ CPU oracle


def _cpu_bf16(rng, shape, scale=1.0):
    """Seeded normal bf16 bit patterns for the CPU samples (input generation only)."""
    f = (rng.standard_normal(shape, dtype=np.float32) * np.float32(scale)).view(np.uint32)
    return ((f + np.uint32(0x7FFF) + ((f >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def cpu_sample(w, tokens_per_layer=9, prefill_rows=16, seed=11):
    """Times the oracle on a bounded sample of workload w: the sparse decode FFN
    of layers {0, L/2, L-1} for the first 8 decode tokens and the last one,
    single-threaded and with OpenMP over rows and neurons, and one prompt's
    selection (|A| of `prefill_rows` rows scaled to the prompt, then top-alpha,
    counts and top-beta on the full prompt). Full-stack figures are
    extrapolated per layer and token. Returns a dict."""
    import oracle
    rng = np.random.default_rng(seed)
    layers = sorted({0, w.L // 2, w.L - 1})
    n_threads = oracle.num_threads()
    t_st = t_mt = 0.0
    n = 0
    t_abs = t_sel = 0.0
    for l in layers:
        Wg = _cpu_bf16(rng, (w.N, w.d), 0.02)
        Wu = _cpu_bf16(rng, (w.N, w.d), 0.02)
        Wd = _cpu_bf16(rng, (w.d, w.N), 0.02)
        s = rng.random(w.N).astype(np.float32)
        loaded, st = oracle.rank_loaded(s, s, w.gamma, w.delta)
        n_sel = oracle.cnt(w.phi, w.N)
        xs = _cpu_bf16(rng, (tokens_per_layer, w.d))
        A = rng.random((w.T * w.B, len(loaded))).astype(np.float32)
        t0 = time.perf_counter()
        S = oracle.select(A, w.T, w.B, len(loaded), st, min(w.alpha, len(loaded)), n_sel)
        t_sel += time.perf_counter() - t0
        X = _cpu_bf16(rng, (prefill_rows, w.d))
        t0 = time.perf_counter()
        oracle.absact(Wg, Wu, loaded, X)
        t_abs += (time.perf_counter() - t0) * (w.T * w.B) / prefill_rows
        for threads in (1, n_threads):
            oracle.set_threads(threads)
            t0 = time.perf_counter()
            for t in range(tokens_per_layer):
                for b in range(w.B):
                    oracle.sparse_ffn(Wg, Wu, Wd, loaded, S[b], xs[t])
            dt = time.perf_counter() - t0
            if threads == 1:
                t_st += dt
            else:
                t_mt += dt
        oracle.set_threads(n_threads)
        n += tokens_per_layer
    per_lt_st, per_lt_mt = t_st / n, t_mt / n     # per layer-token (all B sequences)
    nl = len(layers)
    return {"single_thread_tokens_per_s": round(w.B / (w.L * per_lt_st), 4),
            "openmp_tokens_per_s": round(w.B / (w.L * per_lt_mt), 4), "cores": n_threads,
            "prefill_select_s_openmp": round(w.L * (t_abs + t_sel) / nl, 3),
            "sample": ("oracle sparse_ffn on layers %s x %d decode tokens (the first 8 and the last), "
                       "single-threaded and with %d OpenMP threads; |A| on %d prompt rows scaled to %d, "
                       "top-alpha/top-beta on the full prompt; full-stack figures extrapolated per layer "
                       "and token" % (layers, tokens_per_layer, n_threads, prefill_rows, w.T * w.B)),
            "extrapolated": True}


def cpu_baseline(w):
    c = cpu_sample(w)
    return {"value": c["openmp_tokens_per_s"], "unit": "tokens/s", "cores": c["cores"], "kind": "oracle",
            "sample": c["sample"], "extrapolated": True,
            "single_thread": {"value": c["single_thread_tokens_per_s"], "cores": 1},
            "openmp": {"value": c["openmp_tokens_per_s"], "cores": c["cores"]},
            "prefill_select_s": c["prefill_select_s_openmp"]}


def cpu_baseline_spax(w, tokens=4, seed=12):
    """The oracle's SpAx token (dense activations, tiers, tiered down) on one
    full-size layer for a few tokens, extrapolated to the stack (OpenMP)."""
    import oracle
    rng = np.random.default_rng(seed)
    Wg = _cpu_bf16(rng, (w.N, w.d), 0.02)
    Wu = _cpu_bf16(rng, (w.N, w.d), 0.02)
    Wd = _cpu_bf16(rng, (w.d, w.N), 0.02)
    codes, params = oracle.spax_encode(Wd, w.bits, w.group)
    k_top, k_mid = oracle.cnt(w.top_frac, w.N), oracle.cnt(w.mid_frac, w.N)
    xs = _cpu_bf16(rng, (tokens, w.d))
    t0 = time.perf_counter()
    for t in range(tokens):
        a = oracle.dense_act(Wg, Wu, xs[t]).astype(np.float32)
        top, mid = oracle.spax_tiers(a, k_top, k_mid)
        oracle.spax_down(a, Wd, codes, params, top, mid, w.bits, w.group)
    per = (time.perf_counter() - t0) / tokens
    return {"value": round(1.0 / (w.L * per), 4), "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "oracle dense_act + spax_tiers + spax_down on one full-size layer x %d tokens, "
                      "extrapolated to %d layers" % (tokens, w.L), "extrapolated": True}


def reference_sample(w, seed=21):
    """The reference arm's bounded sample on workload w: one decode token of the
    oracle's sparse FFN on each of layers {0, L/2, L-1}. Returns (step, layer-
    tokens per step, description, cores); step() runs one sample and returns
    its wall time in seconds."""
    import oracle
    rng = np.random.default_rng(seed)
    layers = sorted({0, w.L // 2, w.L - 1})
    data = []
    for l in layers:
        Wg = _cpu_bf16(rng, (w.N, w.d), 0.02)
        Wu = _cpu_bf16(rng, (w.N, w.d), 0.02)
        Wd = _cpu_bf16(rng, (w.d, w.N), 0.02)
        s = rng.random(w.N).astype(np.float32)
        loaded, st = oracle.rank_loaded(s, s, w.gamma, w.delta)
        n_sel = oracle.cnt(w.phi, w.N)
        S = oracle.select(rng.random((64, len(loaded))).astype(np.float32), 64, 1, len(loaded), st, 256, n_sel)
        data.append((Wg, Wu, Wd, loaded, S[0]))
    xs = _cpu_bf16(rng, (len(layers), w.d))

    def step():
        t0 = time.perf_counter()
        for (Wg, Wu, Wd, loaded, S), x in zip(data, xs):
            oracle.sparse_ffn(Wg, Wu, Wd, loaded, S, x)
        return time.perf_counter() - t0

    cores = oracle.num_threads()
    desc = ("oracle sparse_ffn, one decode token on each of layers %s of the %d-layer stack per step "
            "(%d OpenMP threads); tokens/s extrapolated to the full stack" % (layers, w.L, cores))
    return step, len(layers), desc, cores


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores, on the
    headline workload; each step is a bounded sample whose measured time is
    reported as ms_per_step, the full-step figure under its own key."""
    if rank != 0:
        return
    import oracle
    w = HEAD
    t_all = time.perf_counter()
    step, n_lt, desc, cores = reference_sample(w)
    for _ in range(args.warmup):
        step()
    times = [step() for _ in range(args.steps)]
    per_lt = statistics.median(times) / n_lt
    value = 1.0 / (w.L * per_lt)
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(statistics.mean(times) * 1e3, 3),
           "ms_per_step_note": "measured wall time of one step's bounded sample",
           "extrapolated_ms_per_step": round(1e3 * w.decode_tokens / value, 3),
           "extrapolated_note": "time the oracle would take for the step's %d decode tokens over all %d layers"
                                % (w.decode_tokens, w.L),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded generators)",
           "config": {"workload": w.name, "layers": w.L, "d": w.d, "d_ff": w.N, "gamma": w.gamma,
                      "delta": w.delta, "phi": w.phi, "alpha": w.alpha, "prompt_tokens": w.T, "batch": w.B,
                      "decode_tokens": w.decode_tokens, "n_loaded": oracle.cnt(w.gamma, w.N),
                      "n_sel": oracle.cnt(w.phi, w.N), "parallelism": "cpu"},
           "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": desc, "extrapolated": True},
           "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "wall_s": round(time.perf_counter() - t_all, 2)}
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ main GPU arm


def run_gpu(args, world, rank, local):
    import torch
    import activation_sparse_gb300 as si

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        init_dist(world, "nccl")
    w = HEAD
    stream = torch.cuda.Stream(device=dev)
    head = run_selectinfer(si, torch, dev, stream, w, args, 1234 + rank, steps=args.steps, warmup=args.warmup,
                           dec_tokens=w.decode_tokens, world=world, rank=rank, local=local, headline=True)
    clocks = head.pop("_clocks")
    step_total_s = head.pop("_step_total_s")
    t_wall = head.pop("_wall_s")
    n_loaded, _, n_sel, _ = si.si_counts(w.N, w.gamma, w.delta, w.phi)
    out = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_total_s * 1e3 / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded torch generator; shapes and distributions of the Llama3.2-3B FFN stack)",
        "config": {"workload": w.name, "layers": w.L, "d": w.d, "d_ff": w.N, "gamma": w.gamma, "delta": w.delta,
                   "phi": w.phi, "alpha": w.alpha, "prompt_tokens": w.T, "batch": w.B,
                   "decode_tokens": w.decode_tokens, "n_loaded": n_loaded, "n_sel": n_sel,
                   "parallelism": "replicas x%d" % world,
                   "l2": "inputs larger than L2: 2.11 GB of selected weights per decode token, 3.0 GB packed"},
        "hbm_gbs": head["hbm_gbs"], "decode_ms_per_token": head["ms_per_token"],
        "prefill_select_ms": head["prefill_select_ms"], "prefill_gemm_ms": head["prefill_gemm_ms"],
        "offline_ms": head["offline_ms"], "roofline": head["roofline"],
        "prefill_roofline": head["prefill_roofline"], "e2e": head["e2e"],
        "gpu_launches": head["gpu_launches_per_step"] * args.steps,
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"], "reasons": clocks["reasons"]},
        "wall_s_timed": round(t_wall, 4),
        "stack": head["stack"], "overwrite_form": head["overwrite_form"], "layer_range": head["layer_range"],
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w)
    if not args.headline_only:
        subs = {}
        for key in SUB_WORKLOADS:
            ws = synth.WORKLOADS[key]
            if ws.spax:
                r = run_spax(si, torch, dev, stream, args)
                if rank == 0 and not args.no_cpu_baseline:
                    r["cpu_baseline"] = cpu_baseline_spax(ws)
            else:
                tokens = min(ws.decode_tokens, 64)
                r = run_selectinfer(si, torch, dev, stream, ws, args, 4321 + rank, steps=3, warmup=1,
                                    dec_tokens=tokens)
                if rank == 0 and not args.no_cpu_baseline:
                    r["cpu_baseline"] = cpu_baseline(ws)
            subs[key] = r
        out["workloads"] = subs
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_profile_case(args):
    """A few launches of one kernel on one full-size layer, for ncu captures.
    Cases: decode (k_sparse_decode_b1, residual form with a plan, Llama3.2-3B
    layer, as the headline runs it), decode1b (Llama3.2-1B layer), batch8
    (k_sparse_decode_mma<16>, Qwen2.5-3B layer, 8 sequences), prefill (k_act_gemm, 1024-token
    prompt, Llama3.2-3B layer), stack (k_sparse_decode_stack, 4 Llama3.2-3B
    layers), dense (k_dense_act), tiered (k_tiered_down) and gateup
    (k_spax_gate_up, channel tiers 30 % / 30 %) on a Llama-3.1-8B layer. Prints one JSON line with the CUDA-event time per launch."""
    import torch
    import activation_sparse_gb300 as si
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    case = args.profile_case
    keep = []
    if case in ("decode", "decode1b", "prefill", "batch8", "stack"):
        w = {"decode1b": synth.WORKLOADS["llama3.2-1b"], "batch8": synth.WORKLOADS["qwen2.5-3b"]}.get(case, HEAD)
        nl = 4 if case == "stack" else 1
        layers, Ss = [], []
        n_sel = si.si_count(w.phi, w.N)
        for l in range(nl):
            Wg, Wu, Wd = gpu_weights(torch, 7, l, w.d, w.N, w.sigma, dev)
            s = torch.rand(w.N, device=dev)
            layer = si.si_pack_loaded(Wg, Wu, Wd, s, s, w.gamma, w.delta)
            X = gpu_tokens(torch, 7, 1 + l, w.T * w.B, w.d, dev)
            S = torch.empty((w.B, n_sel), dtype=torch.int32, device=dev)
            A = torch.empty((w.T * w.B, layer.n_pad), dtype=torch.float32, device=dev)
            si.si_select_dynamic(layer, X, w.T, w.B, w.alpha, w.phi, S, A)
            si.si_decode_plan(layer, S, n_sel, w.B)
            layers.append(layer)
            Ss.append(S)
            keep += [Wg, Wu, Wd, X, A]
        x = gpu_tokens(torch, 7, 2, w.B, w.d, dev)
        y = torch.zeros((w.B, w.d), dtype=torch.float32, device=dev)
        if case in ("decode", "decode1b"):
            fn = lambda: si.si_sparse_ffn_decode_residual(layers[0], Ss[0], n_sel, 1, x, y)  # noqa: E731
        elif case == "batch8":
            fn = lambda: si.si_sparse_ffn_decode(layers[0], Ss[0], n_sel, w.B, x, y)  # noqa: E731
        elif case == "prefill":
            fn = lambda: si.si_prefill_absact(layers[0], keep[3], w.T, w.B, keep[4])  # noqa: E731
        else:
            stack = si.si_stack_create(layers)
            si.si_stack_plan(stack, [S.view(-1) for S in Ss], [n_sel] * nl)
            h = torch.randn(w.d, device=dev)
            fn = lambda: si.si_sparse_ffn_decode_stack(stack, h)  # noqa: E731
    else:
        w = synth.WORKLOADS["llama3.1-8b-spax"]
        Wg, Wu, Wd = gpu_weights(torch, 7, 0, w.d, w.N, w.sigma, dev)
        enc = si.spax_encode(Wd, w.bits, w.group)
        x = gpu_tokens(torch, 7, 2, 1, w.d, dev)[0]
        a = torch.empty(w.N, dtype=torch.float32, device=dev)
        y = torch.empty(w.d, dtype=torch.float32, device=dev)
        si.spax_dense_act(Wg, Wu, x, a)
        if case == "gateup":
            gate, upe = si.spax_encode_rows(Wg, w.bits, w.group), si.spax_encode_rows(Wu, w.bits, w.group)
            keep += [gate, upe]
            fn = lambda: si.spax_gate_up(gate, upe, x, 0.3, 0.3, a)  # noqa: E731
        elif case == "dense":
            fn = lambda: si.spax_dense_act(Wg, Wu, x, a)  # noqa: E731
        else:
            fn = lambda: si.spax_tiered_down(enc, a, w.top_frac, w.mid_frac, y)  # noqa: E731
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
    print(json.dumps({"profile_case": case, "launches": args.steps, "ms_per_launch": e0.elapsed_time(e1) / args.steps,
                      "source_hash": kernel_source_hash()}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true", help="skip the other workloads' objects")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--out-dir", default=None, help="directory for the clock samples (optional)")
    ap.add_argument("--profile-case", choices=["decode", "decode1b", "batch8", "prefill", "stack", "dense", "tiered",
                                               "gateup"],
                    default=None, help="run only a few launches of one kernel (for ncu captures)")
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
