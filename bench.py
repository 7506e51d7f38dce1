#!/usr/bin/env python
"""Benchmark of the streamed NF4-LoRA training step on GB300.

Workload: the Qwen2.5-32B-shaped stack (64 layers; hidden 5120, kv 1024,
intermediate 27648; head_dim 128), 512 tokens, LoRA r 16 / alpha 32 on all
seven linears, dropout 0.1, blocks of 4 layers, one Adam step per step.
Synthetic data: random-init NF4 base (N(0, 0.02) before quantisation) and
adapters, residual-stream input N(0, 1) regenerated per step.

One step = one pass of the whole hot path: per block the NF4-LoRA linears
forward (dropout mask + down projection + dequant GEMM with the fused up
projection), the stack's pointwise ops, loss, the reverse-order backward
(for the streamed run: reload + recompute each block), Adam.

  value : linear fwd+bwd TFLOPS of the RESIDENT step (NF4 base already in
          HBM when the timed region starts; no recompute);
  e2e   : the same metric for the STREAMED step through the public API:
          the NF4 base flows from pinned host memory through the 2-slot HBM
          window inside the timed region, plus the h0 host->device copy and
          the loss device->host read each step.
The flop count is the useful linear work, 4MNK + 6Mr(K+N) per linear whose
adapters get gradients (v, o, gate, up, down) and 2MNK + 2Mr(K+N) for q and
k (forward only: they feed the replaced attention core); recompute flops
of the streamed step are not counted.

Run:  python bench.py [--steps K] [--warmup W]   (torchrun for N > 1:
independent replicas, one per GPU, no collective on the data path).
``--impl reference`` times the CPU oracle (plain C, fp64) on a bounded sample
of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "NF4-LoRA linear fwd+bwd TFLOPS (% bf16 peak); streamed 32B-shape s/step"
SHAPE_32B = dict(M=512, H=5120, KV=1024, I=27648, head_dim=128, n_layers=64)
BLOCK = 4
SHAPE_7B = dict(H=3584, KV=512, I=18944)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"],
                    bf16_sustained=p["bf16_tflops_sustained"], src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


def lin_shapes(H, KV, I):
    return [(H, H), (KV, H), (KV, H), (H, H), (I, H), (I, H), (H, I)]


def step_flops(M, H, KV, I, n_layers, r=16):
    """Useful linear flops of one training step (see module docstring)."""
    tot = 0
    for i, (N, K) in enumerate(lin_shapes(H, KV, I)):
        if i in (0, 1):
            tot += 2 * M * N * K + 2 * M * r * (K + N)
        else:
            tot += 4 * M * N * K + 6 * M * r * (K + N)
    return tot * n_layers


def nf4_bytes(H, KV, I, n_layers):
    return sum(N * K // 2 + N * K // 64 * 4 for N, K in lin_shapes(H, KV, I)) * n_layers


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        except Exception:
            pass
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["unsampled"], samples=0)
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        pw = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(mx) if mx else None, reasons=reasons, samples=len(rows),
                    power_w_max=max(pw) if pw else None)


# ------------------------------------------------------------------------------ reference arm
def oracle_sample(M_sample, H, KV, I, seed=0):
    """One layer of the workload's seven NF4-LoRA linears, forward + backward,
    on the first M_sample tokens, timed in the CPU oracle."""
    import numpy as np

    import oracle
    from weight_streaming_nf4_gb300 import synth
    oracle.build()
    prepared = []
    for li, (N, K) in enumerate(lin_shapes(H, KV, I)):
        d = synth.linear_inputs(seed, M_sample, N, K, 16, tag=f"cpu{li}")
        Wq = oracle.dequant_nf4(*oracle.quantize_nf4(d["W"]))
        mask = oracle.dropout_mask(seed, 0, 0, li, 0, 0.1, M_sample, K)
        prepared.append((d, Wq, mask))
    flops = sum(4 * M_sample * N * K + 6 * M_sample * 16 * (N + K) for N, K in lin_shapes(H, KV, I))

    def run():
        t0 = time.perf_counter()
        for d, Wq, mask in prepared:
            oracle.lora_fwd(d["x"], Wq, d["A"], d["B"], mask, 2.0 / 0.9)
            oracle.lora_bwd(d["x"], Wq, d["A"], d["B"], mask, d["dY"], 2.0 / 0.9)
        return time.perf_counter() - t0
    return run, flops, oracle.num_threads(), np


def arm_config(world):
    return {"workload": "qwen2.5-32b-shaped stack, 64 layers, seq 512, batch 1, "
                        "LoRA r16 a32 dropout 0.1, blocks of 4, Adam",
            "global_batch": world, "seq_len": SHAPE_32B["M"], "parallelism": f"replicas{world}",
            "l2": "inputs larger than L2 (17.55 GB NF4 base per step)"}


def run_reference(args, rank):
    from weight_streaming_nf4_gb300 import replicas
    if not replicas.is_reporter(rank):
        return
    M_s = 64
    run, flops, cores, _ = oracle_sample(M_s, SHAPE_32B["H"], SHAPE_32B["KV"], SHAPE_32B["I"])
    for _ in range(args.warmup):
        run()
    ts = [run() for _ in range(args.steps)]
    t = sum(ts)
    v = flops * args.steps / t / 1e12
    sample = (f"one 32B-shaped layer's 7 NF4-LoRA linears fwd+bwd on {M_s} of the 512 tokens "
              f"({flops / 1e9:.1f} GFLOP per step), plain C oracle, fp64")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": arm_config(args.gpus),
        "cpu_baseline": {"value": v, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ------------------------------------------------------------------------------ our arm
class Graphed:
    """A StackRun whose step is replayed from one captured CUDA graph (for a
    streamed run, with timing events around every block copy)."""

    def __init__(self, ops, run, lr, stream):
        l0 = ops.kernel_launches()
        self.run, self.stream = run, stream
        self.g = run.graph(lr, stream, time_copies=run.streamed)
        self.launches_per_step = ops.kernel_launches() - l0
        self.loss = run.loss

    def step(self, s, h0):
        self.g.step(s, h0, self.stream)

    def copy_times_ms(self):
        return self.g.copy_times_ms()


def make_runs(ops, StackRun, torch, cfg, dev, streamed=True, resident=True):
    """The streamed run (quantised straight into its pinned image) and the
    resident run (a device copy of the same image)."""
    def gen(layer, lin):
        g = torch.Generator(device=dev)
        g.manual_seed(1_000_003 * layer + 7919 * lin + 17)
        return g

    def wfn(layer, lin, N, K):
        return (torch.randn(N, K, generator=gen(layer, lin), device=dev) * 0.02).to(torch.bfloat16)

    def pfn(layer, lin, N, K):
        g = gen(layer, lin + 100)
        A = (torch.rand(16, K, generator=g, device=dev) * 2 - 1) / (K ** 0.5)
        B = torch.randn(N, 16, generator=g, device=dev) * 0.01
        return A, B
    stm = StackRun(cfg, BLOCK, True, wfn, pfn, device=dev) if streamed else None
    res = None
    if resident:
        res = StackRun(cfg, BLOCK, False, wfn, pfn, device=dev, image_from=stm)
    return res, stm


def time_steps(torch, dist, run, h0s, K, W, stream, e2e=None, nvtx=False, losses=None):
    """W warm-up steps, then K timed steps bracketed by barrier + sync.
    Returns (seconds of the K steps, per-step ms from events on the stream).
    losses: a device tensor [W + K] that receives every step's loss."""
    for i in range(W):
        run.step(i, h0s[i % len(h0s)])
        if losses is not None:
            losses[i:i + 1].copy_(run.loss)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    if nvtx:
        torch.cuda.nvtx.range_push("timed")
    ev[0].record(stream)
    for i in range(K):
        s = W + i
        if e2e is None:
            run.step(s, h0s[s % len(h0s)])
        else:
            host_h0, dev_h0, host_loss = e2e
            dev_h0.copy_(host_h0[s % len(host_h0)], non_blocking=True)
            run.step(s, dev_h0)
            host_loss[s].copy_(run.loss, non_blocking=True)
        if losses is not None:
            losses[s:s + 1].copy_(run.loss)
        ev[i + 1].record(stream)
    if nvtx:
        torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(K)]
    return ev[0].elapsed_time(ev[K]) / 1e3, per


def dist_ms(v):
    v = list(v)
    if not v:
        return None
    med = statistics.median(v)
    return {"median": med, "min": min(v), "max": max(v), "mean": sum(v) / len(v), "n": len(v),
            "n_above_1.2x_median": sum(1 for x in v if x > 1.2 * med)}


def streamed_breakdown(torch, gstm, h0s, first_step, n, stream, t_compute_ms, block_bytes):
    """n more streamed steps, each read back on its own: step time (events on
    the compute stream), the copy stream's busy time (the sum of its block
    copies' durations, from timing events captured in the graph) and the
    per-copy rates.  Overlap per step = (T_compute + T_copy - T_step) / T_copy
    with T_compute the resident step's median."""
    steps, busy, rates, overlap = [], [], [], []
    for i in range(n):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gstm.step(first_step + i, h0s[i % len(h0s)])
        e1.record(stream)
        e1.synchronize()
        t = e0.elapsed_time(e1)
        cp = gstm.copy_times_ms()
        tc = sum(cp)
        steps.append(t)
        busy.append(tc)
        rates += [block_bytes / (c / 1e3) / 1e9 for c in cp if c > 0]
        overlap.append(max(0.0, min(1.0, (t_compute_ms + tc - t) / tc)) if tc > 0 else None)
    ov = [o for o in overlap if o is not None]
    return {"step_ms": dist_ms(steps), "copy_busy_ms": dist_ms(busy),
            "copy_gbs": dist_ms(rates), "copies_per_step": len(cp),
            "overlap_fraction": dist_ms(ov)}


def measure_stack(ops, StackRun, torch, dist, cfg, dev, steps, warmup, e2e=True):
    """Resident and streamed steps of one stack shape, both replayed from
    CUDA graphs: timings, the streamed step's copy and overlap breakdown, the
    bitwise comparison of every step, and the runs' device footprints."""
    t0 = time.time()
    res, stm = make_runs(ops, StackRun, torch, cfg, dev)
    setup_s = time.time() - t0
    M, H = cfg.M, cfg.H
    nh0 = 4
    h0s = [torch.randn(M * H, device=dev, generator=torch.Generator(device=dev).manual_seed(s))
           for s in range(nh0)]
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.set_stream(stream)
    gres = Graphed(ops, res, 2e-4, stream)
    gstm = Graphed(ops, stm, 2e-4, stream)
    n_all = warmup + steps
    loss_res = torch.zeros(n_all, device=dev)
    loss_stm = torch.zeros(n_all, device=dev)
    # ---- resident step, replayed from one CUDA graph
    torch.cuda.reset_peak_memory_stats(dev)
    base_alloc = torch.cuda.memory_allocated(dev)
    with ClockSampler(int(os.environ.get("LOCAL_RANK", 0))) as clk:
        t_res, per_res = time_steps(torch, dist, gres, h0s, steps, warmup, stream, nvtx=True,
                                    losses=loss_res)
    clocks = clk.summary()
    # ---- streamed step through the public API with host buffers (e2e)
    host_h0 = [h.cpu().pin_memory() for h in h0s]
    dev_h0 = torch.empty(M * H, device=dev)
    host_loss = torch.zeros(n_all, 1).pin_memory()
    with ClockSampler(int(os.environ.get("LOCAL_RANK", 0))) as clk2:
        t_stm, per_stm = time_steps(torch, dist, gstm, h0s, steps, warmup, stream,
                                    e2e=(host_h0, dev_h0, host_loss) if e2e else None,
                                    losses=loss_stm)
    clocks2 = clk2.summary()
    alloc_growth = torch.cuda.max_memory_allocated(dev) - base_alloc - dev_h0.numel() * 4
    err = ops.device_error()
    # every step's loss, and after the same steps the whole optimizer state
    bitwise = {"loss_every_step": bool(torch.equal(loss_res, loss_stm))}
    for name in ("params", "grads", "adam_m", "adam_v"):
        bitwise[name] = bool(torch.equal(getattr(res, name), getattr(stm, name)))
    bitwise["all"] = all(bitwise.values())
    bitwise["steps"] = n_all
    nb = cfg.n_layers // BLOCK
    bb = res.sizes["block_bytes"]
    breakdown = streamed_breakdown(torch, gstm, h0s, n_all, 6, stream,
                                   statistics.median(per_res), bb)
    out = {
        "t_res": t_res, "t_stm": t_stm, "per_res": per_res, "per_stm": per_stm,
        "clocks": clocks, "clocks2": clocks2, "device_error_flags": err, "setup_s": setup_s,
        "bitwise": bitwise, "breakdown": breakdown, "res": res, "stm": stm, "gres": gres,
        "launches_per_step": gres.launches_per_step,
        # the two turnaround blocks are not reloaded, and a replayed step starts from
        # the window the previous step left (blocks 0 and 1)
        "h2d_w": (2 * nb - 4) * bb, "block_bytes": bb, "nb": nb,
        "alloc_growth_during_steps": int(alloc_growth),
    }
    torch.cuda.set_stream(torch.cuda.default_stream(dev))
    return out


def streaming_report(m, link_gbs, steps):
    s_res, s_stm = m["t_res"] / steps, m["t_stm"] / steps
    med_res = statistics.median(m["per_res"]) / 1e3
    med_stm = statistics.median(m["per_stm"]) / 1e3
    h2d_w = m["h2d_w"]
    bd = m["breakdown"]
    return {
        "s_per_step_streamed": s_stm, "s_per_step_resident": s_res,
        "s_per_step_streamed_median": med_stm, "s_per_step_resident_median": med_res,
        "step_ms_streamed": dist_ms(m["per_stm"]), "step_ms_resident": dist_ms(m["per_res"]),
        "slowdown": s_stm / s_res, "slowdown_median": med_stm / med_res,
        "h2d_bytes_per_step": h2d_w, "block_copies_per_step": bd["copies_per_step"],
        "h2d_link_peak_gbs": link_gbs,
        "h2d_effective_gbs": h2d_w / s_stm / 1e9,
        "h2d_effective_gbs_median_step": h2d_w / med_stm / 1e9,
        "h2d_frac_of_link": (h2d_w / s_stm / 1e9) / link_gbs,
        "h2d_frac_of_link_median_step": (h2d_w / med_stm / 1e9) / link_gbs,
        "copy_floor_s_at_link_peak": h2d_w / (link_gbs * 1e9),
        "breakdown_of_6_extra_steps": bd,
        "bitwise_streamed_eq_resident": m["bitwise"],
        "device_bytes_streamed": m["stm"].device_bytes(),
        "device_bytes_resident": m["res"].device_bytes(),
        "library_static_device_bytes": (48 << 20) + (4 << 20),
        "torch_alloc_growth_during_steps": m["alloc_growth_during_steps"],
        "pinned_host_bytes": m["nb"] * m["block_bytes"],
        "setup_s": m["setup_s"], "device_error_flags": m["device_error_flags"],
    }


def roofline_calls(ops, torch, res, cfg):
    """The dominant kernel's launches: the NF4 dequant GEMM (forward and
    input-gradient directions) on the workload's seven linear shapes of eight
    layers, weights read from the resident image (different layers back to
    back: no L2 reuse)."""
    M = cfg.M
    st = torch.cuda.current_stream()
    shapes = cfg.shapes()
    bb = res.sizes["block_bytes"]
    flops = 0
    calls = []
    for layer in range(8):
        b, li = divmod(layer, BLOCK)
        img = res.dev_weights[b * bb:(b + 1) * bb]
        for lin, (N, K) in enumerate(shapes):
            oc, oa = ops.stack_weight_offset(cfg, li, lin)
            W = ops.NF4Weight(img[oc:oc + N * K // 2].view(N, K // 2),
                              img[oa:oa + 4 * N * K // 64].view(torch.float32).view(K // 64, N), N, K)
            for tw in (False, True):
                act = torch.randn(M, N if tw else K, device=st.device).to(torch.bfloat16)
                out = torch.empty(M, K if tw else N, device=st.device, dtype=torch.bfloat16)
                ws = torch.empty(ops.nf4_matmul_workspace_size(M, N, K, tw), dtype=torch.uint8,
                                 device=st.device)
                calls.append((W, act, tw, out, ws))
                flops += 2 * M * N * K
    return calls, flops


def gemm_roofline(ops, torch, res, cfg, peak_bf16):
    """Average launch of the dominant kernel (roofline_calls), timed with CUDA
    events on the launching stream."""
    st = torch.cuda.current_stream()
    calls, flops = roofline_calls(ops, torch, res, cfg)
    for c in calls:
        ops.nf4_matmul(c[0], c[1], c[2], out=c[3], workspace=c[4])
    torch.cuda.synchronize()
    reps = 3
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        for c in calls:
            ops.nf4_matmul(c[0], c[1], c[2], out=c[3], workspace=c[4])
    e1.record(st)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / 1e3
    launches = reps * len(calls)
    achieved = flops * reps / t / 1e12
    return dict(bound="tensor", achieved=achieved, peak=peak_bf16, unit="TFLOP/s",
                frac=achieved / peak_bf16, launches=launches,
                avg_launch_us=1e6 * t / launches, flops_per_launch=flops / len(calls))


def profile_roofline(torch):
    """The roofline launches on an 8-layer resident image (a few GB): one warm
    pass, then one pass to capture (skip the first len(calls) launches)."""
    from weight_streaming_nf4_gb300 import ops
    from weight_streaming_nf4_gb300.stack import StackRun
    dev = torch.device("cuda:0")
    cfg = ops.StackCfg(**dict(SHAPE_32B, n_layers=8))
    res, _ = make_runs(ops, StackRun, torch, cfg, dev, streamed=False)
    calls, flops = roofline_calls(ops, torch, res, cfg)
    for _ in range(2):
        for c in calls:
            ops.nf4_matmul(c[0], c[1], c[2], out=c[3], workspace=c[4])
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    print(json.dumps({"profile_roofline": len(calls), "flops_per_launch": flops / len(calls)}))


def linear_7b(ops, torch, dev, M, reps=5):
    """Seven 7B-layer NF4-LoRA linears forward + backward, weights rotated over
    4 layer copies (larger than L2), two ways: one ws_lora_linear_fwd / _bwd
    call per linear, and the grouped calls a layer makes (q, k, v and gate, up
    forward together; k, v and gate, up backward together)."""
    H, KV, I = SHAPE_7B["H"], SHAPE_7B["KV"], SHAPE_7B["I"]
    shapes = lin_shapes(H, KV, I)
    copies = []
    for c in range(4):
        lins = []
        xa = torch.randn(M, H, device=dev).to(torch.bfloat16)      # q, k, v, gate, up input
        for li, (N, K) in enumerate(shapes):
            W = (torch.randn(N, K, device=dev) * 0.02).to(torch.bfloat16)
            codes, absmax = ops.quantize_nf4(W)
            del W
            A = (torch.rand(16, K, device=dev) * 2 - 1) / (K ** 0.5)
            B = torch.randn(N, 16, device=dev) * 0.01
            x = xa if li in (0, 1, 2, 4, 5) else torch.randn(M, K, device=dev).to(torch.bfloat16)
            dY = torch.randn(M, N, device=dev).to(torch.bfloat16)
            y = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
            U = torch.empty(M, 16, device=dev)
            mask = torch.empty(M, K // 32, device=dev, dtype=torch.int32)
            dX = torch.empty(M, K, device=dev, dtype=torch.float32)
            dA, dB = torch.empty_like(A), torch.empty_like(B)
            ws = torch.empty(ops.lora_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
            lins.append(dict(W=ops.NF4Weight(codes, absmax, N, K), x=x, A=A, B=B, dY=dY, y=y,
                             U=U, mask=mask, dX=dX, dA=dA, dB=dB, ws=ws,
                             key=ops.dropout_key(linear=li)))
        gws = torch.empty(max(ops.lora_group_workspace_size([H, KV, KV], M, H),
                              ops.lora_group_workspace_size([KV, KV], M, H),
                              ops.lora_group_workspace_size([H], M, H),
                              ops.lora_group_workspace_size([I, I], M, H),
                              ops.lora_group_workspace_size([H], M, I)),
                          dtype=torch.uint8, device=dev)
        copies.append((lins, gws))
    flops = sum(4 * M * N * K + 6 * M * 16 * (N + K) for N, K in shapes)

    def single(c):
        lins, _ = c
        for l in lins:
            ops.lora_linear_fwd(l["W"], l["x"], l["A"], l["B"], l["key"], y=l["y"], U=l["U"],
                                mask=l["mask"], workspace=l["ws"])
        for l in lins:
            ops.lora_linear_bwd(l["W"], l["x"], l["A"], l["B"], l["key"], l["U"], l["mask"],
                                l["dY"], dX=l["dX"], dA=l["dA"], dB=l["dB"], workspace=l["ws"])

    def grouped(c):
        lins, gws = c

        def fwd(ids):
            ls = [lins[i] for i in ids]
            ops.lora_linear_fwd_group([l["W"] for l in ls], ls[0]["x"], [l["A"] for l in ls],
                                      [l["B"] for l in ls], [l["key"] for l in ls],
                                      ys=[l["y"] for l in ls], Us=[l["U"] for l in ls],
                                      masks=[l["mask"] for l in ls], workspace=gws)

        def bwd(ids):
            ls = [lins[i] for i in ids]
            ops.lora_linear_bwd_group([l["W"] for l in ls], ls[0]["x"], [l["A"] for l in ls],
                                      [l["B"] for l in ls], [l["key"] for l in ls],
                                      [l["U"] for l in ls], [l["mask"] for l in ls],
                                      [l["dY"] for l in ls], dX=ls[0]["dX"],
                                      dAs=[l["dA"] for l in ls], dBs=[l["dB"] for l in ls],
                                      workspace=gws)
        fwd((0, 1, 2))
        fwd((3,))
        fwd((4, 5))
        fwd((6,))
        bwd((6,))
        bwd((4, 5))
        bwd((3,))
        bwd((1, 2))
        bwd((0,))

    out = {}
    for name, one in (("per_linear", single), ("grouped", grouped)):
        for c in copies:
            one(c)
        torch.cuda.synchronize()
        st = torch.cuda.current_stream()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for r in range(reps):
            for c in copies:
                one(c)
        e1.record(st)
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) / 1e3
        n = reps * len(copies)
        out[name] = dict(tflops=flops * n / t / 1e12, ms_per_layer=1e3 * t / n)
    out["flops_per_layer"] = flops
    out["tflops"] = max(out["per_linear"]["tflops"], out["grouped"]["tflops"])
    return out


def profile_gemm(torch, which):
    from weight_streaming_nf4_gb300 import ops
    dev = torch.device("cuda:0")
    H, KV, I = SHAPE_32B["H"], SHAPE_32B["KV"], SHAPE_32B["I"]
    N, K = dict(gate=(I, H), down=(H, I), o=(H, H))[which]
    M = SHAPE_32B["M"]
    W = (torch.randn(N, K, device=dev) * 0.02).to(torch.bfloat16)
    codes, absmax = ops.quantize_nf4(W)
    Wn = ops.NF4Weight(codes, absmax, N, K)
    x = torch.randn(M, K, device=dev).to(torch.bfloat16)
    dY = torch.randn(M, N, device=dev).to(torch.bfloat16)
    for _ in range(2):
        ops.nf4_matmul(Wn, x)
        ops.nf4_matmul(Wn, dY, transpose_w=True)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    print(json.dumps({"profile_gemm": which, "M": M, "N": N, "K": K}))


def profile_lora(torch, which):
    """One 32B-shaped NF4-LoRA linear, ws_lora_linear_fwd then _bwd, three
    times at M=512: the skinny products, weight gradients and dequant GEMM
    of one linear (a few hundred MB on the device), for an ncu capture of the
    LoRA-side kernels."""
    from weight_streaming_nf4_gb300 import ops
    dev = torch.device("cuda:0")
    H, KV, I = SHAPE_32B["H"], SHAPE_32B["KV"], SHAPE_32B["I"]
    N, K = dict(gate=(I, H), down=(H, I), o=(H, H))[which]
    M = SHAPE_32B["M"]
    W = (torch.randn(N, K, device=dev) * 0.02).to(torch.bfloat16)
    codes, absmax = ops.quantize_nf4(W)
    Wn = ops.NF4Weight(codes, absmax, N, K)
    A = (torch.rand(16, K, device=dev) * 2 - 1) / (K ** 0.5)
    B = torch.randn(N, 16, device=dev) * 0.01
    x = torch.randn(M, K, device=dev).to(torch.bfloat16)
    dY = torch.randn(M, N, device=dev).to(torch.bfloat16)
    key = ops.dropout_key(linear=6)
    for _ in range(3):
        y, U, mask = ops.lora_linear_fwd(Wn, x, A, B, key)
        ops.lora_linear_bwd(Wn, x, A, B, key, U, mask, dY)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    print(json.dumps({"profile_lora": which, "M": M, "N": N, "K": K}))


def attn_inputs(torch, dev, S, nh, nkv, d):
    g = torch.Generator(device=dev)
    g.manual_seed(4242)
    mk = lambda w: torch.randn(S, w * d, generator=g, device=dev).to(torch.bfloat16)
    return mk(nh), mk(nkv), mk(nkv), mk(nh)


def attention_32b(ops, torch, dev, reps=50):
    """The attention core at the 32B layer's shape (one sequence of 512 tokens,
    40 query heads over 8 kv heads, head_dim 128): forward and backward timed
    with CUDA events over `reps` back-to-back calls each.  Algorithmic flops:
    the causal half of the two forward products (QK^T, PV) and of the five
    backward ones (QK^T, dO V^T, dQ, dK, dV)."""
    S, nh, nkv, d = SHAPE_32B["M"], 40, 8, 128
    q, k, v, dO = attn_inputs(torch, dev, S, nh, nkv, d)
    ws = torch.empty(ops.attention_workspace_size(S, nh, d), dtype=torch.uint8, device=dev)
    o, o32, lse = ops.attention_fwd(q, k, v, 1, d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = torch.cuda.current_stream()
    for _ in range(5):
        ops.attention_fwd(q, k, v, 1, d, o=o, o32=o32, lse=lse)
        ops.attention_bwd(q, k, v, o32, lse, dO, 1, d, dq, dk, dv, ws)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    ev[0].record(st)
    for _ in range(reps):
        ops.attention_fwd(q, k, v, 1, d, o=o, o32=o32, lse=lse)
    ev[1].record(st)
    for _ in range(reps):
        ops.attention_bwd(q, k, v, o32, lse, dO, 1, d, dq, dk, dv, ws)
    ev[2].record(st)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    tf = ev[0].elapsed_time(ev[1]) / reps * 1e-3
    tb = ev[1].elapsed_time(ev[2]) / reps * 1e-3
    f_fwd = 2 * 2.0 * (S * (S + 1) / 2) * d * nh
    return {"workload": "causal attention, 1 x 512 tokens, 40 query heads over 8 kv heads, "
                        "head_dim 128 (the 32B layer)",
            "fwd_us": tf * 1e6, "bwd_us": tb * 1e6,
            "fwd_tflops": f_fwd / tf / 1e12, "bwd_tflops": 2.5 * f_fwd / tb / 1e12,
            "per_step_ms_64_layers": 64 * (tf + tb) * 1e3,
            "launches": {"fwd": 1, "bwd": 3}}


def attention_stack_32b(ops, StackRun, torch, dev, steps):
    """The resident 32B-shaped step with the causal attention core in place of
    repeat(v): ms per step (graph replay, median of `steps`)."""
    cfg = ops.StackCfg(**SHAPE_32B, attn=ops.ATTN_CAUSAL)
    res, _ = make_runs(ops, StackRun, torch, cfg, dev, streamed=False)
    st = torch.cuda.Stream(device=dev)
    g = Graphed(ops, res, 2e-4, st)
    h0 = torch.randn(cfg.M * cfg.H, device=dev)
    with torch.cuda.stream(st):
        _, per = time_steps(torch, None, g, [h0], steps, 3, st)
    assert ops.device_error() == 0
    loss = float(res.loss.item())
    del g, res
    return {"workload": "qwen2.5-32b-shaped stack, 64 layers, seq 512, causal attention core, "
                        "resident", "ms_per_step_median": statistics.median(per),
            "steps": steps, "loss_finite": bool(loss == loss)}


def profile_attention(torch):
    """The attention core at the 32B layer's shape, forward and backward three
    times (a few MB on the device), for an ncu capture of its kernels."""
    from weight_streaming_nf4_gb300 import ops
    dev = torch.device("cuda:0")
    S, nh, nkv, d = SHAPE_32B["M"], 40, 8, 128
    q, k, v, dO = attn_inputs(torch, dev, S, nh, nkv, d)
    for _ in range(3):
        o, o32, lse = ops.attention_fwd(q, k, v, 1, d)
        ops.attention_bwd(q, k, v, o32, lse, dO, 1, d)
    torch.cuda.synchronize()
    assert ops.device_error() == 0
    print(json.dumps({"profile_attention": "32b layer", "S": S, "nh": nh, "nkv": nkv, "d": d}))


def h2d_peak(torch, dev):
    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8).pin_memory()
    dst = torch.empty(n, dtype=torch.uint8, device=dev)
    st = torch.cuda.Stream(device=dev)
    best = 0.0
    for _ in range(6):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        with torch.cuda.stream(st):
            dst.copy_(src, non_blocking=True)
        e1.record(st)
        e1.synchronize()
        best = max(best, n / (e0.elapsed_time(e1) / 1e3) / 1e9)
    return best


def profile_link(torch):
    """Host-link measurements: pinned host -> HBM copies of 32B-block size
    (one cudaMemcpyAsync each, or cut into pieces, or split over two
    streams), per-copy rates, the same copies beside a tensor-core load, and
    the distribution over ~20 s of back-to-back copies."""
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    bb, nb = 1097072640, 16
    host = torch.empty(nb * bb, dtype=torch.uint8, pin_memory=True)
    host[::4096] = 1
    win = torch.empty(2 * bb, dtype=torch.uint8, device=dev)
    cs = torch.cuda.Stream(device=dev)

    def copies(n, piece=None):
        evs = []
        with torch.cuda.stream(cs):
            for i in range(n):
                src = host[(i % nb) * bb:((i % nb) + 1) * bb]
                dst = win[(i % 2) * bb:((i % 2) + 1) * bb]
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(cs)
                if piece is None:
                    dst.copy_(src, non_blocking=True)
                else:
                    for o in range(0, bb, piece):
                        dst[o:o + piece].copy_(src[o:o + piece], non_blocking=True)
                e1.record(cs)
                evs.append((e0, e1))
        torch.cuda.synchronize()
        return [bb / (a.elapsed_time(b) / 1e3) / 1e9 for a, b in evs]

    def d(g):
        g = sorted(g)
        return {"n": len(g), "min": round(g[0], 1), "median": round(statistics.median(g), 1),
                "max": round(g[-1], 1), "below_0.8x_median": sum(1 for x in g if x < 0.8 * statistics.median(g))}
    copies(4)
    out = {"block_bytes": bb, "whole_block": d(copies(48)), "pieces_128MB": d(copies(32, 128 << 20)),
           "pieces_32MB": d(copies(32, 32 << 20))}
    a = torch.randn(8192, 8192, device=dev, dtype=torch.bfloat16)
    b = torch.randn(8192, 8192, device=dev, dtype=torch.bfloat16)
    ms = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(ms):
        for _ in range(400):
            a @ b
    out["beside_bf16_matmul"] = d(copies(24))
    torch.cuda.synchronize()
    t_end = time.time() + 20
    long = []
    while time.time() < t_end:
        long += copies(16)
    out["back_to_back_20s"] = d(long)
    hist = {}
    for g in long:
        k = int(g // 20) * 20
        hist[k] = hist.get(k, 0) + 1
    out["back_to_back_20s_histogram_gbs_bins_of_20"] = dict(sorted(hist.items()))
    print(json.dumps({"profile_link": out}))


def traffic_counters():
    """Per-launch DRAM traffic of the dominant kernel from the committed ncu
    summary, valid only while the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "nf4_gemm_qwen32b_m512.txt")
    src = os.path.join(ROOT, "weight_streaming_nf4_gb300", "csrc", "nf4_gemm.cu")
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        kv = {}
        for line in open(path):
            if "=" in line and line.startswith("bench:"):
                k, v = line[len("bench:"):].strip().split("=", 1)
                kv[k.strip()] = v.strip()
        if kv.get("source_sha256_16") == sha:
            return float(kv["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


SHAPE_72B = dict(M=512, H=8192, KV=1024, I=29568, head_dim=128, n_layers=80)


def host_mem_available():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except Exception:
        pass
    return None


def release_host_cache(torch):
    torch.cuda.empty_cache()
    try:
        torch._C._host_emptyCache()
    except Exception:
        pass


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="skip the 7B and 72B sub-benchmarks")
    ap.add_argument("--no-72b", action="store_true", help="skip the 72B-shaped streamed run")
    ap.add_argument("--no-bf16", action="store_true", help="skip the bf16-base 32B-shaped run")
    ap.add_argument("--profile-step", action="store_true",
                    help="only the resident run: W warm-up steps and one step inside the NVTX "
                         "range 'timed'; for an ncu launch list of one step")
    ap.add_argument("--profile-roofline", action="store_true",
                    help="only launch the roofline's dequant GEMM calls twice on an 8-layer "
                         "image; for an ncu capture of their DRAM traffic")
    ap.add_argument("--profile-lora", choices=["gate", "down", "o"], default=None,
                    help="only run ws_lora_linear_fwd + _bwd three times on one 32B linear shape "
                         "at M=512; for an ncu capture of the LoRA-side kernels")
    ap.add_argument("--profile-link", action="store_true",
                    help="only measure pinned host -> HBM copies (block-sized, pieces, beside a "
                         "matmul, 20 s back to back) and print their rate distributions")
    ap.add_argument("--no-attn", action="store_true",
                    help="skip the attention-core measurements (kernels and 32B resident step)")
    ap.add_argument("--profile-attention", action="store_true",
                    help="only run the attention core fwd + bwd three times at the 32B layer's "
                         "shape; for an ncu capture of its kernels")
    ap.add_argument("--profile-gemm", choices=["gate", "down", "o"], default=None,
                    help="only launch the dequant GEMM (forward + input gradient) twice on one "
                         "32B linear shape at M=512; for an ncu capture of that kernel")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    args.warmup = max(args.warmup, 3)

    import torch
    if args.profile_gemm:
        profile_gemm(torch, args.profile_gemm)
        return
    if args.profile_lora:
        profile_lora(torch, args.profile_lora)
        return
    if args.profile_roofline:
        profile_roofline(torch)
        return
    if args.profile_link:
        profile_link(torch)
        return
    if args.profile_attention:
        profile_attention(torch)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from weight_streaming_nf4_gb300 import ops, replicas
    from weight_streaming_nf4_gb300.stack import StackRun
    pk = peaks()

    cfg = ops.StackCfg(**SHAPE_32B)
    M, H = cfg.M, cfg.H
    flops = step_flops(M, H, cfg.KV, cfg.I, cfg.n_layers)
    if args.profile_step:
        res, _ = make_runs(ops, StackRun, torch, cfg, dev, streamed=False)
        h0 = torch.randn(M * H, device=dev)
        time_steps(torch, None, res, [h0], 1, args.warmup, torch.cuda.current_stream(), nvtx=True)
        assert ops.device_error() == 0
        print(json.dumps({"profile_step": "resident", "launches": ops.kernel_launches()}))
        return
    m = measure_stack(ops, StackRun, torch, dist, cfg, dev, args.steps, args.warmup)
    t_res = replicas.max_over_ranks(m["t_res"], dist, dev)
    t_stm = replicas.max_over_ranks(m["t_stm"], dist, dev)
    value = replicas.whole_job_rate(flops, args.steps, world, t_res) / 1e12
    e2e_val = replicas.whole_job_rate(flops, args.steps, world, t_stm) / 1e12
    h2d_bytes = m["h2d_w"] + M * H * 4

    extra = {}
    if rank == 0:
        res = m["res"]
        roof = gemm_roofline(ops, torch, res, cfg, pk["bf16"])
        roof["traffic"] = traffic_counters()
        link = h2d_peak(torch, dev)
        extra["roofline"] = {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac",
                                                   "traffic")}
        extra["roofline"]["kernel"] = ("k_nf4_gemm (fwd + input-gradient), the 7 linear shapes "
                                       "of 8 layers, M=512")
        extra["roofline"]["peak_kind"] = ("bf16 dense burst, " + pk["src"])
        extra["roofline"]["avg_launch_us"] = roof["avg_launch_us"]
        extra["streaming"] = streaming_report(m, link, args.steps)
        # the eager resident step (one launch per kernel), for comparison with the graph replay
        t_eager, _ = time_steps(torch, None, res, [torch.zeros(M * H, device=dev)], 2, 1,
                                torch.cuda.current_stream())
        extra["streaming"]["s_per_step_resident_eager"] = t_eager / 2
        if not args.quick:
            extra["linear_7b"] = {f"M{mm}": linear_7b(ops, torch, dev, mm) for mm in (512, 2048)}
        if not args.no_attn:
            extra["attention_32b"] = attention_32b(ops, torch, dev)
        if world == 1 and not args.no_cpu_baseline:
            run, cflops, cores, _ = oracle_sample(256, H, cfg.KV, cfg.I)
            tc = run()
            extra["cpu_baseline"] = {
                "value": cflops / tc / 1e12, "unit": "TFLOPS", "cores": cores, "kind": "oracle",
                "sample": (f"one 32B-shaped layer's 7 NF4-LoRA linears fwd+bwd on 256 of 512 tokens "
                           f"({cflops / 1e9:.1f} GFLOP, {tc:.1f} s), plain C oracle fp64")}
    out = None
    if rank == 0:
        out = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t_res / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (random-init NF4 base and adapters, N(0,1) residual input)",
            "config": arm_config(world),
            "pct_bf16_peak": 100.0 * value / world / pk["bf16_sustained"],
            "e2e": {"value": e2e_val, "unit": "TFLOPS", "h2d_bytes_per_step": h2d_bytes,
                    "d2h_bytes_per_step": 4, "s_per_step": t_stm / args.steps,
                    "s_per_step_median": statistics.median(m["per_stm"]) / 1e3},
            "gpu_launches": int(m["launches_per_step"] * args.steps),
            "clocks": m["clocks"], "clocks_streamed": m["clocks2"],
            "device_error_flags": m["device_error_flags"], "setup_s": m["setup_s"],
        }
        out.update(extra)
    # ---- the 72B-shaped stack, streamed and resident (one GPU only)
    if rank == 0:
        del m, res
    if rank == 0 and world == 1 and not args.quick and not args.no_attn:
        out["attention_32b"]["stack_resident"] = attention_stack_32b(
            ops, StackRun, torch, dev, min(max(args.steps, 3), 10))
    if rank == 0 and world == 1 and not args.quick and not args.no_72b:
        release_host_cache(torch)
        cfg72 = ops.StackCfg(**SHAPE_72B)
        need = nf4_bytes(cfg72.H, cfg72.KV, cfg72.I, cfg72.n_layers)
        avail = host_mem_available()
        if avail is not None and avail < need + (16 << 30):
            out["qwen72b"] = {"skipped": f"host memory available {avail} < pinned image {need} + 16 GiB"}
        else:
            k72 = min(args.steps, 5)
            m72 = measure_stack(ops, StackRun, torch, None, cfg72, dev, k72, 3)
            rep = streaming_report(m72, extra["streaming"]["h2d_link_peak_gbs"], k72)
            f72 = step_flops(cfg72.M, cfg72.H, cfg72.KV, cfg72.I, cfg72.n_layers)
            rep["workload"] = ("qwen2.5-72b-shaped stack, 80 layers, H 8192, kv 1024, I 29568, "
                               "seq 512, blocks of 4, 2-slot window")
            rep["steps"] = k72
            rep["tflops_resident"] = f72 * k72 / m72["t_res"] / 1e12
            rep["tflops_streamed"] = f72 * k72 / m72["t_stm"] / 1e12
            rep["host_mem_available_bytes"] = avail
            out["qwen72b"] = rep
            del m72
            release_host_cache(torch)
    # ---- the 32B-shaped stack with a bf16 base (the pages' bf16 streaming mode)
    if rank == 0 and world == 1 and not args.quick and not args.no_bf16:
        release_host_cache(torch)
        cfgb = ops.StackCfg(**SHAPE_32B, base=ops.BASE_BF16)
        need = 2 * sum(N * K for N, K in lin_shapes(cfgb.H, cfgb.KV, cfgb.I)) * cfgb.n_layers
        avail = host_mem_available()
        if avail is not None and avail < need + (16 << 30):
            out["bf16_base_32b"] = {"skipped": f"host memory available {avail} < pinned image {need} + 16 GiB"}
        else:
            kb = min(args.steps, 3)
            mb = measure_stack(ops, StackRun, torch, None, cfgb, dev, kb, 3)
            rep = streaming_report(mb, out["streaming"]["h2d_link_peak_gbs"], kb)
            rep["workload"] = ("qwen2.5-32b-shaped stack with a bf16 base (2 bytes per weight), "
                               "64 layers, seq 512, blocks of 4, 2-slot window")
            rep["steps"] = kb
            rep["tflops_resident"] = flops * kb / mb["t_res"] / 1e12
            rep["tflops_streamed"] = flops * kb / mb["t_stm"] / 1e12
            out["bf16_base_32b"] = rep
            del mb
            release_host_cache(torch)
    if rank == 0:
        print(json.dumps(out))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
