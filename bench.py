"""Benchmark: block-diffusion attention, forward + backward, on GB300.

One step = one forward and one backward pass of attention under the
block-diffusion mask over one batch of the workload, through the C ABI of
libdfa (device-resident inputs).  Throughput counts visible (query, key)
pairs only: 4 * pairs * headdim * heads FLOPs per sample forward, 2.5x that
backward ("Fast Diffusion Attention", section "The right yardstick").

Printed on one JSON line (rank 0): the headline TFLOPS, the end-to-end
number through the public API with host buffers, the roofline of the
dominant kernel, the causal yardstick (the same kernels on the 2B halves of
length n) and the oracle timed on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload small]
    python bench.py --impl reference   # the float64 CPU oracle as the reference arm
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_diffusion_masked_gb300 import inputs  # noqa: E402

METRIC = "visible-pair TFLOPS fwd+bwd on 1 GB300; % of BF16 peak; × vs causal yardstick"


# ------------------------------------------------------------------ counting

def visible_pairs_per_sample(n, bs):
    """Visible pairs of one [noisy | clean] sample: each half holds, for every
    row r, min(n, (r // bs + 1) * bs) pairs ("The right yardstick")."""
    bs = min(bs, n)
    r = np.arange(n, dtype=np.int64)
    return int(2 * np.minimum(n, (r // bs + 1) * bs).sum())


def flops(w: inputs.Workload):
    pairs = visible_pairs_per_sample(w.n, w.block_size) * w.batch
    fwd = 4.0 * pairs * w.headdim * w.heads
    return fwd, 2.5 * fwd


def causal_flops(w: inputs.Workload):
    pairs = 2 * w.batch * w.n * (w.n + 1) // 2
    fwd = 4.0 * pairs * w.headdim * w.heads
    return fwd, 2.5 * fwd


def max_over_ranks(values, device=None):
    """Element-wise maximum of per-rank timings (a no-op on one rank)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_tflops(flop_per_rank_step, ms_per_step, world):
    """Whole-job throughput: every rank processes its own workload (weak scaling)."""
    return world * flop_per_rank_step / (ms_per_step * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": d.get("bf16_tflops", 1900.0),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", 1700.0),
                "hbm_gbs": d.get("hbm_gbs", 6800.0), "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            import tempfile

            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, x in enumerate(r)
                          if x.lower() == "active"})
        loaded = [r[0] for r in rows if r[0] > 0.5 * r[1]] or [r[0] for r in rows]
        return {"sm_mhz": float(np.median(loaded)), "sm_max_mhz": rows[0][1],
                "samples": len(rows), "reasons": reasons}


# ------------------------------------------------------------------ CPU baseline

def cpu_baseline(w: inputs.Workload, budget_s=12.0, max_heads=None):
    """The float64 oracle on the host cores over a bounded sample of heads."""
    import oracle

    q, k, v, do = inputs.make_workload_inputs(w)
    qn, kn, vn, don = (t.float().double().numpy() for t in (q, k, v, do))
    fwd_pairs = visible_pairs_per_sample(w.n, w.block_size)
    per_head_flops = 3.5 * 4.0 * fwd_pairs * w.headdim
    heads = [(b, h) for b in range(w.batch) for h in range(w.heads)]
    if max_heads:
        heads = heads[:max_heads]
    t0 = time.perf_counter()
    done = 0
    for bh in heads:
        oracle.diffusion_forward(qn, kn, vn, w.block_size, heads=[bh])
        oracle.diffusion_backward(qn, kn, vn, don, w.block_size, heads=[bh])
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": done * per_head_flops / dt / 1e12, "unit": "TFLOPS",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"{done} of {len(heads)} (batch, head) pairs of workload '{w.name}', "
                      f"forward + backward, float64 NumPy (BLAS default threads), {dt:.1f} s"}


# ------------------------------------------------------------------ GPU arm

# DRAM traffic (read + write bytes) per launch of the dominant kernel from
# one ncu capture (profiles/dfa_bwd2_kernel_small_b8_n1024_h16_d128_bs16.md),
# keyed by workload and kernel; any other pair reports null.
NCU_TRAFFIC = {("small", "dfa_bwd2_kernel<128>"): 803.4e6}


def run_gpu(args, w, rank, world):
    import torch

    from block_diffusion_masked_gb300 import binding

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    binding.lib()
    stream = torch.cuda.current_stream(dev)
    q, k, v, do = (t.to(dev) for t in inputs.make_workload_inputs(w))
    B, L, H, d = q.shape
    n = L // 2
    out = torch.empty_like(q)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dq_acc = torch.empty(q.shape, dtype=torch.float32, device=dev)
    delta = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    # causal yardstick buffers on the (2B, n) view
    qc, kc, vc, doc = (t.view(2 * B, n, H, d) for t in (q, k, v, do))
    outc = torch.empty_like(qc)
    lsec = torch.empty((2 * B, H, n), dtype=torch.float32, device=dev)
    dqc, dkc, dvc = torch.empty_like(qc), torch.empty_like(qc), torch.empty_like(qc)

    def diff_step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        # the forward launch also zeroes the dq accumulator
        binding.dfa_fwd_main(q, k, v, out, lse, dq_acc, w.block_size)
        if ev is not None:
            ev[1].record(stream)
        binding.dfa_bwd_preprocess(out, do, delta, None)
        if ev is not None:
            ev[2].record(stream)
        binding.dfa_bwd_main(q, k, v, do, lse, delta, dq_acc, dk, dv, w.block_size)
        if ev is not None:
            ev[3].record(stream)
        binding.dfa_bwd_dq_convert(dq_acc, dq)
        if ev is not None:
            ev[4].record(stream)

    def causal_step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        binding.dfa_fwd_main(q, k, v, outc.view(B, L, H, d), lsec, dq_acc, 1,
                             mode=binding.MODE_CAUSAL)
        if ev is not None:
            ev[1].record(stream)
        binding.dfa_bwd_preprocess(outc.view(B, L, H, d), do, delta, None)
        if ev is not None:
            ev[2].record(stream)
        binding.dfa_bwd_main(q, k, v, do, lsec, delta, dq_acc, dkc.view(B, L, H, d),
                             dvc.view(B, L, H, d), 1, mode=binding.MODE_CAUSAL)
        if ev is not None:
            ev[3].record(stream)
        binding.dfa_bwd_dq_convert(dq_acc, dqc.view(B, L, H, d))
        if ev is not None:
            ev[4].record(stream)

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(step, K):
        # K steps back to back, events only around the whole region: an event
        # between two launches would stop the second from being launched
        # while the first is still running (chained launches).
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        start.record(stream)
        for _ in range(K):
            step()
        end.record(stream)
        barrier()
        return start.elapsed_time(end)

    def per_kernel(step, K):
        # A separate pass with events between the launches: each kernel's
        # own duration (launch gaps included, overlap excluded).
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
        barrier()
        for i in range(K):
            step(evs[i])
        barrier()
        parts = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(4)] for e in evs])
        return parts.mean(axis=0)

    for _ in range(args.warmup):
        diff_step()
        causal_step()
    torch.cuda.synchronize(dev)
    if binding.dfa_status() != 0:
        raise RuntimeError("device status set during warm-up")

    with ClockSampler(dev.index) as clk:
        t_ms = timed(diff_step, args.steps)
    clocks = clk.summary()
    tc_ms = timed(causal_step, args.steps)
    parts = per_kernel(diff_step, args.steps)
    parts_c = per_kernel(causal_step, args.steps)
    if binding.dfa_status() != 0:
        raise RuntimeError("device status set during the timed region")

    t_ms, tc_ms = max_over_ranks([t_ms, tc_ms], dev)

    f_fwd, f_bwd = flops(w)
    c_fwd, c_bwd = causal_flops(w)
    ms_step = t_ms / args.steps
    value = job_tflops(f_fwd + f_bwd, ms_step, world)
    causal_value = job_tflops(c_fwd + c_bwd, tc_ms / args.steps, world)
    fwd_ms, pre_ms, main_ms, conv_ms = parts.tolist()
    peaks = measured_peaks()

    # e2e: public API with host buffers, copies inside the timed region.
    # Every step copies its q/k/v/dout from pinned host memory and its
    # out/dq/dk/dv/lse back; the copies run on their own streams (one per
    # direction) and overlap the neighbouring steps' compute, as in a training
    # loop that stages its next batch, with two device buffer sets.
    host_in = [t.cpu().pin_memory() for t in inputs.make_workload_inputs(w)]
    host_out = [torch.empty(q.shape, dtype=torch.bfloat16).pin_memory() for _ in range(4)]
    host_lse = torch.empty((B, H, L), dtype=torch.float32).pin_memory()
    sets = []
    for _ in range(2):
        sets.append({"in": [torch.empty_like(q) for _ in range(4)],
                     "out": torch.empty_like(q), "lse": torch.empty_like(lse),
                     "grads": [torch.empty_like(q) for _ in range(3)]})
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def issue_h2d(i):
        b = i % 2
        with torch.cuda.stream(h2d_s):
            if i >= 2:
                h2d_s.wait_event(ev_done[b])  # step i-2 has finished reading set b
            for hbuf, dbuf in zip(host_in, sets[b]["in"]):
                dbuf.copy_(hbuf, non_blocking=True)
            ev_in[b].record(h2d_s)

    def e2e_run(steps, start_event=None):
        if start_event is not None:
            h2d_s.wait_event(start_event)
        issue_h2d(0)
        for i in range(steps):
            b = i % 2
            st = sets[b]
            if i + 1 < steps:
                issue_h2d(i + 1)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # step i-2's results have left set b
            o, l = binding.dfa_forward(st["in"][0], st["in"][1], st["in"][2], w.block_size,
                                       out=st["out"], lse=st["lse"])
            g = binding.dfa_backward(st["in"][0], st["in"][1], st["in"][2], o, st["in"][3], l,
                                     w.block_size, dq=st["grads"][0], dk=st["grads"][1],
                                     dv=st["grads"][2])
            ev_done[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_done[b])
                for hbuf, dbuf in zip(host_out, (o,) + tuple(g)):
                    hbuf.copy_(dbuf, non_blocking=True)
                host_lse.copy_(l, non_blocking=True)
                ev_out[b].record(d2h_s)
        stream.wait_event(ev_out[(steps - 1) % 2])

    e2e_run(max(1, args.warmup))
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    e2e_run(args.steps, start_event=e0)
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1)], dev)[0]
    tensor_bytes = q.numel() * 2
    e2e = {"value": job_tflops(f_fwd + f_bwd, e2e_ms / args.steps, world),
           "unit": "TFLOPS", "h2d_bytes_per_step": 4 * tensor_bytes,
           "d2h_bytes_per_step": 4 * tensor_bytes + host_lse.numel() * 4}

    # Optional context: the vendor library's causal attention on the same halves.
    sdpa = None
    if args.sdpa:
        try:
            sdpa = (c_fwd + c_bwd) / (sdpa_causal(qc, kc, vc, doc, args.warmup, args.steps)
                                      * 1e-3) / 1e12
        except Exception as exc:  # context only
            sdpa = f"unavailable: {exc}"

    # kernel names as the library launches them for this head dimension
    fwd_name = "dfa_fwd_kernel<256>" if d == 256 else f"dfa_fwd2_kernel<{d}>"
    bwd_name = "dfa_bwd_kernel<64>" if d == 64 else f"dfa_bwd2_kernel<{d}>"
    dominant = max(((fwd_name, fwd_ms, f_fwd), (bwd_name, main_ms, f_bwd)), key=lambda x: x[1])
    achieved = dominant[2] / (dominant[1] * 1e-3) / 1e12
    res = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: i.i.d. N(0,1)*std bf16 q/k/v/dout from a seeded CPU generator",
        "config": {"workload": w.name, "batch": w.batch, "n": w.n, "seqlen": 2 * w.n,
                   "heads": w.heads, "headdim": w.headdim, "block_size": w.block_size,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2 ({4 * tensor_bytes / 1e6:.0f} MB of q/k/v/dout)"},
        "pct_of_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
        "fwd_tflops": f_fwd / (fwd_ms * 1e-3) / 1e12,
        "bwd_tflops": f_bwd / ((pre_ms + main_ms + conv_ms) * 1e-3) / 1e12,
        "kernel_ms": {"fwd": fwd_ms, "bwd_preprocess": pre_ms, "bwd_main": main_ms,
                      "dq_convert": conv_ms},
        "yardstick": {"what": "same kernels, causal attention on the 2B halves of length n",
                      "value": causal_value, "unit": "TFLOPS",
                      "ratio": value / causal_value,
                      "kernel_ms": dict(zip(("fwd", "bwd_preprocess", "bwd_main", "dq_convert"),
                                            parts_c.tolist()))},
        "gpu_launches": 4 * args.steps,
        "e2e": e2e,
        "roofline": {"kernel": dominant[0], "bound": "tensor", "achieved": achieved,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"],
                     "peak_source": peaks["source"] + " bf16 burst (cuBLAS 8192^3)",
                     "traffic": NCU_TRAFFIC.get((w.name, dominant[0])),
                     "traffic_unit": "bytes per launch (ncu dram read + write)"},
        "clocks": clocks,
    }
    if sdpa is not None:
        res["sdpa_causal_tflops"] = sdpa
    return res


def sdpa_causal(qc, kc, vc, doc, warmup, steps):
    """ms per fwd+bwd step of torch SDPA causal on the (2B, H, n, d) halves."""
    import torch

    qt, kt, vt = (t.transpose(1, 2).contiguous().requires_grad_(True) for t in (qc, kc, vc))
    dot = doc.transpose(1, 2).contiguous()

    def step():
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True)
        o.backward(dot)

    for _ in range(warmup):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_reference(args, w, rank, world):
    """The reference arm: the float64 oracle on the host cores, bounded steps."""
    f_fwd, f_bwd = flops(w)
    per_step = []
    base = None
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(w, budget_s=args.ref_step_s, max_heads=1)
        if i >= args.warmup:
            per_step.append(r["value"])
            base = r
    value = float(np.median(per_step))
    base = dict(base)
    base["value"] = value
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "n": w.n, "seqlen": 2 * w.n,
                       "heads": w.heads, "headdim": w.headdim, "block_size": w.block_size},
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# Half lengths of the packed varlen batch: a mix of sample lengths with the
# rows of the workload it stands beside (8 x 2048 rows for "small").
VARLEN_HALVES = (1536, 1280, 1152, 1024, 1024, 896, 768, 512)


def run_variant(args, w):
    """Time the one-call API on a grouped-head or packed version of `w`.

    gqa: k and v with heads // 4 heads; varlen: the samples of VARLEN_HALVES
    (scaled to the workload's rows) packed along the rows.  One step is the
    forward and the backward (scratch, preprocess, main, dq convert) through
    dfa_forward_gqa / dfa_backward_gqa or dfa_forward_varlen /
    dfa_backward_varlen; FLOPs count the visible pairs of every sample.
    """
    import torch

    from block_diffusion_masked_gb300 import binding

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.lib()
    stream = torch.cuda.current_stream(dev)
    H, d, bs = w.heads, w.headdim, w.block_size
    if args.variant in ("gqa", "onecall"):
        # onecall: the one-call API with every head its own key/value head,
        # the baseline of the packed line; gqa: the step API (the headline's
        # path) with a key/value head per 4 query heads
        Hk = max(1, H // 4) if args.variant == "gqa" else H
        q, _, _, do = inputs.make_workload_inputs(w)
        _, k, v = inputs.make_inputs(w.batch, w.n, Hk, d, seed=w.seed + 1, with_dout=False)
        q, k, v, do = (t.to(dev) for t in (q, k, v, do))
        halves = [w.n] * w.batch
        shape = {"batch": w.batch, "n": w.n, "heads": H, "kv_heads": Hk}
        if args.variant == "onecall":
            fwd = lambda: binding.dfa_forward_gqa(q, k, v, bs)  # noqa: E731
            bwd = lambda o, l: binding.dfa_backward_gqa(q, k, v, o, do, l, bs)  # noqa: E731
        else:
            B_, L_ = q.shape[0], q.shape[1]
            out = torch.empty_like(q)
            lse = torch.empty((B_, H, L_), dtype=torch.float32, device=dev)
            dq_acc = torch.empty(q.shape, dtype=torch.float32, device=dev)
            delta = torch.empty((B_, H, L_), dtype=torch.float32, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            shape["api"] = "step (forward zeroing dq_acc, preprocess, main, convert)"

            def fwd():
                binding.dfa_fwd_main_gqa(q, k, v, out, lse, dq_acc, bs)
                return out, lse

            def bwd(o, l):
                binding.dfa_bwd_preprocess(o, do, delta, None)
                binding.dfa_bwd_main_gqa(q, k, v, do, l, delta, dq_acc, dk, dv, bs)
                binding.dfa_bwd_dq_convert(dq_acc, dq)
    elif args.variant == "fp8":
        # forward only: per-tensor e4m3 quantisation of the workload's q, k, v
        q, k, v = inputs.make_workload_inputs(w, with_dout=False)
        qs, ks, vs = (float(t.float().abs().max()) / 448.0 for t in (q, k, v))
        q, k, v = ((t.float() / s_).to(torch.float8_e4m3fn).to(dev)
                   for t, s_ in ((q, qs), (k, ks), (v, vs)))
        halves = [w.n] * w.batch
        # V^T made once, as a caller that quantises V would (its own cost is
        # reported as transpose_ms); the timed forward runs on it
        vt = binding.dfa_fp8_transpose_v(v)
        fwd = lambda: binding.dfa_forward_fp8_vt(q, k, vt, H, qs, ks, vs, bs)  # noqa: E731
        bwd = lambda o, l: None  # noqa: E731
        shape = {"batch": w.batch, "n": w.n, "heads": H, "inputs": "e4m3, per-tensor descale",
                 "api": "dfa_forward_fp8_vt on a V^T from dfa_fp8_transpose_v"}
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(3):
            binding.dfa_fp8_transpose_v(v, vt)
        t0.record(stream)
        for _ in range(10):
            binding.dfa_fp8_transpose_v(v, vt)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        shape["transpose_ms"] = t0.elapsed_time(t1) / 10
    else:
        scale = w.batch * w.n / sum(VARLEN_HALVES)
        halves = [max(1, int(round(h * scale))) for h in VARLEN_HALVES]
        rows = 2 * sum(halves)
        q, k, v, do = (t[0].to(dev) for t in inputs.make_inputs(1, rows // 2, H, d, seed=w.seed))
        cu = np.concatenate([[0], np.cumsum([2 * h for h in halves])]).astype(int).tolist()
        fwd = lambda: binding.dfa_forward_varlen(q, k, v, cu, bs)  # noqa: E731
        bwd = lambda o, l: binding.dfa_backward_varlen(q, k, v, o, do, l, cu, bs)  # noqa: E731
        shape = {"halves": halves, "rows": rows, "heads": H}
    pairs = sum(visible_pairs_per_sample(n, bs) for n in halves)
    f_fwd = 4.0 * pairs * d * H
    f_bwd = 0.0 if args.variant == "fp8" else 2.5 * f_fwd

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        o, l = fwd()
        if ev is not None:
            ev[1].record(stream)
        bwd(o, l)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        start.record(stream)
        for _ in range(args.steps):
            step()
        end.record(stream)
        torch.cuda.synchronize(dev)
    ms = start.elapsed_time(end) / args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for e in evs:
        step(e)
    torch.cuda.synchronize(dev)
    if binding.dfa_status() != 0:
        raise RuntimeError("device status set during the timed region")
    split = np.array([[e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])] for e in evs]).mean(0)
    return {
        "metric": "visible-pair TFLOPS fwd+bwd on 1 GB300 (" + args.variant + ")",
        "variant": args.variant,
        "value": (f_fwd + f_bwd) / (ms * 1e-3) / 1e12,
        "unit": "TFLOPS",
        "ms_per_step": ms,
        "steps": args.steps,
        "warmup": args.warmup,
        "fwd_tflops": f_fwd / (split[0] * 1e-3) / 1e12,
        "bwd_tflops": f_bwd / (split[1] * 1e-3) / 1e12 if f_bwd else None,
        "kernel_ms": {"fwd": float(split[0]), "bwd": float(split[1])},
        "dtype": "bf16",
        "data": "synthetic: i.i.d. N(0,1) bf16 from a seeded CPU generator",
        "config": dict({"workload": w.name, "headdim": d, "block_size": bs}, **shape),
        "clocks": clk.summary(),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="small", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-baseline-s", type=float, default=12.0)
    ap.add_argument("--ref-step-s", type=float, default=5.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sdpa", action="store_true", help="also time torch SDPA causal (context)")
    ap.add_argument("--variant", default="mha", choices=["mha", "onecall", "gqa", "varlen", "fp8"],
                    help="gqa / varlen / fp8: time the one-call API on that version of the "
                    "workload (fp8: the forward alone)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    w = inputs.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w, rank, world)), flush=True)
        return

    if args.variant != "mha":
        if rank == 0:
            print(json.dumps(run_variant(args, w)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    res = run_gpu(args, w, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_baseline_s)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
