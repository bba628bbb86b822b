"""Benchmark: block-diffusion attention, forward + backward, on GB300.

One step = one forward and one backward pass of attention under the
block-diffusion mask over one batch of the workload, through the C ABI of
libdfa (device-resident inputs).  Throughput counts visible (query, key)
pairs only: 4 * pairs * headdim * heads FLOPs per sample forward, 2.5x that
backward ("Fast Diffusion Attention", section "The right yardstick").

Timing follows "Measuring on power-capped GPUs": after at least 300 ms of
warm-up, rounds of back-to-back steps of the diffusion kernels and of the
causal yardstick (the same kernels, causal, on the 2B halves of length n)
alternate, each round at least 300 ms long; the reported step time is the
median round.  Inputs smaller than the L2 cache are timed step by
step with L2 flushed (a 512 MB write) before every step, outside the timed
interval (at most FLUSHED_STEPS steps a round).

Printed on one JSON line (rank 0): the headline (the "mid" workload: the
largest headdim-128 configuration), the end-to-end number through the public
API with host buffers, the roofline of the dominant kernel with its DRAM
traffic from the ncu summary kept under profiles/, the causal yardstick, the
oracle timed on the host cores, and a `per_config` entry for every other
workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mid]
    python bench.py --impl reference   # the float64 CPU oracle as the reference arm
    python bench.py --profile-workload mid   # a few steps for an ncu capture
    python bench.py --summarize-ncu CSV --workload mid --kernel NAME --out FILE
"""

from __future__ import annotations

import os

# BLAS threads of the CPU oracle: every core this process may run on (set
# before NumPy loads its BLAS).
_CORES = len(os.sched_getaffinity(0))
for _var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_var, str(_CORES))

import argparse  # noqa: E402
import glob  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import math  # noqa: E402
import re  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_diffusion_masked_gb300 import inputs  # noqa: E402

METRIC = "visible-pair TFLOPS fwd+bwd on 1 GB300; % of BF16 peak; × vs causal yardstick"
HEADLINE = "mid"
PER_CONFIG = ("tiny", "small", "long", "hd256_bs1", "hd256_bs64", "hd256_bs128")
ROUND_MS = 300.0
ROUNDS = 10
L2_FLUSH_BYTES = 512 << 20
GB300_L2_BYTES = 126 << 20  # nominal; the GPU arm uses the device's own figure
FLUSHED_STEPS = 100
CSRC = os.path.join(ROOT, "block_diffusion_masked_gb300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")


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


# ------------------------------------------------------------------ kernels and traffic

# The translation unit that defines each kernel; a kernel's identity for the
# traffic records is the hash of that file and of the shared headers.
KERNEL_SOURCES = {
    "dfa_fwd2_kernel": "fwd2.cu",
    "dfa_fwd_kernel": "fwd.cu",
    "dfa_bwd2_kernel": "bwd2.cu",
}


def kernel_names(d):
    """(forward, backward main) kernel names as the library launches them."""
    fwd = "dfa_fwd_kernel<256>" if d == 256 else f"dfa_fwd2_kernel<{d}>"
    bwd = f"dfa_bwd2_kernel<{d}>"
    return fwd, bwd


def source_hash(kernel):
    """sha256 over the kernel's own .cu file and every shared header."""
    base = kernel.split("<")[0]
    files = [os.path.join(CSRC, KERNEL_SOURCES[base])]
    files += sorted(glob.glob(os.path.join(CSRC, "*.cuh")))
    h = hashlib.sha256()
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def read_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` on `workload` from a profiles/ summary.

    Each summary holds `key: value` lines (workload, kernel, source_sha256,
    dram_bytes_per_launch).  Returns (bytes or None, file name or reason):
    None when no summary matches or the kernel's sources changed since.
    """
    for path in sorted(glob.glob(os.path.join(PROFILES, "*.md"))):
        rec = {}
        with open(path) as f:
            for line in f:
                m = re.match(r"^\s*-?\s*`?(workload|kernel|source_sha256|dram_bytes_per_launch)`?"
                             r"\s*:\s*`?([^`\s]+)`?", line)
                if m:
                    rec[m.group(1)] = m.group(2)
        if rec.get("workload") != workload or rec.get("kernel") != kernel:
            continue
        name = os.path.relpath(path, ROOT)
        if rec.get("source_sha256") != source_hash(kernel):
            return None, f"{name}: kernel sources changed since the capture"
        try:
            return float(rec["dram_bytes_per_launch"]), name
        except (KeyError, ValueError):
            return None, f"{name}: no dram_bytes_per_launch"
    return None, "no ncu summary for this kernel and workload"


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
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for *_, r in rows for i, x in enumerate(r)
                          if x.lower() == "active"})
        loaded = [r for r in rows if r[0] > 0.5 * r[1]] or rows
        return {"sm_mhz": float(np.median([r[0] for r in loaded])), "sm_max_mhz": rows[0][1],
                "power_w_median": float(np.median([r[2] for r in loaded])),
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
    c0 = time.process_time()
    done = 0
    for bh in heads:
        oracle.diffusion_forward(qn, kn, vn, w.block_size, heads=[bh])
        oracle.diffusion_backward(qn, kn, vn, don, w.block_size, heads=[bh])
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    busy = (time.process_time() - c0) / dt
    threads = os.environ.get("OPENBLAS_NUM_THREADS", str(_CORES))
    return {"value": done * per_head_flops / dt / 1e12, "unit": "TFLOPS",
            "cores": _CORES, "kind": "oracle", "blas_threads": int(threads),
            "cpu_busy_cores": round(busy, 2),
            "sample": f"{done} of {len(heads)} (batch, head) pairs of workload '{w.name}', "
                      f"forward + backward, float64 NumPy, BLAS threads = {threads} "
                      f"(= cores in this process's affinity set), {dt:.1f} s"}


# ------------------------------------------------------------------ GPU arm

class Steps:
    """Device buffers and the step functions of one workload.

    diff(): dfa_fwd_main (zeroing the dq accumulator) + the three backward
    steps on the (B, 2n) tensors; causal(): the same kernels in the causal
    mode on the (2B, n) view.  Each takes an optional list of 5 events
    recorded between the launches.
    """

    def __init__(self, w, dev):
        import torch

        from block_diffusion_masked_gb300 import binding as b

        self.b = b
        self.w = w
        q, k, v, do = (t.to(dev) for t in inputs.make_workload_inputs(w))
        self.q, self.k, self.v, self.do = q, k, v, do
        B, L, H, d = q.shape
        n = L // 2
        self.out = torch.empty_like(q)
        self.lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
        self.dq, self.dk, self.dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        self.dq_acc = torch.empty(q.shape, dtype=torch.float32, device=dev)
        self.delta = torch.empty((B, H, L), dtype=torch.float32, device=dev)
        self.c = [t.view(2 * B, n, H, d) for t in (q, k, v, do)]
        self.outc = torch.empty_like(self.c[0])
        self.lsec = torch.empty((2 * B, H, n), dtype=torch.float32, device=dev)
        self.deltac = torch.empty((2 * B, H, n), dtype=torch.float32, device=dev)
        self.dqc, self.dkc, self.dvc = (torch.empty_like(self.c[0]) for _ in range(3))
        self.dq_accc = self.dq_acc.view(2 * B, n, H, d)
        self.input_bytes = 4 * q.numel() * q.element_size()

    def diff(self, ev=None):
        b, w = self.b, self.w
        stream = _stream(self.q)
        if ev is not None:
            ev[0].record(stream)
        b.dfa_fwd_main(self.q, self.k, self.v, self.out, self.lse, self.dq_acc, w.block_size)
        if ev is not None:
            ev[1].record(stream)
        b.dfa_bwd_preprocess(self.out, self.do, self.delta, None)
        if ev is not None:
            ev[2].record(stream)
        b.dfa_bwd_main(self.q, self.k, self.v, self.do, self.lse, self.delta, self.dq_acc,
                       self.dk, self.dv, w.block_size)
        if ev is not None:
            ev[3].record(stream)
        b.dfa_bwd_dq_convert(self.dq_acc, self.dq)
        if ev is not None:
            ev[4].record(stream)

    def causal(self, ev=None):
        b = self.b
        cm = b.MODE_CAUSAL
        qc, kc, vc, doc = self.c
        stream = _stream(self.q)
        if ev is not None:
            ev[0].record(stream)
        b.dfa_fwd_main(qc, kc, vc, self.outc, self.lsec, self.dq_accc, 1, mode=cm)
        if ev is not None:
            ev[1].record(stream)
        b.dfa_bwd_preprocess(self.outc, doc, self.deltac, None, mode=cm)
        if ev is not None:
            ev[2].record(stream)
        b.dfa_bwd_main(qc, kc, vc, doc, self.lsec, self.deltac, self.dq_accc, self.dkc,
                       self.dvc, 1, mode=cm)
        if ev is not None:
            ev[3].record(stream)
        b.dfa_bwd_dq_convert(self.dq_accc, self.dqc, mode=cm)
        if ev is not None:
            ev[4].record(stream)


LAUNCHES_PER_STEP = 4


def _stream(t):
    import torch

    return torch.cuda.current_stream(t.device)


def _barrier(world, dev):
    import torch

    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize(dev)


def time_workload(args, w, dev, world):
    """Interleaved rounds of diffusion and causal steps on one workload."""
    import torch

    from block_diffusion_masked_gb300 import binding

    st = Steps(w, dev)
    stream = _stream(st.q)
    flush = st.input_bytes < torch.cuda.get_device_properties(dev).L2_cache_size
    l2 = l2_note(st.input_bytes, flush)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
    arms = (("diff", st.diff), ("causal", st.causal))

    def run(fn, steps):
        """ms of `steps` steps on the device (flushed and timed per step when
        the inputs fit in L2; else back to back, events at the two ends)."""
        if flush:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(steps)]
            for e0, e1 in evs:
                flush_buf.fill_(1.0)
                e0.record(stream)
                fn()
                e1.record(stream)
            torch.cuda.synchronize(dev)
            return sum(e0.elapsed_time(e1) for e0, e1 in evs)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    # warm-up: at least W steps of each arm and at least ROUND_MS of work
    t0 = time.perf_counter()
    warm = 0
    per_step = {}
    while warm < args.warmup or (time.perf_counter() - t0) * 1e3 < ROUND_MS:
        for name, fn in arms:
            per_step[name] = run(fn, 1)
        warm += 1
    torch.cuda.synchronize(dev)
    if binding.dfa_status() != 0:
        raise RuntimeError(f"device status set during warm-up ({w.name})")
    per_step = dict(zip(per_step, max_over_ranks(list(per_step.values()), dev)))

    if args.steps:
        spr = {name: max(1, math.ceil(args.steps / ROUNDS)) for name, _ in arms}
    else:
        spr = {name: max(1, math.ceil(ROUND_MS / max(per_step[name], 1e-3))) for name, _ in arms}
        if flush:
            spr = {name: min(v_, FLUSHED_STEPS) for name, v_ in spr.items()}
    rounds = {name: [] for name, _ in arms}
    with ClockSampler(dev.index) as clk:
        for _ in range(ROUNDS):
            for name, fn in arms:
                _barrier(world, dev)
                ms = run(fn, spr[name])
                _barrier(world, dev)
                rounds[name].append(max_over_ranks([ms], dev)[0] / spr[name])
    clocks = clk.summary()
    # per-kernel durations: a separate pass with events between the launches
    kparts = {}
    for name, fn in arms:
        k = max(3, min(spr[name], 50))
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(k)]
        _barrier(world, dev)
        for e in evs:
            if flush:
                flush_buf.fill_(1.0)
            fn(e)
        _barrier(world, dev)
        kparts[name] = np.median(np.array([[e[j].elapsed_time(e[j + 1]) for j in range(4)]
                                           for e in evs]), axis=0).tolist()
    if binding.dfa_status() != 0:
        raise RuntimeError(f"device status set during the timed region ({w.name})")

    f_fwd, f_bwd = flops(w)
    c_fwd, c_bwd = causal_flops(w)
    ms = float(np.median(rounds["diff"]))
    ms_c = float(np.median(rounds["causal"]))
    value = job_tflops(f_fwd + f_bwd, ms, world)
    cvalue = job_tflops(c_fwd + c_bwd, ms_c, world)
    peaks = measured_peaks()
    names = ("fwd", "bwd_preprocess", "bwd_main", "dq_convert")
    fwd_ms, pre_ms, main_ms, conv_ms = kparts["diff"]
    fwd_name, bwd_name = kernel_names(w.headdim)
    dominant = max(((fwd_name, fwd_ms, f_fwd), (bwd_name, main_ms, f_bwd)), key=lambda x: x[1])
    achieved = dominant[2] / (dominant[1] * 1e-3) / 1e12
    traffic, traffic_src = read_traffic(w.name, dominant[0])
    timed_steps = ROUNDS * spr["diff"]
    res = {
        "workload": w.name,
        "value": value, "unit": "TFLOPS", "ms_per_step": ms,
        "pct_of_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
        "steps": timed_steps,
        "timing": {"rounds": ROUNDS, "steps_per_round": spr,
                   "round_ms_median": {k_: float(np.median(v_)) * spr[k_]
                                       for k_, v_ in rounds.items()},
                   "spread_pct": 100.0 * (max(rounds["diff"]) - min(rounds["diff"])) / ms,
                   "l2": l2},
        "fwd_tflops": f_fwd / (fwd_ms * 1e-3) / 1e12,
        "bwd_tflops": f_bwd / ((pre_ms + main_ms + conv_ms) * 1e-3) / 1e12,
        "kernel_ms": dict(zip(names, kparts["diff"])),
        "yardstick": {"what": "same kernels, causal attention on the 2B halves of length n",
                      "value": cvalue, "unit": "TFLOPS", "ms_per_step": ms_c,
                      "ratio": value / cvalue, "kernel_ms": dict(zip(names, kparts["causal"]))},
        "roofline": {"kernel": dominant[0], "bound": "tensor", "achieved": achieved,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"],
                     "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                     "peak_source": peaks["source"] + " bf16 burst (cuBLAS 8192^3)",
                     "traffic": traffic, "traffic_source": traffic_src,
                     "traffic_unit": "bytes per launch (ncu dram read + write)"},
        "clocks": clocks,
        "gpu_launches": LAUNCHES_PER_STEP * ROUNDS * (spr["diff"] + spr["causal"]),
    }
    return res, st


def e2e_measure(args, w, st, dev, world):
    """The public one-call API with host buffers, copies inside the timed region.

    Every step copies its q/k/v/dout from pinned host memory and its
    out/dq/dk/dv/lse back; the copies run on their own streams (one per
    direction) and overlap the neighbouring steps' compute, as in a training
    loop that stages its next batch, with two device buffer sets.
    """
    import torch

    from block_diffusion_masked_gb300 import binding

    stream = _stream(st.q)
    q, lse = st.q, st.lse
    B, L, H, d = q.shape
    host_in = [t.cpu().pin_memory() for t in (st.q, st.k, st.v, st.do)]
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
        bset = i % 2
        with torch.cuda.stream(h2d_s):
            if i >= 2:
                h2d_s.wait_event(ev_done[bset])  # step i-2 has finished reading the set
            for hbuf, dbuf in zip(host_in, sets[bset]["in"]):
                dbuf.copy_(hbuf, non_blocking=True)
            ev_in[bset].record(h2d_s)

    def e2e_run(steps, start_event=None):
        if start_event is not None:
            h2d_s.wait_event(start_event)
        issue_h2d(0)
        for i in range(steps):
            bset = i % 2
            s = sets[bset]
            if i + 1 < steps:
                issue_h2d(i + 1)
            stream.wait_event(ev_in[bset])
            if i >= 2:
                stream.wait_event(ev_out[bset])  # step i-2's results have left the set
            o, l_ = binding.dfa_forward(s["in"][0], s["in"][1], s["in"][2], w.block_size,
                                        out=s["out"], lse=s["lse"])
            g = binding.dfa_backward(s["in"][0], s["in"][1], s["in"][2], o, s["in"][3], l_,
                                     w.block_size, dq=s["grads"][0], dk=s["grads"][1],
                                     dv=s["grads"][2])
            ev_done[bset].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_done[bset])
                for hbuf, dbuf in zip(host_out, (o,) + tuple(g)):
                    hbuf.copy_(dbuf, non_blocking=True)
                host_lse.copy_(l_, non_blocking=True)
                ev_out[bset].record(d2h_s)
        stream.wait_event(ev_out[(steps - 1) % 2])

    steps = max(args.warmup, 3)
    e2e_run(steps)
    torch.cuda.synchronize(dev)
    k = max(10, args.steps or 0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world, dev)
    e0.record(stream)
    e2e_run(k, start_event=e0)
    e1.record(stream)
    _barrier(world, dev)
    e2e_ms = max_over_ranks([e0.elapsed_time(e1)], dev)[0]
    f_fwd, f_bwd = flops(w)
    tensor_bytes = q.numel() * 2
    return {"value": job_tflops(f_fwd + f_bwd, e2e_ms / k, world), "unit": "TFLOPS",
            "steps": k, "ms_per_step": e2e_ms / k,
            "h2d_bytes_per_step": 4 * tensor_bytes,
            "d2h_bytes_per_step": 4 * tensor_bytes + host_lse.numel() * 4}


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


def l2_note(input_bytes, flush):
    """How the timed steps treat L2 (the same text on both arms)."""
    if flush:
        return "inputs fit in L2: 512 MB flush before every step, outside the timed interval"
    return f"inputs ({input_bytes / 1e6:.0f} MB of q/k/v/dout) larger than L2: no flush"


def _config(w, world, l2):
    return {"workload": w.name, "batch": w.batch, "n": w.n, "seqlen": 2 * w.n,
            "heads": w.heads, "headdim": w.headdim, "block_size": w.block_size,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU", "l2": l2,
            "why_headline": "mid is the largest headdim-128 configuration (964 GFLOP per step, "
                            "537 MB of q/k/v/dout); long and hd256 are of the same FLOP size "
                            "and are reported in per_config"}


def run_gpu(args, rank, world):
    import torch

    from block_diffusion_masked_gb300 import binding

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    binding.lib()
    w = inputs.WORKLOADS[args.workload]
    head, st = time_workload(args, w, dev, world)
    e2e = e2e_measure(args, w, st, dev, world)
    sdpa = None
    if args.sdpa:
        c_fwd, c_bwd = causal_flops(w)
        try:
            sdpa = (c_fwd + c_bwd) / (sdpa_causal(*st.c, args.warmup, 10) * 1e-3) / 1e12
        except Exception as exc:  # context only
            sdpa = f"unavailable: {exc}"
    del st
    torch.cuda.empty_cache()
    per = {}
    launches = head["gpu_launches"]
    if not args.headline_only:
        for name in PER_CONFIG:
            if name == w.name:
                continue
            r, st_ = time_workload(args, inputs.WORKLOADS[name], dev, world)
            del st_
            torch.cuda.empty_cache()
            launches += r.pop("gpu_launches")
            r.pop("workload")
            per[name] = r
    res = {
        "metric": METRIC, "value": head["value"], "unit": "TFLOPS", "n_gpus": world,
        "steps": head["steps"], "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: i.i.d. N(0,1)*std bf16 q/k/v/dout from a seeded CPU generator",
        "config": _config(w, world, head["timing"]["l2"]),
        "pct_of_bf16_peak": head["pct_of_bf16_peak"],
        "timing": head["timing"],
        "fwd_tflops": head["fwd_tflops"], "bwd_tflops": head["bwd_tflops"],
        "kernel_ms": head["kernel_ms"],
        "yardstick": head["yardstick"],
        "gpu_launches": launches,
        "e2e": e2e,
        "roofline": head["roofline"],
        "clocks": head["clocks"],
        "per_config": per,
    }
    if sdpa is not None:
        res["sdpa_causal_tflops"] = sdpa
    return res


def run_profile(args):
    """A few steps of one workload (no e2e, no CPU baseline) for an ncu capture."""
    import torch

    from block_diffusion_masked_gb300 import binding

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.lib()
    st = Steps(inputs.WORKLOADS[args.profile_workload], dev)
    for _ in range(args.profile_steps):
        st.diff()
    torch.cuda.synchronize(dev)
    if binding.dfa_status() != 0:
        raise RuntimeError("device status set")
    print(json.dumps({"profiled": args.profile_workload, "steps": args.profile_steps}))


def algorithmic_bytes(w, backward):
    """Bytes a launch must move at least, as the step runs it: forward reads
    q, k, v, writes out and lse, and zeroes the float32 dq accumulator;
    backward main reads q, k, v, dout, lse, D, writes dk, dv and reads and
    writes the float32 dq accumulator once."""
    T = w.batch * 2 * w.n * w.heads * w.headdim  # elements of one tensor
    rows = w.batch * w.heads * 2 * w.n
    if backward:
        return 4 * 2 * T + 2 * 4 * rows + 2 * 2 * T + 2 * 4 * T, \
            "q, k, v, dout, lse, D read; dk, dv written; dq accumulator read and written"
    return 4 * 2 * T + 4 * rows + 4 * T, "q, k, v read; out, lse written; dq accumulator zeroed"


def summarize_ncu(args):
    """Write a profiles/ summary of an ncu --csv capture of one kernel.

    The capture holds dram__bytes_read.sum, dram__bytes_write.sum (and
    optionally gpu__time_duration.sum, sm__pipe_tensor_cycles_active) for
    each launch of the kernel; the summary records the per-launch mean with
    the kernel's source hash, the keys bench.py reads back.
    """
    import csv

    rows = []
    with open(args.summarize_ncu) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for r in csv.DictReader(lines):
        if args.kernel.split("<")[0] in r.get("Kernel Name", ""):
            rows.append(r)
    by_launch = {}
    for r in rows:
        by_launch.setdefault(r["ID"], {})[r["Metric Name"]] = (r["Metric Unit"], r["Metric Value"])

    def val(m, unit_scale):
        out = []
        for d in by_launch.values():
            if m in d:
                u, v = d[m]
                out.append(float(v.replace(",", "")) * unit_scale.get(u, 1.0))
        return out

    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6,
             "GB": 1e9, "nsecond": 1e-9, "usecond": 1e-6, "msecond": 1e-3, "second": 1.0,
             "ns": 1e-9, "us": 1e-6, "ms": 1e-3, "s": 1.0, "%": 1.0}
    rd = val("dram__bytes_read.sum", scale)
    wr = val("dram__bytes_write.sum", scale)
    if not rd or len(rd) != len(wr):
        raise SystemExit("no dram__bytes_read.sum / dram__bytes_write.sum for that kernel")
    traffic = float(np.mean(np.array(rd) + np.array(wr)))
    dur = val("gpu__time_duration.sum", scale)
    tens = val("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active", scale)
    w = inputs.WORKLOADS[args.workload]
    f_fwd, f_bwd = flops(w)
    is_bwd = "bwd" in args.kernel
    algo = f_bwd if is_bwd else f_fwd
    algo_bytes, algo_what = algorithmic_bytes(w, is_bwd)
    lines = [f"# {args.kernel} on {args.workload}", "",
             f"Workload: B {w.batch}, n {w.n}, H {w.heads}, d {w.headdim}, bs {w.block_size}.",
             f"Launches captured: {len(rd)}.", "",
             f"- workload: {args.workload}",
             f"- kernel: {args.kernel}",
             f"- source_sha256: {source_hash(args.kernel)}",
             f"- dram_bytes_per_launch: {traffic:.6g}",
             f"- dram_read_bytes: {np.mean(rd):.6g}",
             f"- dram_write_bytes: {np.mean(wr):.6g}",
             f"- algorithmic_bytes: {algo_bytes:.6g} ({algo_what})",
             f"- traffic / algorithmic: {traffic / algo_bytes:.2f}"]
    if dur:
        lines.append(f"- ncu_duration_us (serialised, cold): {np.mean(dur) * 1e6:.1f}")
        lines.append(f"- algorithmic_tflops_at_ncu_duration: {algo / np.mean(dur) / 1e12:.1f}")
    if tens:
        lines.append(f"- tensor_pipe_active_pct: {np.mean(tens):.1f}")
    lines += ["", "Command (one GB300, from the repository root; the plain run must exit 0 "
              "before the capture):", "", "```", args.command or "(not given)", "```", ""]
    with open(args.out, "w") as f:
        f.write("\n".join(lines))
    print(args.out, traffic)


def run_reference(args, rank, world):
    """The reference arm: the float64 oracle on the host cores, bounded steps."""
    w = inputs.WORKLOADS[args.workload]
    per_step = []
    base = None
    for i in range(args.warmup + (args.steps or 3)):
        r = cpu_baseline(w, budget_s=args.ref_step_s, max_heads=1)
        if i >= args.warmup:
            per_step.append(r["value"])
            base = r
    value = float(np.median(per_step))
    base = dict(base)
    base["value"] = value
    nbytes = 4 * w.batch * 2 * w.n * w.heads * w.headdim * 2
    cfg = _config(w, world, l2_note(nbytes, nbytes < GB300_L2_BYTES))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
            "n_gpus": world, "steps": len(per_step), "warmup": args.warmup,
            "ms_per_step": None, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg, "cpu_baseline": base,
            "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# Half lengths of the packed varlen batch: a mix of sample lengths with the
# rows of the workload it stands beside (8 x 2048 rows for "small").
VARLEN_HALVES = (1536, 1280, 1152, 1024, 1024, 896, 768, 512)


def run_variant(args, w):
    """Time the one-call API on a grouped-head or packed version of `w`.

    gqa: k and v with heads // 4 heads (the step API); step: the same step
    API with every head its own key/value head (the baseline of gqa);
    onecall: the one-call API, multi-head; diagpass: the step API with the
    noisy-diagonal backward option (DFA_NOISY_DIAG_PASS; step is its
    baseline); varlen: the samples of
    VARLEN_HALVES (scaled to the workload's rows) packed along the rows;
    fp8: the FP8 forward.  FLOPs count the visible pairs of every sample.
    """
    import torch

    from block_diffusion_masked_gb300 import binding

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    binding.lib()
    stream = torch.cuda.current_stream(dev)
    H, d, bs = w.heads, w.headdim, w.block_size
    if args.variant in ("gqa", "onecall", "step", "diagpass"):
        Hk = max(1, H // 4) if args.variant == "gqa" else H
        q, _, _, do = inputs.make_workload_inputs(w)
        _, k, v = inputs.make_inputs(w.batch, w.n, Hk, d, seed=w.seed + 1, with_dout=False)
        q, k, v, do = (t.to(dev) for t in (q, k, v, do))
        halves = [w.n] * w.batch
        shape = {"batch": w.batch, "n": w.n, "heads": H, "kv_heads": Hk}
        if args.variant == "onecall":
            fwd = lambda: binding.dfa_forward_gqa(q, k, v, bs)  # noqa: E731
            bwd = lambda o, l: binding.dfa_backward_gqa(q, k, v, o, do, l, bs)  # noqa: E731
            shape["api"] = "one call (dfa_forward_gqa / dfa_backward_gqa)"
        else:
            B_, L_ = q.shape[0], q.shape[1]
            out = torch.empty_like(q)
            lse = torch.empty((B_, H, L_), dtype=torch.float32, device=dev)
            dq_acc = torch.empty(q.shape, dtype=torch.float32, device=dev)
            delta = torch.empty((B_, H, L_), dtype=torch.float32, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            shape["api"] = "step (forward zeroing dq_acc, preprocess, main, convert)"
            diag = args.variant == "diagpass"
            if diag:
                shape["api"] += ", noisy-diagonal pass"

            def fwd():
                binding.dfa_fwd_main_gqa(q, k, v, out, lse, dq_acc, bs)
                return out, lse

            def bwd(o, l):
                binding.dfa_bwd_preprocess(o, do, delta, None)
                binding.dfa_bwd_main_ex(q, k, v, do, l, delta, dq_acc, dk, dv, bs,
                                        noisy_diag_pass=diag)
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
        Hk = k.shape[2]
        fwd = lambda: binding.dfa_forward_fp8_vt(q, k, vt, Hk, qs, ks, vs, bs)  # noqa: E731
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
    steps = args.steps or 20

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        o, l_ = fwd()
        if ev is not None:
            ev[1].record(stream)
        bwd(o, l_)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        start.record(stream)
        for _ in range(steps):
            step()
        end.record(stream)
        torch.cuda.synchronize(dev)
    ms = start.elapsed_time(end) / steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
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
        "steps": steps,
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
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps of the diffusion arm, spread over the rounds (0: as many "
                         "as make each round at least 300 ms)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-baseline-s", type=float, default=12.0)
    ap.add_argument("--ref-step-s", type=float, default=5.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true", help="skip the per_config workloads")
    ap.add_argument("--sdpa", action="store_true", help="also time torch SDPA causal (context)")
    ap.add_argument("--variant", default="mha",
                    choices=["mha", "onecall", "step", "diagpass", "gqa", "varlen", "fp8"],
                    help="gqa / step / diagpass / onecall / varlen / fp8: time that API on that "
                    "version of the workload (fp8: the forward alone)")
    ap.add_argument("--profile-workload", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--profile-steps", type=int, default=3)
    ap.add_argument("--summarize-ncu")
    ap.add_argument("--kernel")
    ap.add_argument("--out")
    ap.add_argument("--command")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.summarize_ncu:
        summarize_ncu(args)
        return
    if args.profile_workload:
        run_profile(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    if args.variant != "mha":
        if rank == 0:
            print(json.dumps(run_variant(args, inputs.WORKLOADS[args.workload])), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    res = run_gpu(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(inputs.WORKLOADS[args.workload],
                                               budget_s=args.cpu_baseline_s)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
