#!/usr/bin/env python
"""Benchmark of the Gated DeltaNet forward on one node of GB300 GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one gdn_chunk_fwd call over the single-sequence prefill workload
(B=1, T=4096, Hq=16, Hv=32, d=128, bf16 q/k/v, f32 g/beta, zero initial
state, f32 final state), inputs resident in HBM. Between timed steps the L2 is
flushed by writing a 512 MiB buffer (the inputs, 104 MB, would fit in the
126 MB L2). Prints ONE JSON line (rank 0). The decode step (256 sequences x 32
v-heads, f32 state read and written in place) is measured in the same run and
reported under "decode"; the same step fed raw q/k and gate projections (the
front-end and the output gate computed in the kernel) under "decode_gated",
and that with a bf16 state cache and bf16 beta under "decode_sglang";
the stand-alone output gate (gdn_gated_rmsnorm) over the prefill's
[4096, 32, 128] read-out under "output_gate"; the short convolution (prefill
projections and one decode step) and the gating under "front_end"; the prefill
step with the output gate fused in (gdn_chunk_fwd_gated) under "prefill_gated";
the plain prefill on 8 packed sequences of U[100, 8000] tokens with initial
states and on one T=65536 sequence under "prefill_configs".

Multi-GPU (torchrun, one rank per GPU): every rank runs its own replica of the
workload (weak scaling: the GDN core shards over sequences and heads with no
exchange); a barrier brackets the timed region and the slowest rank's time is
taken.

--impl reference times the CPU oracle (plain C, float64, OpenMP on every host
core) on the same workload: each step is one chunk-form pass over all tokens
and all heads, and the line reports the median step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from gated_deltanet_chunked_gb300 import workloads as W  # noqa: E402

METRIC = "GDN prefill tokens/s (T=4096,Hv=32,d=128) & % roofline; decode state GB/s"
PREFILL = W.WORKLOADS["prefill_T4096_hq16_hv32"]
DECODE = W.WORKLOADS["decode_N256_hq16_hv32"]
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 512 << 20
L2_NOTE = "flushed between timed launches (512 MiB write)"


class L2Flush:
    """Evicts the L2 between timed launches by writing a buffer four times its
    size. (Measured on the prefill step: as fast as no flush at all, since
    the step's own 240 MB of traffic evicts its inputs anyway; the dirty
    lines the write leaves cost it nothing measurable.)"""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.w.fill_(1)


# --------------------------------------------------------------------------
# algorithmic byte / flop model (per token, per sequence, per chunk)
# --------------------------------------------------------------------------
def prefill_bytes(T, N, hq, hv, io_bytes=2, s0=False, final=True, d=128):
    per_tok = hq * d * io_bytes * 2 + hv * d * io_bytes * 2 + hv * 8  # q,k + v,o + g,beta
    per_seq = hv * d * d * 4 * (int(s0) + int(final))
    return T * per_tok + N * per_seq


def prefill_flops(n_chunk_heads, hv, hq, C=64, d=128):
    G = hv // hq
    per = 6 * C * d * d + C * C * (d + d) + C * C * d + 2 * C * C * d / G
    return n_chunk_heads * per


def kernel_bytes(name, T, N, hq, hv, io_bytes=2, s0=False, final=True, d=128):
    """Compulsory HBM bytes of one launch of a kernel (its share of the path's
    inputs and outputs; intermediates kept in workspace are not counted)."""
    qk = T * hq * d * io_bytes
    vv = T * hv * d * io_bytes
    gb = T * hv * 8
    st = N * hv * d * d * 4 * (int(s0) + int(final))
    return {
        "chunk_table": 4 * (N + 1),
        "prep_simt": qk + vv + gb,
        "state_simt": qk + st,
        "output_simt": 2 * qk + vv,
        "chunk_fused_tc": 2 * qk + 2 * vv + gb + st,
    }.get(name)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_deltanet_chunked_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != source_hash():
        return None
    k = d.get("kernels", {}).get(kernel)
    return None if k is None else k.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_ms=50):
        self.gpu_index, self.period_ms = gpu_index, period_ms
        self.samples, self.proc, self.thread = [], None, None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        win = [s for t, s in self.samples if t0 - 0.06 <= t <= t1 + 0.06]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm = []
        for s in win:
            try:
                sm.append(float(s[1]))
            except ValueError:
                pass
            for i, n in enumerate(names):
                if len(s) > 5 + i and s[5 + i].lower() == "active":
                    reasons.add(n)
        try:
            smax = float(win[-1][2])
        except ValueError:
            smax = None
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(win), "power_w_max": max((float(s[3]) for s in win if _isnum(s[3])), default=None)}


def _isnum(x):
    try:
        float(x)
        return True
    except ValueError:
        return False


# --------------------------------------------------------------------------
# distributed plumbing (timing only; the data path has no collective)
# --------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend, init_method="env://")
    return world, rank, local


def barrier(world, dev=None):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world, dev):
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    from gated_deltanet_chunked_gb300 import gdn

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the CUDA path has no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gdn.load()
    peaks, peak_src = load_peaks()

    w = PREFILL
    host = W.make_prefill(w)
    T, N = host["total_tokens"], host["num_seqs"]
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    out = torch.empty_like(d["v"])
    fin = torch.empty((N, w.hv, 128, 128), dtype=torch.float32, device=dev)
    prob = gdn.prefill_problem(d["q"], d["v"], N, packed=True)
    ws = torch.empty(gdn.gdn_chunk_fwd_workspace_size(prob), dtype=torch.uint8, device=dev)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    flush = L2Flush(dev)

    def step():
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], initial_state=None, cu_seqlens=cu,
                          out=out, final_state=fin, workspace=ws)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    assert gdn.gdn_read_device_status() == gdn.GDN_OK

    clocks = ClockSampler(local).start()
    time.sleep(0.3)
    # the timed steps run without the library's per-kernel events (their
    # records would sit inside every step); launches are counted regardless
    gdn.gdn_profile_enable(False)
    gdn.gdn_profile_collect(reset=True)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_start = time.time()
    for i in range(args.steps):
        flush()
        ev0[i].record()
        step()
        ev1[i].record()
    torch.cuda.synchronize()
    t_end = time.time()
    barrier(world)
    counts = gdn.gdn_profile_collect(reset=True)
    # per-kernel times: a second, profiled pass over the same steps
    prof_steps = min(args.steps, 50)
    gdn.gdn_profile_enable(True)
    for i in range(prof_steps):
        flush()
        step()
    torch.cuda.synchronize()
    gdn.gdn_profile_enable(False)
    prof = gdn.gdn_profile_collect(reset=True)
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    ms_local = statistics.median(step_ms)
    ms = max_over_ranks(ms_local, world, dev)
    value = world * T / (ms * 1e-3)

    # dominant kernel of the timed region
    kernels = {k: {"launches": counts.get(k, (0,))[0], "ms_per_launch": t / max(nt, 1), "timed_launches": nt}
               for k, (n, t, nt) in prof.items()}
    dom = max(kernels, key=lambda k: kernels[k]["ms_per_launch"] * kernels[k]["launches"])
    dom_bytes = kernel_bytes(dom, T, N, w.hq, w.hv)
    dom_ms = kernels[dom]["ms_per_launch"]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    path_bytes = prefill_bytes(T, N, w.hq, w.hv)
    n_chunk_heads = math.ceil(T / 64) * w.hv
    path_flops = prefill_flops(n_chunk_heads, w.hv, w.hq)
    roofline = {
        "kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
        "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(dom),
        "peak_source": f"{peak_src} (hbm_gbs, burst copy)",
        "algorithmic_bytes_per_launch": dom_bytes,
        "path": {
            "bytes": path_bytes, "flops": path_flops,
            "t_bytes_us": path_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6,
            "t_flops_us": path_flops / (peaks["bf16_tflops"] * 1e12) * 1e6,
            "frac_of_roofline": max(path_bytes / (peaks["hbm_gbs"] * 1e9),
                                    path_flops / (peaks["bf16_tflops"] * 1e12)) / (ms * 1e-3),
        },
    }
    gpu_launches = sum(n for (n, _, _) in counts.values())

    # end to end through the public API: pinned host inputs -> device -> host.
    # Serving-loop form: the copies in of step i+1 and out of step i-1 run on
    # their own streams while step i computes (two buffer sets, ordered by
    # events); every step's copies lie inside the timed region, which spans
    # the first copy in to the last copy out. The strictly serial time per
    # step (copy in, compute, copy out, one after another) is reported too.
    pin = {k: host[k].pin_memory() for k in ("q", "k", "v", "g", "beta")}
    nb = 2
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(nb)]
    fin_h = [torch.empty(fin.shape, dtype=fin.dtype).pin_memory() for _ in range(nb)]
    dev_in = [{k: torch.empty_like(d[k]) for k in pin} for _ in range(nb)]
    outs = [(torch.empty_like(out), torch.empty_like(fin)) for _ in range(nb)]
    bi = sum(t.numel() * t.element_size() for t in pin.values())
    bo = out_h[0].numel() * out_h[0].element_size() + fin_h[0].numel() * fin_h[0].element_size()
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(steps, serial):
        ev = lambda: torch.cuda.Event()
        h2d, cmp, d2h = [ev() for _ in range(steps)], [ev() for _ in range(steps)], [ev() for _ in range(steps)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(steps):
            b = i % nb
            with torch.cuda.stream(s_in):
                if i >= nb:
                    s_in.wait_event(cmp[i - nb])  # step i-2 has read this input set
                if serial and i > 0:
                    s_in.wait_event(d2h[i - 1])
                for k in pin:
                    dev_in[b][k].copy_(pin[k], non_blocking=True)
                h2d[i].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(h2d[i])
                if i >= nb:
                    s_cmp.wait_event(d2h[i - nb])  # step i-2's outputs have been copied out
                gdn.gdn_chunk_fwd(dev_in[b]["q"], dev_in[b]["k"], dev_in[b]["v"], dev_in[b]["g"], dev_in[b]["beta"],
                                  d["scale"], cu_seqlens=cu, out=outs[b][0], final_state=outs[b][1], workspace=ws,
                                  stream=s_cmp)
                cmp[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(cmp[i])
                out_h[b].copy_(outs[b][0], non_blocking=True)
                fin_h[b].copy_(outs[b][1], non_blocking=True)
                d2h[i].record(s_out)
        s_out.wait_event(d2h[steps - 1])
        t1.record(s_out)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / steps

    e2e_run(max(3, args.warmup), serial=False)
    barrier(world)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e2e_run(args.steps, serial=False), world, dev)
    e2e_serial_ms = max_over_ranks(e2e_run(min(args.steps, 50), serial=True), world, dev)
    barrier(world)
    e2e = {"value": world * T / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": bi,
           "d2h_bytes_per_step": bo, "ms_per_step": e2e_ms,
           "mode": "copies of neighbouring steps overlap the compute (streams + events, two buffer sets)",
           "serial_ms_per_step": e2e_serial_ms}

    decode = None if args.no_decode else run_decode(args, dev, world, peaks, peak_src)
    decode_gated = None if args.no_decode else run_decode(args, dev, world, peaks, peak_src, gated=True)
    decode_sglang = None if args.no_decode else run_decode(args, dev, world, peaks, peak_src, gated=True,
                                                           sglang=True)
    output_gate = None if args.no_decode else run_gate_norm(args, dev, world, peaks, peak_src)
    prefill_gated = None if args.no_decode else run_prefill_gated(args, dev, world)
    prefill_configs = None if (args.no_decode or args.no_configs) else run_prefill_configs(args, dev, world, peaks,
                                                                                           peak_src)
    front_end = None if args.no_decode else run_front_end(args, dev, world, peaks, peak_src)
    clocks.stop()
    clk = clocks.summary(t_start, t_end)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(host, w)

    # One JSON line. The headline keys come first and the decode figures
    # (half of the metric) last, with the f32-state decode as the final key,
    # so that a reader keeping only the line's tail still sees them; the
    # per-kernel tables and secondary legs are compact unless --detail.
    r3 = lambda x: None if x is None else round(x, 4)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": 1, "T": T, "hq": w.hq, "hv": w.hv, "dk": 128, "dv": 128,
                   "chunk": 64, "initial_state": "zero", "final_state": "f32",
                   "l2": L2_NOTE, "parallelism": f"replicas x{world}"},
        "step_ms": {"median": statistics.median(step_ms), "mean": statistics.mean(step_ms),
                    "p10": sorted(step_ms)[len(step_ms) // 10], "p90": sorted(step_ms)[(9 * len(step_ms)) // 10]},
        "roofline": roofline, "e2e": e2e, "clocks": clk, "gpu_launches": gpu_launches,
        "kernels_ms": {k: r3(v["ms_per_launch"]) for k, v in kernels.items()},
        "cpu_baseline": cpu,
    }
    if args.detail:
        line.update({"kernels": kernels, "front_end": front_end, "output_gate": output_gate})
    else:
        line["front_end_frac"] = None if front_end is None else {
            k: r3(v["roofline"]["frac"]) for k, v in front_end.items() if isinstance(v, dict) and "roofline" in v}
        line["output_gate_frac"] = None if output_gate is None else r3(output_gate["roofline"]["frac"])
    line["prefill_gated"] = None if prefill_gated is None else (
        prefill_gated if args.detail else {"ms_per_step": prefill_gated["ms_per_step"], "value": prefill_gated["value"]})
    line["prefill_configs"] = None if prefill_configs is None else (
        prefill_configs if args.detail else {
            k: {"ms_per_step": v["ms_per_step"], "value": v["value"], "roofline_us": r3(v["roofline_us"]),
                "frac_of_roofline": r3(v["frac_of_roofline"])} for k, v in prefill_configs.items()})

    def compact_decode(x):
        if x is None or args.detail:
            return x
        rf = x["roofline"]
        return {"ms_per_step": x["ms_per_step"], "value": x["value"], "unit": x["unit"],
                "roofline": {"kernel": rf["kernel"], "achieved": rf["achieved"], "peak": rf["peak"],
                             "frac": rf["frac"], "traffic": rf["traffic"]}}

    line["decode_sglang"] = compact_decode(decode_sglang)
    line["decode_gated"] = compact_decode(decode_gated)
    line["decode"] = compact_decode(decode)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_decode(args, dev, world, peaks, peak_src, gated=False, sglang=False):
    """Times the decode step; ``gated`` runs gdn_recurrent_step_gated (raw q/k
    and gate projections in, front-end in the kernel) instead; ``sglang`` adds
    the packed SGLang kernel's precision (bf16 state cache, bf16 beta)."""
    from gated_deltanet_chunked_gb300 import gdn

    w = DECODE
    state = W.make_decode_state(w).to(dev)
    if sglang:
        state = state.to(torch.bfloat16)
    make = W.make_decode_step_gated if gated else W.make_decode_step
    sets = []
    for s in range(4):
        inp = make(w, s)
        sets.append({k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()})
    out = torch.empty_like(sets[0]["v"])
    A_log, dt_bias = (t.to(dev) for t in W.make_decode_gate_params(w))
    z, norm_w = (t.to(dev) for t in W.make_output_gate(w.seed, w.num_seqs, w.hv, w.io_dtype))

    def step(i):
        x = sets[i % len(sets)]
        if gated:
            gdn.gdn_recurrent_step_gated(x["q"], x["k"], x["v"], x["a"], x["b"], A_log, dt_bias, x["scale"],
                                         state, out=out, z=z, norm_weight=norm_w, norm_eps=1e-6, beta_bf16=sglang)
        else:
            gdn.gdn_recurrent_step(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], state, out=out)

    for i in range(max(3, args.warmup)):
        step(i)
    steps = max(10, min(args.steps, 100))
    gdn.gdn_profile_collect(reset=True)
    gdn.gdn_profile_enable(True)
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        e0[i].record()
        step(i)
        e1[i].record()
    torch.cuda.synchronize()
    barrier(world)
    gdn.gdn_profile_enable(False)
    prof = gdn.gdn_profile_collect(reset=True)
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(e0, e1)) / steps, world, dev)
    n_pairs = w.num_seqs * w.hv
    state_bytes = 2 * n_pairs * 128 * 128 * state.element_size()
    # q, k, v, out in bf16; g, beta (or a, b) f32 per (sequence, v-head); A_log, dt_bias f32 per v-head
    # gated: + z (bf16, like v) per (sequence, v-head) and the 128-float norm weight
    io_bytes = w.num_seqs * (w.hq * 128 * 2 * 2 + w.hv * 128 * 2 * 2 + w.hv * 8)
    if gated:
        io_bytes += w.hv * 8 + w.num_seqs * w.hv * 128 * 2 + 128 * 4
    total = state_bytes + io_bytes
    kname = "recurrent_step_gated" if gated else "recurrent_step"
    n, kms, nt = prof.get(kname, (0, 0.0, 0))
    k_ms = kms / max(nt, 1)
    return {
        "workload": w.name, "steps": steps, "ms_per_step": ms, "value": world * total / (ms * 1e-3) / 1e9,
        "unit": "GB/s", "state_bytes_per_step": state_bytes, "bytes_per_step": total,
        "inputs": ("raw q/k, gate projections a/b, A_log/dt_bias, output gate z + RMSNorm weight "
                   "(front-end and output gate in the kernel)" if gated else "normalised q/k, g, beta")
                  + ("; bf16 state cache, bf16 beta" if sglang else "; f32 state"),
        "roofline": {"kernel": kname, "bound": "hbm", "achieved": total / (k_ms * 1e-3) / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": total / (k_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                     "traffic": ncu_traffic(kname + ("_bf16state" if sglang else "")),
                     "peak_source": f"{peak_src} (hbm_gbs, burst copy)"},
        "l2": f"state ({state.numel() * state.element_size() / 1e6:.0f} MB) larger than L2; no flush",
    }


def run_prefill_configs(args, dev, world, peaks, peak_src):
    """Times the plain prefill on the two other prefill workloads: 8 packed
    sequences of U[100, 8000] tokens with initial states, and one T=65536
    sequence. Each reports its step time, tokens/s and the fraction of the
    path's roofline max(bytes / HBM peak, FLOPs / bf16 peak), as the main
    line does for T=4096."""
    from gated_deltanet_chunked_gb300 import gdn

    res = {}
    flush = L2Flush(dev)
    for name in ("varlen_8seq_hq16_hv32", "long_T65536_hq16_hv32"):
        w = W.WORKLOADS[name]
        host = W.make_prefill(w)
        T, N = host["total_tokens"], host["num_seqs"]
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
        cu = d["cu_seqlens"] if d.get("cu_seqlens") is not None else torch.tensor([0, T], dtype=torch.int32,
                                                                                   device=dev)
        lens = (cu[1:] - cu[:-1]).tolist()
        s0 = d.get("initial_state")
        out = torch.empty_like(d["v"])
        fin = torch.empty((N, w.hv, 128, 128), dtype=torch.float32, device=dev)
        prob = gdn.prefill_problem(d["q"], d["v"], N, packed=True)
        ws = torch.empty(gdn.gdn_chunk_fwd_workspace_size(prob), dtype=torch.uint8, device=dev)

        def step():
            gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], initial_state=s0,
                              cu_seqlens=cu, out=out, final_state=fin, workspace=ws)

        for _ in range(max(3, args.warmup)):
            flush()
            step()
        torch.cuda.synchronize()
        assert gdn.gdn_read_device_status() == gdn.GDN_OK
        steps = max(5, min(args.steps, 30))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        barrier(world)
        torch.cuda.synchronize()
        for a, b in ev:
            flush()
            a.record()
            step()
            b.record()
        torch.cuda.synchronize()
        ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / steps, world, dev)
        nbytes = prefill_bytes(T, N, w.hq, w.hv, s0=s0 is not None)
        flops = prefill_flops(sum(math.ceil(n / 64) for n in lens) * w.hv, w.hv, w.hq)
        t_roof = max(nbytes / (peaks["hbm_gbs"] * 1e9), flops / (peaks["bf16_tflops"] * 1e12))
        res[name] = {"ms_per_step": ms, "value": world * T / (ms * 1e-3), "unit": "tokens/s", "tokens": T,
                     "sequences": N, "longest": max(lens), "initial_state": s0 is not None,
                     "path_bytes": nbytes, "path_flops": flops, "roofline_us": t_roof * 1e6,
                     "frac_of_roofline": t_roof / (ms * 1e-3), "peak_source": peak_src, "l2": L2_NOTE}
        del d, out, fin, ws, host
        torch.cuda.empty_cache()
    return res


def run_prefill_gated(args, dev, world):
    """Times the T=4096 prefill step with the output gate fused in
    (gdn_chunk_fwd_gated) the way the main line times the plain step."""
    from gated_deltanet_chunked_gb300 import gdn

    w = PREFILL
    host = W.make_prefill(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    z, weight = (t.to(dev) for t in W.make_output_gate(w.seed, w.seqlen, w.hv, w.io_dtype))
    T = host["total_tokens"]
    out = torch.empty_like(d["v"])
    fin = torch.empty((1, w.hv, 128, 128), dtype=torch.float32, device=dev)
    prob = gdn.prefill_problem(d["q"], d["v"], 1, packed=True)
    ws = torch.empty(gdn.gdn_chunk_fwd_workspace_size(prob), dtype=torch.uint8, device=dev)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    flush = L2Flush(dev)

    def step():
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], cu_seqlens=cu, out=out,
                          final_state=fin, workspace=ws, z=z, norm_weight=weight, norm_eps=1e-6)

    for _ in range(max(3, args.warmup)):
        flush()
        step()
    steps = max(10, min(args.steps, 100))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for a, b in ev:
        flush()
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / steps, world, dev)
    return {"workload": f"{w.name} + output gate", "ms_per_step": ms, "value": world * T / (ms * 1e-3),
            "unit": "tokens/s", "l2": L2_NOTE, "traffic": ncu_traffic("chunk_fused_tc_gated"),
            "what": "prefill with RMSNorm(o) * weight * silu(z) applied in the fused kernel (gdn_chunk_fwd_gated)"}


def graph_ms_per_launch(launch, n, reps=3):
    """Device time per launch of launch(0) .. launch(n - 1), captured back to
    back in one CUDA graph and replayed `reps` times between one pair of CUDA
    events. A kernel of a few microseconds timed by its own event pair on an
    idle stream also counts the host's launch latency (the start event is
    taken before the launch reaches the GPU); inside a graph the launches
    follow each other on the device."""
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        for i in range(n):
            launch(i)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (reps * n)
    del g
    return ms


def roofline_hbm(kname, total, k_ms, peaks, peak_src):
    return {"kernel": kname, "bound": "hbm", "achieved": total / (k_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": total / (k_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], "traffic": ncu_traffic(kname),
            "peak_source": f"{peak_src} (hbm_gbs, burst copy)"}


def run_gate_norm(args, dev, world, peaks, peak_src):
    """Times gdn_gated_rmsnorm over the prefill workload's read-out tensor
    [4096, 32, 128] bf16 (o, z in; y out). Launches rotate over four sets of
    (o, z, y), 403 MB in all, so each launch finds its inputs evicted from L2
    by the three launches before it (a write flush would instead leave 126 MB
    of dirty lines whose write-back this streaming kernel would pay for)."""
    from gated_deltanet_chunked_gb300 import gdn

    w = PREFILL
    sets = []
    for i in range(4):
        z, weight, o = (t.to(dev) for t in W.make_output_gate(w.seed + 97 * i, w.seqlen, w.hv, w.io_dtype,
                                                                with_o=True))
        sets.append((o, z, weight, torch.empty_like(o)))
    for i in range(max(3, args.warmup)):
        o, z, weight, y = sets[i % 4]
        gdn.gdn_gated_rmsnorm(o, z, weight, 1e-6, out=y)
    steps = max(12, min(args.steps, 100))
    gdn.gdn_profile_collect(reset=True)
    gdn.gdn_profile_enable(True)
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        o, z, weight, y = sets[i % 4]
        gdn.gdn_gated_rmsnorm(o, z, weight, 1e-6, out=y)
    torch.cuda.synchronize()
    barrier(world)
    gdn.gdn_profile_enable(False)
    prof = gdn.gdn_profile_collect(reset=True)
    n, kms, nt = prof.get("gated_rmsnorm", (0, 0.0, 0))
    ev_ms = max_over_ranks(kms / max(nt, 1), world, dev)

    def launch(i):
        o, z, weight, y = sets[i % 4]
        gdn.gdn_gated_rmsnorm(o, z, weight, 1e-6, out=y)
    barrier(world)
    k_ms = max_over_ranks(graph_ms_per_launch(launch, 16), world, dev)
    total = 3 * o.numel() * o.element_size() + 128 * 4
    return {
        "workload": f"{w.name} read-out", "rows": w.seqlen * w.hv, "steps": steps, "ms_per_launch": k_ms,
        "ms_per_launch_own_events": ev_ms,
        "value": world * total / (k_ms * 1e-3) / 1e9, "unit": "GB/s", "bytes_per_launch": total,
        "roofline": roofline_hbm("gated_rmsnorm", total, k_ms, peaks, peak_src),
        "timing": "16 launches back to back in a CUDA graph, 3 replays between two CUDA events",
        "l2": "inputs rotate over 4 sets of o, z, y (403 MB, larger than L2); no flush",
    }


def run_front_end(args, dev, world, peaks, peak_src):
    """Times the short convolution (gdn_causal_conv1d_silu, q/k norm fused) on
    the prefill workload's projections (T = 4096, C = 8192 bf16, with state)
    and on one decode step (256 sequences), and the per-token gating, each
    rotating over input sets larger than L2."""
    from gated_deltanet_chunked_gb300 import gdn

    res = {}
    hq, hv = PREFILL.hq, PREFILL.hv
    for name, T, N in (("conv_prefill_T4096", PREFILL.seqlen, 1), ("conv_decode_N256", DECODE.num_seqs,
                                                                    DECODE.num_seqs)):
        nsets = 4 if N == 1 else 16
        sets = []
        for i in range(nsets):
            x, w, b, st = W.make_conv_inputs(7000 + i, T, hq, hv, PREFILL.io_dtype, slots=N)
            cu = torch.arange(N + 1, dtype=torch.int32) if N > 1 else torch.tensor([0, T], dtype=torch.int32)
            q = torch.empty((T, hq, 128), dtype=x.dtype, device=dev)
            k, v = torch.empty_like(q), torch.empty((T, hv, 128), dtype=x.dtype, device=dev)
            sets.append([t.to(dev) for t in (x, w, b, st, cu)] + [q, k, v])

        def launch(i):
            x, w, b, st, cu, q, k, v = sets[i % nsets]
            if N > 1:  # one token per sequence: the decode step kernel
                gdn.gdn_causal_conv1d_silu_step(x, w, hq, hv, bias=b, conv_state=st, norm_qk=True, q=q, k=k, v=v)
            else:
                gdn.gdn_causal_conv1d_silu(x, w, hq, hv, bias=b, conv_state=st, cu_seqlens=cu, norm_qk=True,
                                           q=q, k=k, v=v)
        for i in range(max(3, args.warmup)):
            launch(i)
        steps = max(16, min(args.steps, 100))
        gdn.gdn_profile_collect(reset=True)
        gdn.gdn_profile_enable(True)
        torch.cuda.synchronize()
        for i in range(steps):
            launch(i)
        torch.cuda.synchronize()
        gdn.gdn_profile_enable(False)
        prof = gdn.gdn_profile_collect(reset=True)
        kname = "conv1d_step" if N > 1 else "conv1d_silu"
        _, kms, nt = prof.get(kname, (0, 0.0, 0))
        ev_ms = max_over_ranks(kms / max(nt, 1), world, dev)
        barrier(world)
        k_ms = max_over_ranks(graph_ms_per_launch(launch, 2 * nsets), world, dev)
        C = (2 * hq + hv) * 128
        # x in, q/k/v out (bf16); conv state 3 rows read + written per sequence; weight and bias (f32)
        total = 2 * T * C * 2 + 2 * N * 3 * C * 2 + C * 4 * 4 + C * 4
        res[name] = {"ms_per_launch": k_ms, "ms_per_launch_own_events": ev_ms, "bytes_per_launch": total,
                     "roofline": roofline_hbm(kname, total, k_ms, peaks, peak_src),
                     "timing": f"{2 * nsets} launches back to back in a CUDA graph, 3 replays between two CUDA events",
                     "l2": f"inputs rotate over {nsets} sets; no flush"}
        del sets
    # gating of every token of the prefill workload ([4096, 32] a, b in; g, beta out)
    T = PREFILL.seqlen
    A_log, dt_bias = (t.to(dev) for t in W.make_decode_gate_params(DECODE))
    gs = [tuple(torch.randn((T, hv), device=dev) for _ in range(4)) for _ in range(4)]
    for i in range(3):
        a, b, g, beta = gs[i % 4]
        gdn.gdn_gating(a, b, A_log, dt_bias, g=g, beta=beta)
    gdn.gdn_profile_collect(reset=True)
    gdn.gdn_profile_enable(True)
    for i in range(20):
        a, b, g, beta = gs[i % 4]
        gdn.gdn_gating(a, b, A_log, dt_bias, g=g, beta=beta)
    torch.cuda.synchronize()
    gdn.gdn_profile_enable(False)
    _, kms, nt = gdn.gdn_profile_collect(reset=True).get("gating", (0, 0.0, 0))

    def launch_g(i):
        a, b, g, beta = gs[i % 4]
        gdn.gdn_gating(a, b, A_log, dt_bias, g=g, beta=beta)
    k_ms = max_over_ranks(graph_ms_per_launch(launch_g, 16), world, dev)
    res["gating_T4096"] = {"ms_per_launch": k_ms, "ms_per_launch_own_events": max_over_ranks(kms / max(nt, 1), world, dev),
                           "bytes_per_launch": 4 * T * hv * 4,
                           "bound": "launch / latency (2 MB per launch; the 4 rotating sets, 8 MB, stay in L2)"}
    res["peak_source"] = f"{peak_src} (hbm_gbs, burst copy)"
    return res


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, where Arm hosts
    list only implementer/part numbers) and the processor count."""
    name = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                name = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read() if name is None else ""
        for key in ("model name", "Model name", "Hardware", "CPU part"):
            for line in info.splitlines():
                if line.split(":")[0].strip() == key:
                    name = line.split(":", 1)[1].strip()
                    break
            if name:
                break
    except OSError:
        pass
    arm_parts = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd0c": "Arm Neoverse-N1",
                 "0xd49": "Arm Neoverse-N2"}
    name = arm_parts.get(name, name)
    return {"model": name or "unknown", "nproc": os.cpu_count()}


def _oracle_rate(fn, host, nk, G, min_seconds, max_passes=50):
    """Tokens/s of one oracle routine over all tokens of the first nk q/k head
    groups (nk * G v-heads), scaled to the whole workload by the head
    fraction, with whole passes repeated until `min_seconds` have passed."""
    T = host["total_tokens"]
    q, k = host["q"][:, :nk], host["k"][:, :nk]
    v, g, beta = host["v"][:, :nk * G], host["g"][:, :nk * G], host["beta"][:, :nk * G]
    passes, t0 = 0, time.perf_counter()
    while passes < max_passes and (passes == 0 or time.perf_counter() - t0 < min_seconds):
        fn(q, k, v, g, beta, host["scale"], None, [0, T])
        passes += 1
    dt = time.perf_counter() - t0
    hq = host["q"].shape[1]
    return {"tokens_per_s": passes * T * (nk / hq) / dt, "passes": passes, "seconds": dt,
            "v_heads": nk * G}


def cpu_baseline(host, w, min_seconds=2.5):
    """The CPU oracle as it stands on this host's cores: the token-by-token
    recurrence (R) and the chunk form (Ch), each on one thread and on every
    core. One thread runs a sample of one q/k head group (2 of 32 v-heads,
    all tokens); all cores run every head. Rates are whole-workload tokens/s
    (the one-thread sample scaled by its head fraction). `value` is Ch on all
    cores, the routine and setting the reference arm times."""
    import oracle

    G = w.hv // w.hq
    oracle.build()
    procs = oracle.num_procs()
    legs = {}
    for threads, nk in ((1, 1), (procs, w.hq)):
        oracle.set_threads(threads)
        for name, fn in (("R", oracle.recurrent), ("Ch", oracle.chunked)):
            legs[f"{name}_{'1thread' if threads == 1 else 'all_cores'}"] = {
                **_oracle_rate(fn, host, nk, G, min_seconds), "threads": threads}
    oracle.set_threads(procs)
    best = legs["Ch_all_cores"]
    T = host["total_tokens"]
    return {"value": best["tokens_per_s"], "unit": "tokens/s", "cores": procs, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": (f"f64 oracle on this host: R and Ch over all {T} tokens; one thread on 1 of {w.hq} q/k head "
                       f"groups ({G} v-heads, rate scaled by the head fraction), all {procs} cores on all "
                       f"{w.hv} v-heads; passes repeated for >= {min_seconds} s each; value = Ch on all cores"),
            "legs": {k: {"tokens_per_s": v["tokens_per_s"], "threads": v["threads"], "v_heads": v["v_heads"],
                         "passes": v["passes"], "seconds": round(v["seconds"], 2)} for k, v in legs.items()}}


# --------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands
# --------------------------------------------------------------------------
def run_reference(args, world, rank):
    """Times the chunk-form oracle (f64, OpenMP on every host core) on the
    whole T=4096 workload, every head, once per step: ms_per_step is the
    measured time of what ran, value the median step's tokens/s."""
    if rank != 0:
        return
    import oracle

    w = PREFILL
    host = W.make_prefill(w)
    T = host["total_tokens"]
    oracle.build()
    procs = oracle.num_procs()
    oracle.set_threads(procs)
    run = lambda: oracle.chunked(host["q"], host["k"], host["v"], host["g"], host["beta"], host["scale"], None,
                                 [0, T])
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        run()
        times.append(time.perf_counter() - t)
    sec = statistics.median(times)
    value = T / sec
    sample = (f"chunk-form oracle (f64, OpenMP, {procs} threads) per step over the whole workload: all {T} tokens, "
              f"all {w.hv} v-heads; median of {args.steps} timed steps")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": 1, "T": T, "hq": w.hq, "hv": w.hv, "dk": 128, "dv": 128, "chunk": 64},
        "step_ms": {"median": sec * 1e3, "mean": statistics.mean(times) * 1e3, "min": min(times) * 1e3,
                    "max": max(times) * 1e3},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": procs, "kind": "oracle", "sample": sample,
                         "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the varlen and T=65536 prefill legs")
    ap.add_argument("--detail", action="store_true", help="full per-kernel and per-leg objects in the JSON line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
