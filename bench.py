"""Benchmark of the chunked Q-Delta forward on GB300 (one JSON line on rank 0).

Workload of a step: one qdelta_fwd over one batch of the 1.3B-model layer shape,
B=8, H=16, T=2048, dk=dv=128, bf16 inputs, fp32 state, full Q-Delta gates
(alpha, beta, lambda), synthetic seeded inputs (synth.layer_1p3b).

  value    tokens/s (B*T per step, summed over ranks) from CUDA events around
           exactly K steps on the launching stream, inputs resident in HBM and
           larger than L2, rotated over several buffer sets between steps
  e2e      the same metric through the C ABI with pinned HOST buffers: every step
           copies its inputs host->device and its outputs (o, S_final) back, steps
           pipelined over three streams (copy in / compute / copy out)
  roofline the dominant kernel against the measured HBM copy bandwidth
  tensor   its GEMM work against the measured bf16 tensor peak
  decode   qdelta_step on 512 sequences x 16 heads (fp32 128x128 state), GB/s
  qed_decode  qed_step on the same shape, GB/s
  qed      qed_fwd at B=4, H=8, T=4096, d=128 bf16, tokens/s, against HBM
  deltanet, gdn  qdelta_fwd on the step's workload with alpha and lambda dropped
           (DeltaNet) or lambda dropped (Gated DeltaNet), against HBM
  long_context  qdelta_fwd at B=1, H=16, T=32768 (mean alpha 0.995, S0 != 0),
           the segment scan, against HBM
  prologue qdelta_fwd_prologue on the step's workload (projections and logits in)
  eda      eda_fwd (erase-then-delta) on the step's shape, tokens/s
  backward qdelta_bwd on the step's workload (all input gradients), against the
           TF32 tensor peak its products run on
  cpu_baseline  the fp64 oracle timed on this host's cores on a bounded sample
  clocks   nvidia-smi samples over the timed K steps and about 0.6 s of the same
           back-to-back steps (untimed) on either side of them

--impl reference times the oracle itself (the CPU reference of this build) on
a bounded sample of the same workload each step, and prints the same line.
Multi-GPU: replicas (each rank runs its own batch; no data-path collective).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "chunked Q-Delta fwd tokens/s at H=16,d=128,T=2048; % tensor peak; step GB/s"
B, T, H, DK, DV, CHUNK = 8, 2048, 16, 128, 128, 64
TOKEN_HEADS = B * T * H
# algorithmic bytes of one forward: q, k, v, o in bf16 + alpha, beta, lambda in bf16
# per token-head, + the fp32 final state
BYTES_PER_TOKEN_HEAD = 2 * (DK + DK + DV + DV) + 3 * 2
ALG_BYTES = TOKEN_HEADS * BYTES_PER_TOKEN_HEAD + B * H * DV * DK * 4
# GEMM work per token-head at chunk C: Grams 4Cd + solve-apply 2Cd + intra output 2Cd
# + the three state products 6 d^2  (= 8Cd + 6d^2 with d = dk = dv)
FLOPS_PER_TOKEN_HEAD = 8 * CHUNK * DK + 6 * DK * DV
ALG_FLOPS = TOKEN_HEADS * FLOPS_PER_TOKEN_HEAD
N_BUFFERS = 3
SOAK_S = 0.6     # untimed back-to-back steps around the timed region, for the clock samples


def mode_bytes(mode, token_heads, heads):
    """Algorithmic bytes of one forward in a gate mode: q, k, v, o in bf16, the gates the
    mode reads (beta always; alpha unless DeltaNet; lambda only for Q-Delta) in bf16, and
    the fp32 final state (plus the fp32 initial state when one is read)."""
    gates = {"deltanet": 1, "gdn": 2, "qdelta": 3}[mode]
    return token_heads * (2 * (DK + DK + DV + DV) + 2 * gates) + heads * DV * DK * 4
DOMINANT_KERNEL_SOURCES = ["delta_rule_linear_qdelta_gb300/csrc/chunk_tc.cu",
                           "delta_rule_linear_qdelta_gb300/csrc/tc_common.cuh",
                           "delta_rule_linear_qdelta_gb300/csrc/sm103_ptx.cuh"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_hash():
    h = hashlib.sha256()
    for rel in DOMINANT_KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    return h.hexdigest()[:16]


def traffic_from_profile():
    """DRAM bytes per launch from the committed ncu summary, if it matches the kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    ent = d.get("qdelta_fwd_bf16_B8_H16_T2048_d128")
    if not ent or ent.get("source_hash") != kernel_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        win = [s for t, s in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        if not win:   # a timed region shorter than the sampling period: nearest samples
            mid = 0.5 * (t0 + t1)
            win = [min(self.samples, key=lambda ts: abs(ts[0] - mid))[1]]
        sm = [float(s[1]) for s in win if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in win if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in win for n, v in zip(names, s[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win)}


def dist_setup(n_gpus):
    import torch
    if n_gpus > 1 or int(os.environ.get("WORLD_SIZE", "1")) > 1:
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        return rank, int(os.environ["WORLD_SIZE"]), local
    torch.cuda.set_device(0)
    return 0, 1, 0


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """Max of a per-rank scalar over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(ms_per_step, world):
    """Whole-job throughput: every rank processes its own B*T-token batch per step."""
    return B * T * world / (ms_per_step * 1e-3)


def to_dev(x, dtype):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).to("cuda", dtype)


def make_buffers(n_sets, seed_base=1):
    """n_sets independent input sets of the workload, resident on the device."""
    import torch
    sets = []
    for i in range(n_sets):
        d = synth.qdelta_inputs(B, T, H, DK, DV, seed=seed_base + 1000 * i, dtype="bf16", mode="qdelta")
        sets.append({k: to_dev(d[k], torch.bfloat16) for k in ("q", "k", "v", "alpha", "beta", "lam")})
    return sets


def soak(step, seconds):
    """Back-to-back untimed steps for about `seconds` of wall time (keeps the GPU under
    the timed workload's load while the clocks are sampled)."""
    import torch
    if seconds <= 0:
        return
    t0 = time.time()
    i = 0
    while time.time() - t0 < seconds:
        for _ in range(50):
            step(i)
            i += 1
        torch.cuda.synchronize()


def time_device(qd, sets, steps, warmup, world, mode="qdelta", soak_s=0.0):
    """Times exactly `steps` forwards after `warmup` untimed ones (plus `soak_s` seconds
    of untimed steps on either side when asked, for the clock samples).  Returns the
    event-timed total, the mean per-launch time, the kernels launched and the wall
    window (soak included)."""
    import torch
    o = torch.empty(B, T, H, DV, dtype=torch.bfloat16, device="cuda")
    S = torch.empty(B, H, DV, DK, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    use_a, use_l = mode != "deltanet", mode == "qdelta"

    def step(i):
        s = sets[i % len(sets)]
        qd.qdelta_fwd(s["q"], s["k"], s["v"], s["alpha"] if use_a else None, s["beta"], s["lam"] if use_l else None,
                      None, o=o, S_final=S, stream=stream)
        return qd.last_launch_count()

    for i in range(warmup):
        step(i)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    soak(step, soak_s)
    barrier(world)
    torch.cuda.synchronize()
    launches = 0
    start.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        launches += step(warmup + i)
        ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    soak(step, soak_s)
    t_wall1 = time.time()
    total_ms = start.elapsed_time(end)
    per_launch_ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    return total_ms, per_launch_ms, launches, (t_wall0, t_wall1)


def hbm_roofline(nbytes, kernel_ms, hbm_peak, peak_kind, flops=None, tc_peak=None):
    gbs = nbytes / (kernel_ms * 1e-3) / 1e9
    r = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
         "peak_kind": peak_kind, "alg_bytes_per_launch": nbytes, "kernel_ms": kernel_ms}
    if flops is not None:
        tf = flops / (kernel_ms * 1e-3) / 1e12
        r["tensor"] = {"achieved": tf, "peak": tc_peak, "unit": "TFLOP/s", "frac": tf / tc_peak,
                       "alg_flops_per_launch": flops}
    return r


def time_mode(qd, sets, mode, hbm_peak, tc_peak, peak_kind, steps=50, warmup=5):
    """qdelta_fwd on the step's workload in one of the special-case gate modes."""
    total_ms, launch_ms, launches, _ = time_device(qd, sets, steps, warmup, 1, mode=mode)
    ms = total_ms / steps
    nbytes = mode_bytes(mode, TOKEN_HEADS, B * H)
    return {"workload": f"{mode}_bf16_B{B}_H{H}_T{T}_d{DK}", "ms_per_step": ms, "tokens_per_s": B * T / (ms * 1e-3),
            "launches_per_step": launches / steps,
            "roofline": hbm_roofline(nbytes, launch_ms, hbm_peak, peak_kind, TOKEN_HEADS * FLOPS_PER_TOKEN_HEAD,
                                     tc_peak)}


def time_long_context(qd, hbm_peak, tc_peak, peak_kind, steps=20, warmup=3):
    """qdelta_fwd at B=1, H=16, T=32768, d=128 bf16, mean alpha 0.995, S0 ~ N(0, 0.01):
    the segment scan (a workspace from the caller).  q, k, v, o are 128 MiB each, so
    the inputs do not fit in L2."""
    import torch
    name, d = synth.long_context()
    bf = torch.bfloat16
    args = [to_dev(d[k], bf) for k in ("q", "k", "v", "alpha", "beta", "lam")]
    S0 = to_dev(d["S0"], torch.float32)
    Bl, Tl, Hl = d["q"].shape[:3]
    o = torch.empty(Bl, Tl, Hl, DV, dtype=bf, device="cuda")
    S = torch.empty(Bl, Hl, DV, DK, dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, qd.qdelta_workspace_bytes(Bl, Tl, Hl, DK, DV)), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        qd.qdelta_fwd(*args, S0, o=o, S_final=S, workspace=ws, stream=stream)

    for _ in range(warmup):
        step()
    launches = qd.last_launch_count()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    call_ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    th = Bl * Tl * Hl
    nbytes = mode_bytes("qdelta", th, Bl * Hl) + Bl * Hl * DV * DK * 4     # + the fp32 S0 read
    return {"workload": name, "ms_per_step": ms, "tokens_per_s": Bl * Tl / (ms * 1e-3),
            "launches_per_step": launches,
            "segments": max(1, ws.numel() // (3 * Bl * Hl * DV * DK * 4)) if launches > 1 else 1,
            "roofline": hbm_roofline(nbytes, call_ms, hbm_peak, peak_kind, th * FLOPS_PER_TOKEN_HEAD, tc_peak)}


def time_e2e(qd, steps, warmup, world):
    """Host buffers in pinned memory; every step copies its inputs in and its results
    (o, S_final) out, all inside the timed region.  Steps are pipelined the way a
    serving loop runs them: step i+1's inputs travel host -> device on one stream while
    step i computes on a second and step i-1's results travel back on a third, with two
    device buffer sets and events ordering each set's reuse."""
    import torch
    d = synth.qdelta_inputs(B, T, H, DK, DV, seed=5, dtype="bf16", mode="qdelta")
    names = ("q", "k", "v", "alpha", "beta", "lam")
    host = {k: torch.from_numpy(d[k]).to(torch.bfloat16).pin_memory() for k in names}
    devb = [{k: torch.empty_like(v, device="cuda") for k, v in host.items()} for _ in range(2)]
    o = [torch.empty(B, T, H, DV, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    S = [torch.empty(B, H, DV, DK, dtype=torch.float32, device="cuda") for _ in range(2)]
    o_h = [torch.empty(o[0].shape, dtype=o[0].dtype).pin_memory() for _ in range(2)]
    S_h = [torch.empty(S[0].shape, dtype=S[0].dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o[0].numel() * o[0].element_size() + S[0].numel() * S[0].element_size()
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    in_done = [torch.cuda.Event() for _ in range(2)]
    cmp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(cmp_done[b])              # step i-2 has read this input set
            for k in names:
                devb[b][k].copy_(host[k], non_blocking=True)
            in_done[b].record(s_in)
        s_cmp.wait_event(in_done[b])
        if i >= 2:
            s_cmp.wait_event(out_done[b])                 # step i-2's results have left this set
        x = devb[b]
        qd.qdelta_fwd(x["q"], x["k"], x["v"], x["alpha"], x["beta"], x["lam"], None, o=o[b], S_final=S[b],
                      stream=s_cmp)
        cmp_done[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(cmp_done[b])
            o_h[b].copy_(o[b], non_blocking=True)
            S_h[b].copy_(S[b], non_blocking=True)
            out_done[b].record(s_out)

    for i in range(warmup):
        step(i)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    start.record(s_in)
    for i in range(steps):
        step(warmup + i)
    for b in range(2):
        s_in.wait_event(out_done[b])                      # the end waits for every step's results
    end.record(s_in)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(end) / steps, world)
    return {"value": B * T * world / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "pipeline": "inputs in, compute, results out on three streams, two buffer sets"}


def time_decode(qd, steps=50, warmup=5, N=512):
    import torch
    d = synth.decode_inputs(N, 16, 128, 128, 4, seed=4, dtype="bf16", s0_var=None)
    S = torch.empty(N, 16, 128, 128, dtype=torch.float32, device="cuda").normal_(0, 0.1)
    tok = [{k: to_dev(d[k][i], torch.bfloat16) for k in ("q", "k", "v", "alpha", "beta", "lam")} for i in range(4)]
    o = torch.empty(N, 16, 128, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i):
        t = tok[i % 4]
        qd.qdelta_step(S, t["q"], t["k"], t["v"], t["alpha"], t["beta"], t["lam"], o=o, stream=stream)

    for i in range(warmup):
        step(i)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    heads = N * 16
    nbytes = heads * (2 * 128 * 128 * 4 + 2 * (128 + 128 + 128 + 128) + 3 * 2)
    return {"workload": f"qdelta_step_bf16_N{N}_H16_d128", "ms_per_step": ms, "tokens_per_s": N / (ms * 1e-3),
            "bytes_per_step": nbytes, "GBps": nbytes / (ms * 1e-3) / 1e9}


def time_qed_decode(qd, steps=50, warmup=5, N=512):
    """qed_step on N sequences x 16 heads, fp32 128x128 state (the decode shape)."""
    import torch
    d = synth.qed_decode_inputs(N, 16, 128, 128, 4, seed=6, dtype="bf16", s0_var=None)
    S = torch.empty(N, 16, 128, 128, dtype=torch.float32, device="cuda").normal_(0, 0.1)
    tok = [{k: to_dev(d[k][i], torch.bfloat16) for k in ("q", "k", "v", "g", "b", "w")} for i in range(4)]
    lam_h = to_dev(d["lam_h"], torch.float32)
    o = torch.empty(N, 16, 128, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i):
        t = tok[i % 4]
        qd.qed_step(S, t["q"], t["k"], t["v"], t["g"], t["b"], t["w"], lam_h, o=o, stream=stream)

    for i in range(warmup):
        step(i)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(steps):
        step(i)
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    heads = N * 16
    nbytes = heads * (2 * 128 * 128 * 4 + 2 * (4 * 128 + 3 * 128))
    return {"workload": f"qed_step_bf16_N{N}_H16_d128", "ms_per_step": ms, "tokens_per_s": N / (ms * 1e-3),
            "bytes_per_step": nbytes, "GBps": nbytes / (ms * 1e-3) / 1e9}


def time_qed(qd, hbm_peak, tc_peak, peak_kind, steps=20, warmup=3):
    import torch
    _, d = synth.qed_gdn2()
    bf = torch.bfloat16
    args = [to_dev(d[k], bf) for k in ("q", "k", "v", "g", "b", "w")] + [to_dev(d["lam_h"], torch.float32)]
    o = torch.empty(4, 4096, 8, 128, dtype=bf, device="cuda")
    S = torch.empty(4, 8, 128, 128, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        qd.qed_fwd(*args, o=o, S_final=S, stream=stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        qd.qed_fwd(*args, o=o, S_final=S, stream=stream)
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    th = 4 * 4096 * 8
    # q, k, v, g, b, w and o in bf16 (seven d-vectors) per token-head, lambda_h, the fp32 final state
    nbytes = th * (2 * 7 * 128) + 8 * 4 + 4 * 8 * 128 * 128 * 4
    return {"workload": "qed_bf16_B4_H8_T4096_d128", "ms_per_step": ms, "tokens_per_s": 4 * 4096 / (ms * 1e-3),
            "GBps": nbytes / (ms * 1e-3) / 1e9, "launches_per_step": qd.last_launch_count(),
            "roofline": hbm_roofline(nbytes, ms, hbm_peak, peak_kind, th * FLOPS_PER_TOKEN_HEAD, tc_peak)}


def time_prologue(qd, steps=20, warmup=3):
    """qdelta_fwd_prologue on the headline workload: q, k projections and gate logits
    in, feature map and gates computed inside the forward."""
    import torch
    d = synth.qdelta_raw_inputs(B, T, H, DK, DV, seed=7, dtype="bf16")
    bf = torch.bfloat16
    args = [to_dev(d[k], bf) for k in ("q", "k", "v", "alpha", "beta", "lam")]
    o = torch.empty(B, T, H, DV, dtype=bf, device="cuda")
    S = torch.empty(B, H, DV, DK, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        qd.qdelta_fwd(*args, None, o=o, S_final=S, stream=stream, prologue=True)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        qd.qdelta_fwd(*args, None, o=o, S_final=S, stream=stream, prologue=True)
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    return {"workload": f"qdelta_prologue_bf16_B{B}_H{H}_T{T}_d{DK}", "ms_per_step": ms,
            "tokens_per_s": B * T / (ms * 1e-3), "GBps": ALG_BYTES / (ms * 1e-3) / 1e9}


# Backward work per token-head (multiply-adds x 2), C = 64, d = dk = dv: the checkpoint
# forward (X S^T, Z^T K: 4 d^2; Grams and solve-apply 5 C d), the reverse sweep (dZ,
# dS update: 6 d^2; Grams, P^T dO, back substitution 7 C d) and the gradient kernel
# (XS, QS, K dS^T, the three S/dS products: 12 d^2; Grams, Z, dZ, dR, dA, dP and the
# four masked products: 22 C d).
BWD_FLOPS_PER_TOKEN_HEAD = 22 * DK * DV + 34 * CHUNK * DK



def time_bwd(qd, tc_peak, steps=5, warmup=3):
    """qdelta_bwd on the step's workload (B=8, H=16, T=2048, d=128, bf16), dO and
    dS_final ~ N(0,1)."""
    import torch
    _, d = synth.layer_1p3b()
    c = synth.cotangents(B, T, H, DK, DV, seed=8, dtype="bf16")
    bf = torch.bfloat16
    args = [to_dev(d[k], bf) for k in ("q", "k", "v", "alpha", "beta", "lam")]
    dO, dS = to_dev(c["dO"], bf), to_dev(c["dS_final"], torch.float32)
    ws = torch.empty(qd.qdelta_bwd_workspace_bytes(B, T, H, DK, DV), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        qd.qdelta_bwd(*args, None, dO, dS, workspace=ws, stream=stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        qd.qdelta_bwd(*args, None, dO, dS, workspace=ws, stream=stream)
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    tflops = TOKEN_HEADS * BWD_FLOPS_PER_TOKEN_HEAD / (ms * 1e-3) / 1e12
    peak = tc_peak                                    # its products are kind::f16 (bf16 and fp16 operands)
    return {"workload": f"qdelta_bwd_bf16_B{B}_H{H}_T{T}_d{DK}", "ms_per_step": ms,
            "tokens_per_s": B * T / (ms * 1e-3), "launches": qd.last_launch_count(),
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "peak_kind": "measured bf16 (fp16 runs at the same rate)",
                         "alg_flops_per_launch": TOKEN_HEADS * BWD_FLOPS_PER_TOKEN_HEAD}}


def time_eda(qd, steps=20, warmup=3):
    """eda_fwd on the step's shape (B=8, H=16, T=2048, d=128, bf16; random unit erase
    directions, beta = sigmoid(N(0,1)))."""
    import torch
    d = synth.eda_inputs(B, T, H, DK, DV, seed=9, dtype="bf16")
    bf = torch.bfloat16
    args = [to_dev(d[k], bf) for k in ("q", "k", "v", "e", "beta")]
    o = torch.empty(B, T, H, DV, dtype=bf, device="cuda")
    S = torch.empty(B, H, DV, DK, dtype=torch.float32, device="cuda")
    ws = torch.empty(qd.eda_workspace_bytes(B, T, H, DK, DV), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        qd.eda_fwd(*args, None, o=o, S_final=S, workspace=ws, stream=stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        qd.eda_fwd(*args, None, o=o, S_final=S, workspace=ws, stream=stream)
    end.record(stream)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / steps
    nbytes = TOKEN_HEADS * (5 * DK * 2 + 2) + B * H * DV * DK * 4     # q, k, v, e, o and beta; S_final
    return {"workload": f"eda_bf16_B{B}_H{H}_T{T}_d{DK}", "ms_per_step": ms, "tokens_per_s": B * T / (ms * 1e-3),
            "GBps": nbytes / (ms * 1e-3) / 1e9, "launches": qd.last_launch_count()}


def oracle_sample(n_streams, seed=1, min_seconds=0.0):
    """Runs the fp64 oracle on n_streams (b, h) streams of the workload (full T) on
    all host cores, repeated until min_seconds have passed; returns
    (tokens/s equivalent, seconds per pass, cores, passes)."""
    import oracle
    d = synth.qdelta_inputs(1, T, n_streams, DK, DV, seed=seed, dtype="bf16", mode="qdelta")
    cores = os.cpu_count() or 1
    passes, t0 = 0, time.perf_counter()
    while True:
        oracle.qdelta_fwd(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["lam"], None, nthreads=cores)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    per = dt / passes
    return (n_streams * T / H) / per, per, min(cores, n_streams), passes


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    n_streams = 16
    for _ in range(args.warmup):
        oracle_sample(n_streams)
    times = []
    for _ in range(args.steps):
        _, dt, cores, _ = oracle_sample(n_streams)
        times.append(dt)
    sec = sum(times) / len(times)
    value = (n_streams * T / H) / sec
    sample = f"{n_streams} of {B * H} (b,h) streams at full T={T} per step (fp64, all host cores)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"qdelta_bf16_B{B}_H{H}_T{T}_d{DK}", "B": B, "T": T, "H": H, "dk": DK,
                       "dv": DV, "chunk": CHUNK},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="skip the decode / QED / e2e / CPU legs")
    ap.add_argument("--profile", nargs="?", const="fwd",
                    choices=["fwd", "bwd", "eda", "decode", "qed_decode", "qed", "long"],
                    help="profiling case: run warmup + steps calls of one leg untimed (fwd: the step's "
                         "forward; bwd, eda, decode, qed_decode, qed, long: those legs' workloads), "
                         "print no JSON line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
        return

    import torch
    import delta_rule_linear_qdelta_gb300 as qd
    if not os.path.exists(qd.LIB_PATH):
        from delta_rule_linear_qdelta_gb300 import build
        build.build()
    rank, world, local = dist_setup(args.gpus)
    hbm_peak, tc_peak, tc_sustained, peak_kind = load_peaks()
    if args.profile == "fwd":
        sets = make_buffers(1, seed_base=1 + rank)
        time_device(qd, sets, args.steps, args.warmup, world)
        torch.cuda.synchronize()
        print(f"profile case done: {args.warmup + args.steps} forwards, status {qd.qd_device_status()}", flush=True)
        return
    if args.profile == "eda":
        time_eda(qd, steps=args.steps, warmup=args.warmup)
        print(f"profile case done: {args.warmup + args.steps} EDA forwards, status {qd.qd_device_status()}",
              flush=True)
        return
    if args.profile == "bwd":
        time_bwd(qd, tc_peak, steps=args.steps, warmup=args.warmup)
        print(f"profile case done: {args.warmup + args.steps} backwards, status {qd.qd_device_status()}", flush=True)
        return
    legs = {"decode": lambda: time_decode(qd, steps=args.steps, warmup=args.warmup),
            "qed_decode": lambda: time_qed_decode(qd, steps=args.steps, warmup=args.warmup),
            "qed": lambda: time_qed(qd, hbm_peak, tc_peak, peak_kind, steps=args.steps, warmup=args.warmup),
            "long": lambda: time_long_context(qd, hbm_peak, tc_peak, peak_kind, steps=args.steps,
                                              warmup=args.warmup)}
    if args.profile in legs:
        legs[args.profile]()
        print(f"profile case done: {args.warmup + args.steps} calls of {args.profile}, "
              f"status {qd.qd_device_status()}", flush=True)
        return

    sets = make_buffers(N_BUFFERS, seed_base=1 + rank)
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    smi_index = int(vis.split(",")[local]) if vis and vis.split(",")[local].isdigit() else local
    sampler = ClockSampler(smi_index)
    sampler.start()
    time.sleep(0.3)
    total_ms, launch_ms, launches, (tw0, tw1) = time_device(qd, sets, args.steps, args.warmup, world,
                                                            soak_s=SOAK_S)
    sampler.stop()
    clocks = sampler.summary(tw0, tw1)
    clocks["window"] = f"the {args.steps} timed steps and {SOAK_S} s of the same steps, untimed, on either side"
    ms_step = max_over_ranks(total_ms / args.steps, world)
    value = job_tokens_per_s(ms_step, world)
    launch_ms = max_over_ranks(launch_ms, world)
    achieved_gbs = ALG_BYTES / (launch_ms * 1e-3) / 1e9
    achieved_tf = ALG_FLOPS / (launch_ms * 1e-3) / 1e12

    extras = {}
    if not args.no_extras:
        extras["e2e"] = time_e2e(qd, max(3, min(args.steps, 20)), 3, world)
        if rank == 0:
            dec = time_decode(qd)
            dec["frac_hbm"] = dec["GBps"] / hbm_peak
            extras["decode"] = dec
            qdec = time_qed_decode(qd)
            qdec["frac_hbm"] = qdec["GBps"] / hbm_peak
            extras["qed_decode"] = qdec
            extras["qed"] = time_qed(qd, hbm_peak, tc_peak, peak_kind)
            extras["deltanet"] = time_mode(qd, sets, "deltanet", hbm_peak, tc_peak, peak_kind)
            extras["gdn"] = time_mode(qd, sets, "gdn", hbm_peak, tc_peak, peak_kind)
            extras["long_context"] = time_long_context(qd, hbm_peak, tc_peak, peak_kind)
            extras["prologue"] = time_prologue(qd)
            extras["backward"] = time_bwd(qd, tc_peak)
            extras["eda"] = time_eda(qd)
    del sets
    torch.cuda.synchronize()

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"qdelta_bf16_B{B}_H{H}_T{T}_d{DK}", "B": B, "T": T, "H": H, "dk": DK,
                       "dv": DV, "chunk": CHUNK, "gates": "alpha,beta,lambda bf16",
                       "l2": f"inputs > L2 (q,k,v 192 MiB per set), rotated over {N_BUFFERS} sets",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved_gbs / hbm_peak, "traffic": traffic_from_profile(),
                         "peak_kind": peak_kind, "alg_bytes_per_launch": ALG_BYTES,
                         "kernel_ms": launch_ms},
            "tensor": {"achieved": achieved_tf, "peak": tc_peak, "unit": "TFLOP/s", "frac": achieved_tf / tc_peak,
                       "alg_flops_per_launch": ALG_FLOPS, "peak_kind": peak_kind},
            "gpu_launches": launches,
            "clocks": clocks}
    if "e2e" in extras:
        line["e2e"] = extras.pop("e2e")
    line.update(extras)
    if rank == 0 and not args.no_extras:
        import oracle
        oracle.build()
        v, sec, cores, passes = oracle_sample(B * H, min_seconds=10.0)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"the whole workload ({B * H} (b,h) streams, T={T}, fp64), "
                                          f"{passes} passes of {sec:.2f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
