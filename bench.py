#!/usr/bin/env python3
"""Selective-scan benchmark on B300.

One step = one forward selective scan (softplus(delta + bias), exp(Delta A)
decay, Delta B u input, C.h + D u output, silu(z) gate, last_state) over the
Mamba-2.8B layer shape: batch 4, 5120 channels, N = 16, L = 4096, bf16 I/O,
fp32 state, synthetic seeded inputs.  Inputs (674 MB) exceed the 126 MB L2,
so no flush is needed between iterations.

Prints ONE JSON line (rank 0).  ``value`` is whole-job elements/s, an
element being one (batch, channel, token) triple; ``gbps`` is the I/O bytes
the scan must move per second.  ``roofline`` compares the kernel with the
slower of its two bounds: the exp count (one per element and state entry) over
the special-function unit's rate, and the I/O bytes over HBM bandwidth.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank scans its own full-size layer (weak
scaling; the channels are independent, there is no collective on the data
path); ranks only meet at barriers and at the max-over-ranks timing.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io as _io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from selective_state_space_116_b300.workloads import (WORKLOADS, make_scan_inputs,  # noqa: E402
                                                      make_step_inputs)

METRIC = "selective-scan GB/s and elements(B*D*L)/s at 1 B300; % of HBM/SFU roofline"
# MUFU ex2 results per clock per SM on B300 (sm_103a), measured by the library's
# ssm_probe_ex2 throughput probe (python bench.py --probe-only).
EX2_PER_CLK_PER_SM = 32
L2_BYTES = 126 * 1024 * 1024


# --------------------------------------------------------------------------- setup
def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="m2p8", choices=["tiny", "m130", "m2p8", "dna"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-step", action="store_true", help="skip the generation-step line")
    p.add_argument("--only", choices=["step", "bwd", "bwd_zoh", "train", "conv", "zoh"], default=None,
                   help="time one part alone and print its line (for profiling commands)")
    p.add_argument("--probe-only", action="store_true",
                   help="only measure the special-function unit's 2^x rate")
    return p.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif args.impl == "ours":
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- work model
def scan_work(w):
    """Algorithmic I/O bytes and exp count of one scan of workload w."""
    es = 2 if w.io == "bf16" else 4
    elems = w.batch * w.dim * w.seqlen
    seq_tensors = 3 + (1 if w.gate else 0)          # u, delta, y (+ z)
    byts = seq_tensors * elems * es
    byts += 2 * w.batch * w.seqlen * w.dstate * es   # B, C
    byts += w.dim * w.dstate * 4                     # A
    byts += w.dim * 4 * ((1 if w.skip else 0) + (1 if w.bias_range else 0))
    if w.last_state:
        byts += w.batch * w.dim * w.dstate * 4
    return elems, byts, elems * w.dstate


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    out = {"hbm_gbs": 6400.0, "sm_max_mhz": 2032.0, "source": "fallback"}
    if os.path.exists(path):
        with open(path) as f:
            mp = json.load(f)
        out.update(hbm_gbs=float(mp["hbm_gbs"]), sm_max_mhz=float(mp.get("sm_max_mhz", 2032.0)),
                   source="measured")
    return out


def kernel_source_hash() -> str:
    """Hash of the forward scan's sources (the kernel the headline times)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_116_b300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith(("scan_fwd", "fwd_", "common", "host_plan")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per launch of the forward kernel at this workload, from the
    ncu capture recorded in profiles/traffic.json, if it was taken on the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(f"scan_fwd/{workload}")
    if not rec or rec.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return float(rec["dram_bytes_per_launch"])


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.file = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            gid = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            gid = str(device_index)
        self.gid = gid

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", self.gid], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        self.t_begin = time.time()

    def stop(self):
        t_end = time.time()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r for r in csv.reader(_io.StringIO(self.file.read())) if len(r) >= 9]
        self.file.close()
        os.unlink(self.file.name)
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        import datetime
        for r in rows:
            try:
                ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if not (self.t_begin - 0.05 <= ts <= t_end + 0.05):
                    continue
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                power.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- ours
def time_scan(w, steps, warmup, world, rank, local):
    import selective_state_space_116_b300 as ssm
    dev = torch.device("cuda", local)
    inp = make_scan_inputs(w, seed=rank)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.empty_like(g["u"])
    last = (torch.empty(w.batch, w.dim, w.dstate, device=dev) if w.last_state else None)
    nbytes = ssm.ssm_scan_fwd_workspace_size(w.batch, w.dim, w.dstate, w.seqlen, g["u"].dtype)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev) if nbytes else None
    _, io_bytes, _ = scan_work(w)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) \
        if io_bytes < 2 * L2_BYTES else None
    stream = torch.cuda.current_stream(dev)

    def step():
        ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                         delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                         return_last_state=w.last_state, y=y, last_state=last, workspace=ws)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    launches = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    t0.record(stream)
    for a, b in launches:
        if flush is not None:
            flush.zero_()
        a.record(stream)
        step()
        b.record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    total_ms = t0.elapsed_time(t1)
    per_launch_ms = [a.elapsed_time(b) for a, b in launches]
    return {"total_ms": total_ms, "launch_ms": per_launch_ms, "clocks": clk,
            "launches_per_step": launches_per_scan(w), "host_inputs": inp}


def launches_per_scan(w) -> int:
    """Kernels one scan launches: three for the chunked schedule the library
    picks for long sequences over few channels (channel groups of the
    state-split kernel covering fewer than 4096 channels, and at least 64
    tiles of 32 tokens), else one."""
    ch = 128 // (w.dstate // min(w.dstate, 8))   # channels per CTA of the chunked schedule
    groups = w.batch * -(-w.dim // ch)
    tiles = -(-w.seqlen // 32)
    return 3 if groups * ch < 4096 and tiles >= 64 else 1


def time_other(name, reps=20, variant=None):
    """Kernel time of one scan of another workload: `reps` scans captured in
    one CUDA graph (so that host-side call overhead, which dominates the tiny
    workload, is not counted), L2 flushed before each scan.  variant: None;
    "conv" (the fused short convolution, width 4, on the block input x);
    "zoh" (the exact zero-order-hold input term)."""
    import selective_state_space_116_b300 as ssm
    w = WORKLOADS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = make_scan_inputs(w, seed=0)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y = torch.empty_like(g["u"])
    last = torch.empty(w.batch, w.dim, w.dstate, device=dev) if w.last_state else None
    nbytes = ssm.ssm_scan_fwd_workspace_size(w.batch, w.dim, w.dstate, w.seqlen, g["u"].dtype)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev)
    _, io_bytes, _ = scan_work(w)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    opts = {}
    if variant == "conv":
        gen = torch.Generator(device=dev).manual_seed(0)
        opts = dict(conv_weight=torch.randn(w.dim, 4, device=dev, generator=gen) * 0.5,
                    conv_bias=torch.randn(w.dim, device=dev, generator=gen) * 0.5)
        io_bytes += w.dim * 5 * 4
    elif variant == "zoh":
        opts = dict(input_term="zoh")

    def scan():
        ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], D=g["D"], z=g["z"],
                         delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                         return_last_state=w.last_state, y=y, last_state=last, workspace=ws,
                         **opts)

    with torch.cuda.stream(stream):
        for _ in range(3):
            scan()
    torch.cuda.synchronize(dev)
    # a graph of flush + scan pairs and a graph of the flushes alone: the
    # scans' time is the difference
    both, flushes = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(both, stream=stream):
        for _ in range(reps):
            flush.zero_()
            scan()
    with torch.cuda.graph(flushes, stream=stream):
        for _ in range(reps):
            flush.zero_()
    both.replay()
    flushes.replay()
    torch.cuda.synchronize(dev)
    a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
    cur = torch.cuda.current_stream(dev)
    a.record(cur)
    both.replay()
    b.record(cur)
    flushes.replay()
    c.record(cur)
    torch.cuda.synchronize(dev)
    t = max(a.elapsed_time(b) - b.elapsed_time(c), 1e-6) * 1e-3 / reps
    elems, _, exps = scan_work(w)
    pk = peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    t_sfu = exps / (EX2_PER_CLK_PER_SM * sms * pk["sm_max_mhz"] * 1e6)
    t_hbm = io_bytes / (pk["hbm_gbs"] * 1e9)
    label = {None: "", "conv": ", fused short convolution (width 4) + SiLU prologue",
             "zoh": ", exact zero-order-hold input term"}[variant]
    del g, y, last, ws, flush
    torch.cuda.empty_cache()
    return {"workload": f"{w.name}: batch={w.batch}, D={w.dim}, N={w.dstate}, L={w.seqlen}, "
                        f"{w.io} I/O{label}", "kernel_time_us": t * 1e6, "elements_per_s": elems / t,
            "bytes_per_launch": io_bytes, "exps_per_launch": exps,
            "roofline_time_us": max(t_sfu, t_hbm) * 1e6, "bound": "alu" if t_sfu >= t_hbm else "hbm",
            "frac": max(t_sfu, t_hbm) / t, "launches_per_scan": launches_per_scan(w),
            "timing": f"{reps} scans in a CUDA graph, L2 flushed before each; flush time subtracted"}


def time_selective_copy(local, gap=1024, n_seq=400):
    """The selective-copying experiment (a target scalar, then `gap` Gaussian
    distractors; fixed step 0.25 against a selective 6 / 0.002) through the
    scan with the exact zero-order-hold input term: the mean recall error of
    each memory and the time of one scan of the 400 sequences."""
    import selective_state_space_116_b300 as ssm
    from selective_state_space_116_b300.workloads import selective_copy_inputs
    dev = torch.device("cuda", local)
    out = {"workload": f"selective copying: {n_seq} sequences, gap {gap}, N=1, A=-1, B=C=1, "
                       "exact zero-order hold"}
    for selective in (False, True):
        inp = selective_copy_inputs(gap, n_seq=n_seq, seed=gap, selective=selective)
        g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}

        def scan():
            return ssm.ssm_scan_fwd(g["u"], g["delta"], g["A"], g["B"], g["C"], input_term="zoh")
        for _ in range(3):
            y, _ = scan()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(20):
            scan()
        b.record()
        torch.cuda.synchronize(dev)
        key = "selective" if selective else "fixed"
        out[f"recall_error_{key}"] = float((y[0, :, -1] - g["target"]).abs().mean().item())
        out[f"us_per_scan_{key}"] = a.elapsed_time(b) * 1e3 / 20
    out["timing"] = "20 calls through the Python binding, CUDA events (latency-bound: 400 x 1025 tokens)"
    return out


def time_e2e(w, inp, steps, warmup, local):
    """Same scan through the public API from pinned host buffers: H2D of every
    input, the scan, D2H of y and last_state, every step."""
    import selective_state_space_116_b300 as ssm
    dev = torch.device("cuda", local)
    h = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    y_h = torch.empty(h["u"].shape, dtype=h["u"].dtype, pin_memory=True)
    last_h = (torch.empty(w.batch, w.dim, w.dstate, pin_memory=True) if w.last_state else None)
    h2d = sum(v.numel() * v.element_size() for v in h.values() if isinstance(v, torch.Tensor))
    d2h = y_h.numel() * y_h.element_size() + (0 if last_h is None else last_h.numel() * 4)

    def step():
        ssm.ssm_scan_fwd(h["u"], h["delta"], h["A"], h["B"], h["C"], D=h["D"], z=h["z"],
                         delta_bias=h["delta_bias"], delta_softplus=h["delta_softplus"],
                         return_last_state=w.last_state, y=y_h, last_state=last_h)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    t = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize(dev)
    sec = (time.perf_counter() - t) / steps
    return sec, h2d, d2h


def time_scan_bwd(w, local, reps=5, input_term="delta_b"):
    """Backward scan (gradients of every input from dy, forward recomputed
    inside the kernel) at the workload's shape, CUDA events on the current
    stream.  Roofline: the forward states are computed twice (checkpoint pass
    and tile recompute) and the decay once more in the adjoint pass, 3 x
    batch*dim*L*N exps; bytes: the forward inputs twice, dy and the fp32
    gradients of the (batch, dim, L) tensors once.  input_term "zoh": the
    exact zero-order-hold term, same exps and bytes."""
    import selective_state_space_116_b300 as ssm
    from selective_state_space_116_b300.workloads import make_scan_inputs
    dev = torch.device("cuda", local)
    inp = make_scan_inputs(w, seed=0)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dy = torch.randn(w.batch, w.dim, w.seqlen, device=dev,
                     generator=torch.Generator(device=dev).manual_seed(0))

    def run():
        return ssm.ssm_scan_bwd(g["u"], g["delta"], g["A"], g["B"], g["C"], dy, D=g["D"], z=g["z"],
                                delta_bias=g["delta_bias"], delta_softplus=g["delta_softplus"],
                                input_term=input_term)
    for _ in range(2):
        run()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        run()
    b.record()
    torch.cuda.synchronize(dev)
    sec = a.elapsed_time(b) / 1e3 / reps
    es = 2 if w.io == "bf16" else 4
    elems = w.batch * w.dim * w.seqlen
    nseq = 3 if w.gate else 2                                   # u, delta (, z)
    byts = 2 * (nseq * elems * es + 2 * w.batch * w.seqlen * w.dstate * es)
    byts += elems * 4 + nseq * elems * 4 + 2 * w.batch * w.seqlen * w.dstate * 4
    exps = 3 * elems * w.dstate
    pk = peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    t_roof = max(byts / (pk["hbm_gbs"] * 1e9),
                 exps / (EX2_PER_CLK_PER_SM * sms * pk["sm_max_mhz"] * 1e6))
    out_gb = (2 + (1 if w.gate else 0)) * elems * 4 / 1e9
    # chunked (the chunks' maps, their composition, then the chunks): the
    # workspace then holds more than the checkpoints
    ckpt = w.batch * w.dim * -(-w.seqlen // 8) * w.dstate * 4
    chunked = ssm.ssm_scan_bwd_workspace_size(w.batch, w.dim, w.dstate, w.seqlen, w.torch_io) > ckpt
    return {"workload": w.name, "input_term": input_term, "ms": sec * 1e3,
            "roofline_ms": t_roof * 1e3, "frac": t_roof / sec,
            "launches": 3 if chunked else 1,
            "timing": f"{reps} calls, CUDA events (outputs {out_gb:.1f} GB: larger than L2)"}


def time_train_step(w, local, reps=5):
    """One training step of the scan through the autograd wrapper
    (selective_scan forward, then backward from a fixed upstream gradient of
    y and last_state), as a user's training loop runs it: the library's
    forward and backward kernels plus the wrapper's casts of the gradients
    to the inputs' dtype.  CUDA events on the current stream."""
    import selective_state_space_116_b300 as ssm
    dev = torch.device("cuda", local)
    inp = make_scan_inputs(w, seed=0)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    names = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")
    leaves = {k: g[k].clone().requires_grad_(True) for k in names if g[k] is not None}
    gen = torch.Generator(device=dev).manual_seed(1)
    wy = torch.randn(w.batch, w.dim, w.seqlen, device=dev, generator=gen).to(w.torch_io)
    wl = torch.randn(w.batch, w.dim, w.dstate, device=dev, generator=gen)

    def step():
        for t in leaves.values():
            t.grad = None
        y, last = ssm.selective_scan(leaves["u"], leaves["delta"], leaves["A"], leaves["B"], leaves["C"],
                                     D=leaves.get("D"), z=leaves.get("z"),
                                     delta_bias=leaves.get("delta_bias"),
                                     delta_softplus=g["delta_softplus"])
        torch.autograd.backward((y, last), (wy, wl))
    for _ in range(2):
        step()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        step()
    b.record()
    torch.cuda.synchronize(dev)
    sec = a.elapsed_time(b) / 1e3 / reps
    elems = w.batch * w.dim * w.seqlen
    return {"workload": w.name, "ms": sec * 1e3, "elements_per_s": elems / sec,
            "timing": f"{reps} steps (forward + backward through selective_scan), CUDA events"}


def time_state_step(local, graph_steps=1024, reps=5):
    """Generation: 128 x 5120 channels, N = 16, bf16 inputs, fp32 state, one token
    per launch, 1024 consecutive launches captured in one CUDA graph.  The state
    (42 MB) would stay in L2 across launches, so four state buffers (168 MB)
    rotate: four independent token streams, each with its own state."""
    import selective_state_space_116_b300 as ssm
    dev = torch.device("cuda", local)
    w = WORKLOADS["gen"]
    nsteps_in = 64   # distinct token inputs cycled through; 4 GB for 1024 would be wasteful
    inp = make_step_inputs(w, seed=0, steps=nsteps_in)
    g = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    states = [torch.zeros(w.batch, w.dim, w.dstate, device=dev) for _ in range(4)]
    ys = torch.empty(nsteps_in, w.batch, w.dim, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(dev)

    def run(n):
        for t in range(n):
            k = t % nsteps_in
            ssm.ssm_state_step(states[t % 4], g["x"][k], g["delta"][k], g["A"], g["B"][k],
                               g["C"][k], D=g["D"], z=g["z"][k], delta_bias=g["delta_bias"],
                               delta_softplus=True, y=ys[k])

    with torch.cuda.stream(stream):
        run(8)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        run(graph_steps)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream(dev)
    a.record(cur)
    for _ in range(reps):
        graph.replay()
    b.record(cur)
    torch.cuda.synchronize(dev)
    us = a.elapsed_time(b) * 1e3 / (reps * graph_steps)
    chan = w.batch * w.dim
    byts = chan * w.dstate * 4 * 2 + chan * 2 * 4 + 2 * w.batch * w.dstate * 2 \
        + w.dim * w.dstate * 4 + 2 * w.dim * 4
    return {"workload": "gen: 128 x 5120 channels, N=16, bf16 x/delta/z/B/C, fp32 state",
            "us_per_token": us, "elements_per_s": chan / (us * 1e-6),
            "gbps": byts / (us * 1e-6) / 1e9, "bytes_per_token": byts,
            "launches": reps * graph_steps, "state_buffers": 4,
            "timing": "CUDA graph of 1024 launches, CUDA events"}


def probe_ex2(local, seconds=1.5):
    """Measured 2^x rate of the special-function unit, through ssm_probe_ex2."""
    import selective_state_space_116_b300 as ssm
    lib = ssm._lib.load()
    dev = torch.device("cuda", local)
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    sink = torch.zeros(1024, device=dev)
    stream = torch.cuda.current_stream(dev)
    blocks, threads, iters = sms * 8, 256, 4096
    launch = lambda: lib.ssm_probe_ex2(blocks, threads, iters, sink.data_ptr(), stream.cuda_stream)
    assert launch() == 0
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    assert launch() == 0
    b.record(stream)
    torch.cuda.synchronize(dev)
    reps = max(1, int(seconds / max(a.elapsed_time(b) * 1e-3, 1e-4)))
    clocks = ClockSampler(local)
    clocks.start()
    a.record(stream)
    for _ in range(reps):
        assert launch() == 0
    b.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    rate = blocks * threads * iters * 8 * reps / (a.elapsed_time(b) * 1e-3)
    per_clk = rate / sms / (clk["sm_mhz"] * 1e6) if clk.get("sm_mhz") else None
    return {"ex2_per_s": rate, "ex2_per_clk_per_sm": per_clk, "sm_mhz_median": clk.get("sm_mhz"),
            "clocks": clk, "launch": f"{blocks} x {threads} threads, {iters} x 8 chains, {reps} reps"}


# --------------------------------------------------------------------------- oracle
def oracle_rate(w, inp, target_s=8.0, max_threads=None):
    """Elements/s of the fp64 oracle on a bounded channel sample of workload w."""
    import oracle
    threads = max(1, min(os.cpu_count() or 1, max_threads or 1024))
    nch_total = w.batch * w.dim

    def run(n, nthreads=threads):
        chans = np.arange(n, dtype=np.int64) % nch_total
        t = time.perf_counter()
        oracle.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                        z=inp["z"], delta_bias=inp["delta_bias"],
                        delta_softplus=inp["delta_softplus"], channels=chans, nthreads=nthreads)
        return time.perf_counter() - t

    n = threads
    sec = run(n)
    n = int(min(nch_total, max(threads, n * target_s / max(sec, 1e-3))))
    n = max(threads, (n // threads) * threads)
    sec = run(n)
    out = {"value": n * w.seqlen / sec, "unit": "elements/s", "cores": threads,
           "kind": "oracle",
           "sample": f"{n} of {nch_total} channels x {w.seqlen} tokens of the {w.name} "
                     f"workload, fp64, {threads} threads, {sec:.1f} s"}
    if threads > 1:   # the same oracle on one core, ~1 s
        n1 = int(max(1, min(nch_total, n / threads * min(1.0, target_s) / max(sec, 1e-3))))
        sec1 = run(n1, 1)
        out["single_thread"] = {"value": n1 * w.seqlen / sec1, "unit": "elements/s",
                                "sample": f"{n1} channels x {w.seqlen} tokens, 1 thread, {sec1:.1f} s"}
    return out


# --------------------------------------------------------------------------- main
def run_reference(args, world, rank):
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    inp = make_scan_inputs(w, seed=0)
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    # each step: a bounded sample of the workload (channels x full length)
    per_step_target = max(1.0, 90.0 / max(1, args.steps + args.warmup))
    cal = oracle_rate(w, inp, target_s=min(per_step_target, 3.0))
    nch = int(max(threads, min(w.batch * w.dim,
                               cal["value"] * per_step_target / w.seqlen)))
    nch = max(threads, nch // threads * threads)
    chans = np.arange(nch, dtype=np.int64)

    def step():
        oracle.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                        z=inp["z"], delta_bias=inp["delta_bias"],
                        delta_softplus=inp["delta_softplus"], channels=chans, nthreads=threads)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    sec = (time.perf_counter() - t) / max(1, args.steps)
    value = nch * w.seqlen / sec
    out = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "elements/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": f"{w.name}: batch={w.batch}, D={w.dim}, N={w.dstate}, "
                               f"L={w.seqlen}, {w.io} I/O", "sample_channels": nch},
        "cpu_baseline": {"value": value, "unit": "elements/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{nch} of {w.batch * w.dim} channels x {w.seqlen} tokens "
                                   f"per step, fp64, {threads} threads"},
        "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def run_ours(args, world, rank, local):
    w = WORKLOADS[args.workload]
    elems, io_bytes, exps = scan_work(w)
    res = time_scan(w, args.steps, args.warmup, world, rank, local)
    total_ms = max_over_ranks(res["total_ms"], world)
    launch_ms = statistics.mean(res["launch_ms"])
    ms_per_step = total_ms / args.steps
    value = world * elems / (ms_per_step * 1e-3)
    pk = peaks()
    props = torch.cuda.get_device_properties(local)
    sms = props.multi_processor_count
    exp_peak = EX2_PER_CLK_PER_SM * sms * pk["sm_max_mhz"] * 1e6     # exp/s
    t_sfu = exps / exp_peak
    t_hbm = io_bytes / (pk["hbm_gbs"] * 1e9)
    t_launch = launch_ms * 1e-3
    sfu_achieved = exps / t_launch
    hbm_achieved = io_bytes / t_launch / 1e9
    bound = "alu" if t_sfu >= t_hbm else "hbm"
    traffic = committed_traffic(args.workload)
    roofline = {
        "bound": bound,
        "achieved": sfu_achieved / 1e9 if bound == "alu" else hbm_achieved,
        "peak": exp_peak / 1e9 if bound == "alu" else pk["hbm_gbs"],
        "unit": "Gexp/s" if bound == "alu" else "GB/s",
        "frac": (t_sfu if bound == "alu" else t_hbm) / t_launch,
        "traffic": traffic,
        "kernel": "ssm::scan_fwd_kernel",
        "peak_source": (f"SFU: {EX2_PER_CLK_PER_SM} ex2/clk/SM (probe) x {sms} SMs x "
                        f"{pk['sm_max_mhz']:.0f} MHz max clock; HBM: {pk['hbm_gbs']:.0f} GB/s "
                        f"copy ({pk['source']})"),
        "hbm": {"achieved": hbm_achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": t_hbm / t_launch, "bytes_per_launch": io_bytes},
        "sfu": {"achieved": sfu_achieved / 1e9, "peak": exp_peak / 1e9, "unit": "Gexp/s",
                "frac": t_sfu / t_launch, "exps_per_launch": exps},
        "roofline_time_us": max(t_sfu, t_hbm) * 1e6,
        "kernel_time_us": launch_ms * 1e3,
    }
    out = {
        "metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if w.io == "f32" else "bf16 I/O, f32 state and math",
        "data": "synthetic (seeded numpy PCG64)",
        "config": {"workload": f"{w.name}: Mamba-2.8B layer scan, batch={w.batch}, D={w.dim}, "
                               f"N={w.dstate}, L={w.seqlen}, {w.io} I/O, softplus+bias, "
                               f"z gate, last_state" if w.name == "m2p8" else w.name,
                   "batch": w.batch, "dim": w.dim, "dstate": w.dstate, "seqlen": w.seqlen,
                   "l2": "inputs larger than L2" if io_bytes >= 2 * L2_BYTES else "L2 flushed",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gbps": world * io_bytes / (ms_per_step * 1e-3) / 1e9,
        "roofline": roofline,
        "clocks": res["clocks"],
        "gpu_launches": res["launches_per_step"] * args.steps,
        "kernel_source_sha256": kernel_source_hash(),
    }
    if not args.no_e2e:
        sec, h2d, d2h = time_e2e(w, res["host_inputs"], max(3, args.steps // 4), 3, local)
        sec = max_over_ranks(sec, world)
        out["e2e"] = {"value": world * elems / sec, "unit": "elements/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "ms_per_step": sec * 1e3}
    if not args.no_step and rank == 0:
        out["state_step"] = time_state_step(local)
        out["scan_bwd"] = time_scan_bwd(w, local)
        out["scan_bwd_zoh"] = time_scan_bwd(w, local, input_term="zoh")
        out["scan_bwd_dna"] = time_scan_bwd(WORKLOADS["dna"], local, reps=3)
        out["train_step"] = time_train_step(w, local)
        out["other_workloads"] = [time_other("m130"), time_other("tiny"),
                                  time_other("dna", reps=5),
                                  time_other(args.workload, variant="conv"),
                                  time_other(args.workload, variant="zoh")]
        out["selective_copy"] = time_selective_copy(local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = oracle_rate(w, res["host_inputs"])
    if rank == 0:
        print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.probe_only:
        if rank == 0:
            print(json.dumps({"sfu_probe": probe_ex2(local)}), flush=True)
    elif args.only:
        if rank == 0:
            w = WORKLOADS[args.workload]
            part = {"step": lambda: time_state_step(local),
                    "bwd": lambda: time_scan_bwd(w, local),
                    "bwd_zoh": lambda: time_scan_bwd(w, local, input_term="zoh"),
                    "train": lambda: time_train_step(w, local),
                    "conv": lambda: time_other(args.workload, variant="conv"),
                    "zoh": lambda: time_other(args.workload, variant="zoh")}[args.only]()
            print(json.dumps({args.only: part}), flush=True)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
