#!/usr/bin/env python3
"""Benchmark of the Mamba2 recurrent-state update on GB300.

One step = one Nemotron-H-8B-shaped decode token through all 48 Mamba2 layers for a batch of
256 requests drawn (random, non-contiguous) from a 512-slot pool per layer: per layer one
fused launch (conv shift + conv1d + SiLU, softplus step, state update, C.h + D.x, SiLU(z) gate)
reading and writing each request's 2 MiB bf16 state in place.  The chunked prefill (8 varlen
sequences of 512..8192 tokens summing to 32768, chunk 256, checkpoints every 1024 tokens) is
timed after it and reported in the same line.

Metric: decode state-update GB/s (algorithmic bytes / time) and token-layers/s against HBM
peak; prefill tokens/s.  Inputs are synthetic and seeded (no dataset): the value distributions
are the ones in recurrent_state_update_gb300.workloads.  The state pool of one layer
(512 MiB touched per launch) is larger than L2, so no L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gb300,reference}]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from recurrent_state_update_gb300 import workloads as wl  # noqa: E402

DECODE = wl.NEMOTRON_DECODE
PREFILL = wl.CHUNKED_PREFILL
SHAPE = wl.NEMOTRON_H_8B
H, P, N, G = SHAPE.nheads, SHAPE.head_dim, SHAPE.d_state, SHAPE.n_groups
CD = SHAPE.conv_dim
W1 = SHAPE.conv_kernel - 1

# Algorithmic bytes of one decode token-layer (bf16 state and activations, fp32 dt):
#   state read + write 2*H*P*N*2, conv state read + write 2*CD*(W-1)*2, xBC in CD*2,
#   z in H*P*2, dt in H*4, y out H*P*2.  Per-launch constants (conv taps, A, D, dt_bias) excluded.
DECODE_BYTES_PER_TOKEN_LAYER = 2 * H * P * N * 2 + 2 * CD * W1 * 2 + CD * 2 + H * P * 2 + H * 4 + H * P * 2


def prefill_bytes(T: int, nseq: int, n_state_writes: int) -> int:
    """Algorithmic bytes of one prefill launch: x, B, C, dt in, y out, state writes (bf16)."""
    return T * H * P * 2 + 2 * T * G * N * 2 + T * H * 4 + T * H * P * 2 + n_state_writes * H * P * N * 2


def prefill_conv_bytes(T: int, nseq: int) -> int:
    """Algorithmic bytes of the varlen prefill conv: xBC in, x | B | C out, each sequence's conv
    window read (W-1 columns) and written (W-1 columns), bf16."""
    Cd = SHAPE.conv_dim
    return 2 * T * Cd * 2 + nseq * Cd * (SHAPE.conv_kernel - 1) * 2 * 2


def prefill_flops(lengths, chunk: int) -> float:
    """Algorithmic flops of the chunked form (causal halves of the intra-chunk matmuls counted):
    per chunk of length L and group: C B^T L(L+1)/2 * 2N; per head: masked (G . L) X L(L+1)/2 * 2P,
    chunk state 2 L P N, off-diagonal C h 2 L N P."""
    total = 0.0
    for Ls in lengths:
        for c0 in range(0, int(Ls), chunk):
            L = min(chunk, int(Ls) - c0)
            tri = L * (L + 1) / 2
            total += G * tri * 2 * N + H * (tri * 2 * P + 2 * L * P * N + 2 * L * N * P)
    return total


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), float(pk["bf16_tflops"]), float(pk["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _profile_traffic(kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or None when the summary
    is missing or was taken on a different version of the kernel source."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            v = v.strip()
            if v.startswith("`") and v.count("`") >= 2:
                v = v[1:v.index("`", 1)]  # the value is the first backticked field
            vals[k.strip()] = v
    src = vals.get("source")
    if not src or "traffic_bytes_per_launch" not in vals:
        return None
    try:
        digest = hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    if digest != vals.get("source_sha256_16"):
        return None
    return float(vals["traffic_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=10)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
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
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------------------
# GPU arm
# ------------------------------------------------------------------------------------------

def e2e_groups(layers: int):
    """Group sizes of the end-to-end pipeline: one layer first and last (its upload, or its
    download, is the part not hidden behind compute), doubling up to eight layers between."""
    up = [1, 2, 4]
    if layers < 2 * sum(up) + 8:
        return [1] * layers
    mid = layers - 2 * sum(up)
    return up + [8] * (mid // 8) + ([mid % 8] if mid % 8 else []) + up[::-1]


class DecodeWorkload:
    """48 layers of pools, parameters and one step's inputs, resident on the device."""

    def __init__(self, torch, rank: int, layers: int, batch: int, pool: int):
        from recurrent_state_update_gb300 import binding as bd
        self.torch, self.bd = torch, bd
        self.layers, self.batch, self.pool = layers, batch, pool
        self.desc = bd.layer_desc(SHAPE, state=wl.BF16, act=wl.BF16, dt=wl.F32)
        dev = torch.device("cuda")
        seed = DECODE["seed"] * 1000 + rank
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)
        bf = torch.bfloat16
        # slot pools [layer, slot, ...], N(0, 0.1^2), generated on the device
        self.ssm = torch.empty(layers, pool, H, P, N, dtype=bf, device=dev)
        self.conv = torch.empty(layers, pool, CD, W1, dtype=bf, device=dev)
        for l in range(layers):
            self.ssm[l].copy_(torch.randn(pool, H, P, N, generator=gen, device=dev).mul_(0.1))
            self.conv[l].copy_(torch.randn(pool, CD, W1, generator=gen, device=dev).mul_(0.1))
        # Every layer's step inputs (xbc, dt, z, slot ids) packed back to back in one pinned host
        # buffer and its device copy, so that the inputs of a run of layers move in one copy.
        self.prm, self.slot, self.inp = [], [], []
        host_np = []
        for l in range(layers):
            g = wl.rng(seed, l)
            prm = wl.layer_params(g, SHAPE)
            self.prm.append({k: torch.from_numpy(v).to(dev) for k, v in prm.items()})
            ids = wl.slot_ids(g, pool, batch)
            inp = wl.decode_inputs(g, SHAPE, prm, batch, 1, wl.BF16)
            host_np.append({"xbc": (inp["xbc"].view(np.int16), bf), "dt": (inp["dt"], torch.float32),
                            "z": (inp["z"].view(np.int16), bf), "slot": (ids, torch.int32)})
        fields = list(host_np[0])
        nbytes = {k: host_np[0][k][0].nbytes for k in fields}
        self.layer_bytes = sum((nbytes[k] + 255) // 256 * 256 for k in fields)
        self.host_flat = torch.empty(layers * self.layer_bytes, dtype=torch.uint8, pin_memory=True)
        self.dev_flat = torch.empty(layers * self.layer_bytes, dtype=torch.uint8, device=dev)
        for l in range(layers):
            off = l * self.layer_bytes
            devv = {}
            for k in fields:
                arr, dtype = host_np[l][k]
                nb = nbytes[k]
                self.host_flat[off:off + nb].copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)))
                devv[k] = self.dev_flat[off:off + nb].view(dtype).view(arr.shape)
                off += (nb + 255) // 256 * 256
            self.slot.append(devv.pop("slot"))
            self.inp.append(devv)
        self.dev_flat.copy_(self.host_flat)
        self.y = torch.empty(layers, batch, 1, H * P, dtype=bf, device=dev)
        self.y_host = torch.empty(layers, batch, 1, H * P, dtype=bf).pin_memory()
        self.launches_per_step = layers
        # end-to-end pipeline: uploads on one stream, downloads on another, the launches on the
        # caller's stream; events order each group of layers' buffers across streams and steps
        self.s_up, self.s_down = torch.cuda.Stream(), torch.cuda.Stream()
        self.groups = e2e_groups(layers)
        ev = lambda: [torch.cuda.Event() for _ in self.groups]
        self.ev_in, self.ev_used, self.ev_out = ev(), ev(), ev()
        self.ev_start = torch.cuda.Event()

    def step(self, stream=None):
        bd = self.bd
        for l in range(self.layers):
            inp, prm = self.inp[l], self.prm[l]
            bd.mamba_state_update(self.desc, self.ssm[l], self.slot[l], inp["xbc"], inp["dt"], prm["A"], self.y[l],
                                  conv_pool=self.conv[l], conv_w=prm["conv_w"], D=prm["D"],
                                  dt_bias=prm["dt_bias"], z=inp["z"], stream=stream)

    def step_e2e(self):
        """Host buffers in, result out: every layer's inputs copied from pinned memory, the 48
        launches, and every layer's y copied back, all inside the step.  Layers go in groups
        (`e2e_groups`): group g+1's upload runs while group g computes and group g's y is
        downloaded while group g+1 computes (three streams, one event per group and stream).  The
        launches inside a group follow each other with no stream dependency between them, so each
        starts as the previous one completes (programmatic dependent launch); a group boundary
        waits on that group's upload.  Only the first group's upload and the last group's download
        (one layer each) are not overlapped with compute.  No upload starts before the previous
        step has ended with its result on the host, as in a decode loop whose next inputs come
        from the previous step's outputs."""
        torch, bd = self.torch, self.bd
        cur = torch.cuda.current_stream()
        self.ev_start.record(cur)  # after the previous step's final wait: its y is on the host
        l0 = 0
        for gi, n in enumerate(self.groups):
            layers = range(l0, l0 + n)
            with torch.cuda.stream(self.s_up):
                if gi == 0:
                    self.s_up.wait_event(self.ev_start)
                self.s_up.wait_event(self.ev_used[gi])  # the previous step's group has read its inputs
                a, b = l0 * self.layer_bytes, (l0 + n) * self.layer_bytes
                self.dev_flat[a:b].copy_(self.host_flat[a:b], non_blocking=True)
                self.ev_in[gi].record(self.s_up)
            cur.wait_event(self.ev_in[gi])
            cur.wait_event(self.ev_out[gi])  # the previous step's y of the group has been downloaded
            for l in layers:
                d, prm = self.inp[l], self.prm[l]
                bd.mamba_state_update(self.desc, self.ssm[l], self.slot[l], d["xbc"], d["dt"], prm["A"], self.y[l],
                                      conv_pool=self.conv[l], conv_w=prm["conv_w"], D=prm["D"],
                                      dt_bias=prm["dt_bias"], z=d["z"])
            self.ev_used[gi].record(cur)
            with torch.cuda.stream(self.s_down):
                self.s_down.wait_event(self.ev_used[gi])
                self.y_host[l0:l0 + n].copy_(self.y[l0:l0 + n], non_blocking=True)
                self.ev_out[gi].record(self.s_down)
            l0 += n
        cur.wait_event(self.ev_out[-1])  # the step ends when the last y is on the host

    def h2d_bytes(self):
        return self.host_flat.numel()  # the inputs plus at most 255 bytes of padding per field

    def d2h_bytes(self):
        return self.y_host.numel() * self.y_host.element_size()

    def bytes_per_step(self):
        return self.layers * self.batch * DECODE_BYTES_PER_TOKEN_LAYER


class PrefillWorkload:
    """One layer of the varlen chunked prefill, inputs resident on the device."""

    def __init__(self, torch, rank: int):
        from recurrent_state_update_gb300 import binding as bd
        self.torch, self.bd = torch, bd
        dev = torch.device("cuda")
        seed = PREFILL["seed"] * 1000 + rank
        g = wl.rng(seed, 0)
        self.lengths = wl.prefill_lengths(g, PREFILL["nseq"], PREFILL["len_lo"], PREFILL["len_hi"], PREFILL["total"])
        T = int(self.lengths.sum())
        self.T = T
        cu = wl.cu_seqlens(self.lengths)
        prm = wl.layer_params(g, SHAPE)
        inp = wl.prefill_inputs(g, SHAPE, prm, T, wl.BF16)
        bf = torch.bfloat16
        self.desc = bd.layer_desc(SHAPE, state=wl.BF16, act=wl.BF16, dt=wl.F32)
        nseq = len(self.lengths)
        interval = PREFILL["ckpt_interval"]
        max_ckpt = int(self.lengths.max()) // interval
        n_ckpt = int(sum(int(L) // interval for L in self.lengths))
        S = nseq + nseq * max_ckpt
        self.pool = torch.zeros(S, H, P, N, dtype=bf, device=dev)
        self.slot = torch.arange(nseq, dtype=torch.int32, device=dev)
        ck = np.arange(nseq, nseq + nseq * max_ckpt, dtype=np.int32).reshape(nseq, max_ckpt)
        self.ckpt = torch.from_numpy(ck).to(dev)
        self.cu = torch.from_numpy(cu).to(dev)
        self.prm = {k: torch.from_numpy(v).to(dev) for k, v in prm.items()}
        self.x = torch.from_numpy(inp["x"].view(np.int16)).to(dev).view(bf)
        self.B = torch.from_numpy(inp["B"].view(np.int16)).to(dev).view(bf)
        self.C = torch.from_numpy(inp["C"].view(np.int16)).to(dev).view(bf)
        self.dt = torch.from_numpy(inp["dt"]).to(dev)
        self.y = torch.empty_like(self.x)
        wsb = bd.mamba_chunk_scan_workspace_bytes(self.desc, T, nseq, PREFILL["chunk"])
        self.ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        self.interval = interval
        self.n_state_writes = nseq + n_ckpt
        # raw xBC and conv windows for the conv in front of the scan (every sequence continues
        # from its stored window)
        self.xbc = torch.from_numpy(wl.prefill_xbc(g, SHAPE, T, wl.BF16).view(np.int16)).to(dev).view(bf)
        self.conv_pool = torch.from_numpy(
            wl.initial_states(g, SHAPE, nseq, wl.F32, wl.BF16)["conv"].view(np.int16)).to(dev).view(bf)
        self.has_init = torch.ones(nseq, dtype=torch.uint8, device=dev)

    def step_conv(self):
        T = self.T
        self.bd.mamba_conv_varlen(self.desc, self.cu, self.xbc, self.prm["conv_w"], self.x.view(T, H * P),
                                  self.B.view(T, G * N), self.C.view(T, G * N), conv_pool=self.conv_pool,
                                  slot_ids=self.slot, has_initial_state=self.has_init)

    def step_layer(self):
        self.step_conv()
        self.step()

    def step(self):
        self.bd.mamba_chunk_scan(self.desc, self.pool, self.cu, self.slot, self.x, self.dt, self.prm["A"], self.B,
                                 self.C, self.y, self.ws, ckpt_slots=self.ckpt, ckpt_interval=self.interval,
                                 chunk=PREFILL["chunk"], D=self.prm["D"], dt_bias=self.prm["dt_bias"])


def _time(torch, fn, steps, warmup, dist=None):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1) / steps  # ms per step


def _time_graph(torch, fn, steps, warmup, dist=None, reps=1):
    """ms per call of `fn` replayed from a CUDA graph: launch-bound sequences of short kernels are
    timed on the GPU instead of on the host's launch rate.  `fn` runs eagerly `warmup` times
    (first-call set-up happens outside the capture), then `reps` calls are captured once and the
    graph is replayed `steps` times between CUDA events."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(reps):
            fn()
    graph.replay()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        graph.replay()
    e1.record(s)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1) / (steps * reps)


def _max_over_ranks(torch, dist, v, device="cuda"):
    """The slowest rank's time: every rank contributes its own, all get the maximum."""
    if dist is None:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_gbs(bytes_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job GB/s: the bytes all ranks moved over the slowest rank's time."""
    return bytes_per_rank * world / (ms_max * 1e-3) / 1e9


def cpu_baseline_decode(budget_s: float = 10.0, rows: int = 32):
    """The fp64 oracle (as it stands) on a bounded sample of the decode workload: `rows` rows of
    one layer's batch, repeated until about `budget_s` seconds of CPU time have passed."""
    import oracle
    seed = DECODE["seed"] * 1000
    g = wl.rng(seed, 0)
    prm = wl.layer_params(g, SHAPE)
    inp = wl.decode_inputs(g, SHAPE, prm, rows, 1, wl.BF16)
    st = wl.initial_states(wl.rng(seed, 99), SHAPE, rows, wl.BF16, wl.BF16)
    ssm = wl.upcast(st["ssm"], wl.BF16)
    conv = wl.upcast(st["conv"], wl.BF16)
    xbc = wl.upcast(inp["xbc"], wl.BF16)
    z = wl.upcast(inp["z"], wl.BF16).reshape(rows, 1, H, P)
    dt = inp["dt"].astype(np.float64)
    o = {k: v.astype(np.float64) for k, v in prm.items()}
    slot = np.arange(rows, dtype=np.int32)
    threads = oracle.default_threads()
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.decode(ssm, slot, xbc, dt, o["A"], conv_pool=conv, conv_w=o["conv_w"], D=o["D"],
                      dt_bias=o["dt_bias"], z=z, n_groups=G, nthreads=threads)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    gbs = n * rows * DECODE_BYTES_PER_TOKEN_LAYER / el / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} x {rows} rows of one Nemotron-H-8B decode layer (fp64 C oracle, {el:.1f} s)",
            "token_layers_per_s": n * rows / el}


def run_gpu(args):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from recurrent_state_update_gb300 import build as bld
    bld.build()
    hbm_peak, bf16_peak, bf16_sus, peak_src = _peaks()

    if args.only in ("prefill", "spec", "sweep", "checkpoint", "mamba1"):
        if args.only == "prefill":
            res = run_prefill(torch, args, rank, world, dist, hbm_peak, bf16_peak)
        elif args.only == "spec":
            res = run_spec(torch, args, rank, dist, hbm_peak)
        elif args.only == "checkpoint":
            res = run_checkpoint(torch, args, rank, dist, hbm_peak)
        elif args.only == "mamba1":
            res = run_mamba1(torch, args, rank, dist, hbm_peak)
        else:
            res = run_sweep(torch, args, rank, dist, hbm_peak)
        if rank == 0:
            print(json.dumps({args.only: res}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    layers = args.layers or DECODE["layers"]
    dec = DecodeWorkload(torch, rank, layers, DECODE["batch"], DECODE["pool"])
    clocks = ClockSampler(local)
    # the sampler runs across the warm-up and the timed steps, so its samples see the GPU under load
    clocks.start()
    time.sleep(0.2)
    for _ in range(args.warmup):
        dec.step()
    torch.cuda.synchronize()
    ms = _time(torch, dec.step, args.steps, 0, dist)
    ck = clocks.stop()
    ms = _max_over_ranks(torch, dist, ms)
    total_bytes = dec.bytes_per_step() * world
    value = weak_scaling_gbs(dec.bytes_per_step(), world, ms)
    token_layers = layers * DECODE["batch"] * world / (ms * 1e-3)
    launch_ms = ms / dec.launches_per_step
    achieved = DECODE["batch"] * DECODE_BYTES_PER_TOKEN_LAYER / (launch_ms * 1e-3) / 1e9

    # end to end: pinned host inputs in, every layer's y out, inside the timed region
    e2e = None
    if args.only in ("all", "decode"):
        ms_e2e = _max_over_ranks(torch, dist, _time(torch, dec.step_e2e, args.steps, max(args.warmup, 3), dist))
        e2e = {"value": total_bytes / (ms_e2e * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": ms_e2e,
               "h2d_bytes_per_step": dec.h2d_bytes(), "d2h_bytes_per_step": dec.d2h_bytes()}
    del dec
    torch.cuda.empty_cache()
    prefill = spec = sweep = ckpt = m1 = None
    if args.only == "all":
        prefill = run_prefill(torch, args, rank, world, dist, hbm_peak, bf16_peak)
        torch.cuda.empty_cache()
        spec = run_spec(torch, args, rank, dist, hbm_peak)
        torch.cuda.empty_cache()
        sweep = run_sweep(torch, args, rank, dist, hbm_peak)
        torch.cuda.empty_cache()
        ckpt = run_checkpoint(torch, args, rank, dist, hbm_peak)
        torch.cuda.empty_cache()
        m1 = run_mamba1(torch, args, rank, dist, hbm_peak)
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and args.only == "all" and not args.no_cpu_baseline:
        cpu = cpu_baseline_decode()

    if rank == 0:
        emit(args, world, layers, ms, value, token_layers, achieved, launch_ms, hbm_peak, peak_src, e2e, ck,
             prefill, cpu, spec, sweep, ckpt, m1)
    if dist is not None:
        dist.destroy_process_group()


SPEC = wl.SPEC_DECODE
SWEEP = wl.PADDING_SWEEP


def spec_bytes(rows: int, accepted_rows: int, K: int, Wc: int) -> int:
    """Algorithmic bytes of one speculative step (draft launch + commit) for `rows` requests:
    draft: state read once, K states written to scratch, conv state read + written, K tokens of
    xBC, z, y, dt; commit: the accepted rows copy one state (read + write) and every row re-seats
    its conv state (read + write)."""
    st = H * P * N * 2
    conv = CD * Wc * 2
    draft = rows * (st + K * st + 2 * conv + K * (CD * 2 + H * P * 2 * 2 + H * 4))
    commit = accepted_rows * 2 * st + rows * 2 * conv
    return draft + commit


def run_spec(torch, args, rank, dist, hbm_peak):
    """Speculative decode: batch 128, 4 draft tokens, 4 scratch slots per request, then the commit
    of random accept lengths (one layer per step)."""
    from recurrent_state_update_gb300 import binding as bd
    dev = torch.device("cuda")
    shape = SHAPE.with_spec(SPEC["ntok"])
    batch, K = SPEC["batch"], SPEC["ntok"]
    S = batch * (1 + K)
    g = wl.rng(SPEC["seed"] * 1000 + rank, 0)
    prm_np = wl.layer_params(g, shape)
    prm = {k: torch.from_numpy(v).to(dev) for k, v in prm_np.items()}
    gen = torch.Generator(device=dev)
    gen.manual_seed(SPEC["seed"] * 1000 + rank)
    bf = torch.bfloat16
    ssm = torch.randn(S, H, P, N, generator=gen, device=dev).mul_(0.1).to(bf)
    conv = torch.randn(S, CD, shape.conv_cols, generator=gen, device=dev).mul_(0.1).to(bf)
    ids = g.permutation(S).astype(np.int32)
    slot = torch.from_numpy(ids[:batch]).to(dev)
    scratch = torch.from_numpy(ids[batch:].reshape(batch, K).copy()).to(dev)
    inp = wl.decode_inputs(g, shape, prm_np, batch, K, wl.BF16)
    xbc = torch.from_numpy(inp["xbc"].view(np.int16)).to(dev).view(bf)
    z = torch.from_numpy(inp["z"].view(np.int16)).to(dev).view(bf)
    dt = torch.from_numpy(inp["dt"]).to(dev)
    accept_np = wl.accept_lengths(g, batch, K)
    accept = torch.from_numpy(accept_np).to(dev)
    y = torch.empty(batch, K, H * P, dtype=bf, device=dev)
    desc = bd.layer_desc(shape)

    def step():
        bd.mamba_state_update(desc, ssm, slot, xbc, dt, prm["A"], y, conv_pool=conv, conv_w=prm["conv_w"],
                              scratch_slots=scratch, D=prm["D"], dt_bias=prm["dt_bias"], z=z)
        bd.mamba_spec_commit(desc, ssm, slot, scratch, accept, conv_pool=conv)

    ms = _max_over_ranks(torch, dist, _time(torch, step, max(args.steps, 10), max(args.warmup, 3), dist))
    by = spec_bytes(batch, int((accept_np > 0).sum()), K, shape.conv_cols)
    return {"workload": SPEC["name"], "ms_per_step": ms, "draft_tokens_per_s": batch * K / (ms * 1e-3),
            "gbs": by / (ms * 1e-3) / 1e9, "hbm_frac": by / (ms * 1e-3) / 1e9 / hbm_peak,
            "algorithmic_bytes": by, "launches_per_step": 2, "kernels": "k_decode (4 tokens), k_spec_commit"}


def run_sweep(torch, args, rank, dist, hbm_peak):
    """Decode at batch 1, 8, 64, 256, 1024 of a 1536-slot pool with 10 % of rows padded (-1):
    per-launch time and GB/s over the non-padded rows (one layer)."""
    from recurrent_state_update_gb300 import binding as bd
    dev = torch.device("cuda")
    bf = torch.bfloat16
    pool = SWEEP["pool"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(SWEEP["seed"] * 1000 + rank)
    ssm = torch.randn(pool, H, P, N, generator=gen, device=dev).mul_(0.1).to(bf)
    conv = torch.randn(pool, CD, W1, generator=gen, device=dev).mul_(0.1).to(bf)
    g = wl.rng(SWEEP["seed"] * 1000 + rank, 0)
    prm_np = wl.layer_params(g, SHAPE)
    prm = {k: torch.from_numpy(v).to(dev) for k, v in prm_np.items()}
    desc = bd.layer_desc(SHAPE)
    out = []
    for batch in SWEEP["batches"]:
        ids = wl.slot_ids(g, pool, batch, SWEEP["pad_frac"])
        live = int((ids >= 0).sum())
        slot = torch.from_numpy(ids).to(dev)
        inp = wl.decode_inputs(g, SHAPE, prm_np, batch, 1, wl.BF16)
        xbc = torch.from_numpy(inp["xbc"].view(np.int16)).to(dev).view(bf)
        z = torch.from_numpy(inp["z"].view(np.int16)).to(dev).view(bf)
        dt = torch.from_numpy(inp["dt"]).to(dev)
        y = torch.empty(batch, 1, H * P, dtype=bf, device=dev)

        def step():
            bd.mamba_state_update(desc, ssm, slot, xbc, dt, prm["A"], y, conv_pool=conv, conv_w=prm["conv_w"],
                                  D=prm["D"], dt_bias=prm["dt_bias"], z=z)

        # a graph of 16 launches replayed: small batches are timed on the GPU, not on the host's launch rate
        ms = _max_over_ranks(torch, dist, _time_graph(torch, step, max(args.steps // 4, 10), max(args.warmup, 3), dist,
                                                      reps=16))
        gbs = live * DECODE_BYTES_PER_TOKEN_LAYER / (ms * 1e-3) / 1e9
        out.append({"batch": batch, "live_rows": live, "us_per_launch": ms * 1e3, "gbs": gbs,
                    "hbm_frac": gbs / hbm_peak})
    return {"workload": SWEEP["name"], "launch": "CUDA graph replay (16 launches per graph)", "points": out}


M1 = wl.MAMBA1_DECODE
M1D, M1N, M1W = M1["d_inner"], M1["d_state"], M1["conv_kernel"]
# Mamba1 decode, per token-layer (bf16): state read + write, conv state read + write, x into the
# conv, its output written and read by the update, z in, y out, dt (fp32), B and C
M1_BYTES_PER_TOKEN_LAYER = 2 * M1D * M1N * 2 + 2 * M1D * (M1W - 1) * 2 + 5 * M1D * 2 + M1D * 4 + 2 * M1N * 2
# the state-update kernel alone: state read + write, x, z, y, dt, B, C
M1_UPDATE_BYTES = 2 * M1D * M1N * 2 + 3 * M1D * 2 + M1D * 4 + 2 * M1N * 2


def run_mamba1(torch, args, rank, dist, hbm_peak):
    """Mamba1 decode: every layer runs the conv update then the state update for batch 256 of a
    512-slot pool (bf16), 64 layers per step; the state-update kernel is also timed alone."""
    from recurrent_state_update_gb300 import binding as bd
    dev = torch.device("cuda")
    bf = torch.bfloat16
    L, batch, S = args.layers or M1["layers"], M1["batch"], M1["pool"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(M1["seed"] * 1000 + rank)
    ssm = [torch.randn(S, M1D, M1N, generator=gen, device=dev).mul_(0.1).to(bf) for _ in range(L)]
    conv = [torch.randn(S, M1D, M1W - 1, generator=gen, device=dev).mul_(0.1).to(bf) for _ in range(L)]
    g = wl.rng(M1["seed"] * 1000 + rank, 0)
    prm_np = wl.mamba1_params(g, M1D, M1N, M1W)
    prm = {k: torch.from_numpy(v).to(dev) for k, v in prm_np.items()}
    inp = wl.mamba1_inputs(g, prm_np, batch, M1N, wl.BF16)
    to = lambda a: torch.from_numpy(a.view(np.int16)).to(dev).view(bf)
    x_in = to(inp["x"]).view(batch, 1, M1D)
    x_c = torch.empty(batch, 1, M1D, dtype=bf, device=dev)
    B, C, z = to(inp["B"]), to(inp["C"]), to(inp["z"])
    dt = torch.from_numpy(inp["dt"]).to(dev)
    y = torch.empty(batch, M1D, dtype=bf, device=dev)
    slot = torch.from_numpy(wl.slot_ids(g, S, batch)).to(dev)
    desc = bd.mamba1_desc(M1D, M1N, M1W)

    def update(l):
        bd.mamba1_state_update(desc, ssm[l], slot, x_c.view(batch, M1D), dt, prm["A"], B, C, y, D=prm["D"],
                               dt_bias=prm["dt_bias"], z=z)

    def step():
        for l in range(L):
            bd.mamba1_conv_update(desc, conv[l], slot, x_in, prm["conv_w"], x_c)
            update(l)

    def updates():
        for l in range(L):
            update(l)

    # 128 short launches per step: timed from a CUDA graph (the host's launch rate would dominate)
    ms = _max_over_ranks(torch, dist, _time_graph(torch, step, max(args.steps // 4, 10), max(args.warmup, 3), dist))
    ms_u = _max_over_ranks(torch, dist, _time_graph(torch, updates, max(args.steps // 4, 10), max(args.warmup, 3),
                                                    dist))
    by = L * batch * M1_BYTES_PER_TOKEN_LAYER
    by_u = L * batch * M1_UPDATE_BYTES
    out = {"workload": M1["name"], "ms_per_step": ms, "gbs": by / (ms * 1e-3) / 1e9,
           "hbm_frac": by / (ms * 1e-3) / 1e9 / hbm_peak, "token_layers_per_s": L * batch / (ms * 1e-3),
           "algorithmic_bytes_per_token_layer": M1_BYTES_PER_TOKEN_LAYER, "launches_per_step": 2 * L,
           "launch": "CUDA graph replay (one graph per step)",
           "state_update": {"kernel": "k_mamba1_stream", "us_per_launch": ms_u * 1e3 / L,
                            "gbs": by_u / (ms_u * 1e-3) / 1e9, "hbm_frac": by_u / (ms_u * 1e-3) / 1e9 / hbm_peak,
                            "algorithmic_bytes_per_launch": batch * M1_UPDATE_BYTES}}
    del ssm, conv
    return out


CKPT_ROWS = 256  # slots restored, stored or loaded per call


def run_checkpoint(torch, args, rank, dist, hbm_peak):
    """Prefix-cache checkpoint operations at the Nemotron-H-8B shape on a 512-slot bf16 pool:
    restore (copy) of 256 slots into fresh slots, int8 store of 256 slots, int8 load of 256
    entries.  GB/s = algorithmic bytes (each state read once and written once) / time."""
    from recurrent_state_update_gb300 import binding as bd
    dev = torch.device("cuda")
    bf = torch.bfloat16
    gen = torch.Generator(device=dev)
    gen.manual_seed(7000 + rank)
    S = DECODE["pool"]
    ssm = torch.randn(S, H, P, N, generator=gen, device=dev).mul_(0.1).to(bf)
    conv = torch.randn(S, CD, W1, generator=gen, device=dev).mul_(0.1).to(bf)
    desc = bd.layer_desc(SHAPE)
    eb = bd.mamba_int8_entry_bytes(desc)
    store = torch.empty(CKPT_ROWS * eb, dtype=torch.uint8, device=dev)
    g = wl.rng(7000 + rank, 0)
    perm = g.permutation(S).astype(np.int32)
    src = torch.from_numpy(perm[:CKPT_ROWS].copy()).to(dev)
    dst = torch.from_numpy(perm[CKPT_ROWS:2 * CKPT_ROWS].copy()).to(dev)
    ent = torch.from_numpy(g.permutation(CKPT_ROWS).astype(np.int32)).to(dev)
    st_b, cv_b = H * P * N * 2, CD * W1 * 2
    q_b = H * P * N + H * N * 4 + cv_b
    legs = {
        "restore_copy": (lambda: bd.mamba_slot_copy(desc, ssm, src, dst, conv_pool=conv), 2 * (st_b + cv_b)),
        "int8_store": (lambda: bd.mamba_ckpt_store_int8(desc, ssm, src, ent, store, conv_pool=conv), st_b + cv_b + q_b),
        "int8_load": (lambda: bd.mamba_ckpt_load_int8(desc, ssm, ent, dst, store, conv_pool=conv), q_b + st_b + cv_b),
    }
    out = {"workload": f"{CKPT_ROWS} slots of a {S}-slot Nemotron-H-8B bf16 pool (2 MiB SSM + 60 KiB conv each)",
           "int8_entry_bytes": eb}
    for name, (fn, per_row) in legs.items():
        ms = _max_over_ranks(torch, dist, _time(torch, fn, max(args.steps, 20), max(args.warmup, 3), dist))
        gbs = CKPT_ROWS * per_row / (ms * 1e-3) / 1e9
        out[name] = {"us_per_call": ms * 1e3, "gbs": gbs, "hbm_frac": gbs / hbm_peak,
                     "algorithmic_bytes": CKPT_ROWS * per_row}
    return out


def run_prefill(torch, args, rank, world, dist, hbm_peak, bf16_peak):
    pre = PrefillWorkload(torch, rank)
    ms_pre = _max_over_ranks(torch, dist, _time(torch, pre.step, args.steps, max(args.warmup, 3), dist))
    fl = prefill_flops(pre.lengths, PREFILL["chunk"])
    by = prefill_bytes(pre.T, len(pre.lengths), pre.n_state_writes)
    prefill = {
        "tokens_per_s": pre.T * world / (ms_pre * 1e-3), "ms_per_layer": ms_pre,
        "workload": PREFILL["name"], "lengths": [int(v) for v in pre.lengths],
        "hbm_frac": by / (ms_pre * 1e-3) / 1e9 / hbm_peak,
        "tensor_frac": fl / (ms_pre * 1e-3) / 1e12 / bf16_peak,
        "algorithmic_bytes": by, "algorithmic_flops": fl,
        "launches_per_layer": 2,
        "kernel": "k_ssd_tc (tcgen05) after k_tc_meta",
    }
    ms_conv = _max_over_ranks(torch, dist, _time(torch, pre.step_conv, args.steps, max(args.warmup, 3), dist))
    by_conv = prefill_conv_bytes(pre.T, len(pre.lengths))
    prefill["conv"] = {
        "ms_per_layer": ms_conv, "gbs": by_conv / (ms_conv * 1e-3) / 1e9,
        "hbm_frac": by_conv / (ms_conv * 1e-3) / 1e9 / hbm_peak, "algorithmic_bytes": by_conv,
        "launches_per_layer": 2, "kernel": "k_conv_varlen, then k_conv_varlen_state",
    }
    ms_layer = _max_over_ranks(torch, dist, _time(torch, pre.step_layer, args.steps, max(args.warmup, 3), dist))
    prefill["conv_then_scan"] = {"ms_per_layer": ms_layer, "tokens_per_s": pre.T * world / (ms_layer * 1e-3)}
    del pre
    torch.cuda.empty_cache()
    return prefill


def decode_config(world, layers):
    """The decode workload as both arms report it."""
    return {"workload": DECODE["name"], "layers": layers, "global_batch": DECODE["batch"] * world,
            "pool_slots": DECODE["pool"], "shape": "H128 P64 N128 G8 W4 (conv_dim 10240)",
            "state_dtype": "bf16", "parallelism": f"dp{world} (independent slot pools)",
            "l2": "no flush: each launch touches 512 MiB of state (> 129 MB L2)"}


def emit(args, world, layers, ms, value, token_layers, achieved, launch_ms, hbm_peak, peak_src, e2e, ck, prefill,
         cpu, spec=None, sweep=None, ckpt=None, m1=None):
    line = {
        "metric": "decode state-update GB/s (and token-layers/s) vs HBM peak; prefill tokens/s",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded; no dataset)",
        "config": decode_config(world, layers),
        "token_layers_per_s": token_layers,
        "roofline": {"bound": "hbm", "kernel": "k_decode_stream", "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak, "peak_source": peak_src,
                     "traffic": _profile_traffic("decode_nemotron_b256"),
                     "algorithmic_bytes_per_launch": DECODE["batch"] * DECODE_BYTES_PER_TOKEN_LAYER,
                     "avg_launch_ms": launch_ms},
        "e2e": e2e,
        "gpu_launches": args.steps * layers,
        "clocks": ck,
        "prefill": prefill,
        "spec_decode": spec,
        "padding_sweep": sweep,
        "checkpoint": ckpt,
        "mamba1_decode": m1,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ------------------------------------------------------------------------------------------

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    rows = 32
    # one step = the oracle on `rows` rows of one decode layer (a bounded sample of the workload)
    import oracle
    seed = DECODE["seed"] * 1000
    g = wl.rng(seed, 0)
    prm = wl.layer_params(g, SHAPE)
    inp = wl.decode_inputs(g, SHAPE, prm, rows, 1, wl.BF16)
    st = wl.initial_states(wl.rng(seed, 99), SHAPE, rows, wl.BF16, wl.BF16)
    ssm, conv = wl.upcast(st["ssm"], wl.BF16), wl.upcast(st["conv"], wl.BF16)
    xbc, z = wl.upcast(inp["xbc"], wl.BF16), wl.upcast(inp["z"], wl.BF16).reshape(rows, 1, H, P)
    dt = inp["dt"].astype(np.float64)
    o = {k: v.astype(np.float64) for k, v in prm.items()}
    slot = np.arange(rows, dtype=np.int32)
    threads = oracle.default_threads()

    def step():
        oracle.decode(ssm, slot, xbc, dt, o["A"], conv_pool=conv, conv_w=o["conv_w"], D=o["D"],
                      dt_bias=o["dt_bias"], z=z, n_groups=G, nthreads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    value = rows * DECODE_BYTES_PER_TOKEN_LAYER / (el / args.steps) / 1e9
    sample = f"{rows} rows of one Nemotron-H-8B decode layer per step (fp64 C oracle)"
    line = {
        "impl": "reference",
        "metric": "decode state-update GB/s (and token-layers/s) vs HBM peak; prefill tokens/s",
        "value": value, "unit": "GB/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; no dataset)",
        "config": dict(decode_config(1, DECODE["layers"]), sample_rows_per_step=rows),
        "token_layers_per_s": rows / (el / args.steps),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--layers", type=int, default=0, help="decode layers per step (default: the workload's 48)")
    ap.add_argument("--only", choices=["all", "decode", "prefill", "spec", "sweep", "checkpoint", "mamba1"],
                    default="all",
                    help="time one form alone (profiling runs)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        # one process per GPU: N > 1 is launched by torch.distributed.run, which sets WORLD_SIZE
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch N > 1 ranks with "
                 f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py --gpus {args.gpus}")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
