"""Benchmark of the LCT codec hot path on GB300 (one JSON line on stdout).

A step is one pass of the whole hot path over one synthetic batch:
  1. lct_encode         shift estimate + block encode (byte split, stream
                        packing, overflow placement)
  2. lct_decode         streams -> BF16
  3. lct_sgd_step_fused W <- W - eta*M on the compressed W (the tensor just
                        encoded) and a compressed momentum M
value = uncompressed BF16 GB/s through the codec: 2N bytes encoded plus 2N
bytes decoded per step, over the time from the step's start to the end of its
decode (an event between the decode and the fused SGD; the fused SGD's own
time and rate are reported beside it, and ms_per_step covers the whole step).

Default workload: 2^24 BF16 values ~ Laplace(0, 0.01), Laplace codebook,
CLEAN blocks; M ~ Laplace(0, 1e-3).  L2 is flushed (256 MiB write) before
every timed step, outside the step's events.  The per-kernel times (and the
roofline of the dominant kernel) come from a second pass with the L2 flushed
before every kernel.  breakdown.configs holds the five workload
configurations (one block of N(0,0.02); 2^24 Laplace; 2^26 heavy-tailed
MEDIUM; 162M fused SGD; GELU activations at 9 scales, HIGH), each with the
oracle timed on a block sample of it.

--impl reference times the CPU oracle (single thread) on the same workload.
--gpus N runs one replica per GPU (weak scaling, no collective on the data
path); under torchrun the ranks come from the environment, otherwise bench.py
starts its N ranks itself.  Timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import socket
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD_TEXT = {
    "gauss_block": "65,536 BF16 ~ N(0,0.02), Gaussian codebook, CLEAN (one block); step = encode + decode + fused "
                   "SGD (M ~ Laplace(0,1e-3))",
    "laplace_16m": "2^24 BF16 ~ Laplace(0,0.01), Laplace codebook, CLEAN; step = encode + decode + fused SGD "
                   "(M ~ Laplace(0,1e-3))",
    "heavy_64m": "2^26 BF16 Student-t(3)*1e-3 with 0.1% x1e4 outliers and 1% subnormals, power-law codebook, "
                 "MEDIUM; step = encode + decode + fused SGD (M ~ Laplace(0,1e-3))",
    "gelu_act": "[8,4096,3072] GELU(N(0,1)) with 30% zeros, Gaussian(1) codebook, HIGH; step = encode + decode + "
                "fused SGD (M ~ Laplace(0,1e-3))",
    "gelu_act_zero": "[8,4096,3072] GELU(N(0,1)) with 30% zeros, Gaussian(1) codebook with a 0.3 point mass at zero, "
                     "HIGH; step = encode + decode + fused SGD (M ~ Laplace(0,1e-3))",
    "sgd_162m": "162,000,000 BF16 W ~ N(0,0.02), M ~ N(0,1e-3), Gaussian codebooks, CLEAN; step = encode + decode "
                "+ fused SGD",
    "adamw_162m": "162,000,000 BF16 W ~ N(0,0.02), M ~ N(0,1e-4), V = |N(0,1e-8)|, dense BF16 gradient ~ "
                  "N(0,1e-4), CLEAN, W, M and V updated in place; step = one fused AdamW step (moments pass + "
                  "weight pass; lr 1e-3, betas 0.9/0.999, eps 1e-8, weight decay 0.01)",
    "momentum_162m": "162,000,000 BF16 W ~ N(0,0.02), M ~ N(0,1e-3), dense BF16 gradient ~ N(0,1e-4), Gaussian "
                     "codebooks, CLEAN, W and M updated in place; step = one fused SGD-with-momentum step "
                     "(mu = 0.9, eta = 1e-3)",
}
SGD_MOMENTUM = {"gauss_block": ("laplace", 1e-3), "laplace_16m": ("laplace", 1e-3), "heavy_64m": ("laplace", 1e-3),
                "gelu_act": ("laplace", 1e-3), "gelu_act_zero": ("laplace", 1e-3), "sgd_162m": ("gaussian", 1e-3)}
ETA = float(np.float32(1e-3))
L2_FLUSH_BYTES = 256 << 20


# The headline metric: GB/s of uncompressed BF16 through the codec, the
# fraction of HBM bandwidth on the bytes actually moved, and the ratio.
METRIC = "encode/decode GB/s (uncompressed BF16) and % of HBM peak; compression ratio"


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), ws


def dist_backend() -> str:
    return os.environ.get("LCT_DIST_BACKEND", "nccl")


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (the job's time is its slowest
    rank's); `value` itself when no process group is running."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_units(n_per_rank: int, world: int) -> int:
    """Values the whole job processes per step: every rank runs its own
    replica of the workload (weak scaling, no collective on the data path)."""
    return n_per_rank * world


# ----------------------------------------------------------- rank launch

def _free_port() -> int:
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_entry(rank, world, port, backend, target, targs, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), LOCAL_RANK=str(rank),
                      WORLD_SIZE=str(world), LCT_DIST_BACKEND=backend)
    q.put((rank, target(*targs)))


def spawn_ranks(world: int, target, targs=(), backend: str = "nccl", timeout: float = 1800.0) -> dict:
    """Run target(*targs) in `world` fresh processes, one rank each (RANK,
    LOCAL_RANK, WORLD_SIZE and a 127.0.0.1 rendezvous in the environment, as
    torchrun would set them); returns {rank: target's return value}.  A rank
    that fails makes this raise."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_entry, args=(r, world, port, backend, target, targs, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=timeout)
    bad = [r for r, p in enumerate(procs) if p.exitcode != 0]
    for p in procs:
        if p.is_alive():
            p.kill()
    if bad:
        raise RuntimeError("ranks %s failed" % bad)
    out = {}
    while not q.empty():
        r, v = q.get()
        out[r] = v
    return out


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, bus_id: str | None):
        self.bus_id = bus_id
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits", "-lms", "200"]
        if self.bus_id:
            cmd += ["-i", self.bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ GPU arm

def placement_launches(n: int, level: str) -> int:
    """Extra launches per written tensor: the writers place block offsets in a
    separate one-CTA kernel on grids of at least four blocks per SM."""
    import torch
    block = 65536 if level == "CLEAN" else 32768
    nblocks = (n + block - 1) // block
    return 1 if nblocks >= 4 * torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count else 0


def algorithmic_bytes(sizes, ovf_used: int) -> int:
    """Bytes of one compressed tensor that a pass over it moves: sign-fraction
    bytes, full fixed slots, markers, block offsets and the overflow used.
    Callers add the 2 bytes per value of the uncompressed side where there is
    one (encode reads it, decode writes it)."""
    return int(sizes.sf_bytes + sizes.slot_bytes + sizes.marker_bytes + sizes.blk_off_bytes + ovf_used)


class KernelTimer:
    """Device time of one call with the L2 flushed (a 256 MiB write) before
    it: events on the launching stream around the call only."""

    def __init__(self, torch, stream):
        self.torch = torch
        self.stream = stream
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")

    def __call__(self, fn, reps: int) -> float:
        torch = self.torch
        ts = []
        for _ in range(reps):
            self.flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            fn()
            e1.record(self.stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.mean(ts)


def codebooks_for(B, wl):
    if "zero_frac" in wl:
        return B.lct_codebook_build_zero_atom(wl["model"], wl["scale"], wl["shape"], wl["zero_frac"])
    return B.lct_codebook_build(wl["model"], wl["scale"], wl["shape"])


def run_gpu(args):
    import torch
    import torch.distributed as dist

    rank, local_rank, world = dist_env()
    if world > 1:
        dist.init_process_group(dist_backend())
    torch.cuda.set_device(local_rank)
    from lossless_bf16_tensor_gb300 import binding as B
    from lossless_bf16_tensor_gb300 import synth

    wl = synth.WORKLOADS[args.workload]
    if "adamw" in wl:
        return run_gpu_adamw(args, rank, local_rank, world)
    if "gradient" in wl:
        return run_gpu_momentum(args, rank, local_rank, world)
    n = wl["n"]
    level = B.LEVELS[wl["level"]]
    x_np = synth.generate(args.workload)
    mm, ms = SGD_MOMENTUM[args.workload]
    m_np = synth.laplace(n, ms, seed=2) if mm == "laplace" else synth.momentum(args.workload)
    cb = codebooks_for(B, wl)
    cbm = B.lct_codebook_build(mm, ms)

    stream = torch.cuda.current_stream()
    x = torch.from_numpy(x_np.view(np.int16)).cuda()
    md = torch.from_numpy(m_np.view(np.int16)).cuda()
    X = B.CompressedTensor(n, level)
    Mc = B.CompressedTensor(n, level)
    Wn = B.CompressedTensor(n, level)
    y = torch.empty_like(x)
    B.lct_encode(md, cbm, Mc)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")

    def step(evs=None, st=stream):
        # evs: (step start, decode end, step end)
        if evs:
            evs[0].record(st)
        B.lct_encode(x, cb, X, st)
        B.lct_decode(X, cb, y, st)
        if evs:
            evs[1].record(st)
        B.lct_sgd_step_fused(X, cb, Mc, cbm, ETA, Wn, st)
        if evs:
            evs[2].record(st)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    # correctness of what is timed: the round trip is exact and nothing latched
    assert torch.equal(y, x), "decode(encode(x)) != x"
    for t in (X, Mc, Wn):
        assert t.state().status == 0

    bus = None
    try:
        bus = torch.cuda.get_device_properties(local_rank).pci_bus_id
    except AttributeError:
        pass
    clocks = ClockSampler(None if world == 1 and bus is None else bus)
    # The timed steps carry one event between the decode and the fused SGD
    # (the encode -> decode hand-over keeps its programmatic early launch).
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.4)
    for k in range(args.steps):
        flush.zero_()
        step(evs[k])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ed_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in evs), device="cuda") / args.steps
    ms_step = max_over_ranks(sum(e[0].elapsed_time(e[2]) for e in evs), device="cuda") / args.steps
    # Per-kernel device times, the L2 flushed before every kernel.
    timer = KernelTimer(torch, stream)
    reps = max(3, args.steps // 2)
    t_ms = {"encode": timer(lambda: B.lct_encode(x, cb, X, stream), reps),
            "decode": timer(lambda: B.lct_decode(X, cb, y, stream), reps),
            "sgd": timer(lambda: B.lct_sgd_step_fused(X, cb, Mc, cbm, ETA, Wn, stream), reps)}
    # The same step captured once in a CUDA graph and replayed (every call
    # only enqueues work, so it captures); reported beside the direct step.
    graph_ms = None
    if world == 1:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):  # captured on torch's side stream
            step(st=torch.cuda.current_stream())
        gevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for k in range(args.steps):
            flush.zero_()
            gevs[k][0].record(stream)
            g.replay()
            gevs[k][1].record(stream)
        torch.cuda.synchronize()
        graph_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in gevs)
        assert torch.equal(y, x), "decode(encode(x)) != x after graph replay"
    clk = clocks.stop()

    sx, sm_, sw = X.state(), Mc.state(), Wn.state()
    sizes = X.sizes
    bytes_x = algorithmic_bytes(sizes, sx.ovf_used)
    bytes_m = algorithmic_bytes(sizes, sm_.ovf_used)
    bytes_w = algorithmic_bytes(sizes, sw.ovf_used)
    alg = {"encode": 2 * n + bytes_x, "decode": 2 * n + bytes_x, "sgd": bytes_x + bytes_m + bytes_w}
    peak, peak_kind = hbm_peak()
    frac = {k: alg[k] / (t_ms[k] * 1e-3) / 1e9 / peak for k in alg}
    dom = max(t_ms, key=t_ms.get)
    achieved = alg[dom] / (t_ms[dom] * 1e-3) / 1e9
    value = 4 * replica_units(n, world) / (ed_ms * 1e-3) / 1e9

    traffic = stored_traffic(args.workload, dom)

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, B, x_np, n, level, cb, world)

    configs = None
    if world == 1 and not args.no_configs:
        configs = run_configs(B, synth, timer, stream, peak)

    if rank != 0:
        return None
    ratio_all_in = 2.0 * n / (sizes.fixed_bytes + sx.ovf_used)
    ratio_payload = 2.0 * n / (sizes.sf_bytes + sizes.slot_bytes + sx.ovf_used)
    cpu = None if args.no_cpu_baseline or world > 1 else cpu_baseline(args.workload, args.cpu_blocks)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "u32+f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload, "n": n,
                   "level": wl["level"], "l2": "flushed before every step (256 MiB write, outside the events); "
                   "per-kernel times flushed before every kernel",
                   "value": "4N uncompressed bytes (encode 2N + decode 2N) per step / time from step start to "
                            "decode end; the fused SGD runs in every step after the decode",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": alg[dom]},
        "breakdown": {
            "encode_gbs_uncompressed": round(2 * n / (t_ms["encode"] * 1e-3) / 1e9, 1),
            "decode_gbs_uncompressed": round(2 * n / (t_ms["decode"] * 1e-3) / 1e9, 1),
            "sgd_gelem_per_s": round(n / (t_ms["sgd"] * 1e-3) / 1e9, 3),
            "ms": {k: round(v, 4) for k, v in t_ms.items()},
            "ms_encode_decode_in_step": round(ed_ms, 4),
            "kernel_times": "each kernel alone, L2 flushed before it, mean of %d" % reps,
            "ms_per_step_cuda_graph": None if graph_ms is None else round(graph_ms, 4),
            "hbm_frac_of_%s" % peak_kind: {k: round(v, 4) for k, v in frac.items()},
            "compression_ratio_all_in": round(ratio_all_in, 5),
            "compression_ratio_payload": round(ratio_payload, 5),
            "overflow_bytes": int(sx.ovf_used),
            "spill_fraction": round(sx.ovf_used / n, 6),
            "allocated_bits_per_exponent": round(8.0 * sizes.slot_bytes / n, 4),
            "configs": configs,
        },
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": (5 + 2 * placement_launches(n, wl["level"])) * args.steps,
        "cpu_baseline": cpu,
    }
    return line


def run_e2e(args, B, x_np, n, level, cb, world):
    """Encode and decode through the public API with host buffers: every step
    uploads its input from pinned host memory, encodes, decodes and downloads
    the decoded values.  Steps are pipelined as a user streaming tensors
    would: uploads, compute and downloads run on three streams with two buffer
    sets, so step k+1's upload overlaps step k's compute and step k-1's
    download.  Timed from the first upload to the last download; the working
    set (two buffer sets, ~115 MB each at 2^24) exceeds L2."""
    import torch
    dev = torch.device("cuda")
    hx = torch.from_numpy(x_np.view(np.int16)).pin_memory()
    hy = [torch.empty(n, dtype=torch.int16).pin_memory() for _ in range(2)]
    xs = [torch.empty(n, dtype=torch.int16, device=dev) for _ in range(2)]
    ys = [torch.empty(n, dtype=torch.int16, device=dev) for _ in range(2)]
    Xs = [B.CompressedTensor(n, level) for _ in range(2)]
    s_up, s_run, s_down = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("up", "run", "down")}
    started = [False, False]

    def step(k):
        i = k % 2
        if started[i]:
            s_up.wait_event(ev["run"][i])     # step k-2's encode has read xs[i]
            s_run.wait_event(ev["down"][i])   # step k-2's download has read ys[i]
        started[i] = True
        with torch.cuda.stream(s_up):
            xs[i].copy_(hx, non_blocking=True)
            ev["up"][i].record(s_up)
        s_run.wait_event(ev["up"][i])
        B.lct_encode(xs[i], cb, Xs[i], s_run)
        B.lct_decode(Xs[i], cb, ys[i], s_run)
        ev["run"][i].record(s_run)
        s_down.wait_event(ev["run"][i])
        with torch.cuda.stream(s_down):
            hy[i].copy_(ys[i], non_blocking=True)
            ev["down"][i].record(s_down)

    torch.cuda.synchronize()
    for k in range(4):
        step(k)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_up)
    for k in range(args.steps):
        step(k)
    s_up.wait_stream(s_down)
    t1.record(s_up)
    torch.cuda.synchronize()
    for i in range(2):
        assert torch.equal(hy[i], hx), "decoded values differ from the input"
        assert Xs[i].state().status == 0, "a status was latched"
    e_ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, device="cuda")
    return {"value": round(4 * replica_units(n, world) / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(e_ms, 4), "h2d_bytes_per_step": 2 * n, "d2h_bytes_per_step": 2 * n,
            "pipelined": "upload / encode + decode / download on three streams, two buffer sets"}


# ------------------------------------------------- the five configurations

def oracle_codec_sample(x, cb_args, level, nblocks):
    """The oracle's encode and decode of the first `nblocks` blocks of x on
    one host core: (values, encode seconds, decode seconds)."""
    import oracle
    block, _ = oracle.geometry(level)
    k = min(x.size, nblocks * block)
    xs = np.ascontiguousarray(x[:k])
    model, scale, shape, zf = cb_args
    cb = oracle.codebook_build_zero_atom(model, scale, shape, zf) if zf else oracle.codebook_build(model, scale, shape)
    t0 = time.perf_counter()
    c = oracle.encode(xs, cb, level)
    t1 = time.perf_counter()
    rc, y = oracle.decode(c, cb)
    t2 = time.perf_counter()
    assert rc == 0 and np.array_equal(y, xs)
    return k, t1 - t0, t2 - t1


def run_configs(B, synth, timer, stream, peak):
    """encode / decode GB/s, fused-SGD rate, HBM fractions and ratios for the
    five workload configurations, each beside the oracle on a block sample."""
    import torch
    reps = 5
    model_id = {"gaussian": 0, "laplace": 1, "powerlaw": 2}
    out = {}

    def codec_record(name, x_np, wl, n, level, rounds=None, sample_blocks=8):
        cb = codebooks_for(B, wl)
        x = torch.from_numpy(x_np.view(np.int16)).cuda()
        X = B.CompressedTensor(n, level)
        y = torch.empty_like(x)
        xs = [x] if rounds is None else [
            (x.view(torch.bfloat16).float() * (2.0 ** k)).to(torch.bfloat16).view(torch.int16) for k in rounds]
        te, td, ratios = [], [], []
        for xr in xs:
            B.lct_encode(xr, cb, X, stream)
            B.lct_decode(X, cb, y, stream)
            torch.cuda.synchronize()
            assert torch.equal(y, xr), name + ": decode(encode(x)) != x"
            st = X.state()
            assert st.status == 0, name
            te.append(timer(lambda: B.lct_encode(xr, cb, X, stream), reps))
            td.append(timer(lambda: B.lct_decode(X, cb, y, stream), reps))
            ratios.append((2.0 * n / (X.sizes.fixed_bytes + st.ovf_used),
                           2.0 * n / (X.sizes.sf_bytes + X.sizes.slot_bytes + st.ovf_used), st.ovf_used))
        sizes = X.sizes
        ovf = statistics.mean(r[2] for r in ratios)
        alg = 2 * n + algorithmic_bytes(sizes, int(ovf))
        t_e, t_d = statistics.mean(te), statistics.mean(td)
        ocb = (model_id[wl["model"]], wl["scale"], wl["shape"], wl.get("zero_frac", 0.0))
        on, oe, od = oracle_codec_sample(x_np, ocb, level, sample_blocks)
        rec = {"n": n, "level": wl["level"], "encode_gbs_uncompressed": round(2 * n / (t_e * 1e-3) / 1e9, 1),
               "decode_gbs_uncompressed": round(2 * n / (t_d * 1e-3) / 1e9, 1), "ms": {"encode": round(t_e, 4),
               "decode": round(t_d, 4)}, "hbm_frac": {"encode": round(alg / (t_e * 1e-3) / 1e9 / peak, 4),
               "decode": round(alg / (t_d * 1e-3) / 1e9 / peak, 4)},
               "compression_ratio_all_in": round(statistics.mean(r[0] for r in ratios), 5),
               "compression_ratio_payload": round(statistics.mean(r[1] for r in ratios), 5),
               "spill_fraction": round(ovf / n, 6),
               "oracle": {"values": on, "encode_s": round(oe, 4), "decode_s": round(od, 4),
                          "encode_gbs": round(2 * on / oe / 1e9, 5), "decode_gbs": round(2 * on / od / 1e9, 5),
                          "cores": 1, "host_cpus": os.cpu_count() or 0,
                          "sample": "first %d block(s), oracle single-threaded" % -(-on // sizes.block)}}
        if rounds is not None:
            rec["rounds"] = "x * 2^k for k = %d..%d, shift re-estimated by every encode" % (rounds[0], rounds[-1])
            rec["per_round_gbs"] = {"encode": [round(2 * n / (t * 1e-3) / 1e9, 1) for t in te],
                                    "decode": [round(2 * n / (t * 1e-3) / 1e9, 1) for t in td]}
        del X, x, y, xs
        torch.cuda.empty_cache()
        return rec

    for name in ("gauss_block", "laplace_16m", "heavy_64m", "sgd_162m", "gelu_act"):
        wl = synth.WORKLOADS[name]
        n, level = wl["n"], B.LEVELS[wl["level"]]
        x_np = synth.generate(name)
        rec = codec_record(name, x_np, wl, n, level, rounds=wl.get("pow2"), sample_blocks=8)
        if name == "sgd_162m":
            rec["sgd"] = run_sgd_config(B, synth, timer, stream, peak, x_np, wl, n, level)
        rec["workload"] = WORKLOAD_TEXT[name]
        out[name] = rec
        del x_np
    return out


def run_sgd_config(B, synth, timer, stream, peak, w_np, wl, n, level):
    """Fused SGD steps W <- W - eta*M on compressed W and M (out of place,
    two W tensors used in turn), the codebook and shift fixed."""
    import torch
    cbw = B.lct_codebook_build(wl["model"], wl["scale"], wl["shape"])
    cbm = B.lct_codebook_build(wl["momentum"]["model"], wl["momentum"]["scale"])
    Ws = [B.CompressedTensor(n, level), B.CompressedTensor(n, level)]
    M = B.CompressedTensor(n, level)
    B.lct_encode(torch.from_numpy(w_np.view(np.int16)).cuda(), cbw, Ws[0], stream)
    B.lct_encode(torch.from_numpy(synth.momentum("sgd_162m").view(np.int16)).cuda(), cbm, M, stream)
    eta = float(np.float32(wl["eta"]))
    steps = 10
    k = [0]

    def one():
        B.lct_sgd_step_fused(Ws[k[0] % 2], cbw, M, cbm, eta, Ws[(k[0] + 1) % 2], stream)
        k[0] += 1
    for _ in range(2):  # untimed: the kernel's first launch also loads its code
        one()
    torch.cuda.synchronize()
    t = timer(one, steps)
    torch.cuda.synchronize()
    cur = Ws[k[0] % 2]
    st, sm_ = cur.state(), M.state()
    assert st.status == 0
    sizes = cur.sizes
    alg = 2 * algorithmic_bytes(sizes, st.ovf_used) + algorithmic_bytes(sizes, sm_.ovf_used)
    res = {"steps": steps, "ms_per_step": round(t, 4), "gelem_per_s": round(n / (t * 1e-3) / 1e9, 3),
           "hbm_frac": round(alg / (t * 1e-3) / 1e9 / peak, 4),
           "compression_ratio_all_in_after": round(2.0 * n / (sizes.fixed_bytes + st.ovf_used), 5),
           "eta": eta, "l2": "flushed before every step"}
    del Ws, M
    torch.cuda.empty_cache()
    return res


def run_gpu_momentum(args, rank, local_rank, world):
    """One fused SGD-with-momentum step per timed step on compressed W and M
    (both in place, overflow regions ping-pong between steps)."""
    import torch
    import torch.distributed as dist
    from lossless_bf16_tensor_gb300 import binding as B
    from lossless_bf16_tensor_gb300 import synth

    wl = synth.WORKLOADS[args.workload]
    n = wl["n"]
    level = B.LEVELS[wl["level"]]
    eta, mu = float(np.float32(wl["eta"])), float(np.float32(wl["mu"]))
    cbw = B.lct_codebook_build(wl["model"], wl["scale"], wl["shape"])
    cbm = B.lct_codebook_build(wl["momentum"]["model"], wl["momentum"]["scale"])
    stream = torch.cuda.current_stream()
    W = B.CompressedTensor(n, level)
    M = B.CompressedTensor(n, level)
    B.lct_encode(torch.from_numpy(synth.generate(args.workload).view(np.int16)).cuda(), cbw, W, stream)
    B.lct_encode(torch.from_numpy(synth.momentum(args.workload).view(np.int16)).cuda(), cbm, M, stream)
    grads = [torch.from_numpy(synth.gradient(args.workload, s).view(np.int16)).cuda() for s in (1, 2)]
    Wb = [W, B.CompressedTensor(n, level, like=W)]
    Mb = [M, B.CompressedTensor(n, level, like=M)]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    count = [0]

    def step():
        k = count[0]
        B.lct_sgd_momentum_step_fused(Wb[k % 2], cbw, Mb[k % 2], cbm, grads[k % 2], eta, mu,
                                      Wb[(k + 1) % 2], Mb[(k + 1) % 2], stream)
        count[0] += 1

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    cur_w, cur_m = Wb[count[0] % 2], Mb[count[0] % 2]
    assert cur_w.state().status == 0 and cur_m.state().status == 0
    clocks = ClockSampler(None)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.4)
    for k in range(args.steps):
        flush.zero_()
        evs[k][0].record(stream)
        step()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    per = [a.elapsed_time(b) for a, b in evs]
    ms_step = max_over_ranks(sum(per), device="cuda") / args.steps
    sw, sm_ = Wb[count[0] % 2].state(), Mb[count[0] % 2].state()
    assert sw.status == 0 and sm_.status == 0
    sizes = W.sizes
    # read W, M compressed and the dense gradient; write W, M compressed
    alg = 2 * algorithmic_bytes(sizes, sw.ovf_used) + 2 * algorithmic_bytes(sizes, sm_.ovf_used) + 2 * n
    peak, peak_kind = hbm_peak()
    t_ms = statistics.mean(per)
    achieved = alg / (t_ms * 1e-3) / 1e9
    value = replica_units(n, world) / (ms_step * 1e-3) / 1e9
    traffic = stored_traffic(args.workload, "momentum")
    if rank != 0:
        return None
    cpu = None
    if not (args.no_cpu_baseline or world > 1):
        dt, nv = oracle_momentum_time(args.workload, args.cpu_blocks or 256)
        cpu = {"value": round(nv / dt / 1e9, 5), "unit": "Gelem/s", "cores": 1, "kind": "oracle",
               "sample": "first %d values of %s, one momentum step; host %s, oracle single-threaded"
                         % (nv, args.workload, cpu_model()), "seconds": round(dt, 3)}
    return {
        "metric": "fused SGD-with-momentum step on compressed W and M: elements per second",
        "value": round(value, 3), "unit": "Gelem/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u32+f32", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload, "n": n, "level": wl["level"],
                   "l2": "flushed before every step (256 MiB write, outside the events)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "kernel": "momentum", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": alg},
        "breakdown": {"compression_ratio_all_in_w": round(2.0 * n / (sizes.fixed_bytes + sw.ovf_used), 5),
                      "compression_ratio_all_in_m": round(2.0 * n / (sizes.fixed_bytes + sm_.ovf_used), 5),
                      "overflow_bytes_w": int(sw.ovf_used), "overflow_bytes_m": int(sm_.ovf_used)},
        "clocks": clk, "e2e": None, "gpu_launches": (2 + placement_launches(n, wl["level"])) * args.steps,
        "cpu_baseline": cpu,
    }


def run_gpu_adamw(args, rank, local_rank, world):
    """One fused AdamW step per timed step on compressed W, M and V (all in
    place, overflow regions ping-pong between steps)."""
    import torch
    import torch.distributed as dist
    from lossless_bf16_tensor_gb300 import binding as B
    from lossless_bf16_tensor_gb300 import synth

    wl = synth.WORKLOADS[args.workload]
    n = wl["n"]
    level = B.LEVELS[wl["level"]]
    hp = wl["adamw"]
    cbs = [B.lct_codebook_build(wl["model"], wl["scale"], wl["shape"]),
           B.lct_codebook_build(wl["momentum"]["model"], wl["momentum"]["scale"]),
           B.lct_codebook_build(wl["second"]["model"], wl["second"]["scale"])]
    stream = torch.cuda.current_stream()
    data = [synth.generate(args.workload), synth.momentum(args.workload), synth.second_moment(args.workload)]
    T = [B.CompressedTensor(n, level) for _ in range(3)]
    for x, cb, t in zip(data, cbs, T):
        B.lct_encode(torch.from_numpy(x.view(np.int16)).cuda(), cb, t, stream)
    del data
    grads = [torch.from_numpy(synth.gradient(args.workload, s).view(np.int16)).cuda() for s in (1, 2)]
    bufs = [T, [B.CompressedTensor(n, level, like=t) for t in T]]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    count = [0]

    def step():
        k = count[0]
        cur, nxt = bufs[k % 2], bufs[(k + 1) % 2]
        B.lct_adamw_step_fused(cur[0], cbs[0], cur[1], cbs[1], cur[2], cbs[2], grads[k % 2], hp["lr"], hp["beta1"],
                               hp["beta2"], hp["eps"], hp["weight_decay"], k + 1, nxt[0], nxt[1], nxt[2], stream)
        count[0] += 1

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert all(t.state().status == 0 for t in bufs[count[0] % 2])
    clocks = ClockSampler(None)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.4)
    for k in range(args.steps):
        flush.zero_()
        evs[k][0].record(stream)
        step()
        evs[k][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    per = [a.elapsed_time(b) for a, b in evs]
    ms_step = max_over_ranks(sum(per), device="cuda") / args.steps
    st = [t.state() for t in bufs[count[0] % 2]]
    assert all(s_.status == 0 for s_ in st)
    sizes = T[0].sizes
    ab = [algorithmic_bytes(sizes, s_.ovf_used) for s_ in st]
    # moments pass: read M, V, g, write M, V; weight pass: read W, M, V, write W
    alg = 2 * ab[1] + 2 * ab[2] + 2 * n + 2 * ab[0] + ab[1] + ab[2]
    peak, peak_kind = hbm_peak()
    achieved = alg / (statistics.mean(per) * 1e-3) / 1e9
    if rank != 0:
        return None
    cpu = None
    if not (args.no_cpu_baseline or world > 1):
        dt, nv = oracle_adamw_time(args.workload, args.cpu_blocks or 64)
        cpu = {"value": round(nv / dt / 1e9, 5), "unit": "Gelem/s", "cores": 1, "kind": "oracle",
               "sample": "first %d values of %s, one AdamW step; host %s, oracle single-threaded"
                         % (nv, args.workload, cpu_model()), "seconds": round(dt, 3)}
    return {
        "metric": "fused AdamW step on compressed W, M and V: elements per second",
        "value": round(replica_units(n, world) / (ms_step * 1e-3) / 1e9, 3), "unit": "Gelem/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u32+f32", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload, "n": n, "level": wl["level"],
                   "l2": "flushed before every step (256 MiB write, outside the events)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "roofline": {"bound": "hbm", "kernel": "adamw (moments pass + weight pass, one call)",
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": stored_traffic(args.workload, "adamw"),
                     "algorithmic_bytes_per_launch": alg},
        "breakdown": {"compression_ratio_all_in": [round(2.0 * n / (sizes.fixed_bytes + s_.ovf_used), 5) for s_ in st],
                      "overflow_bytes": [int(s_.ovf_used) for s_ in st]},
        "clocks": clk, "e2e": None, "gpu_launches": (4 + 2 * placement_launches(n, wl["level"])) * args.steps,
        "cpu_baseline": cpu,
    }


def oracle_adamw_time(workload: str, nblocks_sample: int):
    """Time one oracle AdamW step on the first `nblocks_sample` blocks."""
    import oracle
    from lossless_bf16_tensor_gb300 import synth
    wl = synth.WORKLOADS[workload]
    level = {"CLEAN": 0, "MEDIUM": 1, "HIGH": 2}[wl["level"]]
    block, _ = oracle.geometry(level)
    k = min(wl["n"], nblocks_sample * block)
    xs = [synth.generate(workload, k), synth.momentum(workload, k), synth.second_moment(workload, k)]
    g = synth.gradient(workload, 1, k)
    model = {"gaussian": 0, "laplace": 1, "powerlaw": 2}
    cbs = [oracle.codebook_build(model[wl["model"]], wl["scale"]),
           oracle.codebook_build(model[wl["momentum"]["model"]], wl["momentum"]["scale"]),
           oracle.codebook_build(model[wl["second"]["model"]], wl["second"]["scale"])]
    T = [oracle.encode(x, cb, level) for x, cb in zip(xs, cbs)]
    hp = wl["adamw"]
    kc = oracle.adamw_constants(hp["lr"], hp["beta1"], hp["beta2"], hp["eps"], hp["weight_decay"], 1)
    t0 = time.perf_counter()
    oracle.adamw_step(T[0], cbs[0], T[1], cbs[1], T[2], cbs[2], g, kc)
    return time.perf_counter() - t0, k


def oracle_momentum_time(workload: str, nblocks_sample: int):
    """Time one oracle momentum step on the first `nblocks_sample` blocks."""
    import oracle
    from lossless_bf16_tensor_gb300 import synth
    wl = synth.WORKLOADS[workload]
    level = {"CLEAN": 0, "MEDIUM": 1, "HIGH": 2}[wl["level"]]
    block, _ = oracle.geometry(level)
    k = min(wl["n"], nblocks_sample * block)
    w, m = synth.generate(workload, k), synth.momentum(workload, k)
    g = synth.gradient(workload, 1, k)
    cbw = oracle.codebook_build(0, wl["scale"])
    cbm = oracle.codebook_build(0, wl["momentum"]["scale"])
    W, M = oracle.encode(w, cbw, level), oracle.encode(m, cbm, level)
    t0 = time.perf_counter()
    oracle.sgd_momentum_step(W, cbw, M, cbm, g, float(np.float32(wl["eta"])), float(np.float32(wl["mu"])))
    return time.perf_counter() - t0, k


# Device source each kernel's DRAM traffic depends on (the shared device
# header and the kernel's own file); host code does not enter the hash.
KERNEL_SOURCES = {"encode": ("encode.cu",), "decode": ("decode.cu",), "sgd": ("sgd.cu",),
                  "momentum": ("momentum.cu",), "adamw": ("momentum.cu", "sgd.cu")}


def stored_traffic(workload: str, kernel: str):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the
    ncu summary in profiles/traffic.json, or None when none was taken of the
    kernel's current source."""
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tpath):
        return None
    with open(tpath) as f:
        entry = json.load(f).get(workload, {}).get(kernel)
    if entry and entry.get("source_hash") == kernel_source_hash(kernel):
        return entry["bytes_per_launch"]
    return None


def kernel_source_hash(kernel: str) -> str:
    """Hash of the source a kernel's measured traffic belongs to: a stored
    ncu traffic figure is used only while this hash is unchanged."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lossless_bf16_tensor_gb300", "csrc")
    for fn in ("codec_dev.cuh", "internal.h") + KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------ oracle (CPU) arm

def oracle_step_inputs(workload: str, nblocks_sample: int | None):
    """The oracle's inputs for one step of the workload (or of its first
    `nblocks_sample` blocks): x, its codebook, the encoded M and M's codebook."""
    import oracle
    from lossless_bf16_tensor_gb300 import synth
    wl = synth.WORKLOADS[workload]
    x = synth.generate(workload)
    mm, ms = SGD_MOMENTUM[workload]
    m = synth.laplace(x.size, ms, seed=2) if mm == "laplace" else synth.momentum(workload)
    level = {"CLEAN": 0, "MEDIUM": 1, "HIGH": 2}[wl["level"]]
    block, _ = oracle.geometry(level)
    if nblocks_sample:
        k = min(x.size, nblocks_sample * block)
        x, m = x[:k], m[:k]
    model = {"gaussian": 0, "laplace": 1, "powerlaw": 2}
    if "zero_frac" in wl:
        cb = oracle.codebook_build_zero_atom(model[wl["model"]], wl["scale"], wl["shape"], wl["zero_frac"])
    else:
        cb = oracle.codebook_build(model[wl["model"]], wl["scale"], wl["shape"])
    cbm = oracle.codebook_build(model[mm], ms)
    return x, cb, oracle.encode(m, cbm, level), cbm, level


def oracle_step(x, cb, M, cbm, level) -> float:
    """One timed oracle encode + decode (the metric's two passes); returns
    seconds.  M and cbm are unused (kept so the inputs match the GPU step)."""
    import oracle
    t0 = time.perf_counter()
    X = oracle.encode(x, cb, level)
    rc, y = oracle.decode(X, cb)
    dt = time.perf_counter() - t0
    assert rc == 0 and np.array_equal(y, x)
    return dt


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


CPU_BASELINE_SECONDS = 10.0


def cpu_baseline(workload: str, nblocks_sample: int | None):
    """The oracle on one host core, stepped (encode + decode) over the same
    inputs until at least CPU_BASELINE_SECONDS of oracle work are timed."""
    inputs = oracle_step_inputs(workload, nblocks_sample)
    nvals = inputs[0].size
    total, steps = 0.0, 0
    while total < CPU_BASELINE_SECONDS:
        total += oracle_step(*inputs)
        steps += 1
    return {"value": round(4 * nvals * steps / total / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "%d steps (encode + decode) over %d values of the %s workload (%s); "
                      "host %s, %d logical CPUs, oracle single-threaded" % (
                          steps, nvals, workload, "first %d blocks" % nblocks_sample if nblocks_sample else "all",
                          cpu_model(), os.cpu_count() or 0),
            "seconds": round(total, 3)}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return None
    from lossless_bf16_tensor_gb300 import synth
    if "adamw" in synth.WORKLOADS[args.workload]:
        return run_reference_timed(args, world, oracle_adamw_time,
                                   "fused AdamW step on compressed W, M and V: elements per second")
    if "gradient" in synth.WORKLOADS[args.workload]:
        return run_reference_momentum(args, world)
    inputs = oracle_step_inputs(args.workload, args.cpu_blocks)
    nvals = inputs[0].size
    for _ in range(args.warmup):
        oracle_step(*inputs)
    times = [oracle_step(*inputs) for _ in range(args.steps)]
    s = sum(times) / len(times)
    value = 4 * nvals / s / 1e9
    sample = "%d values of %s per step (%s)" % (nvals, args.workload,
                                               "first %d blocks" % args.cpu_blocks if args.cpu_blocks else "all")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32+f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_reference_timed(args, world, timer, metric):
    for _ in range(args.warmup):
        timer(args.workload, args.cpu_blocks)
    times, nvals = [], 0
    for _ in range(args.steps):
        dt, nvals = timer(args.workload, args.cpu_blocks)
        times.append(dt)
    s = sum(times) / len(times)
    value = nvals / s / 1e9
    sample = "first %d values of %s per step (%d blocks)" % (nvals, args.workload, args.cpu_blocks)
    return {"impl": "reference", "metric": metric, "value": round(value, 5), "unit": "Gelem/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u32+f32", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload},
            "cpu_baseline": {"value": round(value, 5), "unit": "Gelem/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 5), "unit": "Gelem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_reference_momentum(args, world):
    for _ in range(args.warmup):
        oracle_momentum_time(args.workload, args.cpu_blocks)
    times, nvals = [], 0
    for _ in range(args.steps):
        dt, nvals = oracle_momentum_time(args.workload, args.cpu_blocks)
        times.append(dt)
    s = sum(times) / len(times)
    value = nvals / s / 1e9
    sample = "first %d values of %s per step (%d blocks)" % (nvals, args.workload, args.cpu_blocks)
    return {"impl": "reference", "metric": "fused SGD-with-momentum step on compressed W and M: elements per second",
            "value": round(value, 5), "unit": "Gelem/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u32+f32", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload], "name": args.workload},
            "cpu_baseline": {"value": round(value, 5), "unit": "Gelem/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 5), "unit": "Gelem/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["lct", "reference"], default="lct")
    ap.add_argument("--workload", default="laplace_16m", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--cpu-blocks", type=int, default=0, help="oracle sample: first N blocks (0 = whole workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the five-configuration breakdown")
    args = ap.parse_args()
    if args.impl == "reference":
        # each oracle step is a bounded sample of the workload (32 blocks
        # unless given) so that --steps K --warmup W ends within minutes
        if not args.cpu_blocks:
            args.cpu_blocks = 32
        line = run_reference(args)
    elif args.gpus > 1 and int(os.environ.get("WORLD_SIZE", "1")) == 1:
        # not under torchrun: start one process per GPU here
        line = spawn_ranks(args.gpus, run_gpu, (args,)).get(0)
    else:
        line = run_gpu(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
