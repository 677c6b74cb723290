"""Benchmark: quantized Muon optimizer steps on one GB300 (replicas for N > 1).

One step = the whole hot path: the blockwise 8-bit momentum update over every
matrix, grouped Frobenius norms, batched Newton-Schulz (5 quintic
iterations) and the weight update, with the MuonBP schedule (block NS on
1 x 8 column tiles, full NS every 5th step).  Default workload: 4 layers of a
Llama-8B-shaped model (q/o 4096x4096, k/v 1024x4096, gate/up 14336x4096,
down 4096x14336), 872,415,232 parameters, synthetic seeded gradients.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  ``value`` = parameters processed per second (Mparams/s)
over K timed steps, inputs resident in HBM, timed with CUDA events and taken
as the max over ranks.  Every step reads its own pre-generated gradient batch
(one plan per batch; a step overwrites its gradients with the momentum and
then the update), so nothing but the optimizer runs in the timed region.
The inputs (1.75 GB of gradients per step) are larger than L2.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "qMuon update HBM GB/s + Newton-Schulz TFLOP/s; Mparams/s per optimizer step"
UPDATE_BYTES_PER_ELEM = 1 + 2 + 1 + 2 + 8.0 / 256   # q8 r/w, bf16 grad r/w, absmax r/w
MAX_BATCHES = 40   # pre-generated gradient batches (1.75 GB each at the default workload)
L2_BYTES = 129 * 2 ** 20          # GB300 L2
L2_FLUSH_BYTES = 512 * 2 ** 20    # a write that evicts it


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def load_traffic():
    """Per-launch (or per-call) DRAM bytes from the committed ncu summaries
    (``key = bytes`` lines in the profiles listed below)."""
    out = {}
    for name in ("dram_traffic_llama8b_x4_muonbp.md", "grasp_llama8b_x4.md", "dram_traffic_update_rowscale4.md"):
        try:
            with open(os.path.join(ROOT, "profiles", name)) as f:
                for line in f:
                    parts = line.split("=")
                    if len(parts) == 2 and parts[0].strip().endswith(("_per_launch", "_per_call")):
                        out[parts[0].strip()] = float(parts[1])
        except Exception:
            pass
    return out


def ns_flops_of(rows, cols, iters):
    m, n = min(rows, cols), max(rows, cols)
    return iters * 2.0 * (2.0 * n * m * m + float(m) ** 3)


def step_ns_flops(w, full):
    tr, tc = (1, 1) if full else w.tile
    tot = 0.0
    for m in w.matrices:
        tot += tr * tc * ns_flops_of(m.rows // tr, m.cols // tc, w.iters)
    return tot


def ns_executed_flops_of(rows, cols, iters):
    """FLOPs the tensor cores execute for one matrix: 256 x 256 output tiles
    (the symmetric products only those on or above the diagonal, SYRK) and
    K loops in steps of 64."""
    m, n = min(rows, cols), max(rows, cols)
    tm, tn = -(-m // 256), -(-n // 256)
    kpad = lambda k: -(-k // 64) * 64   # noqa: E731
    sym = tm * (tm + 1) // 2
    return iters * 2.0 * 256 * 256 * (sym * kpad(n) + sym * kpad(m) + tm * tn * kpad(m))


def step_ns_executed(w, full):
    tr, tc = (1, 1) if full else w.tile
    return sum(tr * tc * ns_executed_flops_of(m.rows // tr, m.cols // tc, w.iters) for m in w.matrices)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


E2E_MIN_STEPS = 60   # host-fed steps timed by the end-to-end leg of the MuonBP workload
# gradient batches in flight in that leg: step k's copies start once step
# k - E2E_DEPTH has finished with its buffers.  Three measured slower than two
# on hosts whose copy-engine transfers stall (a larger page-locked footprint)
E2E_DEPTH = 2


_HOST_MAPS = []   # keeps the huge-page mappings of pinned_host_bf16 alive


def pinned_host_bf16(n: int) -> torch.Tensor:
    """A page-locked host bf16 buffer of n elements for the end-to-end leg,
    backed by transparent huge pages where the host allows it (anonymous
    mapping advised MADV_HUGEPAGE, then registered with cudaHostRegister and
    mapped into the device's address space, so that the host-fed step reads
    it with the device's own loads).  Falls back to torch's page-locked
    allocation, which is mapped as well, if any step fails."""
    import mmap
    try:
        mm = mmap.mmap(-1, 2 * n, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
        mm.madvise(mmap.MADV_HUGEPAGE)
        arr = np.frombuffer(mm, dtype=np.uint16)
        arr[:] = 0   # touch: the pages exist before they are registered
        buf = torch.from_numpy(arr).view(torch.bfloat16)
        r = torch.cuda.cudart().cudaHostRegister(buf.data_ptr(), 2 * n, 2)   # cudaHostRegisterMapped
        status = int(r[0] if isinstance(r, tuple) else r)
        if status == 0 and buf.is_pinned():
            _HOST_MAPS.append(mm)
            return buf
    except Exception:
        pass
    return torch.empty(n, dtype=torch.bfloat16, pin_memory=True)


def audit_per_step(q, before, steps):
    """The library's path and dtype tallies added by the timed steps, per step
    (fields that moved only)."""
    after = q.qmuon_get_counters()
    return {k: (after[k] - before[k]) / steps for k in after if after[k] != before[k]}


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time (replicas: the job ends when the last one does)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(n_params: int, steps: int, world: int, ms_max: float) -> float:
    """Whole-job Mparams/s: every rank runs its own replica of the workload."""
    return world * n_params * steps / (ms_max / 1e3) / 1e6


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------
# the CPU oracle leg (cpu_baseline and --impl reference)
# --------------------------------------------------------------------------

CODEC_SLICE = 1 << 20   # elements per thread in one sample step of the oracle's codec


def _block_tiles(w):
    """(rows, cols, params of the workload with that matrix shape) per shape,
    and the tile shape each one's block-step Newton-Schulz runs on."""
    shapes = {}
    for m in w.matrices:
        shapes[(m.rows, m.cols)] = shapes.get((m.rows, m.cols), 0) + m.numel
    tr, tc = w.tile if w.P != 1 else (1, 1)
    return [((r, c), wt, (r // tr, c // tc)) for (r, c), wt in sorted(shapes.items(), key=lambda kv: kv[0][0] * kv[0][1])]


def _oracle_codec(n, beta, seed):
    """The oracle's momentum update on n elements from a zero state; returns
    its duration (the inputs are drawn first, untimed)."""
    import numpy as np
    from oracle import codec
    rng = np.random.default_rng(seed)
    q8 = np.zeros(n, np.int8)
    a = np.zeros((n + 255) // 256, np.float32)
    g = codec.bf16_bits_from_f32(rng.standard_normal(n).astype(np.float32))
    t0 = time.perf_counter()
    codec.momentum_update(q8, a, g, beta)
    return time.perf_counter() - t0


NS_SAMPLE_FLOPS = 4e11   # larger tiles are timed on a bounded one (m <= 1792, n <= 4096), scaled by FLOPs


def _sample_tile(th, tw, iters):
    if ns_flops_of(th, tw, iters) <= NS_SAMPLE_FLOPS:
        return th, tw
    m, n = min(min(th, tw), 1792), min(max(th, tw), 4096)
    return (m, n) if th <= tw else (n, m)


def _oracle_ns_tiles(w, seed):
    """fp64 Newton-Schulz of the oracle on one tile of every shape (or on a
    bounded tile of the same orientation, scaled by the FLOP count); returns
    per shape (seconds for the tile, flops actually run, seconds measured)."""
    import numpy as np
    from oracle import ns as ons
    rng = np.random.default_rng(seed)
    out = []
    for _, _, (th, tw) in _block_tiles(w):
        sh, sw = _sample_tile(th, tw, w.iters)
        M = rng.standard_normal((sh, sw))
        t0 = time.perf_counter()
        ons.newton_schulz(M, iters=w.iters)
        dt = time.perf_counter() - t0
        f_run = ns_flops_of(sh, sw, w.iters)
        out.append((dt * ns_flops_of(th, tw, w.iters) / f_run, f_run, dt))
    return out


_SINGLE_CORE = r"""
import sys, time, numpy as np
sys.path.insert(0, sys.argv[1])
from oracle import codec, ns
n, rows, cols, iters = (int(x) for x in sys.argv[2:6])
rng = np.random.default_rng(7)
q8 = np.zeros(n, np.int8); a = np.zeros((n + 255) // 256, np.float32)
g = codec.bf16_bits_from_f32(rng.standard_normal(n).astype(np.float32))
t0 = time.perf_counter(); codec.momentum_update(q8, a, g, 0.95); tc = time.perf_counter() - t0
M = rng.standard_normal((rows, cols))
t0 = time.perf_counter(); ns.newton_schulz(M, iters=iters); tn = time.perf_counter() - t0
print(tc, tn)
"""


def _per_param_seconds(w, codec_s_per_elem, tile_costs, fp64_flops_per_s):
    """Seconds per parameter of one optimizer step averaged over the
    workload's step schedule: the codec on every parameter, block-step
    Newton-Schulz from the measured tiles (weighted by the shapes' parameter
    counts), full-step Newton-Schulz from the measured fp64 rate."""
    blocks = _block_tiles(w)
    ns_block = sum(c[0] / (th * tw) * wt for c, (_, wt, (th, tw)) in zip(tile_costs, blocks)) / w.numel
    if w.P == 1:
        return codec_s_per_elem + ns_block
    ns_full = step_ns_flops(w, True) / fp64_flops_per_s / w.numel
    n_full = sum(1 for t in range(1, w.steps + 1) if w.P and t % w.P == 0)
    return codec_s_per_elem + (ns_block * (w.steps - n_full) + ns_full * n_full) / w.steps


def oracle_sample(w, steps=3, warmup=1):
    """Time the oracle as it stands on bounded sample steps of the workload.

    One sample step: the codec (numpy, fp32) on CODEC_SLICE elements in each
    of `cores` threads at once, then fp64 Newton-Schulz on one block-step tile
    of every matrix shape (numpy's BLAS on every core).  `warmup` untimed
    steps, then `steps` timed ones.  The workload rate is extrapolated from
    the per-parameter costs (``_per_param_seconds``): the codec's from the
    threads' wall time, the block steps' Newton-Schulz from the tiles, the
    full steps' from the tiles' fp64 FLOP rate.  A single-core figure comes
    from one more run in a subprocess with one BLAS thread.
    Returns a dict: value (all cores, Mparams/s), ms_per_step (measured
    sample step), steps, cores, sample, single_core (Mparams/s)."""
    from concurrent.futures import ThreadPoolExecutor
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    step_ms, codec_rates, tile_runs = [], [], []
    with ThreadPoolExecutor(max_workers=cores) as ex:
        for k in range(warmup + steps):
            t0 = time.perf_counter()
            durs = list(ex.map(lambda i: _oracle_codec(CODEC_SLICE, w.beta, 1000 * k + i), range(cores)))
            tiles = _oracle_ns_tiles(w, k)
            dt = time.perf_counter() - t0
            if k >= warmup:
                step_ms.append(dt * 1e3)
                codec_rates.append(max(durs) / (cores * CODEC_SLICE))
                tile_runs.append(tiles)
    codec_s = statistics.median(codec_rates)
    tile_costs = [(statistics.median(run[i][0] for run in tile_runs), tile_runs[0][i][1],
                   statistics.median(run[i][2] for run in tile_runs)) for i in range(len(tile_runs[0]))]
    fp64_rate = sum(c[1] for c in tile_costs) / sum(c[2] for c in tile_costs)
    value = 1.0 / _per_param_seconds(w, codec_s, tile_costs, fp64_rate) / 1e6
    # one core: the codec and the smallest tile's Newton-Schulz with one BLAS thread
    single = None
    try:
        blocks = _block_tiles(w)
        th, tw = _sample_tile(*blocks[0][2], w.iters)
        env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
        r = subprocess.run([sys.executable, "-c", _SINGLE_CORE, ROOT, str(CODEC_SLICE), str(th), str(tw),
                            str(w.iters)], capture_output=True, text=True, env=env, timeout=300)
        tc1, tn1 = (float(x) for x in r.stdout.split())
        rate1 = ns_flops_of(th, tw, w.iters) / tn1
        tiles1 = [(ns_flops_of(bt[0], bt[1], w.iters) / rate1,) for _, _, bt in blocks]
        single = 1.0 / _per_param_seconds(w, tc1 / CODEC_SLICE, tiles1, rate1) / 1e6
    except Exception:
        single = None
    tiles_desc = "; ".join(f"{th}x{tw}" for _, _, (th, tw) in _block_tiles(w))
    sample = (f"{steps} timed sample steps after {warmup} untimed, each: the numpy fp32 codec on "
              f"{CODEC_SLICE} elements in each of {cores} threads, then fp64 Newton-Schulz ({w.iters} iterations) "
              f"on one tile of each shape ({tiles_desc}; tiles above {NS_SAMPLE_FLOPS:.0e} FLOPs timed on a bounded tile and scaled by FLOPs); the workload rate is extrapolated from these "
              "per-parameter costs weighted by the shapes' parameter counts, full steps from the tiles' fp64 FLOP "
              "rate; single_core: the same with one thread and one BLAS thread")
    return {"value": value, "ms_per_step": statistics.mean(step_ms), "steps": steps, "cores": cores,
            "sample": sample, "single_core": single, "fp64_gflops": fp64_rate / 1e9,
            "codec_mparams_per_s_all_cores": 1.0 / codec_s / 1e6, "extrapolated": True}


# --------------------------------------------------------------------------
# the GPU leg
# --------------------------------------------------------------------------

GRASP_BYTES_PER_PARAM = 0.625 + 2 + 2 + 2 + 2 + 0.625   # state r/w, g, M_t w + 2 reads


def time_grasp(q, mats, grads, stream, reps, dev):
    """The 4-bit GRASP momentum step (qmuon_grasp_step) over the same matrices,
    one call for all of them, from a zero residual and a seeded factor."""
    descs, keep = [], []
    g = torch.Generator(device=dev)
    g.manual_seed(4242)
    for m, grad in zip(mats, grads):
        rows, cols = m.rows, m.cols
        nbr, nbc = (rows + 63) // 64, cols // 64
        t = dict(res=torch.full((rows, cols // 2), 0x88, dtype=torch.uint8, device=dev),
                 res_rmax=torch.zeros(nbc, rows, device=dev), res_cmax=torch.zeros(nbr, cols, device=dev),
                 p=torch.zeros(rows, 8, dtype=torch.int8, device=dev), p_rmax=torch.zeros(rows, device=dev),
                 p_cmax=torch.zeros(nbr, 8, device=dev),
                 r=torch.randint(-127, 128, (cols, 8), generator=g, device=dev, dtype=torch.int32).to(torch.int8),
                 r_rmax=torch.ones(cols, device=dev), r_cmax=torch.ones((cols + 63) // 64, 8, device=dev))
        keep.append(t)
        descs.append(q.grasp_matrix(rows, cols, t["res"], t["res_rmax"], t["res_cmax"], t["p"], t["p_rmax"],
                                    t["p_cmax"], t["r"], t["r_rmax"], t["r_cmax"], grad))
    ws = torch.empty(q.qmuon_grasp_workspace_size(descs), dtype=torch.uint8, device=dev)
    for _ in range(2):
        q.qmuon_grasp_step(descs, 0.95, ws, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        q.qmuon_grasp_step(descs, 0.95, ws, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    q.qmuon_sync_status(ws, stream)
    return e0.elapsed_time(e1) / reps


def run_gpu_carrier(args, world, rank, local, w):
    """Workload 5: per-matrix MXFP8 carrier update (E4M3 payload + E8M0 scales
    + inverse norm; the gradient is only read) followed by full Newton-Schulz
    on every matrix, fed by the carrier.  The orthogonalised update lands in
    the gradient buffer; no weight update is part of this workload."""
    import memory_reduced_muon_gb300 as q

    dev = torch.device("cuda", local)
    mats = w.matrices
    stream = torch.cuda.current_stream()
    states = [workloads.zero_state(m, w.q8_kind, device=dev) for m in mats]
    # the carrier update only reads the gradient, so one resident batch serves every step
    grads = [workloads.make_grad(w, i, 1, device=dev) for i in range(len(mats))]
    outs = [torch.empty(m.rows, m.cols, dtype=torch.bfloat16, device=dev) for m in mats]
    payload = [torch.empty(m.numel, dtype=torch.uint8, device=dev) for m in mats]
    scale = [torch.empty(m.rows * (m.cols // 32), dtype=torch.uint8, device=dev) for m in mats]
    inv = torch.zeros(len(mats), dtype=torch.float32, device=dev)
    probs = [q.ns_problem(o, m.rows, m.cols, inv_norm=inv.data_ptr() + 4 * i, input_kind=q.QMUON_NS_MXFP8,
                          payload=payload[i], scale_inv=scale[i]) for i, (o, m) in enumerate(zip(outs, mats))]
    ws_n = torch.empty(q.qmuon_ns_workspace_size(probs), dtype=torch.uint8, device=dev)

    # one launch over every matrix (one norm group per matrix)
    plan_c = q.qmuon_plan_create([(s[0], s[1], g, m.rows, m.cols) for s, g, m in zip(states, grads, mats)],
                                 w.q8_kind, "bf16")
    ws_c = torch.empty(q.qmuon_workspace_size(plan_c), dtype=torch.uint8, device=dev)

    def carrier_all():
        q.qmuon_update_mxfp8_carrier_multi(plan_c, w.beta, payload, scale, inv, ws_c, stream=stream)

    def step(t):
        carrier_all()
        q.qmuon_newton_schulz_batched(probs, w.iters, w.coeffs, ws_n, stream=stream)

    t = 0
    for _ in range(max(args.warmup, 1)):
        t += 1
        step(t)
    q.qmuon_sync_status(ws_n, stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(str(local))
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    tallies = q.qmuon_get_counters()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        t += 1
        step(t)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    audit = audit_per_step(q, tallies, args.steps)
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    q.qmuon_sync_status(ws_n, stream)
    # the carrier update alone and the Newton-Schulz alone
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    u0.record(stream)
    for _ in range(3):
        carrier_all()
    u1.record(stream)
    torch.cuda.synchronize()
    upd_ms = u0.elapsed_time(u1) / 3
    n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0.record(stream)
    for _ in range(3):
        q.qmuon_newton_schulz_batched(probs, w.iters, w.coeffs, ws_n, stream=stream)
    n1.record(stream)
    torch.cuda.synchronize()
    ns_ms = n0.elapsed_time(n1) / 3
    n_params = w.numel
    upd_bytes = (1 + 2 + 1 + 1 + 1.0 / 32 + 8.0 / 256) * n_params
    flop = step_ns_flops(w, True)
    return dict(value=world * n_params * args.steps / (ms / 1e3) / 1e6, ms=ms, clocks=clocks, audit=audit,
                per_step=[], upd_ms=upd_ms, upd_gbs=upd_bytes / (upd_ms / 1e3) / 1e9, upd_bytes=upd_bytes,
                ns_ms={"full": ns_ms}, ns_flop={"full": flop}, ns_exec={"full": step_ns_executed(w, True)},
                e2e_value=None, h2d=0, d2h=0, n_full=args.steps,
                launches=(1 + 1 + 3 * w.iters) * args.steps, n_params=n_params, w=w,
                l2=f"inputs larger than L2 ({sum(2 * m.numel for m in mats) / 1e9:.2f} GB of bf16 gradients and "
                   f"{sum(m.numel for m in mats) / 1e9:.2f} GB of codes read per step)")


def run_gpu_grouped(args, world, rank, local, w):
    """Workloads 2 and 3: the grouped momentum update
    (qmuon_update_multi_normalize_groups, deferred norms) over every matrix
    with the workload's norm groups (its segments, or one group per matrix),
    then, when the workload has Newton-Schulz, one batched call over its
    problems (its row slices, each scaled by its own group's inverse norm),
    in place in the gradient buffers.  These workloads update no weights."""
    import memory_reduced_muon_gb300 as q

    dev = torch.device("cuda", local)
    mats = w.matrices
    stream = torch.cuda.current_stream()
    states = [workloads.zero_state(m, w.q8_kind, device=dev) for m in mats]
    n_steps_total = max(args.warmup, 1) + args.steps
    n_batches = min(n_steps_total, MAX_BATCHES)
    batches = [[workloads.make_grad(w, i, b + 1, device=dev) for i in range(len(mats))] for b in range(n_batches)]
    segs = ([(sg.tensor_index, sg.start, sg.length, sg.group_id) for sg in w.segments]
            if w.segments is not None else None)
    n_groups = w.groups
    plans = [q.qmuon_plan_create([(st[0], st[1], g, m.rows, m.cols) for st, g, m in zip(states, grads, mats)],
                                 w.q8_kind, "bf16", segments=segs, n_groups=n_groups if segs else 0)
             for grads in batches]
    ws = torch.empty(q.qmuon_workspace_size(plans[0]), dtype=torch.uint8, device=dev)
    sums = torch.zeros(n_groups, dtype=torch.float32, device=dev)
    inv = torch.zeros(n_groups, dtype=torch.float32, device=dev)

    def group_of(t, row0):
        if segs is None:
            return t
        for ti, start, _, gid in segs:
            if ti == t and start == row0 * mats[t].cols:
                return gid
        raise ValueError("a Newton-Schulz slice that starts no norm segment")

    slices = w.ns_slices if w.ns_slices is not None else [(i, 0, m.rows) for i, m in enumerate(mats)]

    def problems(grads):
        out = []
        for t, row0, rows in slices:
            cols = mats[t].cols
            out.append(q.ns_problem(grads[t].data_ptr() + 2 * row0 * cols, rows, cols, ld=cols,
                                    inv_norm=inv.data_ptr() + 4 * group_of(t, row0)))
        return out

    probs = [problems(grads) for grads in batches] if w.ns else None
    ws_n = torch.empty(q.qmuon_ns_workspace_size(probs[0]), dtype=torch.uint8, device=dev) if w.ns else None

    def step(t):
        b = (t - 1) % n_batches
        q.qmuon_update_multi_normalize_groups(plans[b], w.beta, 2, sums, inv, ws, stream=stream)
        if w.ns:
            q.qmuon_newton_schulz_batched(probs[b], w.iters, w.coeffs, ws_n, stream=stream)

    t = 0
    for _ in range(max(args.warmup, 1)):
        t += 1
        step(t)
    q.qmuon_sync_status(ws, stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(str(local))
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    tallies = q.qmuon_get_counters()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        t += 1
        step(t)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    audit = audit_per_step(q, tallies, args.steps)
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    q.qmuon_sync_status(ws, stream)
    if w.ns:
        q.qmuon_sync_status(ws_n, stream)
    n_params = w.numel
    # the update alone and the Newton-Schulz alone, on the last batch
    reps = max(3, min(args.steps, 20))   # the per-kernel legs: a few calls back to back
    b_last = (t - 1) % n_batches
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    u0.record(stream)
    for _ in range(reps):
        q.qmuon_update_multi_normalize_groups(plans[b_last], w.beta, 2, sums, inv, ws, stream=stream)
    u1.record(stream)
    torch.cuda.synchronize()
    upd_ms = u0.elapsed_time(u1) / reps
    upd_bytes = UPDATE_BYTES_PER_ELEM * n_params
    ns_ms, ns_flop, ns_exec = {}, {}, {}
    if w.ns:
        n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n0.record(stream)
        for _ in range(3):
            q.qmuon_newton_schulz_batched(probs[b_last], w.iters, w.coeffs, ws_n, stream=stream)
        n1.record(stream)
        torch.cuda.synchronize()
        q.qmuon_sync_status(ws_n, stream)
        ns_ms["full"] = n0.elapsed_time(n1) / 3
        ns_flop["full"] = sum(ns_flops_of(rows, mats[ti].cols, w.iters) for ti, _, rows in slices)
        ns_exec["full"] = sum(ns_executed_flops_of(rows, mats[ti].cols, w.iters) for ti, _, rows in slices)
    # end to end: each step's gradients copied in from page-locked host memory
    # (two batches alternate), the step, and its group sums copied back
    h2d = sum(g.numel() * g.element_size() for g in batches[0])
    host = []
    for b in range(2):
        buf = torch.empty(sum(g.numel() for g in batches[b % n_batches]), dtype=torch.bfloat16, pin_memory=True)
        views, o = [], 0
        for g in batches[b % n_batches]:
            v = buf[o:o + g.numel()].view(g.shape)
            v.copy_(g.cpu())
            views.append(v)
            o += g.numel()
        host.append(views)
    sums_host = torch.zeros(n_groups).pin_memory()
    e2e_steps = max(2, args.steps)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for k in range(e2e_steps):
        t += 1
        b = (t - 1) % n_batches
        for dst, src in zip(batches[b], host[k % 2]):
            dst.copy_(src, non_blocking=True)
        step(t)
        sums_host.copy_(sums, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    q.qmuon_sync_status(ws, stream)
    launches = (1 + (3 * w.iters + (1 if w.iters == 1 else 0) if w.ns else 0)) * args.steps
    return dict(value=job_throughput(n_params, args.steps, world, ms), ms=ms, clocks=clocks, audit=audit, per_step=[],
                upd_ms=upd_ms, upd_gbs=upd_bytes / (upd_ms / 1e3) / 1e9, upd_bytes=upd_bytes, ns_ms=ns_ms,
                ns_flop=ns_flop, ns_exec=ns_exec, e2e_value=world * n_params * e2e_steps / e2e_s / 1e6, e2e_steps=e2e_steps, h2d=h2d,
                d2h=4 * n_groups, n_full=args.steps if w.ns else 0, launches=launches, n_params=n_params, w=w,
                l2=f"inputs larger than L2 ({h2d / 1e9:.2f} GB of bf16 gradients per step)")


def run_gpu(args, world, rank, local):
    import memory_reduced_muon_gb300 as q

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workloads.get(args.workload)
    if args.row_scale > 1:
        w.matrices = [workloads.Matrix(m.name, max(8, m.rows // args.row_scale), m.cols) for m in w.matrices]
    if args.q8:
        w.q8_kind = args.q8
    if w.carrier:
        return run_gpu_carrier(args, world, rank, local, w)
    if w.segments is not None or not w.ns:
        return run_gpu_grouped(args, world, rank, local, w)
    mats = w.matrices
    n_params = w.numel
    stream = torch.cuda.current_stream()

    states = [workloads.zero_state(m, w.q8_kind, device=dev) for m in mats]
    weights = [workloads.make_weight(w, i, device=dev) for i in range(len(mats))]
    # every step gets its own pre-generated gradient batch, resident in HBM
    # before timing starts (a step overwrites its gradients with m and then U);
    # past MAX_BATCHES steps the batches are reused in turn
    n_steps_total = max(args.warmup, 1) + 1 + args.steps
    n_batches = min(n_steps_total, MAX_BATCHES)
    batches = [[workloads.make_grad(w, i, b + 1, device=dev) for i in range(len(mats))] for b in range(n_batches)]
    plans = [q.qmuon_plan_create([(s[0], s[1], g, m.rows, m.cols) for s, g, m in zip(states, grads, mats)],
                                 w.q8_kind, "bf16", tile=w.tile) for grads in batches]
    info = q.qmuon_plan_info(plans[0])
    # pinned host copies of two gradient batches for the end-to-end leg, taken
    # before any step overwrites them
    host_pool = []
    for b in range(E2E_DEPTH):   # one page-locked buffer per batch, a view per matrix
        src = batches[b % n_batches]
        buf = pinned_host_bf16(sum(g.numel() for g in src))
        views, o = [], 0
        for g in src:
            v = buf[o:o + g.numel()].view(g.shape)
            v.copy_(g.cpu())
            views.append(v)
            o += g.numel()
        host_pool.append(views)
    ws = torch.empty(q.qmuon_workspace_size(plans[0], q.QMUON_WS_STEP), dtype=torch.uint8, device=dev)
    for p in plans:   # Newton-Schulz tables of both step kinds, built before any timing
        q.qmuon_step_prepare(p, weights, ws)
    sums = torch.zeros(max(info["n_full_groups"], info["n_block_groups"]), dtype=torch.float32, device=dev)
    grads = batches[0]

    def step(t):
        q.qmuon_step(plans[(t - 1) % n_batches], t, w.P, w.beta, w.eta_full, w.eta_block, weights, w.coeffs,
                     w.iters, sums, ws, stream=stream)

    t = 0
    for _ in range(max(args.warmup, 1)):
        t += 1
        step(t)
    if w.P > 1 and not any((t0 % w.P) == 0 for t0 in range(1, t + 1)):
        t += 1
        step(w.P)   # a full step before timing as well (t only counts the batch used)
    q.qmuon_sync_status(ws, stream)
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps ----
    t_first = t + 1
    n_full = sum(1 for k in range(t_first, t_first + args.steps) if w.P and k % w.P == 0)
    try:
        bus = torch.cuda.get_device_properties(local).pci_bus_id
        sel = f"{torch.cuda.get_device_properties(local).pci_domain_id:08X}:{bus:02X}:{torch.cuda.get_device_properties(local).pci_device_id:02X}.0"
    except Exception:
        sel = str(local)
    # a step whose inputs fit in L2 is timed alone, with L2 flushed before it
    # (a write larger than L2, outside the step's events)
    step_bytes = sum(m.numel * (2 + 1 + 4) for m in mats)   # bf16 gradient, q8 state, fp32 weights
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev) if step_bytes < 2 * L2_BYTES else None
    l2_note = (f"L2 flushed before every step ({L2_FLUSH_BYTES >> 20} MB write outside the step's CUDA events; "
               f"the step's inputs are {step_bytes / 1e6:.1f} MB)" if flush is not None else
               f"inputs larger than L2 ({sum(2 * m.numel for m in mats) / 1e9:.2f} GB of bf16 gradients per step)")
    sampler = ClockSampler(sel)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    tallies = q.qmuon_get_counters()
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    kinds = []
    for k in range(args.steps):
        t += 1
        if flush is not None:
            flush.zero_()
        ev0[k].record(stream)
        step(t)
        ev1[k].record(stream)
        kinds.append("full" if (w.P and t % w.P == 0) else "block")
    torch.cuda.synchronize()
    per_step = [{"kind": kinds[k], "step_ms": ev0[k].elapsed_time(ev1[k])} for k in range(args.steps)]
    barrier(world)
    clocks = sampler.stop()
    audit = audit_per_step(q, tallies, args.steps)
    # back-to-back steps: first event to last; flushed steps: the sum of the steps
    ms = (ev0[0].elapsed_time(ev1[-1]) if flush is None else sum(p["step_ms"] for p in per_step))
    q.qmuon_sync_status(ws, stream)
    ms_max = max_over_ranks(ms, world)
    value = job_throughput(n_params, args.steps, world, ms_max)

    # ---- per-kernel timing: the update alone and the Newton-Schulz engine alone ----
    plan_u = q.qmuon_plan_create([(s[0], s[1], g, m.rows, m.cols) for s, g, m in zip(states, grads, mats)],
                                 w.q8_kind, "bf16")
    ws_u = torch.empty(q.qmuon_workspace_size(plan_u), dtype=torch.uint8, device=dev)
    inv_u = torch.zeros(len(mats), dtype=torch.float32, device=dev)
    reps = max(3, min(args.steps, 20))   # the per-kernel legs: a few calls back to back
    for _ in range(2):
        q.qmuon_update_multi_normalize_groups(plan_u, w.beta, 2, None, inv_u, ws_u, stream=stream)
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    u0.record(stream)
    for _ in range(reps):
        q.qmuon_update_multi_normalize_groups(plan_u, w.beta, 2, None, inv_u, ws_u, stream=stream)
    u1.record(stream)
    torch.cuda.synchronize()
    upd_ms = u0.elapsed_time(u1) / reps
    upd_bytes = UPDATE_BYTES_PER_ELEM * n_params
    upd_gbs = upd_bytes / (upd_ms / 1e3) / 1e9
    # the same update with stochastic requantisation (Philox4x32-10 per element)
    q.qmuon_update_multi_normalize_groups_sr(plan_u, w.beta, 2, 1234, 1, None, inv_u, ws_u, stream=stream)
    torch.cuda.synchronize()
    u0.record(stream)
    for k in range(reps):
        q.qmuon_update_multi_normalize_groups_sr(plan_u, w.beta, 2, 1234, 2 + k, None, inv_u, ws_u, stream=stream)
    u1.record(stream)
    torch.cuda.synchronize()
    upd_sr_ms = u0.elapsed_time(u1) / reps
    grasp_ms = time_grasp(q, mats, grads, stream, reps, dev)

    def ns_problems(full):
        tr, tc = (1, 1) if full else w.tile
        probs = []
        k = 0
        for m, g in zip(mats, grads):
            th, tw = m.rows // tr, m.cols // tc
            for i in range(tr):
                for j in range(tc):
                    off = (i * th * m.cols + j * tw) * 2
                    probs.append(q.ns_problem(g.data_ptr() + off, th, tw, ld=m.cols,
                                              inv_norm=inv_u.data_ptr() + 4 * (k % len(mats))))
                    k += 1
        return probs

    ns_ms, ns_flop, ns_exec = {}, {}, {}
    for full in ([False, True] if w.P != 1 else [True]):
        probs = ns_problems(full)
        ws_n = torch.empty(q.qmuon_ns_workspace_size(probs), dtype=torch.uint8, device=dev)
        q.qmuon_newton_schulz_batched(probs, w.iters, w.coeffs, ws_n, stream=stream)
        torch.cuda.synchronize()
        n0, n1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        nrep = 3
        n0.record(stream)
        for _ in range(nrep):
            q.qmuon_newton_schulz_batched(probs, w.iters, w.coeffs, ws_n, stream=stream)
        n1.record(stream)
        torch.cuda.synchronize()
        q.qmuon_sync_status(ws_n, stream)
        key = "full" if full else "block"
        ns_ms[key] = n0.elapsed_time(n1) / nrep
        ns_flop[key] = step_ns_flops(w, full)
        ns_exec[key] = step_ns_executed(w, full)
        del ws_n

    # e2e through the host-fed entry: every step copies its gradients in from
    # page-locked host memory and reads its group sums (the step's metric)
    # back to host memory.  E2E_DEPTH plans over the same state and weights
    # take turns, so a step's copies (on a copy stream) overlap the kernels of
    # the steps before it; the clock stops once the last read-back has landed.
    torch.cuda.synchronize()
    # at least 60 steps (about a second): a periodic host-to-device stall of
    # the host (copy-engine transfers at 12-19 GB/s for ~180 ms every ~510 ms,
    # seen on some hosts and not on others) then weighs in proportion instead
    # of taking a third of a 20-step leg
    e2e_steps = max(E2E_MIN_STEPS, args.steps)
    h2d = sum(g.numel() * g.element_size() for g in grads)
    ngr = max(info["n_block_groups"], info["n_full_groups"])
    copy_stream = torch.cuda.Stream(device=dev)
    sums_host = [torch.zeros(ngr).pin_memory() for _ in range(e2e_steps)]
    d2h = 0
    # untimed warm-up of the same leg: the first host-fed steps of a process
    # run slower (about 30 ms instead of 18 in a probe of ten and ten)
    for k in range(max(10, args.warmup)):
        t += 1
        q.qmuon_step_from_host(plans[(k % E2E_DEPTH) % n_batches], t, w.P, w.beta, w.eta_full, w.eta_block, weights,
                               w.coeffs, w.iters, host_pool[k % E2E_DEPTH], sums_host[0], sums, ws, stream=stream,
                               copy_stream=copy_stream)
    torch.cuda.synchronize()
    # the host runs at most E2E_DEPTH steps ahead of the GPU, as a training
    # loop that prefetches its batches would
    done = [torch.cuda.Event() for _ in range(e2e_steps)]
    barrier(world)
    t0 = time.perf_counter()
    for k in range(e2e_steps):
        t += 1
        b = k % E2E_DEPTH
        if k >= E2E_DEPTH:
            done[k - E2E_DEPTH].synchronize()
        q.qmuon_step_from_host(plans[b % n_batches], t, w.P, w.beta, w.eta_full, w.eta_block, weights, w.coeffs,
                               w.iters, host_pool[b], sums_host[k], sums, ws, stream=stream, copy_stream=copy_stream)
        done[k].record(stream)
        full_k = w.P != 0 and t % w.P == 0
        d2h += 4 * (info["n_full_groups"] if full_k else info["n_block_groups"])
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    q.qmuon_sync_status(ws, stream)
    if not all(bool(torch.isfinite(x).all()) for x in sums_host):
        raise RuntimeError("end-to-end leg: non-finite group sums read back")
    e2e_s = max_over_ranks(e2e_s, world)
    e2e_value = world * n_params * e2e_steps / e2e_s / 1e6
    d2h //= e2e_steps

    # launches of our kernels per step: 1 update + 3 per Newton-Schulz iteration
    launches_per_step = 1 + 3 * w.iters + (1 if w.iters == 1 else 0)
    return dict(value=value, ms=ms_max, clocks=clocks, audit=audit, per_step=per_step, upd_ms=upd_ms, upd_gbs=upd_gbs,
                upd_bytes=upd_bytes,
                upd_sr_ms=upd_sr_ms, grasp_ms=grasp_ms,
                ns_ms=ns_ms, ns_flop=ns_flop, ns_exec=ns_exec, e2e_value=e2e_value, e2e_steps=e2e_steps, h2d=h2d, d2h=d2h, n_full=n_full,
                l2=l2_note,
                launches=launches_per_step * args.steps, n_params=n_params, w=w)


def measure_gemm_peaks(n=8192, seconds=2.0):
    """Dense library GEMM rates on this GPU for context: torch._scaled_mm with
    E4M3 operands (per-tensor scales, bf16 out) and torch.mm in bf16, each run
    back to back for about `seconds` and timed with CUDA events."""
    dev = torch.device("cuda", 0)
    a = torch.randn(n, n, device=dev)
    b = torch.randn(n, n, device=dev)
    out = {"n": n}

    def rate(fn):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        reps = max(3, int(seconds * 1e3 / max(e0.elapsed_time(e1), 1e-3)))
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return 2.0 * n ** 3 / (e0.elapsed_time(e1) / reps / 1e3) / 1e12

    a16, b16 = a.to(torch.bfloat16), b.to(torch.bfloat16)
    out["bf16_tflops"] = rate(lambda: torch.mm(a16, b16))
    try:
        a8 = a.to(torch.float8_e4m3fn)
        b8 = b.to(torch.float8_e4m3fn).t().contiguous().t()   # column-major second operand
        one = torch.ones((), device=dev)
        out["fp8_e4m3_tflops"] = rate(lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one,
                                                               out_dtype=torch.bfloat16))
    except Exception as e:   # an FP8 GEMM this torch build cannot run here
        out["fp8_e4m3_tflops"] = None
        out["fp8_error"] = str(e).splitlines()[0][:200]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=4)
    ap.add_argument("--row-scale", type=int, default=1,
                    help="divide every matrix's row count, keeping its columns and tiles (profiling captures only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--q8", choices=["int8", "uint8"], default=None,
                    help="code kind of the 8-bit state (default: the workload's)")
    ap.add_argument("--measure-peaks", action="store_true",
                    help="time cuBLASLt FP8 (E4M3) and bf16 GEMMs at 8192^3 and print one JSON line, nothing else")
    args = ap.parse_args()
    if args.measure_peaks:
        print(json.dumps(measure_gemm_peaks()))
        return
    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    w = workloads.get(args.workload)
    wl_name = {4: "llama8b_x4_muonbp", 1: "single_512", 2: "decoder2048_x24_update", 3: "qkv_mlp_grouped",
               5: "llama8b_x4_mxfp8"}[args.workload]
    config = {"workload": wl_name, "description": w.name, "params": w.numel, "matrices": len(w.matrices),
              "P": w.P, "tile": list(w.tile), "ns_iters": w.iters, "beta": w.beta,
              "q8": args.q8 or w.q8_kind, "parallelism": f"replicas x{world}"}
    if w.carrier:
        config["ns_input"] = ("bf16-expanded: each MXFP8 carrier is expanded exactly to bf16 in one launch, and the "
                              "products run on bf16 tensor cores (no block-scaled FP8 MMA)")
    if args.row_scale > 1:
        config["row_scale"] = f"rows / {args.row_scale} (profiling only, not a reported number)"
        config["params"] = sum(max(8, m.rows // args.row_scale) * m.cols for m in w.matrices)

    if args.impl == "reference":
        if rank != 0:
            return
        o = oracle_sample(w, steps=args.steps, warmup=args.warmup)
        v = o["value"]
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "Mparams/s", "n_gpus": args.gpus,
                "steps": o["steps"], "warmup": args.warmup, "ms_per_step": o["ms_per_step"],
                "step": "one bounded sample step of the oracle (see cpu_baseline.sample); value is the workload "
                        "rate extrapolated from the sample's per-parameter costs",
                "extrapolated": True, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32 codec / f64 NS", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": v, "unit": "Mparams/s", "cores": o["cores"], "kind": "oracle",
                                 "sample": o["sample"], "single_core": o["single_core"],
                                 "codec_mparams_per_s_all_cores": o["codec_mparams_per_s_all_cores"],
                                 "fp64_gflops": o["fp64_gflops"]},
                "e2e": {"value": v, "unit": "Mparams/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    r = run_gpu(args, world, rank, local)
    if rank != 0:
        return
    config["l2"] = r["l2"]
    peaks, peak_src = load_peaks()
    traffic = load_traffic()
    w = r["w"]
    # dominant kernel family: the Newton-Schulz GEMMs (block steps dominate a P=5 schedule)
    key = "block" if "block" in r["ns_ms"] else "full"
    ns_tflops = {k: r["ns_flop"][k] / (r["ns_ms"][k] / 1e3) / 1e12 for k in r["ns_ms"]}
    ns_exec_tflops = {k: r["ns_exec"][k] / (r["ns_ms"][k] / 1e3) / 1e12 for k in r["ns_ms"]}
    # the Newton-Schulz call is timed alone (a few calls back to back): the burst peak
    peak_t = float(peaks.get("bf16_tflops", peaks.get("bf16_tflops_sustained")))
    upd_roof = {"bound": "hbm", "kernel": "update_kernel (one launch over every matrix)",
                "achieved": r["upd_gbs"], "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                "frac": r["upd_gbs"] / float(peaks["hbm_gbs"]), "frac_of_8000": r["upd_gbs"] / 8000.0,
                "peak_source": f"hbm_gbs of {peak_src}",
                "bytes_per_launch": r["upd_bytes"], "ms_per_launch": r["upd_ms"],
                "traffic": traffic.get("update_bytes_per_launch") if args.row_scale == 1 and args.workload == 4 else None}
    if r["ns_ms"]:
        roof = {"bound": "tensor", "kernel": f"ns_gemm ({key} step, {3 * w.iters} launches per call)",
                "achieved": ns_tflops[key], "peak": peak_t, "unit": "TFLOP/s", "frac": ns_tflops[key] / peak_t,
                "peak_source": f"bf16_tflops (burst) of {peak_src}: the call is timed alone",
                "flops_basis": "algorithmic 2(2nm^2+m^3) per matrix and iteration",
                "achieved_executed": ns_exec_tflops[key], "frac_executed": ns_exec_tflops[key] / peak_t,
                "executed_flops_per_call": r["ns_exec"][key],
                "traffic": traffic.get(f"ns_{key}_bytes_per_call")
                if args.row_scale == 1 and args.workload == 4 else None,
                "flops_per_call": r["ns_flop"][key], "ms_per_call": r["ns_ms"][key]}
    else:   # an update-only workload: the update kernel is the step
        roof = upd_roof
    line = {"metric": METRIC, "value": r["value"], "unit": "Mparams/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": r["ms"] / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 (NS operands, fp32 accumulate); int8 state, fp32 codec",
            "data": "synthetic (seeded gradients, zero initial state, N(0,0.02^2) weights)", "config": config,
            "full_steps_timed": r["n_full"], "per_step": r["per_step"],
            "update_gbs": r["upd_gbs"], "ns_tflops": ns_tflops,
            "grasp_step": ({"ms_per_call": r["grasp_ms"], "mparams_per_s": r["n_params"] / (r["grasp_ms"] / 1e3) / 1e6,
                            "bytes_per_param": GRASP_BYTES_PER_PARAM,
                            "gbs": GRASP_BYTES_PER_PARAM * r["n_params"] / (r["grasp_ms"] / 1e3) / 1e9,
                            "frac": GRASP_BYTES_PER_PARAM * r["n_params"] / (r["grasp_ms"] / 1e3) / 1e9
                            / float(peaks["hbm_gbs"]),
                            "traffic": traffic.get("grasp_bytes_per_call")
                            if args.row_scale == 1 and args.workload == 4 else None} if r.get("grasp_ms") else None),
            "update_stochastic_rounding": ({"gbs": r["upd_bytes"] / (r["upd_sr_ms"] / 1e3) / 1e9,
                                            "ms_per_launch": r["upd_sr_ms"],
                                            "frac": r["upd_bytes"] / (r["upd_sr_ms"] / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
                                            "traffic": traffic.get("update_sr_bytes_per_launch")
                                            if args.row_scale == 1 and args.workload == 4 else None}
                                           if r.get("upd_sr_ms") else None),
            "roofline": roof, "roofline_update": upd_roof, "clocks": r["clocks"],
            "audit_per_step": r.get("audit"),
            "e2e": ({"value": r["e2e_value"], "unit": "Mparams/s", "h2d_bytes_per_step": r["h2d"],
                     "d2h_bytes_per_step": r["d2h"], "steps": r.get("e2e_steps", args.steps)}
                    if r["e2e_value"] is not None else None),
            "gpu_launches": r["launches"]}
    if not args.no_cpu_baseline:
        t0 = time.perf_counter()
        o = oracle_sample(w, steps=3, warmup=1)
        line["cpu_baseline"] = {"value": o["value"], "unit": "Mparams/s", "cores": o["cores"], "kind": "oracle",
                                "sample": o["sample"], "single_core": o["single_core"],
                                "codec_mparams_per_s_all_cores": o["codec_mparams_per_s_all_cores"],
                                "fp64_gflops": o["fp64_gflops"], "extrapolated": True,
                                "seconds": time.perf_counter() - t0}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
