"""Benchmark of the codebook-4bit MoE verify layer on GB300.

One step = the whole hot path over one batch: the routed-expert layer at
batch 5 with top-8 of 256 experts (H=4096, F=2048; activation quantization,
gate_up + SwiGLU + requantization, down + weighted combine) plus the
129280 x 4096 output-head matvec at n = 5.  Weights are resident in HBM;
every step takes the next of 16 seeded routing tables and inputs.  The
metric is weight GB/s: the distinct experts' bytes plus the head's bytes,
read once per step, over the device time of the step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Prints one JSON line (rank 0).  For N > 1 (torchrun) every rank runs an
independent replica; the value is the bytes of all ranks over the slowest
rank's time.  `--impl reference` times the CPU oracle on a bounded sample of
the same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from verify_matvec_gb300 import synth  # noqa: E402

E, H, F = 256, 4096, 2048
N_TOK, TOPK = 5, 8
HEAD_M, HEAD_K, HEAD_N = 129280, 4096, 5
N_SETS = 16
QK, BB = 32, 18
EXPERT_BYTES = (2 * F * (H // QK) + H * (F // QK)) * BB        # 14,155,776
GATE_UP_BYTES = 2 * F * (H // QK) * BB                          # 9,437,184
DOWN_BYTES = H * (F // QK) * BB                                 # 4,718,592
HEAD_BYTES = HEAD_M * (HEAD_K // QK) * BB                       # 297,861,120
METRIC = "4-bit MoE matvec weight GB/s vs GB300 HBM peak; us/layer at batch 1 and 5"
WORKLOAD = ("MoE verify layer: 5 tokens x top-8 of 256 codebook-4bit experts (gate_up 4096x4096, "
            "down 4096 rows x 2048) with fused SwiGLU and weighted combine, plus the 129280x4096 "
            "output head at n=5")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, vendor figure

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch from
# one ncu capture of each kernel (summaries in profiles/), valid only for the
# kernel sources they were taken on (digest below); otherwise reported as null.
PROFILED = {
    "source_digest": "86060322c018b6db",
    "k_matvec<5> (head)": 297_930_496 + 5_312_256,          # one launch, 129280 x 4096, n=5
    # one layer call (k_quantize_chunked + k_moe + k_moe_combine) with 28 distinct experts
    "moe call per expert": (89_600 + 396_644_096 + 3_252_736 + 673_536) / 28,
}


# The translation unit that holds the profiled kernels (the layer kernel, its
# quantization and combine, the dense matvec); the digest covers it and every
# header, not the other translation units (the tensor-core path, the sinkhorn
# kernel, the C-ABI layer), whose changes leave those kernels as they were.
PROFILED_TU = "cbq_kernels.cu"


def source_digest(csrc=None):
    """Digest of the CUDA sources the profiled kernels are compiled from (code
    only: comments and whitespace runs are dropped), to match profiler
    captures."""
    import hashlib
    import re
    token = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"|\s+', re.S)

    def code(text):
        text = token.sub(lambda m: m.group(0) if m.group(0).startswith('"') else
                         (" " if m.group(0)[0].isspace() else ""), text)
        return re.sub(r"\s+", " ", text).strip()

    d = csrc or os.path.join(ROOT, "verify_matvec_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        if f == PROFILED_TU or f.endswith((".cuh", ".h")):
            h.update(f.encode())
            with open(os.path.join(d, f), encoding="utf-8") as fh:
                h.update(code(fh.read()).encode())
    return h.hexdigest()[:16]


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--profile", action="store_true",
                    help="time the main loop only (no e2e, per-layer or oracle legs); for profiler runs")
    ap.add_argument("--case", default="step", choices=["step", "b1", "b5", "dense1", "convert", "mmq16", "hc"],
                    help="profile mode only: the whole step, the MoE layer alone at batch 1 (top-4) "
                         "or batch 5 (top-8), the 4096x4096 dense projection at n=1 (cbq_matvec over "
                         "16 weight copies, more than L2), the weight converter on 16384x4096 fp32 "
                         "(two inputs, alternating), or the tensor-core path on 16384x4096 at n=16 "
                         "(cbq_matmat over 8 weight copies, more than L2), or the sinkhorn normalisation of "
                         "2^21 hyper-connection matrices, 20 rounds (two inputs alternating)")
    ap.add_argument("--shared", action="store_true",
                    help="profile mode, b1/b5 cases: give the layer a shared expert (one more expert of the "
                         "routed shape that every token passes through)")
    ap.add_argument("--experts", type=int, default=E,
                    help="experts in the layer (default 256); smaller layers keep profiler captures small")
    return ap.parse_args()


def l2_cache_bytes(torch, dev):
    """The device's L2 size in bytes (the runtime's l2CacheSize device
    property, i.e. cudaDevAttrL2CacheSize)."""
    return int(torch.cuda.get_device_properties(dev).L2_cache_size)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        v = d.get("hbm_gbs")
        if v:
            return float(v), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def routing_sets(seed_base=synth.S_IDS + 100, n_exp=E):
    sets = []
    for i in range(N_SETS):
        ids, wts = synth.router(N_TOK, TOPK, n_exp, stream=seed_base + i)
        h = synth.activations(N_TOK, H, stream=synth.S_H + 100 + i)
        x = synth.activations(HEAD_N, HEAD_K, stream=synth.S_HEAD_X + 100 + i)
        sets.append((ids, wts, h, x))
    return sets


# -------------------------------------------------------------- oracle -----

def oracle_sample(sets, n_steps, threads=1):
    """Time the CPU oracle on a bounded sample of the workload: token 0 of the
    MoE layer (its 8 slots) plus 1/16 of the head rows at n = 5, per step.
    With threads > 1 the same oracle calls are split over a thread pool (the
    slots one per task, the head rows in one chunk per thread; the C oracle
    runs without the interpreter lock), as a row-split baseline on all cores."""
    from concurrent.futures import ThreadPoolExecutor

    from oracle import oracle as O
    ids, wts, h, x = sets[0]
    used = synth.distinct_experts(ids[:1], E)
    gu = np.zeros((E, 2 * F, H // QK, BB), dtype=np.uint8)
    dn = np.zeros((E, H, F // QK, BB), dtype=np.uint8)
    for e in used:
        gu[e] = synth.weight_blocks(2 * F, H, stream=synth.S_GATE_UP * 1000 + int(e))
        dn[e] = synth.weight_blocks(H, F, stream=synth.S_DOWN * 1000 + int(e))
    rows = HEAD_M // 16
    head = synth.weight_blocks(rows, HEAD_K, stream=synth.S_HEAD)
    step_bytes = len(used) * EXPERT_BYTES + rows * (HEAD_K // QK) * BB
    times = []
    if threads <= 1:
        for _ in range(n_steps):
            t0 = time.perf_counter()
            O.moe(gu, dn, E, H, F, h[:1], ids[:1], wts[:1], swiglu=1)
            O.matvec(head, rows, HEAD_K, x)
            times.append(time.perf_counter() - t0)
        kind = "single-threaded oracle"
    else:
        bounds = np.linspace(0, rows, threads + 1).astype(int)
        tasks = [(lambda j=j: O.moe(gu, dn, E, H, F, h[:1], ids[:1, j:j + 1], wts[:1, j:j + 1], swiglu=1))
                 for j in range(ids.shape[1])]
        tasks += [(lambda a=a, b=b: O.matvec(head[a:b], b - a, HEAD_K, x))
                  for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
        with ThreadPoolExecutor(max_workers=threads) as pool:
            for _ in range(n_steps):
                t0 = time.perf_counter()
                list(pool.map(lambda f: f(), tasks))
                times.append(time.perf_counter() - t0)
        kind = f"oracle split over {threads} threads (slots, head row chunks)"
    sample = (f"per step: token 0 of the batch-5 MoE layer ({len(used)} experts, "
              f"{len(used) * EXPERT_BYTES} B) + {rows} of {HEAD_M} head rows at n=5; {kind}")
    return step_bytes, times, sample


def oracle_next_rows():
    """The single-threaded CPU oracle timed beside the next rows of the path,
    each on a bounded sample (a second or two of CPU work): the weight
    converter on 256 x 4096 fp32 weights (bytes in + out per second), the
    quantized matmat at n = 16 on 512 rows of a 4096-wide matrix (weight bytes
    per second), and the sinkhorn normalisation of 2^14 4x4 matrices at 20
    rounds (matrices per second)."""
    from oracle import oracle as O
    out = {}
    Mw, Kw = 256, 4096
    w = (np.random.default_rng(5).standard_normal((Mw, Kw)) * 0.02).astype(np.float32)
    t0 = time.perf_counter()
    O.quantize_weights(w, Mw, Kw)
    dt = time.perf_counter() - t0
    nbytes = Mw * Kw * 4 + Mw * (Kw // QK) * BB
    out["weight_converter"] = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                               "sample": f"{Mw} x {Kw} fp32 weights"}
    Mm, n = 512, 16
    Wm = synth.weight_blocks(Mm, Kw, stream=synth.S_W * 1000 + 3)
    qx, dx = O.quantize_act(synth.activations(n, Kw, stream=synth.S_X))
    t0 = time.perf_counter()
    O.matvec_q(Wm, Mm, Kw, qx, dx)
    dt = time.perf_counter() - t0
    out["tensor_core_path"] = {"value": Mm * (Kw // QK) * BB / dt / 1e9, "unit": "GB/s", "cores": 1,
                               "kind": "oracle", "sample": f"{Mm} rows x {Kw} at n={n}"}
    nh = 1 << 14
    c = synth.hc_logits(nh, stream=synth.S_HC * 1000 + 7)
    t0 = time.perf_counter()
    O.hc_sinkhorn(c, 20)
    dt = time.perf_counter() - t0
    out["hc_sinkhorn"] = {"value": nh / dt, "unit": "matrices/s", "cores": 1, "kind": "oracle",
                          "sample": f"{nh} 4x4 matrices, 20 rounds"}
    return out


REFERENCE_BUDGET_S = 120.0  # whole --impl reference run (warm-up + timed steps), about


def oracle_units(sets):
    """The oracle sample of one step split into 16 units, each one oracle
    call: the 8 slots of token 0 of the MoE layer, then the 1/16 of the head
    rows at n = 5 in 8 row chunks.  Returns [(bytes, call)] and a description."""
    from oracle import oracle as O
    ids, wts, h, x = sets[0]
    used = synth.distinct_experts(ids[:1], E)
    gu = np.zeros((E, 2 * F, H // QK, BB), dtype=np.uint8)
    dn = np.zeros((E, H, F // QK, BB), dtype=np.uint8)
    for e in used:
        gu[e] = synth.weight_blocks(2 * F, H, stream=synth.S_GATE_UP * 1000 + int(e))
        dn[e] = synth.weight_blocks(H, F, stream=synth.S_DOWN * 1000 + int(e))
    rows = HEAD_M // 16
    head = synth.weight_blocks(rows, HEAD_K, stream=synth.S_HEAD)
    units = [(EXPERT_BYTES, lambda j=j: O.moe(gu, dn, E, H, F, h[:1], ids[:1, j:j + 1], wts[:1, j:j + 1], swiglu=1))
             for j in range(ids.shape[1])]
    bounds = np.linspace(0, rows, 9).astype(int)
    units += [((b - a) * (HEAD_K // QK) * BB, lambda a=a, b=b: O.matvec(head[a:b], b - a, HEAD_K, x))
              for a, b in zip(bounds[:-1], bounds[1:])]
    desc = (f"token 0 of the batch-5 MoE layer (8 slots) + {rows} of {HEAD_M} head rows at n=5, "
            f"as 16 single-threaded oracle calls")
    return units, desc


def units_per_step(per_unit_s, n_steps, n_units):
    """Sample units per reference step so that n_steps steps take about
    REFERENCE_BUDGET_S: at least one unit, at most the whole sample."""
    return int(max(1, min(n_units, REFERENCE_BUDGET_S / max(n_steps, 1) / per_unit_s)))


def run_reference(args):
    """The CPU oracle on the arm's workload: each step runs the next n of the
    16 sample units (round robin), n chosen from one untimed pass over all of
    them so that the whole run takes about REFERENCE_BUDGET_S."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    sets = routing_sets()
    units, desc = oracle_units(sets)
    t0 = time.perf_counter()
    for _, call in units:  # calibration pass, untimed
        call()
    per_unit = (time.perf_counter() - t0) / len(units)
    n = units_per_step(per_unit, args.warmup + args.steps, len(units))
    nbytes, times, k = 0, [], 0
    for step in range(args.warmup + args.steps):
        b = 0
        t0 = time.perf_counter()
        for _ in range(n):
            ub, call = units[k % len(units)]
            call()
            b += ub
            k += 1
        dt = time.perf_counter() - t0
        if step >= args.warmup:
            times.append(dt)
            nbytes += b
    total = sum(times)
    value = nbytes / total / 1e9
    sample = f"per step {n} of 16 units, round robin over {desc}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "i8xi4-codebook/f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU ------

class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self, ident):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(ident), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        t0 = time.time()  # wait for the first sample so the timed region is covered
        while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for ln in f:
                p = [v.strip() for v in ln.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for name, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def timing_event(torch, stream):
    """A timing event whose CUDA handle exists (torch creates it lazily, at
    its first record), so the library can record it by handle."""
    e = torch.cuda.Event(enable_timing=True)
    e.record(stream)
    return e


def gpu_ident(torch, local):
    """nvidia-smi's name for this rank's GPU: its UUID when torch exposes it."""
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        parts = [p for p in vis.split(",") if p.strip()]
        return parts[local] if local < len(parts) else local


def aggregate(times_ms, weight_bytes, world, device=None):
    """Whole-job numbers of independent replicas: the slowest rank's time
    (max over ranks of each entry of times_ms) and the bytes of all ranks.
    Returns (max_times_ms list, GB/s of each time)."""
    import torch
    t = torch.tensor(list(times_ms), dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    total = float(weight_bytes) * world
    tmax = [float(v) for v in t.cpu()]
    return tmax, [total / (v * 1e-3) / 1e9 for v in tmax]


def build_layer(torch, cbq, n_exp=E, with_head=True):
    """All experts drawn from their seeded streams, repacked on device."""
    gu = np.empty((n_exp, 2 * F, H // QK, BB), dtype=np.uint8)
    dn = np.empty((n_exp, H, F // QK, BB), dtype=np.uint8)
    synth.expert_blocks(n_exp, 2 * F, H, stream=synth.S_GATE_UP, out=gu)
    synth.expert_blocks(n_exp, H, F, stream=synth.S_DOWN, out=dn)
    L = cbq.Moe(gu, dn, n_exp, H, F)
    del gu, dn
    if not with_head:
        return L
    head = cbq.Weights(synth.weight_blocks(HEAD_M, HEAD_K, stream=synth.S_HEAD), HEAD_M, HEAD_K)
    return L, head


def run_gpu(args):
    import torch
    import torch.distributed as dist
    from verify_matvec_gb300 import build, cbq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    l2_bytes = l2_cache_bytes(torch, dev)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    build.build()  # no-op once built; each rank loads the same in-tree library
    cbq.load()

    n_exp = args.experts
    if args.profile and args.case == "dense1":
        Ws = [cbq.Weights(synth.weight_blocks(4096, 4096, stream=synth.S_W * 1000 + 17 * i + 1), 4096, 4096)
              for i in range(16)]
        xx = torch.from_numpy(synth.activations(1, 4096, stream=synth.S_X)).to(dev)
        yy = torch.empty((1, 4096), dtype=torch.float32, device=dev)
        for i in range(args.warmup):
            cbq.cbq_matvec(Ws[i % 16], xx, y=yy)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for i in range(args.steps):
            cbq.cbq_matvec(Ws[i % 16], xx, y=yy)
        a1.record()
        torch.cuda.synchronize()
        print(json.dumps({"profile": True, "case": args.case, "us_per_call": 1e3 * a0.elapsed_time(a1) / args.steps,
                          "device_error": max(cbq.cbq_weights_get_error(w) for w in Ws)}), flush=True)
        return
    if args.profile and args.case in ("convert", "mmq16", "hc"):
        M, K = 16384, 4096
        if args.case == "hc":
            hb = [torch.from_numpy(synth.hc_logits(1 << 21, stream=synth.S_HC * 1000 + 100 + i)).to(dev)
                  for i in range(2)]
            hb_out = torch.empty_like(hb[0])
            call = lambda i: cbq.cbq_hc_sinkhorn(hb[i % 2], 20, out=hb_out)
            err = lambda: 0
        elif args.case == "convert":
            ws = [torch.randn((M, K), device=dev, generator=torch.Generator(device=dev).manual_seed(5 + i)) * 0.02
                  for i in range(2)]
            out = torch.empty((M, K // 32, 18), dtype=torch.uint8, device=dev)
            call = lambda i: cbq.cbq_quantize_weights(ws[i % 2], out=out)
            err = lambda: 0
        else:
            Ws = [cbq.Weights(synth.weight_blocks(M, K, stream=synth.S_W * 1000 + 31 * i + 3), M, K) for i in range(8)]
            xx = torch.from_numpy(synth.activations(16, K, stream=synth.S_X)).to(dev)
            yy = torch.empty((16, M), dtype=torch.float32, device=dev)
            call = lambda i: cbq.cbq_matmat(Ws[i % 8], xx, y=yy)
            err = lambda: max(cbq.cbq_weights_get_error(w) for w in Ws)
        for i in range(args.warmup):
            call(i)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for i in range(args.steps):
            call(i)
        a1.record()
        torch.cuda.synchronize()
        print(json.dumps({"profile": True, "case": args.case, "us_per_call": 1e3 * a0.elapsed_time(a1) / args.steps,
                          "device_error": err()}), flush=True)
        return
    if args.profile and args.case != "step":
        L = build_layer(torch, cbq, n_exp, with_head=False)
        if args.shared:
            cbq.cbq_moe_set_shared(L, synth.weight_blocks(2 * F, H, stream=synth.S_GATE_UP * 1000 + 999),
                                   synth.weight_blocks(H, F, stream=synth.S_DOWN * 1000 + 999))
        n_tok, k = (1, 4) if args.case == "b1" else (N_TOK, TOPK)
        tabs = []
        for i in range(N_SETS):
            ids_i, wts_i = synth.router(n_tok, k, n_exp, stream=synth.S_IDS + 300 + 17 * n_tok + i)
            tabs.append(tuple(torch.from_numpy(a).to(dev) for a in
                              (ids_i, wts_i, synth.activations(n_tok, H, stream=synth.S_H + 300 + i))))
        yl = torch.empty((n_tok, H), dtype=torch.float32, device=dev)
        for i in range(args.warmup):
            t = tabs[i % N_SETS]
            cbq.cbq_moe_matvec(L, t[2], t[0], t[1], y=yl)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for i in range(args.steps):
            t = tabs[i % N_SETS]
            cbq.cbq_moe_matvec(L, t[2], t[0], t[1], y=yl)
        a1.record()
        torch.cuda.synchronize()
        print(json.dumps({"profile": True, "case": args.case, "experts": n_exp, "shared_expert": args.shared,
                          "us_per_layer": 1e3 * a0.elapsed_time(a1) / args.steps,
                          "device_error": cbq.cbq_moe_get_error(L)}), flush=True)
        return
    L, head = build_layer(torch, cbq, n_exp)
    sets = routing_sets(n_exp=n_exp)
    d_sets = []
    for ids, wts, h, x in sets:
        d_sets.append(tuple(torch.from_numpy(a).to(dev) for a in (ids, wts, h, x)))
    distinct = [len(synth.distinct_experts(s[0], n_exp)) for s in sets]
    y = torch.empty((N_TOK, H), dtype=torch.float32, device=dev)
    yh = torch.empty((HEAD_N, HEAD_M), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    total = args.warmup + args.steps
    # Per-call events on every SAMPLE-th timed step only (the first included):
    # an event between two calls cuts the programmatic-dependent-launch overlap
    # of the one call's last kernel with the next call's first (about 10 us a
    # step with events on every step), so most timed steps run as a decode
    # loop runs them, and the per-call durations come from the sampled steps.
    SAMPLE = 8
    sampled = [i for i in range(args.warmup, total) if (i - args.warmup) % SAMPLE == 0]
    ev = {i: [timing_event(torch, stream) for _ in range(3)] for i in sampled}
    torch.cuda.synchronize()

    def step(i, events):
        # events around whole calls only (none between a call's own kernels,
        # whose programmatic-dependent-launch overlap they would cut): MoE call
        # start, MoE call end = head call start, head call end
        ids, wts, h, x = d_sets[i % N_SETS]
        if events is not None:
            events[0].record(stream)
        cbq.cbq_moe_matvec(L, h, ids, wts, swiglu=1, y=y)
        if events is not None:
            events[1].record(stream)
        cbq.cbq_matvec(head, x, y=yh)
        if events is not None:
            events[2].record(stream)

    # untimed warm-up
    for i in range(args.warmup):
        step(i, None)
    torch.cuda.synchronize()
    clocks = Clocks()
    clocks.start(gpu_ident(torch, local))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.warmup, total):
        step(i, ev.get(i))
    t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    cbq.cbq_moe_set_stage_events(L, None)
    ms = t0.elapsed_time(t1)

    timed = range(args.warmup, total)
    wbytes = [distinct[i % N_SETS] * EXPERT_BYTES + HEAD_BYTES for i in timed]
    k_moe = [ev[i][0].elapsed_time(ev[i][1]) for i in sampled]
    k_head = [ev[i][1].elapsed_time(ev[i][2]) for i in sampled]
    err = cbq.cbq_moe_get_error(L) | cbq.cbq_weights_get_error(head)

    # per-launch algorithmic bytes: weights + activations read + outputs written
    slots = N_TOK * TOPK
    moe_io = 8 * N_TOK * H + 8 * slots  # h in, y out, ids + router weights in (intermediates stay in L2)
    moe_alg = [distinct[i % N_SETS] * EXPERT_BYTES + moe_io for i in sampled]
    head_alg = HEAD_BYTES + 4 * HEAD_N * HEAD_K + 4 * HEAD_N * HEAD_M  # weights, x in, y out
    # each call is a chain of PDL launches and events go around whole calls,
    # so a kernel's figure includes the short launches of its call
    kern = {"k_moe (with its k_quantize and k_moe_combine launches)": (sum(k_moe), sum(moe_alg) / len(k_moe)),
            "k_matvec<5> (head, with its k_quantize launch)": (sum(k_head), head_alg)}
    dom = max(kern, key=lambda k: kern[k][0])
    dom_ms, dom_bytes = kern[dom][0] / len(sampled), kern[dom][1]
    peak, peak_kind = peaks()
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = None
    if source_digest() == PROFILED["source_digest"]:
        if dom.startswith("k_matvec"):
            traffic = PROFILED["k_matvec<5> (head)"]
        elif PROFILED["moe call per expert"] is not None:
            traffic = PROFILED["moe call per expert"] * sum(distinct[i % N_SETS] for i in sampled) / len(sampled)

    if args.profile:
        if rank == 0:
            print(json.dumps({"profile": True, "ms_per_step": ms / args.steps, "experts": n_exp,
                              "kernels_ms_per_step": {"moe call": sum(k_moe) / len(sampled),
                                                      "head": sum(k_head) / len(sampled)},
                              "device_error": err}), flush=True)
        if world > 1:
            dist.destroy_process_group()
        return

    # end to end through the host-buffer entry points (pinned host memory)
    h_sets = []
    for ids, wts, h, x in sets:
        h_sets.append(tuple(torch.from_numpy(a).pin_memory().numpy() for a in (ids, wts, h, x)))
    y_host = torch.empty((N_TOK, H), dtype=torch.float32).pin_memory().numpy()
    yh_host = torch.empty((HEAD_N, HEAD_M), dtype=torch.float32).pin_memory().numpy()

    def e2e_step(i):
        ids, wts, h, x = h_sets[i % N_SETS]
        cbq.cbq_moe_matvec_host(L, h, ids, wts, swiglu=1, y=y_host)
        cbq.cbq_matvec_host(head, x, y=yh_host)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.warmup, total):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)

    # microseconds per layer at batch 1 (top-4) and batch 5 (top-8).  A decode
    # loop replays its launches from a CUDA graph, so the per-call figure is
    # the replay of 16 captured calls (one per routing table) divided by 16;
    # the host-driven loop (one Python call per layer) is reported beside it,
    # with the split into the token quantization and the rest of the call.
    def graph_us(fn, n_calls=N_SETS, replays=25, samples=False):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for i in range(3):
                fn(i)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_calls):
                fn(i)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(replays + 1)]
        ev[0].record()
        for r in range(replays):
            g.replay()
            ev[r + 1].record()
        torch.cuda.synchronize()
        per_call = [1e3 * ev[r].elapsed_time(ev[r + 1]) / n_calls for r in range(replays)]
        return (1e3 * ev[0].elapsed_time(ev[-1]) / (replays * n_calls), per_call) if samples else \
            1e3 * ev[0].elapsed_time(ev[-1]) / (replays * n_calls)

    def layer_us(n_tok, k, reps=50, extra_experts=0):
        tabs = []
        for i in range(N_SETS):
            ids_i, wts_i = synth.router(n_tok, k, E, stream=synth.S_IDS + 300 + 17 * n_tok + i)
            tabs.append((torch.from_numpy(ids_i).to(dev), torch.from_numpy(wts_i).to(dev),
                         torch.from_numpy(synth.activations(n_tok, H, stream=synth.S_H + 300 + i)).to(dev),
                         len(synth.distinct_experts(ids_i, E))))
        yl = torch.empty((n_tok, H), dtype=torch.float32, device=dev)
        for i in range(5):
            t = tabs[i % N_SETS]
            cbq.cbq_moe_matvec(L, t[2], t[0], t[1], y=yl)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        stage_ev = [[timing_event(torch, stream) for _ in range(3)] for _ in range(reps)]
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(reps):
            t = tabs[i % N_SETS]
            cbq.cbq_moe_set_stage_events(L, stage_ev[i])
            cbq.cbq_moe_matvec(L, t[2], t[0], t[1], y=yl)
        b.record(stream)
        torch.cuda.synchronize()
        cbq.cbq_moe_set_stage_events(L, None)
        eager = 1e3 * a.elapsed_time(b) / reps
        split = [1e3 * sum(ev[j].elapsed_time(ev[j + 1]) for ev in stage_ev) / reps for j in range(2)]
        trials, per_replay = [], []
        for _ in range(5):
            mean, each = graph_us(lambda i: cbq.cbq_moe_matvec(L, tabs[i][2], tabs[i][0], tabs[i][1], y=yl),
                                  samples=True)
            trials.append(mean)
            per_replay += each
        us = statistics.median(trials)
        half = 2.776 * statistics.stdev(trials) / 5 ** 0.5  # 95% CI of the mean, 4 degrees of freedom
        ci = [statistics.mean(trials) - half, statistics.mean(trials) + half]
        q = statistics.quantiles(per_replay, n=10)  # per replay of the 16 calls, 5 x 25 replays
        spread = {"p10": q[0], "p50": statistics.median(per_replay), "p90": q[-1]}
        nbytes = (sum(t[3] for t in tabs) / N_SETS + extra_experts) * EXPERT_BYTES
        return us, nbytes / (us * 1e-6) / 1e9, eager, split, ci, spread

    b1_us, b1_gbs, b1_eager, b1_split, b1_ci, b1_q = layer_us(1, 4)
    b5_us, b5_gbs, b5_eager, b5_split, b5_ci, b5_q = layer_us(5, 8)

    # the same layers with an always-on shared expert of the routed shape
    # (one more expert's bytes per call, read in the same layer kernel)
    cbq.cbq_moe_set_shared(L, synth.weight_blocks(2 * F, H, stream=synth.S_GATE_UP * 1000 + 999),
                           synth.weight_blocks(H, F, stream=synth.S_DOWN * 1000 + 999))
    shared = {}
    for name, (n_tok, k) in (("batch1_top4", (1, 4)), ("batch5_top8", (5, 8))):
        us, gbs, _, _, ci, _ = layer_us(n_tok, k, reps=10, extra_experts=1)
        shared[name] = {"us": us, "weight_gbs": gbs, "frac_of_peak": gbs / peak, "ci95_us": ci}
    cbq.cbq_moe_set_shared(L, None, None)

    # dense decode projections (4096x4096, 16384x4096) through cbq_matvec, by
    # graph replay of one call per copy over copies whose bytes together are
    # at least four times L2 (every call reads its weights from HBM)
    dense = {}
    for M, K in ((4096, 4096), (16384, 4096)):
        wb = M * (K // QK) * BB
        copies = max(2, -(-4 * l2_bytes // wb))
        Ws = [cbq.Weights(synth.weight_blocks(M, K, stream=synth.S_W * 1000 + 17 * i + M // 4096), M, K)
              for i in range(copies)]
        for nc in (1, 5):
            xx = torch.from_numpy(synth.activations(nc, K, stream=synth.S_X)).to(dev)
            yy = torch.empty((nc, M), dtype=torch.float32, device=dev)
            us = graph_us(lambda i: cbq.cbq_matvec(Ws[i % copies], xx, y=yy), n_calls=copies, replays=8)
            gbs = wb / (us * 1e-6) / 1e9
            dense[f"{M}x{K}_n{nc}"] = {"us": us, "weight_gbs": gbs, "frac_of_peak": gbs / peak,
                                       "bar75_us": wb / (0.75 * peak * 1e9) * 1e6,
                                       "rotating_copies": copies, "rotating_bytes": copies * wb}
        del Ws

    # the tensor-core path (cbq_matmat) for 8 and 16 columns against
    # ceil(n/5) passes of the dp4a path, on the 16384 x 4096 projection and on
    # the head shape (graph replay; the head is larger than L2 by itself)
    mmq = {}
    for M, K, copies in ((16384, 4096, -(-4 * l2_bytes // (16384 * (4096 // QK) * BB))), (HEAD_M, HEAD_K, 1)):
        Ws = [head] if M == HEAD_M else [cbq.Weights(synth.weight_blocks(M, K, stream=synth.S_W * 1000 + 31 * i + 7),
                                                     M, K) for i in range(copies)]
        for nc in (8, 16):
            xx = torch.from_numpy(synth.activations(nc, K, stream=synth.S_X + nc)).to(dev)
            yy = torch.empty((nc, M), dtype=torch.float32, device=dev)
            t_mmq = graph_us(lambda i: cbq.cbq_matmat(Ws[i % len(Ws)], xx, y=yy), n_calls=len(Ws), replays=8)
            parts = [(c0, min(5, nc - c0)) for c0 in range(0, nc, 5)]
            xs = [xx[c0:c0 + kk].contiguous() for c0, kk in parts]
            ys = [torch.empty((kk, M), dtype=torch.float32, device=dev) for _, kk in parts]

            def passes(i):
                for xp, yp in zip(xs, ys):
                    cbq.cbq_matvec(Ws[i % len(Ws)], xp, y=yp)
            t_dp = graph_us(passes, n_calls=len(Ws), replays=8)
            wb = M * (K // QK) * BB
            mmq[f"{M}x{K}_n{nc}"] = {"tensor_core_us": t_mmq, "dp4a_passes_us": t_dp, "dp4a_passes": len(parts),
                                      "tensor_core_weight_gbs": wb / (t_mmq * 1e-6) / 1e9,
                                      "speedup_vs_dp4a": t_dp / t_mmq}
        del Ws

    # the weight converter (fp32 matrix -> codebook blocks) on a 16384 x 4096
    # matrix: 268 MB read, 38 MB written per call, two inputs alternating
    # (more than four times L2 between two reads of one input)
    Mc, Kc = 16384, 4096
    wc = [torch.randn((Mc, Kc), dtype=torch.float32, device=dev) * 0.02 for _ in range(2)]
    bc = torch.empty((Mc, Kc // QK, BB), dtype=torch.uint8, device=dev)
    conv_us = graph_us(lambda i: cbq.cbq_quantize_weights(wc[i % 2], out=bc), n_calls=2, replays=10)
    conv_bytes = Mc * Kc * 4 + Mc * (Kc // QK) * BB
    converter = {"shape": [Mc, Kc], "us": conv_us, "bytes_per_call": conv_bytes,
                 "gbs": conv_bytes / (conv_us * 1e-6) / 1e9, "frac_of_peak": conv_bytes / (conv_us * 1e-6) / 1e9 / peak}
    del wc, bc

    # the hyper-connection Sinkhorn normalisation (4 x 4 per token, 20 rounds):
    # a decoded token runs it twice per layer, 86 times over the model; timed
    # here on a verify batch of five tokens per call (86 calls per replay), and
    # on 2^21 matrices per call (134 MB in, 134 MB out, two inputs alternating)
    # for its throughput
    hc_iters, hc_calls = 20, 86
    hs = [torch.from_numpy(synth.hc_logits(N_TOK, stream=synth.S_HC * 1000 + i)).to(dev) for i in range(hc_calls)]
    hs_out = torch.empty_like(hs[0])
    hc_dec_us = graph_us(lambda i: cbq.cbq_hc_sinkhorn(hs[i], hc_iters, out=hs_out), n_calls=hc_calls, replays=10)
    n_hc = 1 << 21
    hb = [torch.from_numpy(synth.hc_logits(n_hc, stream=synth.S_HC * 1000 + 100 + i)).to(dev) for i in range(2)]
    hb_out = torch.empty_like(hb[0])
    hc_big_us = graph_us(lambda i: cbq.cbq_hc_sinkhorn(hb[i % 2], hc_iters, out=hb_out), n_calls=2, replays=10)
    hc_bytes = n_hc * 2 * cbq.CBQ_HC_NHC * cbq.CBQ_HC_NHC * 4
    hc = {"nhc": cbq.CBQ_HC_NHC, "iters": hc_iters,
          "verify_batch5_us_per_call": hc_dec_us, "calls_per_token": hc_calls,
          "us_per_token": hc_dec_us * hc_calls,
          "large_batch": {"matrices": n_hc, "us": hc_big_us, "matrices_per_s": n_hc / (hc_big_us * 1e-6),
                          "gbs": hc_bytes / (hc_big_us * 1e-6) / 1e9,
                          "frac_of_hbm_peak": hc_bytes / (hc_big_us * 1e-6) / 1e9 / peak}}
    del hs, hs_out, hb, hb_out

    # slowest rank decides; bytes add up over ranks
    (ms_max, e2e_max), (value, e2e_value) = aggregate([ms, e2e_ms], sum(wbytes), world, dev)
    h2d = N_TOK * H * 4 + 2 * slots * 4 + HEAD_N * HEAD_K * 4
    d2h = N_TOK * H * 4 + HEAD_N * HEAD_M * 4

    cpu = cpu_mt = None
    if rank == 0 and world == 1:
        nxt = oracle_next_rows()
        converter["cpu_oracle"] = nxt["weight_converter"]
        mmq["cpu_oracle"] = nxt["tensor_core_path"]
        hc["cpu_oracle"] = nxt["hc_sinkhorn"]
        n_cpu = 1
        _, t1s = oracle_sample(sets, 1)[0:2]
        n_cpu = max(1, min(20, int(10.0 / max(t1s[0], 1e-3))))
        step_bytes, times, sample = oracle_sample(sets, n_cpu)
        cpu = {"value": step_bytes * len(times) / sum(times) / 1e9, "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": f"{n_cpu} repetitions; " + sample}
        cores = os.cpu_count() or 1
        n_mt = max(1, min(40, int(5.0 * cores / max(t1s[0], 1e-3))))
        step_bytes, times, sample = oracle_sample(sets, n_mt, threads=cores)
        cpu_mt = {"value": step_bytes * len(times) / sum(times) / 1e9, "unit": "GB/s", "cores": cores,
                  "kind": "oracle", "sample": f"{n_mt} repetitions; " + sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "i8xi4-codebook/f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "n_tok": N_TOK, "topk": TOPK, "experts": E, "hidden": H,
                       "ffn": F, "head": [HEAD_M, HEAD_K], "head_cols": HEAD_N,
                       "distinct_experts_per_step": [distinct[i % N_SETS] for i in timed][:N_SETS],
                       "weight_bytes_per_step_mean": sum(wbytes) / len(wbytes),
                       "l2": "inputs larger than L2: every step reads ~0.7 GB of weights out of a 1.2 GB set "
                             "(all experts and the head), 16 rotating routing tables",
                       "l2_bytes": l2_bytes,
                       "rotating_sets_bytes": {"experts": E * EXPERT_BYTES, "head": HEAD_BYTES,
                                               "step_set": E * EXPERT_BYTES + HEAD_BYTES,
                                               "dense": {k_: v_["rotating_bytes"] for k_, v_ in dense.items()}},
                       "parallelism": f"replicas x{world}"},
            "us_per_layer": {"batch1_top4": b1_us, "batch5_top8": b5_us,
                             "batch1_weight_gbs": b1_gbs, "batch5_weight_gbs": b5_gbs,
                             "timing": "CUDA-graph replay of 16 captured calls x 25; median of 5 trials",
                             "ci95_us": {"batch1": b1_ci, "batch5": b5_ci},
                             "per_replay_us": {"batch1": b1_q, "batch5": b5_q},
                             "batch1_frac_of_peak": b1_gbs / peak, "batch5_frac_of_peak": b5_gbs / peak,
                             "bar75_us": {"batch1": b1_gbs * b1_us / (0.75 * peak),
                                          "batch5": b5_gbs * b5_us / (0.75 * peak)},
                             "eager_host_loop": {"batch1": b1_eager, "batch5": b5_eager},
                             "eager_split_us_quantize_layer": {"batch1": b1_split, "batch5": b5_split}},
            "us_per_layer_with_shared_expert": shared,
            "us_per_call_dense": dense,
            "weight_converter": converter,
            "tensor_core_path": mmq,
            "hc_sinkhorn": hc,
            "kernels_ms_per_step": {"moe layer call (k_quantize + k_moe + k_moe_combine)": sum(k_moe) / len(sampled),
                                    "head call (k_quantize + k_matvec<5>)": sum(k_head) / len(sampled),
                                    "sampled_steps": len(sampled)},
            "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "peak_nominal": NOMINAL_HBM_GBS, "frac_nominal": achieved / NOMINAL_HBM_GBS,
                         "traffic": traffic, "algorithmic_bytes_per_launch": dom_bytes},
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_mt,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": 5 * args.steps,  # per step: quantize, layer kernel, combine; quantize, head matvec
            "clocks": clk,
            "device_error": err,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
