"""Benchmark: one decode step of the rotated INT2 KV cache on GB300.

A step is the whole hot path for one batch: kv_append of the current token of
every sequence (rotate, clip, INT2 pack, BF16 window write) followed by
attn_decode over the full mixed INT2/BF16 cache (query rotation, split-K
attention, LSE merge, V un-rotation).  Inputs are synthetic (seeded normal
activations with heavy outlier channels) and resident in HBM; the cache is
pre-filled by untimed appends.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
of the workload (weak scaling, no data-path collective).
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "INT2+BF16 KV decode-attn tokens/s and KV GB/s (% of HBM peak), 1 GB300"
APPEND_METRIC = "INT2 KV append tokens/s (rotate + clip + INT2 pack), 1 GB300"
DEFAULT_WORKLOAD = "qwen3-8b-36L"
L2_FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="run only the first N layers of the workload (profiling a large workload's kernel on a "
                         "smaller cache); 0 = all")
    ap.add_argument("--hadamard", action="store_true",
                    help="data-free in-quant Hadamard rotation instead of the calibrated R_K / R_V")
    ap.add_argument("--v-bf16", action="store_true", help="K-only INT2: V kept BF16 at every position")
    ap.add_argument("--lloyd-max", action="store_true",
                    help="INT2 codes index the Lloyd-Max levels (0, rho, rho + 1, 2 rho + 1) instead of evenly spaced ones")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured once as a CUDA graph and replayed (reported under `graph`)")
    ap.add_argument("--calibrate", action="store_true",
                    help="time the R_K calibration (Sigma, eigenvectors, H P_br) instead of the decode step")
    ap.add_argument("--cpu-sample-worker", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--sample-heads", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--append-pairs", type=int, default=0, help=argparse.SUPPRESS)
    return ap.parse_args()


def workload_of(args):
    """The named workload, with --layers N keeping only its first N layers."""
    import dataclasses
    from int2_kv_cache_append_gb300 import synth as S
    w = S.WORKLOADS[args.workload]
    if getattr(args, "layers", 0) and 0 < args.layers < w.num_layers:
        w = dataclasses.replace(w, num_layers=args.layers)
    return w


def workload_desc(w) -> str:
    return (f"{w.name}: B{w.batch} Hq{w.num_q_heads} Hkv{w.num_kv_heads} D{w.head_dim} T{w.context} "
            f"S{w.sink} W{w.recent} g128 clip{w.k_clip}/{w.v_clip} layers{w.num_layers}"
            f"{' absorbV' if w.absorb_v else ''}")


def rotation_desc(args) -> str:
    return "in-quant Hadamard H_128 (data-free)" if getattr(args, "hadamard", False) else "calibrated R_K, R_V"


def kv_bytes_per_bh(w, T: int, v_bf16: bool = False) -> int:
    """Algorithmic K+V bytes one decode step reads for one (sequence, KV head)
    (with V kept BF16, an INT2 position reads K codes + scale/zero and a BF16 V row)."""
    D = w.head_dim
    S, W = w.sink, w.recent
    if T <= S:
        n_bf, n_i2 = T, 0
    else:
        tq = max(S, T - W)
        n_i2 = tq - S
        n_bf = S + (T - tq)
    if v_bf16:
        return n_i2 * (D // 4 + 4 * (D // 128) + 2 * D) + n_bf * 2 * 2 * D
    return n_i2 * 2 * (D // 4 + 4 * (D // 128)) + n_bf * 2 * 2 * D


def max_over_ranks(ms: float) -> float:
    """Slowest rank's time when torch.distributed is initialised (any backend), else ms."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(batch_per_rank: int, world: int, ms_max: float) -> float:
    """Weak scaling: every rank decodes its own batch; the job's rate uses the slowest rank."""
    return world * batch_per_rank / (ms_max / 1e3)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# DRAM bytes (read + write) per launch of the dominant kernel from ncu captures
# (profiles/<kernel>_<workload>.md), with the source file and its hash at
# capture: reported only while that source is unchanged.  The split-kernel
# entries are for the default mode; the 36-layer workload was captured with
# --layers 1 (every layer's launch reads the same bytes); at head_dim 512 the
# figure is the split kernel's alone (unrot_kernel reads R_V and the merged
# outputs, a few MB from L2).
MEASURED_TRAFFIC = {
    "qwen3-8b-36L": ("attn_decode.cu", "3cdce9215ee18187", 647665664),
    "hd512": ("attn_decode.cu", "3cdce9215ee18187", 753083136),
    "qwen3-32b-decode": ("attn_decode.cu", "3cdce9215ee18187", 77965824),
    "qwen3-4b-layer": ("attn_decode.cu", "3cdce9215ee18187", 152292352),
    "qwen3-32b-append": ("kv_append_tc.cu", "da55696891866101", 143004928),
}


def measured_traffic(workload: str):
    """ncu DRAM bytes per launch of the dominant kernel, or None if not measured on the current source."""
    entry = MEASURED_TRAFFIC.get(workload)
    if not entry:
        return None
    src = os.path.join(ROOT, "int2_kv_cache_append_gb300", "csrc", entry[0])
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return entry[2] if entry[1] == sha else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# CPU oracle sample (test infrastructure, timed as the CPU baseline)
# --------------------------------------------------------------------------
def cpu_sample_worker(workload: str, steps: int, warmup: int, heads: int, hadamard: bool = False,
                      v_bf16: bool = False, lloyd_max: bool = False):
    """Run inside a single-threaded child process: time the oracle's decode step
    (append of the current token + attention) for batch row 0 of the workload,
    restricted to its first `heads` KV heads (and their query heads)."""
    import numpy as np
    from int2_kv_cache_append_gb300 import synth as S
    from oracle import oscar_oracle as O

    w = S.WORKLOADS[workload]
    T = w.context
    G = w.num_q_heads // w.num_kv_heads
    c = O.Config(1, 1, G * heads, heads, w.head_dim, w.sink, w.recent, T, w.k_clip, w.v_clip,
                 flags=(O.FLAG_HADAMARD if hadamard else 0) | (O.FLAG_V_BF16 if v_bf16 else 0)
                 | (O.FLAG_LLOYD_MAX if lloyd_max else 0))
    RK, RV = (None, None) if hadamard else S.rotations(w, 0)
    k, v = S.kv_rows(w, 0, T, batch=1)
    k, v = k[:, :, :heads], v[:, :, :heads]
    cache = O.new_cache(c)
    O.append(c, cache, 0, k[:, :T - 1], v[:, :T - 1], [0], RK, RV)
    q = S.queries(w, 0, batch=1)[:, :G * heads]
    times = []
    for i in range(warmup + steps):
        t0 = time.perf_counter()
        O.append(c, cache, 0, k[:, T - 1:], v[:, T - 1:], [T - 1], RK, RV)
        O.decode(c, cache, 0, q, [T], RK, RV, absorb_v=w.absorb_v)
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    print(json.dumps({"sec_per_step": statistics.mean(times), "steps": len(times)}))


def cpu_append_worker(workload: str, pairs: int):
    """Run inside a single-threaded child process: time the oracle's append of
    the workload's new tokens for `pairs` (sequence, KV head) pairs."""
    import numpy as np
    from int2_kv_cache_append_gb300 import synth as S
    from oracle import oscar_oracle as O

    w = S.WORKLOADS[workload]
    c = O.Config(1, 1, w.num_q_heads // w.num_kv_heads, 1, w.head_dim, w.sink, w.recent, w.context, w.k_clip,
                 w.v_clip)
    RK, RV = S.rotations(w, 0)
    k, v = S.kv_rows(w, 0, w.append_tokens, batch=1)
    cache = O.new_cache(c)
    t0 = time.perf_counter()
    for i in range(pairs):
        h = i % w.num_kv_heads
        O.append(c, cache, 0, k[:, :, h:h + 1], v[:, :, h:h + 1], [w.context - w.append_tokens], RK, RV)
    print(json.dumps({"sec": time.perf_counter() - t0, "pairs": pairs}))


def _sample_cmd(workload: str, steps: int, warmup: int, heads: int, hadamard=False, v_bf16=False, lloyd_max=False,
                append_pairs: int = 0):
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-sample-worker", "--workload", workload,
           "--steps", str(steps), "--warmup", str(warmup), "--sample-heads", str(heads)] + (
               ["--hadamard"] if hadamard else []) + (["--v-bf16"] if v_bf16 else []) + (
               ["--lloyd-max"] if lloyd_max else [])
    if append_pairs:
        cmd += ["--append-pairs", str(append_pairs)]
    return cmd


_SAMPLE_ENV = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
                   CUDA_VISIBLE_DEVICES="")


def run_cpu_sample(workload: str, steps: int, warmup: int, heads: int, hadamard: bool = False,
                   v_bf16: bool = False, lloyd_max: bool = False, append_pairs: int = 0):
    """One single-threaded oracle sample in a child process."""
    cmd = _sample_cmd(workload, steps, warmup, heads, hadamard, v_bf16, lloyd_max, append_pairs)
    r = subprocess.run(cmd, env=_SAMPLE_ENV, capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("cpu sample failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_cpu_samples_parallel(n: int, workload: str, steps: int, warmup: int, heads: int, hadamard: bool = False,
                             v_bf16: bool = False, lloyd_max: bool = False, append_pairs: int = 0):
    """n single-threaded oracle samples at once, one child process per host core."""
    cmd = _sample_cmd(workload, steps, warmup, heads, hadamard, v_bf16, lloyd_max, append_pairs)
    procs = [subprocess.Popen(cmd, env=_SAMPLE_ENV, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for _ in range(n)]
    res = []
    for p in procs:
        out, err = p.communicate(timeout=1800)
        if p.returncode != 0:
            raise RuntimeError("cpu sample failed: " + err[-2000:])
        res.append(json.loads(out.strip().splitlines()[-1]))
    return res


def cpu_baseline_decode(w, args, L: int):
    """The oracle's decode step (append of the current token + attention over T)
    for one sequence and one layer, every KV head, timed on one host thread and
    on every host core at once (one process per core): tokens/s of the whole
    workload = sequences per second / layers."""
    Hkv = w.num_kv_heads
    ncores = os.cpu_count() or 1
    one = run_cpu_sample(w.name, steps=2, warmup=1, heads=Hkv, hadamard=args.hadamard, v_bf16=args.v_bf16,
                         lloyd_max=args.lloyd_max)
    allc = run_cpu_samples_parallel(ncores, w.name, steps=2, warmup=1, heads=Hkv, hadamard=args.hadamard,
                                    v_bf16=args.v_bf16, lloyd_max=args.lloyd_max)
    single = 1.0 / (one["sec_per_step"] * L)
    total = sum(1.0 / (r["sec_per_step"] * L) for r in allc)
    return {"value": total, "unit": "tokens/s", "cores": ncores, "kind": "oracle",
            "single_thread_value": single,
            "sample": (f"oracle (numpy; codec float32, attention float64) decode step of one sequence and one "
                       f"layer of {w.name} (append of the current token, then attention over T={w.context} for "
                       f"all {Hkv} KV heads), {one['steps']} timed steps after 1 warm-up; single thread, and one "
                       f"single-threaded process per host core at once ({ncores}); tokens/s = sequences per "
                       f"second / {L} layers")}


def cpu_baseline_append(w):
    """The oracle's append of the workload in full (every sequence and KV head),
    on one host thread and split over every host core (one process each)."""
    pairs = w.batch * w.num_kv_heads
    ncores = os.cpu_count() or 1
    one = run_cpu_sample(w.name, 0, 0, 0, append_pairs=pairs)
    per = max(1, -(-pairs // ncores))
    allc = run_cpu_samples_parallel(min(ncores, pairs), w.name, 0, 0, 0, append_pairs=per)
    tok_per_pair = w.append_tokens / w.num_kv_heads  # a token spans every KV head
    single = pairs * tok_per_pair / one["sec"]
    total = sum(r["pairs"] * tok_per_pair / r["sec"] for r in allc)
    return {"value": total, "unit": "tokens/s", "cores": ncores, "kind": "oracle", "single_thread_value": single,
            "sample": (f"oracle append (rotate in float64, codec float32, windows) of all {w.batch} x "
                       f"{w.num_kv_heads} (sequence, KV head) pairs of {w.append_tokens} new tokens on one thread; "
                       f"all cores: {min(ncores, pairs)} single-threaded processes with {per} pairs each")}


def reference_arm(args):
    """The oracle as the reference implementation, timed on every host core at
    once (one single-threaded process per core, each running the same bounded
    sample; the rates add up)."""
    from int2_kv_cache_append_gb300 import synth as S
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = S.WORKLOADS[args.workload]
    steps = max(1, args.steps)
    ncores = os.cpu_count() or 1
    t0 = time.time()
    if w.append_tokens > 0:
        # one (sequence, KV head) pair of the append per step
        res = run_cpu_samples_parallel(ncores, args.workload, 0, 0, 0, append_pairs=steps)
        tok_per_pair = w.append_tokens / w.num_kv_heads
        value = sum(r["pairs"] * tok_per_pair / r["sec"] for r in res)
        ms = statistics.mean(r["sec"] / r["pairs"] for r in res) * 1e3
        sample = (f"oracle append of {w.append_tokens} new tokens for one (sequence, KV head) pair of "
                  f"{args.workload} per step, {steps} steps, one single-threaded process per host core "
                  f"({ncores}); tokens/s = pairs x {w.append_tokens} / {w.num_kv_heads} KV heads / s")
        sample_desc = "one (sequence, KV head) append per step"
    else:
        # about 75 ms of oracle work per KV head and step at T = 16384: keep the run near two minutes
        heads = max(1, min(w.num_kv_heads, int(120.0 / (0.075 * (steps + args.warmup) * w.context / 16384))))
        res = run_cpu_samples_parallel(ncores, args.workload, steps, args.warmup, heads, args.hadamard,
                                       args.v_bf16, args.lloyd_max)
        # a sample step is heads / Hkv of one sequence's decode step in one of L layers
        value = sum((heads / w.num_kv_heads) / r["sec_per_step"] / w.num_layers for r in res)
        ms = statistics.mean(r["sec_per_step"] for r in res) * 1e3
        sample = (f"oracle (numpy; codec float32, attention float64) on batch row 0 of {args.workload}, {heads} "
                  f"of {w.num_kv_heads} KV heads of one layer per step: append of the current token + decode over "
                  f"T={w.context}; one single-threaded process per host core ({ncores}); tokens/s scaled by the "
                  f"fraction of a token's work ({heads}/{w.num_kv_heads} heads, 1/{w.num_layers} layers) sampled")
        sample_desc = f"{heads} of {w.num_kv_heads} KV heads of one sequence and layer per step"
    line = {"impl": "reference", "metric": METRIC if w.append_tokens == 0 else APPEND_METRIC, "value": value,
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(w) + (f" append{w.append_tokens}" if w.append_tokens else ""),
                       "rotation": rotation_desc(args),
                       "cache": "int2 K + bf16 V" if args.v_bf16 else "int2+bf16",
                       "levels": "Lloyd-Max (0, rho, rho+1, 2rho+1), rho = 1.16 (float32)" if args.lloyd_max else "uniform",
                       "sample": sample_desc},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": ncores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.time() - t0}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
def ours(args):
    import numpy as np
    import torch

    from int2_kv_cache_append_gb300 import build as B
    from int2_kv_cache_append_gb300 import oscar_kv as K
    from int2_kv_cache_append_gb300 import synth as S

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0:
        B.build()
    if dist is not None:
        dist.barrier()
    K.lib()

    w = workload_of(args)
    L, Bsz, Hq, Hkv, D, T = w.num_layers, w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.context
    flags = ((K.FLAG_ABSORB_V if w.absorb_v else 0) | (K.FLAG_HADAMARD if args.hadamard else 0)
             | (K.FLAG_V_BF16 if args.v_bf16 else 0) | (K.FLAG_LLOYD_MAX if args.lloyd_max else 0))
    cfg = K.KVConfig(L, Bsz, Hq, Hkv, D, w.sink, w.recent, T, w.k_clip, w.v_clip, flags)
    lay = K.layout_query(cfg)
    decode_kernels = K.decode_kernels(cfg)
    stream = torch.cuda.current_stream()

    # ---- setup (untimed): rotations, cache pre-fill of T-1 tokens per sequence
    gen = torch.Generator(device=dev)
    cache = torch.empty(lay["total_bytes"], dtype=torch.uint8, device=dev)
    rots = []
    for layer in range(L):
        if args.hadamard:  # no matrices: the library applies the in-quant Hadamard itself
            rots.append((None, None))
            continue
        RK, RV = S.rotations(w, layer if L == 1 else layer % 4)
        rots.append((torch.from_numpy(RK).to(dev), torch.from_numpy(RV).to(dev)))
    ch = S.outlier_channels(w.config_id, 0, D)
    chunk = max(1, min(T - 1, (1 << 27) // (Bsz * Hkv * D)))
    for layer in range(L):
        gen.manual_seed(1000 * w.config_id + layer + 7919 * rank)
        pos = 0
        while pos < T - 1:
            n = min(chunk, T - 1 - pos)
            k = S.activations_torch(gen, (Bsz, n, Hkv, D), ch, dtype=torch.bfloat16, device=dev)
            v = S.activations_torch(gen, (Bsz, n, Hkv, D), ch, dtype=torch.bfloat16, device=dev)
            K.kv_append(cfg, cache, layer, k, v, torch.full((Bsz,), pos, dtype=torch.int32, device=dev),
                        rots[layer][0], rots[layer][1])
            pos += n
    torch.cuda.synchronize()
    gen.manual_seed(99 + rank)
    q = S.activations_torch(gen, (Bsz, Hq, D), ch, dtype=torch.bfloat16, device=dev)
    k1 = S.activations_torch(gen, (Bsz, 1, Hkv, D), ch, dtype=torch.bfloat16, device=dev)
    v1 = S.activations_torch(gen, (Bsz, 1, Hkv, D), ch, dtype=torch.bfloat16, device=dev)
    start = torch.full((Bsz,), T - 1, dtype=torch.int32, device=dev)
    seq = torch.full((Bsz,), T, dtype=torch.int32, device=dev)
    out = torch.empty((Bsz, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Bsz, Hq), dtype=torch.float32, device=dev)
    ws = torch.empty(lay["decode_workspace_bytes"], dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(qq=q, kk=k1, vv=v1, oo=out):
        for layer in range(L):
            RK, RV = rots[layer]
            K.decode_step(cfg, cache, layer, kk, vv, start, qq, seq, RK, RV, oo, ws, lse=lse, seq_len_hint=T,
                          status=status)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    # clocks: sample across a short untimed load phase and the timed region
    clocks = ClockSampler(dev.index)
    clocks.start()
    t_end = time.time() + 1.5
    while time.time() < t_end:
        flush.zero_()
        step()
        torch.cuda.synchronize()

    K_ = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_ * L)]
    for a_, b_ in kev:  # torch creates the CUDA event on first record; the library re-records them
        a_.record(stream)
        b_.record(stream)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K_):
        flush.zero_()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if dist is not None:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(statistics.mean(step_ms))

    # split-kernel duration: the same steps again with events recorded on the
    # library's stream right around the split kernel (an event between two
    # kernels stops the second from launching early, so this pass is kept out
    # of the step timing above)
    pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_)]
    for i in range(K_):
        flush.zero_()
        pev[i][0].record(stream)
        for layer in range(L):
            RK, RV = rots[layer]
            ks, ke = kev[i * L + layer]
            K.set_profile_events(ks, ke)
            K.decode_step(cfg, cache, layer, k1, v1, start, q, seq, RK, RV, out, ws, lse=lse, seq_len_hint=T,
                          status=status)
            K.set_profile_events(None, None)
        pev[i][1].record(stream)
    torch.cuda.synchronize()
    split_ms = [a.elapsed_time(b) for a, b in kev]
    # the split kernels' share of the very steps they were timed in
    prof_step_ms = statistics.mean(a.elapsed_time(b) for a, b in pev)
    split_share = sum(split_ms) / sum(a.elapsed_time(b) for a, b in pev)
    clocks.stop()

    # ---- optional: the same step captured as one CUDA graph, replayed K times
    graph_line = None
    if args.graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            step()
        stream.wait_stream(side)
        for _ in range(3):
            flush.zero_()
            graph.replay()
        torch.cuda.synchronize()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_)]
        for i in range(K_):
            flush.zero_()
            gev[i][0].record(stream)
            graph.replay()
            gev[i][1].record(stream)
        torch.cuda.synchronize()
        g_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in gev))
        graph_line = {"ms_per_step": g_ms, "value": whole_job_tokens_per_s(Bsz, world, g_ms),
                      "kernels_per_replay": (1 + decode_kernels) * L}

    # ---- end-to-end through the public API with host buffers
    q_h = q.cpu().pin_memory()
    k_h = k1.cpu().pin_memory()
    v_h = v1.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    q_d, k_d, v_d = torch.empty_like(q), torch.empty_like(k1), torch.empty_like(v1)
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K_)]
    for i in range(K_):
        flush.zero_()
        e2e_ev[i][0].record(stream)
        q_d.copy_(q_h, non_blocking=True)
        k_d.copy_(k_h, non_blocking=True)
        v_d.copy_(v_h, non_blocking=True)
        step(q_d, k_d, v_d, out)
        out_h.copy_(out, non_blocking=True)
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = statistics.mean(a.elapsed_time(b) for a, b in e2e_ev)
    h2d = (q.numel() * q.element_size() + 2 * k1.numel() * k1.element_size()) * L
    d2h = out.numel() * out.element_size() * L
    st = int(status.item())

    if rank != 0:
        return
    kv_bytes = kv_bytes_per_bh(w, T, args.v_bf16) * Bsz * Hkv * L
    tokens_per_s = whole_job_tokens_per_s(Bsz, world, ms)
    peak, peak_kind = measured_peaks()
    split_avg_ms = statistics.mean(split_ms)
    achieved = kv_bytes / L / (split_avg_ms / 1e3) / 1e9
    step_gbs = kv_bytes / (ms / 1e3) / 1e9
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline_decode(w, args, L)
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": K_,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": workload_desc(w), "step": "decode_step per layer: kv_append(1 token/seq) + attn_decode in one call",
                   "rotation": rotation_desc(args),
                   "l2": "flushed between steps (512 MiB write)",
                   "cache": "int2 K + bf16 V" if args.v_bf16 else "int2+bf16",
                   "levels": "Lloyd-Max (0, rho, rho+1, 2rho+1), rho = 1.16 (float32)" if args.lloyd_max else "uniform",
                   "parallelism":
                       f"replica x{world}" if world > 1 else "single"},
        "kv_gbs": step_gbs, "kv_pct_hbm": step_gbs / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     # the committed counters were taken with calibrated rotations, INT2 V, uniform levels
                     "traffic": None if (args.v_bf16 or args.hadamard or args.lloyd_max)
                     else measured_traffic(args.workload),
                     "kernel": "split_kernel" + ("" if decode_kernels == 2 else " + unrot_kernel")
                               + " (attn_decode)",
                     "kernel_ms": split_avg_ms, "peak_kind": peak_kind,
                     # kernel_ms comes from a second pass of the same steps with events
                     # recorded around each split launch; that pass's own step time and
                     # the split kernels' share of it:
                     "kernel_pass_ms_per_step": prof_step_ms, "kernel_share_of_step": split_share,
                     "algorithmic_bytes_per_launch": kv_bytes // L},
        "e2e": {"value": world * Bsz / (e2e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        # the append + attn_decode's kernels (qrot, split, and unrot where used)
        "gpu_launches": (1 + decode_kernels) * L * K_,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
        "graph": graph_line,
        "dev_status": st,
        "wall_s_timed": wall,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def ours_append(args):
    """Append-phase workload: every step appends n new tokens per sequence at the
    end of the context (rotation GEMM on the tensor cores, clip, INT2 pack, ring)."""
    import torch

    from int2_kv_cache_append_gb300 import build as B
    from int2_kv_cache_append_gb300 import oscar_kv as K
    from int2_kv_cache_append_gb300 import synth as S

    if args.hadamard or args.v_bf16 or args.lloyd_max:
        raise SystemExit("bench.py: --hadamard, --v-bf16 and --lloyd-max select decode modes; the append "
                         "workload measures the tensor-core append of the default mode only")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    if rank == 0:
        B.build()
    if world > 1:
        dist.barrier()
    w = S.WORKLOADS[args.workload]
    Bsz, H, D, T, n = w.batch, w.num_kv_heads, w.head_dim, w.context, w.append_tokens
    cfg = K.KVConfig(1, Bsz, w.num_q_heads, H, D, w.sink, w.recent, T, w.k_clip, w.v_clip)
    lay = K.layout_query(cfg)
    cache = torch.zeros(lay["total_bytes"], dtype=torch.uint8, device=dev)
    RK, RV = S.rotations(w, 0)
    RK, RV = torch.from_numpy(RK).to(dev), torch.from_numpy(RV).to(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(5 + rank)
    ch = S.outlier_channels(w.config_id, 0, D)
    k = S.activations_torch(gen, (Bsz, n, H, D), ch, dtype=torch.bfloat16, device=dev)
    v = S.activations_torch(gen, (Bsz, n, H, D), ch, dtype=torch.bfloat16, device=dev)
    start = torch.full((Bsz,), T - n, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        K.kv_append(cfg, cache, 0, k, v, start, RK, RV, status=status)
    torch.cuda.synchronize()
    clocks = ClockSampler(dev.index)
    clocks.start()
    t_end = time.time() + 1.5
    while time.time() < t_end:
        flush.zero_()
        K.kv_append(cfg, cache, 0, k, v, start, RK, RV, status=status)
        torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a_, b_ in ev:
        flush.zero_()
        a_.record(stream)
        K.kv_append(cfg, cache, 0, k, v, start, RK, RV, status=status)
        b_.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    ms = max_over_ranks(statistics.mean(a_.elapsed_time(b_) for a_, b_ in ev))
    # e2e: inputs copied from pinned host memory every step, status word read back
    k_h, v_h = k.cpu().pin_memory(), v.cpu().pin_memory()
    st_h = torch.empty(1, dtype=torch.int32).pin_memory()
    k_d, v_d = torch.empty_like(k), torch.empty_like(v)
    e2e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a_, b_ in e2e:
        flush.zero_()
        a_.record(stream)
        k_d.copy_(k_h, non_blocking=True)
        v_d.copy_(v_h, non_blocking=True)
        K.kv_append(cfg, cache, 0, k_d, v_d, start, RK, RV, status=status)
        st_h.copy_(status, non_blocking=True)
        b_.record(stream)
    torch.cuda.synchronize()
    e2e_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in e2e)
    if rank != 0:
        return
    rows = Bsz * n * H * 2
    tokens = world * Bsz * n
    ring_rows = Bsz * H * min(n, w.recent) * 2
    hbm_bytes = rows * (2 * D + D // 4 + 4 * (D // 128)) + ring_rows * 2 * D
    flops = rows * 2 * D * D
    peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
    gbs = hbm_bytes / (ms / 1e3) / 1e9
    tfs = flops / (ms / 1e3) / 1e12
    line = {
        "metric": APPEND_METRIC, "value": tokens / (ms / 1e3),
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(w) + f" append{n}", "l2": "flushed between steps (512 MiB write)"},
        "roofline": {"bound": "hbm" if gbs / peaks["hbm_gbs"] >= tfs / peaks["bf16_tflops"] else "tensor",
                     "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "traffic": measured_traffic(args.workload) if args.workload == "qwen3-32b-append" else None,
                     "kernel": "kv_append_tc_kernel",
                     "tensor_tflops_algorithmic": tfs, "tensor_frac_algorithmic": tfs / peaks["bf16_tflops"],
                     "tensor_frac_issued_3piece": 3 * tfs / peaks["bf16_tflops"],
                     "algorithmic_bytes_per_launch": hbm_bytes, "algorithmic_flops_per_launch": flops},
        "e2e": {"value": tokens / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": 2 * k.numel() * k.element_size(), "d2h_bytes_per_step": 4},
        "gpu_launches": args.steps, "clocks": clocks.summary(),
        "cpu_baseline": None if (args.no_cpu_baseline or world > 1) else cpu_baseline_append(w),
        "dev_status": int(status.item()),
    }
    print(json.dumps(line), flush=True)


def calibrate_arm(args):
    """R_K and R_V calibration from 20,000 calibration tokens of the workload's
    shape (every query head's row pooled for Q, every KV head's for K and V):
    GPU time per calibration, with the oracle (numpy float64 + LAPACK) timed on
    the same rows as the CPU baseline."""
    import numpy as np
    import torch

    from int2_kv_cache_append_gb300 import build as B
    from int2_kv_cache_append_gb300 import oscar_kv as K
    from int2_kv_cache_append_gb300 import synth as S
    B.build()
    w = S.WORKLOADS[args.workload]
    D = w.head_dim
    rows = 20000 * w.num_q_heads
    kv_rows = 20000 * w.num_kv_heads
    gen = torch.Generator(device="cuda")
    gen.manual_seed(7)
    ch = S.outlier_channels(w.config_id, 0, D)
    q = S.activations_torch(gen, (rows, D), ch)
    k = S.activations_torch(gen, (kv_rows, D), ch)
    v = S.activations_torch(gen, (kv_rows, D), ch)
    out = torch.empty((D, D), dtype=torch.float32, device="cuda")
    out_v = torch.empty((D, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(K.calibrate_workspace_bytes(D), dtype=torch.uint8, device="cuda")
    ws_v = torch.empty(K.calibrate_rv_workspace_bytes(D, kv_rows), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    steps = max(1, min(args.steps, 20))

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in ev:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    ms = timed(lambda: K.calibrate_rk(q, out, ws, status=st))
    ms_v = timed(lambda: K.calibrate_rv(q, k, v, out_v, ws_v, status=st))
    qn, kn, vn = q.cpu().numpy(), k.cpu().numpy(), v.cpu().numpy()
    from oracle import oscar_oracle as O
    t0 = time.perf_counter()
    ref = O.calibrate_rk(qn)
    cpu_s = time.perf_counter() - t0
    t0 = time.perf_counter()
    ref_v = O.calibrate_rv(qn, kn, vn)
    cpu_v = time.perf_counter() - t0
    line = {"metric": "R_K calibration time (Sigma = Q^T Q, eigenvectors, H P_br), 1 GB300", "value": ms,
            "unit": "ms", "higher_is_better": False, "n_gpus": 1, "steps": steps, "warmup": max(3, args.warmup),
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(w), "rows": rows, "head_dim": D,
                       "inputs": f"{rows * D * 4 / 1e6:.0f} MB of float32 rows (larger than L2)"},
            "max_abs_diff_vs_oracle": float(np.abs(out.cpu().numpy().astype(np.float64) - ref).max()),
            "dev_status": int(st.item()),
            "cpu_baseline": {"value": cpu_s * 1e3, "unit": "ms", "kind": "oracle", "cores": os.cpu_count(),
                             "sample": "the oracle (numpy float64 Q^T Q + LAPACK eigh) on the same rows"},
            "rv": {"metric": "R_V calibration time (score-weighted Sigma_V, eigenvectors, H P_br)", "value": ms_v,
                   "unit": "ms", "q_rows": rows, "kv_rows": kv_rows,
                   "max_abs_diff_vs_oracle": float(np.abs(out_v.cpu().numpy().astype(np.float64) - ref_v).max()),
                   "cpu_baseline": {"value": cpu_v * 1e3, "unit": "ms", "kind": "oracle", "cores": os.cpu_count(),
                                    "sample": "the oracle (numpy float64 weights, Sigma_V + LAPACK eigh) on the "
                                              "same rows"}}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.calibrate:
        calibrate_arm(args)
        return
    if args.cpu_sample_worker and args.append_pairs:
        cpu_append_worker(args.workload, args.append_pairs)
        return
    if args.cpu_sample_worker:
        cpu_sample_worker(args.workload, args.steps, args.warmup, args.sample_heads, args.hadamard, args.v_bf16,
                          args.lloyd_max)
        return
    if args.impl == "reference":
        reference_arm(args)
        return
    from int2_kv_cache_append_gb300 import synth as S
    if S.WORKLOADS[args.workload].append_tokens > 0:
        ours_append(args)
        return
    ours(args)


if __name__ == "__main__":
    main()
