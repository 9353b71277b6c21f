#!/usr/bin/env python3
"""Benchmark of the FP8-KV decode hot path on GB300.

One step = one decode layer of the batch-16, 8192-token workload (16 query /
2 KV heads, head_dim 128, e4m3 K and V with per-(token, head) fp32 scales):
one fp8kv_decode_step call, which appends the step's new token of every
sequence (position 8191) and attends over the 8192 cached tokens.  On the
tensor-core kernel that is one launch (append, flash-decoding split and the
merge of the fp32 partials all inside it); on the CUDA-core kernel it is
three (append, split, merge).
Each step reads a different one of L distinct layer caches (L * 69 MB well
above the 126 MB L2), so every step streams its cache from HBM.  Steps are
replayed from CUDA graphs; timing uses CUDA events on the launching stream.

Prints ONE JSON line (rank 0).  `--impl reference` times the oracle (plain
fp64 C on the host cores) on the same metric instead.
"""
import argparse
import dataclasses
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp8_quantized_kv_gb300 import synth  # noqa: E402

WORKLOAD = "decode_b16_ctx8192"
METRIC = "decode attn KV-read GB/s (% of HBM peak) and µs/layer at B16 ctx8192, 1 GB300"
KERNEL_IDS = {"auto": 0, "cuda_cores": 1, "tensor_cores": 2, "tensor_cores_k_f16": 3,
              "tensor_cores_k_f16_producer": 4}
PAGE_NUMBER_GBS = 550.0   # the pages' figure for this workload (RTX 5070 Ti, Triton, codes only)
# fp8kv_decode_step flag: each layer's step streams its own cache while the
# previous layer's step finishes (programmatic dependent launch); the layers'
# caches are distinct, as in a model
STEP_EARLY_CACHE_READ = 1
L2_BYTES = 129 * 10**6      # GB300 L2 capacity


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="fp8kv", choices=["fp8kv", "reference"])
    ap.add_argument("--dtype", default="k8v8", choices=["k8v8", "k16v8", "k16v16", "k8v16", "mxk8v8"])
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--chunk", type=int, default=200)
    ap.add_argument("--kernel", default="auto", choices=list(KERNEL_IDS))
    ap.add_argument("--no-controls", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-steps", type=int, default=200)
    ap.add_argument("--plain-launch", action="store_true",
                    help="launch every step only after the previous one finished (no early cache read)")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-shapes", action="store_true")
    ap.add_argument("--no-interval", action="store_true")
    ap.add_argument("--shape", default=None, choices=["decode_b16_ctx512", "decode_b16_ctx8192", "paged_b64_hostile"],
                    help="time only the fused decode step on this workload (for profiling) and exit")
    ap.add_argument("--group", type=int, default=0,
                    help="with --shape: query heads per KV head (default: the workload's own)")
    ap.add_argument("--prefill-size", default=None, metavar="TOKENS,BATCH,QHEADS,KVHEADS",
                    help="time only the tensor-core prefill at this size (head_dim 128) and exit")
    return ap.parse_args(argv)


# ------------------------------------------------------------ distributed --

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(bytes_per_step, steps, local_ms, ws):
    """Whole-job figure of the timed region: the slowest rank's time, and the
    bytes every rank processed (each rank runs its own copy of the workload:
    weak scaling) per second of that time, in GB/s."""
    t_max = max_over_ranks(local_ms, ws)
    return t_max, ws * bytes_per_step * steps / (t_max * 1e-3) / 1e9


# ----------------------------------------------------------------- bytes --

def step_bytes(spec, dtype, T):
    """Algorithmic bytes of one step: KV codes (or bf16) + scales read, Q read,
    O written (bf16), plus the appended token's rows (bf16 in, cache out)."""
    B, Hq, Hkv, D = spec.batch, spec.q_heads, spec.kv_heads, spec.head_dim
    k8, v8 = dtype in ("k8v8", "k8v16", "mxk8v8"), dtype in ("k8v8", "k16v8", "mxk8v8")
    row_bytes = D * ((1 if k8 else 2) + (1 if v8 else 2)) + 4 * (int(k8) + int(v8))
    kv = B * Hkv * T * row_bytes
    qo = 2 * B * Hq * D * 2
    append = B * Hkv * (2 * D * 2 + row_bytes)
    split = kv + B * Hq * D * 2
    return {"step": kv + qo + append, "kv": kv, "split_kernel": split, "qo": qo, "append": append}


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
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

    def summary(self, t0, t1):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        inside = [s for t, s in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        if not inside:
            near = min(self.samples, key=lambda ts: min(abs(ts[0] - t0), abs(ts[0] - t1)))
            inside = [near[1]]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in inside if num(s[1]) is not None]
        mx = [num(s[2]) for s in inside if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in inside for n, v in zip(names, s[5:9]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


# ----------------------------------------------------------------- peaks --

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm_gb_s", "hbm"):
            if key in d:
                v = d[key]
                v = v.get("value", v.get("gbs")) if isinstance(v, dict) else v
                return float(v), "measured"
        for k, v in d.items():
            if "hbm" in k.lower() and isinstance(v, (int, float)):
                return float(v), "measured"
    except (OSError, ValueError, TypeError):
        pass
    return 6800.0, "fallback"


def tensor_peak():
    """Dense bf16 tensor-core peak in TFLOP/s (f16 runs at the same rate):
    the burst figure of MEASURED_PEAKS.json when present, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("bf16_tflops", "bf16_TFLOPs", "bf16"):
            if key in d:
                v = d[key]
                v = v.get("value") if isinstance(v, dict) else v
                return float(v), "measured"
    except (OSError, ValueError, TypeError):
        pass
    return 1900.0, "fallback"


def kernel_source_sha(kernel_file):
    """Hash of one kernel's sources: its .cu file, every shared .cuh header
    and the public headers (a change anywhere else leaves it alone)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_quantized_kv_gb300", "csrc")
    inc = os.path.join(ROOT, "include")
    files = [os.path.join(csrc, kernel_file)]
    files += [os.path.join(csrc, n) for n in sorted(os.listdir(csrc)) if n.endswith(".cuh")]
    files += [os.path.join(inc, n) for n in sorted(os.listdir(inc)) if n.endswith(".h")]
    for path in files:
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode() + f.read())
    return h.hexdigest()[:16]


def traffic_from_profile(kernel_key, sha):
    """dram bytes per launch from a committed ncu summary, only if it was taken
    on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel_key)
        if ent and ent.get("source_sha") == sha:
            return float(ent["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError, TypeError):
        pass
    return None


# ---------------------------------------------------------------- oracle --

def host_description():
    """The host the CPU baseline ran on: architecture, logical CPUs and the
    CPU model where the OS reports one (the baseline itself uses one core)."""
    import platform
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"machine": platform.machine(), "logical_cpus": os.cpu_count(), "model": model}


def oracle_sample(inp, n_seqs, tokens):
    """Oracle work for `n_seqs` sequences over `tokens` cached tokens: e4m3
    dequantisation of their K/V and fp64 decode attention.  Returns seconds
    and the algorithmic KV bytes this sample stands for."""
    import numpy as np
    import oracle
    spec = inp.spec
    D, Hkv = spec.head_dim, spec.kv_heads
    q = oracle.bf16_to_double(synth.bf16_bits(inp.q[:n_seqs]))
    kb, vb = [], []
    for b in range(n_seqs):
        s = int(inp.cu_seqlens[b])
        kb.append(synth.bf16_bits(inp.k[s:s + tokens]).transpose(1, 0, 2))
        vb.append(synth.bf16_bits(inp.v[s:s + tokens]).transpose(1, 0, 2))
    kc, ks = oracle.quantize(np.stack(kb))
    vc, vs = oracle.quantize(np.stack(vb))
    lens = np.full(n_seqs, tokens, np.int32)
    t0 = time.perf_counter()
    k = oracle.dequantize(kc, ks)
    v = oracle.dequantize(vc, vs)
    oracle.decode_attention(q, k, v, lens, 1.0 / math.sqrt(D))
    dt = time.perf_counter() - t0
    nbytes = n_seqs * Hkv * tokens * (2 * D + 8) + 2 * n_seqs * spec.q_heads * D * 2
    return dt, nbytes


# Workloads and sequence samples of the fp8_kv_error report: the lengths of
# the workload (paged: the two ends of its length range), seeded like the
# workload, hostile keys where it has them.
KV_ERROR_SAMPLES = {
    "tiny_decode": (77, 128),
    "decode_b16_ctx512": (512, 512),
    "decode_b16_ctx8192": (8192, 8192),
    "paged_b64_hostile": (1024, 16384),
}
KV_ERROR_DTYPES = ("k8v8", "k16v8", "k8v16", "mxk8v8", "k16v16")


def fp8_kv_errors(samples=None, dtypes=KV_ERROR_DTYPES):
    """fp8_kv_error ("FP8 KV cache (fp8_kv, opt-in)", bullet "Math"): the
    relative L2 change of decode attention (all sequences and query heads of
    the sample together) when the bf16 K/V are replaced by what each cache
    dtype stores -- e4m3 codes with a per-row scale, or MXFP8 keys (e4m3 codes
    with one power-of-two scale per 32 elements), on the e4m3 sides; the bf16
    values on the bf16 sides.  Computed by the oracle in fp64 on the host."""
    import numpy as np
    import oracle
    samples = KV_ERROR_SAMPLES if samples is None else samples
    res = {}
    for name, lens in samples.items():
        spec = synth.WORKLOADS[name]
        inp = synth.decode_inputs(spec, device="cpu", seq_lens=list(lens))
        D = spec.head_dim
        B, T = len(lens), max(lens)
        q = oracle.bf16_to_double(synth.bf16_bits(inp.q))
        kb = np.zeros((B, spec.kv_heads, T, D), np.uint16)
        vb = np.zeros_like(kb)
        for b, n in enumerate(lens):
            s = int(inp.cu_seqlens[b])
            kb[b, :, :n] = synth.bf16_bits(inp.k[s:s + n]).transpose(1, 0, 2)
            vb[b, :, :n] = synth.bf16_bits(inp.v[s:s + n]).transpose(1, 0, 2)
        seq = np.asarray(lens, np.int32)
        sm = 1.0 / math.sqrt(D)
        k16, v16 = oracle.bf16_to_double(kb), oracle.bf16_to_double(vb)
        o_ref = oracle.decode_attention(q, k16, v16, seq, sm)
        k8 = oracle.dequantize(*oracle.quantize(kb))
        v8 = oracle.dequantize(*oracle.quantize(vb))
        kmx = oracle.mx_dequantize(*oracle.mx_quantize(kb)) if D % 32 == 0 else None
        sides = {"k8v8": (k8, v8), "k16v8": (k16, v8), "k8v16": (k8, v16), "mxk8v8": (kmx, v8),
                 "k16v16": (k16, v16)}
        res[name] = {}
        for dt in dtypes:
            k, v = sides[dt]
            if k is None:
                continue
            o = oracle.decode_attention(q, k, v, seq, sm)
            res[name][dt] = float(np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-300))
    return res


def run_reference(args, ws, rank):
    if rank != 0:
        return
    spec = synth.WORKLOADS[WORKLOAD]
    T = spec.seq_lens[0]
    inp = synth.decode_inputs(spec, device="cpu", seq_lens=[T] * 2)
    # size each step so the whole run stays within about two minutes
    dt1, _ = oracle_sample(inp, 1, 512)
    per_token = dt1 / 512
    budget = 120.0 / max(1, args.steps + args.warmup)
    tokens = int(max(16, min(T, budget / per_token)))
    tokens -= tokens % 16 or 0
    tokens = max(16, tokens)
    for _ in range(args.warmup):
        oracle_sample(inp, 1, tokens)
    tot_t, tot_b = 0.0, 0
    for _ in range(args.steps):
        dt, nb = oracle_sample(inp, 1, tokens)
        tot_t += dt
        tot_b += nb
    gbs = tot_b / tot_t / 1e9
    sample = (f"per step: 1 sequence x {spec.kv_heads} KV heads x {tokens} tokens of the {WORKLOAD} "
              f"workload ({spec.q_heads} query heads, head_dim {spec.head_dim}): e4m3 dequantise + fp64 "
              "decode attention by the oracle (C, single thread); value and ms_per_step are this "
              "sample's own: its algorithmic KV + q/out bytes over its measured time")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "batch": 1, "q_heads": spec.q_heads,
                   "kv_heads": spec.kv_heads, "head_dim": spec.head_dim, "ctx": tokens,
                   "cache": "k8v8", "layout": "contiguous", "parallelism": "rank 0 only",
                   "kernel": "oracle", "step": "oracle dequantise + fp64 decode attention",
                   "launch": "host call", "l2": "host memory"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", "host": host_description(),
                         "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm --

class Layer:
    """One layer: its own cache, zero-filled workspace and pre-built C-ABI
    argument tuple for fp8kv_decode_step."""

    def __init__(self, cache, q, lens, ws_tensor, out, knew, vnew, Hq, sm_scale, kernel, flags):
        from fp8_quantized_kv_gb300._lib import get_lib
        self.lib = get_lib()
        self.cache = cache
        self.keep = (q, lens, ws_tensor, out, knew, vnew)
        P = lambda t: ctypes.c_void_p(t.data_ptr())
        self.a_step = (P(q), P(knew), P(vnew), cache.struct_ref, P(lens), Hq, ctypes.c_float(sm_scale), 0,
                       kernel, P(ws_tensor), ws_tensor.numel(), P(out), 0, ctypes.c_uint32(flags))

    def step(self, s):
        r = self.lib.fp8kv_decode_step(*self.a_step, s)
        if r:
            raise RuntimeError(f"fp8kv_decode_step status {r}")


def build_layers(spec, dtype, L, inp, kernel, flags=0):
    import fp8_quantized_kv_gb300 as fk
    B, Hq, Hkv, D = spec.batch, spec.q_heads, spec.kv_heads, spec.head_dim
    T = spec.seq_lens[0]
    cap = T
    base = fk.Fp8KVCache.contiguous(B, Hkv, D, cap, dtype)
    # tokens 0..T-2 are the cached context; token T-1 is appended by each step
    lens_prev = torch.full((B,), T - 1, dtype=torch.int64)
    keep = torch.ones(B * T, dtype=torch.bool)
    keep[T - 1::T] = False
    sidx = torch.repeat_interleave(torch.arange(B), lens_prev).to(torch.int32).cuda()
    pos = torch.cat([torch.arange(T - 1)] * B).to(torch.int32).cuda()
    fk.fp8kv_append(base, inp.k[keep.cuda()].contiguous(), inp.v[keep.cuda()].contiguous(), sidx, pos)
    knew = inp.k[T - 1::T].contiguous()          # [B, Hkv, D]: token T-1 of each sequence
    vnew = inp.v[T - 1::T].contiguous()
    new_sidx = torch.arange(B, dtype=torch.int32, device="cuda")
    new_pos = torch.full((B,), T - 1, dtype=torch.int32, device="cuda")
    lens = torch.full((B,), T, dtype=torch.int32, device="cuda")
    q = inp.q.contiguous()
    layers = []
    for li in range(L):
        if li == 0:
            c = base
        else:
            clone = lambda t: None if t is None else t.clone()
            c = fk.Fp8KVCache(dtype=dtype, layout=0, batch=B, kv_heads=Hkv, head_dim=D,
                              k=clone(base.k), v=clone(base.v), k_scale=clone(base.k_scale),
                              v_scale=clone(base.v_scale), max_tokens=cap)
        wsb = fk.fp8kv_decode_step_workspace_bytes(c, Hq, 0, kernel)
        ws_t = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
        layers.append(Layer(c, q, lens, ws_t, out, knew, vnew, Hq, 1.0 / math.sqrt(D), kernel, flags))
    torch.cuda.synchronize()
    return layers, (q, knew, vnew, lens)


def capture(layers, n_steps, with_events):
    """CUDA graph of n_steps steps cycling over the layers; optionally with
    timing events around each step (event-record nodes)."""
    g = torch.cuda.CUDAGraph()
    evs = []
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            for i in range(n_steps):
                L = layers[i % len(layers)]
                if with_events:
                    e = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
                    e[0].record()
                L.step(sp)
                if with_events:
                    e[1].record()
                    evs.append(e)
    torch.cuda.current_stream().wait_stream(s)
    return g, evs


def spacer():
    """Keep the current stream busy for a few tens of microseconds (a spin
    kernel) just before a device-timed region's start event: the host's
    latency in launching the first timed work (a graph replay) then falls
    before the start timestamp instead of inside the timed region.  The
    end-to-end measurement has no spacer."""
    torch.cuda._sleep(100_000)


def time_graph_steps(layers, K, chunk, ws):
    """Time exactly K steps replayed from CUDA graphs with no event nodes
    (the step time), then replay an instrumented copy of one chunk whose
    event-record nodes bracket every kernel (the per-kernel breakdown)."""
    chunk = max(1, min(chunk, K))
    g, _ = capture(layers, chunk, False)
    rem = K % chunk
    g_rem = capture(layers, rem, False)[0] if rem else None
    reps = K // chunk
    g.replay()                                  # one untimed replay: instantiate, warm
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    spacer()
    start.record()
    for _ in range(reps):
        g.replay()
    if g_rem is not None:
        g_rem.replay()
    end.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(ws)
    total_ms = start.elapsed_time(end)
    per = None
    try:                                         # event-record graph nodes need `external`
        torch.cuda.Event(enable_timing=True, external=True)
        gi, evs = capture(layers, chunk, True)
        gi.replay()
        gi.replay()
        torch.cuda.synchronize()
        per = {"step_ms": statistics.mean([e[0].elapsed_time(e[1]) for e in evs])}
    except TypeError:
        pass
    return total_ms, per, (t_wall0, t_wall1)


def e2e_run(layers, host, K, W, kernel, early=False):
    """Through the public Python API with host buffers: each step's inputs
    (q, k_new, v_new, seq_lens) sit in page-locked host memory and its
    output goes to page-locked host memory; fp8kv_decode_step reads and
    writes them across the host link itself (the device addresses pinned
    host memory directly; no copy calls).  The steps of all layers are
    captured once in a CUDA graph (with `early`, each launched as the
    previous one's programmatic dependent, as in the device-timed run) and
    the graph is replayed, as a serving loop would, so the timed region holds
    the steps with their host-side traffic rather than the Python call
    overhead of issuing them."""
    import fp8_quantized_kv_gb300 as fk
    q, knew, vnew, lens = host["dev"]
    hq, hk, hv, hl = host["pinned"]
    out_h = host["out"]
    wss = [torch.zeros(fk.fp8kv_decode_step_workspace_bytes(L.cache, q.shape[1], 0, kernel),
                       dtype=torch.uint8, device="cuda") for L in layers]

    def step(i, early_read):
        j = i % len(layers)
        fk.fp8kv_decode_step(hq, hk, hv, layers[j].cache, hl, out=out_h, workspace=wss[j], kernel=kernel,
                             early_cache_read=early_read)

    n = len(layers)
    for i in range(max(W, n)):
        step(i, False)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for j in range(n):
            step(j, early and j > 0)
    reps = max(1, (K + n - 1) // n)          # whole replays of the n layers
    for _ in range(max(1, (W + n - 1) // n)):
        g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.Event(enable_timing=True)
    en = torch.cuda.Event(enable_timing=True)
    st.record()
    for _ in range(reps):
        g.replay()
    en.record()
    torch.cuda.synchronize()
    if fk.fp8kv_get_device_error() != 0:
        raise RuntimeError("e2e run raised a device error")
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hl))
    # per step over the steps actually run
    return st.elapsed_time(en) * K / (reps * n), h2d, out_h.numel() * out_h.element_size()


def prefill_flops(n, batch, q_heads, head_dim):
    """Algorithmic FLOPs of one causal prefill: query i attends keys 0..i, and
    each (query, key) pair costs a head_dim dot product for QK and another for
    P.V, 2 FLOPs per multiply-add: 4 D per pair, n (n + 1) / 2 pairs per head."""
    return batch * 4.0 * head_dim * q_heads * n * (n + 1) / 2


def time_prefill(spec, batch, K, warmup, ws, min_sets=1):
    """Launches of the tensor-core causal prefill over K8/V8 caches holding
    `batch` copies of the workload's sequence: enough independent input sets
    (Q, cache, output) rotated launch by launch that they exceed the L2
    twice over (at least `min_sets`, at most 8); `warmup` launches, then K
    timed ones between CUDA events on the launching stream.  Returns
    (max-over-ranks time per launch in us, FLOPs per launch, input sets)."""
    import fp8_quantized_kv_gb300 as fk
    n, Hq, Hkv, D = spec.n_tokens, spec.q_heads, spec.kv_heads, spec.head_dim
    pin = synth.prefill_inputs(spec, device="cuda")
    k_all = pin.k.repeat(batch, 1, 1).contiguous()
    v_all = pin.v.repeat(batch, 1, 1).contiguous()
    sidx = torch.repeat_interleave(torch.arange(batch, dtype=torch.int32), n).cuda()
    pos = torch.arange(n, dtype=torch.int32).repeat(batch).cuda()
    set_bytes = batch * n * (2 * Hq * D * 2 + Hkv * 2 * (D + 4))
    n_sets = max(min_sets, min(8, -(-2 * L2_BYTES // set_bytes)))
    sets = []
    for _ in range(n_sets):
        cache = fk.Fp8KVCache.contiguous(batch, Hkv, D, n, "k8v8")
        fk.fp8kv_append(cache, k_all, v_all, sidx, pos)
        q = pin.q[None].expand(batch, -1, -1, -1).clone(memory_format=torch.contiguous_format)
        out = torch.empty(batch, n, Hq, D, dtype=torch.bfloat16, device="cuda")
        sets.append((cache, q, out))
    p0 = torch.zeros(batch, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()

    def run(i):
        cache, q, out = sets[i % len(sets)]
        fk.fp8kv_prefill_attention(q, cache, p0, out=out, kernel="tensor_cores", stream=stream)

    for i in range(max(3, warmup)):
        run(i)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    spacer()
    e0.record(stream)
    for i in range(K):
        run(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    if fk.fp8kv_get_device_error() != 0:
        raise RuntimeError("prefill raised a device error")
    flops = prefill_flops(n, batch, Hq, D)
    t_max, _ = aggregate(0, K, e0.elapsed_time(e1), ws)
    return t_max / K * 1e3, flops, n_sets


def measure_prefill(args, ws):
    """Causal prefill of the 2048-token, 28 q / 4 KV head workload over a K8/V8
    cache (tensor-core kernel).  Eight independent copies (Q, cache, output:
    ~250 MB, above L2) are rotated; the timed region is `args.prefill_steps`
    launches between CUDA events on the launching stream."""
    spec = synth.PREFILL_WORKLOADS["prefill_2048"]
    n, Hq, Hkv, D = spec.n_tokens, spec.q_heads, spec.kv_heads, spec.head_dim
    K = args.prefill_steps
    us, flops, _ = time_prefill(spec, 1, K, args.warmup, ws, min_sets=8)
    achieved = flops / (us * 1e-6) / 1e12
    peak, kind = tensor_peak()
    return {"workload": "prefill_2048", "batch": 1, "tokens": n, "q_heads": Hq, "kv_heads": Hkv,
            "head_dim": D, "cache": "k8v8", "kernel": "prefill_tc", "launches": K,
            "us_per_launch": us, "value": ws * achieved, "unit": "TFLOP/s",
            "l2": "8 input sets rotated (~250 MB, above L2)",
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "peak_kind": f"{kind} (dense bf16; f16 operands run at the same rate)",
                         "traffic": traffic_from_profile("prefill_k8v8_2048", kernel_source_sha("prefill_tc.cu")),
                         "traffic_unit": "DRAM bytes per launch",
                         "algorithmic_flops_per_launch": flops}}


def measure_shapes(args):
    """The decode step on the other decode workloads: batch 16 at 512 tokens
    (40 rotated layer caches, above L2) and the paged batch-64 serving decode
    (lengths U[1024, 16384], 16-token pages, hostile keys; one 1.2-2.3 GB
    cache), the four cache dtypes, on each kernel.  Plain launches, CUDA-graph
    replay, CUDA events on the launching stream."""
    import fp8_quantized_kv_gb300 as fk
    res = {}
    for wl, n_layers, K in (("decode_b16_ctx512", 40, 400), ("paged_b64_hostile", 1, 20)):
        spec = synth.WORKLOADS[wl]
        inp = synth.decode_inputs(spec, device="cuda")
        B, Hq, Hkv, D = spec.batch, spec.q_heads, spec.kv_heads, spec.head_dim
        lens64 = inp.seq_lens.to(torch.int64)
        sidx = torch.repeat_interleave(torch.arange(B), lens64).to(torch.int32).cuda()
        pos = torch.cat([torch.arange(int(n)) for n in lens64]).to(torch.int32).cuda()
        last = (inp.cu_seqlens[1:] - 1).cuda()
        knew, vnew = inp.k[last].contiguous(), inp.v[last].contiguous()
        lens = inp.seq_lens.cuda()
        q = inp.q.contiguous()
        res[wl] = {"group": spec.group, "tokens": int(lens64.sum())}
        for dtype in ("k8v8", "k16v8", "k8v16", "k16v16"):
            k8, v8 = dtype in ("k8v8", "k8v16"), dtype in ("k8v8", "k16v8")
            row = D * ((1 if k8 else 2) + (1 if v8 else 2)) + 4 * (int(k8) + int(v8))
            nbytes = int(lens64.sum()) * Hkv * row + 2 * B * Hq * D * 2 + B * Hkv * (2 * D * 2 + row)
            caches = []
            for _ in range(n_layers):
                if spec.page_size is None:
                    c = fk.Fp8KVCache.contiguous(B, Hkv, D, int(lens64.max()), dtype)
                else:
                    c = fk.Fp8KVCache.paged(inp.page_table, inp.num_pages, Hkv, D, spec.page_size, dtype)
                fk.fp8kv_append(c, inp.k.contiguous(), inp.v.contiguous(), sidx, pos)
                caches.append(c)
            out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
            res[wl][dtype] = {"algorithmic_bytes": nbytes}
            for kname in ("cuda_cores", "tensor_cores"):
                wss = [torch.zeros(fk.fp8kv_decode_step_workspace_bytes(c, Hq, 0, kname), dtype=torch.uint8,
                                   device="cuda") for c in caches]

                def step(i):
                    fk.fp8kv_decode_step(q, knew, vnew, caches[i % n_layers], lens, out=out,
                                         workspace=wss[i % n_layers], kernel=kname)
                for i in range(max(3, args.warmup)):
                    step(i)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for i in range(K):
                        step(i)
                g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                spacer()
                e0.record()
                g.replay()
                e1.record()
                torch.cuda.synchronize()
                us = e0.elapsed_time(e1) / K * 1e3
                res[wl][dtype][kname] = {"us_per_step": us, "GBps": nbytes / (us * 1e-6) / 1e9}
                del g, wss
            del caches
            torch.cuda.empty_cache()
        if fk.fp8kv_get_device_error() != 0:
            raise RuntimeError(f"{wl}: device error")
    return res


def measure_interval(args):
    """Steady-state tile initiation interval of the tensor-core decode split:
    the slope of the step time against the context length (2K-16K tokens) at
    a fixed 4 splits, batch 16, 16 q / 2 KV heads, head_dim 128, times the
    tokens a CTA covers per 128-token tile.  Per cache dtype; 8 rotated layer
    caches, plain launches, CUDA-graph replay."""
    import fp8_quantized_kv_gb300 as fk
    ctxs = (2048, 4096, 8192, 16384)
    S = 4
    res = {}
    spec0 = synth.WORKLOADS[WORKLOAD]
    B, Hq, Hkv, D = spec0.batch, spec0.q_heads, spec0.kv_heads, spec0.head_dim
    for dtype in ("k8v8", "mxk8v8", "k16v8", "k8v16", "k16v16"):
        pts = []
        for T in ctxs:
            spec = synth.DecodeWorkload("ii", B, Hq, Hkv, D, seed=2, seq_lens=(T,) * B)
            inp = synth.decode_inputs(spec, device="cuda")
            sidx = torch.repeat_interleave(torch.arange(B), torch.full((B,), T)).to(torch.int32).cuda()
            pos = torch.arange(T, dtype=torch.int32).repeat(B).cuda()
            knew, vnew = inp.k[T - 1::T].contiguous(), inp.v[T - 1::T].contiguous()
            lens = inp.seq_lens.cuda()
            q = inp.q.contiguous()
            caches = []
            for _ in range(8):
                c = fk.Fp8KVCache.contiguous(B, Hkv, D, T, dtype)
                fk.fp8kv_append(c, inp.k.contiguous(), inp.v.contiguous(), sidx, pos)
                caches.append(c)
            out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
            wss = [torch.zeros(fk.fp8kv_decode_step_workspace_bytes(c, Hq, S, "tensor_cores"), dtype=torch.uint8,
                               device="cuda") for c in caches]

            def step(i):
                fk.fp8kv_decode_step(q, knew, vnew, caches[i % 8], lens, out=out, workspace=wss[i % 8],
                                     num_splits=S, kernel="tensor_cores")
            for i in range(5):
                step(i)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(200):
                    step(i)
            g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            spacer()
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            pts.append((T, e0.elapsed_time(e1) / 200 * 1e3))
            del g, caches, wss
            torch.cuda.empty_cache()
        n = len(pts)
        mx = sum(t for t, _ in pts) / n
        my = sum(u for _, u in pts) / n
        slope = sum((t - mx) * (u - my) for t, u in pts) / sum((t - mx) ** 2 for t, _ in pts)   # us per token
        res[dtype] = {"us_at_ctx": {str(t): u for t, u in pts}, "fixed_us": my - slope * mx,
                      "interval_us_per_tile": slope * 128 * S,
                      "note": "one CTA's 128-token tile; 128 CTAs stream at once"}
    if fk.fp8kv_get_device_error() != 0:
        raise RuntimeError("interval sweep: device error")
    return res


def measure_variant(spec, dtype, args, ws, inp, flags=None, kernel=None, n_layers=None):
    if flags is None:
        flags = 0 if args.plain_launch else STEP_EARLY_CACHE_READ
    kid = KERNEL_IDS[args.kernel if kernel is None else kernel]
    layers, dev = build_layers(spec, dtype, args.layers if n_layers is None else n_layers, inp, kid, flags)
    for i in range(max(3, args.warmup)):                      # eager warm-up steps
        L = layers[i % len(layers)]
        L.step(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    total_ms, per, wall = time_graph_steps(layers, args.steps, args.chunk, ws)
    return layers, dev, total_ms, per, wall


def run_gpu(args, ws, rank):
    spec = synth.WORKLOADS[WORKLOAD]
    T = spec.seq_lens[0]
    inp = synth.decode_inputs(spec, device="cuda")
    dev_index = torch.cuda.current_device()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = int(vis.split(",")[dev_index]) if vis and vis.split(",")[dev_index].isdigit() else dev_index
    sampler = ClockSampler(smi_index)
    sampler.start()
    time.sleep(0.3)

    layers, dev, total_ms, per, wall = measure_variant(spec, args.dtype, args, ws, inp)
    nb = step_bytes(spec, args.dtype, T)
    t_max, value = aggregate(nb["step"], args.steps, total_ms, ws)
    ms_per_step = t_max / args.steps
    peak, peak_kind = hbm_peak()
    clocks = sampler.summary(*wall)

    # e2e through the public API with host buffers
    pinned = tuple(t.cpu().pin_memory() for t in dev)
    out_h = torch.empty((spec.batch, spec.q_heads, spec.head_dim), dtype=torch.bfloat16).pin_memory()
    e2e_ms, h2d, d2h = e2e_run(layers, {"dev": dev, "pinned": pinned, "out": out_h}, args.steps, args.warmup,
                               KERNEL_IDS[args.kernel], early=not args.plain_launch)
    e2e_ms, e2e_val = aggregate(nb["step"], args.steps, e2e_ms, ws)
    sampler.stop()

    tensor = args.kernel != "cuda_cores"
    roof = None
    if tensor:
        # the tensor-core step is one kernel (append + split + merge): its
        # average launch duration is the timed region's time per step (start
        # and end events around the K back-to-back launches), and its
        # algorithmic bytes are the whole step's
        launch_ms = ms_per_step
        achieved = nb["step"] / (launch_ms * 1e-3) / 1e9
        sha = kernel_source_sha("decode_mma.cu")
        roof = {"bound": "hbm", "kernel": "decode_split_tc (fused decode step)",
                "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak, "peak_kind": f"{peak_kind} (HBM copy)",
                "traffic": traffic_from_profile("decode_split_k8v8_b16_ctx8192", sha)
                if args.dtype == "k8v8" else None,
                "algorithmic_bytes_per_launch": nb["step"],
                "avg_launch_us": launch_ms * 1e3, "source_sha": sha,
                "event_node_step_us": None if per is None else per["step_ms"] * 1e3}

    plain = None
    if not args.plain_launch and tensor:
        del layers
        torch.cuda.empty_cache()
        layers, _, pms, _, _ = measure_variant(spec, args.dtype, args, ws, inp, flags=0)
        pms, pval = aggregate(nb["step"], args.steps, pms, ws)
        plain = {"us_per_layer": pms / args.steps * 1e3, "GBps": pval,
                 "note": "every step launched after the previous one finished"}

    controls = {}
    del layers
    torch.cuda.empty_cache()
    if not args.no_controls:
        for other in ("k8v8", "mxk8v8", "k16v8", "k8v16", "k16v16"):
            if other == args.dtype:
                continue
            ls, _, tms, pr, _ = measure_variant(spec, other, args, ws, inp)
            tms = max_over_ranks(tms, ws)
            ob = step_bytes(spec, other, T)
            controls[other] = {"us_per_layer": tms / args.steps * 1e3,
                               "GBps": ob["step"] * args.steps / (tms * 1e-3) / 1e9,
                               "step_kernel_us": None if pr is None else pr["step_ms"] * 1e3}
            del ls
            torch.cuda.empty_cache()

    # where K is prepared: the native e4m3 QK against the transform path (each
    # K tile converted to f16 in shared memory, 16-bit QK), same step, same
    # launch mode
    transform = None
    if not args.no_controls and args.dtype == "k8v8" and args.kernel in ("auto", "tensor_cores"):
        transform = {"native_e4m3_qk": {"us_per_layer": ms_per_step * 1e3, "GBps": value}}
        for kname, who in (("tensor_cores_k_f16", "the softmax warpgroup that owns the tile"),
                           ("tensor_cores_k_f16_producer", "the TMA producer warp")):
            ls, _, xms, _, _ = measure_variant(spec, "k8v8", args, ws, inp, kernel=kname)
            xms = max_over_ranks(xms, ws)
            transform[kname] = {"us_per_layer": xms / args.steps * 1e3,
                                "GBps": nb["step"] * args.steps / (xms * 1e-3) / 1e9,
                                "converted_by": who}
            del ls
            torch.cuda.empty_cache()
        transform["note"] = ("transform path: each K tile converted to f16 in shared memory, QK as kind::f16 "
                             "on an f16 query; 4 cache stages instead of 6 (the two f16 K buffers take the room)")

    # L2-warm: one layer's cache (69 MB at this shape) replayed, so it stays in
    # the 126 MB L2; the headline keeps 8 layers and streams from HBM
    l2_warm = None
    if not args.no_controls and tensor:
        ls, _, lms, _, _ = measure_variant(spec, args.dtype, args, ws, inp, n_layers=1)
        lms = max_over_ranks(lms, ws)
        l2_warm = {"us_per_layer": lms / args.steps * 1e3,
                   "GBps": nb["step"] * args.steps / (lms * 1e-3) / 1e9,
                   "note": "one layer cache replayed (L2-resident); not the headline"}
        del ls
        torch.cuda.empty_cache()

    prefill = None if args.no_prefill else measure_prefill(args, ws)
    shapes = None if args.no_shapes else measure_shapes(args)
    interval = None if args.no_interval else measure_interval(args)

    cpu = kv_err = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        host_inp = synth.decode_inputs(spec, device="cpu", seq_lens=[T] * 8)
        dt, nbytes = oracle_sample(host_inp, 8, T)
        cpu = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle", "host": host_description(),
               "sample": f"8 of 16 sequences x {T} tokens (e4m3 dequantise + fp64 decode attention), "
                         f"single thread, {dt:.2f} s"}
        kv_err = {"sequences": {k: list(v) for k, v in KV_ERROR_SAMPLES.items()},
                  "note": "rel-L2 of decode attention over the stored cache against the bf16 cache (oracle, fp64)",
                  "rel_l2": fp8_kv_errors()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "us_per_layer": ms_per_step * 1e3,
            "pct_of_hbm_peak": 100.0 * value / peak, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": value / PAGE_NUMBER_GBS,
            "vs_baseline_note": "the pages' ~550 GB/s of codes for this workload, RTX 5070 Ti Triton: context only",
            "dtype": "fp32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batch": spec.batch, "q_heads": spec.q_heads,
                       "kv_heads": spec.kv_heads, "head_dim": spec.head_dim, "ctx": T,
                       "cache": args.dtype, "layout": "contiguous", "parallelism": f"replicas x{ws}",
                       "kernel": args.kernel,
                       "step": "fp8kv_decode_step: append 1 token/seq + split + merge",
            "launch": "plain" if args.plain_launch or not tensor else
                      "programmatic dependent launch: a step streams its layer's cache while the previous step finishes (FP8KV_STEP_EARLY_CACHE_READ)",
                       "l2": f"{args.layers} distinct layer caches rotated (inputs larger than L2)"},
            "roofline": roof, "cpu_baseline": cpu, "fp8_kv_error": kv_err,
            "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": (1 if tensor else 3) * args.steps,
            "kernels_us": None if per is None else {k.replace("_ms", "_us"): v * 1e3 for k, v in per.items()},
            "clocks": clocks, "controls": controls, "transform_path": transform, "plain_launch": plain,
            "l2_warm": l2_warm,
            "prefill": prefill,
            "shapes": shapes, "initiation_interval": interval,
        }
        print(json.dumps(line), flush=True)


def run_shape(args, rank):
    """Only the fused decode step on one of the other decode workloads:
    enough caches of it, rotated step by step, that they do not fit in L2
    together (one for the paged workload), `warmup` eager steps, then
    `steps` timed eager steps (CUDA events).  A small, self-contained
    command for profilers; not a bench line."""
    import fp8_quantized_kv_gb300 as fk
    spec = synth.WORKLOADS[args.shape]
    if args.group:
        spec = dataclasses.replace(spec, q_heads=args.group * spec.kv_heads)
    inp = synth.decode_inputs(spec, device="cuda")
    B, Hq, Hkv, D = spec.batch, spec.q_heads, spec.kv_heads, spec.head_dim
    lens64 = inp.seq_lens.to(torch.int64)
    sidx = torch.repeat_interleave(torch.arange(B), lens64).to(torch.int32).cuda()
    pos = torch.cat([torch.arange(int(n)) for n in lens64]).to(torch.int32).cuda()
    caches = []
    n_caches = 1
    while len(caches) < n_caches:
        if spec.page_size is None:
            cache = fk.Fp8KVCache.contiguous(B, Hkv, D, int(lens64.max()), args.dtype)
        else:
            cache = fk.Fp8KVCache.paged(inp.page_table, inp.num_pages, Hkv, D, spec.page_size, args.dtype)
        fk.fp8kv_append(cache, inp.k.contiguous(), inp.v.contiguous(), sidx, pos)
        caches.append(cache)
        if len(caches) == 1:
            nbytes = sum(t.numel() * t.element_size() for t in (cache.k, cache.v, cache.k_scale, cache.v_scale)
                         if t is not None)
            n_caches = min(8, -(-L2_BYTES * 2 // nbytes))
    last = (inp.cu_seqlens[1:] - 1).cuda()
    knew, vnew = inp.k[last].contiguous(), inp.v[last].contiguous()
    lens = inp.seq_lens.cuda()
    q = inp.q.contiguous()
    kid = KERNEL_IDS[args.kernel]
    wss = [torch.zeros(fk.fp8kv_decode_step_workspace_bytes(c, Hq, 0, kid), dtype=torch.uint8, device="cuda")
           for c in caches]
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")

    def step(i):
        j = i % len(caches)
        fk.fp8kv_decode_step(q, knew, vnew, caches[j], lens, workspace=wss[j], out=out, kernel=kid)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    spacer()
    e0.record()
    for i in range(args.steps):
        step(i)
    e1.record()
    torch.cuda.synchronize()
    if fk.fp8kv_get_device_error() != 0:
        raise RuntimeError(f"{args.shape}: device error")
    if rank == 0:
        print(json.dumps({"shape": args.shape, "group": spec.group, "cache": args.dtype, "kernel": args.kernel,
                          "us_per_step": e0.elapsed_time(e1) / args.steps * 1e3, "steps": args.steps,
                          "caches_rotated": len(caches),
                          "note": "eager launches; a profiling aid, not a bench line"}))


def run_prefill_size(args, ws, rank):
    """Only the tensor-core causal prefill at --prefill-size (tokens, batch,
    query heads, KV heads; head_dim 128; Q, K and V ~ N(0,1) as in the
    2048-token workload): `warmup` launches, then `prefill_steps` timed ones
    over rotated input sets.  A measurement aid, not a bench line."""
    n, batch, hq, hkv = (int(x) for x in args.prefill_size.split(","))
    spec = dataclasses.replace(synth.PREFILL_WORKLOADS["prefill_2048"], name=f"prefill_{n}x{batch}",
                               n_tokens=n, q_heads=hq, kv_heads=hkv)
    us, flops, n_sets = time_prefill(spec, batch, args.prefill_steps, args.warmup, ws)
    if rank == 0:
        peak, kind = tensor_peak()
        tf = flops / (us * 1e-6) / 1e12
        print(json.dumps({"prefill": spec.name, "tokens": n, "batch": batch, "q_heads": hq, "kv_heads": hkv,
                          "head_dim": spec.head_dim, "cache": "k8v8", "kernel": "prefill_tc",
                          "us_per_launch": us, "TFLOPs": tf, "frac_of_peak": tf / peak, "peak_kind": kind,
                          "launches": args.prefill_steps, "input_sets_rotated": n_sets,
                          "note": "a measurement aid, not a bench line"}))


def main():
    args = parse()
    ws, rank = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU (the FP8-KV kernels have no CPU path)")
        from fp8_quantized_kv_gb300._lib import get_lib
        get_lib()
        if args.shape:
            run_shape(args, rank)
        elif args.prefill_size:
            run_prefill_size(args, ws, rank)
        else:
            run_gpu(args, ws, rank)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
