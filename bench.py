"""Benchmark of the W4A16 group-32 MoE layer (libmoe_w4a16) on GB300.

One step = the whole layer (route, group, gate_up+SiLU, down+combine) over
one batch of synthetic inputs already resident in HBM, through the one-call
entry point moe_w4a16_moe_layer (one cooperative launch for decode batches).
Default workload: Qwen4Exp-geometry decode, 1 token (hidden 2560,
intermediate 640, 512 experts, top-10, W4A16 g32).

Timing: W untimed warm-up steps, then K timed steps issued back to back on
the launching stream, one pair of CUDA events around all K (each launch
overlaps the end of the previous step, as in a stack of layers).  Inputs
larger than L2: the layer's weights exist in NL distinct copies used in
turn (a stack of MoE layers), so every step reads its active weights from
HBM; copy i reads its own router-logit and activation set i, so the active
experts change from step to step.  Also reported: each call timed alone
(its own events after a GPU sleep, so its launch latency is inside them),
the same with L2 flushed (a 1 GiB read) before every step, which also
evicts the kernel's code, and the four step calls.

Multi-GPU: the layer has no cross-token exchange, so N GPUs run N independent
replicas (weak scaling); value = all ranks' tokens / max-over-ranks time.

--impl reference times the CPU oracle (the only other implementation there
is) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s + achieved HBM GB/s (decode 1-8 tok), W4A16 g32, 1 GB300"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen4exp_decode_T1_H2560_I640_E512_k10")
    ap.add_argument("--sets", type=int, default=32)
    ap.add_argument("--flush-mb", type=int, default=1024)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--timeline", type=int, default=0,
                    help="also run this many steps with the decode layer's phase timestamps on "
                         "and report their summary (decode batches only)")
    ap.add_argument("--sweep-paths", default="",
                    help="comma-separated batch sizes: instead of the bench line, time the step calls on "
                         "every kernel family (and the one-call layer) at each T on the Qwen4Exp and TP4-shard "
                         "geometries, one JSON line per (geometry, T)")
    ap.add_argument("--around-only", action="store_true",
                    help="print only the router and AWQ-import figures (one JSON line)")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the secondary per-workload figures")
    ap.add_argument("--layers", type=int, default=0,
                    help="weight copies used in turn (0: enough to exceed L2 twice; 1 for profiling)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            hbm = d.get("hbm_gbs") or d.get("hbm_GBps")
            if hbm:
                return float(hbm), "measured", d
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback", None


def tensor_peak():
    """Dense fp16 tensor peak in TFLOP/s: the measured bf16 cuBLAS figure
    (fp16 and bf16 run at the same tensor rate), burst (a kernel timed alone
    in a short step)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            v = d.get("bf16_tflops")
            if v:
                return float(v), "measured (MEASURED_PEAKS.json bf16_tflops, burst; fp16 = bf16 tensor rate)"
        except Exception:
            pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def layer_launches(moe, T: int, E: int, k: int, H: int, I: int) -> int:
    """Kernels the one-call layer launches for a shape, following the
    dispatch in capi.cu (moe_step_kernel_path reports the step kernels'
    family) and the kernel files:
    - decode batches that fit the one-launch layer (T <= 8): one cooperative
      kernel;
    - otherwise route and align (two launches), then
      - decode kernels: gate/up, down with the combine fused (2);
      - tensor cores: x gather + gate/up, down + combine (4);
      - stream kernels: gate/up, down (+ the combine kernel above 8 tokens)."""
    if T <= 8:
        return 1
    ra = 2
    path = moe.moe_step_kernel_path(T, E, k, H, I)
    if path == moe.MOE_PATH_DECODE:
        return ra + 2
    if path == moe.MOE_PATH_TENSOR_CORE:
        return ra + 4
    return ra + 1 + (1 if T <= 8 else 2)


def active_bytes(A: int, T: int, k: int, H: int, I: int, fmt: str = "w4a16"):
    """Algorithmic bytes of one layer step and of the gate/up launch."""
    from w4a16_group_quantized_moe_gb300 import inputs
    b = inputs.bytes_per_expert_nvfp4(H, I) if fmt == "nvfp4" else inputs.bytes_per_expert(H, I)
    P = T * k
    E_meta = 0
    gate_up = A * b["w13"] + T * H * 2 + P * I * 2
    layer = A * (b["w13"] + b["w2"]) + T * H * 2 * 2 + P * I * 2 * 2 + E_meta
    return layer, gate_up


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        # raw samples go to a scratch file; the summary goes into the JSON line
        self.path = os.path.join(tempfile.gettempdir(), f"moe_bench_clocks_gpu{device_index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
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
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
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
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "samples": len(sm), "reasons": sorted(reasons)}


def oracle_threads() -> int:
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_plan(wl):
    """(tokens per oracle step, threads).
    - Decode batches run whole layers on one thread.
    - Larger batches run a token-partitioned sample on every host core: 4
      tokens per core, one token per call. Tokens are independent, and the C
      oracle keeps no state and releases the interpreter lock while it runs."""
    if wl.shape.T <= 8:
        return wl.shape.T, 1
    n = oracle_threads()
    return 4 * n, n


def oracle_step(wl, s: int, sets: int, w13, w2, n_tok: int, pool=None):
    """One oracle step on router-logit set s.
    - The work is the whole layer when n_tok covers the batch.
    - Otherwise it is the outputs of n_tok tokens spread over the batch,
      spread over the pool's threads when a pool is given.
    - Returns (tokens, seconds spent in the oracle). Generating the inputs is
      not timed."""
    import oracle
    from w4a16_group_quantized_moe_gb300 import inputs
    sh = wl.shape
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, wl.seed + 1000 + s % sets,
                                        wl.hot_experts, wl.hot_bias)
    t0 = time.perf_counter()
    if n_tok >= sh.T:
        oracle.moe_forward(logits, x, w13, w2, sh.k)
        return sh.T, time.perf_counter() - t0
    toks = [(s * n_tok + i) * 7919 % sh.T for i in range(n_tok)]
    run = lambda t: oracle.moe_token(t, logits, x, w13, w2, sh.k)
    if pool is None:
        for t in toks:
            run(t)
    else:
        list(pool.map(run, toks))
    return n_tok, time.perf_counter() - t0


def cpu_oracle_rate(wl, seconds: float, sets: int):
    """Tokens/s of the CPU oracle on a bounded sample (oracle_plan's
    threads): oracle steps over successive router-logit sets of the workload
    until `seconds` of oracle time have been spent."""
    import concurrent.futures as cf

    import oracle
    from w4a16_group_quantized_moe_gb300 import inputs
    oracle.build()
    sh = wl.shape
    w13, w2 = inputs.make_weights(sh.E, sh.H, sh.I, wl.seed)
    n_tok, threads = oracle_plan(wl)
    tokens, el, s = 0, 0.0, 0
    with cf.ThreadPoolExecutor(threads) as pool:
        while el < seconds:
            n, dt = oracle_step(wl, s, sets, w13, w2, n_tok, pool if threads > 1 else None)
            tokens += n
            el += dt
            s += 1
    return tokens / el, tokens, el, s, threads


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms: float, device=None) -> float:
    """The slowest rank's time: every rank passes its own, every rank gets
    the maximum (identity without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, tokens_per_step: int, steps: int, max_ms: float) -> float:
    """Tokens/s of the whole job: every rank processes tokens_per_step tokens
    per step (independent replicas), timed by the slowest rank."""
    return world * tokens_per_step * steps / (max_ms / 1e3)


def copies_needed(wl, fmt: str = "w4a16") -> int:
    """Distinct weight copies a workload's steps rotate over so that every
    step reads its active weights from HBM: enough that the other copies'
    active weights stream more than twice the 126 MB L2 between two uses of
    a copy (at least 4, at most 16)."""
    from w4a16_group_quantized_moe_gb300 import inputs
    sh = wl.shape
    b = inputs.bytes_per_expert_nvfp4(sh.H, sh.I) if fmt == "nvfp4" else inputs.bytes_per_expert(sh.H, sh.I)
    per_step = min(sh.E, sh.T * sh.k) * (b["w13"] + b["w2"])
    return max(4, min(16, int(np.ceil(2 * 126e6 / max(per_step, 1))) + 1))


def bench_config(wl, world: int, sets: int) -> dict:
    """The `config` object of the JSON line: the workload, its sizes, the
    replication and how inputs are kept larger than L2 (identical in both
    arms)."""
    from w4a16_group_quantized_moe_gb300 import inputs
    sh = wl.shape
    NL = copies_needed(wl)
    b = inputs.bytes_per_expert(sh.H, sh.I)
    per_step = min(sh.E, sh.T * sh.k) * (b["w13"] + b["w2"])
    return {"workload": wl.name, "T": sh.T, "H": sh.H, "I": sh.I, "E": sh.E, "k": sh.k,
            "group_size": 32, "parallelism": f"replicas x{world}",
            "l2": f"inputs larger than L2: {NL} distinct copies of the layer's weights "
                  f"({NL * (b['w13'] + b['w2']) * sh.E / 1e9:.1f} GB) used in turn, so the {NL - 1} steps "
                  f"between two uses of a copy stream >= {(NL - 1) * per_step / 1e6:.0f} MB of other "
                  f"weights through the 126 MB L2; copy i reads router-logit and activation set i; "
                  f"the K timed steps run back to back"}


def run_reference(args, wl):
    """The CPU oracle timed on the host cores, exactly --warmup untimed and
    --steps timed steps, each a bounded sample of the workload (the whole
    layer for decode batches, sampled tokens for large ones)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import concurrent.futures as cf

    import oracle
    from w4a16_group_quantized_moe_gb300 import inputs
    oracle.build()
    sh = wl.shape
    w13, w2 = inputs.make_weights(sh.E, sh.H, sh.I, wl.seed)
    times = []
    n_tok, threads = oracle_plan(wl)
    toks = 0
    with cf.ThreadPoolExecutor(threads) as pool:
        for s in range(args.warmup + args.steps):
            n, dt = oracle_step(wl, s, args.sets, w13, w2, n_tok, pool if threads > 1 else None)
            if s >= args.warmup:
                times.append(dt)
                toks += n
    steps = len(times)
    tot = sum(times)
    value = toks / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config(wl, args.gpus, args.sets),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{steps} timed steps after {args.warmup} untimed of {wl.name} "
                                   f"(T={sh.T}), each "
                                   + ("the whole layer" if n_tok >= sh.T
                                      else f"{n_tok} sampled tokens of the layer, one per call on {threads} threads")
                                   + f"; router logits rotated over {args.sets} sets; fp64 C oracle"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))


# sources the one-launch decode layer kernel is compiled from
DECODE_LAYER_SOURCES = ("common.cuh", "decode_common.cuh", "route.cuh", "decode_layer.cuh", "decode_layer.cu")


def source_digest() -> str:
    """Digest of the decode layer kernel's sources (to tell whether stored
    ncu counters still describe the kernel that runs)."""
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_LAYER_SOURCES:
        h.update(open(os.path.join(ROOT, "w4a16_group_quantized_moe_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str):
    """DRAM bytes per launch of the layer kernel from the committed ncu
    summary, or None when it was taken on other sources or another workload."""
    p = os.path.join(ROOT, "profiles", "decode_layer_traffic.json")
    try:
        d = json.load(open(p))
    except Exception:
        return None
    e = d.get(workload)
    if not e or e.get("sources") != source_digest():
        return None
    return float(e["dram_bytes_per_launch"])


class LayerRig:
    """One workload on the GPU: NL weight copies (a stack of MoE layers, used
    in turn), `sets` router-logit/activation sets, bound layer calls, and
    per-step CUDA-event timing on the launching stream."""

    def __init__(self, moe, wl, copies, dev, sets: int, NL: int, fmt: str = "w4a16"):
        import torch
        from w4a16_group_quantized_moe_gb300 import inputs
        sh = wl.shape
        self.wl, self.sh, self.moe, self.dev, self.fmt = wl, sh, moe, dev, fmt
        self.NL = min(NL, len(copies))
        cls = moe.MoELayerNvfp4 if fmt == "nvfp4" else moe.MoELayer
        self.layers = [cls(c13, c2, sh.T, sh.k, device=dev) for c13, c2 in copies[:self.NL]]
        self.sets = []
        for si in range(sets):
            lg, xx = inputs.make_activations(sh.T, sh.H, sh.E, wl.seed + 1000 + si, wl.hot_experts, wl.hot_bias)
            self.sets.append((torch.from_numpy(lg).to(dev), torch.from_numpy(xx).to(dev)))
        self.logits_buf = torch.empty((sh.T, sh.E), dtype=torch.float32, device=dev)
        self.x_buf = torch.empty((sh.T, sh.H), dtype=torch.float16, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        # back-to-back steps: weight copy i reads its own input buffers, which
        # hold input set i (staged before the timed region)
        self.b2b_in, self.b2b_calls = [], []
        for ly in self.layers:
            lb, xb = torch.empty_like(self.logits_buf), torch.empty_like(self.x_buf)
            ly.bind(lb, xb, self.stream)
            self.b2b_in.append((lb, xb))
            self.b2b_calls.append(ly.layer_call)
        self.steps4 = [ly.bind(self.logits_buf, self.x_buf, self.stream) for ly in self.layers]
        self.calls = [ly.layer_call for ly in self.layers]
        # active experts of every set (for the algorithmic bytes)
        self.A_of = []
        for lg, xx in self.sets:
            self.logits_buf.copy_(lg)
            self.layers[0].route_align_call()
            self.A_of.append(int(self.layers[0].meta[3].item()))

    def stage(self, s):
        lg, xx = self.sets[s % len(self.sets)]
        self.logits_buf.copy_(lg, non_blocking=True)
        self.x_buf.copy_(xx, non_blocking=True)

    def one_call(self, s):
        self.calls[s % self.NL]()

    def four_calls(self, s):
        """The step calls (route, align, gate/up, down; NVFP4: route+align,
        gate/up, down)."""
        for f in self.steps4[s % self.NL]:
            f()

    def timed(self, n, first, fn, flush=None):
        """Per-step milliseconds of fn over n steps starting at step `first`."""
        import torch
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for j in range(n):
            s = first + j
            self.stage(s)
            if flush is not None:
                flush()
            else:
                # keep the GPU busy (~100 us) while the host enqueues the step, so
                # host launch gaps never fall inside the events
                torch.cuda._sleep(200000)
            ev[j][0].record(self.stream)
            fn(s)
            ev[j][1].record(self.stream)
        torch.cuda.synchronize()
        return np.array([e[0].elapsed_time(e[1]) for e in ev])

    def timed_b2b(self, n, first):
        """Milliseconds of n layer calls issued back to back (step s runs on
        weight copy s % NL with input set s % NL), one event pair around all
        of them: each launch overlaps the end of the previous step, as in a
        stack of layers."""
        import torch
        for i, (lb, xb) in enumerate(self.b2b_in):
            lg, xx = self.sets[i % len(self.sets)]
            lb.copy_(lg)
            xb.copy_(xx)
        # ~1 ms of GPU work ahead of the events: the host enqueues the calls
        # faster than the GPU runs them, so no host gap falls inside
        torch.cuda._sleep(2000000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for j in range(n):
            self.b2b_calls[(first + j) % self.NL]()
        e1.record(self.stream)
        torch.cuda.synchronize()
        return float(e0.elapsed_time(e1))

    def A_b2b(self, first, n):
        return np.array([self.A_of[((first + s) % self.NL) % len(self.sets)] for s in range(n)])

    def check_errors(self, when):
        for ly in self.layers:
            flag = self.moe.moe_get_device_error(ly.workspace)
            if flag:
                raise RuntimeError(f"device error word 0x{flag:x} {when}")

    def A_steps(self, first, n):
        return np.array([self.A_of[(first + s) % len(self.sets)] for s in range(n)])


def roofline_entry(wl, ms, A_steps, fmt: str = "w4a16"):
    """Roofline of one workload from per-step times: HBM bytes up to 128
    tokens (each active expert sees a few rows: about 9 FLOP per weight byte
    at 128 tokens on the Qwen4Exp geometry, far below the ridge of about
    280), tensor FLOPs above (the algorithmic work)."""
    sh = wl.shape
    T, H, I, k = sh.T, sh.H, sh.I, sh.k
    if T <= 128:
        lb = np.array([active_bytes(int(a), T, k, H, I, fmt)[0] for a in A_steps])
        gbs = float(lb.sum() / (ms.sum() / 1e3) / 1e9)
        peak, kind, _ = peaks()
        return {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                "peak_source": f"{kind} (MEASURED_PEAKS.json hbm_gbs)",
                "bytes_per_step": float(lb.mean())}
    flops = T * k * (2 * H * 2 * I + 2 * I * H)
    tf = flops / (ms.mean() / 1e3) / 1e12
    tpk, tsrc = tensor_peak()
    return {"bound": "tensor", "achieved": tf, "peak": tpk, "unit": "TFLOP/s", "frac": tf / tpk,
            "peak_source": tsrc, "flops_per_step": flops}


def per_config_figures(moe, dev, geoms, names, sets: int, fmt: str = "w4a16"):
    """Median/mean layer time, tokens/s and roofline fraction of each named
    workload through the one-call layer (a few seconds of GPU time each)."""
    from w4a16_group_quantized_moe_gb300 import inputs
    out = []
    for name in names:
        wl = name if isinstance(name, inputs.Workload) else inputs.ALL[name]
        name = wl.name
        copies = geoms(wl)
        big = wl.shape.T > 8
        rig = LayerRig(moe, wl, copies, dev, min(sets, 8), copies_needed(wl, fmt), fmt)
        warm, steps = (3, 30) if big else (20, 400)
        rig.timed(warm, 0, rig.one_call)
        rig.timed_b2b(warm, 0)
        rig.check_errors(f"during warm-up of {name}")
        iso = rig.timed(steps, warm, rig.one_call)
        tot = rig.timed_b2b(steps, warm)
        rig.check_errors(f"during {name}")
        ms = np.full(steps, tot / steps)
        A = rig.A_b2b(warm, steps)
        roof = roofline_entry(wl, ms, A, fmt)
        out.append({"workload": name, "steps": steps, "warmup": warm,
                    "layer_us_mean": tot / steps * 1e3,
                    "layer_us_isolated_median": float(np.median(iso) * 1e3),
                    "layer_us_isolated_mean": float(iso.mean() * 1e3),
                    "tokens_per_s": wl.shape.T * steps / (tot / 1e3),
                    "mean_active_experts": float(A.mean()),
                    "roofline": {k: roof[k] for k in ("bound", "achieved", "unit", "frac")},
                    "gpu_launches_per_step": layer_launches(moe, *(getattr(wl.shape, f) for f in "TEkHI"))})
        del rig
    return out


def launch_floor(moe, rig, T, E, k, H, I, n: int):
    """µs of the empty kernel launched with the one-call layer's launch shape
    (moe_decode_layer_floor), back to back and each alone, timed as the
    layer is; None where the shape does not take the one-launch path."""
    import ctypes
    import torch
    if T > 8 or moe.moe_decode_layer_floor(T, E, k, H, I, rig.stream, check=False) != moe.MOE_OK:
        return None
    f = moe.load_library().moe_decode_layer_floor
    sp = ctypes.c_void_p(rig.stream.cuda_stream)
    call = lambda s: f(T, E, k, H, I, sp)
    iso = rig.timed(n, 0, call)
    torch.cuda._sleep(2000000)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(rig.stream)
    for j in range(n):
        call(j)
    e1.record(rig.stream)
    torch.cuda.synchronize()
    return {"back_to_back": e0.elapsed_time(e1) / n * 1e3, "isolated_median": float(np.median(iso) * 1e3),
            "launches": 2 * n, "what": "empty kernel, the layer's grid, block, shared memory and cooperative launch"}


# grouped by weight geometry, so each geometry's weights are generated once
TIMELINE_PHASES = ("entry", "routed_and_grouped", "first_copies_issued", "first_stage_landed",
                   "gate_up_done", "down_inputs_ready", "down_done", "exit")


def phase_timeline(moe, rig, steps: int, dev):
    """Runs `steps` layer calls with the decode layer's phase timestamps on
    (global timer, 8 per CTA) and summarises them: for each phase the median
    and maximum over CTAs of its time since the earliest CTA entry, medians
    over the steps; next to the CUDA-event time of the same calls (the
    difference to the device span is the launch cost)."""
    import torch
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    tl = torch.zeros((n_sm, 8), dtype=torch.int64, device=dev)
    ly = rig.layers[0]
    moe.set_diagnostics(ly.workspace, timeline=tl)
    rows, ev_ms = [], []
    for s in range(steps):
        rig.stage(s)
        tl.zero_()
        torch.cuda._sleep(200000)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(rig.stream)
        rig.calls[0]()
        e1.record(rig.stream)
        torch.cuda.synchronize()
        ev_ms.append(e0.elapsed_time(e1))
        rows.append(tl.cpu().numpy().astype(np.float64))
    moe.set_diagnostics(ly.workspace)
    rig.check_errors("during the timeline steps")
    med, mx = {}, {}
    for i, name in enumerate(TIMELINE_PHASES):
        per_step_med, per_step_max = [], []
        for st in rows[1:] if len(rows) > 1 else rows:
            t0 = st[:, 0].min()
            v = st[:, i]
            v = v[v > 0]
            if len(v):
                per_step_med.append(np.median(v - t0) / 1e3)
                per_step_max.append(np.max(v - t0) / 1e3)
        if per_step_med:
            med[name] = float(np.median(per_step_med))
            mx[name] = float(np.median(per_step_max))
    return {"unit": "us since the first CTA entered", "steps": steps,
            "median_over_ctas": med, "max_over_ctas": mx,
            "event_us_median": float(np.median(ev_ms[1:] if len(ev_ms) > 1 else ev_ms) * 1e3)}


PER_CONFIG = ("qwen4exp_decode_T1_H2560_I640_E512_k10", "qwen4exp_decode_T2_H2560_I640_E512_k10",
              "qwen4exp_decode_T4_H2560_I640_E512_k10", "qwen4exp_decode_T8_H2560_I640_E512_k10",
              "qwen4exp_prefill_T4096_H2560_I640_E512_k10", "tp4shard_decode_T2_H2560_I160_E512_k10_hot16",
              "tp4shard_decode_T4_H2560_I160_E512_k10_hot16", "tp4shard_decode_T8_H2560_I160_E512_k10_hot16")


# batches between decode and prefill on the Qwen4Exp geometry (one-call layer)
MID_SIZES = (9, 12, 16, 24, 32, 64, 128)


def mid_size_workloads():
    from w4a16_group_quantized_moe_gb300 import inputs
    return [inputs.Workload(f"qwen4exp_mid_T{T}_H2560_I640_E512_k10", inputs.MoEShape(T, 2560, 640, 512, 10))
            for T in MID_SIZES]


# the same layer with NVFP4 weights (moe_nvfp4_moe_layer)
NVFP4_CONFIG = ("qwen4exp_decode_T1_H2560_I640_E512_k10", "qwen4exp_decode_T2_H2560_I640_E512_k10",
                "qwen4exp_decode_T4_H2560_I640_E512_k10", "qwen4exp_decode_T8_H2560_I640_E512_k10",
                "qwen4exp_prefill_T4096_H2560_I640_E512_k10")


def around_layer_figures(moe, dev):
    """The steps on either side of the layer on the Qwen4Exp geometry, timed
    with CUDA events on the launching stream (inputs larger than L2 where the
    step reads much; means over the timed launches):
    - moe_router_route_align at T = 1 and 8 (one launch: GEMV of the 2.6 MB
      router matrix, top-k and grouping) and T = 4096 (tcgen05 GEMM, then
      route and align); roofline: router-matrix bytes (HBM) for the GEMV,
      2*T*E*H FLOPs (tensor) for the GEMM;
    - moe_awq_import of a 512-expert gate layer (K 2560, N 640) into the
      gate half of W13; roofline: bytes read + written (HBM)."""
    import torch
    from w4a16_group_quantized_moe_gb300 import inputs
    E, H, I, k = 512, 2560, 640, 10
    hbm, kind, _ = peaks()
    tpk, tsrc = tensor_peak()
    stream = torch.cuda.current_stream(dev)
    out = {}
    copies = 64  # router matrices used in turn: 168 MB, more than the L2 holds
    wrs = [torch.from_numpy(inputs.make_router(E, H, seed=s)).to(dev) for s in range(copies)]
    for T in (1, 8, 4096):
        x = torch.from_numpy(inputs.make_activations(T, H, E, seed=T)[1]).to(dev)
        ws = moe.new_workspace(T, E, k, 32, 32, device=dev)  # the router uses its control block only
        bufs = moe.moe_router_route_align(x, wrs[0], k, ws)
        n = 200 if T <= 8 else 30
        for i in range(10):
            moe.moe_router_route_align(x, wrs[i % copies], k, ws, *bufs[:3], meta=bufs[3])
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
        for i in range(n):
            torch.cuda._sleep(100000)
            ev[2 * i].record(stream)
            moe.moe_router_route_align(x, wrs[i % copies], k, ws, *bufs[:3], meta=bufs[3])
            ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        if moe.moe_get_device_error(ws):
            raise RuntimeError("device error in the router")
        us = float(np.mean([ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(n)]) * 1e3)
        if T <= 16:
            b = E * H * 2 + T * H * 2 + T * E * 4
            roof = {"bound": "hbm", "achieved": b / us / 1e3, "peak": hbm, "unit": "GB/s",
                    "frac": b / us / 1e3 / hbm, "bytes": b}
        else:
            f = 2.0 * T * E * H
            roof = {"bound": "tensor", "achieved": f / us / 1e6, "peak": tpk, "unit": "TFLOP/s",
                    "frac": f / us / 1e6 / tpk, "flops": f, "peak_source": tsrc}
        out[f"router_route_align_T{T}"] = {"us": us, "launches": 1 if T <= 16 else 3, "roofline": roof}
    del wrs
    # AWQ import: two source stacks used in turn (1.9 GB together)
    K, N = H, I
    srcs = []
    for s in range(2):
        aq, az, as_ = inputs.make_awq_layer(E, K, N, seed=s)
        srcs.append((torch.from_numpy(aq.view(np.int32)).to(dev), torch.from_numpy(az.view(np.int32)).to(dev),
                     torch.from_numpy(as_).to(dev)))
    dst = (torch.zeros((E, 2 * N, K // 8), dtype=torch.int32, device=dev),
           torch.zeros((E, 2 * N, K // 32), dtype=torch.float16, device=dev),
           torch.zeros((E, 2 * N // 8, K // 32), dtype=torch.int32, device=dev))
    for i in range(3):
        moe.moe_awq_import(srcs[i % 2], dst, 0)
    n = 20
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    for i in range(n):
        ev[2 * i].record(stream)
        moe.moe_awq_import(srcs[i % 2], dst, 0)
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize()
    us = float(np.mean([ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(n)]) * 1e3)
    b = 2 * (E * K * N // 2 + E * (K // 32) * N * 2 + E * (K // 32) * (N // 8) * 4)
    out["awq_import_E512_K2560_N640"] = {"us": us, "launches": 1, "roofline": {
        "bound": "hbm", "achieved": b / us / 1e3, "peak": hbm, "unit": "GB/s", "frac": b / us / 1e3 / hbm,
        "bytes": b}}
    return out


SWEEP_GEOMS = (("qwen4exp", 2560, 640, 512, 10, (), 0.0),
               ("tp4shard", 2560, 160, 512, 10, tuple(range(16)), 2.0))


def sweep_paths(moe, dev, ts, steps: int = 200):
    """For each geometry and T: mean us per layer of the one-call layer, of
    the fused route+align call, of route then align, and of the step calls
    with every kernel family forced (None where the family cannot take the
    shape).  Weights rotate over copies as in the bench line."""
    import torch
    from w4a16_group_quantized_moe_gb300 import inputs
    rows = []
    for gname, H, I, E, k, hot, bias in SWEEP_GEOMS:
        w13, w2 = inputs.make_weights(E, H, I, 0)
        base = (moe.to_device_weights(w13, dev), moe.to_device_weights(w2, dev))
        del w13, w2
        copies = [base]
        for T in ts:
            wl = inputs.Workload(f"{gname}_T{T}", inputs.MoEShape(T, H, I, E, k), hot_experts=hot, hot_bias=bias)
            NL = copies_needed(wl)
            while len(copies) < NL:
                copies.append((tuple(t.clone() for t in base[0]), tuple(t.clone() for t in base[1])))
            rig = LayerRig(moe, wl, copies, dev, 8, NL)
            row = {"geom": gname, "T": T, "auto_path": moe.moe_step_kernel_path(T, E, k, H, I)}
            warm = 5 if T > 64 else 20
            rig.timed(warm, 0, rig.one_call)
            row["one_call_us"] = float(rig.timed(steps, warm, rig.one_call).mean() * 1e3)

            def ra(s):
                rig.layers[s % rig.NL].route_align_call()

            def r_then_a(s):
                st = rig.steps4[s % rig.NL]
                st[0]()
                st[1]()
            for name, fn in (("route_align_fused_us", ra), ("route_then_align_us", r_then_a)):
                rig.timed(warm, 0, fn)
                row[name] = float(rig.timed(steps, warm, fn).mean() * 1e3)
            for p, pname in ((moe.MOE_PATH_DECODE, "decode"), (moe.MOE_PATH_TENSOR_CORE, "tensor_core"),
                             (moe.MOE_PATH_STREAM, "stream")):
                for ly in rig.layers:
                    ly.path = p
                try:
                    rig.steps4 = [ly.bind(rig.logits_buf, rig.x_buf, rig.stream) for ly in rig.layers]
                    rig.timed(warm, 0, rig.four_calls)
                    row[pname + "_us"] = float(rig.timed(steps, warm, rig.four_calls).mean() * 1e3)
                    rig.check_errors(f"{gname} T{T} {pname}")
                except moe.MoEError as e:
                    if e.status != moe.MOE_ERR_UNSUPPORTED:
                        raise
                    row[pname + "_us"] = None
            print(json.dumps(row), flush=True)
            rows.append(row)
            del rig
        del copies, base
        torch.cuda.empty_cache()
    return rows


def main():
    args = parse()
    from w4a16_group_quantized_moe_gb300 import inputs
    wl = inputs.ALL[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
        return

    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import w4a16_group_quantized_moe_gb300 as moe
    if args.sweep_paths:
        sweep_paths(moe, dev, [int(t) for t in args.sweep_paths.split(",")])
        return
    if args.around_only:
        print(json.dumps({"around_layer": around_layer_figures(moe, dev)}))
        return

    sh = wl.shape
    T, H, I, E, k = sh.T, sh.H, sh.I, sh.E, sh.k

    # weight copies per geometry, made once and shared by every workload of
    # that geometry (the copies are a stack of MoE layers used in turn)
    geo_cache = {}

    def geoms(w, need=None, fmt="w4a16"):
        key = (w.shape.E, w.shape.H, w.shape.I, w.seed, fmt)
        n = max(copies_needed(w, fmt), need or 0)
        if key not in geo_cache:
            geo_cache.clear()
            if fmt == "nvfp4":
                w13, w2 = inputs.make_weights_nvfp4(*key[:4])
                geo_cache[key] = [(moe.to_device_weights_nvfp4(w13, dev), moe.to_device_weights_nvfp4(w2, dev))]
            else:
                w13, w2 = inputs.make_weights(*key[:4])
                geo_cache[key] = [(moe.to_device_weights(w13, dev), moe.to_device_weights(w2, dev))]
            del w13, w2
        c = geo_cache[key]
        while len(c) < n:
            c.append((tuple(t.clone() for t in c[0][0]), tuple(t.clone() for t in c[0][1])))
        return c

    NL = args.layers if args.layers > 0 else copies_needed(wl)
    rig = LayerRig(moe, wl, geoms(wl, NL), dev, args.sets, NL)
    flush = torch.zeros((args.flush_mb << 20) // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():  # a read of 1 GiB: evicts every line of L2 (data and code)
        torch.sum(flush, dim=0, out=flush_out)

    with Clocks(local) as clk:
        # the sampler runs across warm-up, the timed steps and the secondary
        # figures, so that it sees the GPU under this load for several periods
        rig.timed(min(args.warmup, 50), 0, rig.one_call)
        rig.timed(min(args.warmup, 50), 0, rig.four_calls)
        rig.timed_b2b(args.warmup, 0)
        rig.check_errors("during warm-up")
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        # the timed region: K layer calls back to back
        tot_ms_rank = rig.timed_b2b(args.steps, args.warmup)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        rig.check_errors("during timed steps")
        A_steps = rig.A_b2b(args.warmup, args.steps)
        # secondary figures: each call alone (a ~100 us GPU sleep ahead of
        # it, so its launch latency is inside its events), the four step
        # calls, and one call with L2 flushed
        n2 = max(200, min(args.steps, 2000))
        iso_ms = rig.timed(n2, args.warmup, rig.one_call)
        four_ms = rig.timed(n2, 0, rig.four_calls)
        flushed_ms = rig.timed(n2, 0, rig.one_call, flush=flush_l2)

        # end to end through the C ABI with host buffers: H2D of the step's
        # inputs from pinned memory, the layer call, D2H of the output
        h_logits = [lg.cpu().pin_memory() for lg, _ in rig.sets]
        h_x = [xx.cpu().pin_memory() for _, xx in rig.sets]
        h_out = torch.empty((T, H), dtype=torch.float16).pin_memory()
        e2e_steps = max(20, min(args.steps, 2000))
        e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(e2e_steps)]
        for s in range(e2e_steps):
            i = s % len(rig.sets)
            e2e_ev[s][0].record(rig.stream)
            rig.logits_buf.copy_(h_logits[i], non_blocking=True)
            rig.x_buf.copy_(h_x[i], non_blocking=True)
            rig.calls[s % rig.NL]()
            h_out.copy_(rig.layers[s % rig.NL].out, non_blocking=True)
            e2e_ev[s][1].record(rig.stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in e2e_ev), dev)
        e2e_val = whole_job_rate(world, T, e2e_steps, e2e_ms)
        floor = launch_floor(moe, rig, T, E, k, H, I, n2)
        timeline = None
        if args.timeline > 0 and T <= 8:
            timeline = phase_timeline(moe, rig, args.timeline, dev)
        del rig

        per_config = nvfp4 = mid = around = None
        if rank == 0 and not args.no_per_config:
            per_config = per_config_figures(moe, dev, geoms, [n for n in PER_CONFIG if n != wl.name],
                                            args.sets)
            mid = per_config_figures(moe, dev, geoms, mid_size_workloads(), args.sets)
            for m in mid:
                m["path"] = {1: "decode", 2: "tensor_core", 3: "stream"}.get(
                    moe.moe_step_kernel_path(int(m["workload"].split("_T")[1].split("_")[0]), 512, 10, 2560, 640))
            nvfp4 = per_config_figures(moe, dev, lambda w: geoms(w, fmt="nvfp4"), NVFP4_CONFIG, args.sets,
                                       fmt="nvfp4")
            geo_cache.clear()
            torch.cuda.empty_cache()
            around = around_layer_figures(moe, dev)
    geo_cache.clear()

    tot_ms = max_over_ranks(tot_ms_rank, dev)
    value = whole_job_rate(world, T, args.steps, tot_ms)
    layer_ms = np.full(args.steps, tot_ms / args.steps)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, toks, el, n, threads = cpu_oracle_rate(wl, args.cpu_seconds, args.sets)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} steps ({toks} tokens: "
                         + ("whole layers" if oracle_plan(wl)[0] >= T else "sampled tokens, one per call")
                         + f") of {wl.name} over {el:.1f} s of oracle time, fp64 C oracle on "
                         + f"{threads} thread{'s' if threads > 1 else ''}"}

    if rank == 0:
        med = lambda a: float(np.median(a) * 1e3)
        roof = roofline_entry(wl, layer_ms, A_steps)
        if T <= 8:
            roof["kernel"] = "decode_layer_kernel (moe_w4a16_moe_layer, one cooperative launch)"
            roof["traffic"] = stored_traffic(wl.name)
        else:
            roof["kernel"] = "tc_kernel (tcgen05) x2 + gather, route, align, combine (moe_w4a16_moe_layer)"
            roof["traffic"] = None
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16", "data": "synthetic",
            "config": bench_config(wl, world, args.sets),
            "mean_active_experts": float(A_steps.mean()),
            "layer_hbm_gbs": roof["achieved"] if roof["bound"] == "hbm" else None,
            "layer_us": tot_ms / args.steps * 1e3,
            "layer_us_isolated": {"median": med(iso_ms), "mean": float(iso_ms.mean() * 1e3),
                                  "p10": float(np.percentile(iso_ms, 10) * 1e3),
                                  "p90": float(np.percentile(iso_ms, 90) * 1e3), "steps": len(iso_ms)},
            "layer_us_l2_flushed_each_step": med(flushed_ms),
            "layer_us_four_step_calls": med(four_ms),
            "roofline": roof,
            "per_config": per_config,
            "nvfp4_per_config": nvfp4,
            "mid_size": mid,
            "around_layer": around,
            "timeline": timeline,
            "launch_floor_us": floor,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "tokens/s",
                    "h2d_bytes_per_step": T * E * 4 + T * H * 2,
                    "d2h_bytes_per_step": T * H * 2, "steps": e2e_steps},
            "gpu_launches": layer_launches(moe, T, E, k, H, I) * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
