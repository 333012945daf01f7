"""Benchmark of the W4A16 group-32 MoE layer (libmoe_w4a16) on GB300.

One step = the whole layer (route, group, gate_up+SiLU, down+combine) over
one batch of synthetic inputs already resident in HBM, through the one-call
entry point moe_w4a16_moe_layer (one cooperative launch for decode batches).
Default workload: Qwen4Exp-geometry decode, 1 token (hidden 2560,
intermediate 640, 512 experts, top-10, W4A16 g32).

Timing: W untimed warm-up steps, then K timed steps, each bracketed by CUDA
events on the launching stream.  Inputs larger than L2: the layer's weights
exist in NL distinct copies used in turn (a stack of MoE layers), so every
step reads its active weights from HBM; the router logits rotate over 32
pre-generated sets so the active experts change from step to step.  Also
reported: the same step with L2 flushed (a 1 GiB read) before every step,
which also evicts the kernel's code, and the four step calls.

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


def layer_launches(T: int, k: int) -> int:
    """Kernels the one-call layer launches for T tokens, following the
    dispatch in capi.cu, decode_gemv.cu and prefill_tc.cu.
    - Decode batches (T <= 8): one cooperative kernel.
    - Otherwise route+align, in one launch for T <= 32, then gate/up and
      down.
    - On the tensor-core path (T >= 9 and T*k >= 128): gate/up adds the
      sorted x gather and down adds the combine.
    - On the decode step kernels (up to 16 tokens, when their shared-memory
      layout fits; on the benchmarked geometry that happens only below 128
      pairs): one launch per step.
    - On the stream kernels: down adds the combine."""
    if T <= 8:
        return 1
    ra = 1 if T <= 32 else 2
    if T * k >= 128:
        return ra + 2 + 2
    return ra + 1 + (1 if T <= 16 else 2)


def active_bytes(A: int, T: int, k: int, H: int, I: int):
    """Algorithmic bytes of one layer step and of the gate/up launch."""
    from w4a16_group_quantized_moe_gb300 import inputs
    b = inputs.bytes_per_expert(H, I)
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


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    budget = 60.0
    import concurrent.futures as cf

    import oracle
    from w4a16_group_quantized_moe_gb300 import inputs
    oracle.build()
    sh = wl.shape
    w13, w2 = inputs.make_weights(sh.E, sh.H, sh.I, wl.seed)
    times = []
    t_start = time.perf_counter()
    n_tok, threads = oracle_plan(wl)
    toks = 0
    with cf.ThreadPoolExecutor(threads) as pool:
        for s in range(args.warmup + args.steps):
            n, dt = oracle_step(wl, s, args.sets, w13, w2, n_tok, pool if threads > 1 else None)
            if s >= min(args.warmup, 1):
                times.append(dt)
                toks += n
            if time.perf_counter() - t_start > budget and len(times) >= 3:
                break
    steps = len(times)
    tot = sum(times)
    value = toks / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": min(args.warmup, 1),
        "ms_per_step": 1e3 * tot / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name,
                   "parallelism": f"cpu, {threads} thread{'s' if threads > 1 else ''}"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"{steps} steps of {wl.name} (T={sh.T}), each "
                                   + ("the whole layer" if n_tok >= sh.T
                                      else f"{n_tok} sampled tokens of the layer, one per call on {threads} threads")
                                   + f"; router logits rotated over {args.sets} sets; run capped "
                                   f"at {budget:.0f} s of CPU time (requested {args.steps} steps after "
                                   f"{args.warmup} warm-up; the oracle needs one untimed step)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))


# sources the one-launch decode layer kernel is compiled from
DECODE_LAYER_SOURCES = ("common.cuh", "decode_common.cuh", "route.cuh", "decode_layer.cuh", "decode_layer.cu",
                        "decode_layer_spec.cu", "decode_layer_gen16.cu", "decode_layer_gen4.cu",
                        "decode_layer_gen1.cu")


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

    sh = wl.shape
    T, H, I, E, k = sh.T, sh.H, sh.I, sh.E, sh.k
    w13, w2 = inputs.make_weights(E, H, I, wl.seed)
    dw13, dw2 = moe.to_device_weights(w13, dev), moe.to_device_weights(w2, dev)
    del w13, w2
    # NL distinct copies of the layer's weights (a stack of MoE layers): step s
    # uses copy s % NL, so between two uses of a copy the other NL-1 copies'
    # active weights stream through L2 -- more than twice its 126 MB at every
    # workload here -- and each step reads its weights from HBM.
    b = inputs.bytes_per_expert(H, I)
    per_step = min(E, T * k) * (b["w13"] + b["w2"])
    NL = args.layers if args.layers > 0 else max(4, min(16, int(np.ceil(2 * 126e6 / max(per_step, 1))) + 1))
    layers = [moe.MoELayer(dw13, dw2, T, k, device=dev)]
    for _ in range(NL - 1):
        c13 = tuple(t.clone() for t in dw13)
        c2 = tuple(t.clone() for t in dw2)
        layers.append(moe.MoELayer(c13, c2, T, k, device=dev))
    sets = []
    for si in range(args.sets):
        lg, xx = inputs.make_activations(T, H, E, wl.seed + 1000 + si, wl.hot_experts, wl.hot_bias)
        sets.append((torch.from_numpy(lg).to(dev), torch.from_numpy(xx).to(dev)))
    logits_buf = torch.empty((T, E), dtype=torch.float32, device=dev)
    x_buf = torch.empty((T, H), dtype=torch.float16, device=dev)
    stream = torch.cuda.current_stream(dev)
    steps4 = [ly.bind(logits_buf, x_buf, stream) for ly in layers]
    calls = [ly.layer_call for ly in layers]
    flush = torch.zeros((args.flush_mb << 20) // 4, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2():  # a read of 1 GiB: evicts every line of L2 (data and code)
        torch.sum(flush, dim=0, out=flush_out)

    # active-expert count of every logits set (for the algorithmic bytes)
    A_of = []
    r0, a0, _, _ = steps4[0]
    for lg, xx in sets:
        logits_buf.copy_(lg)
        r0(); a0()
        A_of.append(int(layers[0].meta[3].item()))

    def stage(s):
        lg, xx = sets[s % len(sets)]
        logits_buf.copy_(lg, non_blocking=True)
        x_buf.copy_(xx, non_blocking=True)

    def timed(n, first, fn, flush_each=False):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for j in range(n):
            s = first + j
            stage(s)
            if flush_each:
                flush_l2()
            else:
                # keep the GPU busy (~100 us) while the host enqueues the step, so
                # host launch gaps never fall inside the events
                torch.cuda._sleep(200000)
            ev[j][0].record(stream)
            fn(s)
            ev[j][1].record(stream)
        torch.cuda.synchronize()
        return np.array([e[0].elapsed_time(e[1]) for e in ev])

    one_call = lambda s: calls[s % NL]()

    def four_calls(s):
        r, a_, g, d = steps4[s % NL]
        r(); a_(); g(); d()

    timed(args.warmup, 0, one_call)
    timed(min(args.warmup, 50), 0, four_calls)
    for ly in layers:
        if moe.moe_get_device_error(ly.workspace):
            raise RuntimeError("device error during warm-up")

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        layer_ms = timed(args.steps, args.warmup, one_call)
    if world > 1:
        torch.distributed.barrier()
    A_steps = np.array([A_of[(args.warmup + s) % len(sets)] for s in range(args.steps)])
    for ly in layers:
        flag = moe.moe_get_device_error(ly.workspace)
        if flag:
            raise RuntimeError(f"device error word 0x{flag:x} during timed steps")
    # secondary figures: the four step calls, and one call with L2 flushed
    n2 = min(args.steps, 2000)
    four_ms = timed(n2, 0, four_calls)
    flushed_ms = timed(n2, 0, one_call, flush_each=True)

    tot_ms = max_over_ranks(float(layer_ms.sum()), dev)
    value = whole_job_rate(world, T, args.steps, tot_ms)

    lb = np.array([active_bytes(int(a), T, k, H, I)[0] for a in A_steps])
    layer_gbs = float(lb.sum() / (layer_ms.sum() / 1e3) / 1e9)
    peak, peak_kind, _ = peaks()

    # end to end through the C ABI with host buffers: H2D of the step's
    # inputs from pinned memory, the layer call, D2H of the output
    h_logits = [lg.cpu().pin_memory() for lg, _ in sets]
    h_x = [xx.cpu().pin_memory() for _, xx in sets]
    h_out = torch.empty((T, H), dtype=torch.float16).pin_memory()
    e2e_steps = min(args.steps, 2000)
    e2e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(e2e_steps)]
    for s in range(e2e_steps):
        i = s % len(sets)
        e2e_ev[s][0].record(stream)
        logits_buf.copy_(h_logits[i], non_blocking=True)
        x_buf.copy_(h_x[i], non_blocking=True)
        calls[s % NL]()
        h_out.copy_(layers[s % NL].out, non_blocking=True)
        e2e_ev[s][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in e2e_ev), dev)
    e2e_val = whole_job_rate(world, T, e2e_steps, e2e_ms)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, toks, el, n, threads = cpu_oracle_rate(wl, args.cpu_seconds, args.sets)
        cpu = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "sample": f"{n} steps ({toks} tokens: "
                         + ("whole layers" if oracle_plan(wl)[0] >= T else "sampled tokens, one per call")
                         + f") of {wl.name} over {el:.1f} s of oracle time, fp64 C oracle on "
                         + f"{threads} thread{'s' if threads > 1 else ''}"}

    if rank == 0:
        fused = T <= 8
        med = lambda a: float(np.median(a) * 1e3)
        if fused:
            roof = {"kernel": "decode_layer_kernel (moe_w4a16_moe_layer, one cooperative launch)",
                    "bound": "hbm", "achieved": layer_gbs, "peak": peak, "unit": "GB/s",
                    "frac": layer_gbs / peak,
                    "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                    "traffic": stored_traffic(wl.name)}
        else:
            # dense contraction on the tensor cores: useful FLOPs of both GEMMs
            P = T * k
            flops = P * (2 * H * 2 * I + 2 * I * H)
            tf = flops / (np.median(layer_ms) / 1e3) / 1e12
            tpk, tsrc = tensor_peak()
            roof = {"kernel": "tc_kernel (tcgen05) x2 + gather, route, align, combine (moe_w4a16_moe_layer)",
                    "bound": "tensor", "achieved": tf, "peak": tpk, "unit": "TFLOP/s", "frac": tf / tpk,
                    "peak_source": tsrc, "flops_per_step": flops, "traffic": None}
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16", "data": "synthetic",
            "config": {"workload": wl.name, "T": T, "H": H, "I": I, "E": E, "k": k,
                       "group_size": 32, "parallelism": f"replicas x{world}",
                       "l2": f"inputs larger than L2: {NL} distinct copies of the layer's weights "
                             f"({NL * inputs.bytes_per_expert(H, I)['w13'] * E / 1e9 + NL * inputs.bytes_per_expert(H, I)['w2'] * E / 1e9:.1f} GB) "
                             f"used in turn, so the {NL - 1} steps between two uses of a copy "
                             f"stream >= {(NL - 1) * per_step / 1e6:.0f} MB of other weights through "
                             f"the 126 MB L2; router logits rotate over {args.sets} sets",
                       "mean_active_experts": float(A_steps.mean())},
            "layer_hbm_gbs": layer_gbs,
            "layer_us": {"median": med(layer_ms), "p10": float(np.percentile(layer_ms, 10) * 1e3),
                         "p90": float(np.percentile(layer_ms, 90) * 1e3)},
            "layer_us_l2_flushed_each_step": med(flushed_ms),
            "layer_us_four_step_calls": med(four_ms),
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "tokens/s",
                    "h2d_bytes_per_step": T * E * 4 + T * H * 2,
                    "d2h_bytes_per_step": T * H * 2, "steps": e2e_steps},
            "gpu_launches": layer_launches(T, k) * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
