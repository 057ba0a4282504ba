"""Throughput of one Transformer layer forward (Llama-3-8B-shaped, seq 4096) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference] [--workload NAME]

A step is one call of mt_layer_forward (all nine steps of the layer: norm, QKV GEMM + RoPE,
causal GQA flash attention, output projection + residual, norm, fc1 + SwiGLU, fc2 + residual)
on inputs already resident in HBM.  L2 is flushed (a 256 MiB write) between steps, outside the
timed spans; each step is timed with CUDA events on the launching stream (`step_ms`: their median,
10th and 90th percentile; `ms_per_step`: their mean).  `e2e` repeats the
measurement through mt_layer_forward_host with pinned host buffers (x copied in and y copied out
inside every step, in two row chunks overlapped with the layer's first and last GEMMs).  With N > 1 (torchrun) every rank runs an independent replica -- the layer
forward of one data-parallel replica needs no collective -- and the slowest rank's time counts.
`workloads` adds the GPU-only time of the other configurations (tiny, GPT-345M-shaped, one TP=8
rank of the 70B-shaped layer, the 32k-token 8B-shaped layer), timed the same way; `cpu_oracle_extras`
times the oracle on the tiny layer with one thread and on the 70B-shaped layer's eight shards.

--impl reference times the float64 CPU oracle (the "reference" arm of this build) on the host
cores: each step is a bounded sample of the same workload (K and V of every token plus the whole
layer for the last rows of the sequence), reported in the same unit.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Layer fwd TFLOP/s & MFU vs GB300 bf16 dense peak; tokens/s per layer (1 GPU)"
# --backward: the same layer's backward pass (forward recompute included in the time, not in the work)
METRIC_BWD = "Layer bwd TFLOP/s (the backward's own algorithmic work) & MFU vs GB300 bf16 dense peak (1 GPU)"
# --train-step: forward then backward (the forward's and the backward's algorithmic work)
METRIC_TRAIN = "Layer training step (fwd + bwd) TFLOP/s & MFU vs GB300 bf16 dense peak (1 GPU)"
UNIT = "TFLOP/s"
EXTRA_WORKLOADS = ("tiny", "gpt345m", "llama70b_tp8", "llama8b_32k")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def workload_desc(cfg) -> str:
    return (f"{cfg.name}: batch {cfg.batch}, seq {cfg.seq}, hidden {cfg.hidden}, {cfg.heads} heads x {cfg.head_dim}, "
            f"{cfg.groups} query groups, {'SwiGLU' if cfg.act == 'swiglu' else 'GeLU-tanh'} ffn {cfg.ffn}, "
            f"{'RMSNorm' if cfg.norm == 'rms' else 'LayerNorm'}, RoPE base {cfg.rope_base:g}, causal, "
            f"TP {cfg.tp} (one rank)")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def profiled_traffic(summary: str):
    """DRAM bytes per launch recorded in an ncu summary under profiles/, or None when the kernel
    sources it names have changed since the counters were taken."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    shas = re.search(r"source_sha256_16:(.*)", text)
    if not m or not shas:
        return None
    csrc = os.path.join(ROOT, "megatron_tensor_transformer_gpt_gb300", "csrc")
    for name, digest in re.findall(r"([\w.]+)\s+([0-9a-f]{16})", shas.group(1)):
        f = os.path.join(csrc, name)
        if not os.path.exists(f) or hashlib.sha256(open(f, "rb").read()).hexdigest()[:16] != digest:
            return None
    return int(m.group(1))


def max_over_ranks(values, dist=None, device=None):
    """Element-wise maximum of `values` over all ranks (the slowest rank's times), any backend."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(world: int, flops_per_step: float, steps: int, total_ms: float) -> float:
    """Whole-job TFLOP/s: the work of every rank divided by the slowest rank's time."""
    return world * flops_per_step * steps / (total_ms * 1e-3) / 1e12


def dense_convention_flops(cfg) -> float:
    """A forward's FLOPs with the attention counted as if unmasked (4 d S^2 per head and batch row),
    the convention of MFU figures that ignore the causal mask; the line's own count keeps the
    unmasked half only."""
    heads = cfg.heads // cfg.tp
    return cfg.gemm_flops() + 4.0 * cfg.head_dim * cfg.seq * cfg.seq * heads * cfg.batch


def step_stats(ms):
    """Median, 10th and 90th percentile (linear interpolation) of per-step times."""
    a = np.asarray(ms, dtype=np.float64)
    return [float(np.median(a)), float(np.percentile(a, 10)), float(np.percentile(a, 90))]


def sample_flops(cfg, rows) -> float:
    """Algorithmic FLOPs of the oracle's row-sampled pass: K and V of every token, then the whole
    layer for `rows` (causal attention over positions 0..s of each sampled row)."""
    T, H, d = cfg.tokens, cfg.hidden, cfg.head_dim
    qw, kvw, f = cfg.heads * d, cfg.groups * d, cfg.ffn
    f1 = 2 * f if cfg.act == "swiglu" else f
    pos = np.asarray(rows) // cfg.batch
    per_row = 2.0 * H * qw + 2.0 * qw * H + 2.0 * H * f1 + 2.0 * f * H
    attn = float(np.sum(4.0 * d * (pos + 1) * cfg.heads))
    return 2.0 * T * H * 2 * kvw + per_row * len(rows) + attn


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


def oracle_sample(cfg, inp, n_rows):
    import oracle
    rows = np.arange(cfg.tokens - n_rows, cfg.tokens)
    t0 = time.perf_counter()
    oracle.layer_forward(cfg, inp, rows=rows)
    dt = time.perf_counter() - t0
    return sample_flops(cfg, rows), dt


def rank_shapes(cfg):
    """One rank's weight shapes (rank 0 of cfg.tp), rows = output features."""
    H, d, tp = cfg.hidden, cfg.head_dim, cfg.tp
    qw, kvw, f = cfg.heads // tp * d, cfg.groups // tp * d, cfg.ffn // tp
    f1 = 2 * f if cfg.act == "swiglu" else f
    shapes = {"norm1_w": (H,), "w_qkv": (qw + 2 * kvw, H), "w_o": (H, qw), "norm2_w": (H,), "w_fc1": (f1, H),
              "w_fc2": (H, f)}
    if cfg.norm == "layer":
        shapes.update(norm1_b=(H,), norm2_b=(H,))
    if cfg.bias:
        shapes.update(b_qkv=(qw + 2 * kvw,), b_o=(H,), b_fc1=(f1,), b_fc2=(H,))
    return shapes


def device_inputs(cfg, dev, seed):
    """Seeded synthetic inputs of one rank drawn on the device, with the distributions of the seeded
    host inputs (x ~ N(0, 1), projection weights ~ N(0, 0.02), norm gains 1, shifts and biases 0),
    for workloads that are timed but not compared (drawing the 70B-shaped layer on the host would
    take longer than timing it)."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    out = {"x": torch.randn(cfg.tokens, cfg.hidden, generator=g, device=dev).to(torch.bfloat16)}
    for name, shape in rank_shapes(cfg).items():
        if name.startswith("w_"):
            out[name] = (torch.randn(shape, generator=g, device=dev) * 0.02).to(torch.bfloat16)
        else:
            fill = 1.0 if name in ("norm1_w", "norm2_w") else 0.0
            out[name] = torch.full(shape, fill, dtype=torch.bfloat16, device=dev)
    return out


def time_workload(ml, cfg, dev, steps, warmup, flush, peak_tf):
    """GPU-only time of one forward of `cfg` (one rank of cfg.tp in the identity-reduce timing mode),
    timed as the headline: CUDA events around every step, the L2 flushed between steps."""
    import torch
    tens = device_inputs(cfg, dev, seed=7)
    x = tens.pop("x")
    layer = ml.Layer.from_config(cfg, tp_rank=0)
    w = layer.weights(tens)
    y = torch.empty(cfg.tokens, cfg.hidden, dtype=torch.bfloat16, device=dev)
    layer.workspace(cfg.seq, cfg.batch, dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        layer.forward(x, cfg.seq, cfg.batch, w, y)
    torch.cuda.synchronize()
    n0 = ml.mt_layer_launch_count(layer.handle)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        layer.forward(x, cfg.seq, cfg.batch, w, y)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    layer.status()
    launches = ml.mt_layer_launch_count(layer.handle) - n0
    ms = [a.elapsed_time(b) for a, b in ev]
    layer.close()
    mean = sum(ms) / len(ms)
    tf = cfg.flops() / (mean * 1e-3) / 1e12
    return {"workload": workload_desc(cfg), "gflop_per_step": cfg.flops() / 1e9, "steps": steps,
            "ms_per_step": mean, "step_ms_median": float(np.median(ms)), "tflops": tf, "frac_of_burst": tf / peak_tf,
            "tokens_per_s": cfg.tokens / (mean * 1e-3), "gpu_launches": launches}


def cpu_oracle_extras():
    """Two more timings of the float64 oracle on the host cores: the tiny layer whole on one thread,
    and the 70B-shaped TP = 8 layer as its eight shards (K and V of every token for each shard, then
    each shard's partials for the last rows, summed)."""
    import oracle
    out = {}
    cfg = synth.CONFIGS["tiny"]
    # one thread: a child process whose BLAS is limited before NumPy loads it
    code = ("import json, time, oracle, synth\n"
            "cfg = synth.CONFIGS['tiny']\ninp = synth.make_inputs(cfg, seed=0)\n"
            "oracle.layer_forward(cfg, inp)\nt0 = time.perf_counter()\noracle.layer_forward(cfg, inp)\n"
            "print(json.dumps(time.perf_counter() - t0))\n")
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True, timeout=300)
    if r.returncode == 0:
        dt = float(r.stdout.strip().splitlines()[-1])
        out["tiny_one_thread"] = {"value": cfg.flops() / dt / 1e12, "unit": UNIT, "cores": 1, "seconds": dt,
                                  "sample": f"the whole {cfg.tokens}-token layer ({cfg.flops() / 1e9:.3f} GFLOP)"}
    cfg = synth.CONFIGS["llama70b_tp8"]
    t0 = time.perf_counter()
    inp = synth.make_inputs(cfg, seed=0)
    shards = [synth.shard_weights(cfg, inp, cfg.tp, r) for r in range(cfg.tp)]
    gen = time.perf_counter() - t0
    n_rows = 256
    rows = np.arange(cfg.tokens - n_rows, cfg.tokens)
    t0 = time.perf_counter()
    oracle.layer_forward_tp_sum(cfg, cfg.tp, inp["x"], shards, rows=rows)
    dt = time.perf_counter() - t0
    full = cfg.replace(tp=1)
    sf = sample_flops(full, rows)
    out["llama70b_tp8_eight_shards"] = {
        "value": sf / dt / 1e12, "unit": UNIT, "cores": blas_threads(), "seconds": dt,
        "sample": f"all {cfg.tp} shards: K/V of all {cfg.tokens} tokens + both blocks for the last {n_rows} rows, "
                  f"partials summed ({sf / 1e9:.1f} GFLOP algorithmic); drawing the inputs took {gen:.1f} s"}
    return out


# ------------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while a region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------ native arm
def run_native(args):
    import torch
    import torch.distributed as dist

    from megatron_tensor_transformer_gpt_gb300 import mt_layer as ml

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    cfg = synth.CONFIGS[args.workload]
    inp = synth.make_inputs(cfg, seed=rank)

    def to_dev(bits):
        return None if bits is None else torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    shards = inp if cfg.tp == 1 else synth.shard_weights(cfg, inp, cfg.tp, 0)
    tens = {k: to_dev(v) for k, v in shards.items()}
    x = tens.pop("x").reshape(cfg.tokens, cfg.hidden)
    layer = ml.Layer.from_config(cfg, tp_rank=0)
    w = layer.weights(tens)
    y = torch.empty(cfg.tokens, cfg.hidden, dtype=torch.bfloat16, device=dev)
    layer.workspace(cfg.seq, cfg.batch, dev)
    if args.fp8:
        # E4M3 weights (current scaling, outside the timed region); activation scales come from
        # the amax history the warm-up steps build (delayed scaling)
        ml.mt_layer_fp8_enable(layer.handle, 1024)
        w8 = ml.MtFp8Weights()
        keep = []
        for name in ("w_qkv", "w_o", "w_fc1", "w_fc2"):
            t = tens[name]
            codes = torch.empty(t.numel(), dtype=torch.uint8, device=dev)
            slot = torch.empty(2, dtype=torch.float32, device=dev)
            ml.mt_quantize_e4m3(t.data_ptr(), t.numel(), codes.data_ptr(), slot.data_ptr(),
                                torch.cuda.current_stream().cuda_stream)
            keep += [codes, slot]
            setattr(w8, name, codes.data_ptr())
            setattr(w8, name.replace("w_", "deq_"), slot.data_ptr() + 4)

        def fwd_fp8(xx, seq, batch, ww, yy, stream=None):
            ml.mt_layer_forward_fp8(layer.handle, xx.data_ptr(), seq, batch, ww, w8, yy.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
        layer.forward = fwd_fp8
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    flops = cfg.flops()
    if args.backward:
        # the backward's own algorithmic work: dX and dW of every projection (2x the forward GEMMs)
        # and dQ, dK, dV, dP plus the recomputed scores (2.5x the causal attention); the forward
        # recompute it also runs is not counted
        flops = 2.0 * cfg.gemm_flops() + 2.5 * cfg.attn_flops()
        if args.train_step:  # forward and backward: the forward's work plus the backward's
            flops += cfg.flops()
        rng = np.random.default_rng(rank + 100)
        dyb = torch.from_numpy(synth.f32_to_bf16_bits(rng.standard_normal((cfg.tokens, cfg.hidden), dtype=np.float32))
                               .view(np.int16)).view(torch.bfloat16).to(dev)
        dxb = torch.empty_like(dyb)
        grads = {k: (None if v is None else torch.empty_like(v)) for k, v in tens.items()}

    def step():
        if args.train_step == "saved":
            layer.forward_train(x, cfg.seq, cfg.batch, w, y)
            layer.backward_saved(x, dyb, cfg.seq, cfg.batch, w, dxb, grads)
        elif args.train_step == "recompute":
            layer.forward(x, cfg.seq, cfg.batch, w, y)
            layer.backward(x, dyb, cfg.seq, cfg.batch, w, dxb, grads)
        elif args.backward:
            layer.backward(x, dyb, cfg.seq, cfg.batch, w, dxb, grads)
        else:
            layer.forward(x, cfg.seq, cfg.batch, w, y)

    def barrier():
        if world > 1:
            dist.barrier()

    # warm-up, extended to about half a second of load so the clock samples see a busy GPU
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    layer.status()

    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    smi_index = int(vis.split(",")[local]) if vis and vis.split(",")[local].strip().isdigit() else local
    clocks = ClockSampler(smi_index)
    if not args.quick:
        clocks.start()
    t_end = time.perf_counter() + (0.0 if args.quick else 0.5)
    while time.perf_counter() < t_end:
        step()
        torch.cuda.synchronize()

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    # inside the timed steps only the roofline kernel (fc1) is bracketed by events: every event pair
    # costs a little time
    fc1_slot = ml.PROFILE_SLOTS.index("gemm_fc1")
    ml.mt_layer_profile_enable(layer.handle, 0 if args.backward else 1 << fc1_slot)
    ml.mt_layer_profile_read(layer.handle)
    torch.cuda.synchronize()
    barrier()
    launches0 = ml.mt_layer_launch_count(layer.handle)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    kernel_launches = ml.mt_layer_launch_count(layer.handle) - launches0
    prof_timed = ml.mt_layer_profile_read(layer.handle)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    # per-kernel breakdown from a separate, untimed pass with every kernel bracketed
    ml.mt_layer_profile_enable(layer.handle, True)
    for i in range(min(args.steps, 5)):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    prof = ml.mt_layer_profile_read(layer.handle)
    ml.mt_layer_profile_enable(layer.handle, False)

    # the other workloads, GPU time only (their oracle comparisons are the parity tests)
    workloads = {}
    if not (args.quick or args.fp8 or args.backward or args.no_workloads) and args.workload == "llama8b":
        for name in EXTRA_WORKLOADS:
            workloads[name] = time_workload(ml, synth.CONFIGS[name], dev, args.steps, args.warmup, flush,
                                            load_peaks()[0]["bf16_tflops"])

    # end to end through the host-buffer entry point
    xh = x.cpu().pin_memory()
    yh = torch.empty(cfg.tokens, cfg.hidden, dtype=torch.bfloat16).pin_memory()
    n_e2e = 0 if (args.quick or args.fp8 or args.backward) else args.steps
    for _ in range(min(2, n_e2e)):
        layer.forward_host(xh, cfg.seq, cfg.batch, w, yh)
    torch.cuda.synchronize()
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_e2e)]
    barrier()
    for i in range(n_e2e):
        flush.fill_(i & 0xFF)
        ev2[i][0].record(stream)
        layer.forward_host(xh, cfg.seq, cfg.batch, w, yh)
        ev2[i][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    layer.status()
    e2e_ms = [a.elapsed_time(b) for a, b in ev2]

    total_ms = sum(step_ms)
    total_e2e = sum(e2e_ms) if e2e_ms else float("nan")
    total_ms, total_e2e = max_over_ranks([total_ms, total_e2e], dist if world > 1 else None, dev)
    step_med, step_p10, step_p90 = max_over_ranks(step_stats(step_ms), dist if world > 1 else None, dev)
    value = job_throughput(world, flops, args.steps, total_ms)
    e2e_value = job_throughput(world, flops, args.steps, total_e2e)

    peaks, peak_src = load_peaks()
    peak_tf = peaks["bf16_tflops"]
    # the FP8 path is compared with the bf16 measurement times the nominal E4M3 / bf16 ratio (2)
    kernel_peak = 2.0 * peak_tf if args.fp8 else peak_tf
    launches, fc1_ms = prof_timed["gemm_fc1"]
    fc1_avg = fc1_ms / max(1, launches)
    f1 = cfg.fc1_out // cfg.tp
    fc1_flops = 2.0 * cfg.tokens * cfg.hidden * f1
    achieved = fc1_flops / (fc1_avg * 1e-3) / 1e12 if fc1_avg > 0 else None

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline and not args.quick and not args.fp8 and not args.backward:
        # about 10 s of CPU work: rows from the end of the sequence (the costliest under the causal
        # mask), doubled until the oracle runs that long or covers the whole layer
        n_rows = 256
        sf, dt = oracle_sample(cfg, inp, n_rows)
        while dt < 10.0 and n_rows < cfg.tokens:
            n_rows = min(cfg.tokens, 2 * n_rows)
            sf, dt = oracle_sample(cfg, inp, n_rows)
        cpu = {"value": sf / dt / 1e12, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
               "sample": f"float64 NumPy oracle: K/V of all {cfg.tokens} tokens + the whole layer for the last "
                         f"{n_rows} rows ({sf / 1e9:.1f} GFLOP algorithmic, {dt:.1f} s)"}

    cpu_extra = None
    if cpu is not None and args.workload == "llama8b":
        cpu_extra = cpu_oracle_extras()

    out = {
        "metric": METRIC_TRAIN if args.train_step else METRIC_BWD if args.backward else METRIC, "value": value,
        "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "step_ms": {"median": step_med, "p10": step_p10, "p90": step_p90,
                    "note": "CUDA-event time of each timed step; the slowest rank's statistic"},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 GEMMs, bf16 elsewhere" if args.fp8 else "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights)",
        "config": {"workload": workload_desc(cfg), "seq": cfg.seq, "batch": cfg.batch, "tokens": cfg.tokens,
                   "gflop_per_step": flops / 1e9, "l2": "flushed by a 256 MiB write between timed steps",
                   "parallelism": f"replicas x{world}"},
        "mfu": value / peak_tf, "mfu_vs_sustained": value / peaks["bf16_tflops_sustained"],
        "mfu_dense_convention": (None if args.backward else
                                 value * dense_convention_flops(cfg) / flops / peak_tf),
        "mfu_dense_convention_note": "attention counted as 4 d S^2 per head (causal mask ignored); "
                                     "mfu counts the unmasked half only",
        "peak_source": f"{peak_src}: bf16 {peak_tf} TF/s burst, {peaks['bf16_tflops_sustained']} sustained",
        "tokens_per_s": world * cfg.tokens * args.steps / (total_ms * 1e-3),
        "per_kernel_ms": {k: (ms / n if n else 0.0) for k, (n, ms) in prof.items()},
        "per_kernel_note": "separate untimed pass, every launch bracketed by events; the roofline kernel is "
                           "timed inside the timed steps",
        "roofline": {"kernel": "gemm_fc1 (fc1 GEMM + SwiGLU epilogue)", "bound": "tensor", "achieved": achieved,
                     "peak": kernel_peak, "unit": "TFLOP/s",
                     "frac": achieved / kernel_peak if achieved is not None else None,
                     "traffic": (profiled_traffic("gemm_fc1_swiglu_llama8b.md")
                                 if cfg.name == "llama8b" and not args.fp8 and not args.backward else None),
                     "algorithmic_bytes": 2.0 * cfg.tokens * cfg.hidden + 2.0 * f1 * cfg.hidden
                                          + 2.0 * cfg.tokens * (f1 // 2 if cfg.act == "swiglu" else f1),
                     "peak_note": (f"{peak_src} cuBLAS bf16 burst x 2 (nominal E4M3 ratio)" if args.fp8
                                   else f"{peak_src} cuBLAS bf16 burst")},
        "cpu_baseline": cpu,
        "e2e": None if n_e2e == 0 else {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": cfg.tokens * cfg.hidden * 2,
                "d2h_bytes_per_step": cfg.tokens * cfg.hidden * 2, "ms_per_step": total_e2e / args.steps},
        "gpu_launches": kernel_launches,
        "clocks": clk,
        "workloads": workloads or None,
        "workloads_note": ("the other configurations, GPU time only, timed like the headline (events, L2 flushed "
                           "between steps); seeded inputs drawn on the device; the 70B-shaped layer is one TP=8 "
                           "rank with the all-reduce replaced by the identity"),
        "cpu_oracle_extras": cpu_extra,
    }
    print(json.dumps(out))
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------ reference arm
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = synth.CONFIGS[args.workload]
    inp = synth.make_inputs(cfg, seed=0)
    n_rows = 16
    for _ in range(args.warmup):
        oracle_sample(cfg, inp, n_rows)
    fl, tt = 0.0, 0.0
    for _ in range(args.steps):
        f, dt = oracle_sample(cfg, inp, n_rows)
        fl += f
        tt += dt
    value = fl / tt / 1e12
    sample = (f"float64 NumPy oracle per step: K/V of all {cfg.tokens} tokens + the whole layer for the last "
              f"{n_rows} rows ({fl / args.steps / 1e9:.1f} GFLOP algorithmic)")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": tt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": workload_desc(cfg), "seq": cfg.seq, "batch": cfg.batch,
                      "parallelism": "host cores"},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--workload", default="llama8b", choices=sorted(synth.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the GPU-only timings of the other configurations")
    ap.add_argument("--backward", action="store_true",
                    help="time mt_layer_backward (forward recompute + gradients) instead of the forward")
    ap.add_argument("--train-step", choices=("recompute", "saved"), default=None,
                    help="time a training step: mt_layer_forward + mt_layer_backward (recompute) or "
                         "mt_layer_forward_train + mt_layer_backward_saved (saved)")
    ap.add_argument("--fp8", action="store_true",
                    help="time the FP8 (E4M3) forward instead of the bf16 one (no host-buffer pass, no CPU baseline)")
    ap.add_argument("--quick", action="store_true",
                    help="profiling runs: no clock sampling, no host-buffer pass, no CPU baseline")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.train_step:
        args.backward = True  # the backward's buffers and its options (no host-buffer pass, no CPU baseline)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
