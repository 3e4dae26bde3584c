#!/usr/bin/env python3
"""Throughput benchmark of the Qwen3-0.6B-shaped decoder forward on GB300.

One step = one pass of the whole forward over a synthetic request batch: the packed prefill
of every prompt (embedding, 28 decoder layers, last-row lm_head + argmax) followed by the
workload's greedy decode steps, each step's token fed back on the device.  Default workload
"decode_b1": one sequence, a 128-token prompt and 128 greedy decode steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun (N > 1) every rank runs an independent replica of the workload on its own GPU
(no collective on the data path); rank 0 prints one JSON line with the sum of tokens over the
ranks divided by the slowest rank's time.  ``--impl reference`` times the CPU oracle instead
(rank 0 only), on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode tokens/s & prefill tokens/s on 1 GB300; % of HBM / bf16 tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 2 ** 20

# DRAM bytes (read + write) per launch of the roofline kernels: medians of ncu captures
# (dram__bytes_read.sum + dram__bytes_write.sum) of each kernel as it stands, None where no
# capture of the current kernel exists.  The fused decode MLP at one row reads exactly its
# 18.9 MB of weights (launches as timed here, without the next-layer L2 prefetch of the decode
# chain); the decode gate_up GEMV at one row (k_gemv_bulk) reads exactly its 12.6 MB; the
# prefill gate_up GEMM at 23,460 rows (launches of the prefill call, the same kernel) reads A
# (48 MB) and W (12.6 MB) once and writes 86 MB of its 144 MB output before it ends (the rest
# leaves L2 later).
TRAFFIC_BYTES = {"gemv_bulk_gate_up": 12609536, "gemv_mma_gate_up": None, "gemm_gate_up": 147362304,
                 "mlp_fused": 18910976}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default="decode_b1")
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--launch", default="graph", choices=["graph", "graph-nopdl", "direct", "persistent"],
                   help="graph: decode steps as a CUDA graph of the kernel chain; direct: kernel by kernel "
                        "without PDL (for profilers); persistent: steps of up to 8 sequences as one "
                        "persistent kernel")
    p.add_argument("--decode-steps", type=int, default=None,
                   help="override the workload's decode steps (shorter runs for profilers)")
    return p.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None
        self.active = False

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == len(self.FIELDS):
                self.rows.append((self.active, parts))

    def mark(self, active: bool):
        self.active = active

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        load = [p for a, p in self.rows if a] or [p for _, p in self.rows]
        if not load:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(p[0]) for p in load if p[0].replace(".", "").isdigit()]
        mx = [float(p[1]) for p in load if p[1].replace(".", "").isdigit()]
        reasons = sorted({name for p in load for name, v in zip(self.REASONS, p[3:]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(load)}


def clocks_rejected(c) -> bool:
    """A measurement is taken again when the GPU throttled for heat or a hardware slowdown, or
    when its SM clock sat well below the maximum under load with no reason given (a clock lock
    left by someone else); a power-cap limit alone is kept (and reported)."""
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(c["reasons"]):
        return True
    if c["sm_mhz"] and c["sm_max_mhz"] and c["sm_mhz"] < 0.85 * c["sm_max_mhz"] and not c["reasons"]:
        return True
    return False


# --------------------------------------------------------------------------------------
# the workload
# --------------------------------------------------------------------------------------

def workload_desc(wl):
    s = wl.shape
    return (f"{wl.name}: {s.n_layers}-layer Qwen3-0.6B shape (hidden {s.hidden}, {s.n_q_heads}/{s.n_kv_heads} "
            f"heads, vocab {s.vocab}), {wl.n_seqs} sequence(s), prompt lengths "
            f"{wl.lengths[0] if len(set(wl.lengths)) == 1 else list(wl.lengths)}, {wl.decode_steps} greedy decode steps")


def chunk_prefills(lengths, max_tokens):
    """Consecutive groups of sequences whose packed length fits one prefill call."""
    groups, cur, tot = [], [], 0
    for i, n in enumerate(lengths):
        if cur and tot + n > max_tokens:
            groups.append(cur)
            cur, tot = [], 0
        cur.append(i)
        tot += n
    if cur:
        groups.append(cur)
    return groups


class GpuRunner:
    """Holds the model and the device buffers of one replica and runs steps of the workload."""

    def __init__(self, wl, device, flags=0):
        import torch
        from qwen3_decoder_forward_gb300 import binding, synth

        self.torch, self.binding, self.wl, self.device = torch, binding, wl, device
        s = wl.shape
        self.max_prefill = min(max(wl.lengths) if wl.n_seqs == 1 else 32768, wl.n_prompt_tokens)
        self.max_prefill = max(self.max_prefill, max(wl.lengths))
        w = synth.make_weights(s)
        self.model = binding.Model(s, w, max_seqs=wl.n_seqs, max_ctx=wl.max_ctx,
                                   max_prefill_tokens=self.max_prefill, flags=flags, device=str(device))
        del w
        prompts = wl.prompts()
        self.groups = chunk_prefills(wl.lengths, self.max_prefill)
        self.group_tokens = [torch.cat([prompts[i] for i in g]).to(device) for g in self.groups]
        self.group_tokens_host = [torch.cat([prompts[i] for i in g]).pin_memory() for g in self.groups]
        self.B = wl.n_seqs
        self.slots = list(range(self.B))
        self.slots_d = torch.tensor(self.slots, dtype=torch.int32, device=device)
        self.first = torch.zeros(self.B, dtype=torch.int32, device=device)
        self.bufs = [torch.zeros(self.B, dtype=torch.int32, device=device) for _ in range(2)]
        self.gen = torch.zeros(max(wl.decode_steps, 1), self.B, dtype=torch.int32, device=device)
        self.gen_host = torch.zeros(max(wl.decode_steps, 1), self.B, dtype=torch.int32).pin_memory()
        self.stream = torch.cuda.current_stream(device)

    def prefill_all(self, host_inputs=False):
        torch = self.torch
        h2d = 0
        for g, toks, toks_h in zip(self.groups, self.group_tokens, self.group_tokens_host):
            if host_inputs:
                toks = torch.empty_like(toks_h, device=self.device)
                toks.copy_(toks_h, non_blocking=True)
                h2d += toks_h.numel() * 4
            lengths = [self.wl.lengths[i] for i in g]
            nxt, _ = self.model.prefill(toks, lengths, [self.slots[i] for i in g])
            h2d += (len(g) + 1) * 4 + len(g) * 4  # cu_seqlens and slots
            self.first[g[0]: g[-1] + 1].copy_(nxt)
        return h2d

    def decode_all(self, record=False):
        if self.wl.decode_steps == 0:
            return
        self.bufs[0].copy_(self.first)
        for i in range(self.wl.decode_steps):
            src, dst = self.bufs[i % 2], self.bufs[(i + 1) % 2]
            self.model.decode_step(src, self.slots_d, self.slots, dst)
            if record:
                self.gen[i].copy_(dst)

    def step(self, ev=None):
        if ev is not None:
            ev[0].record(self.stream)
        self.prefill_all()
        if ev is not None:
            ev[1].record(self.stream)
        self.decode_all()
        if ev is not None:
            ev[2].record(self.stream)

    def step_e2e(self):
        """The same step from host memory: prompts copied in, generated tokens read back."""
        h2d = self.prefill_all(host_inputs=True)
        self.decode_all(record=True)
        d2h = 0
        if self.wl.decode_steps:
            self.gen_host.copy_(self.gen, non_blocking=True)
            d2h = self.gen.numel() * 4
        else:
            self.gen_host[0].copy_(self.first, non_blocking=True)
            d2h = self.B * 4
        self.stream.synchronize()
        return h2d, d2h


def units_per_step(wl):
    """(units, unit name): generated tokens for decode workloads, prompt tokens for prefill-only."""
    if wl.decode_steps:
        return wl.n_seqs * wl.decode_steps, "tokens/s"
    return wl.n_prompt_tokens, "tokens/s"


def measure_mlp_roofline(torch, binding, wl, peaks, peak_kind):
    """Average duration of the fused decode MLP kernel (RMSNorm + gate_up + SwiGLU + down +
    residual; 60% of a layer's weight bytes), the kernel decode steps of up to 4 sequences run
    for the MLP, over launches cycling through 28 layers' weights (528 MB, larger than L2),
    timed with CUDA events on the launching stream."""
    s = wl.shape
    dev = torch.device("cuda")
    M, C, I = wl.n_seqs, s.hidden, s.intermediate
    g = torch.Generator(device="cpu").manual_seed(5)
    layers = [((torch.randn(2 * I, C, generator=g) * 0.02).to(torch.bfloat16).to(dev),
               (torch.randn(I, C, generator=g) * 0.02).to(torch.bfloat16).to(dev)) for _ in range(s.n_layers)]
    h = torch.randn(M, C, generator=g).to(dev)
    gain = torch.ones(C, device=dev)
    out = torch.zeros(M, C, device=dev)
    stream = torch.cuda.current_stream().cuda_stream

    def launch(wgu, wdt):
        binding.qwen3_op_mlp_decode(h.data_ptr(), M, C, gain.data_ptr(), s.rms_eps, wgu.data_ptr(), wdt.data_ptr(),
                                    I, out.data_ptr(), stream)
    for wgu, wdt in layers:
        launch(wgu, wdt)
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        for wgu, wdt in layers:
            launch(wgu, wdt)
    e1.record()
    torch.cuda.synchronize()
    launches = reps * len(layers)
    avg_s = e0.elapsed_time(e1) / 1e3 / launches
    algo_bytes = 3 * I * C * 2 + M * C * 4 * 3  # weights; h read, out read and written
    achieved = algo_bytes / avg_s / 1e9
    peak = float(peaks["hbm_gbs"])
    return {"kernel": "k_mlp_fused (decode MLP: RMSNorm + gate_up + SwiGLU + down + residual, bf16 weights "
                      f"[{2 * I},{C}] + [{I},{C}], {M} row(s))",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": TRAFFIC_BYTES.get("mlp_fused"),
            "algorithmic_bytes_per_launch": algo_bytes, "avg_launch_us": round(avg_s * 1e6, 3),
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s"}


def measure_gemv_roofline(torch, binding, wl, peaks, peak_kind):
    """Average duration of the decode gate_up projection kernel, the largest decode kernel by
    weight bytes (40% of the layer) at 9-32 rows, over launches cycling through 28 weight
    matrices (352 MB, larger than L2), timed with CUDA events on the launching stream."""
    s = wl.shape
    dev = torch.device("cuda")
    M, K, N = wl.n_seqs, s.hidden, 2 * s.intermediate
    g = torch.Generator(device="cpu").manual_seed(5)
    ws = [(torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).to(dev) for _ in range(s.n_layers)]
    x = (torch.randn(M, K, generator=g)).to(torch.bfloat16).to(dev)
    out = torch.empty(M, N // 2, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    for wt in ws:
        binding.qwen3_op_gemv(x.data_ptr(), M, K, wt.data_ptr(), N, binding.QWEN3_EPI_SWIGLU, out.data_ptr(), stream)
    reps = 20
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        for wt in ws:
            binding.qwen3_op_gemv(x.data_ptr(), M, K, wt.data_ptr(), N, binding.QWEN3_EPI_SWIGLU, out.data_ptr(),
                                  stream)
    e1.record()
    torch.cuda.synchronize()
    launches = reps * len(ws)
    avg_s = e0.elapsed_time(e1) / 1e3 / launches
    algo_bytes = N * K * 2 + M * K * 2 + M * (N // 2) * 2
    achieved = algo_bytes / avg_s / 1e9
    peak = float(peaks["hbm_gbs"])
    kname = "k_gemv_bulk" if M <= 8 else "k_gemv_mma"
    return {"kernel": f"{kname} (decode gate_up projection + SwiGLU, bf16 weights [{N},{K}], {M} rows)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": TRAFFIC_BYTES["gemv_bulk_gate_up" if M <= 8 else "gemv_mma_gate_up"],
            "algorithmic_bytes_per_launch": algo_bytes, "avg_launch_us": round(avg_s * 1e6, 3),
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
            else "fallback 6.8 TB/s"}


def measure_gemm_roofline(torch, binding, wl, peaks, peak_kind):
    """Average duration of the prefill gate_up projection GEMM (tcgen05, SwiGLU epilogue), the
    largest prefill GEMM, at the workload's packed token count N, timed with CUDA events on the
    launching stream.  At N = 23,460 the activations and the output (48 MB + 144 MB) exceed L2;
    the 12.6 MB of weights may stay in it."""
    s = wl.shape
    dev = torch.device("cuda")
    M, K, N = wl.n_prompt_tokens, s.hidden, 2 * s.intermediate
    g = torch.Generator(device="cpu").manual_seed(6)
    x = (torch.randn(M, K, generator=g)).to(torch.bfloat16).to(dev)
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).to(dev)
    out = torch.empty(M, N // 2, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(3):
        binding.qwen3_op_gemm(x.data_ptr(), M, K, w.data_ptr(), N, binding.QWEN3_EPI_SWIGLU, out.data_ptr(), stream)
    reps = 10
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        binding.qwen3_op_gemm(x.data_ptr(), M, K, w.data_ptr(), N, binding.QWEN3_EPI_SWIGLU, out.data_ptr(), stream)
    e1.record()
    torch.cuda.synchronize()
    avg_s = e0.elapsed_time(e1) / 1e3 / reps
    flops = 2 * M * N * K
    achieved = flops / avg_s / 1e12
    peak = float(peaks["bf16_tflops"])
    return {"kernel": f"k_gemm_tcp (prefill gate_up GEMM + SwiGLU, tcgen05, [{M},{K}] x [{N},{K}]^T)",
            "bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": TRAFFIC_BYTES["gemm_gate_up"],
            "algorithmic_flops_per_launch": flops, "avg_launch_us": round(avg_s * 1e6, 3),
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops, burst: kernel timed alone)"
            if peak_kind == "measured" else "fallback 1.9 PFLOP/s"}


def prefill_flops(wl):
    """Algorithmic FLOPs of one prefill call: every linear projection for each packed token,
    causal attention (the lower triangle only, QK^T and PV) and the tied head at each
    sequence's last row."""
    s = wl.shape
    lin = 2 * wl.n_prompt_tokens * s.n_layers * ((s.q_dim + 2 * s.kv_dim) * s.hidden + s.hidden * s.q_dim +
                                                3 * s.intermediate * s.hidden)
    attn = s.n_layers * sum(4 * s.n_q_heads * s.head_dim * n * (n + 1) // 2 for n in wl.lengths)
    head = 2 * s.hidden * s.vocab * wl.n_seqs
    return lin + attn + head


# --------------------------------------------------------------------------------------
# CPU oracle timing (reference arm and the cpu_baseline object)
# --------------------------------------------------------------------------------------

def oracle_sample(wl, n_samples=1, decode_sample=8, warmup=0):
    """Times the CPU oracle on the first sequence: its prefill and `decode_sample` greedy steps,
    extrapolated to the workload's request (prefill + decode_steps) per sequence."""
    import numpy as np  # noqa: F401
    from oracle import qwen3_oracle as oracle
    from qwen3_decoder_forward_gb300 import synth

    s = wl.shape
    w = synth.make_weights(s)
    cfg = oracle.Config(s.n_layers, s.hidden, s.n_q_heads, s.n_kv_heads, s.head_dim, s.intermediate, s.vocab,
                        s.rms_eps, s.rope_theta)
    ow = oracle.Weights(w["embed"].float().numpy(), w["final_norm"].float().numpy(),
                        [{k: v.float().numpy() for k, v in d.items()} for d in w["layers"]])
    del w
    prompt = wl.prompts()[0].tolist()
    steps = decode_sample if wl.decode_steps else 0
    times = []
    for it in range(warmup + n_samples):
        cache = oracle.KVCache(cfg.n_layers)
        t0 = time.perf_counter()
        out = oracle.forward(cfg, ow, prompt, cache)
        t1 = time.perf_counter()
        tok = out["token"]
        for _ in range(steps):
            tok = oracle.forward(cfg, ow, [tok], cache)["token"]
        t2 = time.perf_counter()
        if it >= warmup:
            times.append((t1 - t0, (t2 - t1) / max(steps, 1)))
    return times


def oracle_value(wl, t_prefill, t_step):
    """Extrapolated oracle throughput in the metric's unit for the whole workload."""
    if wl.decode_steps:
        per_seq = t_prefill + wl.decode_steps * t_step  # sequences run one after another
        return wl.decode_steps / per_seq
    return len(wl.prompts()[0]) / t_prefill


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def sample_text(wl, decode_sample):
    if wl.decode_steps:
        return (f"oracle (numpy float64) on the host: prefill of sequence 0's {wl.lengths[0]}-token prompt + "
                f"{decode_sample} greedy steps, extrapolated to its {wl.decode_steps}-step request "
                f"(generated tokens / (prefill time + {wl.decode_steps} x step time))")
    return f"oracle (numpy float64) on the host: prefill of sequence 0 ({wl.lengths[0]} tokens)"


def reference_arm(args, wl):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    decode_sample = 8
    times = oracle_sample(wl, n_samples=args.steps, decode_sample=decode_sample, warmup=args.warmup)
    tp = sum(t[0] for t in times) / len(times)
    ts = sum(t[1] for t in times) / len(times)
    value = oracle_value(wl, tp, ts)
    unit = units_per_step(wl)[1]
    ms = statistics.mean((t[0] + t[1] * (decode_sample if wl.decode_steps else 0)) * 1e3 for t in times)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded random-init weights and token ids)",
            "config": {"workload": workload_desc(wl)},
            "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": cores_used(), "kind": "oracle",
                             "sample": sample_text(wl, decode_sample)},
            "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------------------

def reduce_over_ranks(torch, world, ms, units):
    """(max time, sum of units) over ranks; plain values when running alone."""
    if world == 1:
        return ms, units
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    u = torch.tensor([float(units)], dtype=torch.float64, device=t.device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def gpu_arm(args, wl):
    import torch
    from qwen3_decoder_forward_gb300 import binding, build

    rank, local_rank, world = dist_env()
    build.build()
    binding.load_library()
    torch.cuda.set_device(local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    device = torch.device("cuda", local_rank)
    peaks, peak_kind = load_peaks()
    flags = {"graph": 0, "graph-nopdl": binding.QWEN3_FLAG_NO_PDL,
             "direct": binding.QWEN3_FLAG_NO_GRAPH | binding.QWEN3_FLAG_NO_PDL,
             "persistent": binding.QWEN3_FLAG_PERSISTENT}[args.launch]
    runner = GpuRunner(wl, device, flags)
    units, unit = units_per_step(wl)

    args.warmup = max(args.warmup, 3)  # at least three untimed steps
    for _ in range(args.warmup):
        runner.step()
    torch.cuda.synchronize()

    def timed():
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
        sampler = ClockSampler(local_rank)
        sampler.start()
        time.sleep(0.3)
        n0 = binding.qwen3_launch_count(runner.model.ctx)
        barrier(world)
        torch.cuda.synchronize()
        sampler.mark(True)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for k in range(args.steps):
            runner.step(evs[k])
        end.record()
        torch.cuda.synchronize()
        sampler.mark(False)
        barrier(world)
        n1 = binding.qwen3_launch_count(runner.model.ctx)
        time.sleep(0.2)
        sampler.stop()
        ms = start.elapsed_time(end)
        pre = sum(e[0].elapsed_time(e[1]) for e in evs)
        dec = sum(e[1].elapsed_time(e[2]) for e in evs)
        return ms, pre, dec, n1 - n0, sampler.summary()

    ms, pre_ms, dec_ms, launches, clocks = timed()
    retried = False
    if clocks_rejected(clocks):
        ms, pre_ms, dec_ms, launches, clocks = timed()
        retried = True
    ms_max, units_all = reduce_over_ranks(torch, world, ms, units * args.steps)
    value = units_all / (ms_max / 1e3)

    # end to end: host buffers in, generated tokens out, every step
    for _ in range(2):
        runner.step_e2e()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    h2d = d2h = 0
    for _ in range(args.steps):
        h2d, d2h = runner.step_e2e()
    e2e_s = time.perf_counter() - t0
    e2e_s_max, e2e_units = reduce_over_ranks(torch, world, e2e_s * 1e3, units * args.steps)
    e2e_value = e2e_units / (e2e_s_max / 1e3)

    if not wl.decode_steps:
        roofline = measure_gemm_roofline(torch, binding, wl, peaks, peak_kind)
    elif wl.n_seqs <= 4 and wl.shape.hidden == 1024:
        roofline = measure_mlp_roofline(torch, binding, wl, peaks, peak_kind)
    else:
        roofline = measure_gemv_roofline(torch, binding, wl, peaks, peak_kind)
    assert runner.model.status() == 0, binding.qwen3_last_error(runner.model.ctx)
    runner.model.close()
    del runner
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        decode_sample = 8
        t = oracle_sample(wl, n_samples=1, decode_sample=decode_sample)
        cv = oracle_value(wl, t[0][0], t[0][1])
        cpu = {"value": round(cv, 4), "unit": unit, "cores": cores_used(), "kind": "oracle",
               "sample": sample_text(wl, decode_sample)}

    if rank == 0:
        s = wl.shape
        prompt_tokens = wl.n_prompt_tokens * args.steps
        gen_tokens = wl.n_seqs * wl.decode_steps * args.steps
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded random-init bf16 weights N(0,0.02), gains 1+N(0,0.05), uniform token ids)",
            "config": {"workload": workload_desc(wl),
                       "value_is": ("generated tokens per second of the whole step (prompt prefill included in "
                                    "the time)") if wl.decode_steps else "prompt tokens per second",
                       "l2": "inputs larger than L2: every decode step streams 1.19 GB of weights (L2 is 129 MB)",
                       "replicas": world, "launch": args.launch},
            "breakdown": {"prefill_ms_per_step": round(pre_ms / args.steps, 4),
                          "decode_ms_per_step": round(dec_ms / args.steps, 4),
                          "prefill_tok_s": round(prompt_tokens / (pre_ms / 1e3), 1),
                          "decode_tok_s": round(gen_tokens / (dec_ms / 1e3), 1) if gen_tokens else None},
            "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"], "reasons": clocks["reasons"],
                       "samples": clocks["samples"], "retried": retried},
            "e2e": {"value": round(e2e_value, 2), "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": int(launches),
            "roofline": roofline,
            "cpu_baseline": cpu,
        }
        if wl.decode_steps:
            step_bytes = decode_step_bytes(wl)
            dec_s = dec_ms / 1e3 / args.steps / wl.decode_steps
            line["breakdown"]["decode_step_hbm_frac"] = round(step_bytes / dec_s / 1e9 / float(peaks["hbm_gbs"]), 4)
        pre_s = pre_ms / 1e3 / args.steps
        line["breakdown"]["prefill_tflops"] = round(prefill_flops(wl) / pre_s / 1e12, 1)
        line["breakdown"]["prefill_tensor_frac"] = round(prefill_flops(wl) / pre_s / 1e12 / float(peaks["bf16_tflops"]), 4)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def decode_step_bytes(wl):
    """Algorithmic HBM bytes of one decode step of the workload: all linear weights, the tied
    head, every sequence's cached K/V rows (read) and the new rows (written)."""
    s = wl.shape
    lin = s.n_layers * ((s.q_dim + 2 * s.kv_dim) * s.hidden + s.hidden * s.q_dim + 3 * s.intermediate * s.hidden) * 2
    head = s.vocab * s.hidden * 2
    kv_tok = s.n_layers * 2 * s.kv_dim * 2
    mean_ctx = sum(n + 1 + (wl.decode_steps - 1) / 2 for n in wl.lengths) / wl.n_seqs
    return lin + head + wl.n_seqs * (mean_ctx + 1) * kv_tok


def main():
    args = parse_args()
    from qwen3_decoder_forward_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    if args.decode_steps is not None:
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name} (decode steps {args.decode_steps})",
                                 decode_steps=args.decode_steps)
    if args.impl == "reference":
        return reference_arm(args, wl)
    return gpu_arm(args, wl)


if __name__ == "__main__":
    sys.exit(main())
