#!/usr/bin/env python3
"""Throughput benchmark of the Qwen3-0.6B-shaped decoder forward on GB300.

Default workload "decode_long": 16 sequences whose 16,384-token prompts fill the KV cache
(about 30 GB), then 32 greedy decode steps of all 16 at once.  One timed step is those 32
decode steps, each step's tokens fed back on the device; before each step the slots are
rewound to their prompts (qwen3_truncate_slot), so every step decodes at the same contexts
16,384..16,415 and rewrites the same cache rows.  The prompts' prefill (the KV fill) is timed
once and reported beside it.  The same line carries the ragged prefill workload
("prefill_ragged": 8 prompts of 512..4096 tokens packed into one call), timed on its own, as
its "prefill" object.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A prefill-only workload (prefill_ragged, or --workload tiny / decode_* with --decode-steps 0)
times one packed prefill call per step.  Under torchrun (N > 1) every rank runs an
independent replica of the workload on its own GPU (no collective on the data path); rank 0
prints one JSON line with the units of all ranks over the slowest rank's time.
``--impl reference`` times the CPU oracle instead (rank 0 only), on a bounded sample of the
same workload.
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

# DRAM bytes (read + write) per launch of the roofline kernels, from ncu captures
# (dram__bytes_read.sum + dram__bytes_write.sum) of each kernel as it stands; a kernel without
# an entry reports traffic null.  The fused decode MLP at one row reads exactly its 18.9 MB of
# weights; the prefill gate_up GEMM at 23,460 rows reads A (48 MB) and W (12.6 MB) once and
# writes 86 MB of its 144 MB output before it ends (the rest leaves L2 later).  The decode
# attention entries are DRAM bytes per (sequence, position) row of one layer's K and V, scaled
# by the rows a launch reads (the traffic grows in proportion with the rows).  The decode gate_up
# projections at 16 and 32 rows read their 12.6 MB of weights once and write nothing to DRAM
# before they end.
TRAFFIC_BYTES = {"gemm_gate_up": 146836992, "mlp_fused": 18910976, "attn_decode_per_key_row": 4110.9,
                 "gemv_gate_up_16": 12630912, "gemv_gate_up_32": 12664704}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--workload", default="decode_long")
    p.add_argument("--prefill-workload", default="prefill_ragged",
                   help="workload of the line's 'prefill' object when the main workload decodes ('none': skip)")
    p.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--launch", default="graph", choices=["graph", "graph-nopdl", "direct", "chain"],
                   help="graph: decode steps as CUDA graphs with programmatic dependent launch; direct: kernel "
                        "by kernel without it (for profilers); chain: one-row steps as the four-kernel chain")
    p.add_argument("--decode-steps", type=int, default=None,
                   help="override the workload's decode steps (shorter runs for profilers)")
    p.add_argument("--roofline-only", action="store_true",
                   help="run only the roofline kernel's timing of the workload (for ncu captures)")
    p.add_argument("--roofline-ctx", type=int, default=None,
                   help="context of the decode attention roofline launch (default: the workload's)")
    p.add_argument("--roofline-kernel", default="auto", choices=["auto", "proj"],
                   help="with --roofline-only: proj times the decode gate_up projection instead")
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
# the workload and its algorithmic work
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


def decode_step_bytes(wl):
    """Algorithmic HBM bytes of one decode step of the workload: all linear weights, the tied
    head, every sequence's cached K/V rows (read) and the new rows (written)."""
    s = wl.shape
    lin = s.n_layers * ((s.q_dim + 2 * s.kv_dim) * s.hidden + s.hidden * s.q_dim + 3 * s.intermediate * s.hidden) * 2
    head = s.vocab * s.hidden * 2
    kv_tok = s.n_layers * 2 * s.kv_dim * 2
    mean_ctx = sum(n + 1 + (wl.decode_steps - 1) / 2 for n in wl.lengths) / wl.n_seqs
    return lin + head + wl.n_seqs * (mean_ctx + 1) * kv_tok


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


def decode_positions(wl):
    """Position of each sequence's query in the middle decode step of the workload."""
    return [n + wl.decode_steps // 2 for n in wl.lengths]


# --------------------------------------------------------------------------------------
# GPU runner
# --------------------------------------------------------------------------------------

class DeviceRunner:
    """Holds the model and the device buffers of one replica and runs steps of the workload."""

    def __init__(self, wl, device, flags=0, weights=None, kv_block_tokens=0):
        import torch
        from qwen3_decoder_forward_gb300 import binding, synth

        self.torch, self.binding, self.wl, self.device = torch, binding, wl, device
        s = wl.shape
        self.max_prefill = min(max(wl.lengths) if wl.n_seqs == 1 else 32768, wl.n_prompt_tokens)
        self.max_prefill = max(self.max_prefill, max(wl.lengths))
        w = weights if weights is not None else synth.make_weights(s)
        pool = 0
        if kv_block_tokens:  # a pool holding every slot at the workload's longest context
            pool = wl.n_seqs * ((wl.max_ctx + kv_block_tokens - 1) // kv_block_tokens)
        self.model = binding.Model(s, w, max_seqs=wl.n_seqs, max_ctx=wl.max_ctx,
                                   max_prefill_tokens=self.max_prefill, flags=flags, device=str(device),
                                   kv_block_tokens=kv_block_tokens, kv_pool_blocks=pool)
        del w
        prompts = wl.prompts()
        self.groups = chunk_prefills(wl.lengths, self.max_prefill)
        self.group_tokens = [torch.cat([prompts[i] for i in g]).to(device) for g in self.groups]
        self.group_tokens_host = [torch.cat([prompts[i] for i in g]).pin_memory() for g in self.groups]
        self.B = wl.n_seqs
        self.slots = list(range(self.B))
        self.slots_d = torch.tensor(self.slots, dtype=torch.int32, device=device)
        self.first = torch.zeros(self.B, dtype=torch.int32, device=device)
        self.first_host = torch.zeros(self.B, dtype=torch.int32).pin_memory()
        self.bufs = [torch.zeros(self.B, dtype=torch.int32, device=device) for _ in range(2)]
        self.gen = torch.zeros(max(wl.decode_steps, 1), self.B, dtype=torch.int32, device=device)
        self.gen_host = torch.zeros(max(wl.decode_steps, 1), self.B, dtype=torch.int32).pin_memory()
        self.stream = torch.cuda.current_stream(device)

    def prefill_all(self, host_inputs=False):
        """Every prompt, in packed groups; returns the host->device bytes it copied."""
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
        """Rewinds every slot to its prompt, then runs the workload's decode steps from the
        prefill's next tokens, each step's output fed to the next on the device."""
        for i, n in enumerate(self.wl.lengths):
            self.model.truncate(self.slots[i], n)
        self.bufs[0].copy_(self.first)
        for i in range(self.wl.decode_steps):
            src, dst = self.bufs[i % 2], self.bufs[(i + 1) % 2]
            self.model.decode_step(src, self.slots_d, self.slots, dst)
            if record:
                self.gen[i].copy_(dst)

    def step(self):
        if self.wl.decode_steps:
            self.decode_all()
        else:
            self.prefill_all()

    def step_e2e(self):
        """The same step through host memory: its inputs copied in from pinned host buffers
        (the prompts, or the first tokens of the decode steps), its tokens read back."""
        if self.wl.decode_steps:
            self.first.copy_(self.first_host, non_blocking=True)
            h2d = self.B * 4
            self.decode_all(record=True)
            self.gen_host.copy_(self.gen, non_blocking=True)
            d2h = self.gen.numel() * 4
        else:
            h2d = self.prefill_all(host_inputs=True)
            self.first_host.copy_(self.first, non_blocking=True)
            d2h = self.B * 4
        self.stream.synchronize()
        return h2d, d2h


def units_per_step(wl):
    """(units, unit name): generated tokens for decode workloads, prompt tokens for prefill-only."""
    if wl.decode_steps:
        return wl.n_seqs * wl.decode_steps, "tokens/s"
    return wl.n_prompt_tokens, "tokens/s"


def timed_steps(torch, binding, runner, steps, local_rank, world):
    """`steps` steps between CUDA events on the launching stream (barrier + synchronize on both
    sides), clocks sampled meanwhile; retaken once if the clocks were throttled or locked."""
    def once():
        sampler = ClockSampler(local_rank)
        sampler.start()
        time.sleep(0.3)
        n0 = binding.qwen3_launch_count(runner.model.ctx)
        barrier(world)
        torch.cuda.synchronize()
        sampler.mark(True)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(runner.stream)
        for _ in range(steps):
            runner.step()
        end.record(runner.stream)
        torch.cuda.synchronize()
        sampler.mark(False)
        barrier(world)
        n1 = binding.qwen3_launch_count(runner.model.ctx)
        time.sleep(0.2)
        sampler.stop()
        return start.elapsed_time(end), n1 - n0, sampler.summary()

    ms, launches, clocks = once()
    retried = False
    if clocks_rejected(clocks):
        ms, launches, clocks = once()
        retried = True
    clocks = dict(clocks, retried=retried)
    return ms, launches, clocks


def e2e_steps(torch, runner, steps, world):
    for _ in range(2):
        runner.step_e2e()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    h2d = d2h = 0
    for _ in range(steps):
        h2d, d2h = runner.step_e2e()
    return (time.perf_counter() - t0) * 1e3, h2d, d2h


# --------------------------------------------------------------------------------------
# roofline kernels, each timed alone with CUDA events on its launching stream
# --------------------------------------------------------------------------------------

def _peak_source(peak_kind, key, note=""):
    if peak_kind == "measured":
        return f"measured (MEASURED_PEAKS.json {key}{note})"
    return "fallback " + ("6.8 TB/s" if key == "hbm_gbs" else "1.9 PFLOP/s")


def _time_launches(torch, launch, reps):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        launch()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / reps


def measure_mlp_roofline(torch, binding, wl, peaks, peak_kind):
    """Average duration of the fused decode MLP kernel (RMSNorm + gate_up + SwiGLU + down +
    residual; 60% of a layer's weight bytes), the kernel decode steps of up to 4 sequences run
    for the MLP, over launches cycling through 28 layers' weights (528 MB, larger than L2)."""
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
    it = [0]

    def launch():
        wgu, wdt = layers[it[0] % len(layers)]
        it[0] += 1
        binding.qwen3_op_mlp_decode(h.data_ptr(), M, C, gain.data_ptr(), s.rms_eps, wgu.data_ptr(), wdt.data_ptr(),
                                    I, out.data_ptr(), stream)
    for _ in range(len(layers)):
        launch()
    avg_s = _time_launches(torch, launch, 20 * len(layers))
    algo_bytes = 3 * I * C * 2 + M * C * 4 * 3  # weights; h read, out read and written
    achieved = algo_bytes / avg_s / 1e9
    peak = float(peaks["hbm_gbs"])
    return {"kernel": "k_mlp_fused (decode MLP: RMSNorm + gate_up + SwiGLU + down + residual, bf16 weights "
                      f"[{2 * I},{C}] + [{I},{C}], {M} row(s))",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": TRAFFIC_BYTES.get("mlp_fused"),
            "algorithmic_bytes_per_launch": algo_bytes, "avg_launch_us": round(avg_s * 1e6, 3),
            "peak_source": _peak_source(peak_kind, "hbm_gbs")}


def measure_proj_roofline(torch, binding, wl, peaks, peak_kind):
    """Average duration of the decode gate_up projection (+ SwiGLU; 40% of a layer's weight
    bytes) at the workload's batch, through qwen3_op_gemv (the tensor-core GEMV from 9 rows),
    over launches cycling through 28 layers' weights (352 MB, larger than L2)."""
    s = wl.shape
    dev = torch.device("cuda")
    M, C, I = wl.n_seqs, s.hidden, s.intermediate
    g = torch.Generator(device="cpu").manual_seed(6)
    layers = [(torch.randn(2 * I, C, generator=g) * 0.02).to(torch.bfloat16).to(dev) for _ in range(s.n_layers)]
    x = torch.randn(M, C, generator=g).to(torch.bfloat16).to(dev)
    out = torch.zeros(M, I, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream().cuda_stream
    it = [0]

    def launch():
        w = layers[it[0] % len(layers)]
        it[0] += 1
        binding.qwen3_op_gemv(x.data_ptr(), M, C, w.data_ptr(), 2 * I, binding.QWEN3_EPI_SWIGLU, out.data_ptr(), stream)
    for _ in range(len(layers)):
        launch()
    avg_s = _time_launches(torch, launch, 20 * len(layers))
    algo_bytes = 2 * I * C * 2 + M * C * 2 + M * I * 2  # weights; x read, act written
    achieved = algo_bytes / avg_s / 1e9
    peak = float(peaks["hbm_gbs"])
    kern = "k_gemv_mma (tensor cores)" if M > 8 else "k_gemv_bulk"
    return {"kernel": f"{kern} (decode gate_up + SwiGLU, bf16 weights [{2 * I},{C}], {M} row(s))",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": TRAFFIC_BYTES.get(f"gemv_gate_up_{M}"),
            "algorithmic_bytes_per_launch": algo_bytes, "avg_launch_us": round(avg_s * 1e6, 3),
            "peak_source": _peak_source(peak_kind, "hbm_gbs")}


def measure_attn_roofline(torch, binding, wl, peaks, peak_kind, ctx=None, reps=20):
    """Average duration of the decode attention kernel (QK-norm + RoPE + KV write + attention
    over keys 0..p), the kernel that streams the KV cache, as a decode step of the workload
    plans it (qwen3_op_attn_decode_plan: key ranges per (sequence, KV head)), at
    the workload's batch and the positions of its middle decode step (or every row at position
    ctx - 1), over one layer's K/V rows of the workload's size in their own buffer (larger than
    L2 for the long contexts), through qwen3_op_attn_decode."""
    import math
    s = wl.shape
    dev = torch.device("cuda")
    B, Hq, Hkv, D = wl.n_seqs, s.n_q_heads, s.n_kv_heads, s.head_dim
    positions = decode_positions(wl) if ctx is None else [ctx - 1] * B
    max_ctx = max(positions) + 1
    g = torch.Generator(device=dev).manual_seed(7)
    kc = torch.randn((B, Hkv, max_ctx, D), generator=g, device=dev).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, max_ctx, D), generator=g, device=dev).to(torch.bfloat16)
    qkv = torch.randn((B, (Hq + 2 * Hkv) * D), generator=g, device=dev)
    gain = torch.ones(D, device=dev)
    inv = [s.rope_theta ** (-2.0 * i / D) for i in range(D // 2)]
    rope = torch.tensor([[[math.cos(p * f), math.sin(p * f)] for f in inv] for p in sorted(set(positions))],
                        dtype=torch.float32)
    rope_full = torch.zeros((max_ctx, D // 2, 2), dtype=torch.float32)
    for i, p in enumerate(sorted(set(positions))):
        rope_full[p] = rope[i]  # only the rows of the positions used are read
    rope_d = rope_full.to(dev)
    slots = list(range(B))
    slots_d = torch.tensor(slots, dtype=torch.int32, device=dev)
    pos_d = torch.tensor(positions, dtype=torch.int32, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    ws_bytes = binding.qwen3_op_attn_decode_workspace_bytes(B, Hq, Hkv)
    ws = torch.zeros(ws_bytes + 256, dtype=torch.uint8, device=dev)
    ws_ptr = (ws.data_ptr() + 255) // 256 * 256
    stream = torch.cuda.current_stream().cuda_stream
    n_split = binding.qwen3_op_attn_decode_plan(B, Hq, Hkv, max_ctx, max(max_ctx, wl.max_ctx))

    def launch():
        binding.qwen3_op_attn_decode(qkv.data_ptr(), B, slots_d.data_ptr(), slots, pos_d.data_ptr(), positions,
                                     gain.data_ptr(), gain.data_ptr(), rope_d.data_ptr(), kc.data_ptr(),
                                     vc.data_ptr(), B, max_ctx, Hq, Hkv, s.rms_eps, n_split, out.data_ptr(), ws_ptr,
                                     ws_bytes, stream)
    for _ in range(3):
        launch()
    avg_s = _time_launches(torch, launch, reps)
    rows = sum(p + 1 for p in positions)
    algo_bytes = rows * Hkv * D * 2 * 2  # K and V rows 0..p of every (sequence, KV head), the new one written
    achieved = algo_bytes / avg_s / 1e9
    peak = float(peaks["hbm_gbs"])
    per_row = TRAFFIC_BYTES.get("attn_decode_per_key_row")
    del kc, vc
    name = f"k_attn_decode_fused ({n_split} key range{'s' if n_split > 1 else ''} per pair, tensor cores"
    return {"kernel": f"{name}; QK-norm + RoPE + KV write + attention, {B} rows at "
                      f"positions {min(positions)}..{max(positions)}, {Hq}/{Hkv} heads, one layer)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": round(per_row * rows) if per_row else None,
            "algorithmic_bytes_per_launch": algo_bytes, "avg_launch_us": round(avg_s * 1e6, 3),
            "peak_source": _peak_source(peak_kind, "hbm_gbs")}


def measure_gemm_roofline(torch, binding, wl, peaks, peak_kind):
    """Average duration of the prefill gate_up projection GEMM (tcgen05, SwiGLU epilogue), the
    largest prefill GEMM, at the workload's packed token count N.  At N = 23,460 the activations
    and the output (48 MB + 144 MB) exceed L2; the 12.6 MB of weights may stay in it."""
    s = wl.shape
    dev = torch.device("cuda")
    M, K, N = wl.n_prompt_tokens, s.hidden, 2 * s.intermediate
    g = torch.Generator(device="cpu").manual_seed(6)
    x = (torch.randn(M, K, generator=g)).to(torch.bfloat16).to(dev)
    w = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16).to(dev)
    out = torch.empty(M, N // 2, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream().cuda_stream

    def launch():
        binding.qwen3_op_gemm(x.data_ptr(), M, K, w.data_ptr(), N, binding.QWEN3_EPI_SWIGLU, out.data_ptr(), stream)
    for _ in range(3):
        launch()
    avg_s = _time_launches(torch, launch, 10)
    flops = 2 * M * N * K
    achieved = flops / avg_s / 1e12
    peak = float(peaks["bf16_tflops"])
    return {"kernel": f"k_gemm_tcp (prefill gate_up GEMM + SwiGLU, tcgen05, [{M},{K}] x [{N},{K}]^T)",
            "bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": TRAFFIC_BYTES["gemm_gate_up"],
            "algorithmic_flops_per_launch": flops, "avg_launch_us": round(avg_s * 1e6, 3),
            "peak_source": _peak_source(peak_kind, "bf16_tflops", ", burst: kernel timed alone")}


def roofline_for(torch, binding, wl, peaks, peak_kind, ctx=None):
    """The roofline object of the workload's dominant kernel: the gate_up GEMM for prefill, the
    fused MLP (the most weight bytes) for decode of up to 4 rows, the KV-streaming attention
    for larger decode batches."""
    if not wl.decode_steps:
        return measure_gemm_roofline(torch, binding, wl, peaks, peak_kind)
    if wl.n_seqs <= 4 and wl.shape.hidden == 1024 and ctx is None:
        return measure_mlp_roofline(torch, binding, wl, peaks, peak_kind)
    return measure_attn_roofline(torch, binding, wl, peaks, peak_kind, ctx=ctx)


# --------------------------------------------------------------------------------------
# CPU oracle timing (reference arm and the cpu_baseline objects)
# --------------------------------------------------------------------------------------

ORACLE_PREFILL_SAMPLE = 256   # prompt tokens of one oracle prefill sample
ORACLE_DECODE_STEPS_SHORT = 8  # decode steps of the cpu_baseline sample below 8K of context
ORACLE_DECODE_STEPS_LONG = 3   # ... at 8K of context and more


def _oracle_model(wl):
    from oracle import qwen3_oracle as oracle
    from qwen3_decoder_forward_gb300 import synth

    s = wl.shape
    w = synth.make_weights(s)
    cfg = oracle.Config(s.n_layers, s.hidden, s.n_q_heads, s.n_kv_heads, s.head_dim, s.intermediate, s.vocab,
                        s.rms_eps, s.rope_theta)
    ow = oracle.Weights(w["embed"].float().numpy(), w["final_norm"].float().numpy(),
                        [{k: v.float().numpy() for k, v in d.items()} for d in w["layers"]])
    return oracle, cfg, ow


class OracleSample:
    """Bounded samples of the workload on the CPU oracle, as it stands.

    Decode workloads: greedy decode steps of sequence 0 continuing one cache that starts at
    its prompt's length (rows drawn at random: the oracle's step does the same work whatever
    the cached values), `capacity` steps in all.  The oracle runs sequences one after
    another, so its tokens/s for B sequences equals one sequence's.  Prefill workloads: the
    oracle's prefill of the first ORACLE_PREFILL_SAMPLE tokens of sequence 0."""

    def __init__(self, wl, capacity=0):
        import numpy as np
        self.wl = wl
        self.oracle, self.cfg, self.ow = _oracle_model(wl)
        s = wl.shape
        self.prompt = wl.prompts()[0].tolist()
        self.done = 0
        if wl.decode_steps:
            rng = np.random.default_rng(11)
            n = wl.lengths[0]
            k = rng.standard_normal((n, s.n_kv_heads, s.head_dim))
            v = rng.standard_normal((n, s.n_kv_heads, s.head_dim))
            self.cache = self.oracle.KVCache.from_arrays([k] * s.n_layers, [v] * s.n_layers, spare=capacity)
            self.tok = self.prompt[-1]

    def run(self, steps=1):
        """Seconds per unit (one generated token, or one prompt token) over one sample."""
        o = self.oracle
        if self.wl.decode_steps:
            t0 = time.perf_counter()
            for _ in range(steps):
                self.tok = o.forward(self.cfg, self.ow, [self.tok], self.cache)["token"]
            self.done += steps
            return (time.perf_counter() - t0) / steps
        ids = self.prompt[:ORACLE_PREFILL_SAMPLE]
        t0 = time.perf_counter()
        o.forward(self.cfg, self.ow, ids, o.KVCache(self.cfg.n_layers))
        return (time.perf_counter() - t0) / len(ids)

    def describe(self, steps):
        if self.wl.decode_steps:
            n = self.wl.lengths[0]
            return (f"oracle (numpy float64) on the host: greedy decode steps of one sequence at contexts from "
                    f"{n + 1} ({steps} per sample), continuing a {n}-row cache of seeded random rows; the "
                    f"oracle runs sequences one after another, so its tokens/s for {self.wl.n_seqs} sequences "
                    f"is one sequence's")
        n = min(ORACLE_PREFILL_SAMPLE, self.wl.lengths[0])
        return f"oracle (numpy float64) on the host: prefill of the first {n} tokens of sequence 0"


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(wl, unit):
    steps = (ORACLE_DECODE_STEPS_LONG if max(wl.lengths) >= 8192 else ORACLE_DECODE_STEPS_SHORT) \
        if wl.decode_steps else 1
    smp = OracleSample(wl, capacity=steps)
    t = smp.run(steps)
    return {"value": round(1.0 / t, 4), "unit": unit, "cores": cores_used(), "kind": "oracle",
            "sample": smp.describe(steps)}


def reference_arm(args, wl):
    """The oracle timed as the reference: each of the warm-up and timed steps is one sample
    (one decode step of one sequence, or one ORACLE_PREFILL_SAMPLE-token prefill)."""
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    unit = units_per_step(wl)[1]
    steps = max(args.steps, 1)
    smp = OracleSample(wl, capacity=args.warmup + steps)
    for _ in range(args.warmup):
        smp.run()
    per_unit = [smp.run() for _ in range(steps)]
    t = sum(per_unit) / len(per_unit)
    value = 1.0 / t
    units = 1 if wl.decode_steps else min(ORACLE_PREFILL_SAMPLE, wl.lengths[0])
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t * units * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded random-init weights and token ids)",
            "config": {"workload": workload_desc(wl)},
            "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": cores_used(), "kind": "oracle",
                             "sample": smp.describe(1) + "; each step is one sample"},
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


def prefill_once_timed(torch, runner):
    """One pass of every prompt's prefill between CUDA events (the KV fill of a decode
    workload); milliseconds."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(runner.stream)
    runner.prefill_all()
    e1.record(runner.stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def step_roofline(wl, step_s, peaks, peak_kind, what):
    """The whole step against its roofline: decode steps' HBM bytes, or a prefill's flops."""
    if wl.decode_steps:
        achieved = decode_step_bytes(wl) / (step_s / wl.decode_steps) / 1e9
        peak = float(peaks["hbm_gbs"])
        return {"kernel": f"whole decode step ({what})", "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                "algorithmic_bytes_per_step": int(decode_step_bytes(wl)),
                "peak_source": _peak_source(peak_kind, "hbm_gbs")}
    achieved = prefill_flops(wl) / step_s / 1e12
    peak = float(peaks["bf16_tflops"])
    return {"kernel": f"whole prefill ({what})", "bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
            "algorithmic_flops_per_step": int(prefill_flops(wl)), "peak_source": _peak_source(peak_kind, "bf16_tflops")}


def run_workload(args, wl, device, flags, peaks, peak_kind, world, local_rank, weights=None, cpu=True,
                 kv_block_tokens=0):
    """Runs one workload: warm-up, the timed steps, the end-to-end steps, the roofline kernel
    and (rank 0, one GPU) the CPU oracle sample.  Returns the fields of its JSON object."""
    import torch
    from qwen3_decoder_forward_gb300 import binding

    runner = DeviceRunner(wl, device, flags, weights, kv_block_tokens)
    units, unit = units_per_step(wl)
    out = {}
    if wl.decode_steps:
        runner.prefill_all()  # first pass: graphs and lazily loaded kernels
        fill_ms = prefill_once_timed(torch, runner)
        runner.first_host.copy_(runner.first)  # the decode steps' first tokens, for the e2e steps
        fill_flops = prefill_flops(wl)
        out["kv_fill"] = {"what": f"prefill of the {wl.n_seqs} prompts ({wl.n_prompt_tokens} tokens) that fill "
                                  "the KV cache, timed once", "ms": round(fill_ms, 3),
                          "tokens_s": round(wl.n_prompt_tokens / (fill_ms / 1e3), 1),
                          "tflops": round(fill_flops / (fill_ms / 1e3) / 1e12, 1),
                          "tensor_frac": round(fill_flops / (fill_ms / 1e3) / 1e12 / float(peaks["bf16_tflops"]), 4)}
    for _ in range(max(args.warmup, 3)):
        runner.step()
    torch.cuda.synchronize()
    ms, launches, clocks = timed_steps(torch, binding, runner, args.steps, local_rank, world)
    ms_max, units_all = reduce_over_ranks(torch, world, ms, units * args.steps)
    e2e_ms, h2d, d2h = e2e_steps(torch, runner, args.steps, world)
    e2e_ms_max, e2e_units = reduce_over_ranks(torch, world, e2e_ms, units * args.steps)
    assert runner.model.status() == 0, binding.qwen3_last_error(runner.model.ctx)
    runner.model.close()
    del runner
    torch.cuda.empty_cache()
    if kv_block_tokens:  # the kernels read the cache through the block table: the whole step
        roofline = step_roofline(wl, ms / 1e3 / args.steps, peaks, peak_kind,
                                 f"paged KV cache, {kv_block_tokens}-token blocks")
    else:
        roofline = roofline_for(torch, binding, wl, peaks, peak_kind)
    # batched decode: the projections' share of the step, shown by its largest kernel
    proj = (measure_proj_roofline(torch, binding, wl, peaks, peak_kind)
            if wl.decode_steps and wl.n_seqs > 4 and not kv_block_tokens else None)
    torch.cuda.empty_cache()
    out.update({"value": units_all / (ms_max / 1e3), "unit": unit, "ms_per_step": ms_max / args.steps,
                "units_per_step": units, "launches": launches, "clocks": clocks,
                "e2e": {"value": round(e2e_units / (e2e_ms_max / 1e3), 2), "unit": unit,
                        "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
                "roofline": roofline})
    if proj:
        out["roofline_proj"] = proj
    step_s = ms_max / 1e3 / args.steps
    if wl.decode_steps:
        out["decode_step_hbm_frac"] = round(decode_step_bytes(wl) / (step_s / wl.decode_steps) / 1e9 /
                                            float(peaks["hbm_gbs"]), 4)
        out["decode_step_bytes"] = int(decode_step_bytes(wl))
    else:
        out["tflops"] = round(prefill_flops(wl) / step_s / 1e12, 1)
        out["tensor_frac"] = round(prefill_flops(wl) / step_s / 1e12 / float(peaks["bf16_tflops"]), 4)
    rank = dist_env()[0]
    out["cpu_baseline"] = cpu_baseline(wl, unit) if (cpu and rank == 0 and world == 1) else None
    return out


def run_prefill_chunked(args, device, flags, peaks, peak_kind, world, local_rank, weights):
    """One 16,384-token prompt fed as chunks of 2,048 through qwen3_prefill (the first) and
    qwen3_prefill_append (the rest), one step = the whole prompt; beside it the same prompt as
    one qwen3_prefill call."""
    import dataclasses
    import torch
    from qwen3_decoder_forward_gb300 import binding, synth

    s = synth.QWEN3_0P6B
    n, chunk = synth.CHUNKED_PROMPT, synth.CHUNKED_CHUNK
    wl = synth.Workload("prefill_chunked", s, (n,), 0, synth.KV_FILL_SEED)
    prompt = wl.prompts()[0]
    prompt_d = prompt.to(device)
    prompt_h = prompt.pin_memory()
    m = binding.Model(s, weights, max_seqs=1, max_ctx=n, max_prefill_tokens=n, flags=flags, device=str(device))
    nxt = torch.zeros(1, dtype=torch.int32, device=device)
    nxt_h = torch.zeros(1, dtype=torch.int32).pin_memory()
    stream = torch.cuda.current_stream(device)

    def chunked(toks):
        for c0 in range(0, n, chunk):
            m.prefill(toks[c0: c0 + chunk], [min(chunk, n - c0)], [0], next_out=nxt, append=c0 > 0)

    def whole(toks):
        m.prefill(toks, [n], [0], next_out=nxt)

    def timed(fn, steps):
        for _ in range(max(args.warmup, 3)):
            fn(prompt_d)
        torch.cuda.synchronize()
        n0 = binding.qwen3_launch_count(m.ctx)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn(prompt_d)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1), binding.qwen3_launch_count(m.ctx) - n0

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    sampler.mark(True)
    ms, launches = timed(chunked, args.steps)
    sampler.mark(False)
    sampler.stop()
    ms_whole, _ = timed(whole, args.steps)
    # end to end: the prompt copied in from pinned host memory, the next token read back
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        toks = torch.empty_like(prompt_h, device=device)
        toks.copy_(prompt_h, non_blocking=True)
        chunked(toks)
        nxt_h.copy_(nxt, non_blocking=True)
        stream.synchronize()
    e2e_s = time.perf_counter() - t0
    assert m.status() == 0, binding.qwen3_last_error(m.ctx)
    m.close()
    step_s = ms / 1e3 / args.steps
    flops = prefill_flops(wl) + 2 * s.hidden * s.vocab * (n // chunk - 1)  # one head row per chunk
    return {"workload": (f"prefill_chunked: one {n}-token prompt (28-layer Qwen3-0.6B shape) as {n // chunk} chunks of "
                         f"{chunk} (prefill, then prefill_append)"),
            "value": n * args.steps / (ms / 1e3), "unit": "tokens/s", "ms_per_step": step_s * 1e3,
            "launches": launches, "clocks": dict(sampler.summary(), retried=False),
            "e2e": {"value": round(n * args.steps / e2e_s, 1), "unit": "tokens/s", "h2d_bytes_per_step": n * 4 + 16,
                    "d2h_bytes_per_step": 4},
            "roofline": step_roofline(dataclasses.replace(wl), step_s, peaks, peak_kind, "8 chunk calls")
            | {"algorithmic_flops_per_step": int(flops), "achieved": round(flops / step_s / 1e12, 1),
               "frac": round(flops / step_s / 1e12 / float(peaks["bf16_tflops"]), 4)},
            "one_call": {"ms": round(ms_whole / args.steps, 3), "tokens_s": round(n * args.steps / (ms_whole / 1e3), 1)},
            "chunking_cost": round(ms / ms_whole, 3)}


def run_engine_mixed(args, device, flags, peaks, peak_kind, world, local_rank, weights):
    """48 requests through the continuous-batching engine, one step = submit all, run to the
    last one's end.  Units: generated tokens (prompt tokens reported beside them)."""
    import torch
    from qwen3_decoder_forward_gb300 import binding, synth

    s = synth.QWEN3_0P6B
    reqs = synth.engine_requests(s.vocab)
    max_ctx = 2048 + 128
    m = binding.Model(s, weights, max_seqs=synth.ENGINE_SLOTS, max_ctx=max_ctx,
                      max_prefill_tokens=synth.ENGINE_BUDGET, flags=flags, device=str(device))
    eng = binding.Engine(m, token_budget=synth.ENGINE_BUDGET)
    gen_tokens = sum(n for _, n in reqs)
    prompt_tokens = sum(int(p.numel()) for p, _ in reqs)
    lists = [(p.tolist(), n) for p, n in reqs]
    rid = [0]

    def one_step():
        ids = []
        for prompt, n in lists:
            rid[0] += 1
            eng.submit(rid[0], prompt, n)
            ids.append(rid[0])
        steps = eng.run()
        got = 0
        for i in ids:
            toks, why = eng.result(i)
            got += len(toks)
            eng.forget(i)
        return steps, got

    for _ in range(max(1, min(args.warmup, 2))):
        one_step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    sampler.mark(True)
    n0 = binding.qwen3_launch_count(m.ctx)
    st0 = eng.stats()
    t0 = time.perf_counter()
    steps_total = 0
    K = max(1, min(args.steps, 3))
    for _ in range(K):
        st, got = one_step()
        steps_total += st
        assert got == gen_tokens, (got, gen_tokens)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    sampler.mark(False)
    sampler.stop()
    st1 = eng.stats()
    launches = binding.qwen3_launch_count(m.ctx) - n0
    assert m.status() == 0, binding.qwen3_last_error(m.ctx)
    eng.close()
    m.close()
    return {"workload": (f"engine_mixed: {len(reqs)} requests (28-layer Qwen3-0.6B shape), prompts uniform in "
                         f"[256, 2048] tokens ({prompt_tokens} in all), 16..128 new tokens each ({gen_tokens} in all), "
                         f"{synth.ENGINE_SLOTS} slots, {synth.ENGINE_BUDGET} tokens a step"),
            "value": gen_tokens * K / dt, "unit": "tokens/s", "ms_per_step": dt * 1e3 / K,
            "launches": launches, "clocks": dict(sampler.summary(), retried=False),
            "e2e": {"value": round(gen_tokens * K / dt, 2), "unit": "tokens/s",
                    "h2d_bytes_per_step": prompt_tokens * 4, "d2h_bytes_per_step": gen_tokens * 4},
            "prompt_tokens_s": round(prompt_tokens * K / dt, 1),
            "engine_steps_per_run": steps_total / K,
            "mixed_steps": (st1["mixed_steps"] - st0["mixed_steps"]) / K,
            "decode_steps": (st1["decode_steps"] - st0["decode_steps"]) / K,
            "roofline": None}


def gpu_arm(args, wl):
    import torch
    from qwen3_decoder_forward_gb300 import binding, build, synth

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
             "chain": binding.QWEN3_FLAG_DECODE_CHAIN}[args.launch]
    args.warmup = max(args.warmup, 3)  # at least three untimed steps

    if args.roofline_only:
        r = (measure_proj_roofline(torch, binding, wl, peaks, peak_kind) if args.roofline_kernel == "proj" else
             roofline_for(torch, binding, wl, peaks, peak_kind, ctx=args.roofline_ctx))
        if rank == 0:
            print(json.dumps({"roofline_only": True, "workload": wl.name, "roofline": r}), flush=True)
        return 0
    if args.workload in synth.EXTRA_WORKLOADS:
        return gpu_extra(args, wl, device, flags, peaks, peak_kind, world, local_rank)

    weights = synth.make_weights(wl.shape)
    main = run_workload(args, wl, device, flags, peaks, peak_kind, world, local_rank, weights,
                        cpu=not args.no_cpu_baseline)
    pre = None
    if wl.decode_steps and args.prefill_workload != "none":
        pwl = synth.WORKLOADS[args.prefill_workload]
        if pwl.shape != wl.shape:
            weights = synth.make_weights(pwl.shape)
        pre = run_workload(args, pwl, device, flags, peaks, peak_kind, world, local_rank, weights,
                           cpu=not args.no_cpu_baseline)
    del weights

    if rank == 0:
        s = wl.shape
        line = {
            "metric": METRIC, "value": round(main["value"], 2), "unit": main["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(main["ms_per_step"], 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded random-init bf16 weights N(0,0.02), gains 1+N(0,0.05), uniform token ids)",
            "config": {"workload": workload_desc(wl),
                       "value_is": ("generated tokens per second: one step is the workload's decode steps of all "
                                    "its sequences from their prompts' KV cache (slots rewound before each step; "
                                    "the KV fill timed once, in kv_fill)") if wl.decode_steps
                       else "prompt tokens per second: one step is one packed prefill of every prompt",
                       "l2": "inputs larger than L2: every decode step streams 1.19 GB of weights and the KV "
                             "rows; a prefill streams the weights per layer (L2 is 129 MB)",
                       "replicas": world, "launch": args.launch},
            "clocks": main["clocks"],
            "e2e": main["e2e"],
            "gpu_launches": int(main["launches"] + (pre["launches"] if pre else 0)),
            "roofline": main["roofline"],
            "cpu_baseline": main["cpu_baseline"],
        }
        if main.get("roofline_proj"):
            line["roofline_proj"] = main["roofline_proj"]
        bd = {}
        for k in ("kv_fill", "decode_step_hbm_frac", "decode_step_bytes", "tflops", "tensor_frac"):
            if k in main:
                bd[k] = main[k]
        line["breakdown"] = bd
        if pre is not None:
            line["prefill"] = {"workload": workload_desc(synth.WORKLOADS[args.prefill_workload]),
                               "value": round(pre["value"], 1), "unit": pre["unit"],
                               "ms_per_step": round(pre["ms_per_step"], 4), "tflops": pre["tflops"],
                               "tensor_frac": pre["tensor_frac"], "e2e": pre["e2e"], "clocks": pre["clocks"],
                               "gpu_launches": int(pre["launches"]), "roofline": pre["roofline"],
                               "cpu_baseline": pre["cpu_baseline"]}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def gpu_extra(args, wl, device, flags, peaks, peak_kind, world, local_rank):
    """The lines of the feature workloads: chunked prefill, decode over a paged KV cache, and the
    continuous-batching engine."""
    from qwen3_decoder_forward_gb300 import synth

    rank = dist_env()[0]
    weights = synth.make_weights(synth.QWEN3_0P6B)
    extra = {}
    if args.workload == "decode_long_paged":
        res = run_workload(args, wl, device, flags, peaks, peak_kind, world, local_rank, weights,
                           cpu=not args.no_cpu_baseline, kv_block_tokens=synth.PAGED_BLOCK_TOKENS)
        desc = workload_desc(wl) + f"; paged KV cache of {synth.PAGED_BLOCK_TOKENS}-token blocks"
        extra = {"breakdown": {k: res[k] for k in ("kv_fill", "decode_step_hbm_frac", "decode_step_bytes")}}
    elif args.workload == "prefill_chunked":
        res = run_prefill_chunked(args, device, flags, peaks, peak_kind, world, local_rank, weights)
        desc = res["workload"]
        extra = {"one_call": res["one_call"], "chunking_cost": res["chunking_cost"]}
    else:
        res = run_engine_mixed(args, device, flags, peaks, peak_kind, world, local_rank, weights)
        desc = res["workload"]
        extra = {k: res[k] for k in ("prompt_tokens_s", "engine_steps_per_run", "mixed_steps", "decode_steps")}
    import torch
    ms_all = res["ms_per_step"] * args.steps
    ms_max, units_all = reduce_over_ranks(torch, world, ms_all, res["value"] * ms_all / 1e3)
    if rank == 0:
        line = {"metric": METRIC, "value": round(units_all / (ms_max / 1e3), 2), "unit": res["unit"],
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(res["ms_per_step"], 4), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded random-init bf16 weights N(0,0.02), gains 1+N(0,0.05), uniform token ids)",
                "config": {"workload": desc, "replicas": world, "launch": args.launch},
                "clocks": res["clocks"], "e2e": res["e2e"], "gpu_launches": int(res["launches"]),
                "roofline": res["roofline"], "cpu_baseline": res.get("cpu_baseline")}
        line.update(extra)
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    from qwen3_decoder_forward_gb300 import synth
    # the feature workloads time the workload they extend in the reference arm
    base = {"decode_long_paged": "decode_long", "prefill_chunked": "prefill_long",
            "engine_mixed": "decode_b32"}.get(args.workload, args.workload)
    if base == "prefill_long":
        wl = synth.Workload("prefill_long", synth.QWEN3_0P6B, (synth.CHUNKED_PROMPT,), 0, synth.KV_FILL_SEED)
    else:
        wl = synth.WORKLOADS[base]
    if args.decode_steps is not None:
        import dataclasses
        wl = dataclasses.replace(wl, name=f"{wl.name} (decode steps {args.decode_steps})",
                                 decode_steps=args.decode_steps)
    if args.impl == "reference":
        return reference_arm(args, wl)
    return gpu_arm(args, wl)


if __name__ == "__main__":
    sys.exit(main())
