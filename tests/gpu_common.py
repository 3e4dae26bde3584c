"""Shared pieces of the GPU parity tests: oracle weights from the synthetic bf16 tensors,
the parity gate, and a teacher-forced runner that checks every call against the oracle.

Parity gate (one rule for every test): relative L2 error <= 1e-2 for each layer's hidden
state h_0..h_L (over the rows compared) and for the logits, and the same greedy token
wherever the oracle's top-1/top-2 logit gap exceeds 0.1.  The GPU rounds GEMM operands,
Q and the KV cache to bf16 (relative step 2^-8); accumulations, norms and softmax are fp32.
"""

from __future__ import annotations

import concurrent.futures
import multiprocessing

import numpy as np
import torch

from oracle import qwen3_oracle as oracle
from qwen3_decoder_forward_gb300 import binding, build

REL_L2 = 1e-2
MARGIN = 0.1


def ensure_library():
    build.build()
    return binding.load_library()


def oracle_config(shape) -> oracle.Config:
    return oracle.Config(n_layers=shape.n_layers, hidden=shape.hidden, n_q_heads=shape.n_q_heads,
                         n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim,
                         intermediate=shape.intermediate, vocab=shape.vocab, rms_eps=shape.rms_eps,
                         rope_theta=shape.rope_theta)


def oracle_weights(w) -> oracle.Weights:
    def f(t):
        return t.float().numpy()
    return oracle.Weights(f(w["embed"]), f(w["final_norm"]),
                          [{k: f(v) for k, v in d.items()} for d in w["layers"]])


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


class Gate:
    """Collects parity measurements and asserts the gate at the end."""

    def __init__(self):
        self.worst_hidden = 0.0
        self.worst_logits = 0.0
        self.tokens_checked = 0
        self.tokens_skipped = 0
        self.failures = []

    def hidden(self, gpu, ref, what):
        e = rel_l2(gpu, ref)
        self.worst_hidden = max(self.worst_hidden, e)
        if not e <= REL_L2:
            self.failures.append(f"{what}: hidden rel-L2 {e:.3e}")

    def logits(self, gpu, ref, what):
        e = rel_l2(gpu, ref)
        self.worst_logits = max(self.worst_logits, e)
        if not e <= REL_L2:
            self.failures.append(f"{what}: logits rel-L2 {e:.3e}")

    def token(self, gpu_tok, ref_tok, margin, what):
        if margin > MARGIN:
            self.tokens_checked += 1
            if int(gpu_tok) != int(ref_tok):
                self.failures.append(f"{what}: token {gpu_tok} != oracle {ref_tok} (margin {margin:.3f})")
        else:
            self.tokens_skipped += 1

    def check(self):
        assert not self.failures, "; ".join(self.failures[:10])

    def summary(self):
        return (f"worst hidden rel-L2 {self.worst_hidden:.2e}, worst logits rel-L2 {self.worst_logits:.2e}, "
                f"tokens checked {self.tokens_checked}, skipped (margin <= {MARGIN}) {self.tokens_skipped}")


def _oracle_prefill_job(shape, prompt):
    """Worker: the oracle's prefill of one prompt with the synthetic weights of `shape`
    (drawn again from their seeds in this process); hidden states as float32."""
    from qwen3_decoder_forward_gb300 import synth
    w = synth.make_weights(shape)
    ref = oracle.forward(oracle_config(shape), oracle_weights(w), list(prompt), oracle.KVCache(shape.n_layers))
    ref["hidden"] = ref["hidden"].astype(np.float32)
    return ref


def oracle_prefills(shape, prompts):
    """The oracle's prefill of each prompt (lists of ids), one spawned process per prompt, so
    long prompts run side by side on the host cores.  Spawned, not forked: the parent may
    already hold a CUDA context."""
    ctx = multiprocessing.get_context("spawn")
    with concurrent.futures.ProcessPoolExecutor(max_workers=len(prompts), mp_context=ctx) as ex:
        futs = [ex.submit(_oracle_prefill_job, shape, [int(t) for t in p]) for p in prompts]
        return [f.result() for f in futs]


def splitmix64_draw(seed: int, t: int) -> float:
    """The uniform draw of a sampling request's t-th token in the engine: output t + 1 of
    SplitMix64 (Steele, Lea and Flood 2014) started at `seed`, its top 24 bits over 2^24."""
    m = (1 << 64) - 1
    z = (seed + (t + 1) * 0x9E3779B97F4A7C15) & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    z ^= z >> 31
    return (z >> 40) / 16777216.0
