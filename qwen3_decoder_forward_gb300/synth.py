"""Seeded synthetic inputs shared by the CUDA path's callers and the oracle's tests.

This module holds no arithmetic of the decoder forward itself: it only draws
random weights, token ids and ragged sequence lengths, and names the workloads
they are drawn for.  Every draw uses its own ``torch.Generator`` seeded from a
fixed base seed plus a stable per-tensor offset, so the bytes of one tensor do
not depend on which other tensors were drawn before it.

Shapes follow the Qwen3-0.6B checkpoint listing ("手写Qwen3-0.6B推理", section
"打印模型结构"; "古法手撕简易LLM推理器", section "处理参数和超参数"): per layer
q_proj [Hq*D, C], k_proj/v_proj [Hkv*D, C], o_proj [C, Hq*D], gate/up
[I, C], down [C, I], q_norm/k_norm [D], input/post norms [C]; embed [V, C]
tied with lm_head.  The trained weights are not available, so matrices are
drawn N(0, 0.02) and norm gains 1 + N(0, 0.05), all rounded to bf16.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, List

import torch


@dataclasses.dataclass(frozen=True)
class ModelShape:
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim


# Hyper-parameters of Qwen3-0.6B as the pages print them ("古法手撕简易LLM推理器",
# section "处理参数和超参数"; the config literal in the adg.csdn page, section "模型").
QWEN3_0P6B = ModelShape(n_layers=28, hidden=1024, n_q_heads=16, n_kv_heads=8,
                        head_dim=128, intermediate=3072, vocab=151936)
# One-layer model of the same widths with a 4096-entry vocabulary.
QWEN3_TINY = dataclasses.replace(QWEN3_0P6B, n_layers=1, vocab=4096)

WEIGHT_SEED = 1234
TOKEN_SEED = 1
LENGTH_SEED = 2
KV_FILL_SEED = 3

MATRIX_STD = 0.02
NORM_STD = 0.05

LAYER_KEYS = ("in_norm", "post_norm", "q_norm", "k_norm",
              "wq", "wk", "wv", "wo", "wgate", "wup", "wdown")


def layer_param_shapes(s: ModelShape) -> Dict[str, tuple]:
    return {
        "in_norm": (s.hidden,),
        "post_norm": (s.hidden,),
        "q_norm": (s.head_dim,),
        "k_norm": (s.head_dim,),
        "wq": (s.q_dim, s.hidden),
        "wk": (s.kv_dim, s.hidden),
        "wv": (s.kv_dim, s.hidden),
        "wo": (s.hidden, s.q_dim),
        "wgate": (s.intermediate, s.hidden),
        "wup": (s.intermediate, s.hidden),
        "wdown": (s.hidden, s.intermediate),
    }


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _matrix(shape, seed) -> torch.Tensor:
    return (torch.randn(shape, generator=_gen(seed), dtype=torch.float32) * MATRIX_STD).to(torch.bfloat16)


def _gain(shape, seed) -> torch.Tensor:
    return (1.0 + torch.randn(shape, generator=_gen(seed), dtype=torch.float32) * NORM_STD).to(torch.bfloat16)


def make_weights(s: ModelShape, seed: int = WEIGHT_SEED) -> Dict[str, object]:
    """Random bf16 weights on the CPU: {'embed', 'final_norm', 'layers': [dict]}.

    Tensor t of layer l is drawn from seed ``seed + 1000*(l+1) + index(t)``;
    embed and final_norm use ``seed`` and ``seed + 1``.
    """
    out: Dict[str, object] = {
        "embed": _matrix((s.vocab, s.hidden), seed),
        "final_norm": _gain((s.hidden,), seed + 1),
        "layers": [],
    }
    shapes = layer_param_shapes(s)
    for layer in range(s.n_layers):
        d = {}
        for idx, key in enumerate(LAYER_KEYS):
            sd = seed + 1000 * (layer + 1) + idx
            d[key] = _gain(shapes[key], sd) if key.endswith("norm") else _matrix(shapes[key], sd)
        out["layers"].append(d)
    return out


def make_tokens(n: int, vocab: int, seed: int) -> torch.Tensor:
    """n token ids drawn uniformly from [0, vocab), int32."""
    return torch.randint(0, vocab, (n,), generator=_gen(seed), dtype=torch.int64).to(torch.int32)


def make_lengths(n_seqs: int, lo: int, hi: int, seed: int) -> List[int]:
    """n_seqs integer lengths drawn uniformly from [lo, hi] inclusive."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n_seqs,), generator=_gen(seed), dtype=torch.int64)]


SAMPLE_SEED = 5

# Per-row sampling settings, cycled over the rows of a batch: greedy rows, temperature alone,
# Top-k alone, Top-p alone and both, with k on either side of the candidate count.
SAMPLE_TEMPERATURES = (0.0, 0.7, 1.0, 1.3, 0.9, 0.5)
SAMPLE_TOP_K = (0, 0, 50, 0, 20, 1000, 1, 5000)
SAMPLE_TOP_P = (1.0, 1.0, 1.0, 0.9, 0.8, 0.95, 0.5)


def make_sampling_batch(B: int, V: int, seed: int = SAMPLE_SEED, logit_std: float = 2.0,
                        grid: float = 0.0, spikes: int = 4):
    """Inputs of one sampling call: fp32 logits [B, V] ~ N(0, logit_std) with `spikes` tokens
    per row raised by U(4, 12) (a confident next-token distribution; rounded to multiples of
    `grid` when grid > 0, which makes many ties), the per-row settings above, and one uniform
    draw in [0, 1) per row.  Returns (logits, temperature, top_k, top_p, uniform) on the CPU."""
    g = _gen(seed)
    logits = torch.randn((B, V), generator=g) * logit_std
    if spikes:
        idx = torch.randint(0, V, (B, spikes), generator=g)
        logits.scatter_add_(1, idx, 4.0 + 8.0 * torch.rand((B, spikes), generator=g))
    if grid > 0:
        logits = torch.round(logits / grid) * grid
    temperature = torch.tensor([SAMPLE_TEMPERATURES[b % len(SAMPLE_TEMPERATURES)] for b in range(B)],
                               dtype=torch.float32)
    top_k = torch.tensor([SAMPLE_TOP_K[b % len(SAMPLE_TOP_K)] for b in range(B)], dtype=torch.int32)
    top_p = torch.tensor([SAMPLE_TOP_P[b % len(SAMPLE_TOP_P)] for b in range(B)], dtype=torch.float32)
    uniform = torch.rand((B,), generator=g)
    return logits.float(), temperature, top_k, top_p, uniform


def cu_seqlens(lengths: List[int]) -> List[int]:
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return out


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: the model, its prompts and its decode steps."""
    name: str
    shape: ModelShape
    lengths: tuple          # prompt length of each sequence
    decode_steps: int
    prompt_seed: int

    @property
    def n_seqs(self) -> int:
        return len(self.lengths)

    @property
    def n_prompt_tokens(self) -> int:
        return int(sum(self.lengths))

    @property
    def max_ctx(self) -> int:
        return max(self.lengths) + self.decode_steps

    def prompts(self) -> List[torch.Tensor]:
        """Per-sequence prompt ids; sequence i uses seed prompt_seed + 7919*i."""
        return [make_tokens(n, self.shape.vocab, self.prompt_seed + 7919 * i)
                for i, n in enumerate(self.lengths)]


def _ragged_lengths() -> tuple:
    return tuple(make_lengths(8, 512, 4096, LENGTH_SEED))


WORKLOADS = {
    # one layer, vocab 4096: 32-token prompt then 8 greedy steps
    "tiny": Workload("tiny", QWEN3_TINY, (32,), 8, TOKEN_SEED),
    # 28 layers, one sequence: 128-token prompt then 128 greedy steps
    "decode_b1": Workload("decode_b1", QWEN3_0P6B, (128,), 128, TOKEN_SEED),
    # 32 sequences, 1024-token prompts (the KV fill), then 64 steps
    "decode_b32": Workload("decode_b32", QWEN3_0P6B, (1024,) * 32, 64, KV_FILL_SEED),
    # 8 ragged prompts with lengths uniform in [512, 4096], prefill only
    "prefill_ragged": Workload("prefill_ragged", QWEN3_0P6B, _ragged_lengths(), 0, TOKEN_SEED),
    # 16 sequences, 16384-token prompts (the KV fill), then 32 steps
    "decode_long": Workload("decode_long", QWEN3_0P6B, (16384,) * 16, 32, KV_FILL_SEED),
}

# Workloads of the features beyond the plain forward, each measured with its own runner:
#  - prefill_chunked: one 16,384-token prompt fed as 8 chunks of 2,048 (the first a prefill,
#    the others prefill_append calls continuing the slot);
#  - decode_long_paged: decode_long over a paged KV cache of 256-token blocks;
#  - engine_mixed: 48 requests through the continuous-batching engine, prompts uniform in
#    [256, 2048] tokens and 16..128 new tokens each (seed ENGINE_SEED), 16 slots, 2,048 tokens
#    a step.
CHUNKED_PROMPT = 16384
CHUNKED_CHUNK = 2048
PAGED_BLOCK_TOKENS = 256
ENGINE_SEED = 4
ENGINE_REQUESTS = 48
ENGINE_SLOTS = 16
ENGINE_BUDGET = 2048
EXTRA_WORKLOADS = ("prefill_chunked", "decode_long_paged", "engine_mixed")


def engine_requests(vocab: int, n: int = ENGINE_REQUESTS, seed: int = ENGINE_SEED):
    """(prompt int32 tensor, max_new_tokens) of each request of engine_mixed."""
    lengths = make_lengths(n, 256, 2048, seed)
    new = make_lengths(n, 16, 128, seed + 1)
    return [(make_tokens(L, vocab, seed + 100 + 7919 * i), m) for i, (L, m) in enumerate(zip(lengths, new))]
