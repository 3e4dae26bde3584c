"""CPU oracle of the Qwen3-0.6B-style decoder forward -- TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this module.  It shares no code with the CUDA library: it is a plain, slow
restatement of what the pages define, step by step, in numpy.

Precision: every value is widened to float64 (``DTYPE``) on entry and all
arithmetic runs in that type; matrix products are numpy's ``@``.  The weights
it receives are already bf16-rounded, so the only rounding left is float64's.

Sources (page title, section):
  [P1] "手写Qwen3-0.6B推理" -- Qwen3Model, Qwen3DecoderLayer, Qwen3RMSNorm,
       Attention, Rope, MLP, 推理
  [P2] "第 3 章 前向与生成（代码走读）" -- 3.1 .. 3.4, 4.1, 4.2, 5
  [P3] "从零开始写Qwen3" -- Attn, norm, rope (原理 / 实现)
  [P4] "古法手撕简易LLM推理器" -- 工具函数, 核心计算函数与Transformer层,
       prefill与predict, RoPE的细节
Readings taken where the pages are silent or disagree are listed next to the
function that takes them.

Parity status: every function here is pinned by a closed form, an invariant or
an independent library routine in tests/test_oracle_pins.py, except the
end-to-end model with the real Qwen3-0.6B weights (not available), whose
agreement rests on the per-step pins.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

DTYPE = np.float64


# --------------------------------------------------------------------------- #
# Single steps                                                                 #
# --------------------------------------------------------------------------- #

def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gamma.

    [P1] Qwen3RMSNorm; [P4] 工具函数 ``RMSNorm``; [P3] norm.  eps sits inside
    the square root.  [P1] rounds the normalised value to the input dtype
    before the gain; the oracle keeps every step in float64 (no rounding).
    """
    x = np.asarray(x, dtype=DTYPE)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gamma, dtype=DTYPE)


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """theta_i = theta^(-2i/head_dim), i = 0 .. head_dim/2 - 1.

    [P1] Rope ``inv_freq``; [P3] rope 原理 (base angle beta^(-2i/d));
    [P4] RoPE的细节 (the base comes from the config: 1e6 for Qwen3).
    """
    i = np.arange(head_dim // 2, dtype=DTYPE)
    return np.power(DTYPE(theta), -2.0 * i / head_dim)


def apply_rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotate-half ("neox") RoPE of x[..., T, H, D] at absolute positions[T].

    Pair (i, i + D/2) is rotated by angle p * theta_i:
        x'_i       = x_i cos - x_{i+D/2} sin
        x'_{i+D/2} = x_{i+D/2} cos + x_i sin
    [P1] Rope (``rotate_half = cat(-x2, x1)``, ``emb = cat(freqs, freqs)``);
    [P4] 工具函数 (the rotate_half form) and RoPE的细节 (Qwen3 uses rotate_half,
    not the interleaved pairing); [P3] rope 实现 (neox swaps the halves).
    Angles and their cos/sin are taken in float64.
    """
    x = np.asarray(x, dtype=DTYPE)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(positions, dtype=DTYPE)[:, None] * rope_inv_freq(d, theta)[None, :]  # [T, D/2]
    cos = np.cos(ang)[:, None, :]  # broadcast over heads
    sin = np.sin(ang)[:, None, :]
    x1 = x[..., :half]
    x2 = x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    """silu(x) = x / (1 + e^-x).  [P4] 工具函数 ``SiLU``."""
    x = np.asarray(x, dtype=DTYPE)
    return x / (1.0 + np.exp(-x))


def softmax(s: np.ndarray) -> np.ndarray:
    """Row softmax with the row maximum subtracted first.  [P4] 工具函数 ``softmax``."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def causal_gqa_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                         q_pos: np.ndarray, k_pos: np.ndarray) -> np.ndarray:
    """Causal grouped-query attention for one sequence.

    q [T, Hq, D] at absolute positions q_pos[T]; k, v [S, Hkv, D] at k_pos[S].
    Query head h reads KV head h // (Hq/Hkv) ([P1] Attention: expand+flatten;
    [P2] 3.3: repeat_interleave; [P4] DotProductAttention).  Key j is visible to
    a query at position p iff k_pos[j] <= p ([P1] Qwen3Model causal mask; [P2]
    3.3 and 5: position i reads 0..i only).  Masked keys get weight exactly 0.
    With a cache, a query at position p sees keys 0..p -- the "bottom-right"
    reading of [P3] Attn (is_causal must not be used for a length-1 query) and
    [P4] 核心计算函数 (no mask once offset > 0).  Scores are scaled by
    1/sqrt(D) ([P1] Attention; [P3] Attn ``scale``) and the softmax runs in
    the working precision ([P1] softmax in float32; here float64).
    """
    q = np.asarray(q, dtype=DTYPE)
    k = np.asarray(k, dtype=DTYPE)
    v = np.asarray(v, dtype=DTYPE)
    t, hq, d = q.shape
    hkv = k.shape[1]
    group = hq // hkv
    visible = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]  # [T, S]
    out = np.zeros((t, hq, d), dtype=DTYPE)
    scale = 1.0 / np.sqrt(DTYPE(d))
    for h in range(hq):
        g = h // group
        s = (q[:, h, :] @ k[:, g, :].T) * scale          # [T, S]
        s = np.where(visible, s, -np.inf)
        w = softmax(s)
        out[:, h, :] = w @ v[:, g, :]
    return out


def swiglu_mlp(x: np.ndarray, wgate: np.ndarray, wup: np.ndarray, wdown: np.ndarray) -> np.ndarray:
    """down(silu(gate(x)) * up(x)).  [P1] MLP; [P2] 3.4; [P4] ``FFN``.

    Weight matrices are stored [out, in] as in the checkpoint, so y = x W^T.
    """
    return (silu(x @ wgate.T) * (x @ wup.T)) @ wdown.T


# --------------------------------------------------------------------------- #
# Model                                                                        #
# --------------------------------------------------------------------------- #

@dataclasses.dataclass
class Config:
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6


class Weights:
    """float64 copies of one model's (bf16-rounded) weights.

    ``layers[l]`` holds in_norm, post_norm, q_norm, k_norm, wq, wk, wv, wo,
    wgate, wup, wdown, each [out, in] for matrices.  The lm_head is the
    embedding table itself ([P1] Qwen3Model: ``lm_head.weight =
    embed_tokens.weight``).
    """

    def __init__(self, embed, final_norm, layers: Sequence[Dict[str, np.ndarray]]):
        self.embed = np.asarray(embed, dtype=DTYPE)
        self.final_norm = np.asarray(final_norm, dtype=DTYPE)
        self.layers = [{k: np.asarray(v, dtype=DTYPE) for k, v in d.items()} for d in layers]


class KVCache:
    """Per-layer key/value rows of one sequence: K after q/k-norm and RoPE, V raw.

    [P4] 核心计算函数与Transformer层: the cache keeps projected, normed and
    rotated K and projected V; prefill stores all rows, each step appends one.
    Rows live in preallocated arrays that grow when full, so an append copies
    only the new rows.
    """

    def __init__(self, n_layers: int):
        self._k: List[Optional[np.ndarray]] = [None] * n_layers
        self._v: List[Optional[np.ndarray]] = [None] * n_layers
        self._n = [0] * n_layers

    @property
    def length(self) -> int:
        return self._n[0]

    def keys(self, layer: int) -> np.ndarray:
        return self._k[layer][: self._n[layer]]

    def values(self, layer: int) -> np.ndarray:
        return self._v[layer][: self._n[layer]]

    def append(self, layer: int, k: np.ndarray, v: np.ndarray) -> None:
        n, t = self._n[layer], k.shape[0]
        if self._k[layer] is None or n + t > self._k[layer].shape[0]:
            cap = max(n + t, 2 * n, 16)
            grown_k = np.empty((cap,) + k.shape[1:], dtype=DTYPE)
            grown_v = np.empty((cap,) + v.shape[1:], dtype=DTYPE)
            if n:
                grown_k[:n] = self._k[layer][:n]
                grown_v[:n] = self._v[layer][:n]
            self._k[layer], self._v[layer] = grown_k, grown_v
        self._k[layer][n: n + t] = k
        self._v[layer][n: n + t] = v
        self._n[layer] = n + t

    @staticmethod
    def from_arrays(k_layers: Sequence[np.ndarray], v_layers: Sequence[np.ndarray],
                    spare: int = 0) -> "KVCache":
        """A cache holding given rows, each [S, Hkv, D] (e.g. another implementation's
        cache), with room for `spare` more rows per layer."""
        c = KVCache(len(k_layers))
        for layer, (k, v) in enumerate(zip(k_layers, v_layers)):
            s = k.shape[0]
            c._k[layer] = np.empty((s + spare,) + k.shape[1:], dtype=DTYPE)
            c._v[layer] = np.empty((s + spare,) + v.shape[1:], dtype=DTYPE)
            c._k[layer][:s] = k
            c._v[layer][:s] = v
            c._n[layer] = s
        return c


def decoder_layer(cfg: Config, w: Dict[str, np.ndarray], layer: int, h: np.ndarray,
                  positions: np.ndarray, cache: KVCache, trace: Optional[dict] = None) -> np.ndarray:
    """One pre-norm decoder layer over rows h[T, C] at absolute positions[T].

    h' = h + o_proj(attn(RMSNorm(h)));  out = h' + MLP(RMSNorm(h'))
    ([P1] Qwen3DecoderLayer; [P2] 3.2 -- the fused residual form computes the
    same sums).  Inside attention ([P1] Attention; [P2] 3.3; [P4]
    TransfomerLayer): q/k/v projections without bias, per-head RMSNorm of q
    and k (not v), RoPE of q and k, cache append, causal GQA attention over
    the cache, o_proj.  The new rows are appended before attention, so a
    query sees its own key.
    """
    t = h.shape[0]
    hq, hkv, d = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim
    u = rms_norm(h, w["in_norm"], cfg.rms_eps)
    q = (u @ w["wq"].T).reshape(t, hq, d)
    k = (u @ w["wk"].T).reshape(t, hkv, d)
    v = (u @ w["wv"].T).reshape(t, hkv, d)
    q = rms_norm(q, w["q_norm"], cfg.rms_eps)
    k = rms_norm(k, w["k_norm"], cfg.rms_eps)
    q = apply_rope(q, positions, cfg.rope_theta)
    k = apply_rope(k, positions, cfg.rope_theta)
    cache.append(layer, k, v)
    k_pos = np.arange(cache.keys(layer).shape[0])
    o = causal_gqa_attention(q, cache.keys(layer), cache.values(layer), positions, k_pos)
    if trace is not None:
        trace.setdefault("q", []).append(q)
        trace.setdefault("k", []).append(k)
        trace.setdefault("v", []).append(v)
        trace.setdefault("attn", []).append(o)
    h = h + o.reshape(t, hq * d) @ w["wo"].T
    m = rms_norm(h, w["post_norm"], cfg.rms_eps)
    return h + swiglu_mlp(m, w["wgate"], w["wup"], w["wdown"])


def forward(cfg: Config, w: Weights, ids: Sequence[int], cache: KVCache,
            all_logits: bool = False, trace: Optional[dict] = None) -> dict:
    """Run ids (one sequence) through the model, continuing after ``cache``.

    The rows sit at positions cache.length .. cache.length + T - 1 ([P4]
    prefill与predict: offset = cached length).  Returns
      hidden  [L+1, T, C]  h_0 = embedding rows ([P1] Qwen3Model; [P2] 3.1;
                            no scaling), h_l = residual stream after layer l
      logits  [V] of the last row (or [T, V] if all_logits)
      token, margin        greedy choice on the last row and its top-1/top-2 gap
    The head is RMSNorm(h_L) times the tied embedding ([P1] Qwen3Model;
    [P2] 4.1 keeps the last position only).
    """
    ids = np.asarray(ids, dtype=np.int64)
    t = ids.shape[0]
    start = cache.length
    positions = np.arange(start, start + t)
    h = w.embed[ids]
    hidden = [h]
    for layer in range(cfg.n_layers):
        h = decoder_layer(cfg, w.layers[layer], layer, h, positions, cache, trace)
        hidden.append(h)
    rows = h if all_logits else h[-1:]
    z = rms_norm(rows, w.final_norm, cfg.rms_eps) @ w.embed.T
    token, margin = greedy(z[-1])
    return {"hidden": np.stack(hidden), "logits": z if all_logits else z[0],
            "token": token, "margin": margin}


def greedy(logits: np.ndarray):
    """argmax over the vocabulary, lowest index on ties, and the top-1/top-2 gap.

    [P1] 推理 and [P2] 4.2/4.3 take torch.argmax of the last row; torch
    returns the first maximal index.  [P4] applies a softmax first, which is
    monotone and does not change the choice.
    """
    z = np.asarray(logits, dtype=DTYPE)
    tok = int(np.argmax(z))
    top2 = np.partition(z, -2)[-2:] if z.shape[0] >= 2 else np.array([-np.inf, z[0]])
    return tok, float(top2[1] - top2[0])


# Candidates considered by the sampler: the most likely tokens, at most this many.
SAMPLE_CANDIDATES = 1024


def sample(logits: np.ndarray, temperature: float, top_k: int, top_p: float, u: float,
           candidates: int = SAMPLE_CANDIDATES) -> int:
    """Next token drawn from the logits of one row ([P2] 4.3 Sampler: argmax when no
    temperature, otherwise temperature and Top-k/Top-p sampling; [P4] softmax with a
    temperature).  The pages name the steps but not their exact rule; the reading taken:

      temperature <= 0: the greedy choice (lowest index on ties).
      Otherwise z = logits / temperature; tokens ordered by z descending, index ascending;
      the first min(candidates, V) of that order are the candidates; top_k in [1, V) keeps
      the first top_k of them; p_i proportional to exp(z_i - z_max) over the kept tokens;
      top_p < 1 keeps the shortest prefix whose cumulative probability reaches top_p; the
      token is the first kept one whose cumulative probability exceeds u * (the kept total),
      u in [0, 1) a uniform draw supplied by the caller.
    """
    z = np.asarray(logits, dtype=DTYPE)
    if temperature <= 0:
        return greedy(z)[0]
    z = z / DTYPE(temperature)
    order = np.lexsort((np.arange(z.shape[0]), -z))  # z descending, then index ascending
    n = min(int(candidates), z.shape[0])
    if 1 <= top_k < n:
        n = int(top_k)
    kept = order[:n]
    p = np.exp(z[kept] - z[kept[0]])
    cum = np.cumsum(p)
    if top_p < 1.0:
        n = int(np.searchsorted(cum, DTYPE(top_p) * cum[-1], side="left")) + 1
        n = min(n, len(kept))
    target = DTYPE(u) * cum[n - 1]
    i = int(np.searchsorted(cum[:n], target, side="right"))
    return int(kept[min(i, n - 1)])


def generate(cfg: Config, w: Weights, prompt: Sequence[int], steps: int,
             forced: Optional[Sequence[int]] = None) -> dict:
    """Prefill the prompt, then run ``steps`` single-token decode steps.

    Step s feeds the token chosen at step s-1 (the prefill's choice for s=0),
    or ``forced[s]`` when given (teacher forcing).  [P4] prefill与predict;
    [P2] 4.2 (one token appended per step).  No EOS stop: steps are fixed.
    Returns per call (prefill first, then each step): hidden, logits, token,
    margin, plus the cache.
    """
    cache = KVCache(cfg.n_layers)
    out = [forward(cfg, w, prompt, cache)]
    fed = []
    for s in range(steps):
        tok = out[-1]["token"] if forced is None else int(forced[s])
        fed.append(tok)
        out.append(forward(cfg, w, [tok], cache))
    return {"calls": out, "fed": fed, "cache": cache}
