"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Every ``check_*`` takes the oracle module ``o`` and raises AssertionError on a
mismatch.  tests/test_oracle_pins.py runs them on the real oracle;
tests/test_oracle_mutations.py runs them on copies of the oracle with planted
mistakes and requires that each planted mistake makes some check fail.

Kinds of pins used here (no page prints numbers computed from known inputs):
  * closed forms of single steps on special inputs (constant vectors, one-hot
    vectors, zero queries, two-key softmax);
  * invariants the pages state: causality ("第 3 章 前向与生成", section 5),
    cache consistency (the no-cache loop of section 4.2 against the cached
    prefill/predict of "古法手撕简易LLM推理器"), RoPE's relative-position
    property ("从零开始写Qwen3", rope 原理);
  * independent library routines on tiny shapes: torch's F.rms_norm and
    F.scaled_dot_product_attention(enable_gqa=True), which the pages
    themselves use ("从零开始写Qwen3", sections Attn and norm).
"""

from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

ATOL = 1e-10


def _close(a, b, tol=1e-9, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    scale = max(1.0, float(np.max(np.abs(b)))) if b.size else 1.0
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    assert err <= tol * scale, f"{what}: max abs err {err:.3e} > {tol * scale:.3e}"


def tiny_cfg(o, layers=1, c=32, hq=4, hkv=2, d=8, inter=24, vocab=64):
    """The worked shape example of "第 3 章 前向与生成", section 5 (C=32, Hq=4, Hkv=2, D=8, V=64)."""
    return o.Config(n_layers=layers, hidden=c, n_q_heads=hq, n_kv_heads=hkv, head_dim=d,
                    intermediate=inter, vocab=vocab, rms_eps=1e-6, rope_theta=1e6)


def tiny_weights(o, cfg, seed=0, std=0.3):
    rng = np.random.default_rng(seed)
    c, qd, kd, i = cfg.hidden, cfg.n_q_heads * cfg.head_dim, cfg.n_kv_heads * cfg.head_dim, cfg.intermediate

    def mat(*s):
        return rng.standard_normal(s) * std

    def gain(n):
        return 1.0 + 0.1 * rng.standard_normal(n)

    layers = []
    for _ in range(cfg.n_layers):
        layers.append({
            "in_norm": gain(c), "post_norm": gain(c),
            "q_norm": gain(cfg.head_dim), "k_norm": gain(cfg.head_dim),
            "wq": mat(qd, c), "wk": mat(kd, c), "wv": mat(kd, c), "wo": mat(c, qd),
            "wgate": mat(i, c), "wup": mat(i, c), "wdown": mat(c, i),
        })
    return o.Weights(mat(cfg.vocab, c) * 3.0, gain(c), layers)


# --------------------------------------------------------------------------- #
# RMSNorm                                                                      #
# --------------------------------------------------------------------------- #

def check_rmsnorm_constant_vector(o):
    """c*1 normalises to gamma*c/sqrt(c^2+eps); at c=1e-3 eps=1e-6 matters (0.7071...)."""
    rng = np.random.default_rng(1)
    gamma = 1.0 + 0.1 * rng.standard_normal(1024)
    for c in (3.0, -0.5, 1e-3):
        x = np.full((2, 1024), c)
        want = gamma * c / math.sqrt(c * c + 1e-6)
        _close(o.rms_norm(x, gamma, 1e-6), np.stack([want, want]), what=f"rmsnorm const {c}")
    _close(o.rms_norm(np.full((1, 4), 1e-3), np.ones(4), 1e-6), np.full((1, 4), 1.0 / math.sqrt(2.0)),
           what="rmsnorm eps inside sqrt")


def check_rmsnorm_gain_and_scale(o):
    """Gain acts per element; RMSNorm(a*x) = RMSNorm(x) when eps is negligible."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 128))
    gamma = np.zeros(128)
    gamma[[0, 5, 127]] = [2.0, -1.0, 0.5]
    y = o.rms_norm(x, gamma, 1e-6)
    rms = np.sqrt(np.mean(x * x, axis=-1))
    for j, g in zip([0, 5, 127], [2.0, -1.0, 0.5]):
        _close(y[:, j], x[:, j] / np.sqrt(rms ** 2 + 1e-6) * g, what="rmsnorm gain column")
    assert np.all(np.delete(y, [0, 5, 127], axis=1) == 0.0)
    g1 = 1.0 + 0.1 * rng.standard_normal(128)
    _close(o.rms_norm(1e4 * x, g1, 1e-6), o.rms_norm(x, g1, 0.0), tol=1e-8, what="rmsnorm scale invariance")


def check_rmsnorm_vs_torch(o):
    """torch.nn.functional.rms_norm (the routine "从零开始写Qwen3" calls) in float64."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 1024)) * 0.7
    g = 1.0 + 0.05 * rng.standard_normal(1024)
    want = F.rms_norm(torch.from_numpy(x), (1024,), torch.from_numpy(g), 1e-6).numpy()
    _close(o.rms_norm(x, g, 1e-6), want, tol=1e-12, what="rmsnorm vs torch")


# --------------------------------------------------------------------------- #
# RoPE                                                                         #
# --------------------------------------------------------------------------- #

def _rope1(o, x, p, theta=1e6):
    """Rotate one vector x[D] at position p with the oracle."""
    return o.apply_rope(np.asarray(x, dtype=np.float64)[None, None, :], np.array([p]), theta)[0, 0]


def check_rope_identity_at_zero(o):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 5, 128))
    _close(o.apply_rope(x, np.zeros(3, dtype=np.int64), 1e6), x, tol=0, what="rope p=0")


def check_rope_basis_vectors(o):
    """A basis vector e_i (i < 64) rotates inside the plane (i, i+64) by p*theta^(-2i/128).

    The 2x2 rotation [[cos, -sin], [sin, cos]] of "从零开始写Qwen3" (rope 原理)
    applied to the half-swap pairing of Qwen3 ("古法手撕简易LLM推理器", RoPE的细节).
    """
    d = 128
    for i in (0, 1, 17, 63):
        for p in (1, 7, 1000, 16383):
            a = p * (1e6 ** (-2.0 * i / d))
            e = np.zeros(d)
            e[i] = 1.0
            want = np.zeros(d)
            want[i], want[i + 64] = math.cos(a), math.sin(a)
            _close(_rope1(o, e, p), want, tol=1e-12, what=f"rope e_{i} p={p}")
            e = np.zeros(d)
            e[i + 64] = 1.0
            want = np.zeros(d)
            want[i], want[i + 64] = -math.sin(a), math.cos(a)
            _close(_rope1(o, e, p), want, tol=1e-12, what=f"rope e_{i + 64} p={p}")


def check_rope_complex_form(o):
    """Pair (x_i, x_{i+64}) as the complex number x_i + j x_{i+64}, multiplied by e^{j p theta_i}."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((6, 3, 128))
    pos = np.array([0, 1, 2, 129, 4000, 40959])
    z = x[..., :64] + 1j * x[..., 64:]
    freq = 1e6 ** (-np.arange(64) / 64.0)
    rot = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    want = np.concatenate([rot.real, rot.imag], axis=-1)
    _close(o.apply_rope(x, pos, 1e6), want, tol=1e-12, what="rope complex form")


def check_rope_norm_and_relative_position(o):
    """Each (i, i+64) pair keeps its length; <R_m q, R_n k> depends on m-n only."""
    rng = np.random.default_rng(6)
    q = rng.standard_normal(128)
    k = rng.standard_normal(128)
    for p in (3, 999):
        r = _rope1(o, q, p)
        _close(r[:64] ** 2 + r[64:] ** 2, q[:64] ** 2 + q[64:] ** 2, tol=1e-12, what="rope pair norm")
    for m, n, s in ((5, 2, 11), (100, 40, 1234), (7, 7, 3000)):
        a = float(np.dot(_rope1(o, q, m), _rope1(o, k, n)))
        b = float(np.dot(_rope1(o, q, m + s), _rope1(o, k, n + s)))
        assert abs(a - b) <= 1e-9 * max(1.0, abs(a)), f"rope relative position {a} vs {b}"


def check_rope_not_interleaved(o):
    """The interleaved (2i, 2i+1) pairing gives a different result (negative test)."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal(128)
    freq = 1e6 ** (-np.arange(64) / 64.0)
    a = 5 * freq
    inter = x.copy()
    inter[0::2] = x[0::2] * np.cos(a) - x[1::2] * np.sin(a)
    inter[1::2] = x[1::2] * np.cos(a) + x[0::2] * np.sin(a)
    assert np.max(np.abs(_rope1(o, x, 5) - inter)) > 1e-3, "oracle RoPE matches the interleaved pairing"


# --------------------------------------------------------------------------- #
# Attention                                                                    #
# --------------------------------------------------------------------------- #

def check_attention_zero_query_is_causal_mean(o):
    """q = 0 gives equal weights over visible keys: row t averages v_0..v_t of its KV head."""
    rng = np.random.default_rng(8)
    t, hq, hkv, d = 9, 4, 2, 8
    v = rng.standard_normal((t, hkv, d))
    k = rng.standard_normal((t, hkv, d))
    out = o.causal_gqa_attention(np.zeros((t, hq, d)), k, v, np.arange(t), np.arange(t))
    for r in range(t):
        for h in range(hq):
            _close(out[r, h], v[: r + 1, h // 2].mean(axis=0), tol=1e-12, what=f"causal mean r={r} h={h}")


def check_attention_decode_bottom_right(o):
    """A single query at position p over a cache of p+1 keys sees every cached key."""
    rng = np.random.default_rng(9)
    s, hkv, d = 6, 2, 8
    v = rng.standard_normal((s, hkv, d))
    out = o.causal_gqa_attention(np.zeros((1, 4, d)), rng.standard_normal((s, hkv, d)), v,
                                 np.array([s - 1]), np.arange(s))
    for h in range(4):
        _close(out[0, h], v[:, h // 2].mean(axis=0), tol=1e-12, what="decode mean")


def check_attention_two_key_closed_form(o):
    """q = a e_0, k_0 = b e_0, k_1 = 0: w_0 = logistic(a b / sqrt(D))."""
    d = 128
    a, b = 3.0, 2.5
    q = np.zeros((2, 1, d))
    q[1, 0, 0] = a
    k = np.zeros((2, 1, d))
    k[0, 0, 0] = b
    rng = np.random.default_rng(10)
    v = rng.standard_normal((2, 1, d))
    out = o.causal_gqa_attention(q, k, v, np.arange(2), np.arange(2))
    w0 = 1.0 / (1.0 + math.exp(-a * b / math.sqrt(d)))
    _close(out[1, 0], w0 * v[0, 0] + (1 - w0) * v[1, 0], tol=1e-12, what="two-key softmax")
    _close(out[0, 0], v[0, 0], tol=1e-12, what="first row sees only key 0")


def check_attention_gqa_head_mapping(o):
    """Q heads 2g and 2g+1 read KV head g: constant V per KV head shows the mapping."""
    rng = np.random.default_rng(11)
    t, hq, hkv, d = 5, 16, 8, 8
    v = np.zeros((t, hkv, d))
    for g in range(hkv):
        v[:, g, :] = g + 1
    out = o.causal_gqa_attention(rng.standard_normal((t, hq, d)), rng.standard_normal((t, hkv, d)),
                                 v, np.arange(t), np.arange(t))
    for h in range(hq):
        _close(out[:, h, :], np.full((t, d), h // 2 + 1.0), tol=1e-12, what=f"gqa head {h}")


def check_attention_vs_torch_sdpa(o):
    """torch SDPA with enable_gqa and a causal mask ("从零开始写Qwen3", section Attn), float64."""
    rng = np.random.default_rng(12)
    t, hq, hkv, d = 11, 4, 2, 8
    q = rng.standard_normal((t, hq, d))
    k = rng.standard_normal((t, hkv, d))
    v = rng.standard_normal((t, hkv, d))
    want = F.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(0, 1)[None], torch.from_numpy(k).transpose(0, 1)[None],
        torch.from_numpy(v).transpose(0, 1)[None], is_causal=True, enable_gqa=True,
        scale=d ** -0.5)[0].transpose(0, 1).numpy()
    _close(o.causal_gqa_attention(q, k, v, np.arange(t), np.arange(t)), want, tol=1e-12,
           what="attention vs SDPA")
    # decode: the last 3 queries against all keys, with an explicit bottom-right mask
    mask = torch.from_numpy(np.arange(t)[None, :] <= np.arange(t - 3, t)[:, None])
    want = F.scaled_dot_product_attention(
        torch.from_numpy(q[-3:]).transpose(0, 1)[None], torch.from_numpy(k).transpose(0, 1)[None],
        torch.from_numpy(v).transpose(0, 1)[None], attn_mask=mask, enable_gqa=True,
        scale=d ** -0.5)[0].transpose(0, 1).numpy()
    _close(o.causal_gqa_attention(q[-3:], k, v, np.arange(t - 3, t), np.arange(t)), want, tol=1e-12,
           what="cached attention vs SDPA")


# --------------------------------------------------------------------------- #
# MLP                                                                          #
# --------------------------------------------------------------------------- #

def check_silu_values(o):
    want = {0.0: 0.0, 1.0: 0.7310585786300049, -1.0: -0.2689414213699951,
            2.0: 1.7615941559557646, 30.0: 30.0 / (1.0 + math.exp(-30.0))}
    for x, y in want.items():
        assert abs(float(o.silu(np.array(x))) - y) <= 1e-14, f"silu({x})"


def check_mlp_gate_up_order(o):
    """C=2, I=1 with gate reading x_0 and up reading x_1: out_0 = silu(x_0) * x_1."""
    wg = np.array([[1.0, 0.0]])
    wu = np.array([[0.0, 1.0]])
    wd = np.array([[1.0], [0.0]])
    out = o.swiglu_mlp(np.array([[1.0, 2.0]]), wg, wu, wd)
    _close(out, np.array([[2.0 * 0.7310585786300049, 0.0]]), tol=1e-14, what="swiglu order")


# --------------------------------------------------------------------------- #
# Whole model                                                                  #
# --------------------------------------------------------------------------- #

def check_zero_branches_are_identity(o):
    """With o_proj and down_proj zero, every layer passes h through unchanged (residual form)."""
    cfg = tiny_cfg(o, layers=2)
    w = tiny_weights(o, cfg, seed=13)
    for L in w.layers:
        L["wo"][:] = 0.0
        L["wdown"][:] = 0.0
    out = o.forward(cfg, w, [3, 1, 4, 1, 5], o.KVCache(cfg.n_layers))
    for layer in range(3):
        _close(out["hidden"][layer], w.embed[[3, 1, 4, 1, 5]], tol=0, what=f"identity layer {layer}")


def check_mlp_sees_normalised_input(o):
    """With o_proj zero, h_1 - a*h_0 does not depend on a (pre-norm MLP input)."""
    cfg = tiny_cfg(o, layers=1)
    cfg.rms_eps = 0.0  # exact scale invariance of the norm
    w = tiny_weights(o, cfg, seed=14)
    w.layers[0]["wo"][:] = 0.0
    res = []
    for a in (1.0, 7.0):
        w2 = o.Weights(w.embed * a, w.final_norm, w.layers)
        out = o.forward(cfg, w2, [2, 9, 33], o.KVCache(1))
        res.append(out["hidden"][1] - out["hidden"][0])
    _close(res[0], res[1], tol=1e-9, what="pre-norm MLP")


def check_embedding_rows(o):
    cfg = tiny_cfg(o)
    w = tiny_weights(o, cfg, seed=15)
    out = o.forward(cfg, w, [0, 63, 7], o.KVCache(1))
    _close(out["hidden"][0], w.embed[[0, 63, 7]], tol=0, what="h_0 = E[ids]")


def check_causality_prefix(o):
    """Appending or changing later tokens leaves earlier rows unchanged ("第 3 章", section 5)."""
    cfg = tiny_cfg(o, layers=2)
    w = tiny_weights(o, cfg, seed=16)
    ids = [5, 17, 2, 40, 40, 9, 61]
    full = o.forward(cfg, w, ids, o.KVCache(2), all_logits=True)
    alt = o.forward(cfg, w, ids[:4] + [1, 2, 3], o.KVCache(2), all_logits=True)
    pre = o.forward(cfg, w, ids[:4], o.KVCache(2), all_logits=True)
    _close(pre["hidden"], full["hidden"][:, :4], tol=1e-12, what="prefix hidden")
    _close(pre["logits"], full["logits"][:4], tol=1e-12, what="prefix logits")
    _close(alt["logits"][:4], full["logits"][:4], tol=1e-12, what="future change")
    assert np.max(np.abs(alt["logits"][4:] - full["logits"][4:])) > 1e-6


def check_cache_consistency(o):
    """A decode step at position t equals a no-cache forward of the t+1 prefix at its last row.

    "第 3 章 前向与生成", section 4.2 (the loop that recomputes the whole prefix)
    against "古法手撕简易LLM推理器", section prefill与predict (the cached path).
    """
    cfg = tiny_cfg(o, layers=2)
    w = tiny_weights(o, cfg, seed=17)
    prompt = [11, 3, 50, 7, 7]
    run = o.generate(cfg, w, prompt, steps=4)
    seq = list(prompt)
    for s in range(4):
        seq.append(run["fed"][s])
        ref = o.forward(cfg, w, seq, o.KVCache(2), all_logits=True)
        step = run["calls"][s + 1]
        _close(step["hidden"][:, 0], ref["hidden"][:, -1], tol=1e-10, what=f"step {s} hidden")
        _close(step["logits"], ref["logits"][-1], tol=1e-10, what=f"step {s} logits")
        assert step["token"] == int(np.argmax(ref["logits"][-1]))
    prefill_next = run["calls"][0]["token"]
    assert run["fed"][0] == prefill_next


def check_cache_from_arrays(o):
    """A cache rebuilt from another cache's rows (as the long-context test rebuilds one from the
    GPU's rows) holds exactly those rows and continues exactly as the original: decode steps
    from it equal the steps of the run that filled the original ("古法手撕简易LLM推理器",
    prefill与predict: each step reads the cached K/V and appends one row)."""
    cfg = tiny_cfg(o, layers=2)
    w = tiny_weights(o, cfg, seed=21)
    prompt = [9, 31, 4, 4, 60, 2]
    run = o.generate(cfg, w, prompt, steps=3)
    filled = o.KVCache(2)
    o.forward(cfg, w, prompt, filled)
    ks = [filled.keys(layer).copy() for layer in range(2)]
    vs = [filled.values(layer).copy() for layer in range(2)]
    c = o.KVCache.from_arrays(ks, vs, spare=3)
    assert c.length == len(prompt)
    for layer in range(2):
        assert np.array_equal(c.keys(layer), ks[layer]) and np.array_equal(c.values(layer), vs[layer])
    for s in range(3):
        step = o.forward(cfg, w, [run["fed"][s]], c)
        _close(step["logits"], run["calls"][s + 1]["logits"], tol=1e-12, what=f"rebuilt cache step {s}")
        _close(step["hidden"], run["calls"][s + 1]["hidden"], tol=1e-12, what=f"rebuilt cache step {s} hidden")
    assert c.length == len(prompt) + 3


def check_greedy_ties_and_margin(o):
    tok, margin = o.greedy(np.array([0.5, 2.0, -1.0, 2.0, 1.5]))
    assert tok == 1, "ties resolve to the lowest index"
    assert margin == 0.0
    tok, margin = o.greedy(np.array([0.0, 1.25, 3.0, -4.0]))
    assert tok == 2 and abs(margin - 1.75) < 1e-15


def _sample_brute(logits, temperature, top_k, top_p, candidates):
    """Kept tokens and their probabilities, written independently with Python's sorted and math
    (the reading of "第 3 章", 4.3 stated in the oracle's sample docstring)."""
    z = [float(x) / temperature for x in logits]
    order = sorted(range(len(z)), key=lambda i: (-z[i], i))[:candidates]
    if 1 <= top_k < len(order):
        order = order[:top_k]
    w = [math.exp(z[i] - z[order[0]]) for i in order]
    total = sum(w)
    if top_p < 1.0:
        acc, n = 0.0, 0
        while n < len(order):
            acc += w[n] / total
            n += 1
            if acc >= top_p - 1e-15:
                break
        order, w = order[:n], w[:n]
        total = sum(w)
    return order, [x / total for x in w]


def check_sample_frequencies_brute_force(o):
    """Draws on a fine grid of u reproduce the kept tokens' renormalised probabilities."""
    rng = np.random.default_rng(11)
    for temperature, top_k, top_p, v, cand in [(0.7, 0, 1.0, 9, 1024), (1.3, 4, 1.0, 9, 1024),
                                              (0.9, 0, 0.8, 9, 1024), (1.1, 6, 0.7, 12, 1024),
                                              (0.8, 0, 1.0, 12, 5), (1.0, 3, 0.9, 12, 8)]:
        logits = rng.normal(0.0, 1.5, v)
        logits[3] = logits[7]  # a tie, resolved by the lower index
        kept, probs = _sample_brute(logits, temperature, top_k, top_p, cand)
        grid = 20000
        counts = {}
        for j in range(grid):
            t = o.sample(logits, temperature, top_k, top_p, (j + 0.5) / grid, candidates=cand)
            counts[t] = counts.get(t, 0) + 1
        assert set(counts) <= set(kept), (set(counts), kept)
        for tok, pr in zip(kept, probs):
            assert abs(counts.get(tok, 0) / grid - pr) < 2e-4, (temperature, top_k, top_p, tok, pr)
        # the inverse CDF walks the kept tokens in order: low u gives the first kept token
        assert o.sample(logits, temperature, top_k, top_p, 0.0, candidates=cand) == kept[0]


def check_sample_limits_and_invariance(o):
    rng = np.random.default_rng(12)
    logits = rng.normal(0.0, 2.0, 50)
    logits[17] = logits.max()  # tie with the maximum: argmax takes the lower index
    best = int(np.argmax(logits))
    for u in (0.0, 0.37, 0.999):
        assert o.sample(logits, 0.0, 0, 1.0, u) == best          # no temperature: greedy
        assert o.sample(logits, 0.8, 1, 1.0, u) == best          # top-1
        assert o.sample(logits, 0.8, 0, 1e-9, u) == best         # nucleus of one token
        # softmax(z / T) is unchanged by adding a constant, and by scaling z and T together
        assert o.sample(logits, 0.8, 5, 0.9, u) == o.sample(logits + 3.25, 0.8, 5, 0.9, u)
        assert o.sample(logits, 0.8, 5, 0.9, u) == o.sample(logits * 2.0, 1.6, 5, 0.9, u)
    # flat logits over more tokens than candidates: only the first `candidates` indices are drawn
    flat = np.zeros(3000)
    assert o.sample(flat, 1.0, 0, 1.0, 0.99999, candidates=1024) == 1023
    assert o.sample(flat, 1.0, 0, 1.0, 0.5, candidates=1024) == 512


def check_shapes_worked_example(o):
    """The shape table of "第 3 章 前向与生成", section 5 (B=1, T=3, C=32, Hq=4, Hkv=2, D=8, V=64)."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "shape_example_forward_chapter3.json")
    with open(path) as f:
        g = json.load(f)
    cfg = tiny_cfg(o, layers=1, c=g["C"], hq=g["Hq"], hkv=g["Hkv"], d=g["D"], vocab=g["V"])
    w = tiny_weights(o, cfg, seed=18)
    trace = {}
    ids = list(range(g["T"]))
    full = o.forward(cfg, w, ids, o.KVCache(1), all_logits=True, trace=trace)
    last = o.forward(cfg, w, ids, o.KVCache(1))
    # the pages' tensors are [B, H, T, D]; the oracle keeps one sequence as [T, H, D]
    assert [g["B"]] + [trace["q"][0].shape[i] for i in (1, 0, 2)] == g["Q"]
    assert [g["B"]] + [trace["k"][0].shape[i] for i in (1, 0, 2)] == g["K"]
    assert [g["B"]] + [trace["v"][0].shape[i] for i in (1, 0, 2)] == g["V_raw"]
    assert [g["B"], g["T"], g["C"]] == g["embedding"]
    assert list(full["hidden"][0].shape) == g["embedding"][1:]
    assert [g["B"]] + list(full["logits"].shape) == g["logits_all"]
    assert [g["B"]] + list(last["logits"].shape) == g["logits_next"]
    assert list(trace["attn"][0].shape) == [g["T"], g["Hq"], g["D"]]


def torch_reference_forward(cfg, w, ids):
    """The model composed from torch library routines in float64, rows [T] of one sequence."""
    def t(a):
        return torch.from_numpy(np.asarray(a, dtype=np.float64))

    ids_t = torch.as_tensor(ids)
    h = t(w.embed)[ids_t]
    T = len(ids)
    pos = torch.arange(T, dtype=torch.float64)
    inv = 1.0 / (cfg.rope_theta ** (torch.arange(0, cfg.head_dim, 2, dtype=torch.float64) / cfg.head_dim))
    ang = pos[:, None] * inv[None, :]
    cos = torch.cat([ang.cos(), ang.cos()], -1)[None, :, :]
    sin = torch.cat([ang.sin(), ang.sin()], -1)[None, :, :]

    def rot(x):  # x [H, T, D]
        x1, x2 = x.chunk(2, dim=-1)
        return x * cos + torch.cat([-x2, x1], -1) * sin

    hiddens = [h]
    for L in w.layers:
        u = F.rms_norm(h, (cfg.hidden,), t(L["in_norm"]), cfg.rms_eps)
        q = F.linear(u, t(L["wq"])).view(T, cfg.n_q_heads, cfg.head_dim).transpose(0, 1)
        k = F.linear(u, t(L["wk"])).view(T, cfg.n_kv_heads, cfg.head_dim).transpose(0, 1)
        v = F.linear(u, t(L["wv"])).view(T, cfg.n_kv_heads, cfg.head_dim).transpose(0, 1)
        q = rot(F.rms_norm(q, (cfg.head_dim,), t(L["q_norm"]), cfg.rms_eps))
        k = rot(F.rms_norm(k, (cfg.head_dim,), t(L["k_norm"]), cfg.rms_eps))
        a = F.scaled_dot_product_attention(q[None], k[None], v[None], is_causal=True, enable_gqa=True,
                                           scale=cfg.head_dim ** -0.5)[0]
        h = h + F.linear(a.transpose(0, 1).reshape(T, -1), t(L["wo"]))
        m = F.rms_norm(h, (cfg.hidden,), t(L["post_norm"]), cfg.rms_eps)
        h = h + F.linear(F.silu(F.linear(m, t(L["wgate"]))) * F.linear(m, t(L["wup"])), t(L["wdown"]))
        hiddens.append(h)
    z = F.linear(F.rms_norm(h, (cfg.hidden,), t(w.final_norm), cfg.rms_eps), t(w.embed))
    return torch.stack(hiddens).numpy(), z.numpy()


def check_model_vs_torch_composition(o):
    """Whole forward against the same model assembled from torch routines (float64)."""
    cfg = tiny_cfg(o, layers=2, c=64, hq=4, hkv=2, d=16, inter=48, vocab=80)
    w = tiny_weights(o, cfg, seed=19)
    ids = [4, 70, 12, 12, 0, 33, 79, 5]
    out = o.forward(cfg, w, ids, o.KVCache(2), all_logits=True)
    hid, z = torch_reference_forward(cfg, w, ids)
    _close(out["hidden"], hid, tol=1e-10, what="hidden vs torch")
    _close(out["logits"], z, tol=1e-10, what="logits vs torch")


ALL_CHECKS = [
    check_rmsnorm_constant_vector,
    check_rmsnorm_gain_and_scale,
    check_rmsnorm_vs_torch,
    check_rope_identity_at_zero,
    check_rope_basis_vectors,
    check_rope_complex_form,
    check_rope_norm_and_relative_position,
    check_rope_not_interleaved,
    check_attention_zero_query_is_causal_mean,
    check_attention_decode_bottom_right,
    check_attention_two_key_closed_form,
    check_attention_gqa_head_mapping,
    check_attention_vs_torch_sdpa,
    check_silu_values,
    check_mlp_gate_up_order,
    check_zero_branches_are_identity,
    check_mlp_sees_normalised_input,
    check_embedding_rows,
    check_causality_prefix,
    check_cache_consistency,
    check_cache_from_arrays,
    check_greedy_ties_and_margin,
    check_sample_frequencies_brute_force,
    check_sample_limits_and_invariance,
    check_shapes_worked_example,
    check_model_vs_torch_composition,
]
