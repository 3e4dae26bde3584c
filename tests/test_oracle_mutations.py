"""Each plausible mistake planted in a copy of the oracle makes some pin fail.

The copy is the oracle's own source with one substring replaced, loaded as a
separate module on the CPU; the real oracle is never modified.
"""

import importlib.util
import os
import sys

import pytest

import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "qwen3_oracle.py")

MUTANTS = {
    "eps_outside_sqrt": ("np.sqrt(ms + eps)", "(np.sqrt(ms) + eps)"),
    "sum_not_mean": ("np.mean(x * x, axis=-1, keepdims=True)", "np.sum(x * x, axis=-1, keepdims=True)"),
    "rmsnorm_no_gain": ("return x / np.sqrt(ms + eps) * np.asarray(gamma, dtype=DTYPE)", "return x / np.sqrt(ms + eps)"),
    "rope_freq_i_over_d": ("-2.0 * i / head_dim", "-1.0 * i / head_dim"),
    "rope_sign": ("[x1 * cos - x2 * sin, x2 * cos + x1 * sin]", "[x1 * cos + x2 * sin, x2 * cos - x1 * sin]"),
    "rope_interleaved_pairs": ("x1 = x[..., :half]\n    x2 = x[..., half:]", "x1 = x[..., 0::2]\n    x2 = x[..., 1::2]"),
    "positions_restart_each_call": ("positions = np.arange(start, start + t)", "positions = np.arange(0, t)"),
    "no_attention_scale": ("scale = 1.0 / np.sqrt(DTYPE(d))", "scale = 1.0"),
    "gqa_modulo_mapping": ("g = h // group", "g = h % hkv"),
    "no_causal_mask": ("s = np.where(visible, s, -np.inf)", "s = s"),
    "strict_causal_mask": ("np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]",
                           "np.asarray(k_pos)[None, :] < np.asarray(q_pos)[:, None]"),
    "silu_sign": ("x / (1.0 + np.exp(-x))", "x / (1.0 + np.exp(x))"),
    "gate_up_swapped": ("(silu(x @ wgate.T) * (x @ wup.T))", "(silu(x @ wup.T) * (x @ wgate.T))"),
    "attn_residual_dropped": ('h = h + o.reshape(t, hq * d) @ w["wo"].T', 'h = o.reshape(t, hq * d) @ w["wo"].T'),
    "mlp_residual_dropped": ('return h + swiglu_mlp(m, w["wgate"], w["wup"], w["wdown"])',
                             'return swiglu_mlp(m, w["wgate"], w["wup"], w["wdown"])'),
    "mlp_input_not_normed": ('m = rms_norm(h, w["post_norm"], cfg.rms_eps)', "m = h"),
    "post_norm_uses_input_gain": ('m = rms_norm(h, w["post_norm"]', 'm = rms_norm(h, w["in_norm"]'),
    "k_norm_uses_q_gain": ('k = rms_norm(k, w["k_norm"]', 'k = rms_norm(k, w["q_norm"]'),
    "q_norm_missing": ('q = rms_norm(q, w["q_norm"], cfg.rms_eps)', "q = q"),
    "k_not_rotated": ("k = apply_rope(k, positions, cfg.rope_theta)", "k = k"),
    "v_rotated": ('v = (u @ w["wv"].T).reshape(t, hkv, d)',
                  'v = apply_rope((u @ w["wv"].T).reshape(t, hkv, d), positions, cfg.rope_theta)'),
    "final_norm_missing": ("z = rms_norm(rows, w.final_norm, cfg.rms_eps) @ w.embed.T", "z = rows @ w.embed.T"),
    "argmax_last_tie": ("tok = int(np.argmax(z))", "tok = int(len(z) - 1 - np.argmax(z[::-1]))"),
    "embedding_scaled": ("h = w.embed[ids]", "h = w.embed[ids] * np.sqrt(cfg.hidden)"),
    "wq_transposed_heads": ('q = (u @ w["wq"].T).reshape(t, hq, d)',
                            'q = (u @ w["wq"].T).reshape(t, d, hq).transpose(0, 2, 1)'),
    "o_proj_head_order": ("h = h + o.reshape(t, hq * d)", "h = h + o.transpose(0, 2, 1).reshape(t, hq * d)"),
    "from_arrays_kv_swapped": ("c._k[layer][:s] = k\n            c._v[layer][:s] = v",
                               "c._k[layer][:s] = v\n            c._v[layer][:s] = k"),
    "from_arrays_drops_last_row": ("c._n[layer] = s\n", "c._n[layer] = s - 1\n"),
    "sample_ascending_order": ("np.lexsort((np.arange(z.shape[0]), -z))", "np.lexsort((np.arange(z.shape[0]), z))"),
    "sample_no_temperature": ("z = z / DTYPE(temperature)", "z = z"),
    "sample_top_p_one_short": ("side=\"left\")) + 1", "side=\"left\"))"),
    "sample_cdf_left": ("np.searchsorted(cum[:n], target, side=\"right\")", "np.searchsorted(cum[:n], target, side=\"left\")"),
    "sample_ties_high_index": ("np.lexsort((np.arange(z.shape[0]), -z))", "np.lexsort((-np.arange(z.shape[0]), -z))"),
}


def _load_mutant(name, old, new):
    with open(SRC) as f:
        text = f.read()
    assert text.count(old) >= 1, f"mutant {name}: pattern not found in the oracle source"
    text = text.replace(old, new)
    spec = importlib.util.spec_from_loader(f"oracle_mutant_{name}", loader=None)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod  # dataclasses look their module up by name
    exec(compile(text, f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    mod = _load_mutant(name, old, new)
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(mod)
        except Exception as e:  # an assertion or a crash both count as caught
            failed.append(check.__name__)
    assert failed, f"planted mistake {name!r} passed every pin"
