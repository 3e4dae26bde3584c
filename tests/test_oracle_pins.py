"""The CPU oracle against closed forms, invariants and independent library routines."""

import json
import os

import pytest

from oracle import qwen3_oracle as oracle
import oracle_pins
from qwen3_decoder_forward_gb300 import synth


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(oracle)


def test_hyperparameters_match_pages():
    """The synthetic model's shapes are the ones the pages print for Qwen3-0.6B."""
    with open(os.path.join(os.path.dirname(__file__), "golden", "qwen3_0p6b_hyperparameters.json")) as f:
        g = json.load(f)
    s = synth.QWEN3_0P6B
    assert s.n_layers == g["num_hidden_layers"]
    assert s.hidden == g["hidden_size"]
    assert s.n_q_heads == g["num_attention_heads"]
    assert s.n_kv_heads == g["num_key_value_heads"]
    assert s.head_dim == g["head_dim"]
    assert s.intermediate == g["intermediate_size"]
    assert s.vocab == g["vocab_size"]
    assert s.rms_eps == g["rms_norm_eps"]
    assert s.rope_theta == g["rope_theta"]
    names = {"in_norm": "input_layernorm", "post_norm": "post_attention_layernorm",
             "q_norm": "self_attn.q_norm", "k_norm": "self_attn.k_norm", "wq": "self_attn.q_proj",
             "wk": "self_attn.k_proj", "wv": "self_attn.v_proj", "wo": "self_attn.o_proj",
             "wgate": "mlp.gate_proj", "wup": "mlp.up_proj", "wdown": "mlp.down_proj"}
    shapes = synth.layer_param_shapes(s)
    for k, name in names.items():
        assert list(shapes[k]) == g["layer_tensor_shapes"][name], k


def test_synthetic_weights_are_seeded_and_bf16():
    s = synth.QWEN3_TINY
    a = synth.make_weights(s)
    b = synth.make_weights(s)
    import torch
    assert a["embed"].dtype == torch.bfloat16
    assert list(a["embed"].shape) == [s.vocab, s.hidden]
    assert torch.equal(a["layers"][0]["wq"], b["layers"][0]["wq"])
    assert abs(float(a["layers"][0]["wgate"].float().std()) - 0.02) < 1e-3
    assert abs(float(a["layers"][0]["in_norm"].float().mean()) - 1.0) < 1e-2
    assert not torch.equal(a["layers"][0]["wk"], a["layers"][0]["wv"])


def test_ragged_lengths_in_range():
    w = synth.WORKLOADS["prefill_ragged"]
    assert len(w.lengths) == 8
    assert all(512 <= n <= 4096 for n in w.lengths)
