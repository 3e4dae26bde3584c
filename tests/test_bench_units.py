"""The algorithmic work the bench divides by, against figures computed independently from the
model shape (the decode bytes per step and prefill FLOPs of each workload, the linear
parameters per layer and the KV bytes per token).

Figures: linear parameters per layer (4096 + 1024 + 3 * 3072) * 1024 = 15,728,640; KV bytes
per token 28 layers * 2 (K, V) * 8 heads * 128 * 2 bytes = 114,688; per decode step 880.8 MB
of linear weights + 311.2 MB of tied head + the K/V rows read and written; per prefill call
2 * N * 440.4 M + the causal half of the attention + the head at the last rows.
"""

import pytest

import bench
from qwen3_decoder_forward_gb300 import synth

S = synth.QWEN3_0P6B


def test_per_layer_and_per_token_constants():
    assert (S.q_dim + 2 * S.kv_dim) * S.hidden + S.hidden * S.q_dim + 3 * S.intermediate * S.hidden == 15_728_640
    assert S.n_layers * 2 * S.kv_dim * 2 == 114_688


@pytest.mark.parametrize("name,gb", [("decode_b1", 1.214), ("decode_b32", 5.07), ("decode_long", 31.29)])
def test_decode_step_bytes(name, gb):
    wl = synth.WORKLOADS[name]
    assert bench.decode_step_bytes(wl) / 1e9 == pytest.approx(gb, rel=2e-3)


def test_decode_b1_step_bytes_split():
    """Batch 1 at contexts 129..256: 72.5% linear weights, 25.6% head, 1.8% K/V."""
    wl = synth.WORKLOADS["decode_b1"]
    total = bench.decode_step_bytes(wl)
    assert 28 * 15_728_640 * 2 / total == pytest.approx(0.725, abs=1e-3)
    assert 151_936 * 1024 * 2 / total == pytest.approx(0.256, abs=1e-3)


@pytest.mark.parametrize("name,tflop", [("prefill_ragged", 28.9), ("decode_b32", 32.7), ("decode_long", 723.5)])
def test_prefill_flops(name, tflop):
    wl = synth.WORKLOADS[name]
    assert bench.prefill_flops(wl) / 1e12 == pytest.approx(tflop, rel=2e-3)


def test_prefill_flops_tiny_by_hand():
    """One layer, 32 tokens: 2*32*15,728,640 + 4*16*128*(32*33/2) + 2*1024*4096."""
    wl = synth.WORKLOADS["tiny"]
    assert list(wl.lengths) == [32]
    assert bench.prefill_flops(wl) == 2 * 32 * 15_728_640 + 4 * 16 * 128 * 528 + 2 * 1024 * 4096
