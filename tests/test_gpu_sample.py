"""qwen3_sample against the oracle's sampler ("第 3 章", 4.3 Sampler; "手写Qwen3-0.6B推理",
softmax with a temperature) on seeded logits: greedy rows, temperature, Top-k, Top-p and their
combinations, ties at the candidate boundary, vocabularies below, at and above the candidate
count, and flat rows where only the index order decides.

The candidate set and its order are decided on the fp32 logits on both sides, so they agree
exactly.  The probabilities are fp32 in the kernel and fp64 in the oracle: a draw whose target
lies within about 1e-6 (relative) of a cumulative boundary may pick the neighbouring token.
Such a draw is accepted only when the oracle itself picks the GPU's token after moving u or
top_p by 1e-5, and at most 2% of the rows may need that.
"""

import numpy as np
import pytest
import torch

import gpu_common as gc
from oracle import qwen3_oracle as oracle
from qwen3_decoder_forward_gb300 import binding, synth

pytestmark = pytest.mark.gpu

DELTA = 1e-5


def _oracle(row, T, k, p, u):
    return oracle.sample(row, float(T), int(k), float(p), float(u))


def _gpu(logits, temperature, top_k, top_p, uniform):
    out = binding.sample(logits.cuda(), temperature.cuda(), top_k.cuda(), top_p.cuda(), uniform.cuda())
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _compare(logits, temperature, top_k, top_p, uniform):
    got = _gpu(logits, temperature, top_k, top_p, uniform)
    rows = logits.double().numpy()
    exact, boundary, bad = 0, 0, []
    for b in range(logits.shape[0]):
        T, k, p, u = float(temperature[b]), int(top_k[b]), float(top_p[b]), float(uniform[b])
        want = _oracle(rows[b], T, k, p, u)
        if int(got[b]) == want:
            exact += 1
            continue
        near = {_oracle(rows[b], T, k, min(p * (1 + dp), 1.0) if p < 1 else p, min(max(u + du, 0.0), 1 - 1e-12))
                for du in (-DELTA, DELTA) for dp in (-DELTA, 0.0, DELTA)}
        if T > 0 and int(got[b]) in near:
            boundary += 1
        else:
            bad.append((b, T, k, p, u, int(got[b]), want))
    assert not bad, f"rows that differ from the oracle: {bad[:5]}"
    assert boundary <= max(1, int(0.02 * logits.shape[0])), (exact, boundary)
    return exact, boundary


@pytest.fixture(scope="module", autouse=True)
def lib():
    gc.ensure_library()


@pytest.mark.parametrize("B,V,grid", [
    (64, 151936, 0.0),     # the Qwen3 vocabulary
    (32, 151936, 0.25),    # coarse logits: long runs of ties at the candidate boundary
    (16, 1000, 0.0),       # fewer tokens than candidates
    (16, 1024, 0.5),       # exactly the candidate count
    (16, 1025, 0.5),       # one more
    (8, 5, 0.0),
    (8, 4099, 0.0),        # ragged against the 1024-thread stride
])
def test_sample_matches_oracle(B, V, grid):
    inputs = synth.make_sampling_batch(B, V, seed=synth.SAMPLE_SEED + V, grid=grid)
    exact, boundary = _compare(*inputs)
    print(f"B={B} V={V} grid={grid}: exact {exact}, boundary {boundary}")


def test_many_draws_of_one_row():
    """2048 draws from one row on a grid of u, for three settings: every draw matches the oracle,
    so the draw frequencies are the oracle's kept probabilities."""
    V, n = 32768, 2048
    base = synth.make_sampling_batch(1, V, seed=synth.SAMPLE_SEED + 1, spikes=16)[0]
    logits = base.expand(n, V).contiguous()
    uniform = (torch.arange(n, dtype=torch.float32) + 0.5) / n
    for T, k, p in ((1.0, 0, 1.0), (0.7, 40, 1.0), (1.2, 0, 0.9)):
        _compare(logits, torch.full((n,), T), torch.full((n,), k, dtype=torch.int32), torch.full((n,), p), uniform)


def test_flat_rows_draw_by_index():
    """All logits equal: the candidates are tokens 0..1023 and the draw is floor(u * 1024)."""
    V = 151936
    u = torch.tensor([0.0, 0.5, 0.99999, 0.2503, 0.75], dtype=torch.float32)
    B = u.numel()
    got = _gpu(torch.zeros(B, V), torch.ones(B), torch.zeros(B, dtype=torch.int32), torch.ones(B), u)
    assert got.tolist() == [0, 512, 1023, 256, 768]
    # top_k = 10 keeps tokens 0..9
    got = _gpu(torch.zeros(B, V), torch.ones(B), torch.full((B,), 10, dtype=torch.int32), torch.ones(B), u)
    assert got.tolist() == [0, 5, 9, 2, 7]


def test_greedy_rows_take_lowest_index_of_the_maximum():
    V = 151936
    logits = synth.make_sampling_batch(4, V, seed=synth.SAMPLE_SEED + 2)[0]
    top = logits.max(dim=1).values
    logits[0, 7] = top[0]            # a tie before the original maximum
    logits[1, V - 1] = top[1]        # a tie at the end
    logits[2, :] = -1.0              # all equal
    got = _gpu(logits, torch.zeros(4), torch.zeros(4, dtype=torch.int32), torch.ones(4), torch.full((4,), 0.5))
    want = [oracle.greedy(r)[0] for r in logits.double().numpy()]
    assert got.tolist() == want
    assert want[2] == 0


def test_zero_temperature_repeats_the_decode_choice():
    """Sampling at temperature 0 from the logits a decode step writes returns the token the
    step chose itself (lm_head + argmax)."""
    shape = synth.WORKLOADS["tiny"].shape
    m = binding.Model(shape, synth.make_weights(shape), max_seqs=4, max_ctx=32, max_prefill_tokens=32)
    ids = synth.make_tokens(24, shape.vocab, 77)
    m.prefill(ids.cuda(), [6, 8, 10], [0, 1, 2])
    tok = torch.tensor([3, 4, 5], dtype=torch.int32, device="cuda")
    slots = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    out = torch.zeros(3, dtype=torch.int32, device="cuda")
    lg = torch.zeros(3, shape.vocab, dtype=torch.float32, device="cuda")
    m.decode_step(tok, slots, [0, 1, 2], out, lg)
    z = binding.sample(lg, torch.zeros(3, device="cuda"), torch.zeros(3, dtype=torch.int32, device="cuda"),
                       torch.ones(3, device="cuda"), torch.full((3,), 0.5, device="cuda"))
    torch.cuda.synchronize()
    assert z.tolist() == out.tolist()
    assert m.status() == 0
    m.close()


def test_rejects_bad_arguments():
    x = torch.zeros(2, 8, device="cuda")
    f = torch.zeros(2, device="cuda")
    k = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.Qwen3Error) as e:
        binding.qwen3_sample(x.data_ptr(), 0, 8, f.data_ptr(), k.data_ptr(), f.data_ptr(), f.data_ptr(),
                             k.data_ptr())
    assert e.value.code == binding.QWEN3_E_INVALID
    with pytest.raises(binding.Qwen3Error):
        binding.qwen3_sample(x.data_ptr(), 2, 8, 0, k.data_ptr(), f.data_ptr(), f.data_ptr(), k.data_ptr())


@pytest.mark.parametrize("flags,B", [(0, 4), (binding.QWEN3_FLAG_NO_GRAPH, 4), (0, 1)])
def test_context_sampling_draws_from_the_logits_of_each_call(flags, B):
    """With qwen3_set_sampling on, prefill and decode steps (graph replay, one launch per kernel,
    and one row on the two-kernel layer) return the qwen3_sample draw from the logits they wrote:
    the same token as a separate qwen3_sample call on those logits, and the oracle's draw from
    them.  The uniform draws are rewritten between steps in stream order and the graphs see the
    new ones; clearing the setting returns to the argmax."""
    shape = synth.WORKLOADS["tiny"].shape
    n_steps = 5
    m = binding.Model(shape, synth.make_weights(shape), max_seqs=B, max_ctx=64, max_prefill_tokens=64,
                      flags=flags)
    rows = slice(4 - B, 4)  # one row: the temperature-1.3 row
    temperature = torch.tensor([0.0, 0.8, 1.0, 1.3], device="cuda")[rows].contiguous()
    top_k = torch.tensor([0, 40, 0, 0], dtype=torch.int32, device="cuda")[rows].contiguous()
    top_p = torch.tensor([1.0, 1.0, 0.9, 1.0], device="cuda")[rows].contiguous()
    uniform = torch.zeros(B, device="cuda")
    g = torch.Generator().manual_seed(synth.SAMPLE_SEED + 11)
    m.set_sampling(temperature, top_k, top_p, uniform)
    lengths = [5, 9, 7, 11][rows]
    ids = synth.make_tokens(sum(lengths), shape.vocab, 78)

    def check(next_tok, logits, what):
        torch.cuda.synchronize()
        again = binding.sample(logits, temperature, top_k, top_p, uniform)
        torch.cuda.synchronize()
        assert next_tok.tolist() == again.tolist(), what
        _compare(logits.cpu(), temperature.cpu(), top_k.cpu(), top_p.cpu(), uniform.cpu())

    uniform.copy_(torch.rand(B, generator=g))
    with pytest.raises(binding.Qwen3Error) as e:
        m.prefill(ids.cuda(), lengths, list(range(B)))
    assert e.value.code == binding.QWEN3_E_INVALID
    nxt, lg = m.prefill(ids.cuda(), lengths, list(range(B)), want_logits=True)
    check(nxt, lg, "prefill")
    slots_d = torch.arange(B, dtype=torch.int32, device="cuda")
    tok = nxt.clone()
    out = torch.zeros(B, dtype=torch.int32, device="cuda")
    logits = torch.zeros(B, shape.vocab, device="cuda")
    drawn = []
    for step in range(n_steps):
        uniform.copy_(torch.rand(B, generator=g))
        m.decode_step(tok, slots_d, list(range(B)), out, logits)
        check(out, logits, f"decode step {step}")
        drawn.append(out.tolist())
        tok.copy_(out)
    # different draws give different tokens somewhere in the sampled rows
    assert len({tuple(r[-3:]) for r in drawn}) > 1
    m.set_sampling()
    m.decode_step(tok, slots_d, list(range(B)), out, logits)
    torch.cuda.synchronize()
    assert out.tolist() == [oracle.greedy(r)[0] for r in logits.double().cpu().numpy()]
    assert m.status() == 0
    m.close()
