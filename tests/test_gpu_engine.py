"""Continuous batching (qwen3_engine_*): requests queued beyond the slots, prompts longer than
the step budget (chunked prefill), prompt chunks and generated tokens packed into one call,
slots reused after a request finishes, and the end-of-sequence stop.

Every request's generated tokens are checked teacher-forced: the reference is run on the
request alone, fed the engine's own tokens, and wherever its top-1/top-2 logit margin exceeds
0.1 the engine's token must be its argmax (the parity gate's token rule).  On the one-layer
model the reference is the oracle; on the 28-layer model it is the library's own prefill +
decode path on a separate context, which the other parity tests pin to the oracle.
"""

import numpy as np
import pytest
import torch

import gpu_common as gc
from oracle import qwen3_oracle as oracle
from qwen3_decoder_forward_gb300 import binding, synth

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny"].shape
# (prompt length, max new tokens): 6 requests for 3 slots; with a 16-token budget the prompts
# of 20 and 33 tokens run in chunks, and every step after the first mixes chunks with
# generated tokens until the prompts run out.
REQUESTS = [(5, 6), (20, 4), (9, 8), (33, 3), (3, 10), (12, 5)]


@pytest.fixture(scope="module")
def tiny():
    gc.ensure_library()
    w = synth.make_weights(TINY)
    prompts = [synth.make_tokens(n, TINY.vocab, 300 + i).tolist() for i, (n, _) in enumerate(REQUESTS)]
    return w, prompts


def _oracle_check(cfg, ow, prompt, out, what):
    """Teacher-forced oracle run over the engine's tokens; returns (checked, skipped)."""
    ref = oracle.generate(cfg, ow, prompt, len(out) - 1, forced=out[:-1])
    gate = gc.Gate()
    for i, (tok, call) in enumerate(zip(out, ref["calls"])):
        gate.token(tok, call["token"], call["margin"], f"{what} token {i}")
    gate.check()
    return gate.tokens_checked, gate.tokens_skipped


def _run_engine(w, prompts, eos=None, budget=16):
    m = binding.Model(TINY, w, max_seqs=3, max_ctx=64, max_prefill_tokens=48)
    eng = binding.Engine(m, budget)
    for i, (p, (_, n_new)) in enumerate(zip(prompts, REQUESTS)):
        eng.submit(100 + i, p, n_new, -1 if eos is None else eos.get(i, -1))
    steps = eng.run(max_steps=500)
    results = [eng.result(100 + i) for i in range(len(prompts))]
    stats = eng.stats()
    assert eng.unfinished() == 0
    assert m.status() == 0
    eng.close()
    m.close()
    return results, stats, steps


def test_engine_matches_oracle(tiny):
    w, prompts = tiny
    results, stats, steps = _run_engine(w, prompts)
    cfg, ow = gc.oracle_config(TINY), gc.oracle_weights(w)
    checked = 0
    for i, ((out, why), p, (_, n_new)) in enumerate(zip(results, prompts, REQUESTS)):
        assert why == binding.QWEN3_FINISH_LENGTH and len(out) == n_new, (i, why, out)
        checked += _oracle_check(cfg, ow, p, out, f"request {i}")[0]
    assert checked >= 20
    assert stats["prompt_tokens"] == sum(n for n, _ in REQUESTS)
    assert stats["generated_tokens"] == sum(k for _, k in REQUESTS)
    assert stats["mixed_steps"] >= 5 and stats["decode_steps"] >= 1
    assert stats["steps"] == steps == stats["mixed_steps"] + stats["decode_steps"]


def test_engine_stops_at_eos_and_reuses_the_slot(tiny):
    """Request 4 (10 new tokens) gets an eos id equal to a token it generates midway: it must
    stop right there, keep the eos token last, and the other requests still match the oracle."""
    w, prompts = tiny
    first, _, _ = _run_engine(w, prompts)
    out4 = first[4][0]
    # the latest token that is new in the output (token 0 always is); stopping there also
    # frees the slot before the last requests were admitted
    k = [i for i in range(len(out4) - 1) if out4[i] not in out4[:i]][-1]
    results, stats, _ = _run_engine(w, prompts, eos={4: out4[k]})
    out, why = results[4]
    assert why == binding.QWEN3_FINISH_EOS
    assert out[-1] == out4[k] and out4[k] not in out[:-1]
    assert len(out) == k + 1
    cfg, ow = gc.oracle_config(TINY), gc.oracle_weights(w)
    for i, ((o, r), p) in enumerate(zip(results, prompts)):
        if i != 4:
            assert r == binding.QWEN3_FINISH_LENGTH
        _oracle_check(cfg, ow, p, o, f"request {i}")
    assert stats["generated_tokens"] == sum(k2 for _, k2 in REQUESTS) - (REQUESTS[4][1] - (k + 1))


def test_engine_finishes_a_request_whose_slot_is_full(tiny):
    w, _ = tiny
    m = binding.Model(TINY, w, max_seqs=3, max_ctx=40, max_prefill_tokens=48)
    eng = binding.Engine(m, 16)
    eng.submit(1, synth.make_tokens(36, TINY.vocab, 9).tolist(), 50)
    eng.run(max_steps=100)
    out, why = eng.result(1)
    # 36 prompt tokens (chunks of 16, 16, 4), then the first four generated tokens are fed back
    # (slot lengths 37..40); the fifth cannot be appended
    assert why == binding.QWEN3_FINISH_CONTEXT and len(out) == 5
    assert binding.qwen3_slot_length(m.ctx, 0) == 40
    assert m.status() == 0
    eng.close()
    m.close()


def test_engine_argument_errors(tiny):
    w, _ = tiny
    m = binding.Model(TINY, w, max_seqs=3, max_ctx=64, max_prefill_tokens=48)
    for budget in (2, 49):  # below max_seqs, above max_prefill_tokens
        assert binding.qwen3_engine_workspace_bytes(m.ctx, budget) > 0
        with pytest.raises(binding.Qwen3Error):
            binding.Engine(m, budget)
    eng = binding.Engine(m, 16)
    with pytest.raises(binding.Qwen3Error):
        eng.submit(1, [], 4)
    with pytest.raises(binding.Qwen3Error) as e:
        eng.submit(1, [1] * 65, 4)
    assert e.value.code == binding.QWEN3_E_CAPACITY
    eng.submit(1, [1, 2, 3], 2)
    with pytest.raises(binding.Qwen3Error):
        eng.submit(1, [1, 2, 3], 2)
    with pytest.raises(binding.Qwen3Error):
        eng.forget(1)  # not finished yet
    eng.run()
    eng.forget(1)
    with pytest.raises(binding.Qwen3Error):
        eng.result(1)
    eng.close()
    m.close()


def test_engine_full_model_against_direct_path():
    """28 layers: five prompts of 300-700 tokens through 4 slots with a 512-token budget; each
    request's tokens checked teacher-forced against prefill + decode steps of that request alone."""
    gc.ensure_library()
    s = synth.QWEN3_0P6B
    w = synth.make_weights(s)
    lengths = [300, 700, 450, 520, 333]
    n_new = 6
    prompts = [synth.make_tokens(n, s.vocab, 400 + i).tolist() for i, n in enumerate(lengths)]
    m = binding.Model(s, w, max_seqs=4, max_ctx=1024, max_prefill_tokens=512)
    eng = binding.Engine(m, 512)
    for i, p in enumerate(prompts):
        eng.submit(i, p, n_new)
    eng.run(max_steps=200)
    results = [eng.result(i) for i in range(len(prompts))]
    stats = eng.stats()
    assert m.status() == 0
    eng.close()
    m.close()
    assert stats["prompt_tokens"] == sum(lengths) and stats["mixed_steps"] >= 4

    ref = binding.Model(s, w, max_seqs=1, max_ctx=1024, max_prefill_tokens=1024)
    slots = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    lg = torch.zeros(1, s.vocab, dtype=torch.float32, device="cuda")
    checked = 0
    for i, ((out, why), p) in enumerate(zip(results, prompts)):
        assert why == binding.QWEN3_FINISH_LENGTH and len(out) == n_new
        _, logits = ref.prefill(torch.tensor(p, dtype=torch.int32, device="cuda"), [len(p)], [0], want_logits=True)
        rows = [logits[0].cpu().numpy()]
        for t in out[:-1]:
            tok.fill_(int(t))
            ref.decode_step(tok, slots, [0], nxt, lg)
            rows.append(lg[0].cpu().numpy())
        for j, (got, z) in enumerate(zip(out, rows)):
            top2 = np.partition(z, -2)[-2:]
            if top2[1] - top2[0] > gc.MARGIN:
                checked += 1
                assert got == int(np.argmax(z)), f"request {i} token {j}"
    assert ref.status() == 0
    ref.close()
    assert checked >= 10


# (temperature, top_k, top_p, seed) of the sampling requests; None: greedy
SAMPLING = [(1.0, 40, 0.9, 7), None, (0.7, 0, 1.0, 12345678901234567), (1.3, 5, 0.5, 42), None,
            (1.0, 0, 0.95, 2 ** 63 + 5)]


def test_engine_sampling_requests(tiny):
    """Sampling and greedy requests in one engine.  Greedy requests keep matching the oracle's
    greedy tokens (the parity gate's margin rule).  Every token a sampling request gets is the
    oracle sampler's draw -- with the request's temperature / top-k / top-p and the uniform of
    its own token index from its own seed (SplitMix64) -- from the logits of its row in the step
    that produced it (qwen3_engine_last_step), token-exact except where the fp32 draw sits
    within 1e-5 of a boundary of the cumulative distribution (the rule of the sampler tests)."""
    w, prompts = tiny
    cfg, ow = gc.oracle_config(TINY), gc.oracle_weights(w)
    m = binding.Model(TINY, w, max_seqs=3, max_ctx=64, max_prefill_tokens=48)
    eng = binding.Engine(m, 16)
    ids = {}
    for i, (p, (_, n_new)) in enumerate(zip(prompts, REQUESTS)):
        s = SAMPLING[i]
        ids[200 + i] = i
        if s:
            eng.submit(200 + i, p, n_new, temperature=s[0], top_k=s[1], top_p=s[2], seed=s[3])
        else:
            eng.submit(200 + i, p, n_new)
    checked, near = 0, 0
    seen = {rid: 0 for rid in ids}
    steps = 0
    while eng.unfinished() and steps < 500:
        eng.step()
        steps += 1
        rows, logits = eng.last_step()
        lg = logits.cpu().numpy() if logits is not None else None
        for r, rid in enumerate(rows):
            toks, _ = eng.result(rid)
            if len(toks) == seen[rid]:
                continue  # a prompt chunk that did not end the prompt
            t = len(toks) - 1
            seen[rid] = len(toks)
            s = SAMPLING[ids[rid]]
            if s is None:
                continue
            assert lg is not None
            T, k, p, seed = s
            u = gc.splitmix64_draw(seed, t)
            drawn = oracle.sample(lg[r], T, k, p, u)
            if toks[t] != drawn:
                alt = {oracle.sample(lg[r], T, k, p, min(max(u + d, 0.0), 1.0 - 2 ** -24)) for d in (-1e-5, 1e-5)}
                assert toks[t] in alt, (rid, t, toks[t], drawn)
                near += 1
            checked += 1
    results = [eng.result(200 + i) for i in range(len(prompts))]
    assert m.status() == 0
    eng.close()
    m.close()
    for i, ((toks, why), s) in enumerate(zip(results, SAMPLING)):
        assert len(toks) == REQUESTS[i][1] and why == binding.QWEN3_FINISH_LENGTH
        if s is None:
            _oracle_check(cfg, ow, prompts[i], toks, f"greedy request {i}")
    assert checked == sum(REQUESTS[i][1] for i, s in enumerate(SAMPLING) if s) and near <= 1
