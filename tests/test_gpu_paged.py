"""Paged KV cache (kv_block_tokens > 0): blocks of a shared pool, taken as slots grow.

The paged and the contiguous cache run the same kernels on the same values; only where a
cache row lives differs.  So after a prefill every K/V row of every slot is bit-identical
between the two layouts, and decode steps agree to the last bits of the decode MLP's
unordered fp32 atomics (logits within 1e-3, the bound of the graph-vs-direct test).  On
the one-layer model the paged run is also checked against the oracle with the parity gate.
Lengths are chosen so that prefill and decode both cross block boundaries, and the pool
hands blocks out in an order unrelated to the slots (the highest block first).
"""

import numpy as np
import pytest
import torch

import gpu_common as gc
from oracle import qwen3_oracle as oracle
from qwen3_decoder_forward_gb300 import binding, synth

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny"].shape
BS = 128


def _prefill_and_decode(m, prompts, slots, fed, want_logits=True):
    """Prefill `prompts` into `slots`, then one decode step per row of `fed` (tokens per slot).
    Returns the prefill logits and the logits of every step (numpy)."""
    toks = torch.cat([p for p in prompts]).cuda()
    _, lg0 = m.prefill(toks, [p.numel() for p in prompts], slots, want_logits=True)
    out = [lg0.cpu().numpy()]
    B = len(slots)
    slots_d = torch.tensor(slots, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    lg = torch.zeros(B, m.shape.vocab, device="cuda")
    for row in fed:
        m.decode_step(torch.tensor(row, dtype=torch.int32, device="cuda"), slots_d, slots, nxt, lg)
        out.append(lg.cpu().numpy())
    torch.cuda.synchronize()
    return out


def test_paged_tiny_matches_contiguous_and_oracle():
    gc.ensure_library()
    w = synth.make_weights(TINY)
    lengths = [250, 120, 380]  # 2 + 1 + 3 blocks; 30 steps cross 256, 128 and 384
    steps = 30
    prompts = [synth.make_tokens(n, TINY.vocab, 500 + i) for i, n in enumerate(lengths)]
    fed = synth.make_tokens(steps * 3, TINY.vocab, 510).view(steps, 3).tolist()
    slots = [2, 0, 1]
    paged = binding.Model(TINY, w, max_seqs=3, max_ctx=512, max_prefill_tokens=1024,
                          kv_block_tokens=BS, kv_pool_blocks=10)
    flat = binding.Model(TINY, w, max_seqs=3, max_ctx=512, max_prefill_tokens=1024)
    assert paged.kv_free_blocks() == 10 and flat.kv_free_blocks() == -1
    with pytest.raises(binding.Qwen3Error) as e:
        binding.qwen3_kv_view(paged.ctx, 0, 0)
    assert e.value.code == binding.QWEN3_E_UNSUPPORTED

    # prefill: every cached row bit-identical
    toks = torch.cat(prompts).cuda()
    _, lp = paged.prefill(toks, lengths, slots, want_logits=True)
    _, lf = flat.prefill(toks, lengths, slots, want_logits=True)
    assert paged.kv_free_blocks() == 10 - 6
    assert torch.equal(lp, lf)
    for s, n in zip(slots, lengths):
        kp, vp = paged.kv_copy(0, s, 0, n)
        kf, vf = flat.kv_copy(0, s, 0, n)
        assert torch.equal(kp, kf) and torch.equal(vp, vf), f"slot {s}"

    # decode steps across block boundaries
    slots_d = torch.tensor(slots, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(3, dtype=torch.int32, device="cuda")
    gp = torch.zeros(3, TINY.vocab, device="cuda")
    gf = torch.zeros_like(gp)
    paged_logits = [lp.cpu().numpy()]
    for row in fed:
        t = torch.tensor(row, dtype=torch.int32, device="cuda")
        paged.decode_step(t, slots_d, slots, nxt, gp)
        flat.decode_step(t, slots_d, slots, nxt, gf)
        torch.cuda.synchronize()
        assert gc.rel_l2(gp.cpu().numpy(), gf.cpu().numpy()) <= 1e-3
        paged_logits.append(gp.cpu().numpy())
    assert paged.kv_free_blocks() == 10 - 9
    for s, n in zip(slots, lengths):
        assert binding.qwen3_slot_length(paged.ctx, s) == n + steps
        kp, vp = paged.kv_copy(0, s, 0, n + steps)
        kf, vf = flat.kv_copy(0, s, 0, n + steps)
        assert torch.equal(kp[:n], kf[:n]) and torch.equal(vp[:n], vf[:n])
        assert gc.rel_l2(kp.float().cpu().numpy(), kf.float().cpu().numpy()) <= 1e-3
        assert gc.rel_l2(vp.float().cpu().numpy(), vf.float().cpu().numpy()) <= 1e-3
    assert paged.status() == 0 and flat.status() == 0
    paged.close()
    flat.close()

    # the paged run against the oracle, teacher-forced, every call of every sequence
    cfg, ow = gc.oracle_config(TINY), gc.oracle_weights(w)
    gate = gc.Gate()
    for b, p in enumerate(prompts):
        ref = oracle.generate(cfg, ow, p.tolist(), steps, forced=[row[b] for row in fed])
        for i, call in enumerate(ref["calls"]):
            gate.logits(paged_logits[i][b], call["logits"], f"seq {b} call {i}")
            gate.token(int(np.argmax(paged_logits[i][b])), call["token"], call["margin"], f"seq {b} call {i}")
    print(gate.summary())
    gate.check()


def test_paged_pool_exhaustion_and_release():
    gc.ensure_library()
    w = synth.make_weights(TINY)
    m = binding.Model(TINY, w, max_seqs=3, max_ctx=512, max_prefill_tokens=512, kv_block_tokens=BS,
                      kv_pool_blocks=4)
    m.prefill(synth.make_tokens(300, TINY.vocab, 1).cuda(), [300], [0])  # 3 blocks
    assert m.kv_free_blocks() == 1
    with pytest.raises(binding.Qwen3Error) as e:
        m.prefill(synth.make_tokens(200, TINY.vocab, 2).cuda(), [200], [1])  # 2 blocks
    assert e.value.code == binding.QWEN3_E_CAPACITY
    assert m.kv_free_blocks() == 1 and binding.qwen3_slot_length(m.ctx, 1) == 0
    # restarting slot 0 with a longer prompt gives its blocks back first
    m.prefill(synth.make_tokens(400, TINY.vocab, 3).cuda(), [400], [0])  # 4 blocks
    assert m.kv_free_blocks() == 0
    binding.qwen3_release_slot(m.ctx, 0, 0)
    assert m.kv_free_blocks() == 4
    m.prefill(synth.make_tokens(200, TINY.vocab, 2).cuda(), [200], [1])
    assert m.kv_free_blocks() == 2
    # decode across 256 takes one more block
    slots_d = torch.tensor([1], dtype=torch.int32, device="cuda")
    tok = torch.tensor([5], dtype=torch.int32, device="cuda")
    for _ in range(57):
        m.decode_step(tok, slots_d, [1], tok)
    assert binding.qwen3_slot_length(m.ctx, 1) == 257 and m.kv_free_blocks() == 1
    assert m.status() == 0
    m.close()


def test_engine_on_a_paged_cache():
    """The continuous-batching engine over a paged context whose pool holds fewer blocks than
    slots * max_ctx: requests finish and give their blocks back; tokens pass the oracle gate."""
    gc.ensure_library()
    w = synth.make_weights(TINY)
    m = binding.Model(TINY, w, max_seqs=3, max_ctx=512, max_prefill_tokens=256, kv_block_tokens=BS,
                      kv_pool_blocks=5)
    eng = binding.Engine(m, 64)
    reqs = [(200, 6), (90, 8), (140, 5), (30, 12)]
    prompts = [synth.make_tokens(n, TINY.vocab, 520 + i).tolist() for i, (n, _) in enumerate(reqs)]
    for i, (p, (_, k)) in enumerate(zip(prompts, reqs)):
        eng.submit(i, p, k)
    eng.run(max_steps=500)
    cfg, ow = gc.oracle_config(TINY), gc.oracle_weights(w)
    for i, (p, (_, k)) in enumerate(zip(prompts, reqs)):
        out, why = eng.result(i)
        assert why == binding.QWEN3_FINISH_LENGTH and len(out) == k
        ref = oracle.generate(cfg, ow, p, len(out) - 1, forced=out[:-1])
        gate = gc.Gate()
        for j, (tok, call) in enumerate(zip(out, ref["calls"])):
            gate.token(tok, call["token"], call["margin"], f"request {i} token {j}")
        gate.check()
    assert m.status() == 0
    eng.close()
    # every request has finished; the slots still hold their last blocks until reused
    m.close()


def test_paged_full_model_matches_contiguous():
    """28 layers, 6 sequences of 600-1,100 tokens in 256-token blocks, 12 decode steps."""
    gc.ensure_library()
    s = synth.QWEN3_0P6B
    w = synth.make_weights(s)
    lengths = [600, 1100, 767, 1024, 900, 640]
    steps = 12
    prompts = [synth.make_tokens(n, s.vocab, 530 + i) for i, n in enumerate(lengths)]
    fed = synth.make_tokens(steps * 6, s.vocab, 540).view(steps, 6).tolist()
    slots = [5, 0, 3, 1, 4, 2]
    blocks = sum((n + steps + 255) // 256 for n in lengths)
    paged = binding.Model(s, w, max_seqs=6, max_ctx=1280, max_prefill_tokens=sum(lengths), kv_block_tokens=256,
                          kv_pool_blocks=blocks)
    a = _prefill_and_decode(paged, prompts, slots, fed)
    kp, vp = paged.kv_copy(27, 0, 0, 1100 + steps)
    assert paged.kv_free_blocks() == 0 and paged.status() == 0
    paged.close()
    flat = binding.Model(s, w, max_seqs=6, max_ctx=1280, max_prefill_tokens=sum(lengths))
    b = _prefill_and_decode(flat, prompts, slots, fed)
    kf, vf = flat.kv_copy(27, 0, 0, 1100 + steps)
    assert flat.status() == 0
    flat.close()
    assert np.array_equal(a[0], b[0])  # prefill: the same arithmetic, deterministic
    assert torch.equal(kp[:1100], kf[:1100]) and torch.equal(vp[:1100], vf[:1100])
    for x, y in zip(a[1:], b[1:]):
        assert gc.rel_l2(x, y) <= 1e-3
