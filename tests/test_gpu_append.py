"""Prefill that continues a slot (qwen3_prefill_append): chunked prompts, prompts extended after
decode steps, and packed sequences at different offsets, each checked against the oracle run
with the same cached prefix ("从零开始写Qwen3", Attn: the causal mask of a query block that
follows cached keys; "古法手撕简易LLM推理器", prefill与predict: positions start at the cache
length)."""

import pytest
import torch

import gpu_common as gc
from oracle import qwen3_oracle as oracle
from qwen3_decoder_forward_gb300 import binding, synth

pytestmark = pytest.mark.gpu

TOKEN_SEED = 4242


def _dump(model, shape, n):
    buf = torch.zeros((shape.n_layers + 1) * n * shape.hidden, dtype=torch.float32, device="cuda")
    model.set_debug_dump(buf)
    return buf


def _check_call(gate, shape, buf, rows, ref, logits, token, what, row0=0, n_rows=None):
    """hidden rows row0 .. row0+n_rows-1 of the last call against ref['hidden'] (all its rows)."""
    n = n_rows if n_rows is not None else ref["hidden"].shape[1]
    hid = buf[: (shape.n_layers + 1) * rows * shape.hidden].view(shape.n_layers + 1, rows, shape.hidden)
    hid = hid[:, row0:row0 + n].cpu().numpy()
    for layer in range(shape.n_layers + 1):
        gate.hidden(hid[layer], ref["hidden"][layer], f"{what} h_{layer}")
    gate.logits(logits, ref["logits"], what)
    gate.token(token, ref["token"], ref["margin"], what)


@pytest.fixture(scope="module")
def tiny():
    gc.ensure_library()
    shape = synth.WORKLOADS["tiny"].shape
    w = synth.make_weights(shape)
    return shape, w, gc.oracle_config(shape), gc.oracle_weights(w)


def test_chunked_prompt_then_decode(tiny):
    """A 40-token prompt as chunks of 17, 14 and 9 tokens, then three decode steps; every call
    matches the oracle continuing the same cache, and the chunked rows match a one-call prefill."""
    shape, w, cfg, ow = tiny
    ids = synth.make_tokens(40, shape.vocab, TOKEN_SEED)
    m = binding.Model(shape, w, max_seqs=2, max_ctx=64, max_prefill_tokens=64)
    buf = _dump(m, shape, 40)
    gate = gc.Gate()
    cache = oracle.KVCache(cfg.n_layers)
    start = 0
    for i, n in enumerate((17, 14, 9)):
        chunk = ids[start:start + n]
        ref = oracle.forward(cfg, ow, chunk.tolist(), cache)
        nxt, logits = m.prefill(chunk.cuda(), [n], [1], want_logits=True, append=i > 0)
        _check_call(gate, shape, buf, n, ref, logits[0].cpu().numpy(), int(nxt[0]), f"chunk {i}")
        start += n
        assert binding.qwen3_slot_length(m.ctx, 1) == start
    chunked_last = buf[: (shape.n_layers + 1) * 9 * shape.hidden].view(shape.n_layers + 1, 9, shape.hidden).clone()
    # decode continues the appended slot
    slots_d = torch.tensor([1], dtype=torch.int32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    lg = torch.zeros(1, shape.vocab, dtype=torch.float32, device="cuda")
    fed = int(nxt[0])
    for s in range(3):
        ref = oracle.forward(cfg, ow, [fed], cache)
        tok.fill_(fed)
        m.decode_step(tok, slots_d, [1], out, lg)
        _check_call(gate, shape, buf, 1, ref, lg[0].cpu().numpy(), int(out[0]), f"step {s}")
        fed = int(ref["token"])
    assert binding.qwen3_slot_length(m.ctx, 1) == 43
    # the same 40 tokens in one call (slot 0): the last 9 rows equal the third chunk's rows
    m.prefill(ids.cuda(), [40], [0])
    whole = buf[: (shape.n_layers + 1) * 40 * shape.hidden].view(shape.n_layers + 1, 40, shape.hidden)
    assert gc.rel_l2(chunked_last.cpu().numpy(), whole[:, 31:40].cpu().numpy()) <= 2e-3
    assert m.status() == 0
    m.close()
    print(gate.summary())
    gate.check()


def test_packed_sequences_at_different_offsets(tiny):
    """One append call with three sequences: slot 0 continuing after 30 tokens, slot 3 after 5,
    slot 1 starting empty (offset 0 is an ordinary prefill)."""
    shape, w, cfg, ow = tiny
    m = binding.Model(shape, w, max_seqs=4, max_ctx=96, max_prefill_tokens=96)
    heads = {0: synth.make_tokens(30, shape.vocab, TOKEN_SEED + 1), 3: synth.make_tokens(5, shape.vocab, TOKEN_SEED + 2)}
    caches = {s: oracle.KVCache(cfg.n_layers) for s in (0, 1, 3)}
    for s, t in heads.items():
        oracle.forward(cfg, ow, t.tolist(), caches[s])
        m.prefill(t.cuda(), [t.numel()], [s])
    tails = {0: synth.make_tokens(21, shape.vocab, TOKEN_SEED + 3), 3: synth.make_tokens(40, shape.vocab, TOKEN_SEED + 4),
             1: synth.make_tokens(13, shape.vocab, TOKEN_SEED + 5)}
    order = [0, 3, 1]
    lengths = [tails[s].numel() for s in order]
    N = sum(lengths)
    buf = _dump(m, shape, N)
    nxt, logits = m.prefill(torch.cat([tails[s] for s in order]).cuda(), lengths, order, want_logits=True,
                            append=True)
    gate = gc.Gate()
    row0 = 0
    for b, s in enumerate(order):
        ref = oracle.forward(cfg, ow, tails[s].tolist(), caches[s])
        _check_call(gate, shape, buf, N, ref, logits[b].cpu().numpy(), int(nxt[b]), f"slot {s}", row0=row0,
                    n_rows=lengths[b])
        row0 += lengths[b]
    assert [binding.qwen3_slot_length(m.ctx, s) for s in (0, 1, 3)] == [51, 13, 45]
    assert m.status() == 0
    m.close()
    print(gate.summary())
    gate.check()


def test_append_capacity_error(tiny):
    shape, w, _, _ = tiny
    m = binding.Model(shape, w, max_seqs=1, max_ctx=40, max_prefill_tokens=40)
    ids = synth.make_tokens(40, shape.vocab, TOKEN_SEED)
    m.prefill(ids[:30].cuda(), [30], [0])
    with pytest.raises(binding.Qwen3Error) as e:
        m.prefill(ids[:11].cuda(), [11], [0], append=True)  # 30 + 11 > max_ctx
    assert e.value.code == binding.QWEN3_E_CAPACITY
    m.prefill(ids[30:40].cuda(), [10], [0], append=True)  # exactly max_ctx
    assert binding.qwen3_slot_length(m.ctx, 0) == 40
    assert m.status() == 0
    m.close()


def test_full_model_chunks_across_key_tiles():
    """28 layers: a 300-token prompt as chunks of 130, 100 and 70 tokens, so that the cached
    prefix ends inside a 128-key tile and a chunk's keys span up to three tiles."""
    gc.ensure_library()
    shape = synth.QWEN3_0P6B
    w = synth.make_weights(shape)
    cfg, ow = gc.oracle_config(shape), gc.oracle_weights(w)
    ids = synth.make_tokens(300, shape.vocab, TOKEN_SEED + 6)
    m = binding.Model(shape, w, max_seqs=1, max_ctx=320, max_prefill_tokens=130)
    buf = _dump(m, shape, 130)
    cache = oracle.KVCache(cfg.n_layers)
    gate = gc.Gate()
    start = 0
    for i, n in enumerate((130, 100, 70)):
        chunk = ids[start:start + n]
        ref = oracle.forward(cfg, ow, chunk.tolist(), cache)
        nxt, logits = m.prefill(chunk.cuda(), [n], [0], want_logits=True, append=i > 0)
        _check_call(gate, shape, buf, n, ref, logits[0].cpu().numpy(), int(nxt[0]), f"chunk {i}")
        start += n
    assert binding.qwen3_slot_length(m.ctx, 0) == 300
    assert m.status() == 0
    m.close()
    print(gate.summary())
    gate.check()
