"""Batched decode at full size: 32 sequences with 1024-token prompts (the KV fill), then 64
greedy steps with B=32.  Sequences 0 and 17 are checked against the oracle, teacher-forced:
their prefill logits, their cached K/V rows on all 28 layers, and every layer, logits and
token of all 64 steps.  The other 30 rows run free on their own greedy tokens."""

import numpy as np
import pytest
import torch

import gpu_common as gc
from oracle import qwen3_oracle as oracle
from qwen3_decoder_forward_gb300 import binding, synth

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS["decode_b32"]
SAMPLED = (0, 17)


def test_decode_b32_sampled_parity():
    gc.ensure_library()
    s = WL.shape
    B = WL.n_seqs
    w = synth.make_weights(s)
    cfg, ow = gc.oracle_config(s), gc.oracle_weights(w)
    prompts = WL.prompts()
    refs = {i: oracle.generate(cfg, ow, prompts[i].tolist(), WL.decode_steps) for i in SAMPLED}
    del ow

    m = binding.Model(s, w, max_seqs=B, max_ctx=WL.max_ctx, max_prefill_tokens=WL.n_prompt_tokens)
    gate = gc.Gate()
    nxt, logits = m.prefill(torch.cat(prompts).cuda(), list(WL.lengths), list(range(B)), want_logits=True)
    for i in SAMPLED:
        r = refs[i]["calls"][0]
        gate.logits(logits[i].cpu().numpy(), r["logits"], f"seq {i} prefill")
        gate.token(int(nxt[i]), r["token"], r["margin"], f"seq {i} prefill")
        for layer in range(s.n_layers):
            k, v = m.kv_rows(layer, i, WL.lengths[i])
            gate.hidden(k.float().cpu().numpy(), refs[i]["cache"].keys(layer)[: WL.lengths[i]], f"seq {i} K l{layer}")
            gate.hidden(v.float().cpu().numpy(), refs[i]["cache"].values(layer)[: WL.lengths[i]], f"seq {i} V l{layer}")

    buf = torch.zeros((s.n_layers + 1) * B * s.hidden, dtype=torch.float32, device="cuda")
    m.set_debug_dump(buf)
    slots = list(range(B))
    slots_d = torch.tensor(slots, dtype=torch.int32, device="cuda")
    lg = torch.zeros(B, s.vocab, dtype=torch.float32, device="cuda")
    cur = nxt.clone()
    for t in range(WL.decode_steps):
        inp = cur.clone()
        for i in SAMPLED:
            inp[i] = refs[i]["fed"][t]
        out = torch.zeros(B, dtype=torch.int32, device="cuda")
        m.decode_step(inp, slots_d, slots, out, lg)
        hid = buf.view(s.n_layers + 1, B, s.hidden)
        for i in SAMPLED:
            r = refs[i]["calls"][t + 1]
            h = hid[:, i].cpu().numpy()
            for layer in range(s.n_layers + 1):
                gate.hidden(h[layer], r["hidden"][layer, 0], f"seq {i} step {t} h_{layer}")
            gate.logits(lg[i].cpu().numpy(), r["logits"], f"seq {i} step {t}")
            gate.token(int(out[i]), r["token"], r["margin"], f"seq {i} step {t}")
        cur = out
    assert m.status() == 0
    for i in range(B):
        assert binding.qwen3_slot_length(m.ctx, i) == WL.lengths[i] + WL.decode_steps
    m.close()
    print(gate.summary())
    gate.check()
    assert gate.tokens_checked >= 20
