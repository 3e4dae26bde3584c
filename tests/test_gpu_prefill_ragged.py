"""Ragged prefill at full size: 8 sequences with lengths drawn from [512, 4096], packed into
one [N, C] batch with cu_seqlens.  Sequence 1 (2,024 tokens, packed after sequence 0) and
sequence 7 (4,032 tokens, the longest, packed last) are checked against the oracle on every
layer of every row and on their last-row logits.  Every sequence is then prefilled alone, and
the packed results must equal those (packing changes nothing)."""

import numpy as np
import pytest
import torch

import gpu_common as gc
from oracle import qwen3_oracle as oracle
from qwen3_decoder_forward_gb300 import binding, synth

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS["prefill_ragged"]
SAMPLED = (1, 7)


def test_prefill_ragged_parity_and_packing():
    gc.ensure_library()
    s = WL.shape
    B, N = WL.n_seqs, WL.n_prompt_tokens
    w = synth.make_weights(s)
    prompts = WL.prompts()
    refs = dict(zip(SAMPLED, gc.oracle_prefills(s, [prompts[i].tolist() for i in SAMPLED])))

    m = binding.Model(s, w, max_seqs=B, max_ctx=max(WL.lengths), max_prefill_tokens=N)
    cu = synth.cu_seqlens(list(WL.lengths))
    dump = torch.zeros((s.n_layers + 1) * N * s.hidden, dtype=torch.float32, device="cuda")
    m.set_debug_dump(dump)
    nxt, logits = m.prefill(torch.cat(prompts).cuda(), list(WL.lengths), list(range(B)), want_logits=True)
    gate = gc.Gate()
    for i in SAMPLED:
        ref = refs[i]
        hid = dump.view(s.n_layers + 1, N, s.hidden)[:, cu[i]: cu[i + 1]].cpu().numpy()
        for layer in range(s.n_layers + 1):
            gate.hidden(hid[layer], ref["hidden"][layer], f"seq {i} h_{layer}")
        gate.logits(logits[i].cpu().numpy(), ref["logits"], f"seq {i}")
        gate.token(int(nxt[i]), ref["token"], ref["margin"], f"seq {i}")
    m.set_debug_dump(None)
    del dump
    print(gate.summary())
    gate.check()

    packed_logits = logits.cpu().numpy()
    packed_next = nxt.cpu().numpy()
    for i in range(B):
        n1, l1 = m.prefill(prompts[i].cuda(), [WL.lengths[i]], [i], want_logits=True)
        assert gc.rel_l2(l1[0].cpu().numpy(), packed_logits[i]) <= 1e-6, f"sequence {i}: packed != alone"
        assert int(n1[0]) == int(packed_next[i])
    assert m.status() == 0
    m.close()
