"""Long-context decode at full size: 16 sequences prefilled with 16384 seeded tokens each
(about 30 GB of bf16 KV cache), then 32 greedy steps with B=16.

The oracle cannot redo a 16384-token prefill in a test, so sequence 5 is checked in two
ways that hold at any size:
 * causality: the K/V rows 0..1023 the GPU cached for it equal the oracle's prefill of its
   first 1024 tokens, on every layer;
 * cache consistency: the oracle continues from the GPU's own cached rows (copied to the
   host) and is teacher-forced with the GPU over all 32 steps: every layer, logits, token.
"""

import numpy as np
import pytest
import torch

import gpu_common as gc
from oracle import qwen3_oracle as oracle
from qwen3_decoder_forward_gb300 import binding, synth

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS["decode_long"]
SAMPLED = 5
PREFIX = 1024


def test_decode_long_sampled_parity():
    gc.ensure_library()
    s = WL.shape
    B = WL.n_seqs
    w = synth.make_weights(s)
    cfg, ow = gc.oracle_config(s), gc.oracle_weights(w)
    prompts = WL.prompts()

    m = binding.Model(s, w, max_seqs=B, max_ctx=WL.max_ctx, max_prefill_tokens=2 * WL.lengths[0])
    nxt = torch.zeros(B, dtype=torch.int32, device="cuda")
    for j in range(0, B, 2):
        n2, _ = m.prefill(torch.cat(prompts[j: j + 2]).cuda(), list(WL.lengths[j: j + 2]), [j, j + 1])
        nxt[j: j + 2] = n2
    assert m.status() == 0

    gate = gc.Gate()
    pre = oracle.KVCache(s.n_layers)
    oracle.forward(cfg, ow, prompts[SAMPLED][:PREFIX].tolist(), pre)
    for layer in range(s.n_layers):
        k, v = m.kv_rows(layer, SAMPLED, PREFIX)
        gate.hidden(k.float().cpu().numpy(), pre.keys(layer), f"prefix K l{layer}")
        gate.hidden(v.float().cpu().numpy(), pre.values(layer), f"prefix V l{layer}")
    del pre

    n = WL.lengths[SAMPLED]
    ks, vs = [], []
    for layer in range(s.n_layers):
        k, v = m.kv_rows(layer, SAMPLED, n)
        ks.append(k.float().cpu().numpy())
        vs.append(v.float().cpu().numpy())
    cache = oracle.KVCache.from_arrays(ks, vs, spare=WL.decode_steps)
    del ks, vs

    buf = torch.zeros((s.n_layers + 1) * B * s.hidden, dtype=torch.float32, device="cuda")
    m.set_debug_dump(buf)
    slots = list(range(B))
    slots_d = torch.tensor(slots, dtype=torch.int32, device="cuda")
    lg = torch.zeros(B, s.vocab, dtype=torch.float32, device="cuda")
    cur = nxt.clone()
    feed = int(nxt[SAMPLED])
    for t in range(WL.decode_steps):
        r = oracle.forward(cfg, ow, [feed], cache)
        inp = cur.clone()
        inp[SAMPLED] = feed
        out = torch.zeros(B, dtype=torch.int32, device="cuda")
        m.decode_step(inp, slots_d, slots, out, lg)
        h = buf.view(s.n_layers + 1, B, s.hidden)[:, SAMPLED].cpu().numpy()
        for layer in range(s.n_layers + 1):
            gate.hidden(h[layer], r["hidden"][layer, 0], f"step {t} h_{layer}")
        gate.logits(lg[SAMPLED].cpu().numpy(), r["logits"], f"step {t}")
        gate.token(int(out[SAMPLED]), r["token"], r["margin"], f"step {t}")
        feed = r["token"]
        cur = out
    assert m.status() == 0
    m.close()
    print(gate.summary())
    gate.check()
