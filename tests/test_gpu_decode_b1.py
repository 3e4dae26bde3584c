"""The 28-layer Qwen3-0.6B shape (random weights): a 128-token prompt and 128 greedy decode
steps on one sequence, teacher-forced; every layer of every call and the logits are checked
against the oracle."""

import pytest
import torch

import gpu_common as gc
from oracle import qwen3_oracle as oracle
from qwen3_decoder_forward_gb300 import binding, synth

pytestmark = pytest.mark.gpu

WL = synth.WORKLOADS["decode_b1"]


@pytest.fixture(scope="module")
def setup():
    gc.ensure_library()
    s = WL.shape
    w = synth.make_weights(s)
    prompt = WL.prompts()[0]
    ref = oracle.generate(gc.oracle_config(s), gc.oracle_weights(w), prompt.tolist(), WL.decode_steps)
    return w, prompt, ref


@pytest.mark.parametrize("flags", [0, binding.QWEN3_FLAG_DECODE_CHAIN], ids=["layer", "chain"])
def test_decode_b1_teacher_forced_parity(setup, flags):
    """Decode steps as two kernels per layer (the default) and as the four-kernel chain."""
    w, prompt, ref = setup
    s = WL.shape
    m = binding.Model(s, w, max_seqs=1, max_ctx=WL.max_ctx, max_prefill_tokens=WL.lengths[0], flags=flags)
    n = prompt.numel()
    buf = torch.zeros((s.n_layers + 1) * n * s.hidden, dtype=torch.float32, device="cuda")
    m.set_debug_dump(buf)
    gate = gc.Gate()
    nxt, logits = m.prefill(prompt.cuda(), [n], [0], want_logits=True)
    r = ref["calls"][0]
    hid = buf.view(s.n_layers + 1, n, s.hidden).cpu().numpy()
    for layer in range(s.n_layers + 1):
        gate.hidden(hid[layer], r["hidden"][layer], f"prefill h_{layer}")
    gate.logits(logits[0].cpu().numpy(), r["logits"], "prefill")
    gate.token(int(nxt[0]), r["token"], r["margin"], "prefill")

    slots_d = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    lg = torch.zeros(1, s.vocab, dtype=torch.float32, device="cuda")
    for i, t in enumerate(ref["fed"]):
        tok.fill_(int(t))
        m.decode_step(tok, slots_d, [0], nxt, lg)
        r = ref["calls"][i + 1]
        hid = buf[: (s.n_layers + 1) * s.hidden].view(s.n_layers + 1, 1, s.hidden).cpu().numpy()
        for layer in range(s.n_layers + 1):
            gate.hidden(hid[layer], r["hidden"][layer], f"step {i} h_{layer}")
        gate.logits(lg[0].cpu().numpy(), r["logits"], f"step {i}")
        gate.token(int(nxt[0]), r["token"], r["margin"], f"step {i}")
    assert m.status() == 0
    m.close()
    print(gate.summary())
    gate.check()
    assert gate.tokens_checked >= 32
