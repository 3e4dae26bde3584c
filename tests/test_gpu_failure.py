"""Failure detection without a fault: a bounded wait that runs out reports an error status.

Every wait of a decode kernel on an asynchronous copy is bounded.  The test shortens the
limit to one SM cycle (qwen3_set_wait_limit), so the waits on copies issued just before
give up for real inside the kernels of a decode step of nine rows (tensor-core projections
and head, split-KV attention).  Nothing traps or hangs: the kernels record the timeout in
the device error word, let their copies land and return.  qwen3_get_status must report it
(E_DEVICE, with the reason); the greedy tokens of that call are -1 (invalid).  With the
default limit back, the same context is rewound to before the failed step
(qwen3_truncate_slot) and the step is taken again, and a fresh context runs the same
step: both match the oracle.
"""

import pytest
import torch

import gpu_common as gc
from oracle import qwen3_oracle as oracle
from qwen3_decoder_forward_gb300 import binding, synth

pytestmark = pytest.mark.gpu

S = synth.QWEN3_TINY
LENGTHS = [8, 9, 10, 11, 12, 13, 14, 15, 16]


def _step_gate(m, refs, step, gate, what):
    B = len(LENGTHS)
    slots = list(range(B))
    slots_d = torch.tensor(slots, dtype=torch.int32, device="cuda")
    inp = torch.tensor([refs[i]["fed"][step] for i in range(B)], dtype=torch.int32, device="cuda")
    out = torch.zeros(B, dtype=torch.int32, device="cuda")
    lg = torch.zeros(B, S.vocab, dtype=torch.float32, device="cuda")
    m.decode_step(inp, slots_d, slots, out, lg)
    if gate is not None:
        for i in range(B):
            r = refs[i]["calls"][step + 1]
            gate.logits(lg[i].cpu().numpy(), r["logits"], f"{what} row {i}")
            gate.token(int(out[i]), r["token"], r["margin"], f"{what} row {i}")
    return out


def _model(w, prompts):
    B = len(LENGTHS)
    m = binding.Model(S, w, max_seqs=B, max_ctx=64, max_prefill_tokens=sum(LENGTHS))
    m.prefill(torch.cat(prompts).cuda(), LENGTHS, list(range(B)))
    return m


def test_wait_limit_timeout_is_reported_and_recoverable():
    gc.ensure_library()
    w = synth.make_weights(S)
    cfg, ow = gc.oracle_config(S), gc.oracle_weights(w)
    prompts = [synth.make_tokens(n, S.vocab, 600 + i) for i, n in enumerate(LENGTHS)]
    refs = [oracle.generate(cfg, ow, p.tolist(), 2) for p in prompts]

    m = _model(w, prompts)
    gate = gc.Gate()
    _step_gate(m, refs, 0, gate, "step 0")
    assert m.status() == 0

    m.set_wait_limit(1)
    out = _step_gate(m, refs, 1, None, "limited")
    code = m.status()
    msg = binding.qwen3_last_error(m.ctx)
    assert code == binding.QWEN3_E_DEVICE, (code, msg)
    assert "bounded wait" in msg
    assert torch.all(out == -1), out  # the head's waits gave up too: no valid token
    assert m.status() == 0  # the word was cleared by the read

    # rewind the failed step on the same context and take it again with the default limit
    m.set_wait_limit(0)
    for i, n in enumerate(LENGTHS):
        m.truncate(i, n + 1)
        assert binding.qwen3_slot_length(m.ctx, i) == n + 1
    _step_gate(m, refs, 1, gate, "step 1 again")
    assert m.status() == 0
    m.close()

    # a fresh context is clean
    m2 = _model(w, prompts)
    _step_gate(m2, refs, 0, gate, "fresh step 0")
    _step_gate(m2, refs, 1, gate, "fresh step 1")
    assert m2.status() == 0
    m2.close()
    print(gate.summary())
    gate.check()
