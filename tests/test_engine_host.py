"""The continuous-batching engine's scheduling, on the CPU.

engine.cu is compiled unchanged with g++ against engine_host_mock.cpp, a host-only stand-in
for the context calls it makes (prefill_append, decode_step, release_slot, ...) whose "model"
answers with the FNV-1a hash of a slot's token history.  The tests check what the engine
documents: every request's tokens are the model's continuation of its prompt; it stops at its
eos id (kept), at max_new_tokens, or when its slot holds max_ctx tokens; each step schedules at
most token_budget tokens -- one generated token per running request, then prompt chunks, then
first-come-first-served admissions into free slots; a step with a prompt chunk is one
prefill_append call, a step of generated tokens only is one decode step; each prompt is fed
once, in order; slots are released before reuse.
"""

import ctypes
import os
import random
import shutil
import subprocess

import pytest

from qwen3_decoder_forward_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ENGINE_SRC = os.path.join(ROOT, "qwen3_decoder_forward_gb300", "csrc", "engine.cu")
MOCK_SRC = os.path.join(ROOT, "tests", "engine_host_mock.cpp")
CUDA_INCLUDE = "/usr/local/cuda/include"

P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64


@pytest.fixture(scope="module")
def lib(tmp_path_factory):
    gxx = shutil.which("g++")
    if not gxx or not os.path.isdir(CUDA_INCLUDE):
        pytest.skip("needs g++ and the CUDA headers")
    out = str(tmp_path_factory.mktemp("engine_mock") / "libengine_mock.so")
    # -Bsymbolic: the engine's calls resolve to the stand-ins in this library even when the
    # process has loaded the real CUDA runtime or the real library (other tests do)
    cmd = [gxx, "-std=c++17", "-O1", "-shared", "-fPIC", "-Wl,-Bsymbolic", "-I", os.path.join(ROOT, "include"),
           "-I", CUDA_INCLUDE, "-x", "c++", ENGINE_SRC, "-x", "c++", MOCK_SRC, "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    lib = ctypes.CDLL(out)
    sig = {
        "mock_ctx_create": (P, [I32, I32, I32, I32]),
        "mock_ctx_free": (None, [P]),
        "mock_log_size": (I32, [P]),
        "mock_log": (None, [P, P]),
        "qwen3_engine_workspace_bytes": (ctypes.c_size_t, [P, I32]),
        "qwen3_engine_create": (ctypes.c_int, [P, I32, P, ctypes.c_size_t, ctypes.POINTER(P)]),
        "qwen3_engine_submit": (ctypes.c_int, [P, I64, ctypes.POINTER(I32), I32, I32, I32]),
        "qwen3_engine_submit_sampled": (ctypes.c_int, [P, I64, ctypes.POINTER(I32), I32, I32, I32, ctypes.c_float, I32,
                                                       ctypes.c_float, ctypes.c_uint64]),
        "qwen3_engine_step": (ctypes.c_int, [P, P, ctypes.POINTER(I32)]),
        "qwen3_engine_unfinished": (I32, [P]),
        "qwen3_engine_result": (ctypes.c_int, [P, I64, ctypes.POINTER(I32), I32, ctypes.POINTER(I32),
                                               ctypes.POINTER(I32)]),
        "qwen3_engine_forget": (ctypes.c_int, [P, I64]),
        "qwen3_engine_get_stats": (ctypes.c_int, [P, ctypes.POINTER(binding.qwen3_engine_stats)]),
        "qwen3_engine_last_error": (ctypes.c_char_p, [P]),
        "qwen3_engine_free": (None, [P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    return lib


def fnv_next(history, vocab):
    """The stand-in model's next token: FNV-1a (64-bit) of the token history, modulo vocab."""
    x = 14695981039346656037
    for t in history:
        x ^= t & 0xFFFFFFFF
        x = (x * 1099511628211) % (1 << 64)
    return x % vocab


def splitmix64_draw(seed, t):
    """Uniform draw of a sampling request's t-th token: output t + 1 of SplitMix64 (Steele, Lea
    and Flood 2014) started at `seed`, top 24 bits over 2^24."""
    m = (1 << 64) - 1
    z = (seed + (t + 1) * 0x9E3779B97F4A7C15) & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    z ^= z >> 31
    return (z >> 40) / 16777216.0


def sampled_next(history, vocab, temperature, top_k, top_p, u):
    """The stand-in model's token for a sampling row: the history's hash mixed with the row's
    draw and settings (engine_host_mock.cpp, row_token)."""
    import numpy as np
    x = 14695981039346656037
    for t in history:
        x ^= t & 0xFFFFFFFF
        x = (x * 1099511628211) % (1 << 64)
    x ^= int(np.float32(u) * np.float32(16777216.0)) << 32
    x ^= (top_k & 0xFFFFFFFF) << 8
    x ^= int(np.float32(np.float32(temperature) * np.float32(1000.0) + np.float32(0.5))) << 16
    x ^= int(np.float32(np.float32(top_p) * np.float32(1000.0) + np.float32(0.5))) << 40
    return (x % (1 << 64)) % vocab


def expected(prompt, max_new, eos, max_ctx, vocab, sampling=None):
    """(tokens, finish reason) the engine's rules give for one request on the stand-in model;
    sampling = (temperature, top_k, top_p, seed) for a request submitted with them."""
    gen = []
    while True:
        if gen:
            if eos >= 0 and gen[-1] == eos:
                return gen, binding.QWEN3_FINISH_EOS
            if len(gen) >= max_new:
                return gen, binding.QWEN3_FINISH_LENGTH
            if len(prompt) + len(gen) - 1 >= max_ctx:  # the last token cannot be appended
                return gen, binding.QWEN3_FINISH_CONTEXT
        if sampling and sampling[0] > 0:
            T, k, p, seed = sampling
            gen.append(sampled_next(prompt + gen, vocab, T, k, p, splitmix64_draw(seed, len(gen))))
        else:
            gen.append(fnv_next(prompt + gen, vocab))  # every earlier token has been fed


class Run:
    def __init__(self, lib, max_seqs, max_ctx, max_prefill, vocab, budget):
        self.lib, self.budget, self.max_ctx, self.vocab = lib, budget, max_ctx, vocab
        self.max_seqs = max_seqs
        self.ctx = lib.mock_ctx_create(max_seqs, max_ctx, max_prefill, vocab)
        n = lib.qwen3_engine_workspace_bytes(self.ctx, budget)
        self.ws = ctypes.create_string_buffer(n + 256)
        ptr = (ctypes.addressof(self.ws) + 255) // 256 * 256
        self.eng = P()
        rc = lib.qwen3_engine_create(self.ctx, budget, ptr, n, ctypes.byref(self.eng))
        assert rc == binding.QWEN3_OK

    def submit(self, rid, prompt, max_new, eos=-1, sampling=None):
        arr = (I32 * len(prompt))(*prompt)
        if sampling:
            T, k, p, seed = sampling
            return self.lib.qwen3_engine_submit_sampled(self.eng, rid, arr, len(prompt), max_new, eos, T, k, p, seed)
        return self.lib.qwen3_engine_submit(self.eng, rid, arr, len(prompt), max_new, eos)

    def run(self, max_steps=10000):
        steps = 0
        while self.lib.qwen3_engine_unfinished(self.eng) and steps < max_steps:
            n = I32()
            rc = self.lib.qwen3_engine_step(self.eng, None, ctypes.byref(n))
            assert rc == binding.QWEN3_OK, self.lib.qwen3_engine_last_error(self.eng)
            steps += 1
        assert self.lib.qwen3_engine_unfinished(self.eng) == 0
        return steps

    def result(self, rid):
        n, why = I32(), I32()
        assert self.lib.qwen3_engine_result(self.eng, rid, None, 0, ctypes.byref(n), ctypes.byref(why)) == 0
        buf = (I32 * max(1, n.value))()
        self.lib.qwen3_engine_result(self.eng, rid, buf, n.value, ctypes.byref(n), ctypes.byref(why))
        return list(buf[: n.value]), why.value

    def stats(self):
        st = binding.qwen3_engine_stats()
        assert self.lib.qwen3_engine_get_stats(self.eng, ctypes.byref(st)) == 0
        return {k: getattr(st, k) for k, _ in st._fields_}

    def log(self):
        """Parsed call log: ("release", slot) | (kind, [(slot, tokens), ...]) per call."""
        n = self.lib.mock_log_size(self.ctx)
        buf = (I32 * max(1, n))()
        self.lib.mock_log(self.ctx, buf)
        raw, i, out = list(buf[:n]), 0, []
        while i < n:
            kind = raw[i]
            if kind == 3:
                out.append(("release", raw[i + 1]))
                i += 2
                continue
            B, i = raw[i + 1], i + 3
            rows = []
            for _ in range(B):
                slot, cnt = raw[i], raw[i + 1]
                rows.append((slot, raw[i + 2: i + 2 + cnt]))
                i += 2 + cnt
            out.append(("prefill" if kind == 1 else "decode", rows))
        return out

    def close(self):
        self.lib.qwen3_engine_free(self.eng)
        self.lib.mock_ctx_free(self.ctx)


def check_schedule(run, requests, results):
    """The call log against the documented step rules; requests: [(prompt, max_new, eos)],
    results: [(tokens, finish reason)] of the same requests."""
    log = run.log()
    admitted = []   # request indices in admission order (one slot release per admission)
    holder = {}     # slot -> request index
    fed = {}        # request index -> prompt tokens fed so far
    gen_fed = {}    # request index -> generated tokens fed back
    for ev in log:
        if ev[0] == "release":
            r = len(admitted)
            admitted.append(r)
            holder[ev[1]] = r
            fed[r], gen_fed[r] = [], []
            continue
        kind, rows = ev
        assert 1 <= len(rows) <= run.max_seqs
        assert sum(len(t) for _, t in rows) <= run.budget
        seen_chunk = False
        for slot, toks in rows:
            r = holder[slot]
            prompt = requests[r][0]
            if len(fed[r]) < len(prompt):  # a prompt chunk: the next tokens of the prompt
                assert toks == prompt[len(fed[r]): len(fed[r]) + len(toks)]
                fed[r] += toks
                seen_chunk = True
            else:                          # a generated token fed back: one per row, and the
                assert len(toks) == 1      # generated rows of a step come before its chunks
                assert not seen_chunk
                gen_fed[r] += toks
        assert (kind == "prefill") == seen_chunk
    # first come, first served, and every prompt fed completely
    assert admitted == list(range(len(requests)))
    for r, (prompt, _, _) in enumerate(requests):
        assert fed[r] == prompt
        assert gen_fed[r] == results[r][0][:-1]  # each generated token fed once, in order, but the last
    return log


REQUESTS = [(5, 6), (20, 4), (9, 8), (33, 3), (3, 10), (12, 5)]


def _prompts(seed, lengths, vocab):
    rng = random.Random(seed)
    return [[rng.randrange(vocab) for _ in range(n)] for n in lengths]


def test_engine_schedule_and_tokens(lib):
    vocab, max_ctx = 4096, 64
    run = Run(lib, max_seqs=3, max_ctx=max_ctx, max_prefill=48, vocab=vocab, budget=16)
    prompts = _prompts(1, [n for n, _ in REQUESTS], vocab)
    reqs = [(p, k, -1) for p, (_, k) in zip(prompts, REQUESTS)]
    for i, (p, k, e) in enumerate(reqs):
        assert run.submit(100 + i, p, k, e) == 0
    steps = run.run()
    results = [run.result(100 + i) for i in range(len(reqs))]
    for i, (p, k, e) in enumerate(reqs):
        assert results[i] == expected(p, k, e, max_ctx, vocab), i
    check_schedule(run, reqs, results)
    st = run.stats()
    assert st["steps"] == steps == st["mixed_steps"] + st["decode_steps"]
    assert st["prompt_tokens"] == sum(len(p) for p in prompts)
    assert st["generated_tokens"] == sum(k for _, k in REQUESTS)
    assert st["mixed_steps"] >= 5 and st["decode_steps"] >= 1
    # the first step fills the budget: 5 tokens of request 0, then 11 of request 1's 20
    first = [ev for ev in run.log() if ev[0] != "release"][0]
    assert first[0] == "prefill" and [len(t) for _, t in first[1]] == [5, 11]
    run.close()


def test_engine_eos_context_and_slot_reuse(lib):
    vocab, max_ctx = 4096, 40
    run = Run(lib, max_seqs=2, max_ctx=max_ctx, max_prefill=64, vocab=vocab, budget=8)
    prompts = _prompts(2, [7, 36, 4, 15], vocab)
    # request 0 stops on the third token of its continuation; request 1 fills its slot
    cont0, _ = expected(prompts[0], 10, -1, max_ctx, vocab)
    eos0 = cont0[2] if cont0[2] not in cont0[:2] else -1
    reqs = [(prompts[0], 10, eos0), (prompts[1], 50, -1), (prompts[2], 3, -1), (prompts[3], 6, -1)]
    for i, (p, k, e) in enumerate(reqs):
        assert run.submit(i, p, k, e) == 0
    run.run()
    results = [run.result(i) for i in range(len(reqs))]
    for i, (p, k, e) in enumerate(reqs):
        assert results[i] == expected(p, k, e, max_ctx, vocab), i
    if eos0 >= 0:
        assert run.result(0)[1] == binding.QWEN3_FINISH_EOS and len(run.result(0)[0]) == 3
    assert run.result(1)[1] == binding.QWEN3_FINISH_CONTEXT and len(run.result(1)[0]) == 5
    log = check_schedule(run, reqs, results)
    # two slots, four requests: the slots were released and reused
    releases = [ev[1] for ev in log if ev[0] == "release"]
    assert len(releases) == 4 and set(releases) == {0, 1}
    run.close()


@pytest.mark.parametrize("seed", range(6))
def test_engine_random_workloads(lib, seed):
    """Random prompt lengths, limits, end tokens and budgets."""
    rng = random.Random(100 + seed)
    vocab = rng.choice([7, 64, 4096])  # a tiny vocabulary makes end tokens frequent
    max_seqs = rng.randint(1, 5)
    max_ctx = rng.randint(20, 90)
    max_prefill = rng.randint(max_seqs, 120)
    budget = rng.randint(max_seqs, max_prefill)
    run = Run(lib, max_seqs, max_ctx, max_prefill, vocab, budget)
    reqs = []
    for i in range(rng.randint(1, 25)):
        p = [rng.randrange(vocab) for _ in range(rng.randint(1, max_ctx))]
        reqs.append((p, rng.randint(1, 12), rng.randrange(vocab) if rng.random() < 0.5 else -1))
        assert run.submit(i, *reqs[-1]) == 0
    run.run()
    results = [run.result(i) for i in range(len(reqs))]
    for i, (p, k, e) in enumerate(reqs):
        assert results[i] == expected(p, k, e, max_ctx, vocab), (seed, i)
    check_schedule(run, reqs, results)
    run.close()


def test_engine_argument_checks(lib):
    ctx = lib.mock_ctx_create(3, 64, 48, 100)
    eng = P()
    for budget in (2, 49):  # below max_seqs, above max_prefill_tokens
        n = lib.qwen3_engine_workspace_bytes(ctx, budget)
        ws = ctypes.create_string_buffer(n + 256)
        ptr = (ctypes.addressof(ws) + 255) // 256 * 256
        assert lib.qwen3_engine_create(ctx, budget, ptr, n, ctypes.byref(eng)) == binding.QWEN3_E_INVALID
    n = lib.qwen3_engine_workspace_bytes(ctx, 16)
    ws = ctypes.create_string_buffer(n + 256)
    ptr = (ctypes.addressof(ws) + 255) // 256 * 256
    assert lib.qwen3_engine_create(ctx, 16, ptr + 8, n, ctypes.byref(eng)) == binding.QWEN3_E_INVALID  # alignment
    assert lib.qwen3_engine_create(ctx, 16, ptr, n - 1, ctypes.byref(eng)) == binding.QWEN3_E_INVALID  # size
    assert lib.qwen3_engine_create(ctx, 16, ptr, n, ctypes.byref(eng)) == binding.QWEN3_OK
    one = (I32 * 65)(*([1] * 65))
    assert lib.qwen3_engine_submit(eng, 1, one, 0, 4, -1) == binding.QWEN3_E_INVALID
    assert lib.qwen3_engine_submit(eng, 1, one, 3, 0, -1) == binding.QWEN3_E_INVALID
    assert lib.qwen3_engine_submit(eng, 1, one, 65, 4, -1) == binding.QWEN3_E_CAPACITY
    assert lib.qwen3_engine_submit(eng, 1, one, 3, 2, -1) == binding.QWEN3_OK
    assert lib.qwen3_engine_submit(eng, 1, one, 3, 2, -1) == binding.QWEN3_E_INVALID
    assert lib.qwen3_engine_forget(eng, 1) == binding.QWEN3_E_INVALID  # not finished
    assert lib.qwen3_engine_forget(eng, 2) == binding.QWEN3_E_INVALID  # unknown
    while lib.qwen3_engine_unfinished(eng):
        assert lib.qwen3_engine_step(eng, None, None) == binding.QWEN3_OK
    assert lib.qwen3_engine_step(eng, None, None) == binding.QWEN3_OK  # nothing to run
    assert lib.qwen3_engine_forget(eng, 1) == binding.QWEN3_OK
    n_out, why = I32(), I32()
    assert lib.qwen3_engine_result(eng, 1, None, 0, ctypes.byref(n_out), ctypes.byref(why)) == binding.QWEN3_E_INVALID
    lib.qwen3_engine_free(eng)
    lib.mock_ctx_free(ctx)


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_engine_sampling_requests(lib, seed):
    """Sampling requests mixed with greedy ones: each sampling row gets its own settings and the
    draw of its own token index from its own seed, whatever else shares the step; greedy rows of
    a sampling step stay greedy."""
    rng = random.Random(seed)
    vocab, max_ctx = 97, 60
    run = Run(lib, max_seqs=4, max_ctx=max_ctx, max_prefill=64, vocab=vocab, budget=16)
    reqs = {}
    for rid in range(12):
        prompt = [rng.randrange(vocab) for _ in range(rng.randint(1, 30))]
        max_new = rng.randint(1, 25)
        eos = rng.choice([-1, -1, rng.randrange(vocab)])
        sampling = None
        if rid % 3:
            sampling = (rng.choice([0.6, 1.0, 1.7]), rng.choice([0, 5, 40]), rng.choice([1.0, 0.9, 0.5]),
                        rng.randrange(1 << 64))
        assert run.submit(rid, prompt, max_new, eos, sampling) == binding.QWEN3_OK
        reqs[rid] = (prompt, max_new, eos, sampling)
    run.run()
    for rid, (prompt, max_new, eos, sampling) in reqs.items():
        assert run.result(rid) == expected(prompt, max_new, eos, max_ctx, vocab, sampling), rid
    run.close()


def test_splitmix64_reference_values():
    """The draw generator against the published SplitMix64 outputs for state 0 (the first
    output of seed 0 is 0xE220A8397B1DCDAF)."""
    m = (1 << 64) - 1
    z = 0x9E3779B97F4A7C15
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    z ^= z >> 31
    assert z == 0xE220A8397B1DCDAF
    assert splitmix64_draw(0, 0) == (0xE220A8397B1DCDAF >> 40) / 16777216.0
