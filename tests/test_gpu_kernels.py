"""Single kernels through the C ABI against plain PyTorch fp32 on the GPU.

The projections (prefill GEMM, decode GEMV) are checked on ragged row counts and every
epilogue; the lm_head + argmax on its logits and its choice.  Operands are bf16; the
reference widens them to fp32 and multiplies in fp32, so only summation order differs.
"""

import pytest
import torch
import torch.nn.functional as F

import gpu_common as gc
from qwen3_decoder_forward_gb300 import binding

pytestmark = pytest.mark.gpu


def _rand(shape, seed, scale=1.0):
    g = torch.Generator(device="cpu").manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16).cuda()


def _run(op, M, K, N, epi, seed):
    x = _rand((M, K), seed)
    w = _rand((N, K), seed + 1, 0.02)
    ref = x.float() @ w.float().T
    stream = torch.cuda.current_stream().cuda_stream
    if epi == binding.QWEN3_EPI_F32:
        out = torch.full((M, N), float("nan"), device="cuda")
        op(x.data_ptr(), M, K, w.data_ptr(), N, epi, out.data_ptr(), stream)
        return out, ref
    if epi == binding.QWEN3_EPI_RESID_ADD:
        base = _rand((M, N), seed + 2).float()
        out = base.clone()
        op(x.data_ptr(), M, K, w.data_ptr(), N, epi, out.data_ptr(), stream)
        return out, base + ref
    out = torch.full((M, N // 2), float("nan"), dtype=torch.bfloat16, device="cuda")
    op(x.data_ptr(), M, K, w.data_ptr(), N, epi, out.data_ptr(), stream)
    return out.float(), F.silu(ref[:, 0::2]) * ref[:, 1::2]


EPIS = [binding.QWEN3_EPI_F32, binding.QWEN3_EPI_RESID_ADD, binding.QWEN3_EPI_SWIGLU]


@pytest.mark.parametrize("M,K,N", [(1, 1024, 256), (77, 1024, 4096), (128, 2048, 1024), (300, 3072, 1024),
                                   (1000, 1024, 6144), (4099, 1024, 512)])
@pytest.mark.parametrize("epi", EPIS)
def test_prefill_gemm_vs_torch(M, K, N, epi):
    gc.ensure_library()
    out, ref = _run(binding.qwen3_op_gemm, M, K, N, epi, seed=M + K + N + epi)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    tol = 4e-3 if epi == binding.QWEN3_EPI_SWIGLU else 1e-5
    assert gc.rel_l2(out.cpu().numpy(), ref.cpu().numpy()) <= tol


@pytest.mark.parametrize("M", [1, 3, 8, 12, 16, 17, 32])
@pytest.mark.parametrize("K,N", [(1024, 4096), (2048, 1024), (3072, 1024), (1024, 6144)])
@pytest.mark.parametrize("epi", EPIS)
def test_decode_gemv_vs_torch(M, K, N, epi):
    gc.ensure_library()
    out, ref = _run(binding.qwen3_op_gemv, M, K, N, epi, seed=7 * M + K + N + epi)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    tol = 4e-3 if epi == binding.QWEN3_EPI_SWIGLU else 1e-5
    assert gc.rel_l2(out.cpu().numpy(), ref.cpu().numpy()) <= tol


@pytest.mark.parametrize("B,V", [(1, 151936), (7, 4096), (32, 50021)])
def test_lmhead_argmax_vs_torch(B, V):
    gc.ensure_library()
    C = 1024
    x = _rand((B, C), B + V)
    e = _rand((V, C), B + V + 1, 0.02)
    ws_bytes = binding.qwen3_op_lmhead_workspace_bytes(B)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    logits = torch.empty(B, V, device="cuda")
    binding.qwen3_op_lmhead_argmax(x.data_ptr(), B, C, e.data_ptr(), V, logits.data_ptr(), tok.data_ptr(),
                                   ws.data_ptr(), ws_bytes, torch.cuda.current_stream().cuda_stream)
    ref = x.float() @ e.float().T
    torch.cuda.synchronize()
    assert gc.rel_l2(logits.cpu().numpy(), ref.cpu().numpy()) <= 1e-5
    # the choice is exactly the argmax of the kernel's own logits (first index on ties) ...
    assert torch.equal(tok.long(), torch.argmax(logits, dim=1))
    # ... and the reference's wherever its top-2 gap is clear
    top2 = torch.topk(ref, 2, dim=1).values
    clear = (top2[:, 0] - top2[:, 1]) > 1e-3
    assert torch.equal(tok.long()[clear], torch.argmax(ref, dim=1)[clear])


@pytest.mark.parametrize("M", [1, 2, 4])
def test_decode_mlp_vs_torch(M):
    """The fused decode MLP against fp32: out = base + h + Wd(silu(Wg m) * Wu m), m = RMSNorm(h)
    * gain, rounding m and the activation to bf16 where the kernel stores them."""
    gc.ensure_library()
    C, I, eps = 1024, 3072, 1e-6
    g = torch.Generator(device="cpu").manual_seed(40 + M)
    h = torch.randn((M, C), generator=g).cuda()
    gain = (1 + 0.05 * torch.randn(C, generator=g)).cuda()
    wg = _rand((I, C), 41 + M, 0.02)
    wu = _rand((I, C), 42 + M, 0.02)
    wd = _rand((C, I), 43 + M, 0.02)
    w_gu = torch.stack([wg, wu], dim=1).reshape(2 * I, C).contiguous()  # gate_0, up_0, gate_1, ...
    w_dt = wd.T.contiguous()
    base = torch.randn((M, C), generator=g).cuda()
    out = base.clone()
    binding.qwen3_op_mlp_decode(h.data_ptr(), M, C, gain.data_ptr(), eps, w_gu.data_ptr(), w_dt.data_ptr(), I,
                                out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    m = (h * torch.rsqrt((h * h).mean(dim=1, keepdim=True) + eps) * gain).to(torch.bfloat16).float()
    act = (F.silu(m @ wg.float().T) * (m @ wu.float().T)).to(torch.bfloat16).float()
    ref = base + h + act @ wd.float().T
    assert gc.rel_l2((out - base - h).cpu().numpy(), (ref - base - h).cpu().numpy()) <= 4e-3
    assert gc.rel_l2(out.cpu().numpy(), ref.cpu().numpy()) <= 1e-4
    with pytest.raises(binding.Qwen3Error):
        binding.qwen3_op_mlp_decode(h.data_ptr(), 5, C, gain.data_ptr(), eps, w_gu.data_ptr(), w_dt.data_ptr(), I,
                                    out.data_ptr(), 0)


def test_decode_attention_plan():
    """One wave of key ranges per (row, KV head): as many as the SMs hold CTAs for all pairs,
    at least 64 keys a range (from the context rounded up to a power of two, capped at
    max_ctx), 1..64."""
    gc.ensure_library()
    plan = binding.qwen3_op_attn_decode_plan
    wave = plan(1, 16, 8, 40960, 40960)             # 8 pairs, long context: the wave decides
    assert 1 <= wave <= 64
    assert plan(1, 16, 8, 64, 64) == 1              # a 64-key context: one range
    assert plan(1, 16, 8, 200, 256) == min(wave, 4)  # bucket 256: at most 4 ranges of 64
    b16, b32 = plan(16, 16, 8, 16401, 16416), plan(32, 16, 8, 1057, 2048)
    assert 1 <= b32 <= b16 <= wave                   # more pairs, fewer ranges each
    assert plan(1024, 16, 8, 100, 128) == 1


@pytest.mark.parametrize("positions,n_split,Hq,Hkv", [
    ([0, 64, 200], 0, 16, 8), ([63, 127, 129], 1, 16, 8), ([5, 250, 128], 7, 16, 8), ([255, 1, 100], 64, 16, 8),
    ([4000, 1, 3000], 0, 16, 8), ([4095, 2047, 128], 0, 16, 8),
    # one, four and eight query heads per KV head: heads in every column pair of the fragments
    ([130, 7, 255], 3, 8, 8), ([130, 7, 255], 3, 16, 4), ([130, 7, 1000], 0, 16, 2), ([64, 0, 191], 5, 32, 4)])
def test_decode_attention_op_vs_oracle(positions, n_split, Hq, Hkv):
    """qwen3_op_attn_decode against the oracle's per-head RMSNorm, rotate-half RoPE and causal
    GQA attention, over cached rows drawn at random and the new row at `positions`; n_split 0
    takes the decode step's plan (up to 4 ranges of whole 64-key chunks per pair at 256 keys,
    more for the 4K contexts: ranges that end inside a chunk, empty ranges past the keys).
    Query heads per KV head 1, 2, 4 and 8 (the heads are the N side of the score MMA)."""
    import numpy as np
    from oracle import qwen3_oracle as oracle

    gc.ensure_library()
    max_ctx = 256 if max(positions) < 256 else 4096
    B, D, eps, theta = len(positions), 128, 1e-6, 1e6
    n_slots = B + 1
    slots = [2, 0, 3][:B]
    g = torch.Generator(device="cpu").manual_seed(sum(positions) + n_split)
    qkv = torch.randn((B, (Hq + 2 * Hkv) * D), generator=g)
    qg = 1 + 0.05 * torch.randn(D, generator=g)
    kg = 1 + 0.05 * torch.randn(D, generator=g)
    kc = torch.randn((n_slots, Hkv, max_ctx, D), generator=g).to(torch.bfloat16)
    vc = torch.randn((n_slots, Hkv, max_ctx, D), generator=g).to(torch.bfloat16)
    ang = np.arange(max_ctx)[:, None] * oracle.rope_inv_freq(D, theta)[None, :]
    rope = torch.from_numpy(np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32))
    dev = [t.cuda().contiguous() for t in (qkv, qg, kg, kc, vc, rope)]
    qkv_d, qg_d, kg_d, kc_d, vc_d, rope_d = dev
    slots_d = torch.tensor(slots, dtype=torch.int32, device="cuda")
    pos_d = torch.tensor(positions, dtype=torch.int32, device="cuda")
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws_bytes = binding.qwen3_op_attn_decode_workspace_bytes(B, Hq, Hkv)
    ws = torch.zeros(ws_bytes + 256, dtype=torch.uint8, device="cuda")
    ws_ptr = (ws.data_ptr() + 255) // 256 * 256
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # the second call finds the workspace as the first left it
        binding.qwen3_op_attn_decode(qkv_d.data_ptr(), B, slots_d.data_ptr(), slots, pos_d.data_ptr(), positions,
                                     qg_d.data_ptr(), kg_d.data_ptr(), rope_d.data_ptr(), kc_d.data_ptr(),
                                     vc_d.data_ptr(), n_slots, max_ctx, Hq, Hkv, eps, n_split, out.data_ptr(),
                                     ws_ptr, ws_bytes, stream)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    kc_after, vc_after = kc_d.float().cpu().numpy(), vc_d.float().cpu().numpy()
    for b, (s, p) in enumerate(zip(slots, positions)):
        row = qkv[b].double().numpy()
        q = row[: Hq * D].reshape(1, Hq, D)
        k = row[Hq * D: (Hq + Hkv) * D].reshape(1, Hkv, D)
        v = row[(Hq + Hkv) * D:].reshape(1, Hkv, D)
        q = oracle.apply_rope(oracle.rms_norm(q, qg.double().numpy(), eps), np.array([p]), theta)
        k = oracle.apply_rope(oracle.rms_norm(k, kg.double().numpy(), eps), np.array([p]), theta)
        # the cache row of the new position holds bf16(k), bf16(v)
        assert gc.rel_l2(kc_after[s, :, p], k[0]) <= 8e-3
        assert gc.rel_l2(vc_after[s, :, p], v[0]) <= 8e-3
        keys = kc[s].double().numpy().transpose(1, 0, 2)[: p + 1].copy()   # [p+1, Hkv, D]
        vals = vc[s].double().numpy().transpose(1, 0, 2)[: p + 1].copy()
        keys[p], vals[p] = k[0], v[0]
        ref = oracle.causal_gqa_attention(q, keys, vals, np.array([p]), np.arange(p + 1))
        assert gc.rel_l2(got[b], ref[0]) <= gc.REL_L2, (b, p)
    # rows of other positions and of the unused slot are untouched
    for s in range(n_slots):
        for p in range(max_ctx):
            if (s, p) in zip(slots, positions):
                continue
            if p % 37 == 0 or s == 1:
                assert np.array_equal(kc_after[s, :, p], kc[s, :, p].float().numpy())
