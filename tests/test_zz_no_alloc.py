"""The allocation-free lm_head + argmax entry point, checked against the workspace one.

qwen3_op_lmhead_argmax_noalloc serves callers that cannot allocate device memory (for
example code recording a CUDA graph, or a plug-in whose host framework owns all device
memory).  It keeps its scratch in the library's fixed device array, so two calls in a row
must both match qwen3_op_lmhead_argmax, which uses a caller workspace, and a batch larger
than the array must be refused.
"""

import pytest
import torch

import gpu_common as gc
from qwen3_decoder_forward_gb300 import binding

pytestmark = pytest.mark.gpu


def _inputs(B, V, C, seed):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn(B, C, generator=g).to(torch.bfloat16).cuda()
    e = (torch.randn(V, C, generator=g) * 0.02).to(torch.bfloat16).cuda()
    return x, e


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    gc.ensure_library()
    C = 1024
    stream = torch.cuda.current_stream().cuda_stream
    # 32 rows (tensor-core pass), 5 rows (SIMT pass), then 17 rows on the tensor-core pass again:
    # a smaller batch after a larger one must not pick up the earlier call's partials
    for B, V, seed in ((32, 151936, 21), (5, 50021, 22), (17, 151936, 24)):
        x, e = _inputs(B, V, C, seed)
        ws_bytes = binding.qwen3_op_lmhead_workspace_bytes(B)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        ref_tok = torch.empty(B, dtype=torch.int32, device="cuda")
        ref_log = torch.empty(B, V, dtype=torch.float32, device="cuda")
        binding.qwen3_op_lmhead_argmax(x.data_ptr(), B, C, e.data_ptr(), V, ref_log.data_ptr(), ref_tok.data_ptr(),
                                       ws.data_ptr(), ws_bytes, stream)
        tok = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        log = torch.empty(B, V, dtype=torch.float32, device="cuda")
        binding.qwen3_op_lmhead_argmax_noalloc(x.data_ptr(), B, C, e.data_ptr(), V, log.data_ptr(), tok.data_ptr(),
                                               stream)
        torch.cuda.synchronize()
        assert gc.rel_l2(log.cpu().numpy(), ref_log.cpu().numpy()) <= gc.REL_L2
        assert torch.equal(tok, ref_tok)
        # the chosen token is the argmax of the logits, lowest index on ties
        assert torch.equal(tok.long(), torch.argmax(ref_log, dim=1))
        # and, independently of both entry points, the argmax of x E^T in fp32 (torch) wherever
        # its top-1/top-2 gap exceeds 0.1
        ref = x.float() @ e.float().T
        assert gc.rel_l2(log.cpu().numpy(), ref.cpu().numpy()) <= 1e-5
        top2 = torch.topk(ref, 2, dim=1).values
        clear = (top2[:, 0] - top2[:, 1]) > 0.1
        assert int(clear.sum()) >= 1
        assert torch.equal(tok.long()[clear], torch.argmax(ref, dim=1)[clear])


def test_noalloc_refuses_batches_beyond_its_scratch():
    gc.ensure_library()
    x, e = _inputs(33, 1000, 1024, 23)
    tok = torch.empty(33, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.Qwen3Error) as err:
        binding.qwen3_op_lmhead_argmax_noalloc(x.data_ptr(), 33, 1024, e.data_ptr(), 1000, None, tok.data_ptr(),
                                               torch.cuda.current_stream().cuda_stream)
    assert err.value.code == binding.QWEN3_E_CAPACITY
    assert "32" in str(err.value)
