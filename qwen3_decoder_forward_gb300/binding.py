"""ctypes binding of libqwen3_gb300.so: the C ABI's calls under the same names.

The functions here only marshal arguments (device pointers as integers, host arrays as
ctypes arrays) and turn a negative return code into ``Qwen3Error``.  Every step of the
forward runs in the library's CUDA kernels; there is no fallback path.  ``Model`` is a
convenience owner of the device memory (allocated with PyTorch) around one context.
"""

from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libqwen3_gb300.so")

QWEN3_OK = 0
QWEN3_E_INVALID = -1
QWEN3_E_CAPACITY = -2
QWEN3_E_UNSUPPORTED = -3
QWEN3_E_CUDA = -4
QWEN3_E_DEVICE = -5
QWEN3_FLAG_NO_GRAPH = 1
QWEN3_FLAG_NO_PDL = 2
QWEN3_FLAG_DECODE_CHAIN = 8
QWEN3_EPI_F32 = 0
QWEN3_EPI_RESID_ADD = 1
QWEN3_EPI_SWIGLU = 2

_P = ctypes.c_void_p


class qwen3_sampling(ctypes.Structure):
    _fields_ = [("temperature", _P), ("top_k", _P), ("top_p", _P), ("uniform", _P)]


class qwen3_engine_stats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("mixed_steps", ctypes.c_int64), ("decode_steps", ctypes.c_int64),
                ("prompt_tokens", ctypes.c_int64), ("generated_tokens", ctypes.c_int64)]


QWEN3_FINISH_NONE = 0
QWEN3_FINISH_EOS = 1
QWEN3_FINISH_LENGTH = 2
QWEN3_FINISH_CONTEXT = 3


class qwen3_config(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("intermediate", ctypes.c_int32), ("vocab", ctypes.c_int32), ("rms_eps", ctypes.c_float),
        ("rope_theta", ctypes.c_double), ("max_seqs", ctypes.c_int32), ("max_ctx", ctypes.c_int32),
        ("max_prefill_tokens", ctypes.c_int32), ("flags", ctypes.c_uint32),
        ("kv_block_tokens", ctypes.c_int32), ("kv_pool_blocks", ctypes.c_int32),
    ]


class qwen3_weights(ctypes.Structure):
    _fields_ = [("embed", _P), ("final_norm", _P)] + [
        (k, ctypes.POINTER(_P)) for k in
        ("in_norm", "post_norm", "q_norm", "k_norm", "wq", "wk", "wv", "wo", "wgate", "wup", "wdown")
    ]


class Qwen3Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"qwen3 error {code}: {msg}")
        self.code = code


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the CUDA library (raises if it has not been built: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} is missing: build it with qwen3_decoder_forward_gb300.build.build()")
    lib = ctypes.CDLL(path)
    i32, i64, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    pi32 = ctypes.POINTER(i32)
    sig = {
        "qwen3_arena_bytes": (sz, [ctypes.POINTER(qwen3_config)]),
        "qwen3_create": (ctypes.c_int, [ctypes.POINTER(qwen3_config), ctypes.POINTER(qwen3_weights), _P, sz, _P,
                                        ctypes.POINTER(_P)]),
        "qwen3_prefill": (ctypes.c_int, [_P, _P, _P, pi32, _P, pi32, i32, _P, _P, _P]),
        "qwen3_prefill_append": (ctypes.c_int, [_P, _P, _P, pi32, _P, pi32, i32, _P, _P, _P]),
        "qwen3_decode_step": (ctypes.c_int, [_P, _P, _P, pi32, i32, _P, _P, _P]),
        "qwen3_set_debug_dump": (ctypes.c_int, [_P, _P, sz]),
        "qwen3_set_sampling": (ctypes.c_int, [_P, ctypes.POINTER(qwen3_sampling)]),
        "qwen3_get_status": (ctypes.c_int, [_P]),
        "qwen3_last_error": (ctypes.c_char_p, [_P]),
        "qwen3_slot_length": (i32, [_P, i32]),
        "qwen3_kv_view": (ctypes.c_int, [_P, i32, i32, ctypes.POINTER(_P), ctypes.POINTER(_P)]),
        "qwen3_launch_count": (i64, [_P]),
        "qwen3_get_config": (ctypes.c_int, [_P, ctypes.POINTER(qwen3_config)]),
        "qwen3_kv_copy_rows": (ctypes.c_int, [_P, i32, i32, i32, i32, _P, _P, _P]),
        "qwen3_kv_free_blocks": (i32, [_P]),
        "qwen3_release_slot": (ctypes.c_int, [_P, i32, _P]),
        "qwen3_truncate_slot": (ctypes.c_int, [_P, i32, i32, _P]),
        "qwen3_set_wait_limit": (ctypes.c_int, [_P, ctypes.c_uint32]),
        "qwen3_engine_workspace_bytes": (sz, [_P, i32]),
        "qwen3_engine_create": (ctypes.c_int, [_P, i32, _P, sz, ctypes.POINTER(_P)]),
        "qwen3_engine_submit": (ctypes.c_int, [_P, i64, pi32, i32, i32, i32]),
        "qwen3_engine_submit_sampled": (ctypes.c_int, [_P, i64, pi32, i32, i32, i32, ctypes.c_float, i32,
                                                       ctypes.c_float, ctypes.c_uint64]),
        "qwen3_engine_step": (ctypes.c_int, [_P, _P, pi32]),
        "qwen3_engine_unfinished": (i32, [_P]),
        "qwen3_engine_result": (ctypes.c_int, [_P, i64, pi32, i32, pi32, pi32]),
        "qwen3_engine_forget": (ctypes.c_int, [_P, i64]),
        "qwen3_engine_get_stats": (ctypes.c_int, [_P, ctypes.POINTER(qwen3_engine_stats)]),
        "qwen3_engine_last_step": (ctypes.c_int, [_P, ctypes.POINTER(i64), i32, pi32, ctypes.POINTER(_P)]),
        "qwen3_engine_last_error": (ctypes.c_char_p, [_P]),
        "qwen3_engine_free": (None, [_P]),
        "qwen3_free": (None, [_P]),
        "qwen3_op_gemv": (ctypes.c_int, [_P, i32, i32, _P, i32, i32, _P, _P]),
        "qwen3_op_gemm": (ctypes.c_int, [_P, i32, i32, _P, i32, i32, _P, _P]),
        "qwen3_op_mlp_decode": (ctypes.c_int, [_P, i32, i32, _P, ctypes.c_float, _P, _P, i32, _P, _P]),
        "qwen3_op_lmhead_workspace_bytes": (sz, [i32]),
        "qwen3_op_lmhead_argmax": (ctypes.c_int, [_P, i32, i32, _P, i32, _P, _P, _P, sz, _P]),
        "qwen3_op_lmhead_argmax_noalloc": (ctypes.c_int, [_P, i32, i32, _P, i32, _P, _P, _P]),
        "qwen3_sample": (ctypes.c_int, [_P, i32, i32, _P, _P, _P, _P, _P, _P]),
        "qwen3_op_attn_decode_workspace_bytes": (sz, [i32, i32, i32]),
        "qwen3_op_attn_decode_plan": (i32, [i32, i32, i32, i32, i32]),
        "qwen3_op_attn_decode": (ctypes.c_int, [_P, i32, _P, pi32, _P, pi32, _P, _P, _P, _P, _P, i32, i32, i32, i32,
                                                ctypes.c_float, i32, _P, _P, sz, _P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(rc: int, ctx) -> None:
    if rc != QWEN3_OK:
        msg = load_library().qwen3_last_error(ctx)
        raise Qwen3Error(rc, msg.decode() if msg else "")


def _i32_array(values: Sequence[int]):
    return (ctypes.c_int32 * len(values))(*[int(v) for v in values])


def make_config(shape, max_seqs: int, max_ctx: int, max_prefill_tokens: int, flags: int = 0,
                kv_block_tokens: int = 0, kv_pool_blocks: int = 0) -> qwen3_config:
    return qwen3_config(shape.n_layers, shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                        shape.intermediate, shape.vocab, shape.rms_eps, shape.rope_theta, max_seqs, max_ctx,
                        max_prefill_tokens, flags, kv_block_tokens, kv_pool_blocks)


# --- the C ABI, one wrapper per call ------------------------------------------------------

def qwen3_arena_bytes(cfg: qwen3_config) -> int:
    return int(load_library().qwen3_arena_bytes(ctypes.byref(cfg)))


def qwen3_create(cfg: qwen3_config, weights: qwen3_weights, arena_ptr: int, arena_bytes: int,
                 stream: int = 0):
    ctx = _P()
    rc = load_library().qwen3_create(ctypes.byref(cfg), ctypes.byref(weights), arena_ptr, arena_bytes,
                                     stream, ctypes.byref(ctx))
    _check(rc, None)
    return ctx


def qwen3_prefill(ctx, tokens_ptr: int, cu_dev_ptr: int, cu_host: Sequence[int], slots_dev_ptr: int,
                  slots_host: Sequence[int], B: int, logits_ptr: Optional[int], next_ptr: int, stream: int = 0):
    _check(load_library().qwen3_prefill(ctx, tokens_ptr, cu_dev_ptr, _i32_array(cu_host), slots_dev_ptr,
                                        _i32_array(slots_host), B, logits_ptr, next_ptr, stream), ctx)


def qwen3_prefill_append(ctx, tokens_ptr: int, cu_dev_ptr: int, cu_host: Sequence[int], slots_dev_ptr: int,
                         slots_host: Sequence[int], B: int, logits_ptr: Optional[int], next_ptr: int,
                         stream: int = 0):
    _check(load_library().qwen3_prefill_append(ctx, tokens_ptr, cu_dev_ptr, _i32_array(cu_host), slots_dev_ptr,
                                               _i32_array(slots_host), B, logits_ptr, next_ptr, stream), ctx)


def qwen3_decode_step(ctx, tokens_ptr: int, slots_dev_ptr: int, slots_host: Sequence[int], B: int,
                      logits_ptr: Optional[int], next_ptr: int, stream: int = 0):
    _check(load_library().qwen3_decode_step(ctx, tokens_ptr, slots_dev_ptr, _i32_array(slots_host), B,
                                            logits_ptr, next_ptr, stream), ctx)


def qwen3_set_debug_dump(ctx, hidden_ptr: Optional[int], nbytes: int):
    _check(load_library().qwen3_set_debug_dump(ctx, hidden_ptr, nbytes), ctx)


def qwen3_set_sampling(ctx, temperature_ptr: Optional[int], top_k_ptr: Optional[int] = None,
                       top_p_ptr: Optional[int] = None, uniform_ptr: Optional[int] = None):
    """Per-row sampling arrays (device pointers) for the context's next tokens; a None
    temperature returns to greedy next tokens."""
    if temperature_ptr is None:
        _check(load_library().qwen3_set_sampling(ctx, None), ctx)
        return
    sp = qwen3_sampling(temperature_ptr, top_k_ptr, top_p_ptr, uniform_ptr)
    _check(load_library().qwen3_set_sampling(ctx, ctypes.byref(sp)), ctx)


def qwen3_get_config(ctx) -> qwen3_config:
    cfg = qwen3_config()
    _check(load_library().qwen3_get_config(ctx, ctypes.byref(cfg)), ctx)
    return cfg


def qwen3_release_slot(ctx, slot: int, stream: int = 0):
    _check(load_library().qwen3_release_slot(ctx, slot, stream), ctx)


def qwen3_truncate_slot(ctx, slot: int, length: int, stream: int = 0):
    _check(load_library().qwen3_truncate_slot(ctx, slot, length, stream), ctx)


def qwen3_set_wait_limit(ctx, cycles: int):
    _check(load_library().qwen3_set_wait_limit(ctx, int(cycles)), ctx)


def _engine_check(rc: int, eng) -> None:
    if rc != QWEN3_OK:
        msg = load_library().qwen3_engine_last_error(eng) if eng else b""
        raise Qwen3Error(rc, msg.decode() if msg else "")


def qwen3_engine_workspace_bytes(ctx, token_budget: int) -> int:
    return int(load_library().qwen3_engine_workspace_bytes(ctx, token_budget))


def qwen3_engine_create(ctx, token_budget: int, workspace_ptr: int, nbytes: int):
    eng = _P()
    _engine_check(load_library().qwen3_engine_create(ctx, token_budget, workspace_ptr, nbytes, ctypes.byref(eng)),
                  None)
    return eng


def qwen3_engine_submit(eng, request_id: int, prompt: Sequence[int], max_new_tokens: int, eos_id: int = -1):
    _engine_check(load_library().qwen3_engine_submit(eng, request_id, _i32_array(prompt), len(prompt),
                                                     max_new_tokens, eos_id), eng)


def qwen3_engine_submit_sampled(eng, request_id: int, prompt: Sequence[int], max_new_tokens: int, eos_id: int,
                                temperature: float, top_k: int, top_p: float, seed: int):
    _engine_check(load_library().qwen3_engine_submit_sampled(eng, request_id, _i32_array(prompt), len(prompt),
                                                             max_new_tokens, eos_id, temperature, top_k, top_p,
                                                             seed), eng)


def qwen3_engine_step(eng, stream: int = 0) -> int:
    n = ctypes.c_int32(0)
    _engine_check(load_library().qwen3_engine_step(eng, stream, ctypes.byref(n)), eng)
    return int(n.value)


def qwen3_engine_unfinished(eng) -> int:
    return int(load_library().qwen3_engine_unfinished(eng))


def qwen3_engine_result(eng, request_id: int):
    """(generated tokens, finish reason) of a request."""
    lib = load_library()
    n, why = ctypes.c_int32(0), ctypes.c_int32(0)
    _engine_check(lib.qwen3_engine_result(eng, request_id, None, 0, ctypes.byref(n), ctypes.byref(why)), eng)
    buf = (ctypes.c_int32 * max(1, n.value))()
    _engine_check(lib.qwen3_engine_result(eng, request_id, buf, n.value, ctypes.byref(n), ctypes.byref(why)), eng)
    return [int(buf[i]) for i in range(n.value)], int(why.value)


def qwen3_engine_forget(eng, request_id: int):
    _engine_check(load_library().qwen3_engine_forget(eng, request_id), eng)


def qwen3_engine_get_stats(eng) -> Dict[str, int]:
    st = qwen3_engine_stats()
    _engine_check(load_library().qwen3_engine_get_stats(eng, ctypes.byref(st)), eng)
    return {k: int(getattr(st, k)) for k, _ in qwen3_engine_stats._fields_}


def qwen3_engine_free(eng):
    load_library().qwen3_engine_free(eng)


def qwen3_get_status(ctx) -> int:
    return int(load_library().qwen3_get_status(ctx))


def qwen3_last_error(ctx) -> str:
    m = load_library().qwen3_last_error(ctx)
    return m.decode() if m else ""


def qwen3_slot_length(ctx, slot: int) -> int:
    return int(load_library().qwen3_slot_length(ctx, slot))


def qwen3_kv_view(ctx, layer: int, slot: int):
    k, v = _P(), _P()
    _check(load_library().qwen3_kv_view(ctx, layer, slot, ctypes.byref(k), ctypes.byref(v)), ctx)
    return int(k.value), int(v.value)


def qwen3_launch_count(ctx) -> int:
    return int(load_library().qwen3_launch_count(ctx))


def qwen3_free(ctx) -> None:
    load_library().qwen3_free(ctx)


def qwen3_op_gemv(x_ptr: int, M: int, K: int, w_ptr: int, N: int, epilogue: int, out_ptr: int, stream: int = 0):
    _check(load_library().qwen3_op_gemv(x_ptr, M, K, w_ptr, N, epilogue, out_ptr, stream), None)


def qwen3_op_gemm(x_ptr: int, M: int, K: int, w_ptr: int, N: int, epilogue: int, out_ptr: int, stream: int = 0):
    _check(load_library().qwen3_op_gemm(x_ptr, M, K, w_ptr, N, epilogue, out_ptr, stream), None)


def qwen3_op_lmhead_workspace_bytes(B: int) -> int:
    return int(load_library().qwen3_op_lmhead_workspace_bytes(B))


def qwen3_op_lmhead_argmax(x_ptr: int, B: int, C: int, embed_ptr: int, V: int, logits_ptr: Optional[int],
                           next_ptr: int, ws_ptr: int, ws_bytes: int, stream: int = 0):
    _check(load_library().qwen3_op_lmhead_argmax(x_ptr, B, C, embed_ptr, V, logits_ptr, next_ptr, ws_ptr,
                                                 ws_bytes, stream), None)


def qwen3_op_lmhead_argmax_noalloc(x_ptr: int, B: int, C: int, embed_ptr: int, V: int,
                                   logits_ptr: Optional[int], next_ptr: int, stream: int = 0):
    """lm_head + argmax with the library's fixed scratch instead of a caller workspace (B <= 32)."""
    _check(load_library().qwen3_op_lmhead_argmax_noalloc(x_ptr, B, C, embed_ptr, V, logits_ptr, next_ptr,
                                                         stream), None)


def qwen3_op_mlp_decode(h_ptr: int, M: int, C: int, gain_ptr: int, eps: float, w_gate_up_ptr: int,
                        w_down_t_ptr: int, I: int, out_ptr: int, stream: int = 0):
    """out[M, C] += h + down(silu(gate m) * up m), m = RMSNorm(h) * gain: the fused decode MLP
    (gate/up rows interleaved in w_gate_up [2I, C], down transposed in w_down_t [I, C])."""
    _check(load_library().qwen3_op_mlp_decode(h_ptr, M, C, gain_ptr, eps, w_gate_up_ptr, w_down_t_ptr, I,
                                              out_ptr, stream), None)


def qwen3_op_attn_decode_workspace_bytes(B: int, n_q_heads: int, n_kv_heads: int) -> int:
    return int(load_library().qwen3_op_attn_decode_workspace_bytes(B, n_q_heads, n_kv_heads))


def qwen3_op_attn_decode_plan(B: int, n_q_heads: int, n_kv_heads: int, max_len: int, max_ctx: int) -> int:
    """n_split a decode step of B rows whose longest context is max_len gives its attention
    (0: equal shares of all keys); raises on a bad argument."""
    rc = int(load_library().qwen3_op_attn_decode_plan(B, n_q_heads, n_kv_heads, max_len, max_ctx))
    if rc < 0:
        raise Qwen3Error(rc, qwen3_last_error(None))
    return rc


def qwen3_op_attn_decode(qkv_ptr: int, B: int, slots_ptr: int, slots_host: Sequence[int], positions_ptr: int,
                         positions_host: Sequence[int], q_gain_ptr: int, k_gain_ptr: int, rope_ptr: int,
                         k_cache_ptr: int, v_cache_ptr: int, n_slots: int, max_ctx: int, n_q_heads: int,
                         n_kv_heads: int, eps: float, n_split: int, out_ptr: int, ws_ptr: int, ws_bytes: int,
                         stream: int = 0):
    _check(load_library().qwen3_op_attn_decode(qkv_ptr, B, slots_ptr, _i32_array(slots_host), positions_ptr,
                                               _i32_array(positions_host), q_gain_ptr, k_gain_ptr, rope_ptr,
                                               k_cache_ptr, v_cache_ptr, n_slots, max_ctx, n_q_heads, n_kv_heads,
                                               eps, n_split, out_ptr, ws_ptr, ws_bytes, stream), None)


QWEN3_SAMPLE_CANDIDATES = 1024


def qwen3_sample(logits_ptr: int, B: int, V: int, temperature_ptr: int, top_k_ptr: int, top_p_ptr: int,
                 uniform_ptr: int, next_ptr: int, stream: int = 0):
    """Temperature / top-k / top-p draw of one token per row from fp32 logits [B, V]; the per-row
    parameters and the uniform draws are device arrays of B values."""
    _check(load_library().qwen3_sample(logits_ptr, B, V, temperature_ptr, top_k_ptr, top_p_ptr, uniform_ptr,
                                       next_ptr, stream), None)


def sample(logits, temperature, top_k, top_p, uniform, out=None):
    """qwen3_sample on CUDA tensors: logits fp32 [B, V]; temperature, top_p, uniform fp32 [B];
    top_k int32 [B]; returns (or fills) int32 [B] on the current stream."""
    import torch

    B, V = logits.shape
    for t, dt in ((logits, torch.float32), (temperature, torch.float32), (top_k, torch.int32),
                  (top_p, torch.float32), (uniform, torch.float32)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise Qwen3Error(QWEN3_E_INVALID, "sample: expected contiguous CUDA tensors of the documented dtypes")
    for t in (temperature, top_k, top_p, uniform):
        if t.numel() != B:
            raise Qwen3Error(QWEN3_E_INVALID, "sample: one parameter per row")
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=logits.device)
    qwen3_sample(logits.data_ptr(), B, V, temperature.data_ptr(), top_k.data_ptr(), top_p.data_ptr(),
                 uniform.data_ptr(), out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return out


# --- device-memory owner -------------------------------------------------------------------

class Model:
    """One context plus the device memory it runs in (PyTorch tensors on ``device``).

    ``weights`` is the dict of bf16 tensors from ``synth.make_weights`` (any device).  The
    weights are copied to the GPU, packed by qwen3_create into the arena, then released.
    """

    def __init__(self, shape, weights: Dict, max_seqs: int, max_ctx: int, max_prefill_tokens: int,
                 flags: int = 0, device: str = "cuda", kv_block_tokens: int = 0, kv_pool_blocks: int = 0):
        import torch

        self.torch = torch
        self.shape = shape
        self.device = torch.device(device)
        self.cfg = make_config(shape, max_seqs, max_ctx, max_prefill_tokens, flags, kv_block_tokens, kv_pool_blocks)
        nbytes = qwen3_arena_bytes(self.cfg)
        if nbytes == 0:
            raise Qwen3Error(QWEN3_E_UNSUPPORTED, "configuration not supported")
        self.arena = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.device)
        base = self.arena.data_ptr()
        self.arena_ptr = (base + 255) // 256 * 256
        self.arena_bytes = nbytes
        dev_w = {"embed": weights["embed"].to(self.device).contiguous(),
                 "final_norm": weights["final_norm"].to(self.device).contiguous(),
                 "layers": [{k: v.to(self.device).contiguous() for k, v in d.items()} for d in weights["layers"]]}
        arrays = {}
        for key in ("in_norm", "post_norm", "q_norm", "k_norm", "wq", "wk", "wv", "wo", "wgate", "wup", "wdown"):
            arrays[key] = (_P * shape.n_layers)(*[d[key].data_ptr() for d in dev_w["layers"]])
        w = qwen3_weights(dev_w["embed"].data_ptr(), dev_w["final_norm"].data_ptr(),
                          *[ctypes.cast(arrays[k], ctypes.POINTER(_P)) for k in
                            ("in_norm", "post_norm", "q_norm", "k_norm", "wq", "wk", "wv", "wo",
                             "wgate", "wup", "wdown")])
        stream = torch.cuda.current_stream(self.device).cuda_stream
        self.ctx = qwen3_create(self.cfg, w, self.arena_ptr, self.arena_bytes, stream)
        del dev_w, arrays

    def close(self):
        if getattr(self, "ctx", None) is not None:
            qwen3_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _stream(self):
        return self.torch.cuda.current_stream(self.device).cuda_stream

    def prefill(self, tokens, lengths: Sequence[int], slots: Sequence[int], want_logits: bool = False,
                next_out=None, append: bool = False):
        """tokens: int32 CUDA tensor [N]; returns (next_tok int32 [B], logits fp32 [B, V] or None).
        append=True continues each slot after the tokens it holds (qwen3_prefill_append)."""
        torch = self.torch
        B = len(lengths)
        cu = [0]
        for n in lengths:
            cu.append(cu[-1] + int(n))
        cu_d = torch.tensor(cu, dtype=torch.int32, device=self.device)
        slots_d = torch.tensor(list(slots), dtype=torch.int32, device=self.device)
        nxt = next_out if next_out is not None else torch.empty(B, dtype=torch.int32, device=self.device)
        logits = torch.empty(B, self.shape.vocab, dtype=torch.float32, device=self.device) if want_logits else None
        fn = qwen3_prefill_append if append else qwen3_prefill
        fn(self.ctx, tokens.data_ptr(), cu_d.data_ptr(), cu, slots_d.data_ptr(), list(slots), B,
           logits.data_ptr() if logits is not None else None, nxt.data_ptr(), self._stream())
        self._keep = (cu_d, slots_d)
        return nxt, logits

    def decode_step(self, tokens, slots_dev, slots: Sequence[int], next_out, logits_out=None):
        """tokens: int32 CUDA tensor [B]; writes next_out [B] (and logits_out [B, V] if given)."""
        qwen3_decode_step(self.ctx, tokens.data_ptr(), slots_dev.data_ptr(), list(slots), len(slots),
                          logits_out.data_ptr() if logits_out is not None else None, next_out.data_ptr(),
                          self._stream())

    def set_debug_dump(self, buf):
        qwen3_set_debug_dump(self.ctx, buf.data_ptr() if buf is not None else None,
                             buf.numel() * 4 if buf is not None else 0)

    def set_sampling(self, temperature=None, top_k=None, top_p=None, uniform=None):
        """Per-row sampling settings as CUDA tensors [max_seqs] (fp32, int32, fp32, fp32);
        the tensors are kept alive here and may be rewritten in stream order between calls.
        No arguments: greedy next tokens."""
        torch = self.torch
        if temperature is None:
            qwen3_set_sampling(self.ctx, None)
            self._sampling = None
            return
        for t, dt in ((temperature, torch.float32), (top_k, torch.int32), (top_p, torch.float32),
                      (uniform, torch.float32)):
            if t is None or t.dtype != dt or not t.is_cuda or not t.is_contiguous() or t.numel() < self.cfg.max_seqs:
                raise Qwen3Error(QWEN3_E_INVALID, "set_sampling: contiguous CUDA tensors of max_seqs values")
        qwen3_set_sampling(self.ctx, temperature.data_ptr(), top_k.data_ptr(), top_p.data_ptr(), uniform.data_ptr())
        self._sampling = (temperature, top_k, top_p, uniform)

    def status(self) -> int:
        return qwen3_get_status(self.ctx)

    def truncate(self, slot: int, length: int):
        """Shortens a slot to its first `length` tokens (qwen3_truncate_slot)."""
        qwen3_truncate_slot(self.ctx, slot, length, self._stream())

    def set_wait_limit(self, cycles: int):
        qwen3_set_wait_limit(self.ctx, cycles)

    def kv_copy(self, layer: int, slot: int, pos0: int, n: int):
        """K and V rows pos0 .. pos0+n-1 of (layer, slot) as new bf16 tensors [n, Hkv, D], for
        either cache layout (qwen3_kv_copy_rows)."""
        torch = self.torch
        s = self.shape
        k = torch.empty(s.n_kv_heads, n, s.head_dim, dtype=torch.bfloat16, device=self.device)
        v = torch.empty_like(k)
        rc = load_library().qwen3_kv_copy_rows(self.ctx, layer, slot, pos0, n, k.data_ptr(), v.data_ptr(),
                                               self._stream())
        if rc != QWEN3_OK:
            raise Qwen3Error(rc, "qwen3_kv_copy_rows")
        return k.permute(1, 0, 2).contiguous(), v.permute(1, 0, 2).contiguous()

    def kv_free_blocks(self) -> int:
        return int(load_library().qwen3_kv_free_blocks(self.ctx))

    def kv_rows(self, layer: int, slot: int, n: int):
        """Copies K and V rows 0..n-1 of (layer, slot) to new tensors [n, Hkv, D] (bf16, device)."""
        torch = self.torch
        s = self.shape
        per = s.n_kv_heads * self.cfg.max_ctx * s.head_dim
        whole = self.arena.view(torch.bfloat16)
        out = []
        for p in qwen3_kv_view(self.ctx, layer, slot):
            off = (p - self.arena.data_ptr()) // 2
            t = whole[off: off + per].view(s.n_kv_heads, self.cfg.max_ctx, s.head_dim)
            out.append(t[:, :n].permute(1, 0, 2).contiguous())
        return out[0], out[1]


class Engine:
    """Continuous batching over a ``Model``'s context (qwen3_engine_*): the device workspace is
    a PyTorch buffer kept here; the engine owns every KV slot of the model while it lives."""

    def __init__(self, model: "Model", token_budget: int):
        torch = model.torch
        self.model = model
        nbytes = qwen3_engine_workspace_bytes(model.ctx, token_budget)
        if nbytes == 0:
            raise Qwen3Error(QWEN3_E_INVALID, "engine: bad token budget")
        self.ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=model.device)
        ptr = (self.ws.data_ptr() + 255) // 256 * 256
        self.eng = qwen3_engine_create(model.ctx, token_budget, ptr, nbytes)

    def submit(self, request_id: int, prompt: Sequence[int], max_new_tokens: int, eos_id: int = -1,
               temperature: float = 0.0, top_k: int = 0, top_p: float = 1.0, seed: int = 0):
        """Queues a request; a positive temperature makes it sample (qwen3_engine_submit_sampled)."""
        if temperature > 0:
            qwen3_engine_submit_sampled(self.eng, request_id, [int(t) for t in prompt], max_new_tokens, eos_id,
                                        temperature, top_k, top_p, seed)
        else:
            qwen3_engine_submit(self.eng, request_id, [int(t) for t in prompt], max_new_tokens, eos_id)

    def step(self) -> int:
        return qwen3_engine_step(self.eng, self.model._stream())

    def run(self, max_steps: int = 1 << 20) -> int:
        """Steps until every submitted request has finished; returns the steps taken."""
        n = 0
        while self.unfinished() and n < max_steps:
            self.step()
            n += 1
        return n

    def unfinished(self) -> int:
        return qwen3_engine_unfinished(self.eng)

    def result(self, request_id: int):
        return qwen3_engine_result(self.eng, request_id)

    def forget(self, request_id: int):
        qwen3_engine_forget(self.eng, request_id)

    def stats(self) -> Dict[str, int]:
        return qwen3_engine_get_stats(self.eng)

    def last_step(self):
        """(request ids of the last model step's rows, their fp32 logits [rows, V] as a view of the
        workspace -- or None for an all-greedy step)."""
        lib = load_library()
        n = ctypes.c_int32(0)
        ptr = _P()
        _engine_check(lib.qwen3_engine_last_step(self.eng, None, 0, ctypes.byref(n), None), self.eng)
        ids = (ctypes.c_int64 * max(1, n.value))()
        _engine_check(lib.qwen3_engine_last_step(self.eng, ids, n.value, ctypes.byref(n), ctypes.byref(ptr)), self.eng)
        logits = None
        if ptr.value:
            V = self.model.shape.vocab
            off = ptr.value - self.ws.data_ptr()
            logits = self.ws[off: off + n.value * V * 4].view(self.model.torch.float32).view(n.value, V)
        return [int(ids[i]) for i in range(n.value)], logits

    def close(self):
        if getattr(self, "eng", None) is not None:
            qwen3_engine_free(self.eng)
            self.eng = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
