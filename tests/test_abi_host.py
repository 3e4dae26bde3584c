"""Host-side checks of the C ABI: the library builds, exports every declared call, sizes
its arena and rejects bad arguments before touching the GPU."""

import ctypes
import glob
import os
import re

import pytest

from qwen3_decoder_forward_gb300 import binding, build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(qwen3_\w+)\s*\(", text, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "qwen3_create" in names and "qwen3_decode_step" in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_arena_bytes(lib):
    s = synth.QWEN3_0P6B
    small = binding.qwen3_arena_bytes(binding.make_config(s, 1, 256, 128))
    big = binding.qwen3_arena_bytes(binding.make_config(s, 16, 16416, 16384))
    assert small > 0 and big > small
    kv = 28 * 2 * 16 * 8 * 16416 * 128 * 2
    weights = 28 * 15728640 * 2 + 151936 * 1024 * 2
    assert kv + weights < big < kv + weights + 16 * 2 ** 30


@pytest.mark.parametrize("field,value", [("head_dim", 64), ("n_kv_heads", 3), ("hidden", 1000),
                                         ("max_seqs", 0), ("vocab", 0), ("intermediate", 100)])
def test_unsupported_config_sizes_to_zero(lib, field, value):
    cfg = binding.make_config(synth.QWEN3_0P6B, 4, 512, 512)
    setattr(cfg, field, value)
    assert binding.qwen3_arena_bytes(cfg) == 0


def test_unknown_flag_bits_are_unsupported(lib):
    for flags in (4, 16, 1 << 31):
        assert binding.qwen3_arena_bytes(binding.make_config(synth.QWEN3_TINY, 1, 64, 64, flags)) == 0
    ok = binding.QWEN3_FLAG_NO_GRAPH | binding.QWEN3_FLAG_NO_PDL | binding.QWEN3_FLAG_DECODE_CHAIN
    assert binding.qwen3_arena_bytes(binding.make_config(synth.QWEN3_TINY, 1, 64, 64, ok)) > 0


def test_create_rejects_null_and_unsupported(lib):
    cfg = binding.make_config(synth.QWEN3_TINY, 1, 64, 64)
    w = binding.qwen3_weights()
    with pytest.raises(binding.Qwen3Error) as e:
        binding.qwen3_create(cfg, w, 0, 0)
    assert e.value.code == binding.QWEN3_E_INVALID
    cfg.head_dim = 64
    with pytest.raises(binding.Qwen3Error) as e:
        binding.qwen3_create(cfg, w, 1 << 20, 1 << 30)
    assert e.value.code == binding.QWEN3_E_UNSUPPORTED
    assert "head_dim" in binding.qwen3_last_error(None)


def test_null_context_calls_are_rejected(lib):
    assert lib.qwen3_get_status(None) == binding.QWEN3_E_INVALID
    assert lib.qwen3_slot_length(None, 0) == -1
    assert lib.qwen3_launch_count(None) == 0
    lib.qwen3_free(None)


def test_sample_rejects_null_and_bad_sizes_before_any_launch(lib):
    one = 16  # any non-NULL value: the checks return before a pointer is used
    args = [one, 1, 8, one, one, one, one, one, None]
    for i in (0, 3, 4, 5, 6, 7):
        bad = list(args)
        bad[i] = None
        assert lib.qwen3_sample(*bad) == binding.QWEN3_E_INVALID
        assert "NULL" in binding.qwen3_last_error(None)
    for B, V in ((0, 8), (65536, 8), (1, 0)):
        bad = list(args)
        bad[1], bad[2] = B, V
        assert lib.qwen3_sample(*bad) == binding.QWEN3_E_INVALID


def test_package_import_loads_no_cuda():
    import importlib
    import sys
    mod = importlib.import_module("qwen3_decoder_forward_gb300")
    assert "libqwen3_gb300" not in str(sys.modules.get("qwen3_decoder_forward_gb300.binding", ""))
    assert mod is not None


def test_engine_calls_reject_null_before_any_work(lib):
    assert lib.qwen3_engine_workspace_bytes(None, 16) == 0
    out = ctypes.c_void_p()
    assert lib.qwen3_engine_create(None, 16, 256, 1 << 20, ctypes.byref(out)) == binding.QWEN3_E_INVALID
    assert lib.qwen3_engine_submit(None, 1, binding._i32_array([1, 2]), 2, 4, -1) == binding.QWEN3_E_INVALID
    assert lib.qwen3_engine_step(None, None, None) == binding.QWEN3_E_INVALID
    assert lib.qwen3_engine_unfinished(None) == 0
    assert lib.qwen3_engine_result(None, 1, None, 0, None, None) == binding.QWEN3_E_INVALID
    assert lib.qwen3_engine_forget(None, 1) == binding.QWEN3_E_INVALID
    assert lib.qwen3_engine_get_stats(None, None) == binding.QWEN3_E_INVALID
    assert lib.qwen3_engine_last_step(None, None, 0, None, None) == binding.QWEN3_E_INVALID
    assert lib.qwen3_engine_last_error(None) == b""
    lib.qwen3_engine_free(None)
    cfg = binding.qwen3_config()
    assert lib.qwen3_get_config(None, ctypes.byref(cfg)) == binding.QWEN3_E_INVALID
    assert lib.qwen3_release_slot(None, 0, None) == binding.QWEN3_E_INVALID


def test_paged_kv_config_sizes_and_rejections(lib):
    s = synth.QWEN3_0P6B
    flat = binding.qwen3_arena_bytes(binding.make_config(s, 16, 16384, 4096))
    paged = binding.qwen3_arena_bytes(binding.make_config(s, 16, 16384, 4096, kv_block_tokens=256,
                                                          kv_pool_blocks=64))
    kv_flat = 28 * 2 * 16 * 8 * 16384 * 128 * 2
    kv_paged = 28 * 2 * 64 * 8 * 256 * 128 * 2
    assert 0 < paged < flat
    assert abs((flat - paged) - (kv_flat - kv_paged)) < 2 ** 20  # the pool replaces the per-slot rows
    for bt, pool, flags, heads in ((100, 8, 0, 8), (64, 8, 0, 8), (128, 0, 0, 8), (-128, 8, 0, 8),
                                   (128, 8, 4, 8), (128, 8, 0, 4)):
        cfg = binding.make_config(s, 4, 512, 512, flags, bt, pool)
        cfg.n_kv_heads = heads
        assert binding.qwen3_arena_bytes(cfg) == 0, (bt, pool, flags, heads)


def test_truncate_and_wait_limit_reject_null_context(lib):
    assert lib.qwen3_truncate_slot(None, 0, 0, None) == binding.QWEN3_E_INVALID
    assert lib.qwen3_set_wait_limit(None, 16) == binding.QWEN3_E_INVALID


def test_attn_decode_op_rejects_bad_arguments_before_any_launch(lib):
    assert binding.qwen3_op_attn_decode_workspace_bytes(0, 16, 8) == 0
    assert binding.qwen3_op_attn_decode_workspace_bytes(4, 16, 3) == 0
    ws = binding.qwen3_op_attn_decode_workspace_bytes(4, 16, 8)
    assert ws >= 4 * 16 * 64 * (2 + 128) * 4 + 4 * 8 * 4
    p = 256  # any non-NULL, 256-byte aligned value: the checks return before a pointer is used
    slots, pos = binding._i32_array([0, 1, 2, 3]), binding._i32_array([5, 6, 7, 8])

    def call(**kw):
        a = dict(qkv=p, B=4, slots=p, slots_host=slots, pos=p, pos_host=pos, qg=p, kg=p, rope=p, kc=p, vc=p,
                 n_slots=4, max_ctx=64, hq=16, hkv=8, eps=1e-6, n_split=0, out=p, ws=p, ws_bytes=ws)
        a.update(kw)
        return lib.qwen3_op_attn_decode(a["qkv"], a["B"], a["slots"], a["slots_host"], a["pos"], a["pos_host"],
                                        a["qg"], a["kg"], a["rope"], a["kc"], a["vc"], a["n_slots"], a["max_ctx"],
                                        a["hq"], a["hkv"], a["eps"], a["n_split"], a["out"], a["ws"],
                                        a["ws_bytes"], None)
    for kw in ({"qkv": None}, {"slots_host": None}, {"out": None}, {"B": 0}, {"hkv": 3}, {"hq": 48, "hkv": 3},
               {"n_split": 65}, {"ws_bytes": ws - 1}, {"ws": p + 16}, {"eps": -1.0},
               {"slots_host": binding._i32_array([0, 1, 2, 4])},   # slot >= n_slots
               {"pos_host": binding._i32_array([5, 6, 7, 64])},    # position >= max_ctx
               {"pos_host": binding._i32_array([5, -1, 7, 8])}):
        assert call(**kw) == binding.QWEN3_E_INVALID, kw
        assert "qwen3_op_attn_decode" in binding.qwen3_last_error(None)


def test_gemm_op_rejects_bad_arguments_before_any_launch(lib):
    p = 256  # any non-NULL, 256-byte aligned value: the checks return before a pointer is used
    for args in ((None, 64, 1024, p, 1024, 1, p), (p, 0, 1024, p, 1024, 1, p), (p, 64, 1000, p, 1024, 1, p),
                 (p, 64, 1024, p, 1000, 1, p), (p, 64, 1024, p, 1024, 3, p),
                 (p + 8, 64, 1024, p, 1024, 0, p), (p, 64, 1024, p + 4, 1024, 2, p),
                 (p, 64, 1024, p, 1024, 1, p + 8)):  # residual not 16-byte aligned
        assert lib.qwen3_op_gemm(*args, None) == binding.QWEN3_E_INVALID, args
        assert "qwen3_op_gemm" in binding.qwen3_last_error(None)


def test_attn_decode_plan_rejects_bad_arguments(lib):
    for args in ((0, 16, 8, 10, 64), (4, 16, 3, 10, 64), (4, 16, 8, 0, 64), (4, 16, 8, 65, 64), (1025, 16, 8, 1, 8)):
        assert lib.qwen3_op_attn_decode_plan(*args) == binding.QWEN3_E_INVALID, args
        assert "qwen3_op_attn_decode_plan" in binding.qwen3_last_error(None)


def test_paged_kv_calls_reject_null(lib):
    assert lib.qwen3_kv_copy_rows(None, 0, 0, 0, 1, 16, 16, None) == binding.QWEN3_E_INVALID
    assert lib.qwen3_kv_free_blocks(None) == -1


def test_header_is_c99_and_matches_the_binding_structs(tmp_path):
    """The header compiles as plain C99 (-pedantic, no warnings), and every field of the
    structures the binding mirrors sits at the same offset, with the same size, in both."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("needs gcc")
    structs = {"qwen3_config": binding.qwen3_config, "qwen3_sampling": binding.qwen3_sampling,
               "qwen3_engine_stats": binding.qwen3_engine_stats}
    lines = ['#include <stddef.h>', '#include <stdio.h>', '#include "qwen3_gb300.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'    printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'    printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["    return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    got = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    want = []
    for name, cls in structs.items():
        want.append(f"{name} size {ctypes.sizeof(cls)}")
        want += [f"{name} {field} {getattr(cls, field).offset}" for field, _ in cls._fields_]
    assert [l for l in got if l] == want
