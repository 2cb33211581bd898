"""The C-ABI library builds for sm_103a, loads without a GPU, and exports every
entry point include/q3.h declares (no compute calls are made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "q3.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(q3_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def libq3():
    from qwen3_dense_decoder_gb300 import buildlib
    path = buildlib.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("q3_model_create", "q3_model_destroy", "q3_pool_create", "q3_session_create",
                     "q3_session_set_block_table", "q3_session_eval", "q3_eval_batch",
                     "q3_session_truncate", "q3_session_reset", "q3_session_pos", "q3_sync",
                     "q3_last_error", "q3_quantize_q8_0", "q3_quantize_affine4", "q3_affine4_to_f16"):
        assert required in names


def test_library_exports_every_declared_symbol(libq3):
    missing = [n for n in declared_functions() if not hasattr(libq3, n)]
    assert not missing, missing


def test_last_error_is_empty_string_initially(libq3):
    libq3.q3_last_error.restype = ctypes.c_char_p
    assert isinstance(libq3.q3_last_error(), bytes)


def test_host_side_argument_checks_need_no_gpu(libq3):
    # NULL arguments are rejected before any CUDA call
    libq3.q3_last_error.restype = ctypes.c_char_p
    assert libq3.q3_model_create(None, None, 16, None, None) == -1
    assert libq3.q3_session_eval(None, None, 1, None, None) == -1
    assert libq3.q3_quantize_q8_0(None, ctypes.c_int64(32), None, None) == -1
    assert libq3.q3_quantize_affine4(None, ctypes.c_int64(32), None, None) == -1
    assert libq3.q3_affine4_to_f16(None, ctypes.c_int64(32), None, None) == -1
    # misaligned pointers and ragged lengths are rejected before any memory access
    p16, p1 = ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 1)
    assert libq3.q3_quantize_affine4(p1, ctypes.c_int64(32), p16, None) == -1
    assert libq3.q3_quantize_affine4(p16, ctypes.c_int64(32), p1, None) == -1
    assert libq3.q3_quantize_affine4(p16, ctypes.c_int64(33), p16, None) == -1
    assert libq3.q3_affine4_to_f16(p1, ctypes.c_int64(32), p16, None) == -1
    assert libq3.q3_affine4_to_f16(p16, ctypes.c_int64(32), ctypes.c_void_p((1 << 20) + 8), None) == -1
    assert libq3.q3_op_matmul(None, None, 128, 1, 64, None, 0, None) == -1
    assert b"bad argument" in libq3.q3_last_error()

    # the multi-logit round, the prefill attention operator and the path
    # selectors reject bad arguments the same way
    assert libq3.q3_session_eval_n(None, None, 4, 2, None, None) == -1
    assert libq3.q3_op_prefill_attention(None, None, None, 1, 1, 0, 1, 32, 8, None, 1, None) == -1
    assert libq3.q3_model_set_prefill_tc(None, 1) == -1
    assert libq3.q3_model_set_fused_decode(None, 1) == -1
    assert libq3.q3_model_prefill_tc(None) == 0
    assert libq3.q3_model_fused_decode(None) == 0


def test_config_checks_need_no_gpu(libq3):
    # a config is checked before any CUDA call: an unknown weight scheme fails loudly
    from qwen3_dense_decoder_gb300 import _Config
    libq3.q3_last_error.restype = ctypes.c_char_p
    out = ctypes.c_void_p()
    for scheme, msg in ((3, b"unknown weight scheme 3"), (-1, b"unknown weight scheme -1")):
        cfg = _Config(2, 1024, 16, 8, 128, 3072, 4096, 64, 1e6, 1e-6, 1, scheme)
        assert libq3.q3_model_create(ctypes.byref(cfg), None, 16, None, ctypes.byref(out)) == -1
        assert msg in libq3.q3_last_error()
        assert out.value is None
    cfg = _Config(2, 1024, 16, 8, 64, 3072, 4096, 64, 1e6, 1e-6, 1, 0, 0)
    assert libq3.q3_model_create(ctypes.byref(cfg), None, 16, None, ctypes.byref(out)) == -1
    assert b"head_dim must be 128" in libq3.q3_last_error()


def test_unknown_kv_cache_scheme_is_refused(libq3):
    # a K/V cache scheme other than BF16 and Q8_0 is refused before any CUDA call
    libq3.q3_last_error.restype = ctypes.c_char_p
    from qwen3_dense_decoder_gb300 import _Config
    out = ctypes.c_void_p()
    cfg = _Config(2, 1024, 16, 8, 128, 3072, 4096, 64, 1e6, 1e-6, 1, 0, 7)
    assert libq3.q3_model_create(ctypes.byref(cfg), None, 16, None, ctypes.byref(out)) == -1
    assert b"K/V cache scheme" in libq3.q3_last_error()


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "qwen3_dense_decoder_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "q3_oracle" not in text and "orc_" not in text, f


def test_noalloc_binding_checks_shapes_before_any_launch():
    """The library cannot see a buffer's extent, so the binding refuses a short
    x or y (which the kernels would read or write past its end) before it
    touches the library: CPU tensors never reach a launch."""
    import torch
    import qwen3_dense_decoder_gb300 as q3
    w = torch.zeros(256, 128, dtype=torch.float16)
    y = torch.zeros(40, 256, dtype=torch.float32)
    bad = [
        (w, torch.zeros(40, 128, dtype=torch.float16), y),          # x has n rows, not round_up(n, 256)
        (w, torch.zeros(256, 64, dtype=torch.float16), y),          # x's K differs from w's
        (w, torch.zeros(256, 128, dtype=torch.float16), torch.zeros(39, 256)),   # y too short
        (w, torch.zeros(256, 128, dtype=torch.float16), torch.zeros(40, 256, dtype=torch.float16)),
        (w, torch.zeros(256, 128, dtype=torch.float16).t().contiguous().t(), y),  # not contiguous
        (w, torch.zeros(256, 128, dtype=torch.float16), y),          # CPU tensors
    ]
    for wi, xi, yi in bad:
        with pytest.raises(ValueError):
            q3.op_matmul_splitk_noalloc(wi, xi, 40, 2, yi)
