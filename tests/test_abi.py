"""The C-ABI library loads and exports every symbol include/mt_layer.h declares; host-side argument
checks reject bad input before touching the GPU.  No kernel runs here (CPU only)."""
import ctypes
import os
import re

import pytest

from megatron_tensor_transformer_gpt_gb300 import build as _build
from megatron_tensor_transformer_gpt_gb300 import mt_layer as ml

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return ml.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mt_layer.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mt_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_layer_calls():
    names = declared_functions()
    for n in ("mt_layer_create", "mt_layer_forward", "mt_layer_destroy", "mt_layer_forward_attn",
              "mt_layer_forward_mlp", "mt_layer_status", "mt_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    assert set(declared_functions()) <= set(ml._SIGS)


@pytest.mark.parametrize("args,code,msg", [
    ((256, 4, 4, 96, 688, 0, 0, 1e4, 1, 0), ml.MT_ERR_UNSUPPORTED, "head_dim"),
    ((256, 6, 4, 64, 688, 0, 0, 1e4, 1, 0), ml.MT_ERR_UNSUPPORTED, "query_groups"),
    ((256, 4, 4, 64, 688, 0, 0, 1e4, 8, 0), ml.MT_ERR_UNSUPPORTED, "divisible"),
    ((256, 4, 4, 64, 688, 0, 0, 1e4, 2, 2), ml.MT_ERR_INVALID_ARG, "tp_rank"),
    ((250, 4, 4, 64, 688, 0, 0, 1e4, 1, 0), ml.MT_ERR_UNSUPPORTED, "hidden"),
    ((256, 4, 4, 64, 684, 0, 0, 1e4, 1, 0), ml.MT_ERR_UNSUPPORTED, "ffn"),
    ((256, 4, 4, 64, 688, 7, 0, 1e4, 1, 0), ml.MT_ERR_INVALID_ARG, "norm"),
    ((256, 4, 4, 64, 688, 0, 9, 1e4, 1, 0), ml.MT_ERR_INVALID_ARG, "activation"),
    ((256, 4, 4, 64, 688, 0, 0, -1.0, 1, 0), ml.MT_ERR_INVALID_ARG, "rope_base"),
    ((0, 4, 4, 64, 688, 0, 0, 1e4, 1, 0), ml.MT_ERR_INVALID_ARG, "positive"),
])
def test_create_rejects_bad_shapes_before_the_device(lib, args, code, msg):
    h = ctypes.c_void_p(123)
    rc = lib.mt_layer_create(*args, ctypes.byref(h))
    assert rc == code
    assert h.value is None
    assert msg in ml.mt_last_error()


def test_null_arguments(lib):
    assert lib.mt_layer_create(256, 4, 4, 64, 688, 0, 0, 1e4, 1, 0, None) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_layer_forward(None, None, 1, 1, None, None, None) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_layer_forward_attn(None, None, 1, 1, None, None, None) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_layer_forward_mlp(None, None, 1, 1, None, None, None) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_layer_forward_host(None, None, 1, 1, None, None, None) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_layer_set_eps(None, 1e-5) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_layer_status(None) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_gemm_bf16(None, None, None, 1, 8, 8, None) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_selftest_bounded_wait(0) == ml.MT_ERR_INVALID_ARG
    lib.mt_layer_destroy(None)  # no-op


def test_gemm_checks_shapes_on_host(lib):
    # 16-byte aligned dummy addresses: rejected on the K/N rule before any device work
    a = ctypes.c_void_p(0x1000)
    assert lib.mt_gemm_bf16(a, a, a, 16, 12, 64, None) == ml.MT_ERR_UNSUPPORTED
    assert lib.mt_gemm_bf16(a, a, a, 16, 16, 60, None) == ml.MT_ERR_UNSUPPORTED
    assert lib.mt_gemm_bf16(ctypes.c_void_p(0x1004), a, a, 16, 16, 64, None) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_gemm_bf16(a, a, a, 0, 16, 64, None) == ml.MT_ERR_INVALID_ARG


def test_last_error_is_cleared_by_success_and_thread_local(lib):
    import threading
    lib.mt_layer_set_eps(None, 1.0)
    assert "NULL" in ml.mt_last_error()
    seen = []
    th = threading.Thread(target=lambda: seen.append(ml.mt_last_error()))
    th.start()
    th.join()
    assert seen == [""]


def test_gemm_pairing_mode_is_checked(lib):
    assert lib.mt_gemm_set_pairing(3) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_gemm_set_pairing(-1) == ml.MT_ERR_INVALID_ARG
    assert "pairing" in ml.mt_last_error()
    for mode in (1, 2, 0):                 # 0 (automatic) is left in place
        assert lib.mt_gemm_set_pairing(mode) == ml.MT_OK


def test_gemm_tail_split_mode_is_checked(lib):
    assert lib.mt_gemm_set_tail_split(2) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_gemm_set_tail_split(-1) == ml.MT_ERR_INVALID_ARG
    assert "tail split" in ml.mt_last_error()
    for mode in (1, 0):                    # 0 (automatic) is left in place
        assert lib.mt_gemm_set_tail_split(mode) == ml.MT_OK


def test_profile_mask_and_launch_count_check_arguments(lib):
    assert lib.mt_layer_profile_enable(None, 1) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_layer_launch_count(None, None) == ml.MT_ERR_INVALID_ARG


def test_transposed_gemm_checks_arguments(lib):
    a = ctypes.c_void_p(0x1000)
    assert lib.mt_gemm_bf16_t(None, 0, a, 0, a, 8, 8, 8, None) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_gemm_bf16_t(a, 2, a, 0, a, 8, 8, 8, None) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_gemm_bf16_t(a, 1, a, 0, a, 12, 8, 16, None) == ml.MT_ERR_UNSUPPORTED  # A [K, M] needs M % 8
    assert lib.mt_gemm_bf16_t(a, 0, a, 1, a, 8, 12, 16, None) == ml.MT_ERR_UNSUPPORTED  # B [K, N] needs N % 8
