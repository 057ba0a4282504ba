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


def test_attention_heads_mode_is_checked(lib):
    assert lib.mt_attn_set_heads_per_cta(3) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_attn_set_heads_per_cta(-1) == ml.MT_ERR_INVALID_ARG
    assert "heads-per-CTA" in ml.mt_last_error()
    for mode in (1, 2, 0):                 # 0 (automatic) is left in place
        assert lib.mt_attn_set_heads_per_cta(mode) == ml.MT_OK


# Llama-3-8B-shaped layer, 4096 tokens, on 152 SMs / 76 resident CTA pairs (epilogue codes:
# 0 store, 1 residual, 2 QKV, 3 SwiGLU, 4 GeLU)
LLAMA8B_GEMMS = {
    # name: (N, K, epilogue, expected plan)
    "qkv": (6144, 4096, 2, dict(pair=1, tiles_m=16, tiles_n=24, split=1, ksplit=4, full_units=380,
                                num_units=396, epi_split=2)),
    "o": (4096, 4096, 1, dict(pair=1, tiles_m=16, tiles_n=16, split=1, ksplit=2, full_units=228,
                              num_units=284, epi_split=2)),
    "fc1": (14336, 4096, 3, dict(pair=1, tiles_m=16, tiles_n=112, split=1, ksplit=1, full_units=1792,
                                 num_units=1792, epi_split=1)),
    "fc2": (4096, 14336, 1, dict(pair=1, tiles_m=16, tiles_n=16, split=1, ksplit=2, full_units=228,
                                 num_units=284, epi_split=1)),
}


@pytest.mark.parametrize("name", sorted(LLAMA8B_GEMMS))
def test_gemm_plan_llama8b(lib, name):
    """The tail of each projection as measured: QKV 4 tail tiles in 4 K ranges, the output
    projection and fc2 28 tail tiles in 2, fc1's 44 left whole (88 pieces exceed 76 pairs)."""
    N, K, epi, want = LLAMA8B_GEMMS[name]
    assert ml.mt_gemm_plan(4096, N, K, epi, head_dim=128) == want


def test_gemm_plan_tail_forms(lib):
    o = dict(M=4096, N=4096, K=4096, epilogue=1)
    # handle-less calls and tail split mode 1 cut the 28 tail tiles into 2 pieces along N
    for plan in (ml.mt_gemm_plan(**o, with_handle=False), _with_tail_split(1, lambda: ml.mt_gemm_plan(**o))):
        assert (plan["split"], plan["ksplit"], plan["num_units"]) == (2, 1, 228 + 56)
        assert plan["epi_split"] == 1
    # E4M3 operands: 128-deep K blocks, 32 for K = 4096: QKV's 4 tail tiles still take 4 ranges (each
    # drops 24 blocks), the output projection's 28 take 2
    f8 = ml.mt_gemm_plan(4096, 6144, 4096, 2, head_dim=128, fp8=True)
    assert f8["ksplit"] == 4
    assert ml.mt_gemm_plan(**o, fp8=True)["ksplit"] == 2
    # K = 1024 (16 K blocks): no range would drop 16 of them, so the N cut (GPT-345M's QKV)
    gpt = ml.mt_gemm_plan(4096, 3072, 1024, 2, head_dim=64)
    assert (gpt["ksplit"], gpt["epi_split"]) == (1, 2)
    # 128 rows or fewer: the one-CTA kernel, 128 x 256 tiles, never K ranges
    small = ml.mt_gemm_plan(128, 4096, 4096, 0)
    assert (small["pair"], small["tiles_m"], small["ksplit"]) == (0, 1, 1)
    # a whole wave and no tail: nothing to cut
    full = ml.mt_gemm_plan(256 * 76, 256, 4096, 0)
    assert (full["split"], full["ksplit"], full["num_units"]) == (1, 1, 76)


def test_gemm_plan_of_the_ksplit_test_layers(lib):
    """The GPU K-split tests' layers (hidden 2048, 16 x 128 heads, 4 groups) put 3, 2 and 4 K ranges
    under the QKV, SwiGLU, residual and GeLU epilogues."""
    ks = lambda M, N, K, epi: ml.mt_gemm_plan(M, N, K, epi, head_dim=128)["ksplit"]
    assert ks(2048, 3072, 2048, 2) == 3      # QKV, tail 20 tiles
    assert ks(2048, 4096, 2048, 3) == 2      # fc1 SwiGLU, tail 28
    assert ks(2560, 2048, 2048, 1) == 4      # output projection, tail 4
    assert ks(2560, 2048, 4096, 1) == 4      # fc2
    assert ks(2560, 4096, 2048, 3) == 4      # fc1 SwiGLU, tail 16
    assert ks(2560, 6144, 2048, 2) == 4      # MHA QKV, tail 12
    assert ks(2560, 8192, 2048, 4) == 4      # fc1 GeLU, tail 16
    assert ks(2560, 2048, 2048, 0) == 4      # TP = 2 rank's fc2 partial (K = 2048 per rank)


def test_gemm_plan_of_the_backward_ksplit_layers(lib):
    """The backward's dX GEMMs (dX^T = W^T dY^T: M = the layer's input width, N = the tokens, K = its
    output width) in the GPU backward tests' K-split layers: fc1's is a single partial wave cut into 4
    ranges of K (the second layer with a ragged last K block, K = 2056); at the Llama-3-8B shape the
    dX of the output projection, QKV and fc1 cut their 28-tile tails into 2.  The weight-gradient
    GEMMs, which run beside them on a stream of their own, are planned without K ranges (as the
    handle-less calls are) and cut their tails along N.  Planning does not depend on the operands'
    layout."""
    ks = lambda M, N, K, handle=True: ml.mt_gemm_plan(M, N, K, 0, with_handle=handle)
    for T in (2048, 2064):
        assert ks(512, T, 2048)["ksplit"] == 4       # dX_fc1 (SwiGLU rows 2048)
    assert ks(512, 2064, 2056)["ksplit"] == 4        # dX_fc1, GeLU ffn 2056: a ragged last K block
    assert ks(4096, 4096, 4096)["ksplit"] == 2       # Llama-3-8B dX_o
    assert ks(4096, 4096, 6144)["ksplit"] == 2       # dX_qkv
    assert ks(4096, 4096, 28672)["ksplit"] == 2      # dX_fc1
    for M, N, K in ((512, 1024, 2048), (6144, 4096, 4096), (4096, 4096, 4096)):  # dW_fc2, dW_qkv, dW_o
        plan = ks(M, N, K, handle=False)
        assert plan["ksplit"] == 1 and plan["split"] == 2


def _with_tail_split(mode, fn):
    ml.mt_gemm_set_tail_split(mode)
    try:
        return fn()
    finally:
        ml.mt_gemm_set_tail_split(0)


def test_gemm_plan_invariants(lib):
    """Over a sweep of shapes: the units cover the tiles, a cut tail still fits in one wave, K
    ranges only where each drops at least 16 K blocks."""
    for M in (129, 1000, 4096, 8192):
        for N, epi in ((1024, 0), (4096, 1), (6144, 2), (14336, 3), (8192, 4), (520, 0)):
            for K in (512, 1024, 2048, 4096, 14336):
                for handle in (True, False):
                    p = ml.mt_gemm_plan(M, N, K, epi, head_dim=128, with_handle=handle)
                    tiles = p["tiles_m"] * p["tiles_n"]
                    workers = 76 if p["pair"] else 152
                    rest = tiles - p["full_units"]
                    pieces = max(p["split"], p["ksplit"])
                    assert p["split"] == 1 or p["ksplit"] == 1
                    if pieces == 1:
                        assert p["full_units"] == p["num_units"] == tiles
                    else:
                        assert p["full_units"] % workers == 0 and 0 < rest
                        assert p["num_units"] == p["full_units"] + rest * pieces and rest * pieces <= workers
                    if p["ksplit"] > 1:
                        nkb = (K + 63) // 64
                        assert handle and p["pair"] and nkb - nkb // p["ksplit"] >= 16
                    assert p["epi_split"] in (1, 2)


def test_gemm_plan_checks_arguments(lib):
    out = (ctypes.c_int * 8)()
    assert lib.mt_gemm_plan(0, 1, 1, 0, 0, 0, 1, 152, 76, out) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_gemm_plan(1, 1, 1, 5, 0, 0, 1, 152, 76, out) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_gemm_plan(256, 768, 64, 2, 96, 0, 1, 152, 76, out) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_gemm_plan(256, 256, 64, 0, 0, 0, 1, 152, 77, out) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_gemm_plan(256, 256, 64, 0, 0, 0, 1, 152, 76, None) == ml.MT_ERR_INVALID_ARG
    assert lib.mt_gemm_plan(256, 256, 64, 0, 0, 0, 1, 152, 76, out) == ml.MT_OK


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
