"""GPU parity of the CTA-pair GEMM kernel (two CTAs sharing one M = 256 tcgen05.mma per 256 x 256
tile) against the float64 oracle, through every epilogue the layer uses.

mt_gemm_set_pairing(2) forces the pair kernel wherever M > 128, so small layers, ragged M (a pair
whose second CTA has no valid rows), ragged N and the N-split tail pieces all go through it; mode 1
forces the one-CTA kernel on the same inputs.  Tolerances are those of the other parity tests.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import fp8 as of
from oracle import layer as ol
from megatron_tensor_transformer_gpt_gb300 import mt_layer as ml
from tests.gpu_util import DeviceLayer, assert_layer_close, to_dev, to_f64
from tests.test_gpu_parity import small
from tests import test_gpu_backward as tb
from tests import test_gpu_fp8 as tf

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _pairs():
    torch.cuda.set_device(0)
    ml.mt_gemm_set_pairing(2)
    yield
    torch.cuda.synchronize()
    ml.mt_gemm_set_pairing(0)


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("mode", [2, 1], ids=["pairs", "single"])
@pytest.mark.parametrize("M,N,K", [(129, 256, 64), (256, 512, 128), (300, 520, 200), (1000, 1376, 688),
                                   (777, 264, 1032), (4100, 1032, 256), (2048, 3072, 4096)])
def test_gemm_bf16(M, N, K, mode):
    ml.mt_gemm_set_pairing(mode)
    rng = np.random.default_rng(M * 5 + N * 11 + K)
    a = synth.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    b = synth.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32))
    A, B = to_dev(a), to_dev(b)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ml.mt_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, _stream())
    torch.cuda.synchronize()
    want = ol.linear(ol.bf16_to_f64(a), ol.bf16_to_f64(b))
    err = np.abs(to_f64(C) - want)
    assert np.all(err <= 4e-3 * np.abs(want) + 1e-3 * np.max(np.abs(want))), err.max()


def test_pairs_and_single_agree_bitwise():
    """Both kernels add the same fp32 products in the same K order."""
    M, N, K = 1000, 1376, 688
    rng = np.random.default_rng(5)
    A = to_dev(synth.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32)))
    B = to_dev(synth.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32)))
    out = []
    for mode in (2, 1):
        ml.mt_gemm_set_pairing(mode)
        C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        ml.mt_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, _stream())
        out.append(C)
    torch.cuda.synchronize()
    assert torch.equal(out[0], out[1])


@pytest.mark.parametrize("mode", [2, 1], ids=["pairs", "single"])
@pytest.mark.parametrize("a_layout,b_layout", [(0, 1), (1, 1), (1, 0)], ids=["B_KN", "A_KM_B_KN", "A_KM"])
@pytest.mark.parametrize("M,N,K", [(256, 512, 128), (520, 264, 1000), (1000, 1376, 688), (4096, 1024, 4104)])
def test_gemm_transposed_operands(M, N, K, a_layout, b_layout, mode):
    """Operands stored [K, M] / [K, N] are read MN-major by the MMA (the backward's dW and dX form)."""
    ml.mt_gemm_set_pairing(mode)
    rng = np.random.default_rng(M + 3 * N + 7 * K + 11 * a_layout + 13 * b_layout)
    a = synth.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    b = synth.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32))
    A = to_dev(np.ascontiguousarray(a.T) if a_layout else a)
    B = to_dev(np.ascontiguousarray(b.T) if b_layout else b)
    C = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ml.mt_gemm_bf16_t(A.data_ptr(), a_layout, B.data_ptr(), b_layout, C.data_ptr(), M, N, K, _stream())
    torch.cuda.synchronize()
    want = ol.linear(ol.bf16_to_f64(a), ol.bf16_to_f64(b))
    err = np.abs(to_f64(C) - want)
    assert np.all(err <= 4e-3 * np.abs(want) + 1e-3 * np.max(np.abs(want))), err.max()


@pytest.mark.parametrize("M,N,K", [(300, 520, 208), (1000, 1376, 688), (2048, 3072, 4096)])
def test_gemm_e4m3(M, N, K):
    a = synth.random_e4m3_codes((M, K), seed=M + 3 * K)
    b = synth.random_e4m3_codes((N, K), seed=N + 5 * K)
    deq = torch.tensor([0.01, 0.03], dtype=torch.float32, device="cuda")
    A, B = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ml.mt_gemm_e4m3(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, deq.data_ptr(), deq.data_ptr() + 4, _stream())
    torch.cuda.synchronize()
    want = (of.e4m3_decode(a) @ of.e4m3_decode(b).T) * float(np.float32(0.01)) * float(np.float32(0.03))
    err = np.abs(to_f64(C) - want)
    assert np.all(err <= 4e-3 * np.abs(want) + 1e-3 * np.max(np.abs(want))), err.max()


LAYERS = [
    small(),                                                    # QKV d=64 + RoPE, SwiGLU, residual
    small(batch=3, seq=200),                                    # ragged tokens
    small(seq=129, heads=4, groups=1, head_dim=128),            # MQA, d=128, second CTA of the last pair idle
    small(seq=130, head_dim=128, heads=4, groups=1, norm="layer", act="gelu_tanh", rope_base=0.0, bias=True),
    small(hidden=264, heads=2, groups=2, ffn=520, seq=64, batch=5),  # hidden / ffn off the tile grid
    small(batch=2, seq=384, heads=16, groups=2, ffn=1376),
]


@pytest.mark.parametrize("cfg", LAYERS, ids=lambda c: f"b{c.batch}-s{c.seq}-h{c.hidden}-{c.heads}x{c.groups}x"
                                                      f"{c.head_dim}-{c.norm}-{c.act}")
def test_layer_with_pairs(cfg):
    inp = synth.make_inputs(cfg, seed=13, affine="random", biases="random")
    dl = DeviceLayer(cfg, inp)
    y = dl.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden))
    torch.cuda.synchronize()
    dl.layer.status()
    assert_layer_close(to_f64(y), ol.layer_forward(cfg, inp)["y"], cfg.name)
    dl.close()


def test_fp8_layer_with_pairs():
    cfg = synth.LayerConfig("f8pair", batch=2, seq=192, hidden=512, heads=8, groups=2, head_dim=64, ffn=1024,
                            rope_base=1e4, bias=True)
    inp = synth.make_inputs(cfg, seed=62, affine="random", biases="random")
    scales = tf._scales_from(cfg, inp)
    f8 = tf.Fp8Layer(cfg, inp)
    ml.mt_layer_fp8_set_scales(f8.dl.layer.handle, scales)
    y = f8.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden))
    torch.cuda.synchronize()
    f8.dl.layer.status()
    want = of.layer_forward_fp8(cfg, inp, scales)["y"]
    tf.assert_fp8_close(to_f64(y), want, ol.layer_forward(cfg, inp)["y"], "fp8 layer, CTA pairs")
    f8.dl.close()


@pytest.mark.parametrize("cfg", tb.CFGS[1:3], ids=lambda c: c.name)
def test_backward_with_pairs(cfg):
    tb.test_backward_matches_oracle(cfg)
