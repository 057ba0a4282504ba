"""GPU parity of the FP8 (E4M3) path against the float64 oracle of the same quantised values.

* mt_quantize_e4m3 (current scaling of a weight) gives exactly the oracle's codes and factors.
* mt_gemm_e4m3 on seeded random codes matches the exact product (fp32 accumulation, bf16 out).
* mt_layer_forward_fp8 with given activation scales, stage by stage (tests/fp8_check.py): the
  codes of all four quantised activations (normed x, attention output, normed h, MLP hidden),
  each against the oracle's codes of the same values; the stored h against the oracle's attention
  block; y against the oracle's MLP block run from the GPU's own h.  A quantised code is an integer
  decided by floating point, so the oracle takes the kernels' storage precision for the stored
  intermediates the codes depend on (q, k bf16, v fp16, h bf16), and the MLP stage starts from the
  h the GPU stored.  The delayed-scaling history yields scale = 448 / max(history) after each call.

Whole-layer tolerance as well.  Two FP8 computations whose inputs to a cast differ by bf16
rounding round some values to neighbouring E4M3 codes, 6-12% apart, so y is also checked element
by element against the end-to-end FP8 oracle within
    |gpu - oracle_fp8| <= 2e-2 max|oracle_fp8| + 1e-3 + |oracle_fp8 - oracle_exact|_max,
and the GPU result may be no further from the exact layer than 1.5x the oracle FP8 result is.
That bound alone would not notice a skipped cast (y is dominated by the residual); the stage
checks would (the CPU tests plant each skipped cast in the oracle and see them fail).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import fp8 as of
from oracle import layer as ol
from megatron_tensor_transformer_gpt_gb300 import mt_layer as ml
from tests import fp8_check as fc
from tests.gpu_util import DeviceLayer, assert_layer_close, sample_rows, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _stream():
    return torch.cuda.current_stream().cuda_stream


def quantize_on_device(t):
    """(codes uint8 tensor, amax_deq float tensor[2]) of a bf16 device tensor."""
    codes = torch.empty(t.numel(), dtype=torch.uint8, device="cuda")
    slot = torch.empty(2, dtype=torch.float32, device="cuda")
    ml.mt_quantize_e4m3(t.data_ptr(), t.numel(), codes.data_ptr(), slot.data_ptr(), _stream())
    return codes, slot


@pytest.mark.parametrize("shape,std", [((64, 48), 0.02), ((1376, 256), 0.02), ((4096, 1024), 1.0), ((8, 8), 0.0)])
def test_quantize_matches_oracle_bit_for_bit(shape, std):
    rng = np.random.default_rng(shape[0])
    w = synth.f32_to_bf16_bits((rng.standard_normal(shape) * std).astype(np.float32))
    codes, slot = quantize_on_device(to_dev(w))
    torch.cuda.synchronize()
    want = of.quantize_weight(w)
    assert np.array_equal(codes.cpu().numpy(), want["codes"].reshape(-1))
    amax, deq = slot.cpu().numpy()
    assert amax == np.float32(np.max(np.abs(ol.bf16_to_f64(w))))
    assert deq == np.float32(1.0) / want["scale"]


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 520, 208), (1000, 1376, 688), (1, 8, 16),
                                   (2048, 3072, 4096)])
def test_gemm_e4m3_matches_exact_product(M, N, K):
    a = synth.random_e4m3_codes((M, K), seed=M + K)
    b = synth.random_e4m3_codes((N, K), seed=N + 7 * K)
    deq = torch.tensor([0.01, 0.03], dtype=torch.float32, device="cuda")
    A, B = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ml.mt_gemm_e4m3(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, deq.data_ptr(), deq.data_ptr() + 4, _stream())
    torch.cuda.synchronize()
    want = (of.e4m3_decode(a) @ of.e4m3_decode(b).T) * float(np.float32(0.01)) * float(np.float32(0.03))
    err = np.abs(to_f64(C) - want)
    assert np.all(err <= 4e-3 * np.abs(want) + 1e-3 * np.max(np.abs(want))), err.max()


class Fp8Layer:
    """A layer handle with FP8 enabled and its projection weights quantised on the device."""

    def __init__(self, cfg, inp, history=1024):
        self.dl = DeviceLayer(cfg, inp)
        ml.mt_layer_fp8_enable(self.dl.layer.handle, history)
        self.keep = []
        w8 = ml.MtFp8Weights()
        for name in ("w_qkv", "w_o", "w_fc1", "w_fc2"):
            codes, slot = quantize_on_device(self.dl.tens[name])
            self.keep += [codes, slot]
            setattr(w8, name, codes.data_ptr())
            setattr(w8, name.replace("w_", "deq_"), slot.data_ptr() + 4)
        self.w8 = w8

    def forward(self, x):
        cfg = self.dl.cfg
        y = torch.empty(cfg.tokens, cfg.hidden, dtype=torch.bfloat16, device="cuda")
        self.dl.layer.workspace(cfg.seq, cfg.batch)
        ml.mt_layer_forward_fp8(self.dl.layer.handle, x.data_ptr(), cfg.seq, cfg.batch, self.dl.w, self.w8,
                                y.data_ptr(), _stream())
        return y


def _scales_from(cfg, inp, rows=None, wq=None):
    amax = of.layer_forward_fp8(cfg, inp, (1, 1, 1, 1), rows=rows, wq=wq)["amax"]
    return [float(of.scale_from_amax(amax[n])) for n in of.ACT_NAMES]


def assert_fp8_close(got, want_fp8, want_exact, what):
    envelope = np.max(np.abs(want_fp8 - want_exact))
    err = np.abs(got - want_fp8)
    bound = 2e-2 * np.max(np.abs(want_fp8)) + 1e-3 + envelope
    assert np.all(np.isfinite(got)), what
    assert err.max() <= bound, f"{what}: max |gpu - oracle_fp8| {err.max():.4f} > {bound:.4f}"
    dev_gpu, dev_ref = np.max(np.abs(got - want_exact)), envelope
    assert dev_gpu <= 1.5 * dev_ref + 1e-3, f"{what}: gpu FP8 deviation {dev_gpu:.4f} vs oracle FP8 {dev_ref:.4f}"


def check_first_codes(f8, cfg, inp, scales):
    """The normed input's E4M3 codes: decided from the same bf16 x on both sides."""
    T, H = cfg.tokens, cfg.hidden
    xn8 = f8.dl.layer.region(cfg.seq, cfg.batch, "xn")[: T * H].view(T, H).cpu().numpy()
    xn = ol.apply_norm(cfg, ol._tokens(inp["x"], cfg), ol._w(inp, "norm1_w"), ol._w(inp, "norm1_b"))
    fc.assert_codes_close(xn8, of.quantize(xn, np.float32(scales[0])), 1e-4, "xn codes")


def check_stages(f8, cfg, inp, scales, wq, y, rows=None):
    """The attention output's codes and the stored h against the oracle's attention block; the codes
    of normed h and of the MLP hidden, and y, against the oracle's MLP block from the GPU's own h."""
    T, H, S, B = cfg.tokens, cfg.hidden, cfg.seq, cfg.batch
    rows = np.arange(T) if rows is None else np.asarray(rows)
    L = f8.dl.layer

    def region(name, cols, dtype=torch.uint8):
        t = L.region(S, B, name).view(dtype)[: T * cols].view(T, cols)
        return t[torch.from_numpy(rows).to(t.device)].cpu()

    s = [np.float32(v) for v in scales]
    att = of.attention_block_fp8(cfg, inp, scales, rows=rows, wq=wq, storage_rounding=True)
    # the GPU forms o from fp16 probabilities (relative rounding 2^-11, and 2^-10 from the half-precision
    # exponential): |o_gpu - o| <= 2^-9 max|v| leaves a code at most that far (scaled) from the oracle's
    slack = 2.0 ** -9 * float(np.max(np.abs(att["v"]))) * float(s[1])
    fc.assert_codes_close(region("o", cfg.heads * cfg.head_dim).numpy(), of.quantize(att["o"], s[1]), 5e-2,
                          "attention-output codes", slack=slack)
    h = to_f64(region("h", H, torch.bfloat16))
    fc.assert_attention_stage(h, att["h"], ol.layer_forward(cfg, inp, rows=rows)["h"], "attention stage")
    hn = ol.apply_norm(cfg, h, ol._w(inp, "norm2_w"), ol._w(inp, "norm2_b"))
    hn8 = region("hn", H).numpy()
    fc.assert_codes_close(hn8, of.quantize(hn, s[2]), 1e-3, "normed-h codes")
    w_fc1 = of.dequantize(wq["w_fc1"]["codes"], wq["w_fc1"]["scale"])
    a = ol.activation(cfg, ol.linear(of.dequantize(hn8, s[2]), w_fc1, ol._w(inp, "b_fc1")))
    fc.assert_codes_close(region("a", cfg.ffn).numpy(), of.quantize(a, s[3]), 1e-3, "MLP-hidden codes")
    b_fc2 = ol._w(inp, "b_fc2")
    y_exact = h + ol.mlp_partial(cfg, 1, h, inp) + (0.0 if b_fc2 is None else b_fc2)
    fc.assert_mlp_stage(y, of.mlp_block_fp8(cfg, inp, scales, h, wq=wq)["y"], y_exact, "MLP stage")


@pytest.mark.parametrize("cfg", [
    synth.CONFIGS["tiny"],
    synth.LayerConfig("f8gqa", batch=2, seq=192, hidden=512, heads=8, groups=2, head_dim=64, ffn=1024,
                      rope_base=1e4),
    synth.LayerConfig("f8ln", batch=1, seq=200, hidden=512, heads=4, groups=4, head_dim=128, ffn=1024,
                      norm="layer", act="gelu_tanh", rope_base=0.0, bias=True),
    synth.LayerConfig("f8gqa128", batch=2, seq=300, hidden=512, heads=8, groups=2, head_dim=128, ffn=1024,
                      rope_base=5e5),                     # four heads per group: the CTA-pair attention
], ids=lambda c: c.name)
def test_fp8_layer_matches_oracle(cfg):
    inp = synth.make_inputs(cfg, seed=61, affine="random", biases="random")
    scales = _scales_from(cfg, inp)
    f8 = Fp8Layer(cfg, inp)
    ml.mt_layer_fp8_set_scales(f8.dl.layer.handle, scales)
    y = f8.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden))
    torch.cuda.synchronize()
    f8.dl.layer.status()
    check_first_codes(f8, cfg, inp, scales)
    got = to_f64(y)
    check_stages(f8, cfg, inp, scales, of.quantize_weights(inp), got)
    want = of.layer_forward_fp8(cfg, inp, scales)["y"]
    assert_fp8_close(got, want, ol.layer_forward(cfg, inp)["y"], f"fp8 layer {cfg.name}")
    f8.dl.close()


def test_fp8_layer_llama8b_sampled_rows():
    cfg = synth.CONFIGS["llama8b"]
    inp = synth.make_inputs(cfg, seed=0)
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([np.arange(16), np.arange(cfg.tokens - 16, cfg.tokens),
                                     rng.integers(0, cfg.tokens, 32)]))
    wq = of.quantize_weights(inp)
    scales = _scales_from(cfg, inp, rows=rows, wq=wq)
    f8 = Fp8Layer(cfg, inp)
    ml.mt_layer_fp8_set_scales(f8.dl.layer.handle, scales)
    y = f8.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden))
    torch.cuda.synchronize()
    f8.dl.layer.status()
    check_first_codes(f8, cfg, inp, scales)
    got = to_f64(y[torch.from_numpy(rows).cuda()])
    check_stages(f8, cfg, inp, scales, wq, got, rows=rows)
    f8.dl.close()
    assert_fp8_close(got, of.layer_forward_fp8(cfg, inp, scales, rows=rows, wq=wq)["y"],
                     ol.layer_forward(cfg, inp, rows=rows)["y"], "fp8 llama8b")


def test_delayed_scaling_history():
    cfg = synth.LayerConfig("f8h", batch=1, seq=256, hidden=512, heads=8, groups=2, head_dim=64, ffn=1024,
                            rope_base=1e4)
    inp = synth.make_inputs(cfg, seed=62, affine="random")
    f8 = Fp8Layer(cfg, inp, history=3)
    h = f8.dl.layer.handle
    s0 = _scales_from(cfg, inp)
    ml.mt_layer_fp8_set_scales(h, s0)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    want_amax = of.layer_forward_fp8(cfg, inp, s0)["amax"]
    seen = []
    for call in range(5):
        xs = x * (1.0 + 0.25 * call)            # a different input each call, so the amaxes move
        f8.forward(xs.contiguous())
        sc, last = ml.mt_layer_fp8_state(h)
        seen.append(last)
        window = np.max(np.array(seen[-3:], dtype=np.float32), axis=0)
        expect = [np.float32(448.0) / np.float32(m) for m in window]
        assert np.array_equal(np.array(sc, dtype=np.float32), np.array(expect, dtype=np.float32)), (call, sc, expect)
        if call == 0:
            for i, n in enumerate(of.ACT_NAMES):
                assert abs(last[i] - want_amax[n]) <= 0.03 * want_amax[n], (n, last[i], want_amax[n])
    f8.dl.close()
