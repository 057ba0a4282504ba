"""GPU parity of the sequence-parallel epilogue (mt_sp_reduce_add_norm).

Every rank's attention block writes its row-parallel partial; the epilogue, called once per rank
with that rank's sequence slice, sums the partials, adds residual and bias and applies the
pre-MLP norm.  The slices together must give the unsharded layer's h and Norm2(h) (float64 oracle,
layer tolerance |gpu - oracle| <= 2e-2 max|oracle| + 1e-3).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import layer as ol
from megatron_tensor_transformer_gpt_gb300 import mt_layer as ml
from tests.gpu_util import DeviceLayer, assert_layer_close, sample_rows, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _sp_layer(cfg, inp, tp, bounds):
    """Partials of all ranks, then one epilogue call per slice [lo, hi); returns full h, hn."""
    T, H = cfg.tokens, cfg.hidden
    x = to_dev(inp["x"]).reshape(T, H)
    parts = []
    for r in range(tp):
        dl = DeviceLayer(cfg, inp, tp, r)
        parts.append(dl.forward_attn(x))
        dl.close()
    h = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    hn = torch.empty_like(h)
    b_o = to_dev(inp.get("b_o"))
    g, beta = to_dev(inp["norm2_w"]), to_dev(inp.get("norm2_b"))
    stream = torch.cuda.current_stream().cuda_stream
    for lo, hi in bounds:
        ml.mt_sp_reduce_add_norm([p.data_ptr() for p in parts], x[lo:].data_ptr(),
                                 None if b_o is None else b_o.data_ptr(), g.data_ptr(),
                                 None if beta is None else beta.data_ptr(),
                                 ml.MT_NORM_RMS if cfg.norm == "rms" else ml.MT_NORM_LAYER, cfg.eps, T, H, lo, hi - lo,
                                 h[lo:].data_ptr(), hn[lo:].data_ptr(), stream)
    torch.cuda.synchronize()
    return h, hn


def _even(T, tp):
    step = T // tp
    return [(r * step, T if r == tp - 1 else (r + 1) * step) for r in range(tp)]


@pytest.mark.parametrize("tp,norm", [(2, "rms"), (4, "layer"), (8, "rms")])
def test_sp_epilogue_slices_reproduce_unsharded_h_and_norm(tp, norm):
    cfg = synth.LayerConfig("sp", batch=3, seq=200, hidden=512, heads=8, groups=8, head_dim=64, ffn=1024,
                            norm=norm, act="swiglu", rope_base=1e4, bias=True)
    inp = synth.make_inputs(cfg, seed=41, affine="random", biases="random")
    h, hn = _sp_layer(cfg, inp, tp, _even(cfg.tokens, tp))
    want_h = ol.layer_forward(cfg, inp)["h"]
    assert_layer_close(to_f64(h), want_h, "SP h")
    want_hn = ol.apply_norm(cfg, want_h, ol.bf16_to_f64(inp["norm2_w"]), ol.bf16_to_f64(inp["norm2_b"]))
    assert_layer_close(to_f64(hn), want_hn, "SP Norm2(h)")


def test_sp_epilogue_uneven_slices_and_single_partial():
    cfg = synth.LayerConfig("sp1", batch=1, seq=300, hidden=264, heads=4, groups=2, head_dim=64, ffn=520,
                            norm="rms", act="swiglu", rope_base=1e4)
    inp = synth.make_inputs(cfg, seed=42, affine="random")
    h, hn = _sp_layer(cfg, inp, 1, [(0, 7), (7, 129), (129, 300)])
    want_h = ol.layer_forward(cfg, inp)["h"]
    assert_layer_close(to_f64(h), want_h, "SP h, tp=1")
    assert_layer_close(to_f64(hn), ol.rms_norm(want_h, ol.bf16_to_f64(inp["norm2_w"]), cfg.eps), "SP hn, tp=1")


def test_sp_epilogue_llama70b_tp8_sampled_rows():
    cfg = synth.CONFIGS["llama70b_tp8"]
    inp = synth.make_inputs(cfg, seed=0)
    h, hn = _sp_layer(cfg, inp, cfg.tp, _even(cfg.tokens, cfg.tp))
    rows = sample_rows(cfg.tokens, seed=5, n_random=32)
    idx = torch.from_numpy(rows).cuda()
    got_h, got_hn = to_f64(h[idx]), to_f64(hn[idx])
    del h, hn
    torch.cuda.empty_cache()
    want_h = ol.layer_forward(cfg, inp, rows=rows)["h"]
    assert_layer_close(got_h, want_h, "SP h (70B, 8 ranks)")
    assert_layer_close(got_hn, ol.rms_norm(want_h, ol.bf16_to_f64(inp["norm2_w"]), cfg.eps), "SP hn (70B)")


def test_sp_epilogue_rejects_bad_arguments():
    x = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    p = x.data_ptr()
    with pytest.raises(ml.MtError) as e:
        ml.mt_sp_reduce_add_norm([p] * 17, p, None, p, None, ml.MT_NORM_RMS, 1e-5, 16, 64, 0, 16, p, p, None)
    assert e.value.code == ml.MT_ERR_UNSUPPORTED
    with pytest.raises(ml.MtError) as e:
        ml.mt_sp_reduce_add_norm([p], p, None, p, None, ml.MT_NORM_RMS, 1e-5, 16, 64, 8, 9, p, p, None)
    assert e.value.code == ml.MT_ERR_INVALID_ARG
    with pytest.raises(ml.MtError) as e:
        ml.mt_sp_reduce_add_norm([p], p, None, p, None, ml.MT_NORM_LAYER, 1e-5, 16, 64, 0, 16, p, p, None)
    assert e.value.code == ml.MT_ERR_INVALID_ARG
