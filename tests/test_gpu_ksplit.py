"""GPU parity of the K-split tail of the CTA-pair GEMM.

When the tiles of a GEMM's last, partial wave still fit in one wave of SM pairs after cutting each
into 2 to 4 ranges of K, a layer handle's GEMMs compute those tiles as K ranges on different pairs:
the range holding the first K blocks waits for the others' fp32 partial sums, adds them in K order
and runs the epilogue.  The shapes below (on 152 SMs) put that tail under every epilogue the layer
uses: QKV with RoPE (3 ranges), SwiGLU (2 and 4), the residual add of the output projection and
fc2 (4), GeLU and LayerNorm with biases (4 each), and the plain store of a tensor-parallel rank's
partial (fc2 at TP = 2).  Each is checked against the float64 oracle on sampled rows and against
the N-split form of the same call (mt_gemm_set_tail_split(1)), which differs from it only in the
fp32 summation order of the tail tiles.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import layer as ol
from megatron_tensor_transformer_gpt_gb300 import mt_layer as ml
from tests.gpu_util import DeviceLayer, assert_layer_close, sample_rows, tp_sum_on_device, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _tail():
    torch.cuda.set_device(0)
    ml.mt_gemm_set_tail_split(0)
    yield
    torch.cuda.synchronize()
    ml.mt_gemm_set_tail_split(0)


def _cfg(name, **kw):
    base = dict(batch=1, seq=2560, hidden=2048, heads=16, groups=4, head_dim=128, ffn=4096, norm="rms",
                act="swiglu", rope_base=1e4, bias=False)
    base.update(kw)
    return synth.LayerConfig(name, **base)


CFGS = [
    # 2048 tokens: QKV 96 tiles (tail 20 -> 3 K ranges), fc1 256 tiles (tail 28 -> 2)
    _cfg("ks_qkv3_swiglu2", batch=2, seq=1024),
    # 2560 tokens: output projection and fc2 80 tiles (tail 4 -> 4), fc1 320 tiles (tail 16 -> 4)
    _cfg("ks_o4_fc1x4_fc2x4"),
    # MHA, LayerNorm, GeLU, biases: QKV 240 tiles (tail 12 -> 4), fc1 and the rest 4 ranges
    _cfg("ks_gelu_ln_bias", groups=16, ffn=8192, norm="layer", act="gelu_tanh", rope_base=0.0, bias=True),
]


def _many_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count >= 148


@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: c.name)
def test_ksplit_tail_matches_oracle_and_nsplit(cfg):
    inp = synth.make_inputs(cfg, seed=41, affine="random", biases="random")
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    y_k = dl.forward(x).clone()
    y_k2 = dl.forward(x).clone()
    ml.mt_gemm_set_tail_split(1)
    y_n = dl.forward(x).clone()
    torch.cuda.synchronize()
    dl.layer.status()
    dl.close()
    # the partial sums are added in a fixed order: repeated calls agree bit for bit
    assert torch.equal(y_k, y_k2)
    # only the tail tiles' fp32 summation order differs from the N-split form
    assert_layer_close(to_f64(y_k), to_f64(y_n), f"{cfg.name}: K-split against N-split tails")
    if _many_sms():
        assert not torch.equal(y_k, y_n), "no tail tile was cut along K"
    rows = sample_rows(cfg.tokens, seed=5, n_random=96)
    want = ol.layer_forward(cfg, inp, rows=rows)["y"]
    idx = torch.from_numpy(rows).cuda()
    assert_layer_close(to_f64(y_k[idx]), want, f"{cfg.name}: K-split tails")
    assert_layer_close(to_f64(y_n[idx]), want, f"{cfg.name}: N-split tails")


def test_ksplit_tail_of_rank_partials():
    """TP = 2: fc2 (K = 2048 per rank) stores a rank partial through the plain-store epilogue."""
    cfg = _cfg("ks_tp2", heads=16, groups=4, ffn=4096, bias=True)
    inp = synth.make_inputs(cfg, seed=42, affine="random", biases="random")
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    h, y = tp_sum_on_device(cfg, inp, x, 2)
    torch.cuda.synchronize()
    rows = sample_rows(cfg.tokens, seed=6, n_random=64)
    want = ol.layer_forward(cfg, inp, rows=rows)
    idx = torch.from_numpy(rows).cuda()
    assert_layer_close(to_f64(h[idx]), want["h"], "h from summed partials")
    assert_layer_close(to_f64(y[idx]), want["y"], "y from summed partials")
