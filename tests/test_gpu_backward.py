"""GPU parity of the layer backward pass (mt_layer_backward, TP=1) against the float64 backward
oracle (itself pinned by PyTorch autograd and finite differences).

Gradient tolerance, from the arithmetic: the GPU chains bf16-rounded intermediates (P, dS, the
activation and norm gradients, dqkv; each ~2^-9 relative) through fp32-accumulated GEMMs, so
every gradient tensor must satisfy |gpu - oracle| <= 3e-2 * max|oracle| element by element and a
relative Frobenius error below 2e-2.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import backward as ob
from oracle import layer as ol
from megatron_tensor_transformer_gpt_gb300 import mt_layer as ml
from tests.gpu_util import DeviceLayer, to_dev, to_f64

pytestmark = pytest.mark.gpu


def assert_grad_close(got, want, what):
    got, want = np.asarray(got, np.float64).reshape(want.shape), np.asarray(want, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite"
    scale = np.max(np.abs(want))
    err = np.abs(got - want)
    assert err.max() <= 3e-2 * scale + 1e-12, f"{what}: max err {err.max():.3e} vs max|grad| {scale:.3e}"
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    assert rel < 2e-2, f"{what}: relative Frobenius error {rel:.3e}"


CFGS = [
    synth.CONFIGS["tiny"],
    synth.LayerConfig("bw_gqa", batch=2, seq=128, hidden=256, heads=8, groups=2, head_dim=64, ffn=512,
                      rope_base=1e4),
    synth.LayerConfig("bw_ln", batch=2, seq=64, hidden=256, heads=2, groups=2, head_dim=128, ffn=384,
                      norm="layer", act="gelu_tanh", rope_base=0.0, bias=True),
    synth.LayerConfig("bw_mqa", batch=1, seq=200, hidden=512, heads=4, groups=1, head_dim=128, ffn=1024,
                      rope_base=5e5, bias=True),
]


@pytest.mark.parametrize("cfg", CFGS, ids=lambda c: c.name)
def test_backward_matches_oracle(cfg):
    inp = synth.make_inputs(cfg, seed=81, affine="random", biases="random")
    T, H = cfg.tokens, cfg.hidden
    dy_bits = synth.f32_to_bf16_bits(np.random.default_rng(82).standard_normal((T, H)).astype(np.float32))
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(T, H)
    dy = to_dev(dy_bits)
    dx = torch.empty_like(x)
    grads = {k: (None if v is None else torch.empty_like(v)) for k, v in dl.tens.items()}
    dl.layer.backward(x, dy, cfg.seq, cfg.batch, dl.w, dx, grads)
    torch.cuda.synchronize()
    dl.layer.status()
    want = ob.layer_backward(cfg, inp, ol.bf16_to_f64(dy_bits))
    assert_grad_close(to_f64(dx), want["x"], "dx")
    for name, t in grads.items():
        if t is None:
            assert want[name] is None, name
            continue
        assert_grad_close(to_f64(t), want[name], name)
    dl.close()


def test_backward_rejects_unsupported():
    cfg = synth.CONFIGS["tiny"]
    layer = ml.Layer.from_config(cfg, tp_rank=0, tp_size=2)
    z = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ml.MtError) as e:
        ml.mt_layer_backward(layer.handle, z.data_ptr(), z.data_ptr(), 128, 1, ml.MtWeights(), z.data_ptr(),
                             ml.MtGrads(), None)
    assert e.value.code == ml.MT_ERR_UNSUPPORTED
    layer.close()
