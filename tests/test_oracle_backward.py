"""Pins for the float64 backward oracle: PyTorch autograd through the independent restatement, and
central finite differences of the forward oracle."""
import numpy as np
import pytest
import torch

import synth
from oracle import backward as ob
from oracle import layer as ol
from tests import torch_restatement


def _cfg(**kw):
    base = dict(name="bw", batch=2, seq=12, hidden=32, heads=4, groups=2, head_dim=8, ffn=40, norm="rms",
                act="swiglu", rope_base=1e4, bias=False)
    base.update(kw)
    return synth.LayerConfig(**base)


CFGS = [_cfg(), _cfg(norm="layer", act="gelu_tanh", rope_base=0.0, bias=True, groups=4),
        _cfg(groups=1, bias=True, batch=1, seq=20)]


@pytest.mark.parametrize("cfg", CFGS, ids=["rms_swiglu_gqa", "ln_gelu_bias_mha", "mqa_bias"])
def test_backward_matches_torch_autograd(cfg):
    inp = synth.make_inputs(cfg, seed=71, affine="random", biases="random")
    dy = np.random.default_rng(72).standard_normal((cfg.tokens, cfg.hidden))
    G = ob.layer_backward(cfg, inp, dy)
    tens = {k: (None if v is None else v.clone().requires_grad_(True))
            for k, v in torch_restatement.as_tensors(inp).items()}
    y = torch_restatement.layer_forward(cfg, inp, tens)
    (y * torch.from_numpy(dy)).sum().backward()
    for k, v in tens.items():
        if v is None:
            assert G[k] is None, k
            continue
        want = v.grad.numpy().reshape(G[k].shape)
        np.testing.assert_allclose(G[k], want, rtol=1e-9, atol=1e-11, err_msg=k)


def test_backward_matches_finite_differences():
    cfg = _cfg(norm="layer", bias=True)
    inp = synth.make_inputs(cfg, seed=73, affine="random", biases="random")
    dy = np.random.default_rng(74).standard_normal((cfg.tokens, cfg.hidden))
    G = ob.layer_backward(cfg, inp, dy)
    f64 = {k: (None if v is None else ol.bf16_to_f64(v)) for k, v in inp.items()}
    rng = np.random.default_rng(75)

    def loss(vals):
        return float(np.sum(ol.layer_forward(cfg, vals)["y"] * dy))
    for name in ("x", "w_qkv", "w_o", "w_fc1", "w_fc2", "norm1_w", "norm2_b", "b_qkv", "b_fc2"):
        base = f64[name]
        for _ in range(3):
            idx = tuple(rng.integers(0, n) for n in base.shape)
            eps = 1e-6
            plus, minus = dict(f64), dict(f64)
            plus[name], minus[name] = base.copy(), base.copy()
            plus[name][idx] += eps
            minus[name][idx] -= eps
            fd = (loss(plus) - loss(minus)) / (2 * eps)
            an = G[name].reshape(base.shape)[idx]
            assert abs(fd - an) <= 1e-5 * max(1.0, abs(an)), (name, idx, fd, an)
