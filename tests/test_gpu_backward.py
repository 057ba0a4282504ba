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


# Shapes whose dX GEMMs take the layer handle's K-split tail with an MN-major A operand (dX^T = W^T
# dY^T reads W MN-major): fc1's dX (M = hidden 512, N = the tokens, K = fc1's output width) is a
# single partial wave cut into 4 ranges of K (tests/test_abi.py pins the plans); the second layer's
# K = 2056 leaves a ragged last K block, with batch 2 and 2064 tokens.  (The weight gradients run
# on a stream of their own and cut their tails along N.)
KSPLIT_CFGS = [
    synth.LayerConfig("bw_ksplit", batch=1, seq=2048, hidden=512, heads=8, groups=2, head_dim=64, ffn=1024,
                      rope_base=1e4, bias=True),
    synth.LayerConfig("bw_ksplit_ragged", batch=2, seq=1032, hidden=512, heads=4, groups=1, head_dim=128,
                      ffn=2056, norm="layer", act="gelu_tanh", rope_base=0.0, bias=True),
]

CFGS = [
    synth.CONFIGS["tiny"],
    synth.LayerConfig("bw_gqa", batch=2, seq=128, hidden=256, heads=8, groups=2, head_dim=64, ffn=512,
                      rope_base=1e4),
    synth.LayerConfig("bw_ln", batch=2, seq=64, hidden=256, heads=2, groups=2, head_dim=128, ffn=384,
                      norm="layer", act="gelu_tanh", rope_base=0.0, bias=True),
    synth.LayerConfig("bw_mqa", batch=1, seq=200, hidden=512, heads=4, groups=1, head_dim=128, ffn=1024,
                      rope_base=5e5, bias=True),
    # a sequence shorter than one 64-query block (the backward takes seq % 8 == 0), three samples
    synth.LayerConfig("bw_short", batch=3, seq=24, hidden=256, heads=2, groups=2, head_dim=128, ffn=512,
                      rope_base=1e4),
    # three query heads per kv group (an odd count) and a ragged last 128-key block
    synth.LayerConfig("bw_rep3", batch=1, seq=136, hidden=384, heads=6, groups=2, head_dim=64, ffn=768,
                      rope_base=1e4, bias=True),
]


@pytest.mark.parametrize("cfg", CFGS + KSPLIT_CFGS + [synth.CONFIGS["llama8b"]], ids=lambda c: c.name)
def test_backward_matches_oracle(cfg):
    """Every element of dx and of the twelve weight gradients; the Llama-3-8B-shaped layer at its
    full size (4096 tokens) is the benchmarked backward, whose dW GEMMs for the output projection
    and QKV take K-split tails."""
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
    got = {"x": to_f64(dx)}
    got.update({k: (None if t is None else to_f64(t)) for k, t in grads.items()})
    dl.close()
    del x, dy, dx, grads
    torch.cuda.empty_cache()
    want = ob.layer_backward(cfg, inp, ol.bf16_to_f64(dy_bits))
    assert_grad_close(got["x"], want["x"], "dx")
    for name, t in got.items():
        if name == "x":
            continue
        if t is None:
            assert want[name] is None, name
            continue
        assert_grad_close(t, want[name], name)


def test_backward_rejects_unsupported():
    cfg = synth.CONFIGS["tiny"]
    layer = ml.Layer.from_config(cfg, tp_rank=0, tp_size=2)
    z = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ml.MtError) as e:
        ml.mt_layer_backward(layer.handle, z.data_ptr(), z.data_ptr(), 128, 1, ml.MtWeights(), z.data_ptr(),
                             ml.MtGrads(), None)
    assert e.value.code == ml.MT_ERR_UNSUPPORTED
    layer.close()


@pytest.mark.parametrize("cfg", [CFGS[1], CFGS[2], CFGS[5], KSPLIT_CFGS[1]], ids=lambda c: c.name)
def test_forward_train_and_backward_saved_match_forward_and_backward(cfg):
    """mt_layer_forward_train gives mt_layer_forward's y bit for bit, and mt_layer_backward_saved
    after it gives mt_layer_backward's dx and weight-matrix gradients bit for bit (the same kernels on
    the same intermediates); the norm-weight and bias gradients, whose column sums add per-CTA
    partial rows atomically in no fixed order, agree within the gradient tolerance."""
    inp = synth.make_inputs(cfg, seed=83, affine="random", biases="random")
    T, H = cfg.tokens, cfg.hidden
    dy = to_dev(synth.f32_to_bf16_bits(np.random.default_rng(84).standard_normal((T, H)).astype(np.float32)))
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(T, H)

    def run(saved):
        y, dx = torch.empty_like(x), torch.empty_like(x)
        grads = {k: (None if v is None else torch.empty_like(v)) for k, v in dl.tens.items()}
        if saved:
            dl.layer.forward_train(x, cfg.seq, cfg.batch, dl.w, y)
            dl.layer.backward_saved(x, dy, cfg.seq, cfg.batch, dl.w, dx, grads)
        else:
            dl.layer.forward(x, cfg.seq, cfg.batch, dl.w, y)
            dl.layer.backward(x, dy, cfg.seq, cfg.batch, dl.w, dx, grads)
        torch.cuda.synchronize()
        dl.layer.status()
        return y, dx, grads

    y0, dx0, g0 = run(False)
    y1, dx1, g1 = run(True)
    dl.close()
    assert torch.equal(y0, y1), "forward_train's y differs from forward's"
    assert torch.equal(dx0, dx1), "dx differs"
    for name, t in g0.items():
        if t is None:
            assert g1[name] is None
        elif name.startswith("w_"):
            assert torch.equal(t, g1[name]), name
        else:
            assert_grad_close(to_f64(g1[name]), to_f64(t), name)
