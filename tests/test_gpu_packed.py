"""GPU parity of packed variable-length samples (mt_layer_forward_packed) against the float64 oracle.

cu_seqlens are the cumulative sample lengths; attention stays inside each sample and RoPE
positions restart per sample.  Checked element by element (small) and on sampled rows (a
Llama-3-8B-shaped layer with 4096 packed tokens), plus: each packed sample equals the dense
forward of that sample alone, and inconsistent cu_seqlens are reported without faulting.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import layer as ol
from megatron_tensor_transformer_gpt_gb300 import mt_layer as ml
from tests.gpu_util import DeviceLayer, assert_layer_close, sample_rows, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _cfg(lens, **kw):
    base = dict(name="packed", batch=1, seq=int(sum(lens)), hidden=512, heads=8, groups=2, head_dim=64, ffn=1000,
                norm="rms", act="swiglu", rope_base=1e4, bias=False)
    base.update(kw)
    return synth.LayerConfig(**base)


def _run_packed(cfg, inp, lens):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    y = torch.empty_like(x)
    dl.layer.forward_packed(x, torch.from_numpy(cu).cuda(), int(max(lens)), dl.w, y)
    torch.cuda.synchronize()
    dl.layer.status()
    return dl, cu, y


LENS = [
    [200],
    [100, 37, 129, 1, 256],          # lengths off the 8- and 128-token grids
    [50, 0, 70, 0],                   # empty samples
    [300, 300],
]


@pytest.mark.parametrize("lens", LENS, ids=lambda l: "-".join(map(str, l)))
@pytest.mark.parametrize("shape", ["gqa_d64", "mha_d128_ln_gelu", "gqa4_d128", "mha_d64"])
def test_packed_layer_matches_oracle(lens, shape):
    kw = {"gqa_d64": {}, "gqa4_d128": dict(heads=8, groups=2, head_dim=128), "mha_d64": dict(groups=8),
          "mha_d128_ln_gelu": dict(heads=4, groups=4, head_dim=128, norm="layer", act="gelu_tanh", bias=True)}[shape]
    cfg = _cfg(lens, **kw)
    inp = synth.make_inputs(cfg, seed=51, affine="random", biases="random")
    dl, cu, y = _run_packed(cfg, inp, lens)
    assert_layer_close(to_f64(y), ol.layer_forward(cfg, inp, cu_seqlens=cu)["y"], f"packed {lens}")
    dl.close()


def test_each_packed_sample_equals_its_dense_forward():
    lens = [129, 64, 200]
    cfg = _cfg(lens)
    inp = synth.make_inputs(cfg, seed=52, affine="random")
    dl, cu, y = _run_packed(cfg, inp, lens)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    for i, n in enumerate(lens):
        ci = cfg.replace(seq=n)
        di = DeviceLayer(ci, inp)
        yi = torch.empty(n, cfg.hidden, dtype=torch.bfloat16, device="cuda")
        di.layer.forward(x[cu[i]:cu[i + 1]].contiguous(), n, 1, di.w, yi)
        torch.cuda.synchronize()
        assert_layer_close(to_f64(y[cu[i]:cu[i + 1]]), to_f64(yi), f"sample {i} packed vs alone")
        di.close()
    dl.close()


def test_packed_llama8b_shape_sampled_rows():
    lens = [1000, 2048, 500, 548]
    cfg = synth.CONFIGS["llama8b"]
    inp = synth.make_inputs(cfg, seed=3)
    dl, cu, y = _run_packed(cfg, inp, lens)
    rows = np.unique(np.concatenate([sample_rows(cfg.tokens, seed=6, n_random=64), cu[:-1], cu[1:] - 1]))
    got = to_f64(y[torch.from_numpy(rows).cuda()])
    dl.close()
    assert_layer_close(got, ol.layer_forward(cfg, inp, rows=rows, cu_seqlens=cu)["y"], "packed llama8b")


def test_inconsistent_cu_seqlens_are_reported():
    lens = [64, 64, 64]
    cfg = _cfg(lens)
    inp = synth.make_inputs(cfg, seed=53)
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    y = torch.empty_like(x)
    bad = torch.tensor([0, 100, 40, 192], dtype=torch.int32, device="cuda")  # decreasing boundary
    dl.layer.forward_packed(x, bad, 100, dl.w, y)
    torch.cuda.synchronize()
    with pytest.raises(ml.MtError) as e:
        dl.layer.status()
    assert e.value.code == ml.MT_ERR_INVALID_ARG
    # the context stays usable and a consistent call is correct again
    good = torch.tensor([0, 64, 128, 192], dtype=torch.int32, device="cuda")
    dl.layer.forward_packed(x, good, 64, dl.w, y)
    torch.cuda.synchronize()
    dl.layer.status()
    assert_layer_close(to_f64(y), ol.layer_forward(cfg, inp, cu_seqlens=[0, 64, 128, 192])["y"], "after bad call")
    dl.close()
