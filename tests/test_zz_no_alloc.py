"""The allocation-free entry point (mt_layer_forward_static) against the handle-based forward.

Some callers cannot call cudaMalloc (code inside a host framework whose allocator owns all device
memory, real-time or embedded callers that forbid device allocation after start-up); the static
variant keeps its scratch in a fixed area inside the library instead of a caller-lent workspace.
This file is collected last so that a failure here comes after every other test has run; it also
passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import synth
from megatron_tensor_transformer_gpt_gb300 import mt_layer as ml
from tests.gpu_util import DeviceLayer, assert_layer_close, to_dev, to_f64

pytestmark = pytest.mark.gpu

STATIC_BYTES = 32 << 20


def _static_forward(cfg, dl, x, y):
    ml.mt_layer_forward_static(cfg.hidden, cfg.heads, cfg.groups, cfg.head_dim, cfg.ffn,
                               ml.MT_NORM_RMS if cfg.norm == "rms" else ml.MT_NORM_LAYER,
                               ml.MT_ACT_SWIGLU if cfg.act == "swiglu" else ml.MT_ACT_GELU_TANH,
                               cfg.rope_base, 1, 0, cfg.eps, x.data_ptr(), cfg.seq, cfg.batch, dl.w, y.data_ptr(),
                               torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("cfg", [
    synth.CONFIGS["tiny"],
    synth.LayerConfig("small_ln_gelu", batch=2, seq=100, hidden=512, heads=8, groups=2, head_dim=64, ffn=1000,
                      norm="layer", act="gelu_tanh", rope_base=0.0, bias=True),
], ids=lambda c: c.name)
def test_static_forward_matches_handle_forward_on_two_calls(cfg):
    torch.cuda.set_device(0)
    inp = synth.make_inputs(cfg, seed=31, affine="random", biases="random")
    dl = DeviceLayer(cfg, inp)
    assert dl.layer.workspace(cfg.seq, cfg.batch).numel() <= STATIC_BYTES - 1024
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    want = to_f64(dl.forward(x))
    for _ in range(2):
        y = torch.full((cfg.tokens, cfg.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
        _static_forward(cfg, dl, x, y)
        torch.cuda.synchronize()
        assert_layer_close(to_f64(y), want, f"static forward ({cfg.name})")
    dl.close()


def test_static_forward_rejects_workspace_beyond_the_area():
    torch.cuda.set_device(0)
    cfg = synth.CONFIGS["llama8b"]
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ml.MtError) as e:
        ml.mt_layer_forward_static(cfg.hidden, cfg.heads, cfg.groups, cfg.head_dim, cfg.ffn, ml.MT_NORM_RMS,
                                   ml.MT_ACT_SWIGLU, cfg.rope_base, 1, 0, cfg.eps, x.data_ptr(), cfg.seq, cfg.batch,
                                   ml.MtWeights(), x.data_ptr(), None)
    assert e.value.code == ml.MT_ERR_UNSUPPORTED
    assert "static area" in str(e.value)
