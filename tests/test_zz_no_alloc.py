"""The allocation-free entry point (mt_layer_forward_static) against the float64 oracle and the
handle-based forward.

Some callers cannot call cudaMalloc (code inside a host framework whose allocator owns all device
memory, real-time or embedded callers that forbid device allocation after start-up); the static
variant keeps its scratch in a fixed area inside the library instead of a caller-lent workspace.
After its first call on a device (which looks up the area's address and loads its kernels), a
call must leave the device's free memory unchanged.  This file is collected last so that a
failure here comes after every other test has run; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import layer as ol
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
    synth.LayerConfig("gqa_d128_rope", batch=1, seq=200, hidden=512, heads=8, groups=2, head_dim=128, ffn=1024,
                      rope_base=5e5, bias=True),
], ids=lambda c: c.name)
def test_static_forward_matches_oracle_and_handle_on_two_calls(cfg):
    torch.cuda.set_device(0)
    inp = synth.make_inputs(cfg, seed=31, affine="random", biases="random")
    dl = DeviceLayer(cfg, inp)
    assert dl.layer.workspace(cfg.seq, cfg.batch).numel() <= STATIC_BYTES - 1024
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    handle_y = to_f64(dl.forward(x))
    oracle_y = ol.layer_forward(cfg, inp)["y"]
    ys = [torch.full((cfg.tokens, cfg.hidden), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    _static_forward(cfg, dl, x, ys[0])  # first call: address lookup and kernel loading
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for y in ys[1:]:
        _static_forward(cfg, dl, x, y)
        ml.mt_layer_forward_static_status(torch.cuda.current_stream().cuda_stream)  # no timeout recorded
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "a static call changed the device's free memory"
    for y in ys:
        got = to_f64(y)
        assert_layer_close(got, oracle_y, f"static forward vs oracle ({cfg.name})")
        assert_layer_close(got, handle_y, f"static forward vs handle forward ({cfg.name})")
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


def test_static_forward_replays_from_a_cuda_graph():
    """After its first call a static call is stream-ordered device work only (no allocation, no
    host copy or synchronisation), so it can be captured in a CUDA graph under the global capture
    mode, which rejects any of those; the replay equals an eager static call bit for bit."""
    torch.cuda.set_device(0)
    cfg = synth.LayerConfig("static_graph", batch=1, seq=256, hidden=512, heads=8, groups=2, head_dim=128, ffn=1024,
                            rope_base=5e5, bias=True)
    inp = synth.make_inputs(cfg, seed=33, affine="random", biases="random")
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    want = torch.full((cfg.tokens, cfg.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
    _static_forward(cfg, dl, x, want)  # eager: the first call on the device happens outside the capture
    torch.cuda.synchronize()
    y = torch.full_like(want, float("nan"))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side, capture_error_mode="global"):
            _static_forward(cfg, dl, x, y)
    torch.cuda.current_stream().wait_stream(side)
    y.fill_(float("nan"))
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    ml.mt_layer_forward_static_status(torch.cuda.current_stream().cuda_stream)
    assert torch.equal(want, y)
    assert_layer_close(to_f64(y), ol.layer_forward(cfg, inp)["y"], "static forward replayed from a graph vs oracle")
    dl.close()
