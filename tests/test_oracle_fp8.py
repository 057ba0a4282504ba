"""Pins for the E4M3 oracle: the format's definition checked against PyTorch's float8_e4m3fn, the
rounding rules on hand-picked ties, saturation, and the FP8 layer against the bf16 layer."""
import numpy as np
import pytest
import torch

import synth
from oracle import fp8 as of
from oracle import layer as ol
from tests import fp8_check as fc


def test_decode_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = of.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok]) and np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))
    assert of.e4m3_decode(0x7E) == 448.0 and of.e4m3_decode(0x01) == 2.0 ** -9 and of.e4m3_decode(0x08) == 2.0 ** -6


def test_encode_inverts_decode_on_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(of.e4m3_encode(of.e4m3_decode(codes)), codes)


def test_encode_matches_torch_round_to_nearest_even_inside_range():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.normal(0, 1, 4000), rng.normal(0, 100, 4000), rng.normal(0, 1e-2, 4000),
                        rng.uniform(-463, 463, 4000), rng.uniform(-2 ** -6, 2 ** -6, 4000)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(of.e4m3_encode(x.astype(np.float64)), want)


def test_ties_go_to_the_even_code_and_large_values_saturate():
    assert of.e4m3_encode(1.0625) == 0x38          # halfway 1.0 (0x38) / 1.125 (0x39)
    assert of.e4m3_encode(1.1875) == 0x3A          # halfway 1.125 (0x39) / 1.25 (0x3A)
    assert of.e4m3_encode(2.0 ** -10) == 0x00      # halfway 0 / smallest subnormal
    assert of.e4m3_encode(3 * 2.0 ** -10) == 0x02  # halfway 2^-9 (0x01) / 2^-8 (0x02)
    assert of.e4m3_encode(1e4) == 0x7E and of.e4m3_encode(-1e4) == 0xFE and of.e4m3_encode(460.0) == 0x7E
    assert of.e4m3_encode(np.nan) == 0x7F


def test_weight_quantisation_maps_amax_to_448():
    rng = np.random.default_rng(8)
    w = synth.f32_to_bf16_bits(rng.normal(0, 0.02, (64, 48)).astype(np.float32))
    q = of.quantize_weight(w)
    wf = ol.bf16_to_f64(w)
    i = np.unravel_index(np.argmax(np.abs(wf)), wf.shape)
    assert q["scale"] == np.float32(448.0) / np.float32(np.max(np.abs(wf)))
    assert (q["codes"][i] & 0x7F) == 0x7E
    rel = np.abs(of.dequantize(q["codes"], q["scale"]) - wf) / np.maximum(np.abs(wf), 2 ** -6 / q["scale"])
    assert rel.max() <= 2.0 ** -4 + 1e-12          # half an ulp of a 3-bit mantissa


def _cfg(**kw):
    base = dict(name="f8", batch=2, seq=24, hidden=64, heads=4, groups=2, head_dim=16, ffn=96, norm="rms",
                act="swiglu", rope_base=1e4, bias=True)
    base.update(kw)
    return synth.LayerConfig(**base)


def test_fp8_layer_without_quantisation_is_the_bf16_layer(monkeypatch):
    """With the casts replaced by the identity the FP8 layer is the bf16 layer: it composes the same steps."""
    cfg = _cfg()
    inp = synth.make_inputs(cfg, seed=9, affine="random", biases="random")
    monkeypatch.setattr(of, "_qdq", lambda x, s: x)
    monkeypatch.setattr(of, "quantize_weight", lambda w: {"codes": w, "scale": np.float32(1)})
    monkeypatch.setattr(of, "dequantize", lambda c, s: ol.bf16_to_f64(c))
    np.testing.assert_allclose(of.layer_forward_fp8(cfg, inp, (1, 1, 1, 1))["y"], ol.layer_forward(cfg, inp)["y"],
                               rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("cfg", [_cfg(), _cfg(norm="layer", act="gelu_tanh", rope_base=0.0, groups=4)],
                         ids=["rms_swiglu", "ln_gelu"])
def test_fp8_layer_stays_within_fp8_error_of_the_bf16_layer(cfg):
    inp = synth.make_inputs(cfg, seed=10, affine="random", biases="random")
    ref = ol.layer_forward(cfg, inp)
    # scales from the bf16 layer's own activations (amax -> 448)
    o1 = of.layer_forward_fp8(cfg, inp, (1, 1, 1, 1))
    scales = [of.scale_from_amax(o1["amax"][n]) for n in of.ACT_NAMES]
    y = of.layer_forward_fp8(cfg, inp, scales)["y"]
    dev = np.abs(y - ref["y"]) / np.max(np.abs(ref["y"]))
    assert 1e-4 < dev.max() < 0.05     # quantised (so it differs), but only by FP8 rounding


def test_each_gemm_input_is_quantised(monkeypatch):
    cfg = _cfg()
    inp = synth.make_inputs(cfg, seed=11, affine="random")
    scales = (30.0, 300.0, 40.0, 500.0)
    base = of.layer_forward_fp8(cfg, inp, scales)["y"]
    # changing one activation's scale changes the result: that input does go through E4M3
    for i in range(4):
        s = list(scales)
        s[i] = s[i] * 1.37
        assert np.max(np.abs(of.layer_forward_fp8(cfg, inp, s)["y"] - base)) > 1e-6


# --------------------------------------------------------------------------- storage rounding
def test_round_bf16_and_fp16_match_torch_conversions():
    rng = np.random.default_rng(12)
    x = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-3, 5000), rng.normal(0, 300, 5000)])
    # values exactly halfway between two bf16 numbers (ties go to the even mantissa)
    base = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(rng.normal(0, 1, 2000).astype(np.float32)))
    ties = (base.astype(np.float32).view(np.uint32) + np.uint32(0x8000)).view(np.float32).astype(np.float64)
    x = np.concatenate([x, ties])
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(of.round_bf16(x), want)
    want16 = torch.from_numpy(x.astype(np.float32)).to(torch.float16).to(torch.float64).numpy()
    assert np.array_equal(of.round_fp16(x), want16)


# --------------------------------------------------------------------------- the FP8 stage checks can fail
F8_SHAPES = [
    synth.CONFIGS["tiny"],
    synth.LayerConfig("f8gqa", batch=2, seq=192, hidden=512, heads=8, groups=2, head_dim=64, ffn=1024, rope_base=1e4),
    synth.LayerConfig("f8ln", batch=1, seq=200, hidden=512, heads=4, groups=4, head_dim=128, ffn=1024, norm="layer",
                      act="gelu_tanh", rope_base=0.0, bias=True),
]


def _stage_inputs(cfg):
    inp = synth.make_inputs(cfg, seed=61, affine="random", biases="random")
    amax = of.layer_forward_fp8(cfg, inp, (1, 1, 1, 1))["amax"]
    return inp, [float(of.scale_from_amax(amax[n])) for n in of.ACT_NAMES], of.quantize_weights(inp)


def _skipping(name):
    return lambda n, x, s: x if n == name else of._qdq(x, s)


@pytest.mark.parametrize("cfg", F8_SHAPES, ids=lambda c: c.name)
def test_attention_stage_check_passes_other_rounding_and_rejects_a_skipped_cast(cfg, monkeypatch):
    """A correct FP8 attention block that keeps q, k, v unrounded passes the stage bound; the same
    block with xn or o left unquantised (planted here, in the oracle) fails it."""
    inp, sc, wq = _stage_inputs(cfg)
    ref = of.attention_block_fp8(cfg, inp, sc, wq=wq, storage_rounding=True)["h"]
    exact = ol.layer_forward(cfg, inp)["h"]
    plain = of.attention_block_fp8(cfg, inp, sc, wq=wq)["h"]
    assert fc.assert_attention_stage(of.round_bf16(plain), ref, exact, "unrounded q/k/v") > 0.05
    for name in ("xn", "o"):
        with monkeypatch.context() as m:
            m.setattr(of, "_cast", _skipping(name))
            bad = of.attention_block_fp8(cfg, inp, sc, wq=wq, storage_rounding=True)["h"]
        with pytest.raises(AssertionError, match="attention stage"):
            fc.assert_attention_stage(of.round_bf16(bad), ref, exact, f"{name} left unquantised")


@pytest.mark.parametrize("cfg", F8_SHAPES, ids=lambda c: c.name)
def test_mlp_stage_check_passes_fp32_gemms_and_rejects_a_skipped_cast(cfg, monkeypatch):
    """From a given h: the FP8 MLP block with float32 GEMMs passes the stage bound; with hn or a left
    unquantised it fails."""
    inp, sc, wq = _stage_inputs(cfg)
    h = of.round_bf16(of.attention_block_fp8(cfg, inp, sc, wq=wq, storage_rounding=True)["h"])
    y_fp8 = of.mlp_block_fp8(cfg, inp, sc, h, wq=wq)["y"]
    b_fc2 = ol._w(inp, "b_fc2")
    y_exact = h + ol.mlp_partial(cfg, 1, h, inp) + (0.0 if b_fc2 is None else b_fc2)

    def linear32(x, w, b=None):
        y = np.asarray(x, np.float32) @ np.asarray(w, np.float32).T
        return (y if b is None else y + np.asarray(b, np.float32)).astype(np.float64)

    with monkeypatch.context() as m:
        m.setattr(ol, "linear", linear32)
        y32 = of.mlp_block_fp8(cfg, inp, sc, h, wq=wq)["y"]
    fc.assert_mlp_stage(of.round_bf16(y32), y_fp8, y_exact, "float32 GEMMs")
    for name in ("hn", "a"):
        with monkeypatch.context() as m:
            m.setattr(of, "_cast", _skipping(name))
            bad = of.mlp_block_fp8(cfg, inp, sc, h, wq=wq)["y"]
        with pytest.raises(AssertionError, match="MLP stage"):
            fc.assert_mlp_stage(of.round_bf16(bad), y_fp8, y_exact, f"{name} left unquantised")


def test_code_check_counts_signed_steps():
    want = np.array([0x00, 0x80, 0x01, 0x81, 0x38, 0xB8], dtype=np.uint8)
    fc.assert_codes_close(np.array([0x80, 0x00, 0x00, 0x80, 0x39, 0xB9], dtype=np.uint8), want, 1.0, "neighbours")
    with pytest.raises(AssertionError):      # +min subnormal against -min subnormal: two steps apart
        fc.assert_codes_close(np.array([0x81], dtype=np.uint8), np.array([0x01], dtype=np.uint8), 1.0, "sign")
    with pytest.raises(AssertionError):      # more codes differ than allowed
        fc.assert_codes_close(want ^ np.uint8(1), want, 0.5, "fraction")
