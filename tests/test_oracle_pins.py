"""Pins for the float64 CPU oracle: brute force, closed forms, invariants and library cross-checks.

None of these retypes the oracle's formulas: each compares it with something
else that the pages or the mathematics fix.  Runs on CPU only.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import layer as ol
import synth
from tests import torch_restatement

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def small_cfg(**kw):
    base = dict(name="small", batch=2, seq=24, hidden=64, heads=8, groups=8, head_dim=16,
                ffn=96, norm="rms", act="swiglu", rope_base=1e4, bias=False)
    base.update(kw)
    return synth.LayerConfig(**base)


# --------------------------------------------------------------------------- bf16 decoding
def test_bf16_decode_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3E80, 0x0001, 0x7F7F, 0x0000, 0x8000], dtype=np.uint16)
    want = [1.0, -2.0, 0.25, 2.0 ** -133, 3.3895313892515355e38, 0.0, -0.0]
    got = ol.bf16_to_f64(bits)
    assert got.tolist() == want


# --------------------------------------------------------------------------- norms
@pytest.mark.parametrize("c", [0.5, -3.0, 1e-3])
def test_rms_norm_constant_vector_closed_form(c):
    H, eps = 32, 1e-5
    g = rng.normal(1.0, 0.1, H)
    got = ol.rms_norm(np.full((1, H), c), g, eps)
    np.testing.assert_allclose(got[0], g * c / math.sqrt(c * c + eps), rtol=1e-14)


def test_layer_norm_constant_vector_gives_shift():
    H = 32
    g, b = rng.normal(1.0, 0.1, H), rng.normal(0.0, 0.1, H)
    got = ol.layer_norm(np.full((3, H), 7.25), g, b, 1e-5)
    np.testing.assert_allclose(got, np.broadcast_to(b, (3, H)), atol=1e-15)


def test_layer_norm_moments():
    x = rng.normal(2.0, 3.0, (5, 256))
    y = ol.layer_norm(x, np.ones(256), np.zeros(256), 1e-5)
    var = x.var(axis=1)
    np.testing.assert_allclose(y.mean(axis=1), 0.0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=1), var / (var + 1e-5), rtol=1e-12)


def test_norms_match_torch():
    x = rng.normal(size=(7, 48))
    g, b = rng.normal(1, 0.1, 48), rng.normal(0, 0.1, 48)
    tx, tg, tb = (torch.from_numpy(a) for a in (x, g, b))
    np.testing.assert_allclose(ol.rms_norm(x, g, 1e-5), F.rms_norm(tx, (48,), tg, 1e-5).numpy(), rtol=1e-12)
    np.testing.assert_allclose(ol.layer_norm(x, g, b, 1e-5), F.layer_norm(tx, (48,), tg, tb, 1e-5).numpy(),
                               rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------------------- linear
def test_linear_brute_force():
    x, w, b = rng.normal(size=(3, 5)), rng.normal(size=(4, 5)), rng.normal(size=4)
    want = np.array([[sum(x[i, k] * w[j, k] for k in range(5)) + b[j] for j in range(4)] for i in range(3)])
    np.testing.assert_allclose(ol.linear(x, w, b), want, rtol=1e-13)


# --------------------------------------------------------------------------- RoPE
def test_rope_pairing_and_sign_explicit():
    # d = 4: pairs (0,2) and (1,3); theta_0 = 1, theta_1 = base^(-1/2).
    base, p = 100.0, 3
    c, s = ol.rope_cos_sin(np.array([p]), 4, base)
    x = np.array([[[1.0, 0.0, 0.0, 0.0]]])
    np.testing.assert_allclose(ol.rope(x, c, s)[0, 0], [math.cos(3), 0, math.sin(3), 0], atol=1e-15)
    x = np.array([[[0.0, 1.0, 0.0, 0.0]]])
    a = p * base ** -0.5
    np.testing.assert_allclose(ol.rope(x, c, s)[0, 0], [0, math.cos(a), 0, math.sin(a)], atol=1e-15)


def test_rope_preserves_norm_and_position_zero_is_identity():
    d, n = 128, 50
    x = rng.normal(size=(n, 3, d))
    pos = rng.integers(0, 40000, n)
    c, s = ol.rope_cos_sin(pos, d, 5e5)
    y = ol.rope(x, c, s)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    c0, s0 = ol.rope_cos_sin(np.zeros(n, dtype=int), d, 5e5)
    np.testing.assert_array_equal(ol.rope(x, c0, s0), x)


def test_rope_relative_position_property():
    # <R_p q, R_m k> depends only on p - m (RoFormer): shift both positions by the same amount.
    d = 64
    q, k = rng.normal(size=(1, 1, d)), rng.normal(size=(1, 1, d))
    dots = []
    for shift in (0, 7, 1000):
        cq, sq = ol.rope_cos_sin(np.array([15 + shift]), d, 1e4)
        ck, sk = ol.rope_cos_sin(np.array([4 + shift]), d, 1e4)
        dots.append(float(np.sum(ol.rope(q, cq, sq) * ol.rope(k, ck, sk))))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-10)


def test_rope_matches_complex_rotation():
    d, n = 64, 9
    x = rng.normal(size=(n, 2, d))
    pos = np.arange(n) * 37
    c, s = ol.rope_cos_sin(pos, d, 1e4)
    z = x[..., : d // 2] + 1j * x[..., d // 2:]
    theta = 1e4 ** (-np.arange(d // 2) * 2.0 / d)
    z = z * np.exp(1j * pos[:, None, None] * theta[None, None, :])
    np.testing.assert_allclose(ol.rope(x, c, s), np.concatenate([z.real, z.imag], -1), rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- attention
def brute_force_attention(q, k, v):
    """Explicit loops over i, j: every score, every exponential, every weighted sum."""
    n, nh, d = q.shape
    ng = k.shape[1]
    out = np.zeros_like(q)
    for h in range(nh):
        g = h * ng // nh
        for i in range(n):
            sc = [sum(q[i, h, t] * k[j, g, t] for t in range(d)) / math.sqrt(d) for j in range(i + 1)]
            mx = max(sc)
            e = [math.exp(si - mx) for si in sc]
            z = sum(e)
            for t in range(d):
                out[i, h, t] = sum(e[j] * v[j, g, t] for j in range(i + 1)) / z
    return out


@pytest.mark.parametrize("nh,ng", [(2, 2), (4, 2), (4, 1)])
def test_attention_brute_force(nh, ng):
    S, d = 9, 8
    q, k, v = rng.normal(size=(S, nh, d)), rng.normal(size=(S, ng, d)), rng.normal(size=(S, ng, d))
    np.testing.assert_allclose(ol.causal_attention(q, k, v, np.arange(S)), brute_force_attention(q, k, v),
                               rtol=1e-12, atol=1e-13)


def test_softmax_rows_sum_to_one_and_mask():
    n, S = 20, 20
    p = ol.causal_softmax(rng.normal(size=(n, S)) * 5, np.arange(n))
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(p[np.triu_indices(n, 1)] == 0.0)
    assert np.all(p[np.tril_indices(n)] > 0.0)


def test_attention_single_token_returns_v():
    d = 16
    q, k, v = rng.normal(size=(1, 4, d)), rng.normal(size=(1, 2, d)), rng.normal(size=(1, 2, d))
    o = ol.causal_attention(q, k, v, np.array([0]))
    np.testing.assert_array_equal(o, np.repeat(v, 2, axis=1))


def test_gqa_equals_mha_with_repeated_kv():
    S, nh, ng, d = 17, 8, 2, 16
    q, k, v = rng.normal(size=(S, nh, d)), rng.normal(size=(S, ng, d)), rng.normal(size=(S, ng, d))
    a = ol.causal_attention(q, k, v, np.arange(S))
    b = ol.causal_attention(q, np.repeat(k, nh // ng, 1), np.repeat(v, nh // ng, 1), np.arange(S))
    np.testing.assert_allclose(a, b, rtol=1e-13)


def test_attention_is_causal_and_rows_independent():
    S, nh, d = 30, 2, 8
    q, k, v = rng.normal(size=(S, nh, d)), rng.normal(size=(S, nh, d)), rng.normal(size=(S, nh, d))
    full = ol.causal_attention(q, k, v, np.arange(S), row_chunk=7)
    k2, v2 = k.copy(), v.copy()
    k2[20:], v2[20:] = 99.0, -99.0                       # future keys must not matter for rows < 20
    part = ol.causal_attention(q, k2, v2, np.arange(S))
    np.testing.assert_allclose(part[:20], full[:20], rtol=1e-13)
    rows = np.array([3, 11, 29])
    np.testing.assert_allclose(ol.causal_attention(q[rows], k, v, rows), full[rows], rtol=1e-13)


def test_attention_matches_torch_sdpa():
    S, nh, d = 64, 4, 32
    q, k, v = rng.normal(size=(S, nh, d)), rng.normal(size=(S, nh, d)), rng.normal(size=(S, nh, d))
    want = F.scaled_dot_product_attention(*(torch.from_numpy(a).transpose(0, 1) for a in (q, k, v)),
                                          is_causal=True).transpose(0, 1).numpy()
    np.testing.assert_allclose(ol.causal_attention(q, k, v, np.arange(S)), want, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------------------- activations
def test_activations_special_values_and_torch():
    u = np.linspace(-12, 12, 241)
    assert ol.silu(np.array([0.0]))[0] == 0.0 and ol.gelu_tanh(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(ol.silu(u), F.silu(torch.from_numpy(u)).numpy(), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(ol.gelu_tanh(u), F.gelu(torch.from_numpy(u), approximate="tanh").numpy(),
                               rtol=1e-12, atol=1e-15)
    # far from zero both are the identity for u >> 0 and vanish for u << 0
    assert abs(ol.silu(np.array([40.0]))[0] - 40.0) < 1e-12 and abs(ol.gelu_tanh(np.array([-40.0]))[0]) < 1e-12


def test_swiglu_gate_is_first_half():
    cfg = small_cfg(ffn=3)
    u = np.array([[1.0, -2.0, 0.5, 10.0, 20.0, 30.0]])
    want = np.array([[10.0 / (1 + math.exp(-1.0)), 20.0 * -2.0 / (1 + math.exp(2.0)), 30.0 * 0.5 / (1 + math.exp(-0.5))]])
    np.testing.assert_allclose(ol.activation(cfg, u), want, rtol=1e-14)


# --------------------------------------------------------------------------- weight layout (golden)
def test_weight_slices_follow_name_mapping():
    g = json.load(open(os.path.join(GOLDEN, "weight_slices.json")))
    cfg = synth.CONFIGS["tiny"]
    assert cfg.hidden == g["hidden"] and cfg.ffn == g["intermediate"]
    r = synth.shard_row_ranges(cfg, 1, 0)
    assert [list(t) for t in r["qkv_rows"]] == g["qkv_rows"]
    assert [list(t) for t in r["fc1_rows"]] == g["fc1_rows"]


# --------------------------------------------------------------------------- tensor-parallel invariants
@pytest.mark.parametrize("tp", [2, 4, 8])
def test_column_split_concatenation_reproduces_tp1(tp):
    cfg = small_cfg()
    inp = synth.make_inputs(cfg, seed=5, affine="random")
    xn = ol.rms_norm(ol._tokens(inp["x"], cfg), ol.bf16_to_f64(inp["norm1_w"]), cfg.eps)
    full_qkv = ol.linear(xn, ol.bf16_to_f64(inp["w_qkv"]))
    full_fc1 = ol.linear(xn, ol.bf16_to_f64(inp["w_fc1"]))
    d, nh, ng, f = cfg.head_dim, cfg.heads, cfg.groups, cfg.ffn
    qs, ks, vs, gs, us = [], [], [], [], []
    for r in range(tp):
        sh = synth.shard_weights(cfg, inp, tp, r)
        y = ol.linear(xn, ol.bf16_to_f64(sh["w_qkv"]))
        qw, kw = nh // tp * d, ng // tp * d
        qs.append(y[:, :qw]); ks.append(y[:, qw:qw + kw]); vs.append(y[:, qw + kw:])
        u = ol.linear(xn, ol.bf16_to_f64(sh["w_fc1"]))
        gs.append(u[:, : f // tp]); us.append(u[:, f // tp:])
    # equal up to fp64 reassociation (BLAS blocks a narrower product differently)
    np.testing.assert_allclose(np.concatenate(qs + ks + vs, 1), full_qkv, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(np.concatenate(gs + us, 1), full_fc1, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("tp", [2, 4, 8])
def test_row_split_sum_of_partials_reproduces_tp1(tp):
    cfg = small_cfg(bias=True)
    inp = synth.make_inputs(cfg, seed=6, affine="random", biases="random")
    x = ol._tokens(inp["x"], cfg)
    shards = [synth.shard_weights(cfg, inp, tp, r) for r in range(tp)]
    ya = sum(ol.attn_partial(cfg, tp, x, shards[r]) for r in range(tp))
    np.testing.assert_allclose(ya, ol.attn_partial(cfg, 1, x, inp), rtol=1e-11, atol=1e-13)
    h = x + 0.5
    ym = sum(ol.mlp_partial(cfg, tp, h, shards[r]) for r in range(tp))
    np.testing.assert_allclose(ym, ol.mlp_partial(cfg, 1, h, inp), rtol=1e-11, atol=1e-13)
    full = ol.layer_forward(cfg, inp)["y"]
    np.testing.assert_allclose(ol.layer_forward_tp_sum(cfg, tp, inp["x"], shards)["y"], full, rtol=1e-11, atol=1e-12)


def test_rank_identity_at_tp1_is_the_layer_without_its_mlp_residual_and_bias():
    """At tp = 1 the identity-mode rank is the whole layer: its h is the layer's h (b_o added once)
    and its y_partial is y - h - b_fc2 (the fc2 partial carries neither the residual nor the bias)."""
    cfg = small_cfg(groups=2, bias=True, norm="layer", act="gelu_tanh")
    inp = synth.make_inputs(cfg, seed=7, affine="random", biases="random")
    out = ol.layer_forward_rank_identity(cfg, 1, inp["x"], inp)
    full = ol.layer_forward(cfg, inp)
    np.testing.assert_allclose(out["h"], full["h"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(out["y_partial"], full["y"] - full["h"] - ol.bf16_to_f64(inp["b_fc2"]),
                               rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("tp", [2, 4])
def test_rank_identity_h_carries_b_o_once_per_rank(tp):
    """Each identity-mode rank forms h_r = x + Y_attn,r + b_o, so over the ranks
    sum_r (h_r - x - b_o) is the row-parallel sum sum_r Y_attn,r = h - x - b_o of the unsharded
    layer.  A rank that dropped b_o or added it twice breaks this by b_o per rank."""
    cfg = small_cfg(groups=4, bias=True)
    inp = synth.make_inputs(cfg, seed=17, affine="random", biases="random")
    x = ol._tokens(inp["x"], cfg)
    b_o = ol.bf16_to_f64(inp["b_o"])
    acc = sum(ol.layer_forward_rank_identity(cfg, tp, inp["x"], synth.shard_weights(cfg, inp, tp, r))["h"] - x - b_o
              for r in range(tp))
    np.testing.assert_allclose(acc, ol.layer_forward(cfg, inp)["h"] - x - b_o, rtol=1e-10, atol=1e-12)
    assert np.max(np.abs(b_o)) > 1e-3   # the check above is sensitive to b_o


@pytest.mark.parametrize("tp", [2, 4])
def test_rank_identity_y_partials_sum_when_every_rank_sees_the_same_h(tp):
    """With W_o = 0 every rank's h_r is x + b_o, the unsharded layer's h; the ranks' y_partial then
    sum to the row-parallel MLP output y - h - b_fc2 of the unsharded layer."""
    cfg = small_cfg(groups=4, bias=True, norm="layer")
    inp = dict(synth.make_inputs(cfg, seed=18, affine="random", biases="random"))
    inp["w_o"] = np.zeros_like(inp["w_o"])
    full = ol.layer_forward(cfg, inp)
    parts = [ol.layer_forward_rank_identity(cfg, tp, inp["x"], synth.shard_weights(cfg, inp, tp, r))
             for r in range(tp)]
    for p in parts:
        np.testing.assert_allclose(p["h"], full["h"], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sum(p["y_partial"] for p in parts), full["y"] - full["h"] - ol.bf16_to_f64(inp["b_fc2"]),
                               rtol=1e-10, atol=1e-12)


def test_row_sampling_matches_full_layer():
    cfg = small_cfg(batch=3, seq=20)
    inp = synth.make_inputs(cfg, seed=8, affine="random")
    full = ol.layer_forward(cfg, inp)["y"]
    rows = np.array([0, 1, 2, 17, 31, 59])
    np.testing.assert_allclose(ol.layer_forward(cfg, inp, rows=rows)["y"], full[rows], rtol=1e-12)


# --------------------------------------------------------------------------- whole layer vs independent restatement
@pytest.mark.parametrize("cfg", [
    synth.CONFIGS["tiny"],
    small_cfg(),
    small_cfg(groups=2, batch=3, seq=40),
    synth.CONFIGS["gpt345m"].replace(batch=2, seq=48, hidden=128, heads=4, groups=4, ffn=256),
    small_cfg(groups=1, norm="layer", act="gelu_tanh", rope_base=0.0, bias=True),
], ids=lambda c: c.name + f"-g{c.groups}-b{c.batch}")
def test_layer_matches_torch_restatement(cfg):
    inp = synth.make_inputs(cfg, seed=11, affine="random", biases="random")
    got = ol.layer_forward(cfg, inp)["y"]
    want = torch_restatement.layer_forward(cfg, inp).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-10)


# --------------------------------------------------------------------------- planted mistakes are caught
def _restatement_mismatch(cfg, inp):
    got = ol.layer_forward(cfg, inp)["y"]
    want = torch_restatement.layer_forward(cfg, inp).numpy()
    return np.max(np.abs(got - want))


@pytest.mark.parametrize("mutation", ["rope_sign", "mask_off_by_one", "swiglu_swap", "rms_no_eps_sqrt"])
def test_planted_oracle_mistakes_are_caught(monkeypatch, mutation):
    cfg = small_cfg(groups=2)
    inp = synth.make_inputs(cfg, seed=12, affine="random")
    assert _restatement_mismatch(cfg, inp) < 1e-10
    if mutation == "rope_sign":
        good = ol.rope_cos_sin
        monkeypatch.setattr(ol, "rope_cos_sin", lambda p, d, b: (lambda c, s: (c, -s))(*good(p, d, b)))
    elif mutation == "mask_off_by_one":
        good = ol.causal_softmax
        monkeypatch.setattr(ol, "causal_softmax", lambda s, p: good(s, np.maximum(np.asarray(p) - 1, 0)))
    elif mutation == "swiglu_swap":
        monkeypatch.setattr(ol, "activation", lambda c, u: ol.silu(u[:, u.shape[1] // 2:]) * u[:, : u.shape[1] // 2])
    elif mutation == "rms_no_eps_sqrt":
        monkeypatch.setattr(ol, "rms_norm", lambda x, g, eps: x / (np.sqrt(np.mean(x * x, -1, keepdims=True)) + eps) * g * 1.01)
    assert _restatement_mismatch(cfg, inp) > 1e-4


# --------------------------------------------------------------------------- packed samples
@pytest.mark.parametrize("lens", [[24], [5, 19], [1, 7, 3, 13], [9, 0, 15]])
def test_packed_layer_equals_each_sample_alone(lens):
    """A packed sample must compute exactly what the dense layer computes on it alone."""
    T = sum(lens)
    cfg = small_cfg(batch=1, seq=T, groups=2)
    inp = synth.make_inputs(cfg, seed=13, affine="random")
    cu = np.concatenate([[0], np.cumsum(lens)])
    packed = ol.layer_forward(cfg, inp, cu_seqlens=cu)["y"]
    x = inp["x"].reshape(T, cfg.hidden)
    for i, n in enumerate(lens):
        if n == 0:
            continue
        ci = cfg.replace(seq=n)
        alone = dict(inp, x=x[cu[i]:cu[i + 1]].reshape(n, 1, cfg.hidden))
        np.testing.assert_allclose(packed[cu[i]:cu[i + 1]], ol.layer_forward(ci, alone)["y"], rtol=1e-12, atol=1e-12)


def test_packed_segments_of_boundaries():
    seg, pos = ol.packed_segments([0, 3, 3, 5], 5)
    assert seg.tolist() == [0, 0, 0, 2, 2] and pos.tolist() == [0, 1, 2, 0, 1]
