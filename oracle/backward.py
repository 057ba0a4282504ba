"""Float64 oracle of the layer's backward pass at TP=1 -- TEST INFRASTRUCTURE ONLY.

The pages' subject is training (the forward-backward step of "ai阅读megatron", training loop;
activation recompute, "快速入门" §8): given dL/dy of the layer output, this computes dL/dx and the
gradient of every weight by the chain rule through the forward of oracle.layer (same readings:
pre-norm order, rotate-half RoPE, causal GQA softmax with scale 1/sqrt(d), SwiGLU with the gate
first or GeLU(tanh), biases added once).  Pinned by PyTorch autograd on the independent
restatement and by finite differences (tests/test_oracle_backward.py).
"""
from __future__ import annotations

from typing import Dict

import numpy as np

from . import layer as ol


def _norm_fwd(cfg, x, g, b):
    """Norm with the pieces its backward needs: xhat, 1/sigma."""
    if cfg.norm == "rms":
        r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + cfg.eps)
        xhat = x * r
        return xhat * g, xhat, r
    mu = np.mean(x, axis=-1, keepdims=True)
    r = 1.0 / np.sqrt(np.mean((x - mu) ** 2, axis=-1, keepdims=True) + cfg.eps)
    xhat = (x - mu) * r
    return xhat * g + b, xhat, r


def _norm_bwd(cfg, dy, xhat, r, g):
    """d/dx of y = xhat * g (+ b): with gx = dy * g,
    RMS:  dx = r (gx - xhat mean(gx xhat));  LN: dx = r (gx - mean(gx) - xhat mean(gx xhat))."""
    gx = dy * g
    dx = gx - xhat * np.mean(gx * xhat, axis=-1, keepdims=True)
    if cfg.norm != "rms":
        dx = dx - np.mean(gx, axis=-1, keepdims=True)
    return r * dx, np.sum(dy * xhat, axis=0), (np.sum(dy, axis=0) if cfg.norm != "rms" else None)


def _rope_bwd(dxh, cos, sin):
    """Transpose of the rotate-half rotation: rotate by the opposite angle."""
    return ol.rope(dxh, cos, -sin)


def _silu_grad(g):
    s = 1.0 / (1.0 + np.exp(-g))
    return s * (1.0 + g * (1.0 - s))


def _gelu_tanh_grad(u):
    k0, k1 = np.sqrt(2.0 / np.pi), 0.044715
    t = np.tanh(k0 * (u + k1 * u ** 3))
    return 0.5 * (1.0 + t) + 0.5 * u * (1.0 - t * t) * k0 * (1.0 + 3.0 * k1 * u * u)


def layer_backward(cfg, inp: Dict, dy: np.ndarray) -> Dict[str, np.ndarray]:
    """Gradients of sum(y * dy) for the TP=1 layer; dy is [T, H] (float64).  Returns dx and one
    entry per weight of the inputs (None where the weight is absent)."""
    T, B, S, H, d = cfg.tokens, cfg.batch, cfg.seq, cfg.hidden, cfg.head_dim
    nh, ng = cfg.heads, cfg.groups
    rep = nh // ng
    W = {k: ol._w(inp, k) for k in inp if k != "x"}
    x = ol._tokens(inp["x"], cfg)

    # ---- forward, keeping what the backward needs
    xn, xhat1, r1 = _norm_fwd(cfg, x, W["norm1_w"], W.get("norm1_b"))
    qkv = ol.linear(xn, W["w_qkv"], W.get("b_qkv"))
    q = qkv[:, :nh * d].reshape(T, nh, d)
    k = qkv[:, nh * d:(nh + ng) * d].reshape(T, ng, d)
    v = qkv[:, (nh + ng) * d:].reshape(T, ng, d)
    if cfg.rope_base > 0:
        cs, sn = ol.rope_cos_sin(np.arange(T) // B, d, cfg.rope_base)
        q, k = ol.rope(q, cs, sn), ol.rope(k, cs, sn)
    scale = 1.0 / np.sqrt(d)

    def probs(b, h):
        """Causal softmax of one head's scores (formed again where the backward needs them, so that
        no more than one [S, S] matrix is held at a time)."""
        return ol.causal_softmax((q[b::B, h] @ k[b::B, h // rep].T) * scale, np.arange(S))

    o = np.empty((T, nh, d))
    for b in range(B):
        for h in range(nh):
            o[b::B, h] = probs(b, h) @ v[b::B, h // rep]
    o2 = o.reshape(T, nh * d)
    h_ = x + ol.linear(o2, W["w_o"], W.get("b_o"))
    hn, xhat2, r2 = _norm_fwd(cfg, h_, W["norm2_w"], W.get("norm2_b"))
    u = ol.linear(hn, W["w_fc1"], W.get("b_fc1"))
    a = ol.activation(cfg, u)

    # ---- backward
    G: Dict[str, np.ndarray] = {}
    G["b_fc2"] = np.sum(dy, axis=0) if W.get("b_fc2") is not None else None
    G["w_fc2"] = dy.T @ a
    da = dy @ W["w_fc2"]
    if cfg.act == "swiglu":
        f = cfg.ffn
        gate, up = u[:, :f], u[:, f:]
        du = np.concatenate([da * up * _silu_grad(gate), da * ol.silu(gate)], axis=1)
    else:
        du = da * _gelu_tanh_grad(u)
    G["b_fc1"] = np.sum(du, axis=0) if W.get("b_fc1") is not None else None
    G["w_fc1"] = du.T @ hn
    dhn = du @ W["w_fc1"]
    dh_norm, G["norm2_w"], G["norm2_b"] = _norm_bwd(cfg, dhn, xhat2, r2, W["norm2_w"])
    dh = dy + dh_norm
    G["b_o"] = np.sum(dh, axis=0) if W.get("b_o") is not None else None
    G["w_o"] = dh.T @ o2
    do = (dh @ W["w_o"]).reshape(T, nh, d)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(nh):
            g = h // rep
            p = probs(b, h)
            dob = do[b::B, h]
            dv[b::B, g] += p.T @ dob
            dp = dob @ v[b::B, g].T
            ds = p * (dp - np.sum(dp * p, axis=1, keepdims=True)) * scale
            dq[b::B, h] += ds @ k[b::B, g]
            dk[b::B, g] += ds.T @ q[b::B, h]
    if cfg.rope_base > 0:
        dq, dk = _rope_bwd(dq, cs, sn), _rope_bwd(dk, cs, sn)
    dqkv = np.concatenate([dq.reshape(T, -1), dk.reshape(T, -1), dv.reshape(T, -1)], axis=1)
    G["b_qkv"] = np.sum(dqkv, axis=0) if W.get("b_qkv") is not None else None
    G["w_qkv"] = dqkv.T @ xn
    dxn = dqkv @ W["w_qkv"]
    dx_norm, G["norm1_w"], G["norm1_b"] = _norm_bwd(cfg, dxn, xhat1, r1, W["norm1_w"])
    G["x"] = dh + dx_norm
    return G
