"""An independent PyTorch-CPU (float64) restatement of the layer forward, used only to pin the oracle.

Written separately from the NumPy oracle and built from library routines where
they exist: F.rms_norm / F.layer_norm, F.scaled_dot_product_attention with a
causal mask, F.silu / F.gelu(approximate="tanh"), and RoPE as a multiplication
of complex numbers z_i = x_i + j*x_{i+d/2} by exp(j*p*theta_i).
The layer order is the one of "快速入门" §3.1: input_layernorm -> SelfAttention
(linear_qkv, core_attention, linear_proj) -> bias-dropout-add -> pre_mlp_layernorm
-> MLP(linear_fc1, linear_fc2) -> bias-dropout-add.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F


def _t(bits):
    if bits is None:
        return None
    u = torch.from_numpy(np.asarray(bits, dtype=np.uint16).astype(np.int32) << 16)
    return u.view(torch.float32).to(torch.float64)


def _norm(cfg, x, g, b):
    if cfg.norm == "rms":
        return F.rms_norm(x, (x.shape[-1],), weight=g, eps=cfg.eps)
    return F.layer_norm(x, (x.shape[-1],), weight=g, bias=b, eps=cfg.eps)


def _rope_complex(x, positions, base):
    """x [S, B, heads, d]; rotates pairs (i, i+d/2) by angle p*base^(-2i/d) via complex multiply."""
    d = x.shape[-1]
    half = d // 2
    inv = base ** (-torch.arange(0, half, dtype=torch.float64) * 2.0 / d)
    ang = positions.to(torch.float64)[:, None] * inv[None, :]            # [S, half]
    rot = torch.polar(torch.ones_like(ang), ang)[:, None, None, :]        # [S, 1, 1, half]
    z = torch.complex(x[..., :half], x[..., half:]) * rot
    return torch.cat([z.real, z.imag], dim=-1)


def as_tensors(inp):
    """float64 torch tensors of the bf16 inputs (None stays None)."""
    return {k: _t(v) for k, v in inp.items()}


def layer_forward(cfg, inp, tensors=None):
    """TP=1 layer output y [S*B, H] (float64 torch tensor).  `tensors`: as_tensors(inp), possibly
    requiring gradients, used instead of decoding `inp`."""
    S, B, H, d = cfg.seq, cfg.batch, cfg.hidden, cfg.head_dim
    nh, ng = cfg.heads, cfg.groups
    t = as_tensors(inp) if tensors is None else tensors
    x = t["x"].reshape(S, B, H)
    w = {k: v for k, v in t.items() if k != "x"}

    xn = _norm(cfg, x, w["norm1_w"], w.get("norm1_b"))
    qkv = F.linear(xn, w["w_qkv"], w.get("b_qkv"))
    q = qkv[..., : nh * d].reshape(S, B, nh, d)
    k = qkv[..., nh * d:(nh + ng) * d].reshape(S, B, ng, d)
    v = qkv[..., (nh + ng) * d:].reshape(S, B, ng, d)
    if cfg.rope_base > 0:
        pos = torch.arange(S)
        q, k = _rope_complex(q, pos, cfg.rope_base), _rope_complex(k, pos, cfg.rope_base)
    # SDPA wants [B, heads, S, d]; GQA by repeating each group for its nh/ng heads.
    qb = q.permute(1, 2, 0, 3)
    kb = k.permute(1, 2, 0, 3).repeat_interleave(nh // ng, dim=1)
    vb = v.permute(1, 2, 0, 3).repeat_interleave(nh // ng, dim=1)
    o = F.scaled_dot_product_attention(qb, kb, vb, is_causal=True)      # scale 1/sqrt(d)
    o = o.permute(2, 0, 1, 3).reshape(S, B, nh * d)
    attn = F.linear(o, w["w_o"])
    h = x + attn + (w["b_o"] if w.get("b_o") is not None else 0.0)
    hn = _norm(cfg, h, w["norm2_w"], w.get("norm2_b"))
    u = F.linear(hn, w["w_fc1"], w.get("b_fc1"))
    if cfg.act == "swiglu":
        a = F.silu(u[..., : cfg.ffn]) * u[..., cfg.ffn:]
    else:
        a = F.gelu(u, approximate="tanh")
    y = h + F.linear(a, w["w_fc2"]) + (w["b_fc2"] if w.get("b_fc2") is not None else 0.0)
    return y.reshape(S * B, H)
