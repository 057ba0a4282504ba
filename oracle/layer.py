"""Float64 oracle of one GPT/Llama Transformer layer forward, as one tensor-parallel rank computes it.

TEST INFRASTRUCTURE ONLY (tests, smoke check, bench CPU baseline).  Never on the product path.

Sources (page title, section):
  [CSDN]  "Megatron-LM 深度学习与源码分析文档", Part 2 §2 Tensor Parallel:
          Y = XW; column split W=[W_1..W_p], Y_i = X W_i, Y=[Y_1..Y_p];
          row split W=[W_1;..;W_p], X=[X_1..X_p], Y_i = X_i W_i, Y = sum_i Y_i;
          QKV as a column-parallel linear, heads per rank = heads/TP;
          MLP Z = phi(X W_1), Y = Z W_2 with fc1 column- and fc2 row-parallel.
  [PAI]   "快速入门 / Pai-Megatron-Patch 项目深度学习总结文档", §3.1 (layer tree and layer
          spec: input_layernorm -> SelfAttention(linear_qkv, core_attention with a causal
          mask, linear_proj) -> bias-dropout-add -> pre_mlp_layernorm -> MLP(linear_fc1,
          linear_fc2) -> bias-dropout-add) and §5.1 (q/k/v rows and gate/up rows of the
          fused weights); §6.1 launch flags (dropout 0.0, no query-key layer scaling,
          rotary percent 1.0).
  [VLL]   "ai阅读megatron", TransformerConfig (num_query_groups for GQA, gated linear unit)
          and the model flag sets (--swiglu, --normalization RMSNorm, RoPE).

Readings where the pages are silent (each also listed in the design notes):
  * RMSNorm  y = x / sqrt(mean(x^2) + eps) * g;  LayerNorm y = (x - mu) / sqrt(var + eps) * g + b,
    biased variance.  eps inside the square root.
  * RoPE: rotate-half pairing (i, i + d/2), theta_i = base^(-2i/d), position = sequence index s,
    applied to q and k after the bias; v untouched.
  * Softmax scale 1/sqrt(d) (query-key layer scaling disabled); key j visible to query i iff j <= i.
  * GQA head h reads group floor(h / (heads/groups)).
  * SwiGLU: a = silu(u[:, :f]) * u[:, f:], gate first (fc1 rows [gate | up]); GeLU in its tanh form.
  * Dropout is the identity (forward, rate 0.0).
  * Row-parallel partials carry neither bias nor residual; both are added once after the sum.

Every function is pinned by the CPU tests (tests/test_oracle_pins.py):
brute force, closed forms, invariants, and library cross-checks.  Absolute values of the
whole layer have no printed worked example on the pages; the layer is pinned by its parts
plus an independent PyTorch restatement (tests/torch_restatement.py).
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

__all__ = [
    "bf16_to_f64", "rms_norm", "layer_norm", "apply_norm", "linear", "rope_cos_sin", "rope",
    "causal_softmax", "causal_attention", "silu", "gelu_tanh", "activation",
    "attn_partial", "mlp_partial", "layer_forward", "layer_forward_rank_identity",
    "layer_forward_tp_sum", "split_heads", "packed_segments",
]


def bf16_to_f64(bits) -> Optional[np.ndarray]:
    """bfloat16 bit patterns (uint16) -> float64, exactly (bf16 is the top half of an IEEE float32)."""
    if bits is None:
        return None
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- norms
def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * g  (input_layernorm for LLaMA, [PAI] §3.1)."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def layer_norm(x: np.ndarray, g: np.ndarray, b: np.ndarray, eps: float) -> np.ndarray:
    """LayerNorm over the last axis with the biased variance: (x - mu)/sqrt(var + eps) * g + b."""
    mu = np.mean(x, axis=-1, keepdims=True)
    xc = x - mu
    var = np.mean(xc * xc, axis=-1, keepdims=True)
    return xc / np.sqrt(var + eps) * g + b


def apply_norm(cfg, x, g, b):
    if cfg.norm == "rms":
        return rms_norm(x, g, cfg.eps)
    return layer_norm(x, g, b, cfg.eps)


# --------------------------------------------------------------------------- linear
def linear(x: np.ndarray, w: np.ndarray, b: Optional[np.ndarray] = None) -> np.ndarray:
    """Y = X W with W stored as [out, in] (rows are output features), plus an optional bias ([CSDN] Y=XW)."""
    y = x @ w.T
    if b is not None:
        y = y + b
    return y


# --------------------------------------------------------------------------- rotary embedding
def rope_cos_sin(positions: np.ndarray, d: int, base: float):
    """cos/sin of the angles p * theta_i, theta_i = base^(-2i/d), i < d/2; [n, d/2] each."""
    i = np.arange(d // 2, dtype=np.float64)
    theta = np.power(float(base), -2.0 * i / d)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta[None, :]
    return np.cos(ang), np.sin(ang)


def rope(xh: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate-half RoPE on heads xh [n, heads, d]: pair (i, i+d/2) turns by the angle of row n, index i."""
    half = xh.shape[-1] // 2
    x1, x2 = xh[..., :half], xh[..., half:]
    c, s = cos[:, None, :], sin[:, None, :]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# --------------------------------------------------------------------------- attention
def causal_softmax(scores: np.ndarray, q_pos: np.ndarray) -> np.ndarray:
    """Row softmax of scores [n, S] over the keys j <= q_pos[row] (AttnMaskType.causal, [PAI] §3.1)."""
    S = scores.shape[1]
    visible = np.arange(S)[None, :] <= np.asarray(q_pos)[:, None]
    s = np.where(visible, scores, -np.inf)
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=1, keepdims=True)


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_pos: np.ndarray,
                     row_chunk: int = 1024) -> np.ndarray:
    """Causal GQA attention of one batch row.

    q [n, nh, d] (queries at sequence positions q_pos), k, v [S, ng, d] (keys at 0..S-1).
    o_h = softmax(q_h k_g^T / sqrt(d) + causal mask) v_g, g = floor(h / (nh/ng)).
    Query rows are taken `row_chunk` at a time only to bound memory; every row's
    softmax runs over all of its visible keys at once.
    """
    n, nh, d = q.shape
    ng = k.shape[1]
    rep = nh // ng
    o = np.empty((n, nh, d), dtype=np.float64)
    scale = 1.0 / np.sqrt(d)
    for r0 in range(0, n, row_chunk):
        r1 = min(n, r0 + row_chunk)
        pos = np.asarray(q_pos[r0:r1])
        smax = int(pos.max()) + 1
        for h in range(nh):
            g = h // rep
            scores = (q[r0:r1, h, :] @ k[:smax, g, :].T) * scale
            p = causal_softmax(scores, pos)
            o[r0:r1, h, :] = p @ v[:smax, g, :]
    return o


# --------------------------------------------------------------------------- activations
def silu(u):
    return u / (1.0 + np.exp(-u))


def gelu_tanh(u):
    return 0.5 * u * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (u + 0.044715 * u ** 3)))


def activation(cfg, u: np.ndarray) -> np.ndarray:
    """fc1 output -> MLP hidden: SwiGLU silu(gate) * up with gate = first half, or GeLU(tanh)."""
    if cfg.act == "swiglu":
        f = u.shape[1] // 2
        return silu(u[:, :f]) * u[:, f:]
    return gelu_tanh(u)


# --------------------------------------------------------------------------- layer pieces
def split_heads(cfg, tp: int):
    """(q heads, kv groups, ffn columns) held by one rank: heads/TP, groups/TP, ffn/TP ([CSDN] §2)."""
    return cfg.heads // tp, cfg.groups // tp, cfg.ffn // tp


def _tokens(x_bits_or_f64, cfg) -> np.ndarray:
    x = x_bits_or_f64
    if x.dtype == np.uint16:
        x = bf16_to_f64(x)
    return np.asarray(x, dtype=np.float64).reshape(cfg.seq * cfg.batch, cfg.hidden)


def _w(wd: Dict, name: str):
    a = wd.get(name)
    if a is None:
        return None
    return bf16_to_f64(a) if a.dtype == np.uint16 else np.asarray(a, dtype=np.float64)


def packed_segments(cu_seqlens, T: int):
    """Segment id and in-segment position of each of T packed tokens; sample i holds tokens
    [cu[i], cu[i+1]) ("快速入门" §4.1 / §8: cu_seqlens are the cumulative sample lengths)."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    assert cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0)
    seg = np.searchsorted(cu, np.arange(T), side="right") - 1
    return seg, np.arange(T) - cu[seg]


def attn_partial(cfg, tp: int, x: np.ndarray, wd: Dict, rows: Optional[np.ndarray] = None,
                 cu_seqlens=None) -> np.ndarray:
    """One rank's pre-reduce attention output Y_attn,i = o_i W_o,i^T for token rows `rows` (all if None).

    x: layer input, [T, H] float64 (token t = s*batch + b).  wd: that rank's weights.
    K and V are computed for every token (causality needs all earlier keys);
    queries, attention and the output projection only for the requested rows.
    cu_seqlens (batch 1 only): packed samples; a query sees only the earlier keys of its own
    sample, and RoPE positions restart at 0 in every sample (the reading that makes a packed
    sample compute what it would alone).
    """
    T, B, d = cfg.tokens, cfg.batch, cfg.head_dim
    hr, gr, _ = split_heads(cfg, tp)
    rows = np.arange(T) if rows is None else np.asarray(rows)
    if cu_seqlens is not None:
        assert B == 1
        seg, pos = packed_segments(cu_seqlens, T)
    else:
        seg, pos = np.zeros(T, dtype=np.int64), np.arange(T) // B
    xn = apply_norm(cfg, x, _w(wd, "norm1_w"), _w(wd, "norm1_b"))
    w_qkv, b_qkv = _w(wd, "w_qkv"), _w(wd, "b_qkv")
    qw, kw = hr * d, gr * d
    bq = None if b_qkv is None else b_qkv[:qw]
    bk = None if b_qkv is None else b_qkv[qw:qw + kw]
    bv = None if b_qkv is None else b_qkv[qw + kw:]
    q = linear(xn[rows], w_qkv[:qw], bq).reshape(len(rows), hr, d)
    k = linear(xn, w_qkv[qw:qw + kw], bk).reshape(T, gr, d)
    v = linear(xn, w_qkv[qw + kw:qw + 2 * kw], bv).reshape(T, gr, d)
    if cfg.rope_base > 0:
        cq, sq = rope_cos_sin(pos[rows], d, cfg.rope_base)
        ck, sk = rope_cos_sin(pos, d, cfg.rope_base)
        q, k = rope(q, cq, sq), rope(k, ck, sk)
    o = np.empty((len(rows), hr, d))
    if cu_seqlens is not None:
        cu = np.asarray(cu_seqlens)
        for i in range(len(cu) - 1):
            sel = np.nonzero(seg[rows] == i)[0]
            if len(sel) == 0:
                continue
            lo, hi = cu[i], cu[i + 1]                # keys of sample i, at positions 0..len-1
            o[sel] = causal_attention(q[sel], k[lo:hi], v[lo:hi], pos[rows[sel]])
    else:
        for b in range(B):
            sel = np.nonzero(rows % B == b)[0]
            if len(sel) == 0:
                continue
            kb, vb = k[b::B], v[b::B]                  # [S, gr, d] of batch row b
            o[sel] = causal_attention(q[sel], kb, vb, rows[sel] // B)
    return linear(o.reshape(len(rows), hr * d), _w(wd, "w_o"))


def mlp_partial(cfg, tp: int, h: np.ndarray, wd: Dict) -> np.ndarray:
    """One rank's pre-reduce MLP output Y_mlp,i = phi(norm2(h) W_fc1,i^T + b) W_fc2,i^T."""
    hn = apply_norm(cfg, h, _w(wd, "norm2_w"), _w(wd, "norm2_b"))
    u = linear(hn, _w(wd, "w_fc1"), _w(wd, "b_fc1"))
    return linear(activation(cfg, u), _w(wd, "w_fc2"))


def _add_bias(y, b):
    return y if b is None else y + b


def layer_forward(cfg, inp: Dict, rows: Optional[np.ndarray] = None, cu_seqlens=None) -> Dict[str, np.ndarray]:
    """Whole layer at TP=1: h = x + Y_attn + b_o; y = h + Y_mlp + b_fc2 (pre-norm order, bias-dropout-add).

    Returns {"h", "y"} for the token rows `rows` (all tokens if None); cu_seqlens: packed samples
    (see attn_partial)."""
    x = _tokens(inp["x"], cfg)
    rows = np.arange(cfg.tokens) if rows is None else np.asarray(rows)
    h = x[rows] + attn_partial(cfg, 1, x, inp, rows, cu_seqlens)
    h = _add_bias(h, _w(inp, "b_o"))
    y = _add_bias(h + mlp_partial(cfg, 1, h, inp), _w(inp, "b_fc2"))
    return {"h": h, "y": y}


def layer_forward_rank_identity(cfg, tp: int, x_bits, wd: Dict, rows=None) -> Dict[str, np.ndarray]:
    """One rank with the inter-block all-reduce replaced by the identity:
    h = x + Y_attn,i + b_o and y_partial = Y_mlp,i(h) (the rank-local timing path)."""
    x = _tokens(x_bits, cfg)
    rows = np.arange(cfg.tokens) if rows is None else np.asarray(rows)
    h = _add_bias(x[rows] + attn_partial(cfg, tp, x, wd, rows), _w(wd, "b_o"))
    return {"h": h, "y_partial": mlp_partial(cfg, tp, h, wd)}


def layer_forward_tp_sum(cfg, tp: int, x_bits, shards, rows=None) -> Dict[str, np.ndarray]:
    """The layer computed as `tp` ranks whose row-parallel partials are summed (the all-reduce):
    h = x + sum_i Y_attn,i + b_o; y = h + sum_i Y_mlp,i + b_fc2."""
    x = _tokens(x_bits, cfg)
    rows = np.arange(cfg.tokens) if rows is None else np.asarray(rows)
    ya = sum(attn_partial(cfg, tp, x, shards[r], rows) for r in range(tp))
    h = _add_bias(x[rows] + ya, _w(shards[0], "b_o"))
    ym = sum(mlp_partial(cfg, tp, h, shards[r]) for r in range(tp))
    return {"h": h, "y": _add_bias(h + ym, _w(shards[0], "b_fc2"))}
