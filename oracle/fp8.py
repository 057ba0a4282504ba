"""Float64 oracle of the FP8 (E4M3) forward path -- TEST INFRASTRUCTURE ONLY.

Sources: the FP8 recipe of "ai阅读megatron" (performance flags: --fp8-hybrid, recipe hybrid or
delayed_scaling) and of "快速入门" §8.2 (hybrid format: E4M3 in the forward pass, E5M2 in the
backward; dynamic scaling that tracks each tensor's amax over a history, amax_compute_algo max),
and the E4M3 format of "FP8 Formats for Deep Learning" (the reading list of the tutorial's
Appendix A): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
S.1111.111 is NaN, largest finite 448, subnormals down to 2^-9.

Readings (where the pages are silent):
  * Per-tensor scaling: a tensor with amax A is multiplied by scale = 448 / A (fp32) before the
    cast to E4M3, and the product of the two operand dequantisation factors (1/scale) rescales the
    fp32 GEMM accumulator.  A zero amax keeps scale 1.
  * The cast rounds to nearest, ties to even, and saturates to +-448 (the hardware's satfinite).
  * x * scale is formed in fp32 before the cast, as the kernels do, so both sides round the same
    fp32 value (a quantised code is an integer decided by floating point).
  * Delayed scaling: a forward uses the scales of the amax history before it, then appends its own
    amax; the next scale is 448 / max(history).
  * Which tensors are FP8: the four GEMM inputs of each side -- normed x, the attention output,
    normed h and the MLP hidden (activations, delayed scaling), and the four projection weights
    (current scaling at quantisation time).  q/k/v, the attention itself, h and y stay bf16.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from . import layer as ol

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """E4M3 codes (uint8) -> float64 values (NaN for S.1111.111)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.power(2.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return s * mag


_POS_CODES = np.arange(0, 127, dtype=np.uint8)        # +0 ... +448, ascending
_POS_VALUES = e4m3_decode(_POS_CODES)


def e4m3_encode(x) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to the even code), saturating to +-448; NaN -> NaN code."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, len(_POS_VALUES) - 1)
    lo = np.clip(hi - 1, 0, None)
    d_lo, d_hi = a - _POS_VALUES[lo], _POS_VALUES[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    code = np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def scale_from_amax(amax) -> np.float32:
    """448 / amax in fp32 (1 when amax is 0)."""
    a = np.float32(amax)
    return np.float32(1.0) if a == 0 else np.float32(np.float32(E4M3_MAX) / a)


def quantize(x, scale) -> np.ndarray:
    """E4M3 codes of fp32(x * scale)."""
    prod = np.asarray(x, dtype=np.float32) * np.float32(scale)
    return e4m3_encode(prod.astype(np.float64))


def dequantize(codes, scale) -> np.ndarray:
    return e4m3_decode(codes) / float(np.float32(scale))


def quantize_weight(w_bits) -> Dict[str, np.ndarray]:
    """Current per-tensor scaling of a bf16 weight: {'codes', 'scale'} with scale = 448 / amax."""
    w = ol.bf16_to_f64(w_bits)
    scale = scale_from_amax(np.max(np.abs(w)))
    return {"codes": quantize(w, scale), "scale": scale}


def _qdq(x, scale):
    return dequantize(quantize(x, scale), scale)


ACT_NAMES = ("xn", "o", "hn", "a")


WEIGHT_NAMES = ("w_qkv", "w_o", "w_fc1", "w_fc2")


def quantize_weights(inp: Dict) -> Dict[str, Dict[str, np.ndarray]]:
    return {k: quantize_weight(inp[k]) for k in WEIGHT_NAMES}


def layer_forward_fp8(cfg, inp: Dict, act_scales, rows: Optional[np.ndarray] = None,
                      wq: Optional[Dict] = None) -> Dict[str, np.ndarray]:
    """Whole layer at TP=1 with the four GEMMs on E4M3 operands.

    act_scales: fp32 scales of (xn, o, hn, a).  Weights use quantize_weight (or the precomputed
    `wq` of quantize_weights(inp)).  Returns y and h for `rows` (all tokens if None) and the amax
    of each activation over those rows.
    """
    T, B, d = cfg.tokens, cfg.batch, cfg.head_dim
    nh, ng = cfg.heads, cfg.groups
    rows = np.arange(T) if rows is None else np.asarray(rows)
    s_xn, s_o, s_hn, s_a = (np.float32(s) for s in act_scales)
    wq = quantize_weights(inp) if wq is None else wq
    W = {k: dequantize(v["codes"], v["scale"]) for k, v in wq.items()}
    x = ol._tokens(inp["x"], cfg)
    b = {k: ol._w(inp, k) for k in ("b_qkv", "b_o", "b_fc1", "b_fc2")}

    xn = ol.apply_norm(cfg, x, ol._w(inp, "norm1_w"), ol._w(inp, "norm1_b"))
    xq = _qdq(xn, s_xn)
    qw, kw = nh * d, ng * d
    bq = None if b["b_qkv"] is None else b["b_qkv"][:qw]
    bk = None if b["b_qkv"] is None else b["b_qkv"][qw:qw + kw]
    bv = None if b["b_qkv"] is None else b["b_qkv"][qw + kw:]
    q = ol.linear(xq[rows], W["w_qkv"][:qw], bq).reshape(len(rows), nh, d)
    k = ol.linear(xq, W["w_qkv"][qw:qw + kw], bk).reshape(T, ng, d)
    v = ol.linear(xq, W["w_qkv"][qw + kw:], bv).reshape(T, ng, d)
    if cfg.rope_base > 0:
        cq, sq = ol.rope_cos_sin(rows // B, d, cfg.rope_base)
        ck, sk = ol.rope_cos_sin(np.arange(T) // B, d, cfg.rope_base)
        q, k = ol.rope(q, cq, sq), ol.rope(k, ck, sk)
    o = np.empty((len(rows), nh, d))
    for bb in range(B):
        sel = np.nonzero(rows % B == bb)[0]
        if len(sel):
            o[sel] = ol.causal_attention(q[sel], k[bb::B], v[bb::B], rows[sel] // B)
    o = o.reshape(len(rows), qw)
    h = x[rows] + ol.linear(_qdq(o, s_o), W["w_o"], b["b_o"])
    hn = ol.apply_norm(cfg, h, ol._w(inp, "norm2_w"), ol._w(inp, "norm2_b"))
    u = ol.linear(_qdq(hn, s_hn), W["w_fc1"], b["b_fc1"])
    a = ol.activation(cfg, u)
    y = h + ol.linear(_qdq(a, s_a), W["w_fc2"], b["b_fc2"])
    amax = {"xn": np.max(np.abs(xn[rows])), "o": np.max(np.abs(o)), "hn": np.max(np.abs(hn)), "a": np.max(np.abs(a))}
    return {"y": y, "h": h, "amax": amax}
