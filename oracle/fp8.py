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
  * A quantised code is an integer decided by floating point, so where a comparison needs the
    codes of the attention output or of normed h to be decided from the same values as the
    kernels decide them, the oracle takes the kernels' storage precision for the intermediates
    they store between launches: q and k in bf16, v in fp16 (after RoPE), h in bf16
    (storage_rounding=True).  Everything else stays float64.
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


def round_bf16(x) -> np.ndarray:
    """float64 -> the value a kernel stores: fp32 (nearest even), then bfloat16 (nearest even)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return (u.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_fp16(x) -> np.ndarray:
    """float64 -> fp32 -> IEEE half (nearest even), as a kernel stores v for the P V product."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float16).astype(np.float64)


def _cast(name: str, x, scale):
    """The E4M3 cast of activation `name` (one of ACT_NAMES) as the next GEMM sees it."""
    return _qdq(x, scale)


def attention_block_fp8(cfg, inp: Dict, act_scales, rows: Optional[np.ndarray] = None, wq: Optional[Dict] = None,
                        storage_rounding: bool = False) -> Dict[str, np.ndarray]:
    """Attention half of the FP8 layer at TP=1: xn = Norm1(x) cast to E4M3, QKV, RoPE, causal GQA
    attention, its output o cast to E4M3, the output projection, h = x + Y_attn + b_o (float64).

    storage_rounding: q and k are rounded to bf16 and v to fp16 after RoPE, as the kernels store
    them between launches; the E4M3 code of o is then decided from the same stored operands as the
    kernel decides it.  Returns xn, o and h for `rows` (all tokens if None), and v (all tokens)."""
    T, B, d = cfg.tokens, cfg.batch, cfg.head_dim
    nh, ng = cfg.heads, cfg.groups
    rows = np.arange(T) if rows is None else np.asarray(rows)
    s_xn, s_o = np.float32(act_scales[0]), np.float32(act_scales[1])
    wq = quantize_weights(inp) if wq is None else wq
    w_qkv = dequantize(wq["w_qkv"]["codes"], wq["w_qkv"]["scale"])
    w_o = dequantize(wq["w_o"]["codes"], wq["w_o"]["scale"])
    x = ol._tokens(inp["x"], cfg)
    b_qkv, b_o = ol._w(inp, "b_qkv"), ol._w(inp, "b_o")
    xn = ol.apply_norm(cfg, x, ol._w(inp, "norm1_w"), ol._w(inp, "norm1_b"))
    xq = _cast("xn", xn, s_xn)
    qw, kw = nh * d, ng * d
    bq = None if b_qkv is None else b_qkv[:qw]
    bk = None if b_qkv is None else b_qkv[qw:qw + kw]
    bv = None if b_qkv is None else b_qkv[qw + kw:]
    q = ol.linear(xq[rows], w_qkv[:qw], bq).reshape(len(rows), nh, d)
    k = ol.linear(xq, w_qkv[qw:qw + kw], bk).reshape(T, ng, d)
    v = ol.linear(xq, w_qkv[qw + kw:], bv).reshape(T, ng, d)
    if cfg.rope_base > 0:
        cq, sq = ol.rope_cos_sin(rows // B, d, cfg.rope_base)
        ck, sk = ol.rope_cos_sin(np.arange(T) // B, d, cfg.rope_base)
        q, k = ol.rope(q, cq, sq), ol.rope(k, ck, sk)
    if storage_rounding:
        q, k, v = round_bf16(q), round_bf16(k), round_fp16(v)
    o = np.empty((len(rows), nh, d))
    for bb in range(B):
        sel = np.nonzero(rows % B == bb)[0]
        if len(sel):
            o[sel] = ol.causal_attention(q[sel], k[bb::B], v[bb::B], rows[sel] // B)
    o = o.reshape(len(rows), qw)
    h = x[rows] + ol.linear(_cast("o", o, s_o), w_o, b_o)
    return {"xn": xn[rows], "o": o, "h": h, "v": v}


def mlp_block_fp8(cfg, inp: Dict, act_scales, h: np.ndarray, wq: Optional[Dict] = None) -> Dict[str, np.ndarray]:
    """MLP half of the FP8 layer at TP=1 from h [n, H]: hn = Norm2(h) cast to E4M3, fc1, SwiGLU /
    GeLU, the hidden a cast to E4M3, fc2; y = h + Y_mlp + b_fc2 (float64)."""
    s_hn, s_a = np.float32(act_scales[2]), np.float32(act_scales[3])
    wq = quantize_weights(inp) if wq is None else wq
    w_fc1 = dequantize(wq["w_fc1"]["codes"], wq["w_fc1"]["scale"])
    w_fc2 = dequantize(wq["w_fc2"]["codes"], wq["w_fc2"]["scale"])
    hn = ol.apply_norm(cfg, h, ol._w(inp, "norm2_w"), ol._w(inp, "norm2_b"))
    u = ol.linear(_cast("hn", hn, s_hn), w_fc1, ol._w(inp, "b_fc1"))
    a = ol.activation(cfg, u)
    y = h + ol.linear(_cast("a", a, s_a), w_fc2, ol._w(inp, "b_fc2"))
    return {"hn": hn, "a": a, "y": y}


def layer_forward_fp8(cfg, inp: Dict, act_scales, rows: Optional[np.ndarray] = None,
                      wq: Optional[Dict] = None, storage_rounding: bool = False) -> Dict[str, np.ndarray]:
    """Whole layer at TP=1 with the four GEMMs on E4M3 operands.

    act_scales: fp32 scales of (xn, o, hn, a).  Weights use quantize_weight (or the precomputed
    `wq` of quantize_weights(inp)).  storage_rounding: the stored intermediates q, k (bf16), v (fp16)
    and h (bf16) are rounded as the kernels store them (see attention_block_fp8).  Returns y and h
    for `rows` (all tokens if None) and the amax of each activation over those rows.
    """
    wq = quantize_weights(inp) if wq is None else wq
    att = attention_block_fp8(cfg, inp, act_scales, rows=rows, wq=wq, storage_rounding=storage_rounding)
    h = round_bf16(att["h"]) if storage_rounding else att["h"]
    mlp = mlp_block_fp8(cfg, inp, act_scales, h, wq=wq)
    amax = {"xn": np.max(np.abs(att["xn"])), "o": np.max(np.abs(att["o"])), "hn": np.max(np.abs(mlp["hn"])),
            "a": np.max(np.abs(mlp["a"]))}
    return {"y": mlp["y"], "h": h, "amax": amax}
