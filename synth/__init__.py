"""Seeded synthetic inputs for one Transformer layer forward.

This module is shared by the CPU oracle tests, the GPU parity tests and the
bench.  It holds workload shapes, seeds, value distributions and the index
layout of tensor-parallel weight slices -- and none of the layer's arithmetic
(no norm, projection, rotation, softmax or activation lives here).

Values are drawn in float32 from NumPy's PCG64 generator, one independent
stream per tensor (seed, seed+1, ... in the order of ``WEIGHT_NAMES``), and
rounded once to bfloat16 (round to nearest, ties to even).  Both sides of a
parity check read the same bf16 bit patterns.

Shapes follow the Megatron pages: the Llama-3 8B / 70B flag sets ("ai阅读megatron",
model-configuration section: hidden 4096/8192, ffn 14336/28672, 32/64 heads,
8 query groups) and the GPT experiments of "Megatron-LM 深度学习与源码分析文档"
(Part 7).  Activations use the [seq, batch, hidden] layout the sequence-parallel
sketch of "ai阅读megatron" prints, flattened to rows t = s*batch + b.
"""
from __future__ import annotations

import dataclasses
from typing import Dict

import numpy as np

__all__ = [
    "LayerConfig", "CONFIGS", "WEIGHT_NAMES", "f32_to_bf16_bits", "bf16_bits_to_f32",
    "make_inputs", "shard_weights", "shard_row_ranges", "random_e4m3_codes",
]

NORM_RMS, NORM_LAYER = "rms", "layer"
ACT_SWIGLU, ACT_GELU_TANH = "swiglu", "gelu_tanh"


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """Shape of one layer and of the tensor-parallel split it runs under."""
    name: str
    batch: int
    seq: int
    hidden: int
    heads: int
    groups: int
    head_dim: int
    ffn: int
    norm: str = NORM_RMS
    act: str = ACT_SWIGLU
    rope_base: float = 0.0          # 0 => no rotary embedding
    bias: bool = False              # biases on every linear
    tp: int = 1                     # tensor-parallel size the workload is quoted at
    eps: float = 1e-5

    @property
    def tokens(self) -> int:
        return self.seq * self.batch

    @property
    def fc1_out(self) -> int:
        return 2 * self.ffn if self.act == ACT_SWIGLU else self.ffn

    def replace(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)

    def gemm_flops(self, tp: int = None) -> float:
        """2*M*N*K summed over the four projections of one rank."""
        tp = self.tp if tp is None else tp
        T, H, d = self.tokens, self.hidden, self.head_dim
        qw, kvw = self.heads // tp * d, self.groups // tp * d
        f = self.ffn // tp
        f1 = 2 * f if self.act == ACT_SWIGLU else f
        return 2.0 * T * H * (qw + 2 * kvw) + 2.0 * T * qw * H + 2.0 * T * H * f1 + 2.0 * T * f * H

    def attn_flops(self, tp: int = None) -> float:
        """Causal attention counted over the unmasked half: 4*d*S(S+1)/2 per head and batch row."""
        tp = self.tp if tp is None else tp
        S = self.seq
        return 4.0 * self.head_dim * S * (S + 1) / 2 * (self.heads // tp) * self.batch

    def flops(self, tp: int = None) -> float:
        return self.gemm_flops(tp) + self.attn_flops(tp)


CONFIGS: Dict[str, LayerConfig] = {
    # Tiny Llama-style layer: the oracle finishes it in well under a second.
    "tiny": LayerConfig("tiny", batch=1, seq=128, hidden=256, heads=4, groups=4, head_dim=64,
                        ffn=688, norm=NORM_RMS, act=ACT_SWIGLU, rope_base=1e4),
    # GPT-345M-shaped layer: LayerNorm, GeLU(tanh), biases, no RoPE, micro-batch 4.
    "gpt345m": LayerConfig("gpt345m", batch=4, seq=1024, hidden=1024, heads=16, groups=16,
                           head_dim=64, ffn=4096, norm=NORM_LAYER, act=ACT_GELU_TANH,
                           rope_base=0.0, bias=True),
    # Llama-3-8B-shaped layer.
    "llama8b": LayerConfig("llama8b", batch=1, seq=4096, hidden=4096, heads=32, groups=8,
                           head_dim=128, ffn=14336, rope_base=5e5),
    # Llama-3-70B-shaped layer; the workload is one tensor-parallel rank of eight.
    "llama70b_tp8": LayerConfig("llama70b_tp8", batch=1, seq=4096, hidden=8192, heads=64,
                                groups=8, head_dim=128, ffn=28672, rope_base=5e5, tp=8),
    # Llama-3-8B-shaped layer at a 32k context.
    "llama8b_32k": LayerConfig("llama8b_32k", batch=1, seq=32768, hidden=4096, heads=32,
                               groups=8, head_dim=128, ffn=14336, rope_base=5e5),
}

# Order fixes the per-tensor seed offsets (x takes the base seed).
WEIGHT_NAMES = ("norm1_w", "norm1_b", "w_qkv", "b_qkv", "w_o", "b_o",
                "norm2_w", "norm2_b", "w_fc1", "b_fc1", "w_fc2", "b_fc2")


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _draw(seed: int, shape, std: float, mean: float = 0.0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    if mean != 0.0:
        a += np.float32(mean)
    return f32_to_bf16_bits(a)


def weight_shapes(cfg: LayerConfig) -> Dict[str, tuple]:
    """Full (unsharded) weight shapes, rows = output features (the F.linear convention)."""
    H, d = cfg.hidden, cfg.head_dim
    qkv = (cfg.heads + 2 * cfg.groups) * d
    return {
        "norm1_w": (H,), "norm1_b": (H,),
        "w_qkv": (qkv, H), "b_qkv": (qkv,),
        "w_o": (H, cfg.heads * d), "b_o": (H,),
        "norm2_w": (H,), "norm2_b": (H,),
        "w_fc1": (cfg.fc1_out, H), "b_fc1": (cfg.fc1_out,),
        "w_fc2": (H, cfg.ffn), "b_fc2": (H,),
    }


def make_inputs(cfg: LayerConfig, seed: int = 0, weight_std: float = 0.02,
                affine: str = "standard", biases: str = "auto") -> Dict[str, np.ndarray]:
    """All inputs of one layer as bf16 bit patterns (uint16 arrays).

    x has shape [seq, batch, hidden] ~ N(0, 1); projection weights ~ N(0, weight_std).

    affine   "standard": norm gains 1, norm shifts 0 (the usual initialisation);
             "random":   gains ~ 1 + N(0, 0.1), shifts ~ N(0, 0.1) (pins the indexing).
    biases   "auto":   zero biases when cfg.bias, absent otherwise;
             "random": ~N(0, 0.02) when cfg.bias, absent otherwise;
             "none":   always absent.
    Absent tensors (RMSNorm shifts, biases of a bias-free layer) are None.
    """
    shapes = weight_shapes(cfg)
    out: Dict[str, np.ndarray] = {"x": _draw(seed, (cfg.seq, cfg.batch, cfg.hidden), 1.0)}
    for i, name in enumerate(WEIGHT_NAMES):
        s = seed + 1 + i
        shp = shapes[name]
        if name in ("norm1_w", "norm2_w"):
            out[name] = (_draw(s, shp, 0.1, 1.0) if affine == "random"
                         else f32_to_bf16_bits(np.ones(shp, np.float32)))
        elif name in ("norm1_b", "norm2_b"):
            if cfg.norm != NORM_LAYER:
                out[name] = None
            elif affine == "random":
                out[name] = _draw(s, shp, 0.1)
            else:
                out[name] = f32_to_bf16_bits(np.zeros(shp, np.float32))
        elif name.startswith("b_"):
            if not cfg.bias or biases == "none":
                out[name] = None
            elif biases == "random":
                out[name] = _draw(s, shp, 0.02)
            else:
                out[name] = f32_to_bf16_bits(np.zeros(shp, np.float32))
        else:
            out[name] = _draw(s, shp, weight_std)
    return out


def shard_row_ranges(cfg: LayerConfig, tp: int, rank: int) -> Dict[str, list]:
    """Index ranges [lo, hi) that make up tensor-parallel rank `rank`'s slice.

    Column-parallel weights (QKV, fc1) keep a slice of output rows; row-parallel
    weights (output projection, fc2) keep the matching input columns -- the
    W=[W_1..W_p] / W=[W_1;..;W_p] splits of "Megatron-LM 深度学习与源码分析文档",
    Part 2 §2 (Column/Row Parallel Linear).  QKV rows are the contiguous
    [q | k | v] blocks and fc1 rows the [gate | up] blocks of the HF->Megatron
    name mapping ("快速入门", §5.1).  Heads map to groups consecutively, so a
    rank's q heads use exactly its own k/v groups.
    """
    d, nh, ng, f = cfg.head_dim, cfg.heads, cfg.groups, cfg.ffn
    assert nh % tp == 0 and ng % tp == 0 and f % tp == 0
    hr, gr, fr = nh // tp, ng // tp, f // tp
    q0 = rank * hr * d
    k0 = nh * d + rank * gr * d
    v0 = nh * d + ng * d + rank * gr * d
    qkv_rows = [(q0, q0 + hr * d), (k0, k0 + gr * d), (v0, v0 + gr * d)]
    if cfg.act == ACT_SWIGLU:
        fc1_rows = [(rank * fr, (rank + 1) * fr), (f + rank * fr, f + (rank + 1) * fr)]
    else:
        fc1_rows = [(rank * fr, (rank + 1) * fr)]
    return {"qkv_rows": qkv_rows, "o_cols": [(q0, q0 + hr * d)],
            "fc1_rows": fc1_rows, "fc2_cols": [(rank * fr, (rank + 1) * fr)]}


def shard_weights(cfg: LayerConfig, w: Dict[str, np.ndarray], tp: int, rank: int) -> Dict[str, np.ndarray]:
    """Rank `rank`'s weights (index selection only).  Norm weights and the
    row-parallel biases b_o / b_fc2 are replicated; every rank holds them."""
    r = shard_row_ranges(cfg, tp, rank)

    def rows(a, ranges):
        return None if a is None else np.ascontiguousarray(np.concatenate([a[lo:hi] for lo, hi in ranges], axis=0))

    def cols(a, ranges):
        return None if a is None else np.ascontiguousarray(np.concatenate([a[:, lo:hi] for lo, hi in ranges], axis=1))

    out = dict(w)
    out["w_qkv"], out["b_qkv"] = rows(w["w_qkv"], r["qkv_rows"]), rows(w.get("b_qkv"), r["qkv_rows"])
    out["w_o"] = cols(w["w_o"], r["o_cols"])
    out["w_fc1"], out["b_fc1"] = rows(w["w_fc1"], r["fc1_rows"]), rows(w.get("b_fc1"), r["fc1_rows"])
    out["w_fc2"] = cols(w["w_fc2"], r["fc2_cols"])
    return out


def random_e4m3_codes(shape, seed: int, max_exponent_field: int = 9) -> np.ndarray:
    """Seeded random E4M3 bit patterns: uniform sign, exponent field 0..max_exponent_field (so no
    NaN code and magnitudes below 2^(max_exponent_field-6)), uniform 3-bit mantissa."""
    rng = np.random.Generator(np.random.PCG64(seed))
    sign = rng.integers(0, 2, size=shape, dtype=np.uint8) << np.uint8(7)
    expo = rng.integers(0, max_exponent_field + 1, size=shape, dtype=np.uint8) << np.uint8(3)
    mant = rng.integers(0, 8, size=shape, dtype=np.uint8)
    return (sign | expo | mant).astype(np.uint8)
