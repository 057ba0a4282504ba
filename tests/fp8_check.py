"""Stage checks of the FP8 (E4M3) layer against the float64 FP8 oracle, shared by the GPU FP8
tests and the CPU test that plants skipped casts in the oracle (tests/test_oracle_fp8.py).

A quantised code is an integer decided by floating point, so each stage is checked from inputs
that both sides hold identically wherever the implementation exposes them:

* codes: the E4M3 codes of an activation against the oracle's codes of the same values, as the
  fraction of codes that differ, each by at most one step or, where the two sides' inputs to the
  cast differ by a bounded amount, by at most that amount (`slack`, in the scaled units the codes
  encode: near zero, where E4M3 steps are fine, a small difference spans several codes);
* attention stage: the stored bf16 h = x + Y_attn + b_o against the oracle's attention block with
  the kernels' storage precision (q, k bf16, v fp16), rounded to bf16 the same way; the relative
  Frobenius distance must stay below H_STAGE_FRAC of the FP8 envelope of that block (the distance
  between the oracle's FP8 and exact blocks);
* MLP stage: y against the oracle's MLP block run from the implementation's own stored h, rounded
  to bf16; the distance must stay below Y_STAGE_FRAC of the MLP block's FP8 envelope.

Why these fractions: a float64 attention block that skips the bf16/fp16 storage rounding of q, k,
v (a correct FP8 computation that decides some codes of o one step apart) lands at 0.33-0.36 of
the envelope on the test shapes, while one that leaves xn or o unquantised lands at 0.88-1.46;
an MLP block accumulated in float32 lands below 0.02, one that leaves hn or a unquantised at
0.56-1.27.  H_STAGE_FRAC = 0.6 and Y_STAGE_FRAC = 0.25 sit between those.
"""
import numpy as np

from oracle import fp8 as of

H_STAGE_FRAC = 0.6
Y_STAGE_FRAC = 0.25


def code_positions(codes):
    """Signed position of each E4M3 code on the number line (+0 and -0 are both 0)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def assert_codes_close(got, want, max_mismatch, what, slack=0.0):
    g, w = code_positions(got), code_positions(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    frac = float(np.mean(g != w))
    dv = np.abs(of.e4m3_decode(got) - of.e4m3_decode(want))
    bad = (np.abs(g - w) > 1) & ~(dv <= slack)
    assert frac <= max_mismatch and not bad.any(), (
        f"{what}: {frac:.2e} of the codes differ (bound {max_mismatch:.1e}); {int(bad.sum())} by more than one step "
        f"and more than {slack:.3g} (largest value difference {float(dv.max()) if dv.size else 0.0:.3g})")
    return frac


def rel_distance(got, want, fp8, exact):
    """|got - want|_F over |fp8 - exact|_F: the distance in units of the FP8 envelope."""
    env = np.linalg.norm(np.asarray(fp8, np.float64) - np.asarray(exact, np.float64))
    return float(np.linalg.norm(np.asarray(got, np.float64) - np.asarray(want, np.float64)) / max(env, 1e-300))


def assert_attention_stage(h_got, h_fp8, h_exact, what):
    """h_got: the implementation's stored bf16 h (as float64); h_fp8: the oracle's attention block
    (storage rounding, h unrounded); h_exact: the exact layer's h."""
    r = rel_distance(h_got, of.round_bf16(h_fp8), h_fp8, h_exact)
    assert r <= H_STAGE_FRAC, f"{what}: attention stage at {r:.3f} of the FP8 envelope (bound {H_STAGE_FRAC})"
    return r


def assert_mlp_stage(y_got, y_fp8, y_exact, what):
    """y_got: the implementation's bf16 y; y_fp8, y_exact: the oracle's FP8 and exact MLP blocks run
    from the implementation's own h (y = h + Y_mlp + b_fc2, unrounded)."""
    r = rel_distance(y_got, of.round_bf16(y_fp8), y_fp8, y_exact)
    assert r <= Y_STAGE_FRAC, f"{what}: MLP stage at {r:.3f} of the FP8 envelope (bound {Y_STAGE_FRAC})"
    return r
