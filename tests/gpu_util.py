"""Helpers for the GPU parity tests: moving seeded bf16 inputs to the device and the tolerance."""
import numpy as np
import torch

import oracle
import synth
from megatron_tensor_transformer_gpt_gb300 import mt_layer as ml


def to_dev(bits, device="cuda"):
    if bits is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def assert_layer_close(got, want, what=""):
    """The layer tolerance: |gpu - oracle| <= 2e-2 * max|oracle| + 1e-3 for every element."""
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    bound = 2e-2 * np.max(np.abs(want)) + 1e-3
    i = np.unravel_index(np.argmax(err), err.shape)
    assert np.all(err <= bound), (f"{what}: max err {err.max():.4e} at {i} (got {got[i]:.5f}, want {want[i]:.5f}) "
                                  f"> bound {bound:.4e}")
    return float(err.max()), float(bound)


def sample_rows(T, seed=0, n_random=192):
    """Rows a full-size check samples: the first and last 128, the rows around every 128-row tile
    boundary, and seeded random rows."""
    rows = set(range(min(128, T))) | set(range(max(0, T - 128), T))
    for b in range(128, T, 128):
        rows |= {b - 1, b}
    rng = np.random.default_rng(seed)
    rows |= set(rng.integers(0, T, n_random).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < T))


class DeviceLayer:
    """A layer handle plus the device copies of one rank's weights."""

    def __init__(self, cfg, inp, tp_size=1, tp_rank=0):
        self.cfg = cfg
        self.layer = ml.Layer.from_config(cfg, tp_rank=tp_rank, tp_size=tp_size)
        w = inp if tp_size == 1 else synth.shard_weights(cfg, inp, tp_size, tp_rank)
        self.tens = {k: to_dev(v) for k, v in w.items() if k != "x"}
        self.w = self.layer.weights(self.tens)

    def forward(self, x, out=None):
        cfg = self.cfg
        out = torch.empty(cfg.tokens, cfg.hidden, dtype=torch.bfloat16, device=x.device) if out is None else out
        self.layer.forward(x, cfg.seq, cfg.batch, self.w, out)
        return out

    def forward_attn(self, x):
        out = torch.empty(self.cfg.tokens, self.cfg.hidden, dtype=torch.bfloat16, device=x.device)
        self.layer.forward_attn(x, self.cfg.seq, self.cfg.batch, self.w, out)
        return out

    def forward_mlp(self, h):
        out = torch.empty(self.cfg.tokens, self.cfg.hidden, dtype=torch.bfloat16, device=h.device)
        self.layer.forward_mlp(h, self.cfg.seq, self.cfg.batch, self.w, out)
        return out

    def close(self):
        self.layer.close()


def tp_sum_on_device(cfg, inp, x_dev, tp):
    """Run every rank's staged blocks one after another and sum the row-parallel partials in fp32
    (the all-reduce stand-in): h = x + sum Y_attn,i + b_o, y = h + sum Y_mlp,i + b_fc2."""
    ranks = [DeviceLayer(cfg, inp, tp, r) for r in range(tp)]
    acc = torch.zeros(cfg.tokens, cfg.hidden, dtype=torch.float32, device=x_dev.device)
    for r in ranks:
        acc += r.forward_attn(x_dev).float()
    h = x_dev.float() + acc
    if inp.get("b_o") is not None:
        h += to_dev(inp["b_o"]).float()
    h = h.to(torch.bfloat16)
    acc.zero_()
    for r in ranks:
        acc += r.forward_mlp(h).float()
    y = h.float() + acc
    if inp.get("b_fc2") is not None:
        y += to_dev(inp["b_fc2"]).float()
    for r in ranks:
        r.close()
    return h, y.to(torch.bfloat16)
