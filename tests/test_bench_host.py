"""Host logic of bench.py that needs no GPU: the DRAM traffic a bench line reports for its roofline
kernel comes from an ncu summary under profiles/ only while the kernel sources that summary names
are unchanged (otherwise the line reports null); the per-step statistics of the timed steps; the
dense-convention FLOP count."""
import hashlib
import os
import re

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _tree(tmp, source, recorded_source=None, traffic=412984576):
    csrc = tmp / "megatron_tensor_transformer_gpt_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(source)
    (csrc / "c.cuh").write_text("common")
    sha = hashlib.sha256((recorded_source or source).encode()).hexdigest()[:16]
    common = hashlib.sha256(b"common").hexdigest()[:16]
    prof = tmp / "profiles"
    prof.mkdir()
    (prof / "k.md").write_text(f"# k\n\nsource_sha256_16: k.cu {sha}, c.cuh {common}\n"
                               f"traffic_bytes_per_launch: {traffic}\n")


def test_traffic_is_read_while_the_sources_match(tmp_path, monkeypatch):
    _tree(tmp_path, "kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("k.md") == 412984576


def test_traffic_is_null_once_a_source_changed(tmp_path, monkeypatch):
    _tree(tmp_path, "kernel v1", recorded_source="kernel v0")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("k.md") is None


def test_traffic_is_null_without_a_summary(tmp_path, monkeypatch):
    _tree(tmp_path, "kernel v1")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("missing.md") is None


def test_committed_summaries_name_existing_sources():
    """Every committed summary that records traffic or source hashes names sources that exist, in
    the form the bench parses."""
    csrc = os.path.join(ROOT, "megatron_tensor_transformer_gpt_gb300", "csrc")
    seen = 0
    for name in sorted(os.listdir(os.path.join(ROOT, "profiles"))):
        text = open(os.path.join(ROOT, "profiles", name)).read()
        shas = re.search(r"source_sha256_16:(.*)", text)
        if "traffic_bytes_per_launch" in text:
            assert shas, name
            assert int(re.search(r"traffic_bytes_per_launch:\s*(\d+)", text).group(1)) > 0
        if shas:
            pairs = re.findall(r"([\w.]+)\s+([0-9a-f]{16})", shas.group(1))
            assert pairs, name
            for src, _ in pairs:
                assert os.path.exists(os.path.join(csrc, src)), (name, src)
            seen += 1
    assert seen >= 1


def test_step_statistics():
    assert bench.step_stats([5.0, 1.0, 3.0, 2.0, 4.0]) == [3.0, 1.4, 4.6]
    assert bench.step_stats([2.5]) == [2.5, 2.5, 2.5]


def test_dense_convention_counts_the_whole_score_square():
    cfg = synth.CONFIGS["llama8b"]
    attn_half = cfg.attn_flops()                       # 4 d S (S + 1) / 2 per head
    dense = bench.dense_convention_flops(cfg)
    assert abs(dense - (cfg.flops() - attn_half + 2.0 * attn_half * cfg.seq / (cfg.seq + 1))) < 1e3
    assert round(dense / 1e9, 1) == 2061.6
    rank = synth.CONFIGS["llama70b_tp8"]                # one rank of eight: its own heads only
    assert bench.dense_convention_flops(rank) == rank.gemm_flops() + 4.0 * 128 * 4096 * 4096 * 8


def test_rank_shapes_match_the_sharded_host_inputs():
    """The device-drawn inputs of the bench's other workloads have the shapes of one rank's shard
    of the seeded host inputs (absent tensors absent)."""
    for name in ("tiny", "gpt345m", "llama70b_tp8"):
        cfg = synth.CONFIGS[name]
        small = cfg.replace(hidden=64, heads=cfg.tp * 2, groups=cfg.tp, head_dim=cfg.head_dim, ffn=cfg.tp * 16,
                            seq=8, batch=1)
        inp = synth.make_inputs(small, seed=0)
        shard = synth.shard_weights(small, inp, small.tp, 0) if small.tp > 1 else inp
        want = {k: v.shape for k, v in shard.items() if v is not None and k != "x"}
        assert bench.rank_shapes(small) == want, name
