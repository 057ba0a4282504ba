"""GPU parity: the CUDA path (through the C ABI) against the float64 CPU oracle on the same seeded inputs.

Tolerance (the layer's): |gpu - oracle| <= 2e-2 * max|oracle| + 1e-3 elementwise, bf16 inputs,
fp32 accumulation.  Small cases, the Llama-3-8B-shaped layer and the eight summed shards of the
70B-shaped TP = 8 layer compare every element; the 32k-token layer compares sampled rows that the
oracle computes one by one (K and V for every token, the rest for the sampled rows).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import layer as ol
import synth
from megatron_tensor_transformer_gpt_gb300 import mt_layer as ml
from tests.gpu_util import (DeviceLayer, assert_layer_close, sample_rows, to_dev, to_f64, tp_sum_on_device)

pytestmark = pytest.mark.gpu


def small(**kw):
    base = dict(name="small", batch=1, seq=256, hidden=512, heads=8, groups=2, head_dim=64, ffn=1000,
                norm="rms", act="swiglu", rope_base=1e4, bias=False)
    base.update(kw)
    return synth.LayerConfig(**base)


@pytest.fixture(autouse=True)
def _cuda():
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


# ----------------------------------------------------------------------------------- GEMM
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 128), (300, 520, 200), (1, 8, 8), (1000, 1376, 688),
                                   (777, 264, 1032), (2048, 3072, 4096)])
def test_gemm_matches_oracle_linear(M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    a = synth.f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    b = synth.f32_to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32))
    A, B = to_dev(a), to_dev(b)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ml.mt_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    want = ol.linear(ol.bf16_to_f64(a), ol.bf16_to_f64(b))
    got = to_f64(C)
    err = np.abs(got - want)
    assert np.all(err <= 4e-3 * np.abs(want) + 1e-3 * np.max(np.abs(want))), err.max()


# ----------------------------------------------------------------------------------- intermediates
def _oracle_pieces(cfg, inp):
    T, B, S, d = cfg.tokens, cfg.batch, cfg.seq, cfg.head_dim
    x = ol._tokens(inp["x"], cfg)
    xn = ol.apply_norm(cfg, x, ol.bf16_to_f64(inp["norm1_w"]), ol.bf16_to_f64(inp["norm1_b"]))
    qkv = ol.linear(xn, ol.bf16_to_f64(inp["w_qkv"]), ol.bf16_to_f64(inp["b_qkv"]))
    nh, ng = cfg.heads, cfg.groups
    q = qkv[:, :nh * d].reshape(T, nh, d)
    k = qkv[:, nh * d:(nh + ng) * d].reshape(T, ng, d)
    v = qkv[:, (nh + ng) * d:].reshape(T, ng, d)
    if cfg.rope_base > 0:
        c, s = ol.rope_cos_sin(np.arange(T) // B, d, cfg.rope_base)
        q, k = ol.rope(q, c, s), ol.rope(k, c, s)
    o = np.empty((T, nh, d))
    for b in range(B):
        o[b::B] = ol.causal_attention(q[b::B], k[b::B], v[b::B], np.arange(S))
    return dict(xn=xn, q=q, k=k, v=v, o=o.reshape(T, nh * d))


@pytest.mark.parametrize("cfg", [synth.CONFIGS["tiny"], small(batch=3, seq=200), small(head_dim=128, heads=4, groups=1),
                                 small(batch=2, seq=130, norm="layer", act="gelu_tanh", bias=True)],
                         ids=["tiny", "ragged_b3_s200", "mqa_d128", "ln_gelu_b2_s130"])
def test_intermediates_match_oracle(cfg):
    inp = synth.make_inputs(cfg, seed=21, affine="random")
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    y = dl.forward(x)
    torch.cuda.synchronize()
    dl.layer.status()
    T, B, S, d, nh, ng = cfg.tokens, cfg.batch, cfg.seq, cfg.head_dim, cfg.heads, cfg.groups
    ref = _oracle_pieces(cfg, inp)

    def reg(name, shape, dtype=torch.bfloat16):
        return to_f64(dl.layer.region(S, B, name).view(dtype)[: int(np.prod(shape))].reshape(shape))

    assert_layer_close(reg("xn", (T, cfg.hidden)), ref["xn"], "norm1")
    q = reg("q", (B, nh, S, d))
    assert_layer_close(q, ref["q"].reshape(S, B, nh, d).transpose(1, 2, 0, 3), "q after RoPE")
    k = reg("k", (B, ng, S, d))
    assert_layer_close(k, ref["k"].reshape(S, B, ng, d).transpose(1, 2, 0, 3), "k after RoPE")
    v = reg("v", (B, ng, S, d), torch.float16)
    assert_layer_close(v, ref["v"].reshape(S, B, ng, d).transpose(1, 2, 0, 3), "v (fp16)")
    assert_layer_close(reg("o", (T, nh * d)), ref["o"], "attention output")
    full = ol.layer_forward(cfg, inp)
    assert_layer_close(reg("h", (T, cfg.hidden)), full["h"], "h")
    want_hn = ol.apply_norm(cfg, full["h"], ol._w(inp, "norm2_w"), ol._w(inp, "norm2_b"))
    assert_layer_close(reg("hn", (T, cfg.hidden)), want_hn, "norm2")
    assert_layer_close(to_f64(y), full["y"], "y")
    dl.close()


# ----------------------------------------------------------------------------------- whole layer, small
EDGE = [
    synth.CONFIGS["tiny"],
    small(),
    small(batch=3, seq=200),                                   # ragged tokens, batch > 1
    small(seq=1),                                              # single token
    small(seq=129, heads=4, groups=1, head_dim=128),           # MQA, d=128, one-past-a-tile
    small(seq=130, head_dim=128, heads=4, groups=1, norm="layer", act="gelu_tanh", rope_base=0.0, bias=True),
    small(batch=2, seq=384, heads=16, groups=2, ffn=1376),     # 8 heads per group
    small(hidden=264, heads=2, groups=2, ffn=520, seq=64),     # hidden and ffn not multiples of 64/128
    small(heads=6, groups=2, seq=300),                         # 3 heads per group: a CTA's two heads straddle groups
    small(batch=2, seq=300, heads=8, groups=2, head_dim=128),  # GQA d=128, batch 2, three query blocks
]


@pytest.mark.parametrize("cfg", EDGE, ids=lambda c: f"{c.name}-b{c.batch}-s{c.seq}-h{c.hidden}-"
                                                     f"{c.heads}x{c.groups}x{c.head_dim}-{c.norm}-{c.act}")
@pytest.mark.parametrize("affine", ["standard", "random"])
def test_layer_matches_oracle_small(cfg, affine):
    inp = synth.make_inputs(cfg, seed=3, affine=affine, biases="random")
    dl = DeviceLayer(cfg, inp)
    y = dl.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden))
    torch.cuda.synchronize()
    dl.layer.status()
    assert_layer_close(to_f64(y), ol.layer_forward(cfg, inp)["y"], cfg.name)
    dl.close()


# Attention forms (mt_attn_set_heads_per_cta): the automatic choice takes one head per CTA for all
# of these small layers; mode 2 forces two heads of one group per CTA (and, for MHA at d = 64, two
# heads of two groups).  Ragged sequences, batch > 1, an odd number of query blocks, MQA, GQA with
# eight heads per group.
ATTN_FORMS = [
    small(),
    small(batch=3, seq=200),
    small(seq=129, heads=4, groups=1, head_dim=128),
    small(batch=2, seq=300, heads=8, groups=2, head_dim=128),
    small(batch=2, seq=384, heads=16, groups=2, ffn=1376),
    small(groups=8, seq=300),                                  # MHA, d = 64
    small(heads=6, groups=2, seq=300, head_dim=128),           # 3 heads per group
]


@pytest.mark.parametrize("cfg", ATTN_FORMS, ids=lambda c: f"b{c.batch}-s{c.seq}-{c.heads}x{c.groups}x{c.head_dim}")
def test_attention_forms_match_oracle(cfg):
    inp = synth.make_inputs(cfg, seed=8, affine="random", biases="random")
    want = ol.layer_forward(cfg, inp)["y"]
    ys = {}
    try:
        for mode in (1, 2):
            ml.mt_attn_set_heads_per_cta(mode)
            dl = DeviceLayer(cfg, inp)
            y = dl.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden))
            torch.cuda.synchronize()
            dl.layer.status()
            ys[mode] = y.clone()
            assert_layer_close(to_f64(y), want, f"{cfg.name} heads-per-CTA mode {mode}")
            dl.close()
    finally:
        ml.mt_attn_set_heads_per_cta(0)
    if (cfg.heads // cfg.groups) % 2 == 0:  # one and two heads of one group: the same arithmetic
        assert torch.equal(ys[1], ys[2])


def test_gpt345m_full_layer():
    cfg = synth.CONFIGS["gpt345m"]
    inp = synth.make_inputs(cfg, seed=0)
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    y = dl.forward(x).clone()
    torch.cuda.synchronize()
    dl.layer.status()
    assert_layer_close(to_f64(y), ol.layer_forward(cfg, inp)["y"], "gpt345m")
    # every output element is summed in a fixed order: a second call is bit-identical
    assert torch.equal(dl.forward(x), y)
    dl.close()


# ----------------------------------------------------------------------------------- tensor parallel
@pytest.mark.parametrize("tp", [2, 4])
def test_tp_shards_sum_to_the_unsharded_layer(tp):
    cfg = small(heads=8, groups=4, ffn=1024, bias=True, norm="layer")
    inp = synth.make_inputs(cfg, seed=9, affine="random", biases="random")
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    h, y = tp_sum_on_device(cfg, inp, x, tp)
    torch.cuda.synchronize()
    want = ol.layer_forward(cfg, inp)
    assert_layer_close(to_f64(h), want["h"], "h from summed partials")
    assert_layer_close(to_f64(y), want["y"], "y from summed partials")
    shards = [synth.shard_weights(cfg, inp, tp, r) for r in range(tp)]
    assert_layer_close(to_f64(y), ol.layer_forward_tp_sum(cfg, tp, inp["x"], shards)["y"], "y vs oracle TP sum")


@pytest.mark.parametrize("bias", [False, True], ids=["no-bias", "biases"])
def test_rank_identity_mode(bias):
    """One rank with the all-reduce replaced by the identity: h = x + Y_attn,i + b_o (b_o once) and
    y_partial = Y_mlp,i(h) without residual or b_fc2; with random biases on every linear."""
    cfg = small(heads=8, groups=4, ffn=1024, bias=bias)
    inp = synth.make_inputs(cfg, seed=10, affine="random", biases="random")
    tp, r = 4, 1
    dl = DeviceLayer(cfg, inp, tp, r)
    y = dl.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden))
    torch.cuda.synchronize()
    want = ol.layer_forward_rank_identity(cfg, tp, inp["x"], synth.shard_weights(cfg, inp, tp, r))
    h = to_f64(dl.layer.region(cfg.seq, cfg.batch, "h").view(torch.bfloat16)[: cfg.tokens * cfg.hidden]
               .reshape(cfg.tokens, cfg.hidden))
    assert_layer_close(h, want["h"], "identity-mode h")
    assert_layer_close(to_f64(y), want["y_partial"], "identity-mode y_partial")
    dl.close()


# ----------------------------------------------------------------------------------- full-size workloads
def test_llama8b_full_size_every_row():
    """The Llama-3-8B-shaped layer at its full size (4096 tokens), every element of y against the
    oracle's whole layer."""
    cfg = synth.CONFIGS["llama8b"]
    inp = synth.make_inputs(cfg, seed=0)
    dl = DeviceLayer(cfg, inp)
    y = dl.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden))
    torch.cuda.synchronize()
    dl.layer.status()
    got = to_f64(y)
    dl.close()
    del y
    torch.cuda.empty_cache()
    assert_layer_close(got, ol.layer_forward(cfg, inp)["y"], "llama8b, all rows")


def _full_size_sampled(name, n_random):
    cfg = synth.CONFIGS[name]
    inp = synth.make_inputs(cfg, seed=0)
    dl = DeviceLayer(cfg, inp)
    y = dl.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden))
    torch.cuda.synchronize()
    dl.layer.status()
    rows = sample_rows(cfg.tokens, seed=1, n_random=n_random)
    got = to_f64(y[torch.from_numpy(rows).cuda()])
    dl.close()
    del y
    torch.cuda.empty_cache()
    assert_layer_close(got, ol.layer_forward(cfg, inp, rows=rows)["y"], name)


def test_llama8b_32k_full_size_sampled_rows():
    _full_size_sampled("llama8b_32k", 128)


def test_llama70b_tp8_all_shards_sum_to_unsharded_oracle():
    """The eight TP = 8 ranks of the 70B-shaped layer, run one after another; their row-parallel
    partials summed (fp32) give h and y, compared on every row with the unsharded oracle layer."""
    cfg = synth.CONFIGS["llama70b_tp8"]
    inp = synth.make_inputs(cfg, seed=0)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    h, y = tp_sum_on_device(cfg, inp, x, cfg.tp)
    torch.cuda.synchronize()
    got_h, got_y = to_f64(h), to_f64(y)
    del h, y, x
    torch.cuda.empty_cache()
    want = ol.layer_forward(cfg, inp)
    assert_layer_close(got_h, want["h"], "llama70b tp8 summed h")
    assert_layer_close(got_y, want["y"], "llama70b tp8 summed y")


def test_llama70b_tp8_one_rank_identity_mode():
    cfg = synth.CONFIGS["llama70b_tp8"]
    inp = synth.make_inputs(cfg, seed=0)
    r = 5
    sh = synth.shard_weights(cfg, inp, cfg.tp, r)
    dl = DeviceLayer(cfg, inp, cfg.tp, r)
    y = dl.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden))
    torch.cuda.synchronize()
    dl.layer.status()
    rows = sample_rows(cfg.tokens, seed=3, n_random=32)
    got = to_f64(y[torch.from_numpy(rows).cuda()])
    dl.close()
    want = ol.layer_forward_rank_identity(cfg, cfg.tp, inp["x"], sh, rows=rows)
    assert_layer_close(got, want["y_partial"], "llama70b rank identity")


# ----------------------------------------------------------------------------------- properties
def test_deterministic_and_host_path_matches():
    cfg = small(batch=2, seq=192)
    inp = synth.make_inputs(cfg, seed=4, affine="random")
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    y1 = dl.forward(x).clone()
    y2 = dl.forward(x).clone()
    assert torch.equal(y1, y2)
    # pinned (asynchronous copies) and pageable (staged copies) host buffers give the same y
    for x_pinned in (True, False):
        for y_pinned in (True, False):
            xh = x.cpu().pin_memory() if x_pinned else x.cpu()
            yh = torch.full((cfg.tokens, cfg.hidden), float("nan"), dtype=torch.bfloat16)
            yh = yh.pin_memory() if y_pinned else yh
            dl.layer.forward_host(xh, cfg.seq, cfg.batch, dl.w, yh)
            torch.cuda.synchronize()
            assert torch.equal(y1.cpu(), yh), (x_pinned, y_pinned)


@pytest.mark.parametrize("cfg", [small(), synth.CONFIGS["llama8b"]], ids=["small", "llama8b"])
def test_forward_replays_from_a_cuda_graph(cfg):
    """The forward is stream-ordered (programmatic-dependent launches, no host synchronisation), so a
    CUDA graph captured from it replays it: the output equals the eager forward bit for bit."""
    inp = synth.make_inputs(cfg, seed=8, affine="random")
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    want = dl.forward(x).clone()  # eager first: kernel attributes and workspace are set up here
    y = torch.full_like(want, float("nan"))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        dl.layer.forward(x, cfg.seq, cfg.batch, dl.w, y)  # one run on the capture stream before capturing
        with torch.cuda.graph(graph, stream=side):
            dl.layer.forward(x, cfg.seq, cfg.batch, dl.w, y)
    torch.cuda.current_stream().wait_stream(side)
    y.fill_(float("nan"))
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    dl.layer.status()
    assert torch.equal(want, y)
    dl.close()


@pytest.mark.parametrize("cfg", [small(batch=2, seq=320), small(seq=700, heads=4, groups=1, head_dim=128),
                                 small(batch=2, seq=4096)],
                         ids=["640-tokens-gqa", "700-tokens-mqa-d128", "8192-tokens-four-chunks"])
def test_host_path_chunked_copies_match(cfg):
    """With pinned buffers and 512 tokens or more (8192: four chunks) the host-buffer path copies x and
    y in row chunks on a copy stream, overlapped with norm1 + QKV of the chunks already in and fc2 of
    the chunks still to come; every row still equals the device path bit for bit, over repeated calls."""
    inp = synth.make_inputs(cfg, seed=9, affine="random")
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    want = dl.forward(x).cpu()
    xh = x.cpu().pin_memory()
    for _ in range(3):
        yh = torch.full((cfg.tokens, cfg.hidden), float("nan"), dtype=torch.bfloat16).pin_memory()
        dl.layer.forward_host(xh, cfg.seq, cfg.batch, dl.w, yh)
        torch.cuda.synchronize()
        assert torch.equal(want, yh)
    dl.layer.status()
    dl.close()


@pytest.mark.parametrize("norm", ["rms", "layer"])
def test_launch_count_and_profile_mask(norm):
    """A dense forward launches seven kernels (the RoPE table rides on norm1), with either norm; a
    slot mask brackets only the selected slot."""
    launches = 7
    cfg = small(norm=norm)
    inp = synth.make_inputs(cfg, seed=5)
    dl = DeviceLayer(cfg, inp)
    x = to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden)
    dl.forward(x)
    torch.cuda.synchronize()
    n0 = ml.mt_layer_launch_count(dl.layer.handle)
    fc1 = ml.PROFILE_SLOTS.index("gemm_fc1")
    ml.mt_layer_profile_enable(dl.layer.handle, 1 << fc1)
    dl.forward(x)
    dl.forward(x)
    torch.cuda.synchronize()
    prof = ml.mt_layer_profile_read(dl.layer.handle)
    ml.mt_layer_profile_enable(dl.layer.handle, False)
    assert ml.mt_layer_launch_count(dl.layer.handle) - n0 == 2 * launches
    assert prof["gemm_fc1"][0] == 2 and prof["gemm_fc1"][1] > 0
    assert all(n == 0 for k, (n, _) in prof.items() if k != "gemm_fc1")
    with pytest.raises(ml.MtError):
        ml.mt_layer_profile_enable(dl.layer.handle, 1 << 8)
    dl.close()


def test_output_guard_regions_untouched():
    cfg = small(batch=1, seq=200)
    inp = synth.make_inputs(cfg, seed=5)
    dl = DeviceLayer(cfg, inp)
    n, pad = cfg.tokens * cfg.hidden, 4096
    buf = torch.full((n + 2 * pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[pad:pad + n].view(cfg.tokens, cfg.hidden)
    dl.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden), out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 7.0) and torch.all(buf[pad + n:] == 7.0)
    assert_layer_close(to_f64(out), ol.layer_forward(cfg, inp)["y"], "guarded")


def test_bounded_wait_reports_and_context_survives():
    assert ml.mt_selftest_bounded_wait(2000) == ml.MT_ERR_DEVICE_TIMEOUT
    assert "gave up" in ml.mt_last_error()
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_inputs(cfg, seed=0)
    dl = DeviceLayer(cfg, inp)
    y = dl.forward(to_dev(inp["x"]).reshape(cfg.tokens, cfg.hidden))
    torch.cuda.synchronize()
    dl.layer.status()
    assert_layer_close(to_f64(y), ol.layer_forward(cfg, inp)["y"], "after self test")


def test_workspace_errors():
    cfg = synth.CONFIGS["tiny"]
    layer = ml.Layer.from_config(cfg)
    x = torch.zeros(cfg.tokens, cfg.hidden, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ml.MtError) as e:
        ml.mt_layer_forward(layer.handle, x.data_ptr(), cfg.seq, cfg.batch, ml.MtWeights(), x.data_ptr(), None)
    assert e.value.code == ml.MT_ERR_NO_WORKSPACE
    need = ml.mt_layer_workspace_bytes(layer.handle, cfg.seq, cfg.batch)
    ws = torch.empty(need - 1024, dtype=torch.uint8, device="cuda")
    ml.mt_layer_set_workspace(layer.handle, ws.data_ptr(), ws.numel())
    with pytest.raises(ml.MtError) as e:
        ml.mt_layer_forward(layer.handle, x.data_ptr(), cfg.seq, cfg.batch, ml.MtWeights(), x.data_ptr(), None)
    assert e.value.code == ml.MT_ERR_NO_WORKSPACE
    layer.close()
