"""Python binding of libmt_layer.so (the C ABI in include/mt_layer.h).

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.  The
functions carry the C names; a failing status raises MtError with the library's message.
PyTorch is used only by the ``Layer`` convenience wrapper, for device memory and streams.
There is no fallback: if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmt_layer.so")

MT_NORM_RMS, MT_NORM_LAYER = 0, 1
MT_ACT_SWIGLU, MT_ACT_GELU_TANH = 0, 1
MT_OK, MT_ERR_INVALID_ARG, MT_ERR_UNSUPPORTED, MT_ERR_NO_WORKSPACE = 0, 1, 2, 3
MT_ERR_CUDA, MT_ERR_DEVICE_TIMEOUT, MT_ERR_UNIMPLEMENTED = 4, 5, 6

WEIGHT_FIELDS = ("norm1_w", "norm1_b", "w_qkv", "b_qkv", "w_o", "b_o",
                 "norm2_w", "norm2_b", "w_fc1", "b_fc1", "w_fc2", "b_fc2")

# workspace regions (mt_layer_workspace_region)
REGION = {"xn": 0, "q": 1, "k": 2, "v": 3, "o": 4, "h": 5, "hn": 6, "a": 7, "rope": 8}


class MtWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


class MtGrads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


class MtFp8Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("w_qkv", "w_o", "w_fc1", "w_fc2",
                                                "deq_qkv", "deq_o", "deq_fc1", "deq_fc2")]


class MtError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[mt status {code}] {msg}")
        self.code = code


_lib: Optional[ctypes.CDLL] = None

_SIGS = {
    "mt_layer_create": ([ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                              ctypes.POINTER(ctypes.c_void_p)], ctypes.c_int),
    "mt_layer_set_eps": ([ctypes.c_void_p, ctypes.c_float], ctypes.c_int),
    "mt_layer_workspace_bytes": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_size_t)],
                                 ctypes.c_int),
    "mt_layer_set_workspace": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t], ctypes.c_int),
    "mt_layer_forward": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.POINTER(MtWeights),
                          ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "mt_layer_forward_attn": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                               ctypes.POINTER(MtWeights), ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "mt_layer_forward_mlp": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                              ctypes.POINTER(MtWeights), ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "mt_layer_forward_host": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                               ctypes.POINTER(MtWeights), ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "mt_layer_workspace_region": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "mt_layer_status": ([ctypes.c_void_p], ctypes.c_int),
    "mt_last_error": ([], ctypes.c_char_p),
    "mt_layer_destroy": ([ctypes.c_void_p], None),
    "mt_gemm_set_pairing": ([ctypes.c_int], ctypes.c_int),
    "mt_attn_set_heads_per_cta": ([ctypes.c_int], ctypes.c_int),
    "mt_gemm_set_tail_split": ([ctypes.c_int], ctypes.c_int),
    "mt_gemm_plan": ([ctypes.c_int] * 9 + [ctypes.POINTER(ctypes.c_int)], ctypes.c_int),
    "mt_gemm_bf16_t": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                        ctypes.c_int, ctypes.c_int, ctypes.c_void_p], ctypes.c_int),
    "mt_gemm_bf16": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      ctypes.c_void_p], ctypes.c_int),
    "mt_selftest_bounded_wait": ([ctypes.c_int], ctypes.c_int),
    "mt_layer_profile_enable": ([ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "mt_layer_launch_count": ([ctypes.c_void_p, ctypes.POINTER(ctypes.c_ulonglong)], ctypes.c_int),
    "mt_layer_profile_read": ([ctypes.c_void_p, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_double)],
                              ctypes.c_int),
    "mt_layer_workspace_bytes_packed": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "mt_layer_forward_packed": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                 ctypes.c_int, ctypes.POINTER(MtWeights), ctypes.c_void_p, ctypes.c_void_p],
                                ctypes.c_int),
    "mt_layer_backward_workspace_bytes": ([ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                           ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
    "mt_layer_backward": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                           ctypes.POINTER(MtWeights), ctypes.c_void_p, ctypes.POINTER(MtGrads), ctypes.c_void_p],
                          ctypes.c_int),
    "mt_layer_forward_train": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                ctypes.POINTER(MtWeights), ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "mt_layer_backward_saved": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                 ctypes.POINTER(MtWeights), ctypes.c_void_p, ctypes.POINTER(MtGrads),
                                 ctypes.c_void_p], ctypes.c_int),
    "mt_layer_fp8_enable": ([ctypes.c_void_p, ctypes.c_int], ctypes.c_int),
    "mt_layer_fp8_set_scales": ([ctypes.c_void_p, ctypes.POINTER(ctypes.c_float)], ctypes.c_int),
    "mt_layer_fp8_state": ([ctypes.c_void_p, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)],
                           ctypes.c_int),
    "mt_layer_forward_fp8": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.POINTER(MtWeights),
                              ctypes.POINTER(MtFp8Weights), ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "mt_quantize_e4m3": ([ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p],
                         ctypes.c_int),
    "mt_gemm_e4m3": ([ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int),
    "mt_sp_reduce_add_norm": ([ctypes.POINTER(ctypes.c_void_p), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_void_p], ctypes.c_int),
    "mt_layer_forward_static_status": ([ctypes.c_void_p], ctypes.c_int),
    "mt_layer_forward_static": ([ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                                      ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                                      ctypes.POINTER(MtWeights), ctypes.c_void_p, ctypes.c_void_p],
                                ctypes.c_int),
}

PROFILE_SLOTS = ("attention_bwd", "norm1", "gemm_qkv", "attention", "gemm_o", "norm2", "gemm_fc1", "gemm_fc2")


def lib() -> ctypes.CDLL:
    """Load libmt_layer.so (built in-tree by build.py); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m megatron_tensor_transformer_gpt_gb300.build`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(l, name)
            f.argtypes = args
            f.restype = res
        _lib = l
    return _lib


def mt_last_error() -> str:
    return lib().mt_last_error().decode()


def _check(rc: int):
    if rc != MT_OK:
        raise MtError(rc, mt_last_error())


def mt_layer_create(hidden, heads, query_groups, head_dim, ffn, norm, act, rope_base, tp_size, tp_rank) -> int:
    h = ctypes.c_void_p()
    _check(lib().mt_layer_create(hidden, heads, query_groups, head_dim, ffn, norm, act, float(rope_base),
                                 tp_size, tp_rank, ctypes.byref(h)))
    return h.value


def mt_layer_set_eps(handle, eps):
    _check(lib().mt_layer_set_eps(handle, float(eps)))


def mt_layer_workspace_bytes(handle, seq, batch) -> int:
    n = ctypes.c_size_t()
    _check(lib().mt_layer_workspace_bytes(handle, seq, batch, ctypes.byref(n)))
    return n.value


def mt_layer_set_workspace(handle, dev_ptr, nbytes):
    _check(lib().mt_layer_set_workspace(handle, dev_ptr, nbytes))


def mt_layer_forward(handle, x, seq, batch, weights: MtWeights, y_partial, stream):
    _check(lib().mt_layer_forward(handle, x, seq, batch, ctypes.byref(weights), y_partial, stream))


def mt_layer_forward_attn(handle, x, seq, batch, weights: MtWeights, attn_out, stream):
    _check(lib().mt_layer_forward_attn(handle, x, seq, batch, ctypes.byref(weights), attn_out, stream))


def mt_layer_forward_mlp(handle, h, seq, batch, weights: MtWeights, y_partial, stream):
    _check(lib().mt_layer_forward_mlp(handle, h, seq, batch, ctypes.byref(weights), y_partial, stream))


def mt_layer_forward_host(handle, x_host, seq, batch, weights: MtWeights, y_host, stream):
    _check(lib().mt_layer_forward_host(handle, x_host, seq, batch, ctypes.byref(weights), y_host, stream))


def mt_layer_workspace_bytes_packed(handle, total_tokens, num_seqs, max_seqlen) -> int:
    n = ctypes.c_size_t()
    _check(lib().mt_layer_workspace_bytes_packed(handle, total_tokens, num_seqs, max_seqlen, ctypes.byref(n)))
    return n.value


def mt_layer_forward_packed(handle, x, total_tokens, cu_seqlens_dev, num_seqs, max_seqlen, weights: MtWeights,
                            y_partial, stream):
    _check(lib().mt_layer_forward_packed(handle, x, total_tokens, cu_seqlens_dev, num_seqs, max_seqlen,
                                         ctypes.byref(weights), y_partial, stream))


def mt_layer_workspace_region(handle, seq, batch, which):
    off, n = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().mt_layer_workspace_region(handle, seq, batch, which, ctypes.byref(off), ctypes.byref(n)))
    return off.value, n.value


def mt_layer_status(handle):
    _check(lib().mt_layer_status(handle))


def mt_layer_destroy(handle):
    lib().mt_layer_destroy(handle)


def mt_layer_launch_count(handle) -> int:
    n = ctypes.c_ulonglong(0)
    _check(lib().mt_layer_launch_count(handle, ctypes.byref(n)))
    return n.value


PROFILE_ALL = (1 << 8) - 1


def mt_layer_profile_enable(handle, slots=True):
    """slots: True (every kernel slot), False (none) or an int bit mask over the slots."""
    mask = PROFILE_ALL if slots is True else (0 if slots is False else int(slots))
    _check(lib().mt_layer_profile_enable(handle, mask))


def mt_layer_profile_read(handle):
    """{slot name: (launches, total ms)} since the last read."""
    n = len(PROFILE_SLOTS)
    launches, ms = (ctypes.c_int * n)(), (ctypes.c_double * n)()
    _check(lib().mt_layer_profile_read(handle, launches, ms))
    return {PROFILE_SLOTS[i]: (launches[i], ms[i]) for i in range(n)}


def mt_layer_forward_static_status(stream):
    _check(lib().mt_layer_forward_static_status(stream))


def mt_layer_forward_static(hidden, heads, query_groups, head_dim, ffn, norm, act, rope_base, tp_size, tp_rank, eps,
                            x, seq, batch, weights: MtWeights, y_partial, stream):
    """Whole layer without any device allocation (scratch in the library's fixed static area)."""
    _check(lib().mt_layer_forward_static(hidden, heads, query_groups, head_dim, ffn, norm, act, float(rope_base),
                                         tp_size, tp_rank, float(eps), x, seq, batch, ctypes.byref(weights),
                                         y_partial, stream))


def mt_sp_reduce_add_norm(partials, resid, bias, norm_w, norm_b, norm, eps, tokens, hidden, row0, rows, h_out,
                          hn_out, stream):
    """Sequence-parallel epilogue for one rank's slice; `partials` is a list of device pointers."""
    arr = (ctypes.c_void_p * len(partials))(*partials)
    _check(lib().mt_sp_reduce_add_norm(arr, len(partials), resid, bias, norm_w, norm_b, norm, float(eps), tokens,
                                       hidden, row0, rows, h_out, hn_out, stream))


def mt_layer_backward_workspace_bytes(handle, seq, batch) -> int:
    n = ctypes.c_size_t()
    _check(lib().mt_layer_backward_workspace_bytes(handle, seq, batch, ctypes.byref(n)))
    return n.value


def mt_layer_backward(handle, x, dy, seq, batch, weights: MtWeights, dx, grads: "MtGrads", stream):
    _check(lib().mt_layer_backward(handle, x, dy, seq, batch, ctypes.byref(weights), dx, ctypes.byref(grads), stream))


def mt_layer_forward_train(handle, x, seq, batch, weights: MtWeights, y, stream):
    _check(lib().mt_layer_forward_train(handle, x, seq, batch, ctypes.byref(weights), y, stream))


def mt_layer_backward_saved(handle, x, dy, seq, batch, weights: MtWeights, dx, grads: "MtGrads", stream):
    _check(lib().mt_layer_backward_saved(handle, x, dy, seq, batch, ctypes.byref(weights), dx, ctypes.byref(grads),
                                         stream))


def mt_layer_fp8_enable(handle, amax_history_len=1024):
    _check(lib().mt_layer_fp8_enable(handle, int(amax_history_len)))


def mt_layer_fp8_set_scales(handle, scales):
    arr = (ctypes.c_float * 4)(*[float(s) for s in scales])
    _check(lib().mt_layer_fp8_set_scales(handle, arr))


def mt_layer_fp8_state(handle):
    """(scales[4], last_amax[4]) of the activations (normed x, attention out, normed h, MLP hidden)."""
    sc, am = (ctypes.c_float * 4)(), (ctypes.c_float * 4)()
    _check(lib().mt_layer_fp8_state(handle, sc, am))
    return list(sc), list(am)


def mt_layer_forward_fp8(handle, x, seq, batch, weights: MtWeights, w8: MtFp8Weights, y_partial, stream):
    _check(lib().mt_layer_forward_fp8(handle, x, seq, batch, ctypes.byref(weights), ctypes.byref(w8), y_partial,
                                      stream))


def mt_quantize_e4m3(src, n, dst, amax_deq, stream):
    _check(lib().mt_quantize_e4m3(src, n, dst, amax_deq, stream))


def mt_gemm_e4m3(A, B, C, M, N, K, deq_a, deq_b, stream):
    _check(lib().mt_gemm_e4m3(A, B, C, M, N, K, deq_a, deq_b, stream))


def mt_gemm_bf16_t(A, a_layout, B, b_layout, C, M, N, K, stream):
    _check(lib().mt_gemm_bf16_t(A, a_layout, B, b_layout, C, M, N, K, stream))


def mt_gemm_set_pairing(mode):
    _check(lib().mt_gemm_set_pairing(mode))


def mt_attn_set_heads_per_cta(mode):
    _check(lib().mt_attn_set_heads_per_cta(mode))


def mt_gemm_set_tail_split(mode):
    _check(lib().mt_gemm_set_tail_split(mode))


PLAN_FIELDS = ("pair", "tiles_m", "tiles_n", "split", "ksplit", "full_units", "num_units", "epi_split")


def mt_gemm_plan(M, N, K, epilogue, head_dim=0, fp8=False, with_handle=True, sms=152, pair_slots=76):
    out = (ctypes.c_int * 8)()
    _check(lib().mt_gemm_plan(M, N, K, epilogue, head_dim, int(fp8), int(with_handle), sms, pair_slots, out))
    return dict(zip(PLAN_FIELDS, list(out)))


def mt_gemm_bf16(A, B, C, M, N, K, stream):
    _check(lib().mt_gemm_bf16(A, B, C, M, N, K, stream))


def mt_selftest_bounded_wait(limit_us) -> int:
    """Returns the status code (MT_ERR_DEVICE_TIMEOUT is the expected outcome)."""
    return lib().mt_selftest_bounded_wait(int(limit_us))


# --------------------------------------------------------------------------- torch convenience
class Layer:
    """One rank of a layer bound to torch-owned device memory (weights, workspace) and streams."""

    def __init__(self, hidden, heads, query_groups, head_dim, ffn, norm="rms", act="swiglu", rope_base=0.0,
                 tp_size=1, tp_rank=0, eps=1e-5):
        self.handle = mt_layer_create(hidden, heads, query_groups, head_dim, ffn,
                                      MT_NORM_RMS if norm == "rms" else MT_NORM_LAYER,
                                      MT_ACT_SWIGLU if act == "swiglu" else MT_ACT_GELU_TANH,
                                      rope_base, tp_size, tp_rank)
        mt_layer_set_eps(self.handle, eps)
        self.hidden = hidden
        self._ws = None
        self._ws_key = None
        self._keep = None

    @classmethod
    def from_config(cls, cfg, tp_rank=0, tp_size=None):
        return cls(cfg.hidden, cfg.heads, cfg.groups, cfg.head_dim, cfg.ffn, cfg.norm, cfg.act, cfg.rope_base,
                   cfg.tp if tp_size is None else tp_size, tp_rank, cfg.eps)

    def workspace(self, seq, batch, device=None):
        import torch
        need = mt_layer_workspace_bytes(self.handle, seq, batch)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=device or "cuda")
            mt_layer_set_workspace(self.handle, self._ws.data_ptr(), self._ws.numel())
        return self._ws

    def region(self, seq, batch, name):
        off, n = mt_layer_workspace_region(self.handle, seq, batch, REGION[name])
        return self._ws[off:off + n]

    @staticmethod
    def weights(tensors: Dict[str, "object"]) -> MtWeights:
        w = MtWeights()
        for f in WEIGHT_FIELDS:
            t = tensors.get(f)
            setattr(w, f, None if t is None else t.data_ptr())
        return w

    @staticmethod
    def _stream(stream):
        import torch
        s = torch.cuda.current_stream() if stream is None else stream
        return s.cuda_stream

    def forward(self, x, seq, batch, weights: MtWeights, out, stream=None):
        self.workspace(seq, batch, x.device)
        mt_layer_forward(self.handle, x.data_ptr(), seq, batch, weights, out.data_ptr(), self._stream(stream))
        return out

    def forward_attn(self, x, seq, batch, weights: MtWeights, out, stream=None):
        self.workspace(seq, batch, x.device)
        mt_layer_forward_attn(self.handle, x.data_ptr(), seq, batch, weights, out.data_ptr(), self._stream(stream))
        return out

    def forward_mlp(self, h, seq, batch, weights: MtWeights, out, stream=None):
        self.workspace(seq, batch, h.device)
        mt_layer_forward_mlp(self.handle, h.data_ptr(), seq, batch, weights, out.data_ptr(), self._stream(stream))
        return out

    def forward_packed(self, x, cu_seqlens, max_seqlen, weights: MtWeights, out, stream=None):
        """x, out: [total_tokens, H]; cu_seqlens: int32 device tensor of num_seqs + 1 boundaries."""
        import torch
        total, n = x.shape[0], cu_seqlens.numel() - 1
        need = mt_layer_workspace_bytes_packed(self.handle, total, n, max_seqlen)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=x.device)
            mt_layer_set_workspace(self.handle, self._ws.data_ptr(), self._ws.numel())
        mt_layer_forward_packed(self.handle, x.data_ptr(), total, cu_seqlens.data_ptr(), n, max_seqlen, weights,
                                out.data_ptr(), self._stream(stream))
        return out

    def _backward_workspace(self, seq, batch, device):
        import torch
        need = mt_layer_backward_workspace_bytes(self.handle, seq, batch)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=device)
            mt_layer_set_workspace(self.handle, self._ws.data_ptr(), self._ws.numel())

    @staticmethod
    def _grads(grads):
        g = MtGrads()
        for f in WEIGHT_FIELDS:
            t = grads.get(f)
            setattr(g, f, None if t is None else t.data_ptr())
        return g

    def backward(self, x, dy, seq, batch, weights: MtWeights, dx, grads: Dict[str, "object"], stream=None):
        """dx and the weight gradients into the given torch tensors (grads: name -> tensor or None)."""
        self._backward_workspace(seq, batch, x.device)
        mt_layer_backward(self.handle, x.data_ptr(), dy.data_ptr(), seq, batch, weights, dx.data_ptr(),
                          self._grads(grads), self._stream(stream))
        return dx

    def forward_train(self, x, seq, batch, weights: MtWeights, y, stream=None):
        """y as forward() computes it, keeping the intermediates for backward_saved()."""
        self._backward_workspace(seq, batch, x.device)
        mt_layer_forward_train(self.handle, x.data_ptr(), seq, batch, weights, y.data_ptr(), self._stream(stream))
        return y

    def backward_saved(self, x, dy, seq, batch, weights: MtWeights, dx, grads: Dict[str, "object"], stream=None):
        """backward() without the recompute, from the intermediates of the last forward_train()."""
        self._backward_workspace(seq, batch, x.device)
        mt_layer_backward_saved(self.handle, x.data_ptr(), dy.data_ptr(), seq, batch, weights, dx.data_ptr(),
                                self._grads(grads), self._stream(stream))
        return dx

    def forward_host(self, x_host, seq, batch, weights: MtWeights, y_host, stream=None):
        self.workspace(seq, batch)
        mt_layer_forward_host(self.handle, x_host.data_ptr(), seq, batch, weights, y_host.data_ptr(),
                              self._stream(stream))
        return y_host

    def status(self):
        mt_layer_status(self.handle)

    def close(self):
        if self.handle:
            mt_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
