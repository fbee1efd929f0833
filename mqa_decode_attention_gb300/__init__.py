"""GB300 decode-step grouped-query attention: Python binding of libmqa_decode.so.

The three calls of the C ABI under the same names -- ``kv_append_rope``,
``gqa_decode_attention``, ``splitkv_combine`` -- plus layout builders and a
``decode_step`` that issues them in order. Everything here marshals torch
tensors (device memory, streams) into pointers and sizes; every step of the
computation runs in the CUDA kernels behind the C ABI. A non-OK status raises
``MqaError``.
"""

from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass

import torch

from . import _abi
from ._abi import (
    KVLayout,
    MQA_BF16,
    MQA_DEVERR_PAGE_RANGE,
    MQA_DEVERR_POS_RANGE,
    MQA_DEVERR_SEQ_LEN,
    MQA_DEVERR_TIMEOUT,
    MQA_DEVERR_U8_SCALE,
    MQA_F32,
    MQA_U8,
    MQA_FP8_E5M2,
    MQA_VARIANT_AUTO,
    MQA_VARIANT_CUDA_CORE,
    MQA_VARIANT_TENSOR_CORE,
)

__all__ = [
    "KVLayout",
    "MqaError",
    "DecodeBuffers",
    "layout_contiguous",
    "layout_paged",
    "kv_append_rope",
    "gqa_decode_attention",
    "splitkv_combine",
    "choose_splits",
    "workspace_size",
    "step_launches",
    "decode_step",
    "decode_step_multi",
    "kv_append_rope_multi",
    "gqa_decode_attention_multi",
    "gqa_prefill_attention",
    "prefill_step",
    "library",
    "MQA_VARIANT_AUTO",
    "MQA_VARIANT_CUDA_CORE",
    "MQA_VARIANT_TENSOR_CORE",
    "MQA_DEVERR_POS_RANGE",
    "MQA_DEVERR_PAGE_RANGE",
    "MQA_DEVERR_SEQ_LEN",
    "MQA_DEVERR_TIMEOUT",
    "MQA_DEVERR_U8_SCALE",
    "MQA_U8",
    "MQA_FP8_E5M2",
]


class MqaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = library()
        msg = lib.mqa_status_string(status).decode()
        if status == _abi.MQA_ERR_CUDA:
            msg += ": " + lib.mqa_last_cuda_error().decode()
        super().__init__(f"{fn} failed: {msg} (status {status})")
        self.status = status


def library() -> ctypes.CDLL:
    return _abi.load()


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return MQA_BF16
    if dt == torch.float32:
        return MQA_F32
    if dt == torch.uint8:
        return MQA_U8
    if dt == torch.float8_e5m2:
        return MQA_FP8_E5M2
    raise TypeError(f"unsupported dtype {dt}")


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def layout_contiguous(k_cache: torch.Tensor, v_cache: torch.Tensor, h_q: int, window: int = 0,
                      k_scale_zero: torch.Tensor | None = None, v_scale_zero: torch.Tensor | None = None) -> KVLayout:
    """Layout of a contiguous cache pair, each [batch, h_kv, capacity, head_dim]
    (bf16, fp32, fp8 e5m2, or uint8 codes with float32 [batch, h_kv, capacity,
    2] scale / zero-point pairs); window > 0 restricts the attention to the
    last `window` tokens."""
    assert k_cache.shape == v_cache.shape and k_cache.dim() == 4
    assert k_cache.is_contiguous() and v_cache.is_contiguous()
    B, h_kv, cap, d = k_cache.shape
    lay = KVLayout(_dtype_code(k_cache.dtype), B, h_q, h_kv, d, 0, k_cache.data_ptr(), v_cache.data_ptr(), cap,
                   0, 0, 0, window, None, _ptr(k_scale_zero), _ptr(v_scale_zero))
    lay._tensors = (k_cache, v_cache, k_scale_zero, v_scale_zero)  # the struct holds raw pointers: keep them alive
    return lay


def layout_paged(k_pool: torch.Tensor, v_pool: torch.Tensor, block_table: torch.Tensor, h_q: int,
                 window: int = 0, k_scale_zero: torch.Tensor | None = None,
                 v_scale_zero: torch.Tensor | None = None) -> KVLayout:
    """Layout of a paged pool pair, each [num_pages, h_kv, page_size, head_dim]
    (uint8 pools take [num_pages, h_kv, page_size, 2] scale / zero-point pairs),
    with an int32 block table [batch, max_pages_per_seq]; window > 0 restricts
    the attention to the last `window` tokens."""
    assert k_pool.shape == v_pool.shape and k_pool.dim() == 4
    assert block_table.dtype == torch.int32 and block_table.is_contiguous()
    n, h_kv, ps, d = k_pool.shape
    B, mp = block_table.shape
    lay = KVLayout(_dtype_code(k_pool.dtype), B, h_q, h_kv, d, 1, k_pool.data_ptr(), v_pool.data_ptr(), 0, ps, n,
                   mp, window, block_table.data_ptr(), _ptr(k_scale_zero), _ptr(v_scale_zero))
    lay._tensors = (k_pool, v_pool, block_table, k_scale_zero, v_scale_zero)  # keep the pointed-to tensors alive
    return lay


def kv_append_rope(layout: KVLayout, q_new, k_new, v_new, pos, rope_base: float, q_rot, err, stream=None) -> None:
    st = library().kv_append_rope(ctypes.byref(layout), _ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(pos),
                                  float(rope_base), _ptr(q_rot), _ptr(err), _stream(stream))
    if st != 0:
        raise MqaError("kv_append_rope", st)


def gqa_decode_attention(layout: KVLayout, q_rot, seq_lens, max_seq_len: int, scale: float, num_splits: int, out,
                         lse_out=None, workspace=None, variant: int = MQA_VARIANT_AUTO, err=None,
                         stream=None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = library().gqa_decode_attention(ctypes.byref(layout), _ptr(q_rot), _ptr(seq_lens), int(max_seq_len),
                                        float(scale), int(num_splits), _ptr(out), _dtype_code(out.dtype),
                                        _ptr(lse_out), _ptr(workspace), ws_bytes, int(variant), _ptr(err),
                                        _stream(stream))
    if st != 0:
        raise MqaError("gqa_decode_attention", st)


def splitkv_combine(o_part, lse_part, out, lse_out=None, stream=None) -> None:
    """o_part [batch, h_q, splits, d] fp32, lse_part [batch, h_q, splits] fp32."""
    B, hq, S, d = o_part.shape
    st = library().splitkv_combine(_ptr(o_part), _ptr(lse_part), B, hq, S, d, _ptr(out), _dtype_code(out.dtype),
                                   _ptr(lse_out), _stream(stream))
    if st != 0:
        raise MqaError("splitkv_combine", st)


def kv_append_rope_multi(layout: KVLayout, n_new: int, q_new, k_new, v_new, pos, rope_base: float, q_rot, err,
                         stream=None) -> None:
    """Append n_new tokens per sequence: q_new [B, n, H_q, d], k_new / v_new
    [B, n, H_kv, d]; token i at position pos[b] + i."""
    st = library().kv_append_rope_multi(ctypes.byref(layout), int(n_new), _ptr(q_new), _ptr(k_new), _ptr(v_new),
                                        _ptr(pos), float(rope_base), _ptr(q_rot), _ptr(err), _stream(stream))
    if st != 0:
        raise MqaError("kv_append_rope_multi", st)


def gqa_decode_attention_multi(layout: KVLayout, n_new: int, q_rot, seq_lens, max_seq_len: int, scale: float,
                               num_splits: int, out, lse_out=None, workspace=None, variant: int = MQA_VARIANT_AUTO,
                               err=None, stream=None) -> None:
    """Attention of the last n_new tokens of each sequence, causal among them:
    q_rot [B, n, H_q, d] fp32, out [B, n, H_q, d]."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = library().gqa_decode_attention_multi(ctypes.byref(layout), int(n_new), _ptr(q_rot), _ptr(seq_lens),
                                              int(max_seq_len), float(scale), int(num_splits), _ptr(out),
                                              _dtype_code(out.dtype), _ptr(lse_out), _ptr(workspace), ws_bytes,
                                              int(variant), _ptr(err), _stream(stream))
    if st != 0:
        raise MqaError("gqa_decode_attention_multi", st)


def choose_splits(layout: KVLayout, max_seq_len: int, variant: int = MQA_VARIANT_AUTO, n_new: int = 1) -> int:
    return int(library().mqa_choose_splits_multi(ctypes.byref(layout), int(n_new), int(max_seq_len), int(variant)))


def workspace_size(layout: KVLayout, max_seq_len: int, num_splits: int, variant: int = MQA_VARIANT_AUTO,
                   n_new: int = 1) -> int:
    return int(library().mqa_workspace_size_multi(ctypes.byref(layout), int(n_new), int(max_seq_len),
                                                  int(num_splits), int(variant)))


def step_launches(layout: KVLayout, max_seq_len: int, num_splits: int = 0, variant: int = MQA_VARIANT_AUTO,
                  n_new: int = 1) -> tuple[int, bool]:
    """(kernel launches of one decode step, whether the append runs inside the
    attention launch) through ``mqa_step_launches``; (-1, False) when the step
    would be refused."""
    fused = ctypes.c_int32(0)
    n = int(library().mqa_step_launches(ctypes.byref(layout), int(n_new), int(max_seq_len), int(num_splits),
                                        int(variant), ctypes.byref(fused)))
    return n, bool(fused.value)


@dataclass
class DecodeBuffers:
    """Caller-owned device buffers of one decode step (allocated by torch)."""

    q_rot: torch.Tensor
    out: torch.Tensor
    lse: torch.Tensor
    workspace: torch.Tensor | None
    err: torch.Tensor

    @staticmethod
    def allocate(layout: KVLayout, max_seq_len: int, num_splits: int = 0, variant: int = MQA_VARIANT_AUTO,
                 out_dtype: torch.dtype | None = None, device="cuda", n_new: int = 1) -> "DecodeBuffers":
        """Buffers for n_new query tokens per sequence: [B, H_q, d] (n_new = 1)
        or [B, n_new, H_q, d]."""
        B, hq, d = layout.batch, layout.h_q, layout.head_dim
        if out_dtype is None:
            out_dtype = torch.float32 if layout.cache_dtype == MQA_F32 else torch.bfloat16
        ws = workspace_size(layout, max_seq_len, num_splits, variant, n_new)
        rows = (B, hq) if n_new == 1 else (B, n_new, hq)
        return DecodeBuffers(
            q_rot=torch.empty(*rows, d, dtype=torch.float32, device=device),
            out=torch.empty(*rows, d, dtype=out_dtype, device=device),
            lse=torch.empty(*rows, dtype=torch.float32, device=device),
            workspace=torch.empty(ws, dtype=torch.uint8, device=device) if ws > 0 else None,
            err=torch.zeros(1, dtype=torch.int32, device=device),
        )


def decode_step(layout: KVLayout, q_new, k_new, v_new, pos, seq_lens, max_seq_len: int, bufs: DecodeBuffers,
                rope_base: float = 10000.0, scale: float | None = None, num_splits: int = 0,
                variant: int = MQA_VARIANT_AUTO, stream=None) -> torch.Tensor:
    """One decode step through ``mqa_decode_step``: append with RoPE at ``pos``
    (= seq_lens - 1), then attention over ``seq_lens`` tokens (and the combine
    when it splits). Returns ``bufs.out``."""
    if scale is None:
        scale = 1.0 / math.sqrt(layout.head_dim)
    ws = bufs.workspace
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = library().mqa_decode_step(ctypes.byref(layout), _ptr(q_new), _ptr(k_new), _ptr(v_new), _ptr(pos),
                                   _ptr(seq_lens), int(max_seq_len), float(rope_base), float(scale), int(num_splits),
                                   _ptr(bufs.q_rot), _ptr(bufs.out), _dtype_code(bufs.out.dtype), _ptr(bufs.lse),
                                   _ptr(ws), ws_bytes, int(variant), _ptr(bufs.err), _stream(stream))
    if st != 0:
        raise MqaError("mqa_decode_step", st)
    return bufs.out


def decode_step_multi(layout: KVLayout, n_new: int, q_new, k_new, v_new, pos, seq_lens, max_seq_len: int,
                      bufs: DecodeBuffers, rope_base: float = 10000.0, scale: float | None = None,
                      num_splits: int = 0, variant: int = MQA_VARIANT_AUTO, stream=None) -> torch.Tensor:
    """n_new new tokens per sequence through ``mqa_decode_step_multi`` (the
    verification pass of speculative decoding): tokens appended with RoPE at
    ``pos`` .. ``pos + n_new - 1`` (pos = seq_lens - n_new), then each attends
    causally. q_new [B, n, H_q, d], k_new / v_new [B, n, H_kv, d]; buffers from
    ``DecodeBuffers.allocate(..., n_new=n_new)``. Returns ``bufs.out``."""
    if scale is None:
        scale = 1.0 / math.sqrt(layout.head_dim)
    ws = bufs.workspace
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    st = library().mqa_decode_step_multi(ctypes.byref(layout), int(n_new), _ptr(q_new), _ptr(k_new), _ptr(v_new),
                                         _ptr(pos), _ptr(seq_lens), int(max_seq_len), float(rope_base), float(scale),
                                         int(num_splits), _ptr(bufs.q_rot), _ptr(bufs.out),
                                         _dtype_code(bufs.out.dtype), _ptr(bufs.lse), _ptr(ws), ws_bytes,
                                         int(variant), _ptr(bufs.err), _stream(stream))
    if st != 0:
        raise MqaError("mqa_decode_step_multi", st)
    return bufs.out


def gqa_prefill_attention(layout: KVLayout, n_new: int, q_rot, seq_lens, max_seq_len: int, scale: float, out,
                          lse_out=None, err=None, stream=None) -> None:
    """Causal attention of the last n_new tokens of every sequence on the
    tensor-memory tensor cores: q_rot [B, n, H_q, 128] fp32, out [B, n, H_q, 128]."""
    st = library().gqa_prefill_attention(ctypes.byref(layout), int(n_new), _ptr(q_rot), _ptr(seq_lens),
                                         int(max_seq_len), float(scale), _ptr(out), _dtype_code(out.dtype),
                                         _ptr(lse_out), _ptr(err), _stream(stream))
    if st != 0:
        raise MqaError("gqa_prefill_attention", st)


def prefill_step(layout: KVLayout, n_new: int, q_new, k_new, v_new, pos, seq_lens, max_seq_len: int,
                 bufs: DecodeBuffers, rope_base: float = 10000.0, scale: float | None = None,
                 stream=None) -> torch.Tensor:
    """The prompt's n_new tokens through ``mqa_prefill_step``: appended with RoPE
    at pos .. pos + n_new - 1 (pos = seq_lens - n_new), then causal attention.
    Buffers from ``DecodeBuffers.allocate(..., n_new=n_new, num_splits=1)``."""
    if scale is None:
        scale = 1.0 / math.sqrt(layout.head_dim)
    st = library().mqa_prefill_step(ctypes.byref(layout), int(n_new), _ptr(q_new), _ptr(k_new), _ptr(v_new),
                                    _ptr(pos), _ptr(seq_lens), int(max_seq_len), float(rope_base), float(scale),
                                    _ptr(bufs.q_rot), _ptr(bufs.out), _dtype_code(bufs.out.dtype), _ptr(bufs.lse),
                                    _ptr(bufs.err), _stream(stream))
    if st != 0:
        raise MqaError("mqa_prefill_step", st)
    return bufs.out
