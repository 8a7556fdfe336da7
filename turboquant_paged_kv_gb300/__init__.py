"""TurboQuant paged KV cache for GB300: Python binding of libtq.

Functions carry the C ABI's names (``include/tq.h``) and only marshal
arguments: torch tensors become raw device pointers, the current CUDA stream
becomes the launch stream, and a non-OK status raises ``TQError``. Every step
of the store and the decode runs inside libtq's CUDA kernels; the first call
raises ImportError if the library is not built (there is no fallback path).
"""

from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import (PRESET_IDS, TQ_DEV_BLOCK_OUT_OF_RANGE, TQ_DEV_SEQ_TOO_LONG,  # noqa: F401
                   TQ_DECODE_NOALLOC_SCRATCH_BYTES, TQ_DEV_SLOT_OUT_OF_RANGE, TQ_DEV_TIMEOUT,
                   TQ_DTYPE_BF16, TQ_DTYPE_F16, TQ_DTYPE_F32, TQ_ERR_WORKSPACE_TOO_SMALL,
                   TQError, tq_codebook, tq_config, tq_layout, tq_prod_layout)



class _LazyLib:
    """libtq.so, loaded on first use (raises ImportError if it is not built)."""

    def __getattr__(self, name):
        return getattr(_abi.load(), name)


_LIB = _LazyLib()

_DTYPES = {torch.float16: TQ_DTYPE_F16, torch.bfloat16: TQ_DTYPE_BF16, torch.float32: TQ_DTYPE_F32}

__all__ = ["make_config", "tq_build_codebook", "tq_layout_for", "tq_store", "tq_decode", "tq_decode_append",
           "tq_decode_partials", "tq_decode_reduce", "tq_decode_noalloc", "tq_decode_workspace_size",
           "tq_dequant", "tq_prod_layout_for", "tq_prod_store", "tq_prod_scores_workspace_size",
           "tq_prod_scores", "tq_continue_workspace_size", "tq_continue",
           "tq_status_string",
           "tq_version", "TQError", "lib_path"]


def lib_path() -> str:
    return _abi.lib_path()


TQ_FLAG_INDICES_READY = 1   # include/tq.h: seq_lens / block_table not written by the previous kernel


def make_config(preset: str | int, num_q_heads: int, num_kv_heads: int, head_dim: int = 128,
                block_size: int = 16, partition_tokens: int = 0, flags: int = 0) -> tq_config:
    pid = PRESET_IDS[preset] if isinstance(preset, str) else int(preset)
    return tq_config(pid, head_dim, block_size, num_q_heads, num_kv_heads, partition_tokens, flags)


def tq_build_codebook(head_dim: int, bits: int) -> tq_codebook:
    cb = tq_codebook()
    _abi.check("tq_build_codebook", _LIB.tq_build_codebook(head_dim, bits, ctypes.byref(cb)))
    return cb


def tq_layout_for(cfg: tq_config) -> tq_layout:
    lay = tq_layout()
    _abi.check("tq_layout_for", _LIB.tq_layout_for(ctypes.byref(cfg), ctypes.byref(lay)))
    return lay


def tq_decode_workspace_size(cfg: tq_config, batch: int, max_seq_len: int) -> int:
    return int(_LIB.tq_decode_workspace_size(ctypes.byref(cfg), batch, max_seq_len))


def tq_status_string(status: int) -> str:
    return _LIB.tq_status_string(status).decode()


def tq_version() -> int:
    return int(_LIB.tq_version())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _cb(cb):
    return None if cb is None else ctypes.byref(cb)


def tq_store(cfg: tq_config, cb, key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor,
             cache: torch.Tensor, num_blocks: int | None = None, dev_status: torch.Tensor | None = None,
             stream=None) -> None:
    """key, value [N, n_kv, d] f16/bf16; slot_mapping [N] int64; cache uint8."""
    lay = tq_layout_for(cfg)
    if num_blocks is None:
        num_blocks = cache.numel() // lay.block_bytes
    _abi.check("tq_store", _LIB.tq_store(
        ctypes.byref(cfg), _cb(cb), _ptr(key), _ptr(value), _DTYPES[key.dtype], key.shape[0],
        _ptr(slot_mapping), _ptr(cache), num_blocks, _ptr(dev_status), _stream(stream)))


def tq_decode(cfg: tq_config, cb, q: torch.Tensor, cache: torch.Tensor, block_table: torch.Tensor,
              seq_lens: torch.Tensor, max_seq_len: int, out: torch.Tensor, workspace: torch.Tensor,
              scale: float = 0.0, num_blocks: int | None = None, dev_status: torch.Tensor | None = None,
              stream=None) -> None:
    """q [B, n_q, d]; block_table [B, stride] int32; seq_lens [B] int32; out [B, n_q, d]."""
    lay = tq_layout_for(cfg)
    if num_blocks is None:
        num_blocks = cache.numel() // lay.block_bytes
    _abi.check("tq_decode", _LIB.tq_decode(
        ctypes.byref(cfg), _cb(cb), _ptr(q), _DTYPES[q.dtype], _ptr(cache), num_blocks,
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), q.shape[0], max_seq_len, float(scale),
        _ptr(out), _DTYPES[out.dtype], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream(stream)))


def tq_decode_append(cfg: tq_config, cb, q: torch.Tensor, new_k: torch.Tensor, new_v: torch.Tensor,
                     cache: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                     out: torch.Tensor, workspace: torch.Tensor, scale: float = 0.0, num_blocks: int | None = None,
                     dev_status: torch.Tensor | None = None, stream=None) -> None:
    """One decode step with its new tokens: new_k, new_v [B, n_kv, d] (q's
    dtype) are stored at position seq_lens[b] - 1 of each sequence, then the
    decode runs over all seq_lens[b] positions (one split and one reduce
    launch, no store launch)."""
    lay = tq_layout_for(cfg)
    if num_blocks is None:
        num_blocks = cache.numel() // lay.block_bytes
    if new_k.dtype != q.dtype or new_v.dtype != q.dtype:
        raise ValueError("new_k and new_v must have q's dtype")
    _abi.check("tq_decode_append", _LIB.tq_decode_append(
        ctypes.byref(cfg), _cb(cb), _ptr(q), _DTYPES[q.dtype], _ptr(new_k), _ptr(new_v), _ptr(cache), num_blocks,
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), q.shape[0], max_seq_len, float(scale),
        _ptr(out), _DTYPES[out.dtype], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream(stream)))


def tq_decode_noalloc(cfg: tq_config, cb, q: torch.Tensor, cache: torch.Tensor, block_table: torch.Tensor,
                      seq_lens: torch.Tensor, max_seq_len: int, out: torch.Tensor, scale: float = 0.0,
                      num_blocks: int | None = None, dev_status: torch.Tensor | None = None,
                      stream=None) -> None:
    """tq_decode without a workspace argument: the library's fixed device array
    of TQ_DECODE_NOALLOC_SCRATCH_BYTES serves as workspace (calls whose kernels
    may overlap race on it; the first call on a device does the set-up)."""
    lay = tq_layout_for(cfg)
    if num_blocks is None:
        num_blocks = cache.numel() // lay.block_bytes
    _abi.check("tq_decode_noalloc", _LIB.tq_decode_noalloc(
        ctypes.byref(cfg), _cb(cb), _ptr(q), _DTYPES[q.dtype], _ptr(cache), num_blocks,
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), q.shape[0], max_seq_len, float(scale),
        _ptr(out), _DTYPES[out.dtype], _ptr(dev_status), _stream(stream)))


def tq_decode_partials(cfg: tq_config, cb, q: torch.Tensor, cache: torch.Tensor, block_table: torch.Tensor,
                       seq_lens: torch.Tensor, max_seq_len: int, workspace: torch.Tensor, scale: float = 0.0,
                       num_blocks: int | None = None, dev_status: torch.Tensor | None = None,
                       stream=None) -> None:
    lay = tq_layout_for(cfg)
    if num_blocks is None:
        num_blocks = cache.numel() // lay.block_bytes
    _abi.check("tq_decode_partials", _LIB.tq_decode_partials(
        ctypes.byref(cfg), _cb(cb), _ptr(q), _DTYPES[q.dtype], _ptr(cache), num_blocks,
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), q.shape[0], max_seq_len, float(scale),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)))


def tq_decode_reduce(cfg: tq_config, seq_lens: torch.Tensor, batch: int, max_seq_len: int, bt_stride: int,
                     out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    _abi.check("tq_decode_reduce", _LIB.tq_decode_reduce(
        ctypes.byref(cfg), _ptr(seq_lens), batch, max_seq_len, bt_stride, _ptr(out), _DTYPES[out.dtype],
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def tq_dequant(cfg: tq_config, cb, cache: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor,
               max_seq_len: int, key_out: torch.Tensor, value_out: torch.Tensor, num_blocks: int | None = None,
               dev_status: torch.Tensor | None = None, stream=None) -> None:
    """key_out, value_out [B, max_seq_len, n_kv, d] (f16, bf16 or f32), written in full."""
    if value_out.dtype != key_out.dtype:
        raise ValueError("key_out and value_out must have the same dtype")
    lay = tq_layout_for(cfg)
    if num_blocks is None:
        num_blocks = cache.numel() // lay.block_bytes
    _abi.check("tq_dequant", _LIB.tq_dequant(
        ctypes.byref(cfg), _cb(cb), _ptr(cache), num_blocks, _ptr(block_table), block_table.shape[1],
        _ptr(seq_lens), seq_lens.shape[0], max_seq_len, _ptr(key_out), _ptr(value_out),
        _DTYPES[key_out.dtype], _ptr(dev_status), _stream(stream)))


def tq_prod_layout_for(cfg: tq_config) -> tq_prod_layout:
    lay = tq_prod_layout()
    _abi.check("tq_prod_layout_for", _LIB.tq_prod_layout_for(ctypes.byref(cfg), ctypes.byref(lay)))
    return lay


def tq_prod_store(cfg: tq_config, cb, S: torch.Tensor, key: torch.Tensor, slot_mapping: torch.Tensor,
                  cache: torch.Tensor, num_blocks: int | None = None, dev_status: torch.Tensor | None = None,
                  stream=None) -> None:
    """TurboQuant_prod keys: key [N, n_kv, d] f16/bf16, S fp32 [d, d] (row i =
    projection i), slot_mapping [N] int64, cache uint8 (the prod key cache)."""
    if S.dtype != torch.float32:
        raise ValueError("S must be float32")
    lay = tq_prod_layout_for(cfg)
    if num_blocks is None:
        num_blocks = cache.numel() // lay.block_bytes
    _abi.check("tq_prod_store", _LIB.tq_prod_store(
        ctypes.byref(cfg), _cb(cb), _ptr(S), _ptr(key), _DTYPES[key.dtype], key.shape[0], _ptr(slot_mapping),
        _ptr(cache), num_blocks, _ptr(dev_status), _stream(stream)))


def tq_prod_scores_workspace_size(cfg: tq_config, batch: int) -> int:
    return int(_LIB.tq_prod_scores_workspace_size(ctypes.byref(cfg), batch))


def tq_prod_scores(cfg: tq_config, cb, S: torch.Tensor, q: torch.Tensor, cache: torch.Tensor,
                   block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int, scores: torch.Tensor,
                   workspace: torch.Tensor, scale: float = 0.0, num_blocks: int | None = None,
                   dev_status: torch.Tensor | None = None, stream=None) -> None:
    """scores fp32 [B, n_q, max_seq_len]: scale * the unbiased estimate of <q, k_p>."""
    if S.dtype != torch.float32 or scores.dtype != torch.float32:
        raise ValueError("S and scores must be float32")
    lay = tq_prod_layout_for(cfg)
    if num_blocks is None:
        num_blocks = cache.numel() // lay.block_bytes
    _abi.check("tq_prod_scores", _LIB.tq_prod_scores(
        ctypes.byref(cfg), _cb(cb), _ptr(S), _ptr(q), _DTYPES[q.dtype], _ptr(cache), num_blocks,
        _ptr(block_table), block_table.shape[1], _ptr(seq_lens), q.shape[0], max_seq_len, float(scale),
        _ptr(scores), _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(dev_status),
        _stream(stream)))


def tq_continue_workspace_size(cfg: tq_config, total_q: int, max_seq_len: int) -> int:
    return int(_LIB.tq_continue_workspace_size(ctypes.byref(cfg), total_q, max_seq_len))


def tq_continue(cfg: tq_config, cb, q: torch.Tensor, query_start: torch.Tensor, max_q_len: int,
                cache: torch.Tensor, block_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                out: torch.Tensor, workspace: torch.Tensor, scale: float = 0.0, num_blocks: int | None = None,
                dev_status: torch.Tensor | None = None, stream=None) -> None:
    """Causal attention of continuation chunks: q [total_q, n_q, d], query_start
    int32 [batch + 1], seq_lens int32 [batch] (lengths with the chunk),
    block_table int32 [batch, stride], out [total_q, n_q, d]."""
    lay = tq_layout_for(cfg)
    if num_blocks is None:
        num_blocks = cache.numel() // lay.block_bytes
    _abi.check("tq_continue", _LIB.tq_continue(
        ctypes.byref(cfg), _cb(cb), _ptr(q), _DTYPES[q.dtype], _ptr(query_start), seq_lens.shape[0], q.shape[0],
        max_q_len, _ptr(cache), num_blocks, _ptr(block_table), block_table.shape[1], _ptr(seq_lens), max_seq_len,
        float(scale), _ptr(out), _DTYPES[out.dtype], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(dev_status), _stream(stream)))
