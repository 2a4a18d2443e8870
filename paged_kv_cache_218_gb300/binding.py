"""Thin ctypes binding of libpa.so (include/pa.h).

Argument marshalling only: each function takes torch tensors, checks their
dtype / device / contiguity, and passes raw pointers, sizes and the current
CUDA stream to the C function of the same name.  Every step of the paged
attention path runs in the library's CUDA kernels; there is no fallback.
Importing this module raises if libpa.so has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"libpa.so not found at {_LIB_PATH}; build it first with "
        "`python -m paged_kv_cache_218_gb300.build` (or __graft_entry__.build())")
_lib = ctypes.CDLL(_LIB_PATH)

PA_OK = 0
PA_ERR_INVALID = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_CUDA = -3
PA_ERR_WORKSPACE = -4
PA_ERR_SCRATCH_LIMIT = -5
PA_DEVERR_BLOCK_ID = 1
PA_DEVERR_SEQ_LEN = 2
PA_DEVERR_SLOT = 4
PA_DEVERR_TIMEOUT = 8
PA_DEVERR_CHUNK = 16
PA_DEVERR_GROUP = 32

_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64
_F = ctypes.c_float
_S = ctypes.c_size_t

_SIGS = {
    "pa_status_string": ([_I], ctypes.c_char_p),
    "pa_version": ([], _I),
    "pa_reshape_and_cache": ([_P, _P, _L, _L, _P, _P, _P, _I, _I, _I, _I, _L, _P], _I),
    "pa_copy_blocks": ([_P, _P, _P, _I, _I, _I, _I, _L, _P], _I),
    "pa_decode_workspace_size": ([_I, _I, _I, _I, _I, _I, _I], _S),
    "pa_decode": ([_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _L, _F, _I, _P, _P, _S, _P], _I),
    "pa_merge_partials": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "pa_decode_append": ([_P, _P, _P, _P, _L, _L, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _L, _F,
                          _I, _P, _P, _S, _P], _I),
    "pa_decode_noalloc": ([_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _L, _F, _P, _P], _I),
    "pa_prefill_chunk": ([_P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _L, _F,
                          _P, _P], _I),
    "pa_validate_metadata": ([_P, _I, _P, _I, _P, _I, _P, _L, _I], _I),
    "pa_cascade_workspace_size": ([_I, _I, _I, _I, _I, _I, _I], _S),
    "pa_cascade_decode": ([_P, _P, _P, _P, _P, _I, _P, _I, _P, _I, _I, _P, _I, _P, _I, _I, _I, _I,
                           _L, _F, _I, _P, _P, _S, _P], _I),
    "pa_reshape_and_cache_fp8": ([_P, _P, _L, _L, _P, _P, _P, _P, _P, _I, _I, _I, _I, _L, _P], _I),
    "pa_copy_blocks_fp8": ([_P, _P, _P, _I, _I, _I, _I, _L, _P], _I),
    "pa_decode_fp8": ([_P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _L, _F, _I, _P, _P,
                       _S, _P], _I),
    "pa_device_error_flags": ([ctypes.POINTER(ctypes.c_uint), _I], _I),
    "pa_hybrid_workspace_size": ([_I, _I, _I, _I, _I, _I], _S),
    "pa_hybrid_attention": ([_P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _P,
                             _P, _P, _P, _I, _P, _I, _P,
                             _P, _P, _I, _I, _I, _I, _L, _F, _I, _P, _S, _P], _I),
    "pa_hybrid_attention_append": ([_P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _P,
                                    _P, _P, _P, _P, _P, _I, _P, _I, _P, _L, _L,
                                    _P, _P, _I, _I, _I, _I, _L, _F, _I, _P, _S, _P], _I),
    "pa_test_decode_stalled": ([_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _L, _F, _I, _P,
                                _S, ctypes.c_uint, _P], _I),
    "pa_test_prefill_stalled": ([_P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                 _L, _F, ctypes.c_uint, _P], _I),
}
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res

LIB_PATH = _LIB_PATH


class PAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {pa_status_string(status)} ({status})")
        self.status = status


def _check(fn: str, rc: int) -> None:
    if rc != PA_OK:
        raise PAError(fn, rc)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, dims: Optional[int] = None, contiguous=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {t.dim()}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def pa_status_string(status: int) -> str:
    return _lib.pa_status_string(int(status)).decode()


def pa_version() -> int:
    return int(_lib.pa_version())


def pa_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """Scatter key/value [T, Hkv, D] (row stride may exceed Hkv*D) into the pools."""
    _need(key, "key", torch.bfloat16, 3, contiguous=False)
    _need(value, "value", torch.bfloat16, 3, contiguous=False)
    for t, n in ((key, "key"), (value, "value")):
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} must be contiguous within a token")
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    T, Hkv, D = key.shape
    nb, bs = k_cache.shape[0], k_cache.shape[1]
    _check("pa_reshape_and_cache", _lib.pa_reshape_and_cache(
        _ptr(key), _ptr(value), key.stride(0), value.stride(0), _ptr(k_cache), _ptr(v_cache),
        _ptr(slot_mapping), T, Hkv, D, bs, nb, _stream(stream)))


def pa_copy_blocks(k_cache, v_cache, block_pairs, stream=None) -> None:
    """Copy whole blocks src -> dst of both pools; block_pairs int64 [n, 2]."""
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_pairs, "block_pairs", torch.int64, 2)
    nb, bs, Hkv, D = k_cache.shape
    _check("pa_copy_blocks", _lib.pa_copy_blocks(
        _ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), block_pairs.shape[0], Hkv, D, bs, nb,
        _stream(stream)))


def pa_reshape_and_cache_fp8(key, value, k_cache, v_cache, slot_mapping, k_scales, v_scales,
                             stream=None) -> None:
    """Quantizing scatter of bf16 key/value [T, Hkv, D] into uint8 E4M3 pools
    with per-kv-head fp32 scales: code = E4M3(x / scale[h])."""
    _need(key, "key", torch.bfloat16, 3, contiguous=False)
    _need(value, "value", torch.bfloat16, 3, contiguous=False)
    for t, n in ((key, "key"), (value, "value")):
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} must be contiguous within a token")
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    _need(k_scales, "k_scales", torch.float32, 1)
    _need(v_scales, "v_scales", torch.float32, 1)
    T, Hkv, D = key.shape
    nb, bs = k_cache.shape[0], k_cache.shape[1]
    _check("pa_reshape_and_cache_fp8", _lib.pa_reshape_and_cache_fp8(
        _ptr(key), _ptr(value), key.stride(0), value.stride(0), _ptr(k_cache), _ptr(v_cache),
        _ptr(slot_mapping), _ptr(k_scales), _ptr(v_scales), T, Hkv, D, bs, nb, _stream(stream)))


def pa_copy_blocks_fp8(k_cache, v_cache, block_pairs, stream=None) -> None:
    """Whole-block copies src -> dst of uint8 E4M3 pools; block_pairs int64 [n, 2]."""
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(block_pairs, "block_pairs", torch.int64, 2)
    nb, bs, Hkv, D = k_cache.shape
    _check("pa_copy_blocks_fp8", _lib.pa_copy_blocks_fp8(
        _ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), block_pairs.shape[0], Hkv, D, bs, nb,
        _stream(stream)))


def pa_decode_fp8(out, q, k_cache, v_cache, k_scales, v_scales, block_tables, seq_lens, scale,
                  partition_tokens=0, out_lse=None, workspace=None, stream=None) -> None:
    """pa_decode over uint8 E4M3 pools with per-kv-head fp32 scales."""
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.uint8, 4)
    _need(v_cache, "v_cache", torch.uint8, 4)
    _need(k_scales, "k_scales", torch.float32, 1)
    _need(v_scales, "v_scales", torch.float32, 1)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if out_lse is not None:
        _need(out_lse, "out_lse", torch.float32, 2)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_decode_fp8", _lib.pa_decode_fp8(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scales), _ptr(v_scales),
        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), S, Hq, Hkv, D, bs, nb,
        float(scale), int(partition_tokens), _ptr(out_lse), _ptr(workspace), ws_bytes,
        _stream(stream)))


def pa_cascade_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                              block_size=16, partition_tokens=0) -> int:
    return int(_lib.pa_cascade_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                              max_blocks_per_seq, block_size, partition_tokens))


def pa_cascade_decode(out, q, k_cache, v_cache, block_tables, seq_lens, group_offsets,
                      max_group_size, prefix_tables, shared_blocks, scale, partition_tokens=0,
                      out_lse=None, workspace=None, stream=None) -> None:
    """Decode with each group's shared prefix attended once for all its
    members, merged with their private suffixes (same result as pa_decode)."""
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(group_offsets, "group_offsets", torch.int32, 1)
    _need(prefix_tables, "prefix_tables", torch.int32, 2)
    _need(shared_blocks, "shared_blocks", torch.int32, 1)
    if out_lse is not None:
        _need(out_lse, "out_lse", torch.float32, 2)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_cascade_decode", _lib.pa_cascade_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), S, _ptr(group_offsets), group_offsets.shape[0] - 1,
        int(max_group_size), _ptr(prefix_tables), prefix_tables.shape[1], _ptr(shared_blocks),
        Hq, Hkv, D, bs, nb, float(scale), int(partition_tokens), _ptr(out_lse), _ptr(workspace),
        ws_bytes, _stream(stream)))


def pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                             block_size=16, partition_tokens=0) -> int:
    return int(_lib.pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, block_size, partition_tokens))


def alloc_workspace(nbytes: int, device) -> Optional[torch.Tensor]:
    """A zero-filled, 256-byte aligned workspace (torch allocations are)."""
    if nbytes == 0:
        return None
    return torch.zeros(nbytes, dtype=torch.uint8, device=device)


def pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, scale, partition_tokens=0,
              out_lse=None, workspace=None, stream=None) -> None:
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if out_lse is not None:
        _need(out_lse, "out_lse", torch.float32, 2)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_decode", _lib.pa_decode(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), S, Hq, Hkv, D, bs, nb, float(scale),
        int(partition_tokens), _ptr(out_lse), _ptr(workspace), ws_bytes, _stream(stream)))


def pa_decode_append(out, q, key, value, k_cache, v_cache, block_tables, seq_lens, scale,
                     partition_tokens=0, out_lse=None, workspace=None, stream=None) -> None:
    """One decode step with the slot scatter fused in: row s of key / value
    goes into the slot of position seq_lens[s] - 1, then the decode."""
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(key, "key", torch.bfloat16, 3, contiguous=False)
    _need(value, "value", torch.bfloat16, 3, contiguous=False)
    for t, n in ((key, "key"), (value, "value")):
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} must be contiguous within a token")
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if out_lse is not None:
        _need(out_lse, "out_lse", torch.float32, 2)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("pa_decode_append", _lib.pa_decode_append(
        _ptr(out), _ptr(q), _ptr(key), _ptr(value), key.stride(0), value.stride(0),
        _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), S, Hq, Hkv, D, bs, nb, float(scale),
        int(partition_tokens), _ptr(out_lse), _ptr(workspace), ws_bytes, _stream(stream)))


def pa_decode_noalloc(out, q, k_cache, v_cache, block_tables, seq_lens, scale, out_lse=None,
                      stream=None) -> None:
    """Balanced decode with the library's static scratch: no workspace, no
    allocation (for callers that cannot allocate device memory)."""
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if out_lse is not None:
        _need(out_lse, "out_lse", torch.float32, 2)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    _check("pa_decode_noalloc", _lib.pa_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), S, Hq, Hkv, D, bs, nb, float(scale),
        _ptr(out_lse), _stream(stream)))


def pa_merge_partials(out, part_out, part_lse, num_parts, out_lse=None, stream=None) -> None:
    _need(out, "out", torch.bfloat16, 3)
    _need(part_out, "part_out", torch.float32, 4)
    _need(part_lse, "part_lse", torch.float32, 3)
    _need(num_parts, "num_parts", torch.int32, 1)
    if out_lse is not None:
        _need(out_lse, "out_lse", torch.float32, 2)
    S, Hq, P, D = part_out.shape
    _check("pa_merge_partials", _lib.pa_merge_partials(
        _ptr(out), _ptr(out_lse), _ptr(part_out), _ptr(part_lse), _ptr(num_parts), S, Hq, D, P,
        _stream(stream)))


def pa_prefill_chunk(out, q, k_cache, v_cache, block_tables, cu_q_lens, q_start_pos, seq_lens,
                     max_q_len, scale, out_lse=None, stream=None) -> None:
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(cu_q_lens, "cu_q_lens", torch.int32, 1)
    _need(q_start_pos, "q_start_pos", torch.int32, 1)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    if out_lse is not None:
        _need(out_lse, "out_lse", torch.float32, 2)
    T, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    C = q_start_pos.shape[0]
    _check("pa_prefill_chunk", _lib.pa_prefill_chunk(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(cu_q_lens), _ptr(q_start_pos), _ptr(seq_lens), C, T,
        int(max_q_len), Hq, Hkv, D, bs, nb, float(scale), _ptr(out_lse), _stream(stream)))


def pa_hybrid_workspace_size(num_decode_seqs, num_q_heads, num_kv_heads, head_dim,
                             max_blocks_per_seq, block_size=16) -> int:
    return int(_lib.pa_hybrid_workspace_size(num_decode_seqs, num_q_heads, num_kv_heads, head_dim,
                                             max_blocks_per_seq, block_size))


def pa_hybrid_attention(out_chunk, q_chunk, chunk_block_tables, cu_q_lens, q_start_pos,
                        chunk_seq_lens, max_q_len, out_decode, q_decode, decode_block_tables,
                        decode_seq_lens, k_cache, v_cache, scale, workspace, chunk_sms=0,
                        chunk_lse=None, decode_lse=None, stream=None) -> None:
    """Prefill chunks and balanced decodes of one hybrid batch, co-scheduled."""
    _need(out_chunk, "out_chunk", torch.bfloat16, 3)
    _need(q_chunk, "q_chunk", torch.bfloat16, 3)
    _need(chunk_block_tables, "chunk_block_tables", torch.int32, 2)
    _need(cu_q_lens, "cu_q_lens", torch.int32, 1)
    _need(q_start_pos, "q_start_pos", torch.int32, 1)
    _need(chunk_seq_lens, "chunk_seq_lens", torch.int32, 1)
    _need(out_decode, "out_decode", torch.bfloat16, 3)
    _need(q_decode, "q_decode", torch.bfloat16, 3)
    _need(decode_block_tables, "decode_block_tables", torch.int32, 2)
    _need(decode_seq_lens, "decode_seq_lens", torch.int32, 1)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(workspace, "workspace", torch.uint8, 1)
    if chunk_lse is not None:
        _need(chunk_lse, "chunk_lse", torch.float32, 2)
    if decode_lse is not None:
        _need(decode_lse, "decode_lse", torch.float32, 2)
    T, Hq, D = q_chunk.shape
    nb, bs, Hkv, _ = k_cache.shape
    _check("pa_hybrid_attention", _lib.pa_hybrid_attention(
        _ptr(out_chunk), _ptr(q_chunk), _ptr(chunk_block_tables), chunk_block_tables.shape[1],
        _ptr(cu_q_lens), _ptr(q_start_pos), _ptr(chunk_seq_lens), q_start_pos.shape[0], T,
        int(max_q_len), _ptr(chunk_lse),
        _ptr(out_decode), _ptr(q_decode), _ptr(decode_block_tables), decode_block_tables.shape[1],
        _ptr(decode_seq_lens), q_decode.shape[0], _ptr(decode_lse),
        _ptr(k_cache), _ptr(v_cache), Hq, Hkv, D, bs, nb, float(scale), int(chunk_sms),
        _ptr(workspace), workspace.numel(), _stream(stream)))


def pa_hybrid_attention_append(out_chunk, q_chunk, key_chunk, value_chunk, chunk_block_tables,
                               cu_q_lens, q_start_pos, chunk_seq_lens, max_q_len, out_decode,
                               q_decode, key_decode, value_decode, decode_block_tables,
                               decode_seq_lens, k_cache, v_cache, scale, workspace, chunk_sms=0,
                               chunk_lse=None, decode_lse=None, stream=None) -> None:
    """One hybrid step with its slot scatter fused in: the chunk's and the
    decodes' new K/V rows go into their slots, then pa_hybrid_attention."""
    _need(out_chunk, "out_chunk", torch.bfloat16, 3)
    _need(q_chunk, "q_chunk", torch.bfloat16, 3)
    _need(chunk_block_tables, "chunk_block_tables", torch.int32, 2)
    _need(cu_q_lens, "cu_q_lens", torch.int32, 1)
    _need(q_start_pos, "q_start_pos", torch.int32, 1)
    _need(chunk_seq_lens, "chunk_seq_lens", torch.int32, 1)
    _need(out_decode, "out_decode", torch.bfloat16, 3)
    _need(q_decode, "q_decode", torch.bfloat16, 3)
    _need(decode_block_tables, "decode_block_tables", torch.int32, 2)
    _need(decode_seq_lens, "decode_seq_lens", torch.int32, 1)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    rows = [(key_chunk, "key_chunk"), (value_chunk, "value_chunk"), (key_decode, "key_decode"),
            (value_decode, "value_decode")]
    for t, n in rows:
        _need(t, n, torch.bfloat16, 3, contiguous=False)
        if t.stride(2) != 1 or t.stride(1) != t.shape[2]:
            raise ValueError(f"{n} must be contiguous within a token")
    if key_chunk.stride(0) != key_decode.stride(0) or value_chunk.stride(0) != value_decode.stride(0):
        raise ValueError("the chunk's and the decodes' rows must share their token strides")
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, 1)
    if chunk_lse is not None:
        _need(chunk_lse, "chunk_lse", torch.float32, 2)
    if decode_lse is not None:
        _need(decode_lse, "decode_lse", torch.float32, 2)
    T, Hq, D = q_chunk.shape
    nb, bs, Hkv, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel()
    _check("pa_hybrid_attention_append", _lib.pa_hybrid_attention_append(
        _ptr(out_chunk), _ptr(q_chunk), _ptr(key_chunk), _ptr(value_chunk),
        _ptr(chunk_block_tables), chunk_block_tables.shape[1], _ptr(cu_q_lens), _ptr(q_start_pos),
        _ptr(chunk_seq_lens), q_start_pos.shape[0], T, int(max_q_len), _ptr(chunk_lse),
        _ptr(out_decode), _ptr(q_decode), _ptr(key_decode), _ptr(value_decode),
        _ptr(decode_block_tables), decode_block_tables.shape[1], _ptr(decode_seq_lens),
        q_decode.shape[0], _ptr(decode_lse), key_chunk.stride(0), value_chunk.stride(0),
        _ptr(k_cache), _ptr(v_cache), Hq, Hkv, D, bs, nb, float(scale), int(chunk_sms),
        _ptr(workspace), ws_bytes, _stream(stream)))


def _host_ptr(a):
    import numpy as np
    return None if a is None else np.ascontiguousarray(a).ctypes.data_as(ctypes.c_void_p)


def pa_validate_metadata(block_tables, seq_lens, slot_mapping=None, refcount=None,
                         num_blocks=None, block_size=16) -> int:
    """Host-side metadata check on numpy arrays; returns the pa_status value."""
    import numpy as np
    bt = None if block_tables is None else np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    sm = None if slot_mapping is None else np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = None if refcount is None else np.ascontiguousarray(refcount, dtype=np.int32)
    mb = 0 if bt is None else bt.shape[1]
    return int(_lib.pa_validate_metadata(
        _host_ptr(bt), mb, _host_ptr(sl), sl.shape[0], _host_ptr(sm),
        0 if sm is None else sm.shape[0], _host_ptr(rc), int(num_blocks), int(block_size)))


def pa_device_error_flags(reset: bool = True) -> int:
    v = ctypes.c_uint(0)
    _check("pa_device_error_flags", _lib.pa_device_error_flags(ctypes.byref(v), int(reset)))
    return int(v.value)


# ---------------------------------------------------------------- failure-path tests

def pa_test_decode_stalled(out, q, k_cache, v_cache, block_tables, seq_lens, scale,
                           partition_tokens=0, workspace=None, wait_limit_us=1000,
                           stream=None) -> None:
    """One decode launch whose producer issues no load, every wait bounded by
    wait_limit_us: the kernel must report PA_DEVERR_TIMEOUT and return."""
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    _check("pa_test_decode_stalled", _lib.pa_test_decode_stalled(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), S, Hq, Hkv, D, bs, nb, float(scale),
        int(partition_tokens), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), int(wait_limit_us),
        _stream(stream)))


def pa_test_prefill_stalled(out, q, k_cache, v_cache, block_tables, cu_q_lens, q_start_pos,
                            seq_lens, max_q_len, scale, wait_limit_us=1000,
                            stream=None) -> None:
    """One prefill-chunk launch whose loaders issue no load, every wait
    bounded by wait_limit_us: the kernel must report PA_DEVERR_TIMEOUT."""
    _need(out, "out", torch.bfloat16, 3)
    _need(q, "q", torch.bfloat16, 3)
    _need(k_cache, "k_cache", torch.bfloat16, 4)
    _need(v_cache, "v_cache", torch.bfloat16, 4)
    _need(block_tables, "block_tables", torch.int32, 2)
    for t, name in ((cu_q_lens, "cu_q_lens"), (q_start_pos, "q_start_pos"),
                    (seq_lens, "seq_lens")):
        _need(t, name, torch.int32, 1)
    T, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    C = q_start_pos.shape[0]
    _check("pa_test_prefill_stalled", _lib.pa_test_prefill_stalled(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(cu_q_lens), _ptr(q_start_pos), _ptr(seq_lens), C, T,
        int(max_q_len), Hq, Hkv, D, bs, nb, float(scale), int(wait_limit_us), _stream(stream)))
