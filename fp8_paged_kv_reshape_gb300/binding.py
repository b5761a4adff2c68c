"""Thin Python binding over the kvfp8 C ABI (include/kvfp8.h).

Argument marshalling only: every step of the path runs in libkvfp8.so's CUDA kernels.
PyTorch supplies device memory and the current stream.  There is no CPU or eager
fallback: if the library is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

OK = 0
ERR_NULL, ERR_SHAPE, ERR_DTYPE, ERR_SCALE, ERR_ALIGN, ERR_WORKSPACE, ERR_CUDA, ERR_UNSUPPORTED = \
    range(1, 9)
BF16 = 0
F32 = 1
CACHE_E4M3 = 0
CACHE_BF16 = 1

DEV_BAD_SCALE = 1 << 0
DEV_BAD_SLOT = 1 << 1
DEV_BAD_BLOCK = 1 << 2
DEV_TIMEOUT = 1 << 3

# The functions include/kvfp8.h declares; the library must export every one.
ABI_FUNCTIONS = (
    "kvfp8_reshape_and_cache",
    "kvfp8_rope_reshape_and_cache",
    "kvfp8_paged_decode_workspace_size",
    "kvfp8_paged_decode_attention",
    "kvfp8_paged_decode_attention_noalloc",
    "kvfp8_paged_attention_multi",
    "kvfp8_paged_attention_multi_workspace_size",
    "kvfp8_reshape_and_cache_mixed",
    "kvfp8_paged_decode_attention_mixed",
    "kvfp8_paged_attention_multi_mixed",
    "kvfp8_dequant",
    "kvfp8_check_scale_host",
    "kvfp8_status_string",
)


class KvFp8Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(
            f"kvfp8 CUDA library not built ({path} missing): run "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    lib.kvfp8_reshape_and_cache.argtypes = [P, P, ctypes.c_int, i64, i64, i64, P, P, i32, i32, i32,
                                            i32, P, P, P, ctypes.c_int, P, P]
    lib.kvfp8_reshape_and_cache.restype = ctypes.c_int
    lib.kvfp8_rope_reshape_and_cache.argtypes = [P, P, ctypes.c_int, i64, i64, i64, P, P, i32, i32,
                                                 i32, i32, P, P, P, i64, i32, i32, P, P,
                                                 ctypes.c_int, P, P]
    lib.kvfp8_rope_reshape_and_cache.restype = ctypes.c_int
    lib.kvfp8_paged_decode_workspace_size.argtypes = [i32, i32, i32]
    lib.kvfp8_paged_decode_workspace_size.restype = sz
    lib.kvfp8_paged_decode_attention.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                                 i32, f32, P, P, ctypes.c_int, P, sz, P, P]
    lib.kvfp8_paged_decode_attention.restype = ctypes.c_int
    lib.kvfp8_paged_decode_attention_noalloc.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                                         i32, i32, f32, P, P, ctypes.c_int, P, P]
    lib.kvfp8_paged_decode_attention_noalloc.restype = ctypes.c_int
    lib.kvfp8_paged_attention_multi.argtypes = [P, P, P, i32, i32, P, P, P, i32, P, i32, i32, i32,
                                                i32, i32, i32, f32, P, P, ctypes.c_int, P, sz, P,
                                                P]
    lib.kvfp8_paged_attention_multi.restype = ctypes.c_int
    lib.kvfp8_paged_attention_multi_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.kvfp8_paged_attention_multi_workspace_size.restype = sz
    lib.kvfp8_reshape_and_cache_mixed.argtypes = [P, P, ctypes.c_int, i64, i64, i64, P,
                                                  ctypes.c_int, P, ctypes.c_int, i32, i32, i32,
                                                  i32, P, P, P, ctypes.c_int, P, P]
    lib.kvfp8_reshape_and_cache_mixed.restype = ctypes.c_int
    lib.kvfp8_paged_decode_attention_mixed.argtypes = [P, P, P, ctypes.c_int, P, ctypes.c_int, P,
                                                       i32, P, i32, i32, i32, i32, i32, i32, f32,
                                                       P, P, ctypes.c_int, P, sz, P, P]
    lib.kvfp8_paged_decode_attention_mixed.restype = ctypes.c_int
    lib.kvfp8_paged_attention_multi_mixed.argtypes = [P, P, P, i32, i32, P, ctypes.c_int, P,
                                                      ctypes.c_int, P, i32, P, i32, i32, i32,
                                                      i32, i32, i32, f32, P, P, ctypes.c_int, P,
                                                      sz, P, P]
    lib.kvfp8_paged_attention_multi_mixed.restype = ctypes.c_int
    lib.kvfp8_dequant.argtypes = [P, ctypes.c_int, P, i64, P, ctypes.c_int, P]
    lib.kvfp8_dequant.restype = ctypes.c_int
    lib.kvfp8_check_scale_host.argtypes = [f32]
    lib.kvfp8_check_scale_host.restype = ctypes.c_int
    lib.kvfp8_status_string.argtypes = [ctypes.c_int]
    lib.kvfp8_status_string.restype = ctypes.c_char_p
    return lib


LIB = _load()
LIB_PATH = _build.LIB


def status_string(status: int) -> str:
    return LIB.kvfp8_status_string(int(status)).decode()


def check_scale_host(s: float) -> int:
    return int(LIB.kvfp8_check_scale_host(float(s)))


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _scale_args(k_scale, v_scale):
    dt = None
    for s in (k_scale, v_scale):
        if s is None:
            continue
        if not (isinstance(s, torch.Tensor) and s.numel() == 1 and s.is_cuda
                and s.dtype in (torch.float32, torch.bfloat16)):
            raise TypeError("scales must be 1-element CUDA float32 or bfloat16 tensors (or None)")
        if dt is not None and s.dtype != dt:
            raise TypeError("k_scale and v_scale must share one dtype")
        dt = s.dtype
    return (BF16 if dt == torch.bfloat16 else F32)


def _check(rc: int, what: str):
    if rc != OK:
        raise KvFp8Error(rc, what)


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                      value_cache: torch.Tensor, slot_mapping: torch.Tensor,
                      k_scale: torch.Tensor | None = None, v_scale: torch.Tensor | None = None,
                      status: torch.Tensor | None = None, stream=None) -> None:
    """kvfp8_reshape_and_cache on torch tensors.

    key/value: [num_tokens, n_kv, head_dim] bf16 or float32 (same dtype); the token
    stride may exceed n_kv*head_dim (a slice of a fused QKV), the inner two dims must be
    dense.  Caches: uint8 [num_blocks, block_size, n_kv, head_dim], contiguous.
    slot_mapping: int64 [num_tokens] (-1 = padding).  status: int32 [1] or None.
    """
    if key.dtype != value.dtype or key.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("key and value must share one dtype, bfloat16 or float32")
    if key.dim() != 3 or value.shape != key.shape:
        raise ValueError("key/value must be [num_tokens, n_kv, head_dim] with equal shapes")
    n, n_kv, hd = key.shape
    for t in (key, value):
        if t.stride(2) != 1 or t.stride(1) != hd:
            raise ValueError("key/value inner dims [n_kv, head_dim] must be dense")
    if key_cache.dtype != torch.uint8 or value_cache.dtype != torch.uint8:
        raise TypeError("caches must be uint8")
    if key_cache.shape != value_cache.shape or key_cache.dim() != 4 or \
            tuple(key_cache.shape[2:]) != (n_kv, hd):
        raise ValueError("caches must be [num_blocks, block_size, n_kv, head_dim]")
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != n or \
            not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous int64 [num_tokens] tensor")
    sdt = _scale_args(k_scale, v_scale)
    rc = LIB.kvfp8_reshape_and_cache(
        _ptr(key), _ptr(value), F32 if key.dtype == torch.float32 else BF16,
        key.stride(0) if n > 0 else n_kv * hd, value.stride(0) if n > 0 else n_kv * hd, n,
        _ptr(key_cache), _ptr(value_cache), key_cache.shape[0], key_cache.shape[1], n_kv, hd,
        _ptr(slot_mapping), _ptr(k_scale), _ptr(v_scale), sdt, _ptr(status), _stream(stream))
    _check(rc, "kvfp8_reshape_and_cache")


def rope_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                           value_cache: torch.Tensor, slot_mapping: torch.Tensor,
                           positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                           is_neox: bool = True, k_scale: torch.Tensor | None = None,
                           v_scale: torch.Tensor | None = None,
                           status: torch.Tensor | None = None, stream=None) -> None:
    """kvfp8_rope_reshape_and_cache: rope on K (table cos_sin_cache float32 [max_pos, rot]),
    then the store of reshape_and_cache; positions int64 [num_tokens]."""
    if key.dtype != value.dtype or key.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("key and value must share one dtype, bfloat16 or float32")
    if key.dim() != 3 or value.shape != key.shape:
        raise ValueError("key/value must be [num_tokens, n_kv, head_dim] with equal shapes")
    n, n_kv, hd = key.shape
    for t in (key, value):
        if t.stride(2) != 1 or t.stride(1) != hd:
            raise ValueError("key/value inner dims [n_kv, head_dim] must be dense")
    if key_cache.dtype != torch.uint8 or key_cache.shape != value_cache.shape or \
            key_cache.dim() != 4 or tuple(key_cache.shape[2:]) != (n_kv, hd) or \
            not (key_cache.is_contiguous() and value_cache.is_contiguous()):
        raise ValueError("caches must be contiguous uint8 [num_blocks, block_size, n_kv, head_dim]")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != n or \
            positions.dtype != torch.int64 or positions.numel() != n:
        raise ValueError("slot_mapping and positions must be int64 [num_tokens]")
    if cos_sin_cache.dtype != torch.float32 or cos_sin_cache.dim() != 2 or \
            not cos_sin_cache.is_contiguous():
        raise ValueError("cos_sin_cache must be a contiguous float32 [max_pos, rot_dim] tensor")
    sdt = _scale_args(k_scale, v_scale)
    rc = LIB.kvfp8_rope_reshape_and_cache(
        _ptr(key), _ptr(value), F32 if key.dtype == torch.float32 else BF16,
        key.stride(0) if n > 0 else n_kv * hd, value.stride(0) if n > 0 else n_kv * hd, n,
        _ptr(key_cache), _ptr(value_cache), key_cache.shape[0], key_cache.shape[1], n_kv, hd,
        _ptr(slot_mapping), _ptr(positions), _ptr(cos_sin_cache), cos_sin_cache.shape[0],
        cos_sin_cache.shape[1], 1 if is_neox else 0, _ptr(k_scale), _ptr(v_scale), sdt,
        _ptr(status), _stream(stream))
    _check(rc, "kvfp8_rope_reshape_and_cache")


def paged_decode_workspace_size(num_seqs: int, n_q: int, head_dim: int) -> int:
    return int(LIB.kvfp8_paged_decode_workspace_size(num_seqs, n_q, head_dim))


def _check_tables(block_tables: torch.Tensor, seq_lens: torch.Tensor, num_seqs: int):
    """block_tables int32 [num_seqs, max_blocks] and seq_lens int32 [num_seqs], contiguous:
    the kernels index both for every sequence, so a short or int64 tensor would be read out
    of bounds (or as the halves of 64-bit words)."""
    if block_tables.dtype != torch.int32 or block_tables.dim() != 2 or \
            block_tables.shape[0] != num_seqs or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous int32 [num_seqs, max_blocks] tensor")
    if seq_lens.dtype != torch.int32 or seq_lens.numel() != num_seqs or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be a contiguous int32 [num_seqs] tensor")


def _check_decode_args(query: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                       block_tables: torch.Tensor, seq_lens: torch.Tensor,
                       out: torch.Tensor | None):
    """The argument checks every single-query decode wrapper makes; returns
    (num_seqs, n_q, head_dim, num_blocks, block_size, n_kv)."""
    if query.dtype != torch.bfloat16 or query.dim() != 3 or not query.is_contiguous():
        raise ValueError("query must be a contiguous bf16 [num_seqs, n_q, head_dim] tensor")
    num_seqs, n_q, hd = query.shape
    if key_cache.dtype != torch.uint8 or key_cache.shape != value_cache.shape or \
            key_cache.dim() != 4 or key_cache.shape[3] != hd:
        raise ValueError("caches must be uint8 [num_blocks, block_size, n_kv, head_dim]")
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    num_blocks, bs, n_kv, _ = key_cache.shape
    _check_tables(block_tables, seq_lens, num_seqs)
    if out is not None and (out.dtype != torch.bfloat16 or out.shape != query.shape or
                            not out.is_contiguous()):
        raise ValueError("out must be a contiguous bf16 tensor shaped like query")
    return num_seqs, n_q, hd, num_blocks, bs, n_kv


def paged_decode_attention(query: torch.Tensor, key_cache: torch.Tensor, value_cache: torch.Tensor,
                           block_tables: torch.Tensor, seq_lens: torch.Tensor,
                           k_scale: torch.Tensor | None = None, v_scale: torch.Tensor | None = None,
                           sm_scale: float = 0.0, out: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None,
                           status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kvfp8_paged_decode_attention on torch tensors; returns out (bf16 [num_seqs, n_q, hd])."""
    num_seqs, n_q, hd, num_blocks, bs, n_kv = _check_decode_args(
        query, key_cache, value_cache, block_tables, seq_lens, out)
    if out is None:
        out = torch.empty_like(query)
    need = paged_decode_workspace_size(num_seqs, n_q, hd)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=query.device)
    sdt = _scale_args(k_scale, v_scale)
    rc = LIB.kvfp8_paged_decode_attention(
        _ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), num_seqs, n_q, n_kv, hd, bs, num_blocks,
        float(sm_scale), _ptr(k_scale), _ptr(v_scale), sdt, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream))
    _check(rc, "kvfp8_paged_decode_attention")
    return out


def paged_attention_multi_workspace_size(num_seqs: int, n_q: int, n_kv: int, head_dim: int,
                                         max_query_len: int) -> int:
    return int(LIB.kvfp8_paged_attention_multi_workspace_size(num_seqs, n_q, n_kv, head_dim,
                                                              max_query_len))


def paged_attention_multi(query: torch.Tensor, query_start_loc: torch.Tensor, max_query_len: int,
                          key_cache: torch.Tensor, value_cache: torch.Tensor,
                          block_tables: torch.Tensor, seq_lens: torch.Tensor,
                          k_scale: torch.Tensor | None = None, v_scale: torch.Tensor | None = None,
                          sm_scale: float = 0.0, out: torch.Tensor | None = None,
                          workspace: torch.Tensor | None = None,
                          status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kvfp8_paged_attention_multi: causal multi-query attention; query/out bf16
    [num_query_rows, n_q, head_dim], sequence b's rows from query_start_loc[b] (int32
    [num_seqs + 1])."""
    if query.dtype != torch.bfloat16 or query.dim() != 3 or not query.is_contiguous():
        raise ValueError("query must be a contiguous bf16 [rows, n_q, head_dim] tensor")
    rows, n_q, hd = query.shape
    num_seqs = seq_lens.numel()
    if query_start_loc.dtype != torch.int32 or query_start_loc.numel() != num_seqs + 1 or \
            not query_start_loc.is_contiguous():
        raise ValueError("query_start_loc must be a contiguous int32 [num_seqs + 1] tensor")
    if key_cache.dtype != torch.uint8 or key_cache.shape != value_cache.shape or \
            key_cache.dim() != 4 or key_cache.shape[3] != hd:
        raise ValueError("caches must be uint8 [num_blocks, block_size, n_kv, head_dim]")
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    num_blocks, bs, n_kv, _ = key_cache.shape
    _check_tables(block_tables, seq_lens, num_seqs)
    if out is None:
        out = torch.empty_like(query)
    need = paged_attention_multi_workspace_size(num_seqs, n_q, n_kv, hd, max_query_len)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    sdt = _scale_args(k_scale, v_scale)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = LIB.kvfp8_paged_attention_multi(
        _ptr(out), _ptr(query), _ptr(query_start_loc), rows, max_query_len, _ptr(key_cache),
        _ptr(value_cache), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), num_seqs,
        n_q, n_kv, hd, bs, num_blocks, float(sm_scale), _ptr(k_scale), _ptr(v_scale), sdt,
        _ptr(workspace), ws_bytes, _ptr(status), _stream(stream))
    _check(rc, "kvfp8_paged_attention_multi")
    return out


def paged_decode_attention_noalloc(query: torch.Tensor, key_cache: torch.Tensor,
                                   value_cache: torch.Tensor, block_tables: torch.Tensor,
                                   seq_lens: torch.Tensor, k_scale: torch.Tensor | None = None,
                                   v_scale: torch.Tensor | None = None, sm_scale: float = 0.0,
                                   out: torch.Tensor | None = None,
                                   status: torch.Tensor | None = None,
                                   stream=None) -> torch.Tensor:
    """kvfp8_paged_decode_attention_noalloc: the same call with the library's fixed device
    scratch instead of a workspace, for callers that cannot allocate device memory.  Pass
    ``out`` to keep the call free of allocations on the Python side too.  The arguments are
    checked exactly as paged_decode_attention checks them."""
    num_seqs, n_q, hd, num_blocks, bs, n_kv = _check_decode_args(
        query, key_cache, value_cache, block_tables, seq_lens, out)
    if out is None:
        out = torch.empty_like(query)
    sdt = _scale_args(k_scale, v_scale)
    rc = LIB.kvfp8_paged_decode_attention_noalloc(
        _ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), num_seqs, n_q, n_kv, hd, bs, num_blocks,
        float(sm_scale), _ptr(k_scale), _ptr(v_scale), sdt, _ptr(status), _stream(stream))
    _check(rc, "kvfp8_paged_decode_attention_noalloc")
    return out


def _cache_kind(t: torch.Tensor) -> int:
    if t.dtype == torch.uint8:
        return CACHE_E4M3
    if t.dtype == torch.bfloat16:
        return CACHE_BF16
    raise TypeError("a cache is uint8 (E4M3 codes) or bfloat16")


def _check_mixed_caches(key_cache: torch.Tensor, value_cache: torch.Tensor):
    if key_cache.dim() != 4 or value_cache.shape != key_cache.shape:
        raise ValueError("caches must be [num_blocks, block_size, n_kv, head_dim]")
    if not (key_cache.is_contiguous() and value_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    return _cache_kind(key_cache), _cache_kind(value_cache)


def reshape_and_cache_mixed(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                            value_cache: torch.Tensor, slot_mapping: torch.Tensor,
                            k_scale: torch.Tensor | None = None,
                            v_scale: torch.Tensor | None = None,
                            status: torch.Tensor | None = None, stream=None) -> None:
    """kvfp8_reshape_and_cache_mixed: each cache's dtype picks its side's format (uint8 =
    E4M3 with that side's scale, bfloat16 = the value rounded to bf16, no scale)."""
    if key.dtype != value.dtype or key.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("key and value must share one dtype, bfloat16 or float32")
    if key.dim() != 3 or value.shape != key.shape:
        raise ValueError("key/value must be [num_tokens, n_kv, head_dim] with equal shapes")
    n, n_kv, hd = key.shape
    for t in (key, value):
        if t.stride(2) != 1 or t.stride(1) != hd:
            raise ValueError("key/value inner dims [n_kv, head_dim] must be dense")
    kk, vk = _check_mixed_caches(key_cache, value_cache)
    if tuple(key_cache.shape[2:]) != (n_kv, hd):
        raise ValueError("caches must be [num_blocks, block_size, n_kv, head_dim]")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != n or \
            not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous int64 [num_tokens] tensor")
    sdt = _scale_args(k_scale, v_scale)
    rc = LIB.kvfp8_reshape_and_cache_mixed(
        _ptr(key), _ptr(value), F32 if key.dtype == torch.float32 else BF16,
        key.stride(0) if n > 0 else n_kv * hd, value.stride(0) if n > 0 else n_kv * hd, n,
        _ptr(key_cache), kk, _ptr(value_cache), vk, key_cache.shape[0], key_cache.shape[1], n_kv,
        hd, _ptr(slot_mapping), _ptr(k_scale), _ptr(v_scale), sdt, _ptr(status), _stream(stream))
    _check(rc, "kvfp8_reshape_and_cache_mixed")


def paged_decode_attention_mixed(query: torch.Tensor, key_cache: torch.Tensor,
                                 value_cache: torch.Tensor, block_tables: torch.Tensor,
                                 seq_lens: torch.Tensor, k_scale: torch.Tensor | None = None,
                                 v_scale: torch.Tensor | None = None, sm_scale: float = 0.0,
                                 out: torch.Tensor | None = None,
                                 workspace: torch.Tensor | None = None,
                                 status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kvfp8_paged_decode_attention_mixed: decode attention where each cache's dtype picks
    its side's format (uint8 = E4M3, scaled; bfloat16 = unscaled)."""
    if query.dtype != torch.bfloat16 or query.dim() != 3 or not query.is_contiguous():
        raise ValueError("query must be a contiguous bf16 [num_seqs, n_q, head_dim] tensor")
    num_seqs, n_q, hd = query.shape
    kk, vk = _check_mixed_caches(key_cache, value_cache)
    if key_cache.shape[3] != hd:
        raise ValueError("caches must be [num_blocks, block_size, n_kv, head_dim]")
    num_blocks, bs, n_kv, _ = key_cache.shape
    _check_tables(block_tables, seq_lens, num_seqs)
    if out is None:
        out = torch.empty_like(query)
    need = paged_decode_workspace_size(num_seqs, n_q, hd)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=query.device)
    sdt = _scale_args(k_scale, v_scale)
    rc = LIB.kvfp8_paged_decode_attention_mixed(
        _ptr(out), _ptr(query), _ptr(key_cache), kk, _ptr(value_cache), vk, _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), num_seqs, n_q, n_kv, hd, bs, num_blocks,
        float(sm_scale), _ptr(k_scale), _ptr(v_scale), sdt, _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream))
    _check(rc, "kvfp8_paged_decode_attention_mixed")
    return out


def paged_attention_multi_mixed(query: torch.Tensor, query_start_loc: torch.Tensor,
                                max_query_len: int, key_cache: torch.Tensor,
                                value_cache: torch.Tensor, block_tables: torch.Tensor,
                                seq_lens: torch.Tensor, k_scale: torch.Tensor | None = None,
                                v_scale: torch.Tensor | None = None, sm_scale: float = 0.0,
                                out: torch.Tensor | None = None,
                                workspace: torch.Tensor | None = None,
                                status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """kvfp8_paged_attention_multi_mixed: causal multi-query attention where each cache's
    dtype picks its side's format (uint8 = E4M3, scaled; bfloat16 = unscaled)."""
    if query.dtype != torch.bfloat16 or query.dim() != 3 or not query.is_contiguous():
        raise ValueError("query must be a contiguous bf16 [rows, n_q, head_dim] tensor")
    rows, n_q, hd = query.shape
    num_seqs = seq_lens.numel()
    if query_start_loc.dtype != torch.int32 or query_start_loc.numel() != num_seqs + 1 or \
            not query_start_loc.is_contiguous():
        raise ValueError("query_start_loc must be a contiguous int32 [num_seqs + 1] tensor")
    kk, vk = _check_mixed_caches(key_cache, value_cache)
    if key_cache.shape[3] != hd:
        raise ValueError("caches must be [num_blocks, block_size, n_kv, head_dim]")
    num_blocks, bs, n_kv, _ = key_cache.shape
    _check_tables(block_tables, seq_lens, num_seqs)
    if out is None:
        out = torch.empty_like(query)
    need = paged_attention_multi_workspace_size(num_seqs, n_q, n_kv, hd, max_query_len)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=query.device)
    sdt = _scale_args(k_scale, v_scale)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = LIB.kvfp8_paged_attention_multi_mixed(
        _ptr(out), _ptr(query), _ptr(query_start_loc), rows, max_query_len, _ptr(key_cache), kk,
        _ptr(value_cache), vk, _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
        num_seqs, n_q, n_kv, hd, bs, num_blocks, float(sm_scale), _ptr(k_scale), _ptr(v_scale),
        sdt, _ptr(workspace), ws_bytes, _ptr(status), _stream(stream))
    _check(rc, "kvfp8_paged_attention_multi_mixed")
    return out


def dequant(src: torch.Tensor, dst_dtype: torch.dtype = torch.float32,
            scale: torch.Tensor | None = None, out: torch.Tensor | None = None,
            stream=None) -> torch.Tensor:
    """kvfp8_dequant: uint8 E4M3 codes -> scale * value as float32 or bfloat16 (same shape)."""
    if src.dtype != torch.uint8 or not src.is_contiguous():
        raise ValueError("src must be a contiguous uint8 tensor")
    if dst_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("dst_dtype must be float32 or bfloat16")
    if out is None:
        out = torch.empty(src.shape, dtype=dst_dtype, device=src.device)
    sdt = _scale_args(scale, None)
    rc = LIB.kvfp8_dequant(_ptr(out), BF16 if dst_dtype == torch.bfloat16 else F32, _ptr(src),
                           src.numel(), _ptr(scale), sdt, _stream(stream))
    _check(rc, "kvfp8_dequant")
    return out
