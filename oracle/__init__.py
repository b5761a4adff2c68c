"""kvfp8 oracle: plain, slow CPU statement of the FP8 paged KV-cache path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library (``fp8_paged_kv_reshape_gb300``) and never imports it.

The arithmetic lives in ``kvfp8_oracle.c`` (plain C11, single-threaded); this
module only marshals numpy arrays into it.  Parity status: every function here
is pinned by ``tests/test_oracle_codec.py``, ``tests/test_oracle_store.py`` and
``tests/test_oracle_attention.py`` against values the source pages and
mathematics fix; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import math

import numpy as np

from . import build as _build

BF16 = 0
F32 = 1

STATUS_BAD_SCALE = 1 << 0
STATUS_BAD_SLOT = 1 << 1
STATUS_BAD_BLOCK = 1 << 2

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f32, f64, u8, u32 = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                       ctypes.c_double, ctypes.c_uint8, ctypes.c_uint32)
        lib.kvo_e4m3_decode.argtypes = [u8]
        lib.kvo_e4m3_decode.restype = f64
        lib.kvo_e4m3_encode.argtypes = [f32]
        lib.kvo_e4m3_encode.restype = u8
        lib.kvo_e4m3_encode_n.argtypes = [P, P, i64]
        lib.kvo_e4m3_encode_n.restype = None
        lib.kvo_store_code.argtypes = [f32, f32]
        lib.kvo_store_code.restype = u8
        lib.kvo_scale_ok.argtypes = [f32]
        lib.kvo_scale_ok.restype = ctypes.c_int
        lib.kvo_scale_value.argtypes = [P, ctypes.c_int]
        lib.kvo_scale_value.restype = f32
        lib.kvo_f32_to_bf16.argtypes = [f32]
        lib.kvo_f32_to_bf16.restype = ctypes.c_uint16
        lib.kvo_reshape_and_cache.argtypes = [P, P, ctypes.c_int, i64, i64, i64, P, P, i32, i32,
                                              i32, i32, P, f32, f32]
        lib.kvo_reshape_and_cache.restype = u32
        lib.kvo_rope.argtypes = [P, i32, i32, ctypes.c_int, P]
        lib.kvo_rope.restype = None
        lib.kvo_rope_reshape_and_cache.argtypes = [P, P, ctypes.c_int, i64, i64, i64, P, P, i32,
                                                   i32, i32, i32, P, P, P, i64, i32, ctypes.c_int,
                                                   f32, f32]
        lib.kvo_rope_reshape_and_cache.restype = u32
        lib.kvo_dequant.argtypes = [P, ctypes.c_int, P, i64, ctypes.c_int, f32]
        lib.kvo_dequant.restype = None
        lib.kvo_paged_decode_attention.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                                   i32, f64, f32, f32]
        lib.kvo_paged_decode_attention.restype = u32
        lib.kvo_paged_attention_multi.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32, i32,
                                                  i32, i32, f64, f32, f32]
        lib.kvo_paged_attention_multi.restype = u32
        lib.kvo_reshape_and_cache_mixed.argtypes = [P, P, ctypes.c_int, i64, P, ctypes.c_int, P,
                                                    ctypes.c_int, i32, i32, i32, i32, P, f32, f32]
        lib.kvo_reshape_and_cache_mixed.restype = u32
        lib.kvo_paged_decode_attention_mixed.argtypes = [P, P, P, ctypes.c_int, P, ctypes.c_int, P,
                                                         i32, P, i32, i32, i32, i32, i32, i32, f64,
                                                         f32, f32]
        lib.kvo_paged_decode_attention_mixed.restype = u32
        lib.kvo_paged_attention_multi_mixed.argtypes = [P, P, P, P, ctypes.c_int, P, ctypes.c_int,
                                                        P, i32, P, i32, i32, i32, i32, i32, i32,
                                                        f64, f32, f32]
        lib.kvo_paged_attention_multi_mixed.restype = u32
        lib.kvo_paged_decode_attention_pairs.argtypes = [P, P, i32, P, P, P, P, i32, P, i32, i32,
                                                         i32, i32, i32, f64, f32, f32]
        lib.kvo_paged_decode_attention_pairs.restype = u32
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _as_u16(a) -> np.ndarray:
    """bf16 data as raw uint16 (accepts a uint16 array or a CPU torch bf16 tensor)."""
    if isinstance(a, np.ndarray):
        assert a.dtype == np.uint16
        return np.ascontiguousarray(a)
    import torch  # only for unpacking a caller's CPU bf16 tensor

    assert a.dtype == torch.bfloat16 and a.device.type == "cpu"
    return a.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- codec

def e4m3_decode(code: int) -> float:
    return _load().kvo_e4m3_decode(int(code))


def e4m3_decode_all() -> np.ndarray:
    """The 256 decoded values, index = code."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(y: float) -> int:
    return int(_load().kvo_e4m3_encode(float(np.float32(y))))


def e4m3_encode_array(y: np.ndarray) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float32).ravel()
    out = np.empty(y.size, dtype=np.uint8)
    _load().kvo_e4m3_encode_n(_ptr(y), _ptr(out), y.size)
    return out


def store_code(x: float, s: float) -> int:
    return int(_load().kvo_store_code(float(np.float32(x)), float(np.float32(s))))


def scale_ok(s: float) -> bool:
    return bool(_load().kvo_scale_ok(float(np.float32(s))))


def scale_value(raw: np.ndarray, dtype: int) -> float:
    raw = np.ascontiguousarray(raw)
    return float(_load().kvo_scale_value(_ptr(raw), dtype))


def f32_to_bf16(f: float) -> int:
    return int(_load().kvo_f32_to_bf16(float(np.float32(f))))


# ---------------------------------------------------------------- path

def reshape_and_cache(key, value, key_cache: np.ndarray, value_cache: np.ndarray,
                      slot_mapping: np.ndarray, block_size: int, k_scale: float, v_scale: float,
                      src_dtype: int = BF16, key_stride: int | None = None,
                      value_stride: int | None = None) -> int:
    """Quantize-and-scatter into the caches in place; returns the status bits.

    key/value: [num_tokens, n_kv, head_dim] (bf16 as uint16 or CPU torch bf16,
    or float32 when src_dtype == F32); caches: uint8
    [num_blocks, block_size, n_kv, head_dim].
    """
    if src_dtype == BF16:
        k = _as_u16(key)
        v = _as_u16(value)
    else:
        k = np.ascontiguousarray(key, dtype=np.float32)
        v = np.ascontiguousarray(value, dtype=np.float32)
    num_blocks, bs, n_kv, hd = key_cache.shape
    assert bs == block_size and value_cache.shape == key_cache.shape
    assert key_cache.dtype == np.uint8 and value_cache.dtype == np.uint8
    num_tokens = k.shape[0]
    row = n_kv * hd
    ks = row if key_stride is None else key_stride
    vs = row if value_stride is None else value_stride
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert slots.shape[0] == num_tokens
    return int(_load().kvo_reshape_and_cache(
        _ptr(k), _ptr(v), src_dtype, ks, vs, num_tokens, _ptr(key_cache), _ptr(value_cache),
        num_blocks, block_size, n_kv, hd, _ptr(slots), float(np.float32(k_scale)),
        float(np.float32(v_scale))))


def rope(x: np.ndarray, cos_sin_row: np.ndarray, rot: int, neox: bool) -> np.ndarray:
    """Rotate one head vector (float32) by one table row; returns a new array."""
    v = np.ascontiguousarray(x, dtype=np.float32).copy()
    cs = np.ascontiguousarray(cos_sin_row, dtype=np.float32)
    assert cs.size >= rot and v.size >= rot
    _load().kvo_rope(_ptr(v), v.size, rot, 1 if neox else 0, _ptr(cs))
    return v


def rope_reshape_and_cache(key, value, key_cache: np.ndarray, value_cache: np.ndarray,
                           slot_mapping: np.ndarray, positions: np.ndarray, cos_sin: np.ndarray,
                           rot: int, neox: bool, block_size: int, k_scale: float, v_scale: float,
                           src_dtype: int = BF16) -> int:
    """Rope on K, then quantize-and-scatter K and V in place; returns the status bits.
    cos_sin: float32 [max_pos, rot] (cos then sin halves)."""
    if src_dtype == BF16:
        k = _as_u16(key)
        v = _as_u16(value)
    else:
        k = np.ascontiguousarray(key, dtype=np.float32)
        v = np.ascontiguousarray(value, dtype=np.float32)
    num_blocks, bs, n_kv, hd = key_cache.shape
    assert bs == block_size and value_cache.shape == key_cache.shape
    cs = np.ascontiguousarray(cos_sin, dtype=np.float32)
    assert cs.ndim == 2 and cs.shape[1] == rot
    num_tokens = k.shape[0]
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    assert slots.shape[0] == num_tokens and pos.shape[0] == num_tokens
    return int(_load().kvo_rope_reshape_and_cache(
        _ptr(k), _ptr(v), src_dtype, n_kv * hd, n_kv * hd, num_tokens, _ptr(key_cache),
        _ptr(value_cache), num_blocks, block_size, n_kv, hd, _ptr(slots), _ptr(pos), _ptr(cs),
        cs.shape[0], rot, 1 if neox else 0, float(np.float32(k_scale)),
        float(np.float32(v_scale))))


def dequant(src: np.ndarray, dst_dtype: int = F32, scale: float | None = None) -> np.ndarray:
    src = np.ascontiguousarray(src, dtype=np.uint8).ravel()
    out = np.empty(src.size, dtype=np.float32 if dst_dtype == F32 else np.uint16)
    _load().kvo_dequant(_ptr(out), dst_dtype, _ptr(src), src.size, 0 if scale is None else 1,
                        0.0 if scale is None else float(np.float32(scale)))
    return out


def paged_decode_attention(query, key_cache: np.ndarray, value_cache: np.ndarray,
                           block_tables: np.ndarray, seq_lens: np.ndarray, k_scale: float,
                           v_scale: float, sm_scale: float = 0.0):
    """Full decode attention in double; returns (out[num_seqs, n_q, head_dim] float64, status)."""
    q = _as_u16(query)
    num_seqs, n_q, hd = q.shape
    num_blocks, bs, n_kv, hd2 = key_cache.shape
    assert hd2 == hd and n_q % n_kv == 0
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((num_seqs, n_q, hd), dtype=np.float64)
    st = _load().kvo_paged_decode_attention(
        _ptr(out), _ptr(q), _ptr(np.ascontiguousarray(key_cache)),
        _ptr(np.ascontiguousarray(value_cache)), _ptr(bt), bt.shape[1], _ptr(sl), num_seqs, n_q,
        n_kv, hd, bs, num_blocks, float(sm_scale), float(np.float32(k_scale)),
        float(np.float32(v_scale)))
    return out, int(st)


def paged_attention_multi(query, query_start_loc: np.ndarray, key_cache: np.ndarray,
                          value_cache: np.ndarray, block_tables: np.ndarray, seq_lens: np.ndarray,
                          k_scale: float, v_scale: float, sm_scale: float = 0.0):
    """Causal multi-query attention in double; query [total_q, n_q, hd] (bf16) with
    sequence b's rows at query_start_loc[b]; returns (out float64 like query, status)."""
    q = _as_u16(query)
    total_q, n_q, hd = q.shape
    num_blocks, bs, n_kv, hd2 = key_cache.shape
    assert hd2 == hd and n_q % n_kv == 0
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    assert qsl.size == sl.size + 1 and qsl[-1] == total_q
    out = np.zeros((total_q, n_q, hd), dtype=np.float64)
    st = _load().kvo_paged_attention_multi(
        _ptr(out), _ptr(q), _ptr(qsl), _ptr(np.ascontiguousarray(key_cache)),
        _ptr(np.ascontiguousarray(value_cache)), _ptr(bt), bt.shape[1], _ptr(sl), sl.size, n_q,
        n_kv, hd, bs, num_blocks, float(sm_scale), float(np.float32(k_scale)),
        float(np.float32(v_scale)))
    return out, int(st)


E4M3 = 0      # cache kinds for the mixed-dtype functions
CACHE_BF16 = 1


def reshape_and_cache_mixed(key, value, key_cache: np.ndarray, k_kind: int,
                            value_cache: np.ndarray, v_kind: int, slot_mapping: np.ndarray,
                            block_size: int, k_scale: float, v_scale: float,
                            src_dtype: int = BF16) -> int:
    """Store with a per-side cache kind: E4M3 (uint8 cache, scaled) or CACHE_BF16 (uint16
    cache holding bf16 bits, unscaled).  Caches [num_blocks, block_size, n_kv, head_dim]."""
    if src_dtype == BF16:
        k, v = _as_u16(key), _as_u16(value)
    else:
        k = np.ascontiguousarray(key, dtype=np.float32)
        v = np.ascontiguousarray(value, dtype=np.float32)
    for c, kind in ((key_cache, k_kind), (value_cache, v_kind)):
        assert c.dtype == (np.uint8 if kind == E4M3 else np.uint16) and c.flags["C_CONTIGUOUS"]
    num_blocks, bs, n_kv, hd = key_cache.shape
    assert bs == block_size and value_cache.shape == key_cache.shape
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    return int(_load().kvo_reshape_and_cache_mixed(
        _ptr(k), _ptr(v), src_dtype, k.shape[0], _ptr(key_cache), k_kind, _ptr(value_cache),
        v_kind, num_blocks, block_size, n_kv, hd, _ptr(slots), float(np.float32(k_scale)),
        float(np.float32(v_scale))))


def paged_decode_attention_mixed(query, key_cache: np.ndarray, k_kind: int,
                                 value_cache: np.ndarray, v_kind: int, block_tables: np.ndarray,
                                 seq_lens: np.ndarray, k_scale: float, v_scale: float,
                                 sm_scale: float = 0.0):
    q = _as_u16(query)
    num_seqs, n_q, hd = q.shape
    num_blocks, bs, n_kv, _ = key_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((num_seqs, n_q, hd), dtype=np.float64)
    st = _load().kvo_paged_decode_attention_mixed(
        _ptr(out), _ptr(q), _ptr(np.ascontiguousarray(key_cache)), k_kind,
        _ptr(np.ascontiguousarray(value_cache)), v_kind, _ptr(bt), bt.shape[1], _ptr(sl),
        num_seqs, n_q, n_kv, hd, bs, num_blocks, float(sm_scale), float(np.float32(k_scale)),
        float(np.float32(v_scale)))
    return out, int(st)


def paged_attention_multi_mixed(query, query_start_loc: np.ndarray, key_cache: np.ndarray,
                                k_kind: int, value_cache: np.ndarray, v_kind: int,
                                block_tables: np.ndarray, seq_lens: np.ndarray, k_scale: float,
                                v_scale: float, sm_scale: float = 0.0):
    """Causal multi-query attention with a per-side cache kind (E4M3 or CACHE_BF16), in
    double; query [total_q, n_q, hd] (bf16) with sequence b's rows at query_start_loc[b];
    returns (out float64 like query, status)."""
    q = _as_u16(query)
    total_q, n_q, hd = q.shape
    num_blocks, bs, n_kv, hd2 = key_cache.shape
    assert hd2 == hd and n_q % n_kv == 0
    for c, kind in ((key_cache, k_kind), (value_cache, v_kind)):
        assert c.dtype == (np.uint8 if kind == E4M3 else np.uint16)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    assert qsl.size == sl.size + 1 and qsl[-1] == total_q
    out = np.zeros((total_q, n_q, hd), dtype=np.float64)
    st = _load().kvo_paged_attention_multi_mixed(
        _ptr(out), _ptr(q), _ptr(qsl), _ptr(np.ascontiguousarray(key_cache)), k_kind,
        _ptr(np.ascontiguousarray(value_cache)), v_kind, _ptr(bt), bt.shape[1], _ptr(sl), sl.size,
        n_q, n_kv, hd, bs, num_blocks, float(sm_scale), float(np.float32(k_scale)),
        float(np.float32(v_scale)))
    return out, int(st)


def paged_decode_attention_pairs(pairs: np.ndarray, query, key_cache: np.ndarray,
                                 value_cache: np.ndarray, block_tables: np.ndarray,
                                 seq_lens: np.ndarray, k_scale: float, v_scale: float,
                                 sm_scale: float = 0.0):
    """Decode attention for sampled (seq, head) pairs; returns (out[n_pairs, head_dim], status)."""
    q = _as_u16(query)
    num_seqs, n_q, hd = q.shape
    num_blocks, bs, n_kv, _ = key_cache.shape
    pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    out = np.zeros((pr.shape[0], hd), dtype=np.float64)
    st = _load().kvo_paged_decode_attention_pairs(
        _ptr(out), _ptr(pr), pr.shape[0], _ptr(q), _ptr(np.ascontiguousarray(key_cache)),
        _ptr(np.ascontiguousarray(value_cache)), _ptr(bt), bt.shape[1], _ptr(sl), n_q, n_kv, hd,
        bs, num_blocks, float(sm_scale), float(np.float32(k_scale)), float(np.float32(v_scale)))
    return out, int(st)


def default_sm_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
