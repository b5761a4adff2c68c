"""The C-ABI library loads and exports what include/kvfp8.h declares; host-side
validation returns its documented codes before touching the GPU (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

import fp8_paged_kv_reshape_gb300 as kv
from fp8_paged_kv_reshape_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "kvfp8.h")


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"KVFP8_API\s+[\w\s\*]*?\b(kvfp8_\w+)\s*\(", text)))


def test_header_declares_the_binding_functions():
    assert _declared() == sorted(binding.ABI_FUNCTIONS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(kv.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", kv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kvfp8_\w+)", out))
    assert exported == set(_declared())  # nothing else leaks out of the ABI


def test_status_strings_and_scale_check():
    for code in range(9):
        assert kv.status_string(code) not in ("", "unknown status")
    assert kv.status_string(99) == "unknown status"
    assert kv.check_scale_host(0.05) == binding.OK
    assert kv.check_scale_host(-2.0) == binding.OK
    for bad in (0.0, float("inf"), float("-inf"), float("nan")):
        assert kv.check_scale_host(bad) == binding.ERR_SCALE


def test_workspace_size_grows_with_the_batch():
    a = kv.paged_decode_workspace_size(64, 32, 128)
    b = kv.paged_decode_workspace_size(128, 32, 128)
    assert 0 < a < b
    assert kv.paged_decode_workspace_size(-1, 32, 128) == 0


def _reshape(**over):
    args = dict(key=ctypes.c_void_p(16), value=ctypes.c_void_p(16), src_dtype=binding.BF16,
                key_stride=1024, value_stride=1024, num_tokens=4, key_cache=ctypes.c_void_p(16),
                value_cache=ctypes.c_void_p(16), num_blocks=4, block_size=16, n_kv=8,
                head_dim=128, slot_mapping=ctypes.c_void_p(16), k_scale=None, v_scale=None,
                scale_dtype=binding.F32, status=None, stream=None)
    args.update(over)
    return kv.LIB.kvfp8_reshape_and_cache(*args.values())


def test_reshape_host_validation():
    assert _reshape(key=None) == binding.ERR_NULL
    assert _reshape(slot_mapping=None) == binding.ERR_NULL
    assert _reshape(src_dtype=7) == binding.ERR_DTYPE
    assert _reshape(scale_dtype=5) == binding.ERR_DTYPE
    assert _reshape(n_kv=1, head_dim=3) == binding.ERR_SHAPE        # row not a multiple of 8
    assert _reshape(key_stride=100) == binding.ERR_SHAPE            # stride below the row
    assert _reshape(num_blocks=0) == binding.ERR_SHAPE
    assert _reshape(key=ctypes.c_void_p(24)) == binding.ERR_ALIGN
    assert _reshape(key_stride=1028) == binding.ERR_ALIGN           # 2056 bytes
    assert _reshape(slot_mapping=ctypes.c_void_p(20)) == binding.ERR_ALIGN
    assert _reshape(num_tokens=0, key=None) == binding.OK           # nothing to do


def test_rope_reshape_host_validation():
    def call(**over):
        args = dict(key=ctypes.c_void_p(16), value=ctypes.c_void_p(16), src_dtype=binding.BF16,
                    key_stride=1024, value_stride=1024, num_tokens=4,
                    key_cache=ctypes.c_void_p(16), value_cache=ctypes.c_void_p(16), num_blocks=4,
                    block_size=16, n_kv=8, head_dim=128, slot_mapping=ctypes.c_void_p(16),
                    positions=ctypes.c_void_p(16), cos_sin=ctypes.c_void_p(16), max_pos=4096,
                    rot=128, neox=1, k_scale=None, v_scale=None, scale_dtype=binding.F32,
                    status=None, stream=None)
        args.update(over)
        return kv.LIB.kvfp8_rope_reshape_and_cache(*args.values())
    assert call(positions=None) == binding.ERR_NULL
    assert call(cos_sin=None) == binding.ERR_NULL
    assert call(rot=96) == binding.ERR_SHAPE          # not a power of two
    assert call(rot=256) == binding.ERR_SHAPE         # above head_dim
    assert call(rot=8) == binding.ERR_SHAPE
    assert call(head_dim=96, n_kv=8, key_stride=768, value_stride=768) == binding.ERR_SHAPE
    assert call(max_pos=0) == binding.ERR_SHAPE
    assert call(n_kv=32, key_stride=4096, value_stride=4096) == binding.ERR_UNSUPPORTED
    assert call(cos_sin=ctypes.c_void_p(24)) == binding.ERR_ALIGN
    assert call(positions=ctypes.c_void_p(20)) == binding.ERR_ALIGN
    assert call(num_tokens=0, key=None) == binding.OK


def _decode(**over):
    args = dict(out=ctypes.c_void_p(16), query=ctypes.c_void_p(16), key_cache=ctypes.c_void_p(16),
                value_cache=ctypes.c_void_p(16), block_tables=ctypes.c_void_p(16),
                max_blocks_per_seq=256, seq_lens=ctypes.c_void_p(16), num_seqs=4, n_q=32, n_kv=8,
                head_dim=128, block_size=16, num_blocks=1024, sm_scale=0.0, k_scale=None,
                v_scale=None, scale_dtype=binding.F32, workspace=ctypes.c_void_p(16),
                workspace_bytes=1 << 30, status=None, stream=None)
    args.update(over)
    return kv.LIB.kvfp8_paged_decode_attention(*args.values())


def test_decode_host_validation():
    assert _decode(query=None) == binding.ERR_NULL
    assert _decode(workspace=None) == binding.ERR_NULL
    assert _decode(n_q=30) == binding.ERR_SHAPE                      # not a multiple of n_kv
    assert _decode(n_q=8 * 129) == binding.ERR_UNSUPPORTED           # group above 128
    assert _decode(head_dim=96) == binding.ERR_SHAPE
    assert _decode(block_size=12) == binding.ERR_SHAPE
    assert _decode(sm_scale=float("nan")) == binding.ERR_SCALE
    assert _decode(out=ctypes.c_void_p(8)) == binding.ERR_ALIGN
    assert _decode(workspace_bytes=100) == binding.ERR_WORKSPACE
    assert _decode(num_seqs=0, query=None) == binding.OK


def test_dequant_host_validation():
    lib = kv.LIB
    assert lib.kvfp8_dequant(None, binding.F32, ctypes.c_void_p(16), 16, None, 0, None) == binding.ERR_NULL
    assert lib.kvfp8_dequant(ctypes.c_void_p(16), 9, ctypes.c_void_p(16), 16, None, 0, None) == binding.ERR_DTYPE
    assert lib.kvfp8_dequant(ctypes.c_void_p(16), binding.F32, ctypes.c_void_p(16), -1, None, 0, None) == binding.ERR_SHAPE
    assert lib.kvfp8_dequant(ctypes.c_void_p(16), binding.F32, ctypes.c_void_p(17), 16, None, 0, None) == binding.ERR_ALIGN
    assert lib.kvfp8_dequant(None, binding.F32, None, 0, None, 0, None) == binding.OK


def test_mixed_reshape_host_validation():
    def call(**over):
        args = dict(key=ctypes.c_void_p(16), value=ctypes.c_void_p(16), src_dtype=binding.BF16,
                    key_stride=1024, value_stride=1024, num_tokens=4,
                    key_cache=ctypes.c_void_p(16), k_kind=binding.CACHE_BF16,
                    value_cache=ctypes.c_void_p(16), v_kind=binding.CACHE_E4M3, num_blocks=4,
                    block_size=16, n_kv=8, head_dim=128, slot_mapping=ctypes.c_void_p(16),
                    k_scale=None, v_scale=None, scale_dtype=binding.F32, status=None, stream=None)
        args.update(over)
        return kv.LIB.kvfp8_reshape_and_cache_mixed(*args.values())
    assert call(k_kind=2) == binding.ERR_DTYPE
    assert call(v_kind=-1) == binding.ERR_DTYPE
    assert call(key_cache=None) == binding.ERR_NULL
    assert call(n_kv=1, head_dim=3) == binding.ERR_SHAPE
    assert call(n_kv=32, key_stride=4096, value_stride=4096) == binding.ERR_UNSUPPORTED
    assert call(value_cache=ctypes.c_void_p(8)) == binding.ERR_ALIGN
    assert call(num_tokens=0, key=None) == binding.OK


def test_mixed_decode_host_validation():
    def call(**over):
        args = dict(out=ctypes.c_void_p(16), query=ctypes.c_void_p(16),
                    key_cache=ctypes.c_void_p(16), k_kind=binding.CACHE_E4M3,
                    value_cache=ctypes.c_void_p(16), v_kind=binding.CACHE_BF16,
                    block_tables=ctypes.c_void_p(16), max_blocks_per_seq=256,
                    seq_lens=ctypes.c_void_p(16), num_seqs=4, n_q=32, n_kv=8, head_dim=128,
                    block_size=16, num_blocks=1024, sm_scale=0.0, k_scale=None, v_scale=None,
                    scale_dtype=binding.F32, workspace=ctypes.c_void_p(16),
                    workspace_bytes=1 << 30, status=None, stream=None)
        args.update(over)
        return kv.LIB.kvfp8_paged_decode_attention_mixed(*args.values())
    assert call(k_kind=5) == binding.ERR_DTYPE
    assert call(k_kind=binding.CACHE_BF16, v_kind=binding.CACHE_BF16) == binding.ERR_UNSUPPORTED
    assert call(head_dim=256, n_q=80) == binding.ERR_UNSUPPORTED    # group of 10 at head_dim 256
    assert call(n_q=17 * 8) == binding.ERR_UNSUPPORTED               # group of 17
    assert call(head_dim=96) == binding.ERR_SHAPE
    assert call(n_q=30) == binding.ERR_SHAPE
    assert call(query=None) == binding.ERR_NULL
    assert call(value_cache=ctypes.c_void_p(24)) == binding.ERR_ALIGN
    assert call(workspace_bytes=100) == binding.ERR_WORKSPACE
    assert call(num_seqs=0, query=None) == binding.OK
    # both sides E4M3 is the all-FP8 call, with its own validation
    assert call(v_kind=binding.CACHE_E4M3, head_dim=96) == binding.ERR_SHAPE


def test_multi_query_workspace_follows_the_kernel_that_serves_the_shape():
    dec = kv.paged_decode_workspace_size
    ws = kv.paged_attention_multi_workspace_size
    # split-KV decode kernel: up to 16 score columns per kv head (8 at head_dim 256), n_kv <= 8
    assert ws(4, 32, 8, 128, 4) == dec(4, 32 * 4, 128) > 0
    assert ws(4, 4, 2, 256, 4) == dec(4, 4 * 4, 256) > 0
    # tensor-core kernel: no workspace
    assert ws(4, 32, 8, 128, 5) == 0          # 20 columns
    assert ws(4, 4, 2, 256, 5) == 0           # 10 columns at head_dim 256
    assert ws(4, 16, 16, 128, 1) == dec(4, 16, 128) > 0   # 16 kv heads: two head groups
    assert ws(4, 16, 16, 128, 17) == 0                    # 17 columns
    assert ws(-1, 32, 8, 128, 4) == 0


def test_multi_query_host_validation_on_the_tensor_core_route():
    def call(**over):
        args = dict(out=ctypes.c_void_p(16), query=ctypes.c_void_p(16), qsl=ctypes.c_void_p(16),
                    rows=64, qmax=64, key_cache=ctypes.c_void_p(16),
                    value_cache=ctypes.c_void_p(16), block_tables=ctypes.c_void_p(16),
                    max_blocks_per_seq=256, seq_lens=ctypes.c_void_p(16), num_seqs=1, n_q=32,
                    n_kv=8, head_dim=128, block_size=16, num_blocks=1024, sm_scale=0.0,
                    k_scale=None, v_scale=None, scale_dtype=binding.F32, workspace=None,
                    workspace_bytes=0, status=None, stream=None)
        args.update(over)
        return kv.LIB.kvfp8_paged_attention_multi(*args.values())
    assert call(query=None) == binding.ERR_NULL
    assert call(qsl=ctypes.c_void_p(18)) == binding.ERR_ALIGN
    assert call(n_q=129 * 2, n_kv=2) == binding.ERR_UNSUPPORTED     # group of 129 heads
    # 2^20 sequences x 8 kv heads x 4096 row tiles: 2^35 CTAs, past the 2^31 - 1 grid
    assert call(num_seqs=1 << 20, n_q=128 * 8, qmax=1 << 12) == binding.ERR_UNSUPPORTED
    assert call(num_seqs=0, query=None) == binding.OK
    # the split-KV route still wants its workspace
    assert call(qmax=4, workspace=None) == binding.ERR_NULL


def _noalloc(**over):
    args = dict(out=ctypes.c_void_p(16), query=ctypes.c_void_p(16), key_cache=ctypes.c_void_p(16),
                value_cache=ctypes.c_void_p(16), block_tables=ctypes.c_void_p(16),
                max_blocks_per_seq=256, seq_lens=ctypes.c_void_p(16), num_seqs=4, n_q=32, n_kv=8,
                head_dim=128, block_size=16, num_blocks=1024, sm_scale=0.0, k_scale=None,
                v_scale=None, scale_dtype=binding.F32, status=None, stream=None)
    args.update(over)
    return kv.LIB.kvfp8_paged_decode_attention_noalloc(*args.values())


def test_noalloc_host_validation_matches_the_workspace_entry_point():
    # every argument error comes back with the workspace entry point's code, before the
    # library's scratch array is looked up (so no device is needed to see them)
    for over in (dict(query=None), dict(seq_lens=None), dict(scale_dtype=4), dict(n_q=30),
                 dict(n_q=8 * 129), dict(head_dim=96), dict(block_size=12),
                 dict(num_blocks=0), dict(sm_scale=float("inf")), dict(out=ctypes.c_void_p(8)),
                 dict(block_tables=ctypes.c_void_p(18)), dict(num_seqs=-1),
                 dict(num_seqs=0, query=None)):
        assert _noalloc(**over) == _decode(**over), over
    assert _noalloc(num_seqs=0, query=None) == binding.OK
    # past the fixed scratch: refused without touching a device
    assert kv.paged_decode_workspace_size(40000, 32, 128) > (32 << 20)
    assert _noalloc(num_seqs=40000) == binding.ERR_WORKSPACE


def test_noalloc_binding_checks_tables_like_the_workspace_binding():
    import torch

    q = torch.zeros(4, 32, 128, dtype=torch.bfloat16)
    kc = torch.zeros(8, 16, 8, 128, dtype=torch.uint8)
    bt = torch.zeros(4, 2, dtype=torch.int32)
    sl = torch.ones(4, dtype=torch.int32)
    bad = [(bt.long(), sl), (bt[:3], sl), (bt, sl.long()), (bt, sl[:3]), (bt.t(), sl)]
    for fn in (kv.paged_decode_attention, kv.paged_decode_attention_noalloc):
        for b, s in bad:
            with pytest.raises(ValueError):
                fn(q, kc, kc, b, s)
        with pytest.raises(ValueError):  # out shaped unlike query
            fn(q, kc, kc, bt, sl, out=torch.zeros(4, 32, 64, dtype=torch.bfloat16))


def test_multi_mixed_host_validation():
    def call(**over):
        args = dict(out=ctypes.c_void_p(16), query=ctypes.c_void_p(16), qsl=ctypes.c_void_p(16),
                    rows=16, qmax=4, key_cache=ctypes.c_void_p(16), k_kind=binding.CACHE_BF16,
                    value_cache=ctypes.c_void_p(16), v_kind=binding.CACHE_E4M3,
                    block_tables=ctypes.c_void_p(16), max_blocks_per_seq=256,
                    seq_lens=ctypes.c_void_p(16), num_seqs=4, n_q=32, n_kv=8, head_dim=128,
                    block_size=16, num_blocks=1024, sm_scale=0.0, k_scale=None, v_scale=None,
                    scale_dtype=binding.F32, workspace=ctypes.c_void_p(16),
                    workspace_bytes=1 << 30, status=None, stream=None)
        args.update(over)
        return kv.LIB.kvfp8_paged_attention_multi_mixed(*args.values())
    assert call(k_kind=3) == binding.ERR_DTYPE
    assert call(k_kind=binding.CACHE_BF16, v_kind=binding.CACHE_BF16) == binding.ERR_UNSUPPORTED
    assert call(qmax=5) == binding.ERR_UNSUPPORTED                 # 20 score columns
    assert call(head_dim=256, qmax=3) == binding.ERR_UNSUPPORTED   # 12 columns at head_dim 256
    assert call(head_dim=96) == binding.ERR_SHAPE
    assert call(qsl=None) == binding.ERR_NULL
    assert call(workspace=None) == binding.ERR_NULL
    assert call(qsl=ctypes.c_void_p(18)) == binding.ERR_ALIGN
    assert call(workspace_bytes=100) == binding.ERR_WORKSPACE
    assert call(num_seqs=0, query=None) == binding.OK
    # both sides E4M3 is the all-FP8 call, with its own validation
    assert call(k_kind=binding.CACHE_E4M3, head_dim=96) == binding.ERR_SHAPE
    assert call(k_kind=binding.CACHE_E4M3, query=None) == binding.ERR_NULL
