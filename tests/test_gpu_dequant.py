"""kvfp8_dequant on the GPU vs the oracle (bit-exact), and the rope-shift round trip
dequantize -> rotate -> requantize against quantize(rope(decode(bytes))) from
llama.cpp "llama : Add FP8 KV-cache support (#28392)", tests/test-fp8.cpp
check_fp8_context_shift."""
import numpy as np
import pytest
import torch

import oracle
from tests import gpu_util

pytestmark = pytest.mark.gpu

kv = pytest.importorskip("fp8_paged_kv_reshape_gb300")


def _same(gpu: np.ndarray, ref: np.ndarray):
    gn, rn = np.isnan(gpu.astype(np.float32)), np.isnan(ref.astype(np.float32))
    assert np.array_equal(gn, rn)
    np.testing.assert_array_equal(gpu[~gn], ref[~rn])


@pytest.mark.parametrize("n", [256, 1, 15, 16, 17, 1000, 4096 + 7])
def test_all_codes_bit_exact(n):
    codes = np.resize(np.arange(256, dtype=np.uint8), n)
    src = torch.from_numpy(codes).cuda()
    for scale in (None, 0.05, -3.0):
        sc = None if scale is None else torch.tensor([scale], device="cuda")
        f = kv.dequant(src, torch.float32, sc).cpu().numpy()
        _same(f, oracle.dequant(codes, oracle.F32, scale))
        b = kv.dequant(src, torch.bfloat16, sc)
        b_bits = gpu_util.to_u16(b)
        ref = oracle.dequant(codes, oracle.BF16, scale)
        as_f = lambda u: (u.astype(np.uint32) << 16).view(np.float32)
        _same(as_f(b_bits), as_f(ref))


def _rope(x: np.ndarray, pos: np.ndarray, base: float = 10000.0) -> np.ndarray:
    """Plain rotary rotation of adjacent pairs (test-side, float32), token axis 0."""
    n, h, d = x.shape
    inv = (base ** (-np.arange(0, d, 2, dtype=np.float32) / d)).astype(np.float32)
    ang = (pos[:, None].astype(np.float32) * inv[None, :]).astype(np.float32)
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x0, x1 = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out.astype(np.float32)


@pytest.mark.parametrize("scale", [None, 0.5])
def test_rope_shift_round_trip_is_byte_exact(scale):
    # The shift is scale-free (rope is linear): with the layer scale 0.5 (a power of two)
    # dequant-with-scale -> rope -> requant-with-scale gives the same bytes as the
    # scale-free round trip, as the page's test checks at scales 1.0 and 0.5.
    rng = np.random.Generator(np.random.PCG64(31))
    n, h, d = 64, 2, 64
    codes = rng.integers(0, 256, size=(n, h, d), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C
    shift = np.full(n, -1, np.int32)
    sc = None if scale is None else torch.tensor([scale], device="cuda")
    deq = kv.dequant(torch.from_numpy(codes).cuda(), torch.float32, sc).cpu().numpy()
    rot = _rope(deq, shift)
    kc = torch.zeros(n, 1, h, d, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    kv.reshape_and_cache(torch.from_numpy(rot).cuda(), torch.from_numpy(rot).cuda(), kc, vc,
                         torch.arange(n, dtype=torch.int64, device="cuda"), sc, sc)
    torch.cuda.synchronize()
    # oracle: quantize(rope(decode(bytes))), no scale anywhere
    want_f = _rope(oracle.dequant(codes, oracle.F32).reshape(n, h, d), shift)
    ko = np.zeros((n, 1, h, d), np.uint8)
    oracle.reshape_and_cache(want_f, want_f, ko, ko.copy(), np.arange(n), 1, 1.0, 1.0,
                             src_dtype=oracle.F32)
    got = kc.cpu().numpy()
    assert np.array_equal(got, ko)
    assert not np.array_equal(got.reshape(codes.shape), codes)  # the shift changed bytes
