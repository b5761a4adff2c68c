"""Pins for the oracle's store path: divide by the scale, encode, scatter (CPU only).

[P1] = llama.cpp commit "llama : Add FP8 KV-cache support (#28392)";
[P3] = vllm.cpp PR #1641 "feat(KV-FP8): W3 ...".
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import pins

SCALES = [0.05, 0.04, 0.03, 0.3, 3.7, 0.125, 0.25, 0.03125, 0.5, 1.0, -0.05, 3.0, 1e-3, 7.3e5,
          float(np.float32(0.1)), 2.0 ** -7, 2.0 ** -13, 2.0 ** -11, 2.0 ** -9]


def _store_codes(x: np.ndarray, s: float) -> np.ndarray:
    """Oracle store codes for a 1-D float32 array via the reshape entry point."""
    n = x.size
    key = np.ascontiguousarray(x, dtype=np.float32).reshape(n, 1, 1)
    kc = np.full((n, 1, 1, 1), 0x5A, dtype=np.uint8)
    vc = kc.copy()
    st = oracle.reshape_and_cache(key, key, kc, vc, np.arange(n, dtype=np.int64), 1, s, s,
                                  src_dtype=oracle.F32)
    assert st == 0
    return kc.ravel()


def test_store_is_ieee_division_then_encode_on_every_bf16_value():
    # [P1] llama-graph.cpp build_attn_scale_kv_inputs: K is divided by s_k (ggml_div)
    # before the F8 cache copy.  Expected: brute-force encode of the IEEE float32 quotient
    # (numpy's float32 division is correctly rounded).
    x = pins.all_bf16_as_f32()
    for s in SCALES:
        with np.errstate(all="ignore"):
            q = (x / np.float32(s)).astype(np.float32)
        want = pins.brute_encode(q)
        nan = np.isnan(x)
        want[nan] = 0x7F | (np.signbit(x[nan]).astype(np.uint8) << 7)
        got = _store_codes(x, s)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (s, [(float(x[i]), hex(got[i]), hex(want[i])) for i in bad[:5]])


def test_store_quotient_is_exactly_rounded():
    # Independent of any float division: round the exact rational x/s to float32
    # with integer arithmetic, then brute-force encode.
    rng = np.random.Generator(np.random.PCG64(3))
    bits = rng.integers(0, 1 << 16, size=4000).astype(np.uint32)
    x = pins.bf16_bits_to_f32(bits)
    x = x[np.isfinite(x)]
    for s in (0.05, 0.04, -0.125, 1e-3, 3.0):
        sf = np.float32(s)
        q = np.array([pins.rn_f32(Fraction(float(v)) / Fraction(float(sf))) for v in x],
                     dtype=np.float32)
        np.testing.assert_array_equal(_store_codes(x, s), pins.brute_encode(q))


def test_division_is_distinguishable_from_reciprocal_multiply():
    # Anti-vacuity for the pin above: multiplying by a rounded 1/s gives different bytes
    # for some bf16 inputs (30 of them at s = 0.03; none at 0.05), so a store written
    # that way would fail it.
    x = pins.all_bf16_as_f32()
    x = x[np.isfinite(x)]
    s = np.float32(0.03)
    with np.errstate(all="ignore"):
        div = pins.brute_encode((x / s).astype(np.float32))
        mul = pins.brute_encode((x * (np.float32(1) / s)).astype(np.float32))
    assert np.count_nonzero(div != mul) > 0
    np.testing.assert_array_equal(_store_codes(x, float(s)), div)


def test_store_envelope():
    # [P3] store envelope: |dequant(store(x)) - x| <= 2^-4 |x| + 2^-10 * scale for every
    # element that does not saturate; non-unit, unequal scales 0.125 (K) and 0.25 (V).
    rng = np.random.Generator(np.random.PCG64(5))
    for s in (0.125, 0.25, 0.05, 0.04):
        x = (rng.standard_normal(200_000) * np.exp2(rng.uniform(-8, 4, 200_000)) * s)
        x = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).float().numpy()
        codes = _store_codes(x, s)
        dec = oracle.e4m3_decode_all()[codes]
        unsat = np.abs(x / s) < 448.0
        normal = np.abs(x / s) >= 2.0 ** -6
        assert unsat.mean() > 0.99 and normal.sum() > 1000   # anti-vacuity
        err = np.abs(s * dec - x)
        bound = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * abs(s)
        assert np.all(err[unsat] <= bound[unsat])


def test_envelope_catches_swapped_or_dropped_scales():
    # [P3] mutation table: a store with the other side's scale, or with no scale, leaves
    # the envelope.  Checked on the oracle's own output read back with the wrong scale.
    rng = np.random.Generator(np.random.PCG64(6))
    x = (rng.standard_normal(10_000) * 0.1).astype(np.float32)
    codes = _store_codes(x, 0.125)
    dec = oracle.e4m3_decode_all()[codes]
    for wrong in (0.25, 1.0):
        err = np.abs(wrong * dec - x)
        bound = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * wrong
        assert np.count_nonzero(err > bound) > 0.5 * x.size


@pytest.mark.parametrize("pair", [(2.0 ** -7, 2.0 ** -13), (2.0 ** -11, 2.0 ** -9)])
def test_power_of_two_scale_invariance(pair):
    # [P3] section "Round 4": for power-of-two scales s, s' that keep a value normal and
    # unsaturated, s*D(Q(x/s)) == s'*D(Q(x/s')) bit for bit.
    s, t = pair
    rng = np.random.Generator(np.random.PCG64(8))
    x = (rng.standard_normal(100_000) * 2.0 ** rng.uniform(-16, -4, 100_000)).astype(np.float32)
    ok = np.ones(x.size, bool)
    for sc in pair:
        a = np.abs(x / np.float32(sc))
        ok &= (a >= 2.0 ** -6) & (a < 448.0)
    x = x[ok]
    assert x.size > 1000  # anti-vacuity
    dec = oracle.e4m3_decode_all()
    cs, ct = _store_codes(x, s), _store_codes(x, t)
    assert np.count_nonzero(cs != ct) == x.size  # different bytes...
    np.testing.assert_array_equal(np.float32(s) * dec[cs].astype(np.float32),
                                  np.float32(t) * dec[ct].astype(np.float32))  # ...same values


def test_scatter_places_rows_and_preserves_everything_else():
    # [P1] llama-kv-cache.cpp cpy_k/cpy_v: row i goes to destination slot_mapping[i];
    # slot -1 is a padding row that writes nothing.
    rng = np.random.Generator(np.random.PCG64(9))
    nb, bs, nkv, hd = 6, 4, 2, 8
    n = 10
    slots = rng.permutation(nb * bs)[:n].astype(np.int64)
    slots[[2, 7]] = -1
    k = torch.randn(n, nkv, hd, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    v = torch.randn(n, nkv, hd, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    kc = np.full((nb, bs, nkv, hd), 0x5A, np.uint8)
    vc = kc.copy()
    st = oracle.reshape_and_cache(k, v, kc, vc, slots, bs, 0.05, 0.04)
    assert st == 0
    kf, vf = k.float().numpy(), v.float().numpy()
    written = np.zeros((nb, bs), bool)
    for i, sl in enumerate(slots):
        if sl < 0:
            continue
        b, o = divmod(int(sl), bs)
        written[b, o] = True
        with np.errstate(all="ignore"):
            np.testing.assert_array_equal(kc[b, o], pins.brute_encode(kf[i] / np.float32(0.05)).reshape(nkv, hd))
            np.testing.assert_array_equal(vc[b, o], pins.brute_encode(vf[i] / np.float32(0.04)).reshape(nkv, hd))
    assert np.all(kc[~written] == 0x5A) and np.all(vc[~written] == 0x5A)
    assert written.sum() == n - 2


def test_scatter_honours_row_strides():
    n, nkv, hd = 5, 2, 4
    big = torch.randn(n, 3 * nkv * hd, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    kc = np.zeros((n, 1, nkv, hd), np.uint8)
    vc = kc.copy()
    key = big[:, : nkv * hd].contiguous()
    val = big[:, 2 * nkv * hd:].contiguous()
    oracle.reshape_and_cache(key, val, kc, vc, np.arange(n), 1, 0.5, 0.5)
    kc2, vc2 = np.zeros_like(kc), np.zeros_like(vc)
    raw = big.contiguous()
    raw_u16 = raw.view(torch.int16).numpy().view(np.uint16)
    lib = oracle._load()
    lib.kvo_reshape_and_cache(oracle._ptr(raw_u16), oracle._ptr(raw_u16[:, 2 * nkv * hd:].copy()),
                              oracle.BF16, 3 * nkv * hd, nkv * hd, n, oracle._ptr(kc2),
                              oracle._ptr(vc2), n, 1, nkv, hd,
                              oracle._ptr(np.arange(n, dtype=np.int64)), 0.5, 0.5)
    np.testing.assert_array_equal(kc, kc2)
    np.testing.assert_array_equal(vc, vc2)


def test_bad_slots_and_scales_are_flagged():
    kc = np.zeros((2, 2, 1, 8), np.uint8)
    vc = kc.copy()
    k = torch.ones(3, 1, 8, dtype=torch.bfloat16)
    st = oracle.reshape_and_cache(k, k, kc, vc, np.array([0, 4, -2]), 2, 0.5, 0.5)
    assert st == oracle.STATUS_BAD_SLOT
    assert np.all(kc[0, 0] == oracle.e4m3_encode(2.0)) and np.all(kc.reshape(4, 8)[1:] == 0)
    for bad in (0.0, math.inf, -math.inf, math.nan):
        assert not oracle.scale_ok(bad)
        kc[:] = 0
        assert oracle.reshape_and_cache(k, k, kc, vc, np.array([0, 1, 2]), 2, bad, 0.5) == \
            oracle.STATUS_BAD_SCALE
        assert np.all(kc == 0)
    assert oracle.scale_ok(-0.05) and oracle.scale_ok(1e-30)


def test_bf16_scale_widens_exactly():
    # [P1] conversion/base.py accepts a BF16 or FP32 scale and widens it (scale.float()).
    for v in (0.05, 0.04, 0.125):
        t = torch.tensor([v], dtype=torch.bfloat16)
        raw = t.view(torch.int16).numpy().view(np.uint16).copy()
        assert oracle.scale_value(raw, oracle.BF16) == float(t.float().item())
        assert workloads.stored_scale(v, "bf16") == float(t.float().item())
    raw = np.array([0.05], np.float32)
    assert oracle.scale_value(raw, oracle.F32) == float(np.float32(0.05))


def test_fp8_block_is_half_of_bf16_block():
    # [P3] ApplyCacheDType: KVBytesPerBlock exactly halved.
    for (bs, nkv, hd) in [(16, 8, 128), (32, 8, 128), (16, 2, 64)]:
        fp8 = np.zeros((1, bs, nkv, hd), np.uint8)
        bf16 = torch.zeros((1, bs, nkv, hd), dtype=torch.bfloat16)
        assert 2 * fp8.nbytes == bf16.numel() * bf16.element_size()


def test_dequant_is_exact_and_rounds_bf16_once():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode_all()
    f = oracle.dequant(codes, oracle.F32)
    finite = ~np.isnan(vals)
    np.testing.assert_array_equal(f[finite], vals[finite].astype(np.float32))
    assert np.all(np.isnan(f[~finite]))
    for s in (0.05, 0.5, -3.0):
        fs = oracle.dequant(codes, oracle.F32, s)
        want = np.float32(s) * vals.astype(np.float32)
        np.testing.assert_array_equal(fs[finite], want[finite])
        b = oracle.dequant(codes, oracle.BF16, s)
        want_b = torch.from_numpy(want).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(b[finite], want_b[finite])


def test_requantize_of_dequantized_bytes_is_identity():
    # [P1] tests/test-fp8.cpp check_fp8_context_shift: the stored bytes after a shift are
    # quantize(rope(decode(bytes))); at a zero shift rope is the identity, so the bytes
    # must come back unchanged (scale-free: rope is linear).
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    f = oracle.dequant(codes, oracle.F32)
    np.testing.assert_array_equal(oracle.e4m3_encode_array(f), codes)
    np.testing.assert_array_equal(_store_codes(f, 1.0), codes)
