"""Pins for the oracle's E4M3 codec (CPU only).

Checked against: the format facts the pages print (tests/golden/e4m3_format.txt),
the exact closed form of every code, the exhaustive round-trip contract of
[P2] tests/test-quantize-fns.cpp test_f8_e4m3, and a brute-force nearest-code
search over every bf16 bit pattern and a large seeded sample of float32 bit
patterns.  [P2] = llama.cpp compare osimons/ocp_fp8_kv.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests import pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_format.txt")


def _golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, a, b = line.split()[:3]
            rows.append((kind, a, b))
    return rows


def test_golden_format_facts():
    rows = _golden_rows()
    assert len(rows) >= 15
    for kind, a, b in rows:
        if kind == "decode":
            got = oracle.e4m3_decode(int(a, 16))
            want = float(b)
            if math.isnan(want):
                assert math.isnan(got), (a, got)
            else:
                assert got == want and math.copysign(1, got) == math.copysign(1, want), (a, got)
        elif kind == "encode":
            got = oracle.e4m3_encode(float(a))
            assert got == int(b, 16), (a, hex(got), b)
        else:
            raise AssertionError(kind)


def test_decode_matches_closed_form_for_all_codes():
    for c in range(256):
        got = oracle.e4m3_decode(c)
        want = pins.e4m3_exact(c)
        if want is None:
            assert math.isnan(got), c
            continue
        assert got == float(want), (hex(c), got, want)
        if want == 0:
            assert math.copysign(1.0, got) == (-1.0 if c & 0x80 else 1.0)


def test_decode_value_set():
    vals = oracle.e4m3_decode_all()
    finite = vals[~np.isnan(vals)]
    assert np.isnan(vals).sum() == 2          # 0x7F and 0xFF only
    assert finite.max() == 448.0 and finite.min() == -448.0
    assert np.min(np.abs(finite[finite != 0])) == 2.0 ** -9
    assert len(set(finite.tolist())) == 253   # 254 codes, +0 and -0 compare equal


def test_encode_roundtrips_every_finite_code():
    # [P2] test_f8_e4m3: encode(decode(c)) == c for every code that is not NaN.
    vals = oracle.e4m3_decode_all()
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    got = oracle.e4m3_encode_array(vals[codes].astype(np.float32))
    np.testing.assert_array_equal(got, codes.astype(np.uint8))


def test_encode_matches_brute_force_on_every_bf16_pattern():
    x = pins.all_bf16_as_f32()
    got = oracle.e4m3_encode_array(x)
    want = pins.brute_encode(x)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(hex(int(i)), float(x[i]), hex(got[i]), hex(want[i])) for i in bad[:10]]


def test_encode_matches_brute_force_on_random_f32_patterns():
    rng = np.random.Generator(np.random.PCG64(7))
    bits = rng.integers(0, 1 << 32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    # also values concentrated where E4M3 lives, which random bit patterns rarely hit
    y = (rng.standard_normal(1_000_000) * np.exp2(rng.uniform(-12, 10, 1_000_000))).astype(np.float32)
    for arr in (x, y):
        got = oracle.e4m3_encode_array(arr)
        want = pins.brute_encode(arr)
        assert np.array_equal(got, want)


def test_encode_midpoints_go_to_even_and_neighbours_do_not():
    vals = pins.POS_VALUES
    for c in range(0x7E):
        m = np.float32((vals[c] + vals[c + 1]) / 2)
        assert float(m) == (vals[c] + vals[c + 1]) / 2  # midpoints are exact in float32
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(m) == even, hex(c)
        assert oracle.e4m3_encode(-m) == (even | 0x80)
        up = np.nextafter(m, np.float32(np.inf))
        dn = np.nextafter(m, np.float32(0))
        assert oracle.e4m3_encode(up) == c + 1
        assert oracle.e4m3_encode(dn) == c


def test_encode_named_rounding_cases():
    # 432 lies halfway between 416 (0x7D, odd mantissa) and 448 (0x7E, even).
    assert oracle.e4m3_encode(432.0) == 0x7E
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02   # 1.5 steps -> 2
    assert oracle.e4m3_encode(5 * 2.0 ** -10) == 0x02   # 2.5 steps -> 2
    assert oracle.e4m3_encode(7 * 2.0 ** -10) == 0x04   # 3.5 steps -> 4
    assert oracle.e4m3_encode(15 * 2.0 ** -10) == 0x08  # 7.5 steps -> smallest normal
    assert oracle.e4m3_encode(1.0625) == 0x38           # tie between 1.0 and 1.125 -> 1.0
    assert oracle.e4m3_encode(1.1875) == 0x3A           # tie between 1.125 and 1.25 -> 1.25
    assert oracle.e4m3_encode(464.0) == 0x7E            # past the last midpoint: saturate
    assert oracle.e4m3_encode(np.float32(1e-40)) == 0x00  # float32 subnormal input
    assert oracle.e4m3_encode(np.float32(-1e-40)) == 0x80


def test_f32_to_bf16_matches_torch_rounding():
    rng = np.random.Generator(np.random.PCG64(11))
    bits = rng.integers(0, 1 << 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # ties: low 16 bits exactly 0x8000 with odd and even kept halves
    ties = (np.arange(4096, dtype=np.uint32) << 17) | 0x8000
    bits = np.concatenate([bits, ties, ties | 0x10000])
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f32_to_bf16(float(v)) for v in x[:20000]], dtype=np.uint16)
    np.testing.assert_array_equal(got, want[:20000])
    got_t = np.array([oracle.f32_to_bf16(float(v)) for v in x[-8192:]], dtype=np.uint16)
    np.testing.assert_array_equal(got_t, want[-8192:])


@pytest.mark.slow
def test_encode_matches_brute_force_on_every_f32_pattern():
    step = 1 << 24
    for start in range(0, 1 << 32, step):
        bits = np.arange(start, start + step, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        assert np.array_equal(oracle.e4m3_encode_array(x), pins.brute_encode(x)), hex(start)
