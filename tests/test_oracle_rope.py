"""Pins for the oracle's rope + cache write (CPU only).

The fused write rotates K by its position (rope, from a caller-supplied fp32 cos/sin
table) and then stores it like reshape_and_cache ([P1] llama-graph.cpp build_attn:
"rope fusion which directly writes into k-v cache").  Pinned by exact special angles
(identity, quarter turn), the NeoX/GPT-J layouts being one permutation apart, an
elementwise float32 restatement, norm preservation and pass-through dims.
"""
import numpy as np
import pytest
import torch

import oracle


def _table(max_pos, rot, base=10000.0):
    inv = (base ** (-np.arange(0, rot, 2, dtype=np.float64) / rot))
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def _bf16(a):
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def _store(k, v, slots, nb, bs, ks, vs, table=None, pos=None, rot=None, neox=True):
    n, n_kv, hd = k.shape
    kc = np.full((nb, bs, n_kv, hd), 0x5A, np.uint8)
    vc = kc.copy()
    if table is None:
        st = oracle.reshape_and_cache(k, v, kc, vc, slots, bs, ks, vs)
    else:
        st = oracle.rope_reshape_and_cache(k, v, kc, vc, slots, pos, table, rot, neox, bs, ks, vs)
    assert st == 0
    return kc, vc


def test_identity_angle_is_a_plain_store():
    rng = np.random.default_rng(1)
    k = _bf16(rng.standard_normal((20, 2, 64)))
    v = _bf16(rng.standard_normal((20, 2, 64)))
    slots = rng.permutation(32)[:20].astype(np.int64)
    table = np.concatenate([np.ones((4, 32)), np.zeros((4, 32))], axis=1).astype(np.float32)
    pos = rng.integers(0, 4, 20)
    for neox in (True, False):
        a = _store(k, v, slots, 2, 16, 0.05, 0.04)
        b = _store(k, v, slots, 2, 16, 0.05, 0.04, table, pos, 64, neox)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("neox", [True, False])
def test_quarter_turn_permutes_exactly(neox):
    # cos = 0, sin = 1: (a, b) -> (-b, a) with no rounding at all
    rng = np.random.default_rng(2)
    k = rng.standard_normal((8, 1, 16)).astype(np.float32)
    table = np.concatenate([np.zeros((1, 8)), np.ones((1, 8))], axis=1).astype(np.float32)
    want = k.copy()
    if neox:
        want[..., :8], want[..., 8:] = -k[..., 8:], k[..., :8]
    else:
        want[..., 0::2], want[..., 1::2] = -k[..., 1::2], k[..., 0::2]
    for row in range(8):
        got = oracle.rope(k[row, 0], table[0], 16, neox)
        np.testing.assert_array_equal(got, want[row, 0])
    slots = np.arange(8, dtype=np.int64)
    kc = np.zeros((8, 1, 1, 16), np.uint8)
    oracle.rope_reshape_and_cache(k, k, kc, kc.copy(), slots, np.zeros(8, np.int64), table, 16, neox,
                                  1, 0.5, 0.5, src_dtype=oracle.F32)
    np.testing.assert_array_equal(kc.reshape(8, 16),
                                  oracle.e4m3_encode_array(want.reshape(-1) / np.float32(0.5)).reshape(8, 16))


def test_neox_and_gptj_are_one_permutation_apart():
    rng = np.random.default_rng(3)
    rot, hd = 64, 128
    table = _table(50, rot)
    perm = np.empty(rot, np.int64)  # GPT-J position of NeoX dim
    perm[0::2] = np.arange(rot // 2)
    perm[1::2] = np.arange(rot // 2) + rot // 2
    for _ in range(20):
        x = rng.standard_normal(hd).astype(np.float32)
        p = int(rng.integers(0, 50))
        neox = oracle.rope(x, table[p], rot, True)
        xg = x.copy()
        xg[:rot] = x[perm]
        gptj = oracle.rope(xg, table[p], rot, False)
        back = gptj.copy()
        back[perm] = gptj[:rot]
        np.testing.assert_array_equal(neox[:rot], back[:rot])
        np.testing.assert_array_equal(neox[rot:], x[rot:])  # pass-through dims


def test_elementwise_float32_restatement():
    rng = np.random.default_rng(4)
    rot = 128
    table = _table(300, rot)
    x = rng.standard_normal((300, rot)).astype(np.float32)
    c, s = table[:, :64], table[:, 64:]
    a, b = x[:, :64], x[:, 64:]
    want = np.concatenate([(a * c) - (b * s), (a * s) + (b * c)], axis=1)  # float32, no fusing
    got = np.stack([oracle.rope(x[i], table[i], rot, True) for i in range(300)])
    np.testing.assert_array_equal(got, want)
    n0 = np.sum(x.astype(np.float64) ** 2, axis=1)
    n1 = np.sum(got.astype(np.float64) ** 2, axis=1)
    np.testing.assert_allclose(n1, n0, rtol=1e-5)  # a rotation keeps the norm


def test_bad_position_is_flagged():
    k = _bf16(np.ones((3, 1, 16)))
    kc = np.zeros((4, 1, 1, 16), np.uint8)
    st = oracle.rope_reshape_and_cache(k, k, kc, kc.copy(), np.arange(3), np.array([0, 5, -1]),
                                       _table(4, 16), 16, True, 1, 1.0, 1.0)
    assert st == oracle.STATUS_BAD_SLOT
