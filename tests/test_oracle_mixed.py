"""Pins for the oracle's mixed cache dtypes (CPU only): FP8 on K only, on V only, or on
both ([P1] tests/test-fp8.cpp check_fp8_attention, scaled = 1/2/3; the non-FP8 side is
kept at 16 bits and unscaled -- here bf16)."""
import math

import numpy as np
import torch

import oracle


def _setup(lengths, seed, n_q=8, n_kv=2, hd=32, bs=4):
    rng = np.random.default_rng(seed)
    need = [math.ceil(L / bs) for L in lengths]
    nb = sum(need) + 1
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((len(lengths), max(need)), -1, np.int32)
    at = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[at:at + n]
        at += n
    total = sum(lengths)
    k = torch.as_tensor(rng.standard_normal((total, n_kv, hd)).astype(np.float32)).to(torch.bfloat16)
    v = torch.as_tensor(rng.standard_normal((total, n_kv, hd)).astype(np.float32)).to(torch.bfloat16)
    q = torch.as_tensor(rng.standard_normal((len(lengths), n_q, hd)).astype(np.float32)).to(torch.bfloat16)
    slots = np.concatenate([bt[i, np.arange(L) // bs].astype(np.int64) * bs + np.arange(L) % bs
                            for i, L in enumerate(lengths)])
    return k, v, q, bt, slots, nb


def _caches(nb, kinds, shape=(4, 2, 32)):
    return [np.zeros((nb, *shape), np.uint8 if kind == oracle.E4M3 else np.uint16) for kind in kinds]


def test_both_fp8_equals_the_fp8_path():
    lengths = [5, 13, 30]
    k, v, q, bt, slots, nb = _setup(lengths, 1)
    kc, vc = _caches(nb, (oracle.E4M3, oracle.E4M3))
    assert oracle.reshape_and_cache_mixed(k, v, kc, oracle.E4M3, vc, oracle.E4M3, slots, 4, 0.05, 0.04) == 0
    kc2, vc2 = np.zeros_like(kc), np.zeros_like(vc)
    oracle.reshape_and_cache(k, v, kc2, vc2, slots, 4, 0.05, 0.04)
    np.testing.assert_array_equal(kc, kc2)
    np.testing.assert_array_equal(vc, vc2)
    a, _ = oracle.paged_decode_attention_mixed(q, kc, oracle.E4M3, vc, oracle.E4M3, bt, np.array(lengths), 0.05, 0.04)
    b, _ = oracle.paged_decode_attention(q, kc, vc, bt, np.array(lengths), 0.05, 0.04)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)


def test_bf16_side_is_the_source_value_and_ignores_its_scale():
    lengths = [9, 20]
    k, v, q, bt, slots, nb = _setup(lengths, 2)
    kc, vc = _caches(nb, (oracle.CACHE_BF16, oracle.E4M3))
    oracle.reshape_and_cache_mixed(k, v, kc, oracle.CACHE_BF16, vc, oracle.E4M3, slots, 4, 7.0, 0.04)
    flat = kc.reshape(-1, 2, 32)
    np.testing.assert_array_equal(flat[slots], k.view(torch.int16).numpy().view(np.uint16))
    out1, _ = oracle.paged_decode_attention_mixed(q, kc, oracle.CACHE_BF16, vc, oracle.E4M3, bt,
                                                  np.array(lengths), 7.0, 0.04)
    out2, _ = oracle.paged_decode_attention_mixed(q, kc, oracle.CACHE_BF16, vc, oracle.E4M3, bt,
                                                  np.array(lengths), 0.5, 0.04)
    np.testing.assert_array_equal(out1, out2)  # the bf16 side carries no scale


def test_library_softmax_on_each_mix():
    import scipy.special
    DEC = oracle.e4m3_decode_all()
    lengths = [7, 33]
    k, v, q, bt, slots, nb = _setup(lengths, 3)
    for kinds in ((oracle.CACHE_BF16, oracle.E4M3), (oracle.E4M3, oracle.CACHE_BF16)):
        kc, vc = _caches(nb, kinds)
        oracle.reshape_and_cache_mixed(k, v, kc, kinds[0], vc, kinds[1], slots, 4, 0.125, 0.25)
        out, st = oracle.paged_decode_attention_mixed(q, kc, kinds[0], vc, kinds[1], bt,
                                                      np.array(lengths), 0.125, 0.25)
        assert st == 0

        def val(c, kind, s):
            if kind == oracle.E4M3:
                return s * DEC[c]
            return (c.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        fk, fv = kc.reshape(-1, 2, 32), vc.reshape(-1, 2, 32)
        qf = q.float().numpy().astype(np.float64)
        start = 0
        for b, L in enumerate(lengths):
            sl = slots[start:start + L]
            start += L
            K, V = val(fk[sl], kinds[0], 0.125), val(fv[sl], kinds[1], 0.25)
            for h in range(8):
                s = K[:, h // 4] @ qf[b, h] / math.sqrt(32)
                np.testing.assert_allclose(out[b, h], scipy.special.softmax(s) @ V[:, h // 4],
                                           rtol=1e-12, atol=1e-14)


def _multi_setup(lengths, nbs, seed):
    k, v, _, bt, slots, nb = _setup(lengths, seed)
    rng = np.random.default_rng(seed + 100)
    qsl = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int32)
    q = torch.as_tensor(rng.standard_normal((int(qsl[-1]), 8, 32)).astype(np.float32)).to(torch.bfloat16)
    return k, v, q, bt, slots, nb, qsl


def test_multi_mixed_with_a_bf16_side_holding_fp8_values_equals_the_fp8_multi_form():
    # E4M3 values are exact in bf16: a bf16 side holding dec(code) (scale 1) must give the
    # all-FP8 causal multi-query result -- a check against the separately pinned FP8 form
    lengths, nbs = [6, 17, 30], [3, 1, 5]
    k, v, q, bt, slots, nb, qsl = _multi_setup(lengths, nbs, 5)
    kc8, vc8 = _caches(nb, (oracle.E4M3, oracle.E4M3))
    oracle.reshape_and_cache(k, v, kc8, vc8, slots, 4, 1.0, 0.04)
    DEC = oracle.e4m3_decode_all()
    as_bf16 = lambda c: (DEC[c].astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # noqa: E731
    assert np.array_equal((as_bf16(kc8).astype(np.uint32) << 16).view(np.float32), DEC[kc8].astype(np.float32))
    ref, st = oracle.paged_attention_multi(q, qsl, kc8, vc8, bt, np.array(lengths), 1.0, 0.04)
    assert st == 0
    got, st = oracle.paged_attention_multi_mixed(q, qsl, as_bf16(kc8), oracle.CACHE_BF16, vc8,
                                                 oracle.E4M3, bt, np.array(lengths), 123.0, 0.04)
    assert st == 0
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)
    ref_v, _ = oracle.paged_attention_multi(q, qsl, kc8, vc8, bt, np.array(lengths), 1.0, 1.0)
    got_v, _ = oracle.paged_attention_multi_mixed(q, qsl, kc8, oracle.E4M3, as_bf16(vc8),
                                                  oracle.CACHE_BF16, bt, np.array(lengths), 1.0, 9.0)
    np.testing.assert_allclose(got_v, ref_v, rtol=1e-12, atol=1e-15)


def test_multi_mixed_is_causal_and_its_first_token_sees_one_key():
    lengths, nbs = [12, 9], [12, 4]
    k, v, q, bt, slots, nb, qsl = _multi_setup(lengths, nbs, 6)
    kinds = (oracle.CACHE_BF16, oracle.E4M3)
    kc, vc = _caches(nb, kinds)
    oracle.reshape_and_cache_mixed(k, v, kc, kinds[0], vc, kinds[1], slots, 4, 0.05, 0.25)
    out, st = oracle.paged_attention_multi_mixed(q, qsl, kc, kinds[0], vc, kinds[1], bt,
                                                 np.array(lengths), 0.05, 0.25)
    assert st == 0
    # sequence 0's first query token sits at position 0: its output is V_0 itself
    DEC = oracle.e4m3_decode_all()
    v0 = 0.25 * DEC[vc.reshape(-1, 2, 32)[slots[0]]]
    for h in range(8):
        np.testing.assert_allclose(out[0, h], v0[h // 4], rtol=0, atol=1e-15)
    # rows past a token's position do not change its output
    fk = kc.reshape(-1, 2, 32)
    fk[slots[12 + 8]] ^= 0x1234  # sequence 1's last token (position 8)
    out2, _ = oracle.paged_attention_multi_mixed(q, qsl, kc, kinds[0], vc, kinds[1], bt,
                                                 np.array(lengths), 0.05, 0.25)
    np.testing.assert_array_equal(out2[:12 + 3], out[:12 + 3])  # every row before it
    assert not np.array_equal(out2[12 + 3], out[12 + 3])      # the row at position 8 sees it
