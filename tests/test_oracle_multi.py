"""Pins for the oracle's multi-query causal paged attention (CPU only).

[P1] llama.cpp "llama : Add FP8 KV-cache support (#28392)", tests/test-fp8.cpp
check_fp8_attention: a batch of 4 new tokens, each attending to every cached token up to
and including itself.  Pinned by: one query per sequence equals decode attention; equal
keys give the running mean of V over the causal prefix (closed form); a library softmax
with an explicit causal mask on a separately gathered cache.
"""
import math

import numpy as np
import scipy.special
import torch

import oracle
import workloads

DEC = oracle.e4m3_decode_all()


def _setup(lengths, qlens, n_q=8, n_kv=2, hd=32, bs=4, seed=0, same_k=False):
    rng = np.random.default_rng(seed)
    need = [math.ceil(L / bs) for L in lengths]
    nb = sum(need) + 2
    perm = rng.permutation(nb).astype(np.int32)
    bt = np.full((len(lengths), max(need)), -1, np.int32)
    at = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[at:at + n]
        at += n
    kc = rng.integers(0, 0x70, size=(nb, bs, n_kv, hd)).astype(np.uint8)
    vc = rng.integers(0, 0x70, size=(nb, bs, n_kv, hd)).astype(np.uint8)
    if same_k:
        kc[:] = kc[0, 0]
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = torch.as_tensor(rng.standard_normal((int(qsl[-1]), n_q, hd)).astype(np.float32)).to(torch.bfloat16)
    return q, qsl, kc, vc, bt


def test_one_query_per_sequence_is_decode():
    lengths = [5, 17, 40]
    q, qsl, kc, vc, bt = _setup(lengths, [1, 1, 1])
    multi, st = oracle.paged_attention_multi(q, qsl, kc, vc, bt, np.array(lengths), 0.05, 0.04)
    dec, st2 = oracle.paged_decode_attention(q, kc, vc, bt, np.array(lengths), 0.05, 0.04)
    assert st == 0 and st2 == 0
    np.testing.assert_array_equal(multi, dec)


def test_equal_keys_give_the_causal_running_mean():
    lengths, qlens = [9, 12], [4, 3]
    q, qsl, kc, vc, bt = _setup(lengths, qlens, same_k=True, bs=4)
    out, st = oracle.paged_attention_multi(q, qsl, kc, vc, bt, np.array(lengths), 0.05, 0.04)
    assert st == 0
    G = 8 // 2
    for b, (L, n) in enumerate(zip(lengths, qlens)):
        rows = [vc[bt[b, t // 4], t % 4] for t in range(L)]
        for j in range(n):
            p = L - n + j
            for h in range(8):
                want = float(np.float32(0.04)) * np.mean([DEC[r[h // G]] for r in rows[:p + 1]], axis=0)
                np.testing.assert_allclose(out[qsl[b] + j, h], want, rtol=1e-13, atol=1e-15)


def test_library_softmax_with_a_causal_mask():
    lengths, qlens = [13, 30, 4], [4, 2, 4]
    q, qsl, kc, vc, bt = _setup(lengths, qlens, seed=5)
    out, st = oracle.paged_attention_multi(q, qsl, kc, vc, bt, np.array(lengths), 0.125, 0.25)
    assert st == 0
    qf = q.float().numpy().astype(np.float64)
    sk, sv = 0.125, 0.25
    for b, (L, n) in enumerate(zip(lengths, qlens)):
        K = np.stack([sk * DEC[kc[bt[b, t // 4], t % 4]] for t in range(L)])  # [L, n_kv, hd]
        V = np.stack([sv * DEC[vc[bt[b, t // 4], t % 4]] for t in range(L)])
        pos = L - n + np.arange(n)
        mask = np.arange(L)[None, :] <= pos[:, None]  # [n, L]
        for h in range(8):
            s = qf[qsl[b]:qsl[b] + n, h] @ K[:, h // 4].T / math.sqrt(32)
            s = np.where(mask, s, -np.inf)
            want = scipy.special.softmax(s, axis=1) @ V[:, h // 4]
            np.testing.assert_allclose(out[qsl[b]:qsl[b] + n, h], want, rtol=1e-12, atol=1e-14)


def test_more_queries_than_tokens_is_flagged():
    q, qsl, kc, vc, bt = _setup([2], [3])
    out, st = oracle.paged_attention_multi(q, qsl, kc, vc, bt, np.array([2]), 1.0, 1.0)
    assert st == oracle.STATUS_BAD_BLOCK and np.all(out[0] == 0)  # position -1: nothing
