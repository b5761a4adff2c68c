"""Pins for the oracle's paged decode attention (CPU only).

Definition followed by the oracle: [P1] llama.cpp commit "llama : Add FP8
KV-cache support (#28392)", tests/test-fp8.cpp check_fp8_attention (double
precision softmax(q.k/sqrt(d)) V on K/V that were divided by the scale, E4M3
rounded and multiplied back).  Pinned here by closed forms (one token, two
tokens, uniform scores), selection of a single dominant token at every
position class of the paged layout, the GQA head grouping, block-table
permutation invariance, and a library softmax on a separately gathered cache.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import workloads

DEC = oracle.e4m3_decode_all()


def _bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _layout(lens, bs, rng, spare=0):
    need = [math.ceil(L / bs) for L in lens]
    nb = sum(need) + spare
    perm = rng.permutation(nb)
    bt = np.full((len(lens), max(need)), -1, np.int32)
    at = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[at:at + n]
        at += n
    return bt, nb


def _fill(cache, bt, bs, seq, rows):
    """Write per-token rows [L, n_kv, hd] (uint8 codes) of one sequence into the cache."""
    for t in range(rows.shape[0]):
        cache[bt[seq, t // bs], t % bs] = rows[t]


def test_single_token_returns_scaled_value_row():
    bs, nkv, hd = 4, 1, 8
    rng = np.random.Generator(np.random.PCG64(1))
    bt, nb = _layout([1], bs, rng, spare=2)
    kc = np.full((nb, bs, nkv, hd), 0x5A, np.uint8)
    vc = kc.copy()
    kcodes = rng.integers(0, 0x7E, size=(1, nkv, hd)).astype(np.uint8)
    vcodes = rng.integers(0, 0x7E, size=(1, nkv, hd)).astype(np.uint8) | 0x80
    _fill(kc, bt, bs, 0, kcodes)
    _fill(vc, bt, bs, 0, vcodes)
    q = _bf16(rng.standard_normal((1, 1, hd)))
    out, st = oracle.paged_decode_attention(q, kc, vc, bt, np.array([1]), 0.05, 0.04)
    assert st == 0
    np.testing.assert_array_equal(out[0, 0], np.float64(np.float32(0.04)) * DEC[vcodes[0, 0]])


def test_two_tokens_follow_the_logistic_closed_form():
    bs, nkv, hd = 2, 1, 4
    rng = np.random.Generator(np.random.PCG64(2))
    bt, nb = _layout([2], bs, rng, spare=3)
    kc = np.zeros((nb, bs, nkv, hd), np.uint8)
    vc = kc.copy()
    k = np.array([[0x38, 0x40, 0xB8, 0x30], [0x30, 0x38, 0x44, 0x28]], np.uint8)  # codes
    v = np.array([[0x38, 0x00, 0x48, 0xC0], [0x40, 0x3C, 0x80, 0x50]], np.uint8)
    _fill(kc, bt, bs, 0, k[:, None, :])
    _fill(vc, bt, bs, 0, v[:, None, :])
    qv = np.array([1.5, -2.0, 0.75, 3.0])
    sk, sv = 0.125, 0.25
    for sm in (0.0, 0.3):
        out, _ = oracle.paged_decode_attention(_bf16(qv[None, None]), kc, vc, bt, np.array([2]),
                                               sk, sv, sm_scale=sm)
        s = 0.5 if sm == 0.0 else 0.3  # 1/sqrt(4)
        d = s * sk * float(np.dot(qv, DEC[k[0]] - DEC[k[1]]))
        w0 = 1.0 / (1.0 + math.exp(-d))
        want = sv * (w0 * DEC[v[0]] + (1.0 - w0) * DEC[v[1]])
        np.testing.assert_allclose(out[0, 0], want, rtol=0, atol=1e-14)


def test_equal_keys_or_zero_query_average_the_values():
    bs, nkv, hd, L = 4, 2, 8, 11
    rng = np.random.Generator(np.random.PCG64(3))
    bt, nb = _layout([L], bs, rng, spare=1)
    kc = np.zeros((nb, bs, nkv, hd), np.uint8)
    vc = np.zeros_like(kc)
    vcodes = rng.integers(0, 0x7E, size=(L, nkv, hd)).astype(np.uint8)
    _fill(vc, bt, bs, 0, vcodes)
    same = np.tile(rng.integers(0, 0x70, size=(1, nkv, hd)).astype(np.uint8), (L, 1, 1))
    _fill(kc, bt, bs, 0, same)
    q = _bf16(rng.standard_normal((1, 4, hd)))
    out, _ = oracle.paged_decode_attention(q, kc, vc, bt, np.array([L]), 0.05, 0.04)
    for h in range(4):
        want = float(np.float32(0.04)) * DEC[vcodes[:, h // 2]].mean(axis=0)
        np.testing.assert_allclose(out[0, h], want, rtol=1e-13, atol=1e-15)
    # zero query, arbitrary keys
    _fill(kc, bt, bs, 0, rng.integers(0, 0x7E, size=(L, nkv, hd)).astype(np.uint8))
    out0, _ = oracle.paged_decode_attention(_bf16(np.zeros((1, 4, hd))), kc, vc, bt,
                                            np.array([L]), 0.05, 0.04)
    np.testing.assert_allclose(out0, out, rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("bs", [4, 16])
def test_dominant_token_is_selected_at_every_position(bs):
    # A block-table or in-page offset mistake (P3's read-side pitfalls: wrong page, offset
    # dropped) selects a different value row and fails here.
    nkv, hd = 1, 16
    L = 3 * bs + 3
    rng = np.random.Generator(np.random.PCG64(4))
    bt, nb = _layout([L], bs, rng, spare=2)
    vcodes = rng.integers(0, 0x60, size=(L, nkv, hd)).astype(np.uint8)
    vc = np.zeros((nb, bs, nkv, hd), np.uint8)
    _fill(vc, bt, bs, 0, vcodes)
    q = _bf16(np.ones((1, 1, hd)))
    for star in sorted({0, 1, bs - 1, bs, bs + 1, 2 * bs - 1, L - 2, L - 1}):
        kcodes = np.zeros((L, nkv, hd), np.uint8)          # all keys 0 -> score 0
        kcodes[star] = 0x7E                                 # 448 in every dim
        kc = np.zeros_like(vc)
        _fill(kc, bt, bs, 0, kcodes)
        out, _ = oracle.paged_decode_attention(q, kc, vc, bt, np.array([L]), 1.0, 0.5)
        # score gap 448*16/4 = 1792, so the other weights are below e^-1700
        np.testing.assert_array_equal(out[0, 0], 0.5 * DEC[vcodes[star, 0]])


def test_gqa_heads_read_their_group_kv_head():
    nq, nkv, hd, bs, L = 8, 4, 8, 4, 5
    rng = np.random.Generator(np.random.PCG64(5))
    bt, nb = _layout([L], bs, rng)
    kc = np.zeros((nb, bs, nkv, hd), np.uint8)
    vc = np.zeros_like(kc)
    vrows = np.zeros((L, nkv, hd), np.uint8)
    for h in range(nkv):
        vrows[:, h, :] = 0x38 + 8 * h   # kv head h holds the constant 2^h in every slot
    _fill(vc, bt, bs, 0, vrows)
    q = _bf16(rng.standard_normal((1, nq, hd)))
    out, _ = oracle.paged_decode_attention(q, kc, vc, bt, np.array([L]), 0.05, 1.0)
    for h in range(nq):
        np.testing.assert_allclose(out[0, h], 2.0 ** (h // (nq // nkv)), rtol=1e-14)


def test_block_permutation_invariance():
    w = workloads.WORKLOADS["tiny"]
    lens = [17, 33, 64, 100]
    k = _bf16(np.random.default_rng(6).standard_normal((sum(lens), w.n_kv, w.head_dim)))
    v = _bf16(np.random.default_rng(7).standard_normal((sum(lens), w.n_kv, w.head_dim)))
    q = _bf16(np.random.default_rng(8).standard_normal((4, w.n_q, w.head_dim)))
    outs = []
    for seed in (1, 2):
        bt, nb = _layout(lens, w.block_size, np.random.Generator(np.random.PCG64(seed)), spare=7)
        slots = np.concatenate([bt[i, np.arange(L) // w.block_size].astype(np.int64) * w.block_size
                                + np.arange(L) % w.block_size for i, L in enumerate(lens)])
        kc = np.full((nb, w.block_size, w.n_kv, w.head_dim), 0x5A, np.uint8)
        vc = kc.copy()
        oracle.reshape_and_cache(k, v, kc, vc, slots, w.block_size, 0.05, 0.04)
        out, st = oracle.paged_decode_attention(q, kc, vc, bt, np.array(lens), 0.05, 0.04)
        assert st == 0
        outs.append(out)
    np.testing.assert_array_equal(outs[0], outs[1])


def test_matches_library_softmax_on_a_gathered_cache():
    # Special case that reduces to library routines: gather the dequantized rows of each
    # sequence, then scipy softmax and a numpy contraction.
    w = workloads.WORKLOADS["tiny"]
    lay = workloads.make_layout(w)
    k, v = workloads.make_kv(w, lay.slot_mapping.size)
    q = workloads.make_query(w, lay.num_seqs)
    kc = workloads.new_cache(lay.num_blocks, w).numpy()
    vc = kc.copy()
    oracle.reshape_and_cache(k, v, kc, vc, lay.slot_mapping, w.block_size, w.k_scale, w.v_scale)
    out, st = oracle.paged_decode_attention(q, kc, vc, lay.block_tables, lay.seq_lens,
                                            w.k_scale, w.v_scale)
    assert st == 0
    G = w.n_q // w.n_kv
    qf = q.float().numpy().astype(np.float64)
    sk, sv = float(np.float32(w.k_scale)), float(np.float32(w.v_scale))
    flat_k = kc.reshape(-1, w.n_kv, w.head_dim)
    flat_v = vc.reshape(-1, w.n_kv, w.head_dim)
    for b in range(lay.num_seqs):
        sl = lay.slot_mapping[lay.row_seq == b]
        Kd = sk * DEC[flat_k[sl]]
        Vd = sv * DEC[flat_v[sl]]
        for h in range(w.n_q):
            s = Kd[:, h // G, :] @ qf[b, h] / math.sqrt(w.head_dim)
            want = scipy.special.softmax(s) @ Vd[:, h // G, :]
            np.testing.assert_allclose(out[b, h], want, rtol=1e-12, atol=1e-14)


def test_scale_swap_changes_the_output():
    # [P3] read-side mutation table: V read with K's scale must not pass.
    w = workloads.WORKLOADS["tiny"]
    lay = workloads.make_layout(w)
    k, v = workloads.make_kv(w, lay.slot_mapping.size)
    q = workloads.make_query(w, lay.num_seqs)
    kc = workloads.new_cache(lay.num_blocks, w).numpy()
    vc = kc.copy()
    oracle.reshape_and_cache(k, v, kc, vc, lay.slot_mapping, w.block_size, w.k_scale, w.v_scale)
    ref, _ = oracle.paged_decode_attention(q, kc, vc, lay.block_tables, lay.seq_lens, 0.05, 0.04)
    for ks, vs in ((0.04, 0.05), (0.05, 0.05), (1.0, 0.04), (0.05, 1.0)):
        alt, _ = oracle.paged_decode_attention(q, kc, vc, lay.block_tables, lay.seq_lens, ks, vs)
        tol = 2e-3 + 1e-2 * np.abs(ref)
        assert np.count_nonzero(np.abs(alt - ref) > tol) > 0


def test_empty_sequence_gives_zeros_and_pairs_match_full():
    w = workloads.WORKLOADS["tiny"]
    lay = workloads.make_layout(w, lengths=[0, 33, 1, 100])
    k, v = workloads.make_kv(w, lay.slot_mapping.size)
    q = workloads.make_query(w, lay.num_seqs)
    kc = workloads.new_cache(lay.num_blocks, w).numpy()
    vc = kc.copy()
    oracle.reshape_and_cache(k, v, kc, vc, lay.slot_mapping, w.block_size, w.k_scale, w.v_scale)
    out, st = oracle.paged_decode_attention(q, kc, vc, lay.block_tables, lay.seq_lens, 0.05, 0.04)
    assert st == 0 and np.all(out[0] == 0)
    pairs = np.array([[b, h] for b in range(4) for h in range(w.n_q)], np.int32)
    pout, _ = oracle.paged_decode_attention_pairs(pairs, q, kc, vc, lay.block_tables,
                                                  lay.seq_lens, 0.05, 0.04)
    np.testing.assert_array_equal(pout.reshape(out.shape), out)


def test_bad_block_id_is_flagged():
    bs, nkv, hd = 4, 1, 8
    kc = np.zeros((2, bs, nkv, hd), np.uint8)
    bt = np.array([[0, 5]], np.int32)
    q = _bf16(np.ones((1, 1, hd)))
    out, st = oracle.paged_decode_attention(q, kc, kc, bt, np.array([6]), 1.0, 1.0)
    assert st == oracle.STATUS_BAD_BLOCK
    _, st2 = oracle.paged_decode_attention(q, kc, kc, bt, np.array([9]), 1.0, 1.0)
    assert st2 & oracle.STATUS_BAD_BLOCK
