"""kvfp8_paged_attention_multi on its tensor-core (tcgen05) kernel: query chunks longer than
the split-KV decode kernel's 16 score columns per kv head (8 at head_dim 256), vs the
double-precision oracle.
Tolerance per element: |gpu - oracle| <= 2e-3 + 1e-2 * |oracle|."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import gpu_util

pytestmark = pytest.mark.gpu

kv = pytest.importorskip("fp8_paged_kv_reshape_gb300")


def _inputs(n_q, n_kv, hd, bs, lengths, qlens, seed, k_fn=None, q_fn=None):
    g = torch.Generator().manual_seed(seed)
    need = [math.ceil(L / bs) for L in lengths]
    nb = sum(need) + 3
    perm = torch.randperm(nb, generator=g).numpy().astype(np.int32)
    bt = np.full((len(lengths), max(1, max(need))), -1, np.int32)
    at = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[at:at + n]
        at += n
    total = sum(lengths)
    k = torch.randn(total, n_kv, hd, generator=g)
    v = torch.randn(total, n_kv, hd, generator=g).to(torch.bfloat16)
    pos = np.concatenate([np.arange(L) for L in lengths]) if total else np.zeros(0, np.int64)
    if k_fn is not None:
        k = k_fn(k, torch.from_numpy(pos))
    k = k.to(torch.bfloat16)
    slots = np.concatenate([bt[i, np.arange(L) // bs].astype(np.int64) * bs + np.arange(L) % bs
                            for i, L in enumerate(lengths)]) if total else np.zeros(0, np.int64)
    kc = np.full((nb, bs, n_kv, hd), 0x5A, np.uint8)
    vc = kc.copy()
    assert oracle.reshape_and_cache(k, v, kc, vc, slots, bs, 0.05, 0.04) == 0
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = torch.randn(int(qsl[-1]), n_q, hd, generator=g)
    if q_fn is not None:
        q = q_fn(q)
    return q.to(torch.bfloat16), qsl, kc, vc, bt


def _run(n_q, n_kv, hd, bs, lengths, qlens, seed, expect_status=0, **kw):
    q, qsl, kc, vc, bt = _inputs(n_q, n_kv, hd, bs, lengths, qlens, seed, **kw)
    qmax = max(max(qlens), 1)
    assert kv.paged_attention_multi_workspace_size(len(lengths), n_q, n_kv, hd, qmax) == 0
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((q.shape[0], n_q, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    kv.paged_attention_multi(q.cuda(), torch.from_numpy(qsl).cuda(), qmax,
                             torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                             torch.from_numpy(bt).cuda(),
                             torch.tensor(lengths, dtype=torch.int32, device="cuda"),
                             torch.tensor([0.05], device="cuda"), torch.tensor([0.04], device="cuda"),
                             out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    ref, s2 = oracle.paged_attention_multi(q, qsl, kc, vc, bt, np.array(lengths), 0.05, 0.04)
    assert s2 == expect_status
    return out, ref


CASES = [
    # name, n_q, n_kv, head_dim, block, lengths, query counts
    ("g4_q32", 32, 8, 128, 16, [1000, 64, 4096], [32, 5, 17]),
    ("g4_many_tiles", 32, 8, 128, 16, [2000, 150], [100, 150]),
    ("g8_q9", 64, 8, 128, 16, [333, 9, 70], [9, 9, 3]),
    ("g5_rows_straddle_tiles", 40, 8, 128, 32, [700, 100], [60, 100]),
    ("mha_16_kv_heads", 16, 16, 128, 16, [300, 40], [20, 40]),
    ("hd64_g2", 8, 4, 64, 16, [500, 77], [40, 77]),
    ("hd256_g2", 4, 2, 256, 64, [300, 129], [10, 129]),
    ("bs8", 16, 4, 128, 8, [250, 31], [31, 31]),
    ("bs256", 32, 8, 128, 256, [600, 1], [64, 1]),
    ("prefill_from_empty", 32, 8, 128, 16, [50, 200], [50, 200]),
    ("zero_query_sequences", 32, 8, 128, 16, [80, 0, 300, 5], [0, 0, 40, 5]),
    ("g128_one_token_per_tile", 128, 1, 64, 16, [90], [6]),
    ("bs8_two_row_tiles", 16, 4, 128, 8, [700, 90], [90, 40]),
    ("hd64_long_rotated_passes", 16, 8, 64, 16, [3000, 129], [300, 129]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_prefill_against_oracle(case):
    name, n_q, n_kv, hd, bs, lengths, qlens = case
    out, ref = _run(n_q, n_kv, hd, bs, lengths, qlens, seed=len(name) * 13)
    gpu_util.assert_attention_close(out, ref, name)


@pytest.mark.parametrize("n_q,n_kv,hd,qlen", [(32, 8, 128, 5), (8, 2, 64, 40)],
                         ids=["20_rows", "160_rows"])
def test_many_sequences_of_mixed_lengths_run_longest_first(n_q, n_kv, hd, qlen):
    # The CTAs take the sequences longest first, each CTA ranking every sequence's length
    # itself.  470 sequences are more than a CTA's 448 threads, so its lookup of the
    # sequence of a given rank takes two rounds; lengths repeat within a length bucket, and
    # a few sequences are empty.  Every row must land where it belongs (the output starts
    # as NaN, so a row that no CTA writes fails the comparison).
    rng = np.random.default_rng(qlen)
    lengths = rng.integers(qlen, 120, 470)
    lengths[rng.choice(470, 6, replace=False)] = 0
    qlens = np.where(lengths > 0, qlen, 0)
    out, ref = _run(n_q, n_kv, hd, 16, lengths.tolist(), qlens.tolist(), seed=qlen)
    gpu_util.assert_attention_close(out, ref, "470 sequences, %d query tokens" % qlen)


def test_growing_scores_take_the_rescale_path():
    # scores rise by about 0.3 per key, so the running maximum grows by far more than 2^8
    # from one key tile to the next and O is rescaled in tensor memory
    lengths, qlens = [700, 300], [40, 20]
    q_fn = lambda q: torch.ones_like(q)                                    # noqa: E731
    k_fn = lambda k, pos: (pos.float() * 0.03)[:, None, None].expand_as(k) + 0.1 * k  # noqa: E731
    out, ref = _run(32, 8, 128, 16, lengths, qlens, seed=7, k_fn=k_fn, q_fn=q_fn)
    gpu_util.assert_attention_close(out, ref, "rescale")


def test_growing_scores_rescale_with_one_row_tile():
    # 80 rows per kv head (prefill_kernel, one row tile of 64-key tiles): the rescale waits
    # for the previous tile's O product through that tile's buffer release
    lengths, qlens = [900, 300], [20, 11]
    q_fn = lambda q: torch.ones_like(q)                                    # noqa: E731
    k_fn = lambda k, pos: (pos.float() * 0.03)[:, None, None].expand_as(k) + 0.1 * k  # noqa: E731
    out, ref = _run(32, 8, 128, 16, lengths, qlens, seed=8, k_fn=k_fn, q_fn=q_fn)
    gpu_util.assert_attention_close(out, ref, "rescale, one row tile")


def test_more_new_tokens_than_cached_are_flagged_and_give_zero_rows():
    out, ref = _run(32, 8, 128, 16, [5, 300], [20, 40], seed=9, expect_status=kv.DEV_BAD_BLOCK)
    gpu_util.assert_attention_close(out, ref, "n_b > L")
    assert torch.count_nonzero(out[:15]).item() == 0  # positions below zero see no key


def test_prefill_kernel_agrees_with_the_split_kv_kernel_where_both_apply():
    # 16 score columns go to the split-KV kernel; 17 to the tensor cores: compare each
    # against the oracle on the same cache
    lengths = [400, 64]
    for qlens in ([4, 4], [5, 3]):  # G = 4: 16 and 20 columns
        q, qsl, kc, vc, bt = _inputs(32, 8, 128, 16, lengths, qlens, seed=11)
        qmax = max(qlens)
        used_ws = kv.paged_attention_multi_workspace_size(2, 32, 8, 128, qmax)
        out = kv.paged_attention_multi(q.cuda(), torch.from_numpy(qsl).cuda(), qmax,
                                       torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                                       torch.from_numpy(bt).cuda(),
                                       torch.tensor(lengths, dtype=torch.int32, device="cuda"),
                                       torch.tensor([0.05], device="cuda"),
                                       torch.tensor([0.04], device="cuda"))
        ref, _ = oracle.paged_attention_multi(q, qsl, kc, vc, bt, np.array(lengths), 0.05, 0.04)
        gpu_util.assert_attention_close(out, ref, "qmax %d (workspace %d)" % (qmax, used_ws))
