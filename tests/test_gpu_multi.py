"""kvfp8_paged_attention_multi (causal multi-query) on the GPU vs the double-precision oracle.
Tolerance per element: |gpu - oracle| <= 2e-3 + 1e-2 * |oracle|."""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import gpu_util

pytestmark = pytest.mark.gpu

kv = pytest.importorskip("fp8_paged_kv_reshape_gb300")


def _inputs(n_q, n_kv, hd, bs, lengths, qlens, seed):
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
    k = torch.randn(total, n_kv, hd, generator=g).to(torch.bfloat16)
    v = torch.randn(total, n_kv, hd, generator=g).to(torch.bfloat16)
    slots = np.concatenate([bt[i, np.arange(L) // bs].astype(np.int64) * bs + np.arange(L) % bs
                            for i, L in enumerate(lengths)])
    kc = np.full((nb, bs, n_kv, hd), 0x5A, np.uint8)
    vc = kc.copy()
    assert oracle.reshape_and_cache(k, v, kc, vc, slots, bs, 0.05, 0.04) == 0
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    q = torch.randn(int(qsl[-1]), n_q, hd, generator=g).to(torch.bfloat16)
    return q, qsl, kc, vc, bt


def _gpu(q, qsl, qmax, kc, vc, bt, lengths, status=None):
    return kv.paged_attention_multi(q.cuda(), torch.from_numpy(qsl).cuda(), qmax,
                                    torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                                    torch.from_numpy(bt).cuda(),
                                    torch.tensor(lengths, dtype=torch.int32, device="cuda"),
                                    torch.tensor([0.05], device="cuda"),
                                    torch.tensor([0.04], device="cuda"), status=status)


CASES = [
    # name, n_q, n_kv, head_dim, block, lengths, query counts
    ("p1_like_4tok", 4, 4, 64, 16, [4, 30, 257], [4, 4, 4]),
    ("g4_q4_nt2", 32, 8, 128, 16, [1000, 17, 4096, 5], [4, 1, 3, 4]),
    ("g8_q2", 64, 8, 128, 16, [300, 2, 64], [2, 2, 1]),
    ("g5_q3_bs32", 40, 8, 128, 32, [700, 33, 1024], [3, 3, 2]),
    ("g2_hd256_q4", 4, 2, 256, 64, [129, 300], [4, 4]),
    ("g1_q16", 8, 8, 128, 8, [100, 16], [16, 16]),
    ("zero_queries", 32, 8, 128, 16, [50, 80, 0], [0, 3, 0]),
    ("mha16_head_groups_q1", 16, 16, 128, 16, [300, 33], [1, 1]),
    ("g2_12_kv_heads_q8", 24, 12, 64, 16, [200, 100], [8, 5]),
    # 16 columns at head_dim 128: head groups of 3 (6 kv heads) and of 1 kv head
    ("g4_q4_six_kv_heads", 24, 6, 128, 16, [700, 64], [4, 3]),
    ("g16_q1_one_kv_head", 16, 1, 128, 16, [500, 90], [1, 1]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_multi_query_against_oracle(case):
    name, n_q, n_kv, hd, bs, lengths, qlens = case
    q, qsl, kc, vc, bt = _inputs(n_q, n_kv, hd, bs, lengths, qlens, seed=len(name))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _gpu(q, qsl, max(max(qlens), 1), kc, vc, bt, lengths, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, s2 = oracle.paged_attention_multi(q, qsl, kc, vc, bt, np.array(lengths), 0.05, 0.04)
    assert s2 == 0
    gpu_util.assert_attention_close(out, ref, name)


def test_long_sequence_split_over_many_ctas():
    q, qsl, kc, vc, bt = _inputs(32, 8, 128, 16, [60_000, 300], [4, 2], seed=3)
    out = _gpu(q, qsl, 4, kc, vc, bt, [60_000, 300])
    ref, _ = oracle.paged_attention_multi(q, qsl, kc, vc, bt, np.array([60_000, 300]), 0.05, 0.04)
    gpu_util.assert_attention_close(out, ref, "long")


def test_one_query_each_matches_the_decode_entry_point():
    lengths = [333, 17, 4096]
    q, qsl, kc, vc, bt = _inputs(32, 8, 128, 16, lengths, [1, 1, 1], seed=4)
    multi = _gpu(q, qsl, 1, kc, vc, bt, lengths)
    dec = kv.paged_decode_attention(q.cuda(), torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda(),
                                    torch.from_numpy(bt).cuda(),
                                    torch.tensor(lengths, dtype=torch.int32, device="cuda"),
                                    torch.tensor([0.05], device="cuda"),
                                    torch.tensor([0.04], device="cuda"))
    assert torch.equal(multi, dec)


def test_out_of_range_query_rows_are_flagged_and_skipped():
    lengths = [40, 40]
    q, qsl, kc, vc, bt = _inputs(8, 2, 64, 16, lengths, [2, 2], seed=5)
    bad = np.array([0, 2, 9], np.int32)  # second sequence claims rows past the 4 that exist
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((4, 8, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    kv.paged_attention_multi(q.cuda(), torch.from_numpy(bad).cuda(), 4, torch.from_numpy(kc).cuda(),
                             torch.from_numpy(vc).cuda(), torch.from_numpy(bt).cuda(),
                             torch.tensor(lengths, dtype=torch.int32, device="cuda"),
                             torch.tensor([0.05], device="cuda"), torch.tensor([0.04], device="cuda"),
                             out=out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & kv.DEV_BAD_BLOCK
    assert bool((out[2:] == 7.0).all())          # the bad sequence's rows were not touched
    ref, _ = oracle.paged_attention_multi(q[:2], np.array([0, 2], np.int32), kc, vc, bt[:1],
                                          np.array([40]), 0.05, 0.04)
    gpu_util.assert_attention_close(out[:2], ref, "good sequence")
