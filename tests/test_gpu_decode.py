"""kvfp8_paged_decode_attention on the GPU vs the double-precision CPU oracle.

Tolerance (per element): |gpu - oracle| <= 2e-3 + 1e-2 * |oracle|.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_util

pytestmark = pytest.mark.gpu

kv = pytest.importorskip("fp8_paged_kv_reshape_gb300")


def _case(n_q, n_kv, hd, bs, lengths, seed, ks=0.05, vs=0.04, kv_std=1.0, spare_blocks=3,
          sdt=torch.float32, sm_scale=0.0, null_scales=False):
    """Random inputs; the cache is written by the oracle (so decode is tested alone) and
    copied to the GPU; returns GPU output and oracle output."""
    g = torch.Generator().manual_seed(seed)
    lengths = list(lengths)
    need = [math.ceil(L / bs) for L in lengths]
    nb = sum(need) + spare_blocks
    perm = torch.randperm(nb, generator=g).numpy().astype(np.int32)
    maxb = max(1, max(need) if need else 1)
    bt = np.full((len(lengths), maxb), -1, np.int32)
    at = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[at:at + n]
        at += n
    total = sum(lengths)
    k = (torch.randn(total, n_kv, hd, generator=g) * kv_std).to(torch.bfloat16)
    v = (torch.randn(total, n_kv, hd, generator=g) * kv_std).to(torch.bfloat16)
    q = torch.randn(len(lengths), n_q, hd, generator=g).to(torch.bfloat16)
    slots = np.concatenate([bt[i, np.arange(L) // bs].astype(np.int64) * bs + np.arange(L) % bs
                            for i, L in enumerate(lengths)]) if total else np.zeros(0, np.int64)
    ksf = workloads.stored_scale(ks, "f32" if sdt == torch.float32 else "bf16")
    vsf = workloads.stored_scale(vs, "f32" if sdt == torch.float32 else "bf16")
    if null_scales:
        ksf = vsf = 1.0
    kc = np.full((nb, bs, n_kv, hd), workloads.SENTINEL, np.uint8)
    vc = kc.copy()
    assert oracle.reshape_and_cache(k, v, kc, vc, slots, bs, ksf, vsf) == 0
    ref, st = oracle.paged_decode_attention(q, kc, vc, bt, np.array(lengths, np.int32), ksf, vsf,
                                            sm_scale)
    assert st == 0
    ksc = None if null_scales else torch.tensor([ks], dtype=sdt, device="cuda")
    vsc = None if null_scales else torch.tensor([vs], dtype=sdt, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kv.paged_decode_attention(q.cuda(), torch.from_numpy(kc).cuda(),
                                    torch.from_numpy(vc).cuda(), torch.from_numpy(bt).cuda(),
                                    torch.tensor(lengths, dtype=torch.int32, device="cuda"), ksc,
                                    vsc, sm_scale=sm_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, ref


CASES = [
    # name, n_q, n_kv, head_dim, block_size, lengths
    ("g4_ragged", 32, 8, 128, 16, [1, 15, 16, 17, 31, 33, 100, 257, 1000, 4096]),
    ("g8", 64, 8, 128, 16, [5, 3000, 70, 2]),
    ("g5_bs32", 40, 8, 128, 32, [16, 17, 1023, 2048, 33, 0, 64]),
    ("g1_hd64_bs8", 4, 4, 64, 8, [1, 7, 8, 9, 200]),
    ("g2_hd64", 4, 2, 64, 16, [17, 33, 64, 100]),
    ("g16_nt2", 32, 2, 128, 16, [50, 500]),
    ("g12_hd64_nt2", 24, 2, 64, 16, [77, 1234]),
    ("g2_hd256_bs64", 4, 2, 256, 64, [65, 300, 1]),
    ("mha_g1", 8, 8, 128, 16, [40, 129]),
    ("bs128", 32, 8, 128, 128, [300, 1000, 129]),
    ("bs256_g6", 24, 4, 128, 256, [700, 5]),
    # more than 8 kv heads: head groups of 8 (32 = 4 x 8), 6 (12 = 2 x 6), 5 (10 = 2 x 5)
    ("mha_32_kv_heads", 32, 32, 128, 16, [300, 1000, 17]),
    ("g2_12_kv_heads_bs8", 24, 12, 64, 8, [129, 40]),
    ("g4_10_kv_heads_hd256", 40, 10, 256, 32, [200, 65]),
    ("g1_16_kv_heads_hd64", 16, 16, 64, 16, [5000, 1]),
    # groups past the split-KV kernel's 16 columns (8 at head_dim 256): tensor-core kernel
    ("g32_tensor_route", 64, 2, 128, 16, [700, 33, 0]),
    ("g12_hd256_tensor_route", 24, 2, 256, 64, [300, 5]),
    ("g128_tensor_route", 128, 1, 64, 16, [90, 17]),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_shapes_against_oracle(case):
    name, n_q, n_kv, hd, bs, lengths = case
    out, ref = _case(n_q, n_kv, hd, bs, lengths, seed=hash(name) % 1000)
    gpu_util.assert_attention_close(out, ref, name)


def test_one_long_sequence_spans_every_cta():
    out, ref = _case(32, 8, 128, 16, [100_003], seed=11)
    gpu_util.assert_attention_close(out, ref, "one_long")


def test_many_short_sequences():
    lengths = [1] * 2000 + [17] * 50 + [0] * 10 + [16] * 40
    out, ref = _case(16, 4, 64, 16, lengths, seed=12)
    gpu_util.assert_attention_close(out, ref, "many_short")


def test_more_sequences_than_the_plan_keeps_in_shared_memory():
    # the plan kernel searches its chunk prefix in shared memory up to 4096 sequences and in
    # global memory beyond; lengths 0..40 give empty, one-chunk and multi-chunk sequences
    lengths = list(np.random.default_rng(16).integers(0, 41, 5000))
    out, ref = _case(8, 2, 64, 16, lengths, seed=16)
    gpu_util.assert_attention_close(out, ref, "5000 seqs")


def test_scale_variants():
    lens = [300, 17, 1]
    for kwargs in (dict(sdt=torch.bfloat16), dict(null_scales=True), dict(ks=-0.07, vs=0.5),
                   dict(sm_scale=0.02), dict(ks=0.125, vs=0.25, kv_std=0.05)):
        out, ref = _case(32, 8, 128, 16, lens, seed=13, **kwargs)
        gpu_util.assert_attention_close(out, ref, str(kwargs))


def test_scale_swap_would_be_caught():
    # [P3] read-side mutation table: reading V with K's scale must leave the tolerance.
    out, ref = _case(32, 8, 128, 16, [500, 60], seed=14, ks=0.05, vs=0.02)
    gpu_util.assert_attention_close(out, ref)
    g = out.float().cpu().numpy() * (0.05 / 0.02)
    assert np.count_nonzero(np.abs(g - ref) > 2e-3 + 1e-2 * np.abs(ref)) > 0


def test_all_empty_sequences_give_zeros():
    out, ref = _case(32, 8, 128, 16, [0, 0, 0], seed=15)
    assert torch.count_nonzero(out).item() == 0 and np.all(ref == 0)


def test_deterministic():
    w = workloads.WORKLOADS["tiny"]
    lay = workloads.make_layout(w)
    k, v = workloads.make_kv(w, lay.slot_mapping.size, "cuda")
    q = workloads.make_query(w, lay.num_seqs, "cuda")
    ksc, vsc = gpu_util.scale_pair(w)
    kc = workloads.new_cache(lay.num_blocks, w, "cuda")
    vc = kc.clone()
    kv.reshape_and_cache(k, v, kc, vc, torch.from_numpy(lay.slot_mapping).cuda(), ksc, vsc)
    bt = torch.from_numpy(lay.block_tables).cuda()
    sl = torch.from_numpy(lay.seq_lens).cuda()
    a = kv.paged_decode_attention(q, kc, vc, bt, sl, ksc, vsc)
    b = kv.paged_decode_attention(q, kc, vc, bt, sl, ksc, vsc)
    assert torch.equal(a, b)


def test_bad_block_and_length_are_flagged():
    q = torch.randn(2, 4, 64, device="cuda").to(torch.bfloat16)
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.uint8, device="cuda")
    bt = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kv.paged_decode_attention(q, kc, kc, bt, torch.tensor([20, 20], dtype=torch.int32,
                                                                device="cuda"), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kv.DEV_BAD_BLOCK
    assert torch.isfinite(out.float()).all()
    status.zero_()
    kv.paged_decode_attention(q, kc, kc, bt, torch.tensor([5, 40], dtype=torch.int32,
                                                          device="cuda"), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kv.DEV_BAD_BLOCK


def test_bad_device_scale_writes_nothing():
    q = torch.randn(2, 4, 64, device="cuda").to(torch.bfloat16)
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.uint8, device="cuda")
    bt = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device="cuda")
    sl = torch.tensor([20, 30], dtype=torch.int32, device="cuda")
    for bad in (0.0, float("nan"), float("inf")):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.full_like(q, 7.0)
        kv.paged_decode_attention(q, kc, kc, bt, sl, torch.tensor([bad], device="cuda"),
                                  torch.tensor([1.0], device="cuda"), out=out, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == kv.DEV_BAD_SCALE
        assert bool((out == 7.0).all())


def _full_size(name, n_random_pairs):
    # The bench step at full size: the whole context written (and, for the serving mix, one
    # new token per sequence), then decode.  The oracle attends over its own cache (built
    # from the same host inputs, never from GPU output) for every head of four sequences --
    # the longest, the shortest and two seeded others -- and for seeded random pairs.
    case = gpu_util.full_size_workload(name)
    w, lay = case["w"], case["lay"]
    q = workloads.make_query(w, lay.num_seqs, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kv.paged_decode_attention(q, case["kc"], case["vc"],
                                    torch.from_numpy(lay.block_tables).cuda(),
                                    torch.from_numpy(lay.seq_lens).cuda(), case["ksc"],
                                    case["vsc"], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.isfinite(out.float()).all()
    ko, vo = gpu_util.oracle_full_cache(case)
    rng = np.random.Generator(np.random.PCG64(w.seed + 77))
    whole = [int(np.argmax(lay.seq_lens)), int(np.argmin(lay.seq_lens))]
    for s in rng.permutation(lay.num_seqs):
        if len(whole) == min(4, lay.num_seqs):
            break
        if int(s) not in whole:
            whole.append(int(s))
    pairs = [(b, h) for b in whole for h in range(w.n_q)]
    pairs += [(int(b), int(h)) for b, h in zip(rng.integers(0, lay.num_seqs, n_random_pairs),
                                                rng.integers(0, w.n_q, n_random_pairs))]
    ks, vs = gpu_util.stored_scales(w)
    ref = gpu_util.oracle_pairs_threaded(pairs, q, ko, vo, lay.block_tables, lay.seq_lens, ks, vs)
    got = torch.stack([out[b, h] for b, h in pairs])
    gpu_util.assert_attention_close(got, ref, name)


def test_full_size_llama3_8b_sampled():
    _full_size("llama3_8b", 48)


def test_full_size_long_context_sampled():
    _full_size("long_context", 16)


def test_full_size_mixed_serving_sampled():
    _full_size("mixed_serving", 48)


def test_plan_with_empty_sequences_among_many():
    # 300 sequences, every 7th empty (zeroed by the plan, visited by no CTA), the others
    # split over CTA ranges at every offset of their block tables
    w = workloads.WORKLOADS["mixed_serving"]
    lay = workloads.make_layout(w, num_seqs=300, context=3000)
    lens = lay.seq_lens.copy()
    lens[::7] = 0
    k, v = workloads.make_kv(w, lay.slot_mapping.size, "cuda")
    q = workloads.make_query(w, lay.num_seqs, "cuda")
    ksc, vsc = gpu_util.scale_pair(w)
    kc = workloads.new_cache(lay.num_blocks, w, "cuda")
    vc = kc.clone()
    kv.reshape_and_cache(k, v, kc, vc, torch.from_numpy(lay.slot_mapping).cuda(), ksc, vsc)
    bt = torch.from_numpy(lay.block_tables).cuda()
    sl = torch.from_numpy(lens).cuda()
    out = torch.full_like(q, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.paged_decode_attention(q, kc, vc, bt, sl, ksc, vsc, out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.count_nonzero(out[torch.from_numpy(lens == 0).cuda()]).item() == 0
    ks, vs = gpu_util.stored_scales(w)
    ko, vo = gpu_util.oracle_cache_threaded(gpu_util.to_u16(k), gpu_util.to_u16(v),
                                            lay.slot_mapping, lay.num_blocks, w, ks, vs)
    pairs = [(b, h) for b in range(0, lay.num_seqs, 3) for h in range(0, w.n_q, 3)]
    ref = gpu_util.oracle_pairs_threaded(pairs, q, ko, vo, lay.block_tables, lens, ks, vs)
    gpu_util.assert_attention_close(torch.stack([out[b, h] for b, h in pairs]), ref, "plan")
