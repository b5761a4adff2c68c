"""The widened forms of the path at full workload size, in the launch configuration the
benchmark times (bench.Problem: the same tensors, calls and workspace), checked on sampled
sequences against the oracle's matching functions:

  rope     rope on K fused into the cache write, then decode
  k_bf16   mixed cache dtypes, K bf16 / V E4M3;  v_bf16 the other way round
  multi    causal multi-query attention, 16 // G query tokens per sequence
  prefill  chunked prefill: the last 512 tokens of each sequence (16 on the serving mix)
           written, then causal attention for them on the tensor-core kernel

For each sampled sequence the oracle writes that sequence's rows (as one step leaves them
in the cache) into a cache of its own and attends with every head.
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
import bench  # noqa: E402


def _seq_rows(p, b, ctx):
    """bf16 K/V rows [L, n_kv, hd] of sequence b in position order after one step."""
    w, lay = p.w, p.lay
    rows = np.nonzero(lay.row_seq == b)[0]
    rows = rows[np.argsort(lay.row_pos[rows])]
    if w.kind == "write":
        rows = rows[lay.row_pos[rows] >= 0]
    idx = torch.from_numpy(rows).cuda()
    if not p.serving:
        return p.k.index_select(0, idx).cpu(), p.v.index_select(0, idx).cpu()
    k = ctx[0].index_select(0, idx).clone()
    v = ctx[1].index_select(0, idx).clone()
    L, n = rows.size, p.qlen
    k[L - n:] = p.k[b * n:(b + 1) * n]
    v[L - n:] = p.v[b * n:(b + 1) * n]
    return k.cpu(), v.cpu()


def _oracle_seq(p, b, k, v, ks, vs):
    """(oracle cache pair, oracle output rows of sequence b) for p's variant."""
    w = p.w
    L = k.shape[0]
    bs = w.block_size
    nb = max(1, math.ceil(L / bs))
    shape = (nb, bs, w.n_kv, w.head_dim)
    kinds = (oracle.CACHE_BF16 if p.k_elem == 2 else oracle.E4M3,
             oracle.CACHE_BF16 if p.v_elem == 2 else oracle.E4M3)
    kc = np.full(shape, workloads.SENTINEL, np.uint8 if kinds[0] == oracle.E4M3 else np.uint16)
    vc = np.full(shape, workloads.SENTINEL, np.uint8 if kinds[1] == oracle.E4M3 else np.uint16)
    slots = np.arange(L, dtype=np.int64)
    if p.variant == "rope":
        st = oracle.rope_reshape_and_cache(k, v, kc, vc, slots, slots, p.table.cpu().numpy(),
                                           p.rot, True, bs, ks, vs)
    elif p.variant in ("k_bf16", "v_bf16"):
        st = oracle.reshape_and_cache_mixed(k, v, kc, kinds[0], vc, kinds[1], slots, bs, ks, vs)
    else:
        st = oracle.reshape_and_cache(k, v, kc, vc, slots, bs, ks, vs)
    assert st == 0
    if not p.decode:
        return (kc, vc), None
    bt = np.arange(nb, dtype=np.int32)[None, :]
    lens = np.array([L], np.int32)
    if p.variant in ("multi", "prefill"):
        n = p.qlen
        q = p.q[b * n:(b + 1) * n].cpu()
        out, st = oracle.paged_attention_multi(q, np.array([0, n], np.int32), kc, vc, bt, lens,
                                               ks, vs)
    elif p.variant in ("k_bf16", "v_bf16"):
        out, st = oracle.paged_decode_attention_mixed(p.q[b:b + 1].cpu(), kc, kinds[0], vc,
                                                      kinds[1], bt, lens, ks, vs)
    else:
        out, st = oracle.paged_decode_attention(p.q[b:b + 1].cpu(), kc, vc, bt, lens, ks, vs)
    assert st == 0
    return (kc, vc), out


def _gpu_seq_cache(p, b, L):
    """The GPU cache's rows of sequence b in position order, as host arrays."""
    lay, bs = p.lay, p.w.block_size
    t = torch.arange(L, device="cuda")
    phys = torch.from_numpy(lay.block_tables[b]).cuda().long()[t // bs]
    res = []
    for c in (p.kc, p.vc):
        rows = c[phys, t % bs]
        res.append(rows.cpu().numpy() if c.dtype == torch.uint8
                   else rows.view(torch.int16).cpu().numpy().view(np.uint16))
    return res


CASES = [
    ("llama3_8b", "rope", 5), ("llama3_8b", "k_bf16", 5), ("llama3_8b", "v_bf16", 5),
    ("llama3_8b", "multi", 5), ("mixed_serving", "multi", 8), ("mixed_serving", "v_bf16", 8),
    ("llama3_8b", "prefill", 2), ("mixed_serving", "prefill", 4),
    ("prefill_write", "rope", 4), ("prefill_write", "k_bf16", 4),
]


@pytest.mark.parametrize("case", CASES, ids=["%s-%s" % c[:2] for c in CASES])
def test_bench_variant_full_size_sampled(case):
    name, variant, n_seq = case
    p = bench.Problem(name, torch.device("cuda", 0), None, variant)
    p.reshape()
    if p.decode:
        p.attend()
    torch.cuda.synchronize()
    assert int(p.status.item()) == 0
    w, lay = p.w, p.lay
    ctx = workloads.make_kv(w, lay.slot_mapping.size, "cuda") if p.serving else None
    rng = np.random.Generator(np.random.PCG64(w.seed + 91))
    seqs = list(rng.choice(lay.num_seqs, size=min(n_seq, lay.num_seqs), replace=False))
    seqs[0] = int(np.argmax(lay.seq_lens))
    ks, vs = gpu_util.stored_scales(w)
    for b in seqs:
        b = int(b)
        k, v = _seq_rows(p, b, ctx)
        (kc, vc), ref = _oracle_seq(p, b, k, v, ks, vs)
        L = k.shape[0]
        gk, gv = _gpu_seq_cache(p, b, L)
        assert np.array_equal(gk, kc.reshape(-1, w.n_kv, w.head_dim)[:L]), (name, variant, b, "K")
        assert np.array_equal(gv, vc.reshape(-1, w.n_kv, w.head_dim)[:L]), (name, variant, b, "V")
        if ref is not None:
            got = p.out[b * p.qlen:(b + 1) * p.qlen] if p.qsl is not None else p.out[b:b + 1]
            gpu_util.assert_attention_close(got, ref, "%s %s seq %d" % (name, variant, b))
    if p.decode:
        assert torch.isfinite(p.out.float()).all()
