"""kvfp8_paged_decode_attention_noalloc: decode attention for callers that cannot allocate
device memory (a plug-in whose host runtime owns every device allocation, a serving loop
that must not allocate once it runs).  It keeps its split-KV scratch in a fixed device
array inside the library instead of a caller workspace; its output must match the
workspace entry point's.  Collected last on purpose (file name), so that a run stopping
at its first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests import gpu_util

pytestmark = pytest.mark.gpu

kv = pytest.importorskip("fp8_paged_kv_reshape_gb300")
from fp8_paged_kv_reshape_gb300 import binding  # noqa: E402


def _inputs(seed, lengths, n_q=32, n_kv=8, hd=128, bs=16):
    g = torch.Generator().manual_seed(seed)
    need = [-(-L // bs) for L in lengths]
    nb = sum(need) + 1
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    bt = torch.full((len(lengths), max(1, max(need))), -1, dtype=torch.int32)
    at = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[at:at + n]
        at += n
    # random non-NaN E4M3 codes
    codes = torch.randint(0, 0x70, (2, nb, bs, n_kv, hd), generator=g, dtype=torch.int32)
    signs = torch.randint(0, 2, codes.shape, generator=g, dtype=torch.int32) << 7
    kc, vc = (codes | signs).to(torch.uint8).cuda().unbind(0)
    q = torch.randn(len(lengths), n_q, hd, generator=g).to(torch.bfloat16).cuda()
    sl = torch.tensor(lengths, dtype=torch.int32).cuda()
    ks = torch.tensor([0.05], device="cuda")
    vs = torch.tensor([0.04], device="cuda")
    return q, kc.contiguous(), vc.contiguous(), bt.cuda(), sl, ks, vs


def _noalloc_via_c_abi(q, kc, vc, bt, sl, ks, vs, out, status):
    num_seqs, n_q, hd = q.shape
    nb, bs, n_kv, _ = kc.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return kv.LIB.kvfp8_paged_decode_attention_noalloc(
        p(out), p(q), p(kc), p(vc), p(bt), bt.shape[1], p(sl), num_seqs, n_q, n_kv, hd, bs, nb,
        0.0, p(ks), p(vs), binding.F32, p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _oracle(q, kc, vc, bt, sl, ks, vs):
    ref, st = oracle.paged_decode_attention(q.cpu(), kc.cpu().numpy(), vc.cpu().numpy(),
                                            bt.cpu().numpy(), sl.cpu().numpy(), float(ks.item()),
                                            float(vs.item()))
    assert st == 0
    return ref


def test_no_alloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    # Two different batches back to back through the raw C ABI: each output must equal the
    # workspace entry point's bit for bit (same kernels, same inputs), and both must match the
    # double-precision oracle within the attention tolerance.  The second call reuses the
    # scratch the first one left behind.
    cases = [(1, [1000, 17, 4096, 0, 300, 1]), (2, [30000, 33, 5, 2048])]
    for seed, lengths in cases:
        q, kc, vc, bt, sl, ks, vs = _inputs(seed, lengths)
        ref = kv.paged_decode_attention(q, kc, vc, bt, sl, ks, vs)
        out = torch.full_like(q, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = _noalloc_via_c_abi(q, kc, vc, bt, sl, ks, vs, out, status)
        torch.cuda.synchronize()
        assert rc == binding.OK, kv.status_string(rc)
        assert int(status.item()) == 0
        assert torch.equal(out, ref), f"call {seed}: differs from the workspace entry point"
        gpu_util.assert_attention_close(out, _oracle(q, kc, vc, bt, sl, ks, vs),
                                        f"noalloc call {seed} vs oracle")


def test_no_alloc_through_the_binding_allocates_no_device_memory():
    q, kc, vc, bt, sl, ks, vs = _inputs(3, [5000, 1, 777, 64, 2])
    ref = kv.paged_decode_attention(q, kc, vc, bt, sl, ks, vs)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [torch.full_like(q, float("nan")) for _ in range(3)]
    kv.paged_decode_attention_noalloc(q, kc, vc, bt, sl, ks, vs, out=out, status=status)
    torch.cuda.synchronize()  # the first call has loaded its kernels
    free0 = torch.cuda.mem_get_info()[0]
    for o in outs:
        kv.paged_decode_attention_noalloc(q, kc, vc, bt, sl, ks, vs, out=o, status=status)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0, "device memory changed across no-alloc calls"
    assert int(status.item()) == 0
    for o in [out] + outs:
        assert torch.equal(o, ref)
    gpu_util.assert_attention_close(out, _oracle(q, kc, vc, bt, sl, ks, vs), "noalloc binding")


def test_no_alloc_refuses_a_batch_larger_than_its_scratch():
    # the scratch holds the partials of (num_seqs + max CTAs) x n_q x head_dim floats
    num_seqs = 40000
    assert kv.paged_decode_workspace_size(num_seqs, 32, 128) > (32 << 20)
    q = torch.zeros(num_seqs, 32, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(1, 16, 8, 128, dtype=torch.uint8, device="cuda")
    bt = torch.zeros(num_seqs, 1, dtype=torch.int32, device="cuda")
    sl = torch.ones(num_seqs, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _noalloc_via_c_abi(q, kc, kc, bt, sl, torch.ones(1, device="cuda"),
                            torch.ones(1, device="cuda"), out, status)
    torch.cuda.synchronize()
    assert rc == binding.ERR_WORKSPACE
    assert bool((out == 7.0).all())  # nothing ran
