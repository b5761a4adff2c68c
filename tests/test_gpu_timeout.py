"""The decode kernel's bounded-wait timeout path, driven on the GPU without any fault.

A test-only build of the library (libkvfp8_withhold.so, never loaded by the package)
makes every CTA's producer withhold the copy of its first chunk -- no copy is issued and
no arrival made for that pipeline stage -- and gives every wait a limit of about 1e5
cycles.  The consumers' waits on that stage then run out: each sets KVFP8_DEV_TIMEOUT,
raises the CTA's abort flag and leaves; the producer drains the copies it did issue (they
land) and leaves too.  Nothing traps and no copy is outstanding when a CTA exits.  The
call must return, the status must carry the timeout bit, and a normal call on the same
stream right after must be correct.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

import workloads
from tests import gpu_util

pytestmark = pytest.mark.gpu

kv = pytest.importorskip("fp8_paged_kv_reshape_gb300")
from fp8_paged_kv_reshape_gb300 import _build, binding  # noqa: E402


@pytest.fixture(scope="module")
def withhold_lib():
    lib = ctypes.CDLL(_build.build_withhold_variant())  # its own symbols (RTLD_LOCAL)
    P, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lib.kvfp8_paged_decode_attention.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32,
                                                 i32, f32, P, P, ctypes.c_int, P, sz, P, P]
    lib.kvfp8_paged_decode_attention.restype = ctypes.c_int
    return lib


def _case(lengths, seed):
    w = workloads.WORKLOADS["llama3_8b"]
    lay = workloads.make_layout(w, lengths=lengths)
    k, v = workloads.make_kv(w, lay.slot_mapping.size, "cuda")
    q = workloads.make_query(w, lay.num_seqs, "cuda")
    ksc, vsc = gpu_util.scale_pair(w)
    kc = workloads.new_cache(lay.num_blocks, w, "cuda")
    vc = kc.clone()
    kv.reshape_and_cache(k, v, kc, vc, torch.from_numpy(lay.slot_mapping).cuda(), ksc, vsc)
    return w, lay, k, v, q, ksc, vsc, kc, vc


@pytest.mark.parametrize("lengths", [[17, 33, 64, 100], [50000]], ids=["one_chunk_per_cta",
                                                                       "ten_chunks_per_cta"])
def test_decode_wait_runs_out_and_the_next_call_is_correct(withhold_lib, lengths):
    w, lay, k, v, q, ksc, vsc, kc, vc = _case(lengths, 1)
    bt = torch.from_numpy(lay.block_tables).cuda()
    sl = torch.from_numpy(lay.seq_lens).cuda()
    num_seqs, n_q, hd = q.shape
    ws = torch.empty(kv.paged_decode_workspace_size(num_seqs, n_q, hd), dtype=torch.uint8,
                     device="cuda")
    out = torch.zeros_like(q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = withhold_lib.kvfp8_paged_decode_attention(
        p(out), p(q), p(kc), p(vc), p(bt), bt.shape[1], p(sl), num_seqs, n_q, w.n_kv, hd,
        w.block_size, lay.num_blocks, 0.0, p(ksc), p(vsc), binding.F32, p(ws), ws.numel(),
        p(status), ctypes.c_void_p(stream.cuda_stream))
    torch.cuda.synchronize()  # the kernels ended
    elapsed = time.perf_counter() - t0
    assert rc == binding.OK
    assert int(status.item()) & kv.DEV_TIMEOUT, int(status.item())
    assert elapsed < 10.0
    # the context is usable and the stream healthy: the library's normal call is correct
    status.zero_()
    out2 = kv.paged_decode_attention(q, kc, vc, bt, sl, ksc, vsc, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ks, vs = gpu_util.stored_scales(w)
    ko, vo = gpu_util.oracle_cache_threaded(gpu_util.to_u16(k), gpu_util.to_u16(v),
                                            lay.slot_mapping, lay.num_blocks, w, ks, vs)
    pairs = [(b, h) for b in range(num_seqs) for h in range(0, n_q, 5)]
    ref = gpu_util.oracle_pairs_threaded(pairs, q, ko, vo, lay.block_tables, lay.seq_lens, ks, vs)
    gpu_util.assert_attention_close(torch.stack([out2[b, h] for b, h in pairs]), ref, "after")
    assert np.isfinite(ref).all()
