"""Mixed cache dtypes on the GPU (FP8 on K only or on V only, the other side bf16 and
unscaled) vs the CPU oracle.

[P1] tests/test-fp8.cpp check_fp8_attention quantizes K only, V only or both; the
all-FP8 case is covered by the other GPU tests.  Cache bytes: bit for bit (a NaN on a bf16
side only has to stay a NaN); attention: |gpu - oracle| <= 2e-3 + 1e-2 * |oracle|.
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

K_BF16 = (oracle.CACHE_BF16, oracle.E4M3)  # (k_kind, v_kind)
V_BF16 = (oracle.E4M3, oracle.CACHE_BF16)


def _np_cache(kind, shape):
    dt = np.uint8 if kind == oracle.E4M3 else np.uint16
    return np.full(shape, workloads.SENTINEL, dt)


def _to_gpu(c: np.ndarray) -> torch.Tensor:
    if c.dtype == np.uint8:
        return torch.from_numpy(c).cuda()
    return torch.from_numpy(c.view(np.int16)).cuda().view(torch.bfloat16)


def _from_gpu(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _assert_cache_equal(got: np.ndarray, want: np.ndarray, what: str):
    if got.dtype == np.uint16:  # bf16 side: a NaN's payload is not specified
        gn = (got & 0x7F80) == 0x7F80
        gn &= (got & 0x007F) != 0
        wn = (want & 0x7F80) == 0x7F80
        wn &= (want & 0x007F) != 0
        np.testing.assert_array_equal(gn, wn, err_msg=what + " (NaN positions)")
        got, want = np.where(gn, 0, got), np.where(wn, 0, want)
    mism = np.count_nonzero(got != want)
    assert mism == 0, f"{what}: {mism} elements differ"


def _specials(n, n_kv, hd, g, f32):
    x = torch.randn(n, n_kv, hd, generator=g) * 3.0
    flat = x.view(-1)
    idx = torch.randperm(flat.numel(), generator=g)[:64]
    vals = torch.tensor([0.0, -0.0, 1e30, -1e30, float("inf"), float("-inf"), float("nan"),
                         1e-30, 448.0 * 0.05, -1e-7, 3.0e38, 2.0 ** -140])
    flat[idx] = vals[torch.arange(64) % vals.numel()]
    return x if f32 else x.to(torch.bfloat16)


RESHAPE_CASES = [
    # name, kinds, n_kv, head_dim, block_size, num_tokens, f32 source
    ("kbf16_row1024", K_BF16, 8, 128, 16, 300, False),
    ("vbf16_row1024", V_BF16, 8, 128, 16, 300, False),
    ("kbf16_f32src", K_BF16, 4, 64, 8, 129, True),
    ("vbf16_f32src_row2048", V_BF16, 16, 128, 32, 77, True),
    ("vbf16_row8", V_BF16, 1, 8, 4, 33, False),
]


@pytest.mark.parametrize("case", RESHAPE_CASES, ids=[c[0] for c in RESHAPE_CASES])
def test_mixed_reshape_bytes_match_the_oracle(case):
    name, (kk, vk), n_kv, hd, bs, n, f32 = case
    g = torch.Generator().manual_seed(len(name) * 31 + n)
    k = _specials(n, n_kv, hd, g, f32)
    v = _specials(n, n_kv, hd, g, f32)
    nb = math.ceil(n / bs) + 2
    slots = torch.randperm(nb * bs, generator=g)[:n].to(torch.int64)
    slots[torch.randperm(n, generator=g)[: n // 10]] = -1  # padding tokens
    ks, vs = 0.05, -0.04
    kc, vc = _np_cache(kk, (nb, bs, n_kv, hd)), _np_cache(vk, (nb, bs, n_kv, hd))
    src = oracle.F32 if f32 else oracle.BF16
    kin = k.numpy() if f32 else k
    vin = v.numpy() if f32 else v
    st = oracle.reshape_and_cache_mixed(kin, vin, kc, kk, vc, vk, slots.numpy(), bs, ks, vs,
                                        src_dtype=src)
    assert st == 0
    gk, gv = _to_gpu(_np_cache(kk, kc.shape)), _to_gpu(_np_cache(vk, vc.shape))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.reshape_and_cache_mixed(k.cuda(), v.cuda(), gk, gv, slots.cuda(),
                               torch.tensor([ks], device="cuda"), torch.tensor([vs], device="cuda"),
                               status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _assert_cache_equal(_from_gpu(gk), kc, name + " K")
    _assert_cache_equal(_from_gpu(gv), vc, name + " V")


def test_bf16_side_scale_is_never_read_or_checked():
    # a zero scale on the bf16 side is not an error; on the FP8 side it is
    g = torch.Generator().manual_seed(5)
    k = torch.randn(40, 2, 64, generator=g).to(torch.bfloat16).cuda()
    slots = torch.arange(40, dtype=torch.int64).cuda()
    kc = torch.zeros(5, 8, 2, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros(5, 8, 2, 64, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.reshape_and_cache_mixed(k, k, kc, vc, slots, torch.tensor([0.0], device="cuda"),
                               torch.tensor([0.5], device="cuda"), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(kc.view(-1, 2, 64), k)  # the bf16 copy is exact
    status.zero_()
    vc2 = torch.full_like(vc, 7)
    kv.reshape_and_cache_mixed(k, k, kc, vc2, slots, torch.tensor([0.5], device="cuda"),
                               torch.tensor([0.0], device="cuda"), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & kv.DEV_BAD_SCALE
    assert bool((vc2 == 7).all())  # nothing written


def _decode_case(kinds, n_q, n_kv, hd, bs, lengths, seed, ks=0.05, vs=0.04, sm_scale=0.0,
                 sdt=torch.float32, write_on_gpu=False):
    kk, vk = kinds
    g = torch.Generator().manual_seed(seed)
    need = [math.ceil(L / bs) for L in lengths]
    nb = sum(need) + 2
    perm = torch.randperm(nb, generator=g).numpy().astype(np.int32)
    bt = np.full((len(lengths), max(1, max(need))), -1, np.int32)
    at = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[at:at + n]
        at += n
    total = sum(lengths)
    k = torch.randn(total, n_kv, hd, generator=g).to(torch.bfloat16)
    v = torch.randn(total, n_kv, hd, generator=g).to(torch.bfloat16)
    q = torch.randn(len(lengths), n_q, hd, generator=g).to(torch.bfloat16)
    slots = np.concatenate([bt[i, np.arange(L) // bs].astype(np.int64) * bs + np.arange(L) % bs
                            for i, L in enumerate(lengths)]) if total else np.zeros(0, np.int64)
    sname = "f32" if sdt == torch.float32 else "bf16"
    ksf, vsf = workloads.stored_scale(ks, sname), workloads.stored_scale(vs, sname)
    kc, vc = _np_cache(kk, (nb, bs, n_kv, hd)), _np_cache(vk, (nb, bs, n_kv, hd))
    assert oracle.reshape_and_cache_mixed(k, v, kc, kk, vc, vk, slots, bs, ksf, vsf) == 0
    ref, st = oracle.paged_decode_attention_mixed(q, kc, kk, vc, vk, bt,
                                                  np.array(lengths, np.int32), ksf, vsf, sm_scale)
    assert st == 0
    ksc = torch.tensor([ks], dtype=sdt, device="cuda")
    vsc = torch.tensor([vs], dtype=sdt, device="cuda")
    if write_on_gpu:
        gk, gv = _to_gpu(_np_cache(kk, kc.shape)), _to_gpu(_np_cache(vk, vc.shape))
        kv.reshape_and_cache_mixed(k.cuda(), v.cuda(), gk, gv, torch.from_numpy(slots).cuda(),
                                   ksc, vsc)
    else:
        gk, gv = _to_gpu(kc), _to_gpu(vc)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kv.paged_decode_attention_mixed(q.cuda(), gk, gv, torch.from_numpy(bt).cuda(),
                                          torch.tensor(lengths, dtype=torch.int32, device="cuda"),
                                          ksc, vsc, sm_scale=sm_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, ref


DECODE_CASES = [
    # name, n_q, n_kv, head_dim, block_size, lengths
    ("g4_ragged", 32, 8, 128, 16, [1, 15, 16, 17, 31, 33, 100, 257, 1000, 4096]),
    ("g8_bs32", 64, 8, 128, 32, [5, 3000, 70, 0, 2]),
    ("g1_hd64_bs8", 4, 4, 64, 8, [1, 7, 8, 9, 200]),
    ("g16_nt2", 32, 2, 128, 16, [50, 500]),
    ("g12_hd64_nt2", 24, 2, 64, 16, [77, 1234]),
    ("bs256_g6", 24, 4, 128, 256, [700, 5]),
    ("mha16_head_groups", 16, 16, 128, 16, [400, 17]),
    # head_dim 256: groups of up to 8 on the split-KV kernel
    ("g8_hd256_bs64", 64, 8, 256, 64, [65, 300, 1, 2000]),
    ("g2_hd256", 4, 2, 256, 16, [17, 129]),
]


@pytest.mark.parametrize("kinds", [K_BF16, V_BF16], ids=["k_bf16", "v_bf16"])
@pytest.mark.parametrize("case", DECODE_CASES, ids=[c[0] for c in DECODE_CASES])
def test_mixed_decode_against_oracle(case, kinds):
    name, n_q, n_kv, hd, bs, lengths = case
    out, ref = _decode_case(kinds, n_q, n_kv, hd, bs, lengths, seed=len(name) * 7 + kinds[0])
    gpu_util.assert_attention_close(out, ref, name)


@pytest.mark.parametrize("kinds", [K_BF16, V_BF16], ids=["k_bf16", "v_bf16"])
def test_mixed_decode_long_sequence_and_scales(kinds):
    out, ref = _decode_case(kinds, 32, 8, 128, 16, [60_001, 3], seed=21)
    gpu_util.assert_attention_close(out, ref, "long")
    for kw in (dict(sdt=torch.bfloat16), dict(ks=-0.07, vs=0.5), dict(sm_scale=0.02)):
        out, ref = _decode_case(kinds, 32, 8, 128, 16, [300, 17, 1], seed=22, **kw)
        gpu_util.assert_attention_close(out, ref, str(kw))


@pytest.mark.parametrize("kinds", [K_BF16, V_BF16], ids=["k_bf16", "v_bf16"])
def test_mixed_write_then_decode_on_gpu(kinds):
    out, ref = _decode_case(kinds, 32, 8, 128, 16, [513, 16, 1, 2000], seed=23, write_on_gpu=True)
    gpu_util.assert_attention_close(out, ref, "gpu write + decode")


def test_scaling_the_bf16_side_would_be_caught():
    # V bf16 read as if it carried v_scale: leaves the tolerance (the test can fail)
    out, ref = _decode_case(V_BF16, 32, 8, 128, 16, [400, 31], seed=24, vs=0.04)
    gpu_util.assert_attention_close(out, ref)
    g = out.float().cpu().numpy() * 0.04
    assert np.count_nonzero(np.abs(g - ref) > 2e-3 + 1e-2 * np.abs(ref)) > 0


def _multi_case(kinds, n_q, n_kv, hd, bs, lengths, nbs, seed, ks=0.05, vs=0.04):
    """Causal multi-query attention with one bf16 side: sequence b's last nbs[b] cached tokens
    are its query tokens.  The cache is written by the GPU; the oracle writes its own."""
    kk, vk = kinds
    g = torch.Generator().manual_seed(seed)
    need = [math.ceil(L / bs) for L in lengths]
    nb = sum(need) + 2
    perm = torch.randperm(nb, generator=g).numpy().astype(np.int32)
    bt = np.full((len(lengths), max(1, max(need))), -1, np.int32)
    at = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[at:at + n]
        at += n
    total = sum(lengths)
    k = torch.randn(total, n_kv, hd, generator=g).to(torch.bfloat16)
    v = torch.randn(total, n_kv, hd, generator=g).to(torch.bfloat16)
    qsl = np.concatenate([[0], np.cumsum(nbs)]).astype(np.int32)
    q = torch.randn(int(qsl[-1]), n_q, hd, generator=g).to(torch.bfloat16)
    slots = np.concatenate([bt[i, np.arange(L) // bs].astype(np.int64) * bs + np.arange(L) % bs
                            for i, L in enumerate(lengths)])
    kc, vc = _np_cache(kk, (nb, bs, n_kv, hd)), _np_cache(vk, (nb, bs, n_kv, hd))
    assert oracle.reshape_and_cache_mixed(k, v, kc, kk, vc, vk, slots, bs, ks, vs) == 0
    ref, st = oracle.paged_attention_multi_mixed(q, qsl, kc, kk, vc, vk, bt,
                                                 np.array(lengths, np.int32), ks, vs)
    assert st == 0
    ksc = torch.tensor([ks], device="cuda")
    vsc = torch.tensor([vs], device="cuda")
    gk, gv = _to_gpu(_np_cache(kk, kc.shape)), _to_gpu(_np_cache(vk, vc.shape))
    kv.reshape_and_cache_mixed(k.cuda(), v.cuda(), gk, gv, torch.from_numpy(slots).cuda(), ksc, vsc)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = kv.paged_attention_multi_mixed(q.cuda(), torch.from_numpy(qsl).cuda(), max(nbs), gk, gv,
                                         torch.from_numpy(bt).cuda(),
                                         torch.tensor(lengths, dtype=torch.int32, device="cuda"),
                                         ksc, vsc, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, ref


MULTI_CASES = [
    # name, n_q, n_kv, head_dim, block_size, lengths, query tokens per sequence
    ("g4_q4", 32, 8, 128, 16, [700, 33, 4, 2000], [4, 3, 4, 1]),
    ("g5_q3_bs32", 40, 8, 128, 32, [100, 1000, 3], [3, 2, 3]),
    ("g2_q8_hd64", 8, 4, 64, 16, [50, 17, 300], [8, 5, 1]),
    ("g1_q16", 8, 8, 128, 16, [64, 130], [16, 9]),
    ("g2_q4_hd256", 8, 4, 256, 64, [90, 500], [4, 2]),
]


@pytest.mark.parametrize("kinds", [K_BF16, V_BF16], ids=["k_bf16", "v_bf16"])
@pytest.mark.parametrize("case", MULTI_CASES, ids=[c[0] for c in MULTI_CASES])
def test_mixed_multi_query_against_oracle(case, kinds):
    name, n_q, n_kv, hd, bs, lengths, nbs = case
    out, ref = _multi_case(kinds, n_q, n_kv, hd, bs, lengths, nbs, seed=len(name) * 5 + kinds[1])
    gpu_util.assert_attention_close(out, ref, name)


def test_mixed_multi_query_past_the_split_kv_kernel_is_refused():
    q = torch.zeros(5, 32, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros(4, 16, 8, 128, dtype=torch.uint8, device="cuda")
    bt = torch.zeros(1, 4, dtype=torch.int32, device="cuda")
    sl = torch.tensor([40], dtype=torch.int32, device="cuda")
    qsl = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
    with pytest.raises(kv.KvFp8Error) as e:  # 5 tokens x 4 heads = 20 score columns
        kv.paged_attention_multi_mixed(q, qsl, 5, kc, vc, bt, sl)
    assert e.value.status == kv.ERR_UNSUPPORTED
