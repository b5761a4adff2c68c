"""kvfp8_reshape_and_cache on the GPU vs the CPU oracle: cache bytes bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_util, pins

pytestmark = pytest.mark.gpu

kv = pytest.importorskip("fp8_paged_kv_reshape_gb300")

SCALES = [0.05, 0.04, 0.03, 0.3, 3.7, 0.125, 0.25, 0.03125, 0.5, 1.0, -0.05, 3.0, 1e-3, 7.3e5,
          2.0 ** -7, 2.0 ** -13, 2.0 ** -11, 2.0 ** -9, 1.0e-30, 3.0e30,
          # edges of the reciprocal-and-corrections divide's range [2^-60, 2^60]
          2.0 ** -60, 2.0 ** 60, 1.5 * 2.0 ** -61, 1.5 * 2.0 ** 60, 1.25 * 2.0 ** -60,
          0.75 * 2.0 ** 61]


def _run(key, value, slots, nb, bs, ks, vs, sdt=torch.float32, status=None):
    n_kv, hd = key.shape[1], key.shape[2]
    kc = torch.full((nb, bs, n_kv, hd), workloads.SENTINEL, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    ksc = None if ks is None else torch.tensor([ks], dtype=sdt, device="cuda")
    vsc = None if vs is None else torch.tensor([vs], dtype=sdt, device="cuda")
    kv.reshape_and_cache(key, value, kc, vc, slots, ksc, vsc, status=status)
    torch.cuda.synchronize()
    return kc.cpu().numpy(), vc.cpu().numpy()


def _oracle(key_host, value_host, slots_np, nb, bs, n_kv, hd, ks, vs, src=oracle.BF16):
    kc = np.full((nb, bs, n_kv, hd), workloads.SENTINEL, np.uint8)
    vc = kc.copy()
    st = oracle.reshape_and_cache(key_host, value_host, kc, vc, slots_np, bs,
                                  1.0 if ks is None else ks, 1.0 if vs is None else vs,
                                  src_dtype=src)
    assert st == 0
    return kc, vc


# Row layouts (n_kv, head_dim): 8-element rows take the 8-wide kernel; 512- and 1024-element
# rows with 32-byte aligned sources take the wide kernel (16 elements per lane, one unit or two)
ROW_LAYOUTS = [(1, 8), (4, 128), (8, 128)]


@pytest.mark.parametrize("n_kv,hd", ROW_LAYOUTS)
def test_every_bf16_value_at_many_scales(n_kv, hd):
    bits = np.arange(1 << 16, dtype=np.uint16)
    n = bits.size // (n_kv * hd)
    k = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).reshape(n, n_kv, hd)
    v = torch.from_numpy(bits[::-1].view(np.int16).copy()).view(torch.bfloat16).reshape(n, n_kv, hd)
    slots = torch.arange(n, dtype=torch.int64)
    kd, vd, sd = k.cuda(), v.cuda(), slots.cuda()
    for s in SCALES:
        s32 = float(np.float32(s))
        kc, vc = _run(kd, vd, sd, n, 1, s32, -s32)
        ko, vo = _oracle(gpu_util.to_u16(k), gpu_util.to_u16(v), slots.numpy(), n, 1, n_kv, hd,
                         s32, -s32)
        bad = np.nonzero(kc.ravel() != ko.ravel())[0]
        assert bad.size == 0, (s, [(hex(int(bits[i])), hex(kc.ravel()[i]), hex(ko.ravel()[i]))
                                   for i in bad[:8]])
        np.testing.assert_array_equal(vc, vo)


@pytest.mark.parametrize("n_kv,hd", ROW_LAYOUTS)
def test_float32_source_bit_patterns(n_kv, hd):
    rng = np.random.Generator(np.random.PCG64(21))
    x = rng.integers(0, 1 << 32, size=1 << 21, dtype=np.uint64).astype(np.uint32).view(np.float32)
    y = (rng.standard_normal(1 << 21) * np.exp2(rng.uniform(-14, 12, 1 << 21))).astype(np.float32)
    special = np.array([np.nan, -np.nan, np.inf, -np.inf, 0.0, -0.0, 448.0, 464.0, -464.0, 1e-45,
                        -1e-45, 2.0 ** -10, 3 * 2.0 ** -10, 432.0, 3.4e38, -3.4e38], np.float32)
    neg_nan = np.array([0xFFC00000, 0xFF800001, 0x7F800001], np.uint32).view(np.float32)
    data = np.concatenate([x, y, special, neg_nan])
    row = n_kv * hd
    data = np.concatenate([data, np.zeros((-data.size) % row, np.float32)])
    n = data.size // row
    key = torch.from_numpy(data.reshape(n, n_kv, hd).copy())
    slots = torch.arange(n, dtype=torch.int64)
    for s in (0.05, 0.03, 1.0, -0.125, 2.0 ** -60, -2.0 ** 60, 1e-25, 3.7e22):
        s32 = float(np.float32(s))
        kc, vc = _run(key.cuda(), key.cuda(), slots.cuda(), n, 1, s32, s32)
        ko, _ = _oracle(key.numpy(), key.numpy(), slots.numpy(), n, 1, n_kv, hd, s32, s32,
                        src=oracle.F32)
        bad = np.nonzero(kc.ravel() != ko.ravel())[0]
        assert bad.size == 0, (s, [(hex(int(data.view(np.uint32)[i])), hex(kc.ravel()[i]),
                                    hex(ko.ravel()[i])) for i in bad[:8]])
        np.testing.assert_array_equal(vc, kc)


def test_rows_16_but_not_32_byte_aligned_take_the_8_wide_kernel():
    # a source starting 16 bytes into an allocation: the wide kernel's 32-byte loads would be
    # misaligned, so the call must fall back to 16-byte loads and give the same bytes
    torch.manual_seed(6)
    n, n_kv, hd = 257, 8, 128
    buf = (torch.randn(n * n_kv * hd + 8, device="cuda") * 20).to(torch.bfloat16)
    key = buf[8:].view(n, n_kv, hd)
    assert key.data_ptr() % 32 == 16
    val = torch.flip(key, dims=[0]).contiguous()
    slots = torch.randperm(40 * 16, device="cuda")[:n].to(torch.int64)
    kc, vc = _run(key, val, slots, 40, 16, 0.05, -0.04)
    ko, vo = _oracle(gpu_util.to_u16(key), gpu_util.to_u16(val), slots.cpu().numpy(), 40, 16,
                     n_kv, hd, 0.05, -0.04)
    np.testing.assert_array_equal(kc, ko)
    np.testing.assert_array_equal(vc, vo)


def test_special_values_follow_the_page_encoder():
    # NaN keeps its own sign, +-inf and |x/s| >= 448 saturate, -0 stays 0x80.
    # bf16 bits: +NaN, -NaN, +inf, -inf, -0, +0, 22.375, 23.25, -30, 2^-100
    bits = np.array([0x7FC0, 0xFFC0, 0x7F80, 0xFF80, 0x8000, 0x0000, 0x41B3, 0x41BA, 0xC1F0,
                     0x0D80, 0, 0, 0, 0, 0, 0], np.uint16)
    x = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    key = x.reshape(2, 1, 8).cuda()
    kc, _ = _run(key, key, torch.arange(2, dtype=torch.int64, device="cuda"), 2, 1, 0.05, 0.05)
    got = [int(v) for v in kc.ravel()[:10]]
    assert got == [0x7F, 0xFF, 0x7E, 0xFE, 0x80, 0x00, 0x7E, 0x7E, 0xFE, 0x00]
    ko, _ = _oracle(bits.reshape(2, 1, 8), bits.reshape(2, 1, 8), np.arange(2), 2, 1, 1, 8, 0.05, 0.05)
    assert got == [int(v) for v in ko.ravel()[:10]]


def _workload_inputs(name, **over):
    w = workloads.WORKLOADS[name]
    lay = workloads.make_layout(w, **over)
    k, v = workloads.make_kv(w, lay.slot_mapping.size, device="cuda")
    return w, lay, k, v


@pytest.mark.parametrize("name", ["tiny", "llama3_8b", "long_context", "prefill_write",
                                  "mixed_serving"])
def test_workload_full_cache_bit_exact(name):
    # Every configuration at full size, written as a bench step writes it (all context rows;
    # the serving mix then writes one new token per sequence over its last row), and the
    # whole K and V caches compared byte for byte with the oracle's, sentinels included.
    case = gpu_util.full_size_workload(name)
    ko, vo = gpu_util.oracle_full_cache(case)
    kc = case["kc"].cpu().numpy()
    bad = np.nonzero(kc.ravel() != ko.ravel())[0]
    assert bad.size == 0, (name, bad.size, bad[:8])
    del kc
    vc = case["vc"].cpu().numpy()
    bad = np.nonzero(vc.ravel() != vo.ravel())[0]
    assert bad.size == 0, (name, bad.size, bad[:8])
    lay = case["lay"]
    if name == "prefill_write":
        assert (lay.slot_mapping == -1).sum() > 0  # padding rows were present and skipped
        assert (ko == workloads.SENTINEL).all(axis=(1, 2, 3)).any()  # untouched pool blocks
    if name == "llama3_8b":  # the 0.1% outliers x20 reach the saturation code
        assert ((ko & 0x7F) == 0x7E).any()
    if name == "mixed_serving":  # the last row of every sequence holds its new token
        w = case["w"]
        kn, vn, new_slots = case["new"]
        ks, vs = gpu_util.stored_scales(w)
        kt = np.zeros((lay.num_seqs, 1, w.n_kv, w.head_dim), np.uint8)
        vt = kt.copy()
        assert oracle.reshape_and_cache(kn, vn, kt, vt, np.arange(lay.num_seqs), 1, ks, vs) == 0
        row = w.n_kv * w.head_dim
        np.testing.assert_array_equal(ko.reshape(-1, row)[new_slots], kt.reshape(-1, row))
        np.testing.assert_array_equal(vo.reshape(-1, row)[new_slots], vt.reshape(-1, row))


def test_strided_rows_from_a_fused_projection():
    torch.manual_seed(3)
    n, n_kv, hd, n_q = 300, 8, 128, 32
    qkv = torch.randn(n, (n_q + 2 * n_kv) * hd, device="cuda").to(torch.bfloat16)
    key = qkv[:, n_q * hd:(n_q + n_kv) * hd].view(n, n_kv, hd)
    val = qkv[:, (n_q + n_kv) * hd:].view(n, n_kv, hd)
    assert key.stride(0) == (n_q + 2 * n_kv) * hd
    slots = torch.randperm(64 * 16, device="cuda")[:n].to(torch.int64)
    kc, vc = _run(key, val, slots, 64, 16, 0.05, 0.04)
    ko, vo = _oracle(gpu_util.to_u16(key.contiguous()), gpu_util.to_u16(val.contiguous()),
                     slots.cpu().numpy(), 64, 16, n_kv, hd, 0.05, 0.04)
    np.testing.assert_array_equal(kc, ko)
    np.testing.assert_array_equal(vc, vo)


def test_null_and_bf16_scales():
    torch.manual_seed(4)
    key = (torch.randn(64, 2, 64, device="cuda") * 30).to(torch.bfloat16)
    slots = torch.arange(64, dtype=torch.int64, device="cuda")
    kc, vc = _run(key, key, slots, 4, 16, None, None)
    ko, vo = _oracle(gpu_util.to_u16(key), gpu_util.to_u16(key), slots.cpu().numpy(), 4, 16, 2, 64,
                     1.0, 1.0)
    np.testing.assert_array_equal(kc, ko)
    b = workloads.stored_scale(0.05, "bf16")
    kc, _ = _run(key, key, slots, 4, 16, 0.05, 0.05, sdt=torch.bfloat16)
    ko, _ = _oracle(gpu_util.to_u16(key), gpu_util.to_u16(key), slots.cpu().numpy(), 4, 16, 2, 64, b, b)
    np.testing.assert_array_equal(kc, ko)


def test_device_errors_set_status_and_skip():
    key = torch.ones(4, 1, 8, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.tensor([0, 99, -1, -7], dtype=torch.int64, device="cuda")
    kc, _ = _run(key, key, slots, 2, 2, 0.5, 0.5, status=status)
    assert int(status.item()) == kv.DEV_BAD_SLOT
    flat = kc.reshape(4, 8)
    assert np.all(flat[0] == oracle.e4m3_encode(2.0)) and np.all(flat[1:] == workloads.SENTINEL)
    for bad in (0.0, float("inf"), float("nan")):
        status.zero_()
        kc, vc = _run(key, key, torch.arange(4, dtype=torch.int64, device="cuda"), 2, 2, bad, 0.5,
                      status=status)
        assert int(status.item()) == kv.DEV_BAD_SCALE
        assert np.all(kc == workloads.SENTINEL) and np.all(vc == workloads.SENTINEL)


def test_padding_rows_and_sentinel_survive():
    torch.manual_seed(5)
    key = torch.randn(40, 2, 64, device="cuda").to(torch.bfloat16)
    slots = torch.full((40,), -1, dtype=torch.int64)
    slots[::3] = torch.randperm(64)[: len(slots[::3])]
    kc, vc = _run(key, key, slots.cuda(), 4, 16, 0.05, 0.04)
    ko, vo = _oracle(gpu_util.to_u16(key), gpu_util.to_u16(key), slots.numpy(), 4, 16, 2, 64, 0.05, 0.04)
    np.testing.assert_array_equal(kc, ko)
    np.testing.assert_array_equal(vc, vo)
    assert (kc == workloads.SENTINEL).all(axis=(2, 3)).sum() == 64 - len(slots[::3])


def test_block_is_half_the_bf16_bytes():
    w = workloads.WORKLOADS["llama3_8b"]
    kc = workloads.new_cache(1, w, "cuda")
    bf = torch.empty((1, w.block_size, w.n_kv, w.head_dim), dtype=torch.bfloat16, device="cuda")
    assert 2 * kc.numel() * kc.element_size() == bf.numel() * bf.element_size()
