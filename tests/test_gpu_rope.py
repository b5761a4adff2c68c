"""kvfp8_rope_reshape_and_cache on the GPU vs the CPU oracle: cache bytes bit for bit.
The rotation uses a caller-supplied float32 cos/sin table (see include/kvfp8.h)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import gpu_util

pytestmark = pytest.mark.gpu

kv = pytest.importorskip("fp8_paged_kv_reshape_gb300")


def _table(max_pos, rot, base=10000.0):
    inv = base ** (-np.arange(0, rot, 2, dtype=np.float64) / rot)
    ang = np.arange(max_pos)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


CASES = [  # n_kv, head_dim, rot, neox, src dtype, tokens
    (8, 128, 128, True, torch.bfloat16, 3000),
    (8, 128, 64, True, torch.bfloat16, 1000),
    (8, 128, 128, False, torch.bfloat16, 1000),
    (2, 64, 64, True, torch.bfloat16, 777),
    (2, 64, 32, False, torch.bfloat16, 100),
    (4, 256, 256, True, torch.bfloat16, 500),
    (8, 256, 128, False, torch.bfloat16, 300),
    (1, 128, 16, True, torch.bfloat16, 64),
    (8, 128, 128, True, torch.float32, 600),
    (16, 128, 128, True, torch.bfloat16, 500),   # 2048-element rows: four units a lane
    (4, 128, 128, True, torch.bfloat16, 500),    # 512-element rows: one unit a lane
    (2, 64, 16, False, torch.bfloat16, 100),     # GPT-J over 16 dims: one rotated unit a head
    (4, 64, 32, True, torch.bfloat16, 200),      # NeoX over 32 dims: partner one unit away
]


@pytest.mark.parametrize("case", CASES, ids=[f"nkv{c[0]}_hd{c[1]}_rot{c[2]}_{'neox' if c[3] else 'gptj'}_{str(c[4])[6:]}" for c in CASES])
def test_rope_cache_write_bit_exact(case):
    n_kv, hd, rot, neox, dt, n = case
    g = torch.Generator().manual_seed(n + hd + rot)
    k = (torch.randn(n, n_kv, hd, generator=g) * 3).to(dt)
    v = (torch.randn(n, n_kv, hd, generator=g) * 3).to(dt)
    max_pos = 8192
    pos = torch.randint(0, max_pos, (n,), generator=g, dtype=torch.int64)
    nb, bs = (n + 15) // 16 + 3, 16
    slots = torch.randperm(nb * bs, generator=g)[:n].to(torch.int64)
    slots[::17] = -1
    table = _table(max_pos, rot)
    kc = torch.full((nb, bs, n_kv, hd), 0x5A, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    sc = (torch.tensor([0.05], device="cuda"), torch.tensor([0.04], device="cuda"))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.rope_reshape_and_cache(k.cuda(), v.cuda(), kc, vc, slots.cuda(), pos.cuda(),
                              torch.from_numpy(table).cuda(), neox, *sc, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ko = np.full((nb, bs, n_kv, hd), 0x5A, np.uint8)
    vo = ko.copy()
    src = oracle.F32 if dt == torch.float32 else oracle.BF16
    kin = k.numpy() if dt == torch.float32 else k
    vin = v.numpy() if dt == torch.float32 else v
    assert oracle.rope_reshape_and_cache(kin, vin, ko, vo, slots.numpy(), pos.numpy(), table, rot,
                                         neox, bs, 0.05, 0.04, src_dtype=src) == 0
    got_k = kc.cpu().numpy()
    bad = np.argwhere(got_k != ko)
    assert bad.shape[0] == 0, bad[:5]
    np.testing.assert_array_equal(vc.cpu().numpy(), vo)


def test_rope_changes_k_but_not_v_and_bad_positions_are_flagged():
    w = workloads.WORKLOADS["llama3_8b"]
    n = 64
    k, v = workloads.make_kv(w, n, "cuda")
    table = torch.from_numpy(_table(128, 128)).cuda()
    slots = torch.arange(n, dtype=torch.int64, device="cuda")
    pos = torch.arange(n, dtype=torch.int64, device="cuda") + 1
    pos[5] = 128      # out of range
    pos[9] = -3
    kc = torch.zeros(4, 16, 8, 128, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    kp, vp = kc.clone(), vc.clone()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.rope_reshape_and_cache(k, v, kc, vc, slots, pos, table, True, status=st)
    kv.reshape_and_cache(k, v, kp, vp, slots)
    torch.cuda.synchronize()
    assert int(st.item()) == kv.DEV_BAD_SLOT
    flat_k, flat_v = kc.view(64, -1), vc.view(64, -1)
    assert torch.all(flat_k[[5, 9]] == 0) and torch.all(flat_v[[5, 9]] == 0)  # skipped
    ok = [i for i in range(64) if i not in (5, 9)]
    assert torch.equal(flat_v[ok], vp.view(64, -1)[ok])                      # V untouched by rope
    assert not torch.equal(flat_k[ok], kp.view(64, -1)[ok])                  # K rotated


@pytest.mark.parametrize("scales", [(0.05, 0.04), (1e-25, 3.7e22)], ids=["fast_divide", "slow_divide"])
def test_rope_divide_paths(scales):
    # scales inside the reciprocal-and-corrections range and outside it (IEEE divide)
    n_kv, hd, rot, n = 8, 128, 128, 2000
    g = torch.Generator().manual_seed(99)
    k = (torch.randn(n, n_kv, hd, generator=g) * 3).to(torch.bfloat16)
    v = (torch.randn(n, n_kv, hd, generator=g) * 3).to(torch.bfloat16)
    pos = torch.randint(0, 4096, (n,), generator=g, dtype=torch.int64)
    nb, bs = (n + 15) // 16 + 3, 16
    slots = torch.randperm(nb * bs, generator=g)[:n].to(torch.int64)
    slots[::13] = -1
    table = _table(4096, rot)
    ks = np.float32(scales[0]).item()
    vs = np.float32(scales[1]).item()
    kc = torch.full((nb, bs, n_kv, hd), 0x5A, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    kv.rope_reshape_and_cache(k.cuda(), v.cuda(), kc, vc, slots.cuda(), pos.cuda(),
                              torch.from_numpy(table).cuda(), True,
                              torch.tensor([ks], device="cuda"), torch.tensor([vs], device="cuda"))
    torch.cuda.synchronize()
    ko = np.full((nb, bs, n_kv, hd), 0x5A, np.uint8)
    vo = ko.copy()
    assert oracle.rope_reshape_and_cache(k, v, ko, vo, slots.numpy(), pos.numpy(), table, rot,
                                         True, bs, ks, vs) == 0
    np.testing.assert_array_equal(kc.cpu().numpy(), ko)
    np.testing.assert_array_equal(vc.cpu().numpy(), vo)


def test_rope_special_values_bit_exact():
    # NaN, infinities, values that overflow E4M3 after the divide, zeros of both signs and
    # subnormal quotients, in K (rotated) and V; every byte against the oracle
    n_kv, hd, rot, n = 8, 128, 128, 700
    g = torch.Generator().manual_seed(5)
    k = torch.randn(n, n_kv, hd, generator=g) * 3
    v = torch.randn(n, n_kv, hd, generator=g) * 3
    specials = torch.tensor([float("nan"), float("inf"), -float("inf"), 1e30, -1e30, 0.0, -0.0,
                             1e-38, -3e-39, 448.0 * 0.05, 500.0])
    for t in (k, v):
        idx = torch.randint(0, t.numel(), (4000,), generator=g)
        t.view(-1)[idx] = specials[torch.randint(0, specials.numel(), (4000,), generator=g)]
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    pos = torch.randint(0, 4096, (n,), generator=g, dtype=torch.int64)
    nb, bs = (n + 15) // 16 + 3, 16
    slots = torch.randperm(nb * bs, generator=g)[:n].to(torch.int64)
    table = _table(4096, rot)
    kc = torch.full((nb, bs, n_kv, hd), 0x5A, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    kv.rope_reshape_and_cache(k.cuda(), v.cuda(), kc, vc, slots.cuda(), pos.cuda(),
                              torch.from_numpy(table).cuda(), True,
                              torch.tensor([0.05], device="cuda"), torch.tensor([0.04], device="cuda"))
    torch.cuda.synchronize()
    ko = np.full((nb, bs, n_kv, hd), 0x5A, np.uint8)
    vo = ko.copy()
    assert oracle.rope_reshape_and_cache(k, v, ko, vo, slots.numpy(), pos.numpy(), table, rot,
                                         True, bs, 0.05, 0.04) == 0
    np.testing.assert_array_equal(kc.cpu().numpy(), ko)
    np.testing.assert_array_equal(vc.cpu().numpy(), vo)
