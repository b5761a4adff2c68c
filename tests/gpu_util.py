"""Helpers shared by the GPU parity tests (test code only).

Parity rules: cache bytes are compared bit for bit; attention outputs must satisfy
|gpu - oracle| <= 2e-3 + 1e-2 * |oracle| element by element (max-abs 2e-3 / rel 1e-2 in
allclose form), the oracle being the double-precision CPU reference on the same
dequantized cache.  The oracle's inputs are the same seeded bf16 K/V/q the GPU sees,
never anything the GPU computed.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import workloads

TOL_ABS = 2e-3
TOL_REL = 1e-2


def to_u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> host uint16 array of its bits."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_attention_close(gpu_out: torch.Tensor, ref: np.ndarray, what: str = ""):
    g = gpu_out.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; worst at {i}: "
            f"gpu={g[i]!r} ref={ref[i]!r}; max_abs={err.max():.3e}")
    return float(err.max())


def scale_pair(w: workloads.Workload, device="cuda"):
    return (workloads.scale_tensor(w.k_scale, w.scale_dtype, device),
            workloads.scale_tensor(w.v_scale, w.scale_dtype, device))


def stored_scales(w: workloads.Workload):
    return workloads.stored_scale(w.k_scale, w.scale_dtype), workloads.stored_scale(w.v_scale, w.scale_dtype)


def oracle_seq_cache(k_rows: torch.Tensor, v_rows: torch.Tensor, block_size: int, ks: float, vs: float):
    """The oracle's own cache for one sequence: its L token rows written to blocks
    0..ceil(L/bs)-1 in order (attention does not depend on the physical order)."""
    L, n_kv, hd = k_rows.shape
    nb = max(1, math.ceil(L / block_size))
    kc = np.full((nb, block_size, n_kv, hd), workloads.SENTINEL, np.uint8)
    vc = kc.copy()
    st = oracle.reshape_and_cache(to_u16(k_rows), to_u16(v_rows), kc, vc,
                                  np.arange(L, dtype=np.int64), block_size, ks, vs)
    assert st == 0
    return kc, vc, np.arange(nb, dtype=np.int32)[None, :]


def oracle_pairs(pairs, k_all: torch.Tensor, v_all: torch.Tensor, q: torch.Tensor,
                 lay: workloads.Layout, w: workloads.Workload, ks: float, vs: float,
                 sm_scale: float = 0.0) -> np.ndarray:
    """Oracle output rows for (seq, head) pairs; k_all/v_all are the bf16 rows of every
    context token in the layout's row order (lay.row_seq / lay.row_pos)."""
    out = np.zeros((len(pairs), w.head_dim), np.float64)
    qh = q.detach().cpu()
    by_seq: dict[int, list[int]] = {}
    for i, (b, _h) in enumerate(pairs):
        by_seq.setdefault(int(b), []).append(i)
    for b, idx in by_seq.items():
        rows = np.nonzero(lay.row_seq == b)[0]
        rows = rows[np.argsort(lay.row_pos[rows])]
        L = int(lay.seq_lens[b])
        assert rows.size == L
        ridx = torch.from_numpy(rows).to(k_all.device)
        kc, vc, bt = oracle_seq_cache(k_all.index_select(0, ridx).cpu(),
                                      v_all.index_select(0, ridx).cpu(), w.block_size, ks, vs)
        pr = np.array([[0, int(pairs[i][1])] for i in idx], np.int32)
        o, st = oracle.paged_decode_attention_pairs(pr, qh[b:b + 1], kc, vc, bt,
                                                    np.array([L], np.int32), ks, vs, sm_scale)
        assert st == 0
        out[idx] = o
    return out
