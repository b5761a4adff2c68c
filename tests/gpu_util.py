"""Helpers shared by the GPU parity tests (test code only).

Parity rules: cache bytes are compared bit for bit; attention outputs must satisfy
|gpu - oracle| <= 2e-3 + 1e-2 * |oracle| element by element (max-abs 2e-3 / rel 1e-2 in
allclose form), the oracle being the double-precision CPU reference on the same
dequantized cache.  The oracle's inputs are the same seeded bf16 K/V/q the GPU sees,
never anything the GPU computed.
"""
from __future__ import annotations

import concurrent.futures as cf
import math
import os

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


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_cache_threaded(k_u16: np.ndarray, v_u16: np.ndarray, slots: np.ndarray,
                          num_blocks: int, w: workloads.Workload, ks: float, vs: float,
                          kc: np.ndarray | None = None, vc: np.ndarray | None = None):
    """The oracle's whole cache for host bf16 rows (uint16 [rows, n_kv, head_dim]) written at
    ``slots``: the unchanged single-threaded oracle, called on disjoint row ranges from
    parallel threads (its C calls release the interpreter lock).  The valid slots are
    distinct, so the ranges write disjoint cache rows and the result does not depend on the
    split.  Starts from sentinel-filled caches unless kc/vc are given."""
    valid = slots[slots >= 0]
    assert np.unique(valid).size == valid.size, "overlapping slots would make the split matter"
    if kc is None:
        kc = np.full((num_blocks, w.block_size, w.n_kv, w.head_dim), workloads.SENTINEL, np.uint8)
        vc = kc.copy()
    n = slots.size
    parts = max(1, min(host_threads(), n // 4096 + 1))
    bounds = np.linspace(0, n, parts + 1).astype(np.int64)

    def run(i):
        a, b = int(bounds[i]), int(bounds[i + 1])
        if a == b:
            return 0
        return oracle.reshape_and_cache(k_u16[a:b], v_u16[a:b], kc, vc, slots[a:b],
                                        w.block_size, ks, vs)

    with cf.ThreadPoolExecutor(max_workers=parts) as ex:
        sts = list(ex.map(run, range(parts)))
    assert all(s == 0 for s in sts), sts
    return kc, vc


def oracle_pairs_threaded(pairs, q: torch.Tensor, kc: np.ndarray, vc: np.ndarray,
                          block_tables: np.ndarray, seq_lens: np.ndarray, ks: float, vs: float,
                          sm_scale: float = 0.0) -> np.ndarray:
    """Oracle decode attention rows for (seq, head) pairs over the oracle's own cache, the
    pairs split over parallel threads (each runs the unchanged single-threaded oracle)."""
    qh = to_u16(q)
    pr = np.asarray(pairs, np.int32).reshape(-1, 2)
    parts = max(1, min(host_threads(), pr.shape[0]))
    chunks = np.array_split(np.arange(pr.shape[0]), parts)

    def run(idx):
        o, st = oracle.paged_decode_attention_pairs(pr[idx], qh, kc, vc, block_tables, seq_lens,
                                                    ks, vs, sm_scale)
        assert st == 0
        return o

    with cf.ThreadPoolExecutor(max_workers=parts) as ex:
        outs = list(ex.map(run, chunks))
    return np.concatenate(outs, axis=0) if outs else np.zeros((0, kc.shape[3]))


def serving_write_rows(w: workloads.Workload, lay: workloads.Layout):
    """Slots of the serving step's one new token per sequence, at position len-1."""
    last = lay.seq_lens.astype(np.int64) - 1
    return lay.block_tables[np.arange(lay.num_seqs), last // w.block_size].astype(np.int64) \
        * w.block_size + last % w.block_size


def full_size_workload(name: str):
    """A workload at its full size written through the GPU path exactly as a bench step
    does: every context row with kvfp8_reshape_and_cache, then (the serving workload) one
    new token per sequence at len-1.  Returns the GPU caches and the host inputs."""
    import fp8_paged_kv_reshape_gb300 as kv

    w = workloads.WORKLOADS[name]
    lay = workloads.make_layout(w)
    k, v = workloads.make_kv(w, lay.slot_mapping.size, "cuda")
    ksc, vsc = scale_pair(w)
    kc = workloads.new_cache(lay.num_blocks, w, "cuda")
    vc = kc.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kv.reshape_and_cache(k, v, kc, vc, torch.from_numpy(lay.slot_mapping).cuda(), ksc, vsc,
                         status=status)
    new = None
    if w.kind == "mixed":
        kn, vn = workloads.make_new_token_kv(w, lay.num_seqs, "cuda")
        new_slots = serving_write_rows(w, lay)
        kv.reshape_and_cache(kn, vn, kc, vc, torch.from_numpy(new_slots).cuda(), ksc, vsc,
                             status=status)
        new = (to_u16(kn), to_u16(vn), new_slots)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return dict(w=w, lay=lay, k=k, v=v, kc=kc, vc=vc, ksc=ksc, vsc=vsc, new=new)


def oracle_full_cache(case):
    """The oracle's cache for a full_size_workload case, from the same host inputs."""
    w, lay = case["w"], case["lay"]
    ks, vs = stored_scales(w)
    ko, vo = oracle_cache_threaded(to_u16(case["k"]), to_u16(case["v"]), lay.slot_mapping,
                                   lay.num_blocks, w, ks, vs)
    if case["new"] is not None:
        kn, vn, new_slots = case["new"]
        assert oracle.reshape_and_cache(kn, vn, ko, vo, new_slots, w.block_size, ks, vs) == 0
    return ko, vo
