"""Seeded synthetic inputs for the FP8 paged KV-cache path.

This module only draws inputs: sequence lengths, block tables, slot mappings,
bf16 K/V/q values and scale tensors.  It holds none of the method's arithmetic
(no quantization, no attention), so both the CUDA library's tests/benchmark and
the CPU oracle can be fed from it.

Recipe (one per workload; seed = 1000 + workload index):
  * layout (lengths, physical block permutation, slots) from numpy
    ``Generator(PCG64(seed))`` -- stable across machines and numpy versions;
  * K, V, q values as float32 normals from a seeded ``torch.Generator`` on the
    target device (child seeds seed*16+1/2/3), scaled by the workload's std,
    optional outliers multiplied before rounding, then rounded to bf16 (RNE);
  * caches are pre-filled with the sentinel byte 0x5A by the caller.

Workloads (the shapes the source pages' problem statement names):
  tiny           4 q / 2 kv heads, head_dim 64, block 16, lengths {17,33,64,100},
                 N(0,1), k_scale 0.05, v_scale 0.04, 32-block pool shuffled
  llama3_8b      32 q / 8 kv, head_dim 128, block 16, 64 seqs x 4096 tokens,
                 K/V ~ N(0,1.5) with 0.1% outliers x20, q ~ N(0,1), fp32 scales
  long_context   64 q / 8 kv, head_dim 128, block 16, 8 seqs with lengths
                 uniform in [32768, 131072], N(0,1), bf16-stored scales
  prefill_write  8 kv, head_dim 128, block 16: 32768 new rows across 16 seqs
                 (2048 rows each, the last U[0,127] rows of each are padding,
                 slot -1), K/V ~ N(0,2), 1M-slot pool (65536 blocks)
  mixed_serving  40 q / 8 kv, head_dim 128, block 32, 256 seqs with lengths
                 log-uniform in [16, 32768]; one new token per seq is written
                 at position len-1, then decode
Scales not named by a workload are k_scale 0.05 and v_scale 0.04.

Rope tables (for the rope-fused cache write) are the model's constant input: the
standard rotary table with base theta, cos(p * theta^(-2i/rot)) then sin(...), computed
in float64 and rounded once to float32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

K_SCALE = 0.05
V_SCALE = 0.04
SENTINEL = 0x5A


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    n_q: int
    n_kv: int
    head_dim: int
    block_size: int
    kind: str  # "decode" | "write" | "mixed"
    kv_std: float = 1.0
    q_std: float = 1.0
    outlier_frac: float = 0.0
    outlier_mult: float = 1.0
    scale_dtype: str = "f32"  # "f32" | "bf16"
    k_scale: float = K_SCALE
    v_scale: float = V_SCALE
    extra: dict = field(default_factory=dict)

    @property
    def seed(self) -> int:
        return 1000 + self.index


WORKLOADS = {
    "tiny": Workload("tiny", 0, 4, 2, 64, 16, "decode", extra={"lengths": [17, 33, 64, 100],
                                                                 "pool": 32}),
    "llama3_8b": Workload("llama3_8b", 1, 32, 8, 128, 16, "decode", kv_std=1.5,
                          outlier_frac=1e-3, outlier_mult=20.0,
                          extra={"num_seqs": 64, "context": 4096}),
    "long_context": Workload("long_context", 2, 64, 8, 128, 16, "decode", scale_dtype="bf16",
                             extra={"num_seqs": 8, "len_lo": 32768, "len_hi": 131072}),
    "prefill_write": Workload("prefill_write", 3, 8, 8, 128, 16, "write", kv_std=2.0,
                              extra={"num_seqs": 16, "rows_per_seq": 2048, "pad_max": 127,
                                     "pool_slots": 1 << 20}),
    "mixed_serving": Workload("mixed_serving", 4, 40, 8, 128, 32, "mixed",
                              extra={"num_seqs": 256, "len_lo": 16, "len_hi": 32768}),
}


@dataclass
class Layout:
    """Paged layout of one workload (host numpy arrays)."""
    seq_lens: np.ndarray        # int32 [num_seqs]
    block_tables: np.ndarray    # int32 [num_seqs, max_blocks_per_seq], unused entries -1
    num_blocks: int
    slot_mapping: np.ndarray    # int64 [num_rows]: destination slot of each written row (-1 = pad)
    row_seq: np.ndarray         # int32 [num_rows]: which sequence each written row belongs to
    row_pos: np.ndarray         # int32 [num_rows]: position of the row in its sequence (-1 = pad)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


def _tables(rng: np.random.Generator, lens: np.ndarray, block_size: int, pool_blocks: int | None):
    need = [int(math.ceil(int(L) / block_size)) for L in lens]
    total = int(sum(need))
    num_blocks = total if pool_blocks is None else int(pool_blocks)
    assert num_blocks >= total
    perm = rng.permutation(num_blocks).astype(np.int32)
    max_b = max(1, max(need) if need else 1)
    bt = np.full((len(lens), max_b), -1, dtype=np.int32)
    at = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[at:at + n]
        at += n
    return bt, num_blocks


def _context_rows(lens: np.ndarray, bt: np.ndarray, block_size: int):
    """Slots of every context token 0..len-1 of every sequence, in sequence order."""
    seqs, poss, slots = [], [], []
    for i, L in enumerate(lens):
        L = int(L)
        t = np.arange(L, dtype=np.int64)
        seqs.append(np.full(L, i, dtype=np.int32))
        poss.append(t.astype(np.int32))
        slots.append(bt[i, t // block_size].astype(np.int64) * block_size + t % block_size)
    cat = (lambda xs, dt: np.concatenate(xs).astype(dt) if xs else np.zeros(0, dt))
    return cat(slots, np.int64), cat(seqs, np.int32), cat(poss, np.int32)


def make_layout(w: Workload, *, num_seqs: int | None = None, context: int | None = None,
                lengths: list[int] | None = None) -> Layout:
    """Draw the workload's lengths, block tables and slot mapping (seeded).

    ``num_seqs`` / ``context`` / ``lengths`` override the workload's sizes for
    reduced parity cases; the drawing recipe stays the same.
    """
    rng = np.random.Generator(np.random.PCG64(w.seed))
    bs = w.block_size
    e = w.extra
    if w.kind == "write":
        n = num_seqs or e["num_seqs"]
        rows = context or e["rows_per_seq"]
        pads = rng.integers(0, min(e["pad_max"], rows - 1) + 1, size=n)
        valid = (rows - pads).astype(np.int32)
        pool_blocks = e["pool_slots"] // bs
        bt, num_blocks = _tables(rng, valid, bs, pool_blocks)
        slots = np.full(n * rows, -1, dtype=np.int64)
        row_seq = np.repeat(np.arange(n, dtype=np.int32), rows)
        row_pos = np.full(n * rows, -1, dtype=np.int32)
        for i in range(n):
            t = np.arange(int(valid[i]), dtype=np.int64)
            slots[i * rows:i * rows + valid[i]] = bt[i, t // bs].astype(np.int64) * bs + t % bs
            row_pos[i * rows:i * rows + valid[i]] = t
        return Layout(valid, bt, num_blocks, slots, row_seq, row_pos)

    if lengths is not None:
        lens = np.asarray(lengths, dtype=np.int32)
    elif "lengths" in e:
        lens = np.asarray(e["lengths"], dtype=np.int32)
    elif "context" in e:
        lens = np.full(num_seqs or e["num_seqs"], context or e["context"], dtype=np.int32)
    elif w.kind == "mixed":
        n = num_seqs or e["num_seqs"]
        lo, hi = math.log(e["len_lo"]), math.log(e["len_hi"])
        lens = np.floor(np.exp(rng.uniform(lo, hi, size=n))).astype(np.int64)
        lens = np.clip(lens, e["len_lo"], e["len_hi"]).astype(np.int32)
        if context is not None:  # reduced case: rescale into [len_lo, context]
            lens = np.clip((lens.astype(np.int64) * context) // e["len_hi"], 1, context).astype(np.int32)
    else:
        n = num_seqs or e["num_seqs"]
        hi = context or e["len_hi"]
        lo = min(e["len_lo"], hi)
        lens = rng.integers(lo, hi + 1, size=n).astype(np.int32)
    pool = e.get("pool")
    bt, num_blocks = _tables(rng, lens, bs, pool)
    slots, row_seq, row_pos = _context_rows(lens, bt, bs)
    return Layout(lens, bt, num_blocks, slots, row_seq, row_pos)


def _normal_bf16(shape, std: float, seed: int, device, outlier_frac=0.0, outlier_mult=1.0):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    x.mul_(std)
    if outlier_frac > 0.0:
        sel = torch.rand(shape, generator=g, device=device) < outlier_frac
        x[sel] *= outlier_mult
    return x.to(torch.bfloat16)


def make_kv(w: Workload, num_rows: int, device="cpu"):
    """bf16 K and V rows [num_rows, n_kv, head_dim] for the workload (seeded)."""
    shape = (num_rows, w.n_kv, w.head_dim)
    k = _normal_bf16(shape, w.kv_std, w.seed * 16 + 2, device, w.outlier_frac, w.outlier_mult)
    v = _normal_bf16(shape, w.kv_std, w.seed * 16 + 3, device, w.outlier_frac, w.outlier_mult)
    return k, v


def make_query(w: Workload, num_seqs: int, device="cpu"):
    """bf16 decode queries [num_seqs, n_q, head_dim] (seeded)."""
    return _normal_bf16((num_seqs, w.n_q, w.head_dim), w.q_std, w.seed * 16 + 1, device)


def make_new_token_kv(w: Workload, num_seqs: int, device="cpu"):
    """bf16 K/V of the one new token per sequence of a serving step (seeded)."""
    shape = (num_seqs, w.n_kv, w.head_dim)
    k = _normal_bf16(shape, w.kv_std, w.seed * 16 + 4, device)
    v = _normal_bf16(shape, w.kv_std, w.seed * 16 + 5, device)
    return k, v


def rope_table(max_pos: int, rot: int, theta: float = 500000.0) -> np.ndarray:
    """float32 [max_pos, rot]: cos of every (position, pair) angle, then sin."""
    inv = theta ** (-np.arange(0, rot, 2, dtype=np.float64) / rot)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def scale_tensor(value: float, dtype: str, device="cpu") -> torch.Tensor:
    """A per-layer scalar scale stored as a 1-element fp32 or bf16 tensor."""
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    return torch.tensor([value], dtype=dt, device=device)


def stored_scale(value: float, dtype: str) -> float:
    """The float a stored scale holds (bf16 storage rounds it once, RNE)."""
    return float(scale_tensor(value, dtype).float().item())


def new_cache(num_blocks: int, w: Workload, device="cpu") -> torch.Tensor:
    """A uint8 cache [num_blocks, block_size, n_kv, head_dim] filled with the sentinel."""
    return torch.full((num_blocks, w.block_size, w.n_kv, w.head_dim), SENTINEL,
                      dtype=torch.uint8, device=device)
