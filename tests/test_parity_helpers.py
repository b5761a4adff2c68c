"""The parallel oracle helpers the full-size GPU parity tests use give exactly what one
single-threaded oracle call gives (CPU only)."""
import numpy as np
import torch

import oracle
import workloads
from tests import gpu_util


def test_threaded_cache_equals_one_call():
    w = workloads.WORKLOADS["llama3_8b"]
    lay = workloads.make_layout(w, num_seqs=3, context=700)
    k, v = workloads.make_kv(w, lay.slot_mapping.size, "cpu")
    ks, vs = gpu_util.stored_scales(w)
    ku, vu = gpu_util.to_u16(k), gpu_util.to_u16(v)
    ko, vo = gpu_util.oracle_cache_threaded(ku, vu, lay.slot_mapping, lay.num_blocks, w, ks, vs)
    k1 = workloads.new_cache(lay.num_blocks, w).numpy()
    v1 = k1.copy()
    assert oracle.reshape_and_cache(ku, vu, k1, v1, lay.slot_mapping, w.block_size, ks, vs) == 0
    np.testing.assert_array_equal(ko, k1)
    np.testing.assert_array_equal(vo, v1)


def test_threaded_cache_skips_padding_rows():
    w = workloads.WORKLOADS["prefill_write"]
    lay = workloads.make_layout(w, num_seqs=2, context=300)
    k, v = workloads.make_kv(w, lay.slot_mapping.size, "cpu")
    ku, vu = gpu_util.to_u16(k), gpu_util.to_u16(v)
    ko, vo = gpu_util.oracle_cache_threaded(ku, vu, lay.slot_mapping, lay.num_blocks, w, 0.05,
                                            0.04)
    k1 = workloads.new_cache(lay.num_blocks, w).numpy()
    v1 = k1.copy()
    assert oracle.reshape_and_cache(ku, vu, k1, v1, lay.slot_mapping, w.block_size, 0.05,
                                    0.04) == 0
    np.testing.assert_array_equal(ko, k1)
    np.testing.assert_array_equal(vo, v1)


def test_threaded_pairs_equal_the_full_decode():
    w = workloads.WORKLOADS["tiny"]
    lay = workloads.make_layout(w)
    k, v = workloads.make_kv(w, lay.slot_mapping.size, "cpu")
    q = workloads.make_query(w, lay.num_seqs, "cpu")
    ks, vs = gpu_util.stored_scales(w)
    ko, vo = gpu_util.oracle_cache_threaded(gpu_util.to_u16(k), gpu_util.to_u16(v),
                                            lay.slot_mapping, lay.num_blocks, w, ks, vs)
    full, st = oracle.paged_decode_attention(q, ko, vo, lay.block_tables, lay.seq_lens, ks, vs)
    assert st == 0
    pairs = [(b, h) for b in range(lay.num_seqs) for h in range(w.n_q)][::-1]
    got = gpu_util.oracle_pairs_threaded(pairs, q, ko, vo, lay.block_tables, lay.seq_lens, ks, vs)
    np.testing.assert_array_equal(got, np.stack([full[b, h] for b, h in pairs]))


def test_serving_rows_are_each_sequences_last_slot():
    w = workloads.WORKLOADS["mixed_serving"]
    lay = workloads.make_layout(w, num_seqs=6)
    slots = gpu_util.serving_write_rows(w, lay)
    for b in range(lay.num_seqs):
        ctx = lay.slot_mapping[lay.row_seq == b]
        assert slots[b] == ctx[int(lay.seq_lens[b]) - 1]
