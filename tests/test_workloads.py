"""Host-side checks of the seeded input generators (CPU only)."""
import numpy as np
import torch

import workloads


def test_layouts_are_deterministic_and_valid():
    for name, w in workloads.WORKLOADS.items():
        small = {"num_seqs": 4, "context": 300} if name != "tiny" else {}
        a = workloads.make_layout(w, **small)
        b = workloads.make_layout(w, **small)
        np.testing.assert_array_equal(a.slot_mapping, b.slot_mapping)
        np.testing.assert_array_equal(a.block_tables, b.block_tables)
        valid = a.slot_mapping[a.slot_mapping >= 0]
        assert valid.size == len(set(valid.tolist()))                 # no slot written twice
        assert valid.max() < a.num_blocks * w.block_size
        used = a.block_tables[a.block_tables >= 0]
        assert used.size == len(set(used.tolist())) and used.max() < a.num_blocks
        for i, L in enumerate(a.seq_lens):
            nb = int(np.ceil(L / w.block_size))
            assert np.all(a.block_tables[i, :nb] >= 0) and np.all(a.block_tables[i, nb:] == -1)


def test_full_size_layouts_have_the_stated_shapes():
    w = workloads.WORKLOADS["llama3_8b"]
    lay = workloads.make_layout(w)
    assert lay.num_seqs == 64 and np.all(lay.seq_lens == 4096) and lay.num_blocks == 16384
    w = workloads.WORKLOADS["long_context"]
    lay = workloads.make_layout(w)
    assert lay.num_seqs == 8 and lay.seq_lens.min() >= 32768 and lay.seq_lens.max() <= 131072
    w = workloads.WORKLOADS["prefill_write"]
    lay = workloads.make_layout(w)
    assert lay.slot_mapping.size == 32768 and lay.num_blocks == 65536
    pads = np.count_nonzero(lay.slot_mapping == -1)
    assert 0 < pads <= 16 * 127
    w = workloads.WORKLOADS["mixed_serving"]
    lay = workloads.make_layout(w)
    assert lay.num_seqs == 256 and lay.seq_lens.min() >= 16 and lay.seq_lens.max() <= 32768
    assert lay.block_tables.shape[1] == int(np.ceil(lay.seq_lens.max() / 32))


def test_values_are_seeded_bf16():
    w = workloads.WORKLOADS["llama3_8b"]
    k1, v1 = workloads.make_kv(w, 2000)
    k2, _ = workloads.make_kv(w, 2000)
    assert k1.dtype == torch.bfloat16 and torch.equal(k1, k2) and not torch.equal(k1, v1)
    # 0.1% outliers x20 push some |x|/0.05 past the E4M3 maximum (saturation exercised)
    assert (k1.float().abs() / 0.05 >= 448).any()
    q = workloads.make_query(w, 3)
    assert q.shape == (3, 32, 128)
