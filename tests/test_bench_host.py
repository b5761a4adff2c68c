"""Host-side logic of bench.py on CPU: the multi-rank aggregation under a world_size-2
gloo group, and the reference arm (the CPU oracle) on the tiny workload."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench

    mx = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
    torch.distributed.barrier()
    out_q.put((rank, mx, bench.whole_job_gbs(1_000_000, 10, world, mx)))
    torch.distributed.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [3.0, 5.0]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, val in res:
        assert mx == 5.0  # the slowest rank's time
        assert val == pytest.approx(2 * 1_000_000 * 10 / 5e-3 / 1e9)


def _bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=e, timeout=600)


def test_reference_arm_prints_one_line_with_the_contract_keys():
    r = _bench("--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["config"]["workload"] == "tiny"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    r = _bench("--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3",
               env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_byte_accounting():
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import workloads

    w = workloads.WORKLOADS["llama3_8b"]
    slots = np.array([0, -1, 5, 7], np.int64)
    assert bench.reshape_bytes(w, slots) == 3 * 1024 * 6 + 8 * 4
    lens = np.array([16, 17, 0], np.int32)
    per = bench.decode_bytes(w, lens)
    assert per == 2 * 33 * 1024 + 4 * (1 + 2 + 0) + 4 * 3 + 2 * 2 * 3 * 32 * 128


def test_byte_accounting_of_the_variants():
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import workloads

    w = workloads.WORKLOADS["llama3_8b"]
    slots = np.array([0, -1, 5, 7], np.int64)
    # a bf16 side writes two bytes per element
    assert bench.reshape_bytes(w, slots, 2, 2, 1) == 3 * 1024 * 7 + 8 * 4
    # rope: + the 8-byte position of every row + one float32 table row per distinct position
    pos = np.array([3, 0, 3, 9], np.int64)
    assert bench.reshape_bytes(w, slots, 2, 1, 1, pos, 128) == \
        3 * 1024 * 6 + 8 * 4 + 8 * 4 + 2 * 128 * 4
    lens = np.array([16, 17, 0], np.int32)
    assert bench.decode_bytes(w, lens, 1, 2) == \
        3 * 33 * 1024 + 4 * (1 + 2 + 0) + 4 * 3 + 2 * 2 * 3 * 32 * 128
    # multi-query: the query/output rows and query_start_loc
    assert bench.decode_bytes(w, lens, query_rows=12) == \
        2 * 33 * 1024 + 4 * (1 + 2 + 0) + 4 * 3 + 2 * 2 * 12 * 32 * 128 + 4 * 4
    assert bench.query_len(w, "multi") == 4 and bench.query_len(w, "fp8") == 1


def test_serving_step_rows_are_the_last_query_tokens():
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import workloads

    w = workloads.WORKLOADS["mixed_serving"]
    lay = workloads.make_layout(w, num_seqs=5)
    slots, pos = bench.step_rows(w, lay, 3)
    assert slots.shape == (15,) and pos.shape == (15,)
    for b in range(5):
        L = int(lay.seq_lens[b])
        assert list(pos[3 * b:3 * b + 3]) == [L - 3, L - 2, L - 1]
        # the same slots the context layout gives those positions
        ctx = lay.slot_mapping[(lay.row_seq == b)]
        assert list(slots[3 * b:3 * b + 3]) == list(ctx[L - 3:L])


def test_reference_arm_runs_each_variant():
    for variant in ("rope", "k_bf16", "multi", "prefill"):
        r = _bench("--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3",
                   "--variant", variant)
        assert r.returncode == 0, r.stderr
        d = json.loads(r.stdout.strip().splitlines()[-1])
        assert d["config"]["variant"] == variant and d["value"] > 0


def test_cpu_baselines_report_their_threads():
    sys.path.insert(0, ROOT)
    import bench

    one = bench.cpu_baseline("tiny", target_s=0.2)
    allc = bench.cpu_baseline_all_cores("tiny", target_s=0.3)
    assert one["cores"] == 1 and one["kind"] == "oracle" and one["value"] > 0
    assert allc["cores"] == bench.host_cores() >= 1 and allc["value"] > 0
    assert "threads" in allc["sample"]


def test_prefill_flops_count_the_causal_pairs():
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import workloads

    w = workloads.WORKLOADS["llama3_8b"]
    lens = np.array([5, 8], np.int64)
    # 3 new tokens: sequence 0 sees 3, 4, 5 keys; sequence 1 sees 6, 7, 8
    assert bench.attention_flops(w, lens, 3) == 4 * 128 * 32 * (3 + 4 + 5 + 6 + 7 + 8)
    assert bench.query_len(w, "prefill", np.array([4096, 4096])) == 512
    assert bench.query_len(w, "prefill", np.array([4096, 17])) == 17


def test_cpu_sample_of_a_chunk_is_its_last_tokens_exactly():
    # the CPU baseline of the multi-query forms attends with the last m of a sequence's new
    # tokens: with the same cache and length, those rows equal the full chunk's last m rows
    sys.path.insert(0, ROOT)
    import numpy as np

    import bench
    import oracle
    import workloads

    w = workloads.WORKLOADS["llama3_8b"]
    assert bench.sampled_queries(w, 512, 4096) == 4
    assert bench.sampled_queries(w, 512, 1 << 20) == 1      # never fewer than one token
    assert bench.sampled_queries(w, 3, 10) == 3             # never more than the chunk
    g = torch.Generator().manual_seed(3)
    L, n, m, bs = 40, 8, 3, 16
    k = torch.randn(L, 2, 64, generator=g).to(torch.bfloat16)
    v = torch.randn(L, 2, 64, generator=g).to(torch.bfloat16)
    kc = np.zeros((3, bs, 2, 64), np.uint8)
    vc = kc.copy()
    assert oracle.reshape_and_cache(k, v, kc, vc, np.arange(L), bs, 0.05, 0.05) == 0
    q = torch.randn(n, 4, 64, generator=g).to(torch.bfloat16)
    bt = np.arange(3, dtype=np.int32)[None, :]
    lens = np.array([L], np.int32)
    full, st = oracle.paged_attention_multi(q, np.array([0, n], np.int32), kc, vc, bt, lens,
                                            0.05, 0.05)
    part, st2 = oracle.paged_attention_multi(q[n - m:], np.array([0, m], np.int32), kc, vc, bt,
                                             lens, 0.05, 0.05)
    assert st == st2 == 0
    np.testing.assert_array_equal(np.asarray(part), np.asarray(full)[n - m:])
