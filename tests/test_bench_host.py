"""Host-side logic of bench.py, on CPU: replica aggregation over 2 gloo ranks,
clock-sample parsing, and the traffic record's source check."""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r processed (r+1) GB in (r+1)*0.5 s: slowest rank 1.0 s, total 3 GB
    total, slowest, gbs = bench.aggregate((rank + 1) * 1e9, (rank + 1) * 0.5, world)
    bench.barrier(world)
    q.put((rank, total, slowest, gbs))
    dist.destroy_process_group()


def test_replica_aggregation_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, total, slowest, gbs in res:
        assert total == pytest.approx(3e9)
        assert slowest == pytest.approx(1.0)
        assert gbs == pytest.approx(3.0)


def test_single_rank_aggregation_is_identity():
    total, slowest, gbs = bench.aggregate(2e9, 0.5, 1)
    assert (total, slowest, gbs) == (2e9, 0.5, 4.0)


def test_clock_sampler_parsing():
    c = bench.ClockSampler(0)
    c.proc = type("P", (), {"terminate": lambda s: None, "wait": lambda s, timeout: 0})()
    c.lines = ["0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1980, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
               "garbage"]
    r = c.stop()
    assert r["sm_mhz"] == pytest.approx(1972.5)
    assert r["sm_max_mhz"] == 2070
    assert r["reasons"] == ["sw_power_cap"]


def test_traffic_record_requires_matching_source(tmp_path, monkeypatch):
    h = bench.decode_source_hash()
    assert len(h) == 16
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "decode_traffic.json").write_text(json.dumps(
        {"1": {"source_hash": h, "dram_bytes_per_launch": 123},
         "2": {"source_hash": "stale", "dram_bytes_per_launch": 456}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "decode_source_hash", lambda sources=None: h)
    assert bench.recorded_traffic(1) == 123
    assert bench.recorded_traffic(2) is None
    assert bench.recorded_traffic(3) is None


def test_peak_falls_back_without_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6785.2}))
    assert bench.measured_peak()[0] == 6785.2


def test_multi_query_roofline_bound_follows_arithmetic_intensity():
    """The chunked prefill (about 1,350 FLOP per algorithmic byte) is tensor-bound, the
    draft-tree workload (about 240) HBM-bound, against the ridge of the measured peaks."""
    from paged_kv_cache_87_gb300 import inputs
    r1 = bench.mq_roofline(inputs.make_multi_query_config(1), 500e-6)
    r3 = bench.mq_roofline(inputs.make_multi_query_config(3), 300e-6)
    assert r1["bound"] == "tensor" and r1["unit"] == "TFLOP/s"
    assert r3["bound"] == "hbm" and r3["unit"] == "GB/s"
    assert r3["flops_per_byte"] < r3["ridge_flops_per_byte"] < r1["flops_per_byte"]
    assert r3["achieved"] == pytest.approx(r3["algorithmic_bytes"] / 300e-6 / 1e9, rel=1e-3)


def test_oracle_sample_of_a_tree_workload_counts_visible_pairs():
    """The reference arm's oracle sample on draft trees calls the tree oracle and counts,
    per sampled row, the prior context, the token itself and its ancestors."""
    import numpy as np
    from paged_kv_cache_87_gb300 import inputs
    w = inputs.make_tree_verify("host trees", np.random.default_rng(3), [20, 7], [9, 5],
                                kinds=["random", "star"], num_q_heads=4, num_kv_heads=2,
                                head_dim=128, block_size=16, dtype="bf16")
    tflops, secs, flops, desc = bench.mq_oracle_sample(w, 0.05, 2)
    assert tflops > 0 and secs > 0 and "pairs" in desc
    per_row = [4 * w.head_dim * (int(w.context_lens[s]) - int(w.query_start[s + 1] - w.query_start[s])
                                 + 1 + bin(int(w.tree[r])).count("1"))
               for s in range(w.num_seqs)
               for r in range(int(w.query_start[s]), int(w.query_start[s + 1]))]
    assert flops % (4 * w.head_dim) == 0
    k = flops // min(per_row)                               # sampled pairs: at least 8
    assert k >= 8 and min(per_row) * 8 <= flops


def test_per_config_entry_uses_unique_bytes_for_the_roofline():
    """The roofline fraction divides the unique K/V rows (each shared prompt block once)
    by the decode time; the logical rate of a shared-prefix workload is labelled as not
    a roofline, and is absent when nothing is shared."""
    from types import SimpleNamespace
    w = SimpleNamespace(name="shared", kv_read_bytes=4_000_000_000,
                        unique_kv_bytes=1_000_000_000)
    e = bench.per_config_entry(w, [0.5, 0.5], [0.25, 0.25], 8000.0, "flushed", True)
    assert e["decode_us"] == pytest.approx(250.0)
    assert e["step_us"] == pytest.approx(500.0)
    assert e["decode_gbs"] == pytest.approx(4000.0)
    assert e["frac"] == pytest.approx(0.5)
    assert e["logical_kv_gbs_not_a_roofline"] == pytest.approx(16000.0)
    assert e["entry"] == "prefix-aware"
    w2 = SimpleNamespace(name="plain", kv_read_bytes=10**9, unique_kv_bytes=10**9)
    e2 = bench.per_config_entry(w2, [1.0], [0.5], 4000.0, "flushed", False)
    assert e2["frac"] == pytest.approx(0.5) and "logical_kv_gbs_not_a_roofline" not in e2


def test_launch_count_per_step():
    from types import SimpleNamespace
    import numpy as np
    w = SimpleNamespace(q_dtype="bf16", kv_dtype="e4m3", head_dim=128, num_q_heads=32,
                        num_kv_heads=8, step_pairs=np.zeros((32, 2), np.int32))
    # copy, append, shared-prefix detection, plan, decode, merge
    assert bench.launches_per_step(w, True) == 6
    assert bench.launches_per_step(w, False) == 4
    w.num_q_heads = 128                                # 16 heads per kv head: no groups
    assert bench.launches_per_step(w, True) == 4
    w.num_q_heads = 32
    w.step_pairs = np.zeros((0, 2), np.int32)
    w.q_dtype, w.kv_dtype = "f32", "f32"
    assert bench.launches_per_step(w, True) == 3       # append, plan, decode (CUDA cores)


def test_default_workload_is_the_long_context_split_kv_decode():
    args = bench.parse_args([])
    assert args.workload == 3
    from paged_kv_cache_87_gb300 import inputs
    assert "long-context split-KV" in inputs.CONFIG_NAMES[args.workload]
