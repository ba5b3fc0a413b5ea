"""Host logic of the multi-rank bench path, run as two gloo ranks on CPU:
per-rank batches differ but share a shape, the step time is the MAX over
ranks, and the whole-job value counts every rank's bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from paged_kv_cache_226_gb300 import inputs as pin
        w = pin.build_workload("tiny", seed=bench.rank_seed("tiny", rank))
        local_ms = 1.0 + rank                      # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms)
        q.put((rank, ms, int(w.context_lens.sum()), w.q.shape, float(w.q.float().sum()),
               bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_sharding():
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
    (r0, ms0, n0, s0, q0, env0), (r1, ms1, n1, s1, q1, env1) = res
    assert ms0 == ms1 == 2.0                      # MAX over ranks on both
    assert s0 == s1 and n0 == n1                  # same shape (tiny has fixed lengths)
    assert q0 != q1                               # different draws per rank
    assert env0 == (0, 2, 0) and env1 == (1, 2, 1)


def test_whole_job_value_counts_all_ranks():
    import bench
    assert bench.whole_job_gbs(1_000_000_000, 4, 2.0) == pytest.approx(2000.0)
    assert bench.max_over_ranks(3.5) == 3.5       # no process group: identity


def test_prefill_flops_counts_every_attended_key():
    """The closed form in bench.prefill_flops against a count over every new
    token's position (4 D FLOPs per query head per attended key)."""
    import bench
    from paged_kv_cache_226_gb300 import inputs as pin
    w = pin.build_prefill_workload(params=dict(dtype="bf16", lens=[1, 17, 300, 64, 5],
                                               chunks=[1, 17, 29, 0, 3], num_q_heads=8,
                                               num_kv_heads=2, head_dim=64, block_size=16),
                                   seed=5)
    attended = 0
    for L, C in zip(w.context_lens.tolist(), (w.query_start[1:] - w.query_start[:-1]).tolist()):
        for i in range(C):
            attended += (L - C + i) + 1            # keys 0 .. position of new token i
    assert bench.prefill_flops(w) == 4 * 64 * 8 * attended


def test_profiled_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    """A committed DRAM-traffic figure is reported only while the kernel's
    sources hash to the value it was captured on."""
    import json
    import bench
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"source_sha256_16": bench.source_hash("paged_prefill"), "dram_bytes_per_launch": 1234}
    (prof / "paged_prefill_w.json").write_text(json.dumps(rec))
    assert bench.profiled_traffic("w", "paged_prefill") == 1234
    rec["source_sha256_16"] = "0" * 16
    (prof / "paged_prefill_w.json").write_text(json.dumps(rec))
    assert bench.profiled_traffic("w", "paged_prefill") is None
    assert bench.profiled_traffic("absent", "paged_prefill") is None


def test_profiled_traffic_follows_the_partition_size(tmp_path, monkeypatch):
    """A partitioned launch's figure is reported only at the partition size
    it was captured with."""
    import json
    import bench
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"source_sha256_16": bench.source_hash("paged_decode_step"), "partition_tokens": 2048,
           "dram_bytes_per_launch": 99}
    (prof / "paged_decode_step_w.json").write_text(json.dumps(rec))
    assert bench.profiled_traffic("w", "paged_decode_step", 2048) == 99
    assert bench.profiled_traffic("w", "paged_decode_step", 1536) is None
    del rec["partition_tokens"]
    (prof / "paged_decode_step_w.json").write_text(json.dumps(rec))
    assert bench.profiled_traffic("w", "paged_decode_step", 2048) is None


def test_choose_partition_rule():
    """The partition size rule on a 152-SM part with six decode CTAs per SM
    (912 slots): many (sequence, KV head) pairs get 1024-token partitions,
    few pairs the smallest multiple of 512 giving at most 729 CTAs (4.8 per
    SM) with each context's last piece counted, short contexts 512."""
    from paged_kv_cache_226_gb300 import lib
    if __import__("torch").cuda.is_available():
        pytest.skip("the rule is checked here for the 152-SM default only")
    assert lib.choose_partition(64, 8, 2048) == 1024            # 512 pairs
    assert lib.choose_partition(256, 8, 4608) == 1024           # shared-prefix batch
    assert lib.choose_partition(32, 8, 4096) == 2048            # 1536: 768 CTAs; 2048: 512
    assert lib.choose_partition(8, 8, 50000) == 4608            # 64 x ceil(50000 / 4608) = 704
    assert lib.choose_partition(8, 8, 45056) == 4096            # 64 x 11 = 704; 3584: 64 x 13
    assert lib.choose_partition(1, 1, 10 ** 6) == 1536          # 652 pieces; 1024: 977
    assert lib.choose_partition(1, 1, 10 ** 7) == 13824         # 724 pieces; 13312: 752
    assert lib.choose_partition(4, 2, 250) == 512               # short contexts
    assert lib.choose_partition(64, 8, 2048, block_size=32) % 32 == 0


def test_choose_partition_counts_ragged_contexts():
    """With the context lengths given, the short contexts' single pieces are
    counted as such: one 49152-token context and seven of 1024 tokens, 8 KV
    heads, fit 729 CTAs at 1024 tokens (8 x (48 + 7) = 440), while taking
    every context at the maximum needs 4608 (8 x 8 x 11 = 704)."""
    import numpy as np
    import torch
    from paged_kv_cache_226_gb300 import lib
    if torch.cuda.is_available():
        pytest.skip("the rule is checked here for the 152-SM default only")
    lens = [49152] + [1024] * 7
    assert lib.choose_partition(8, 8, 49152) == 4608
    assert lib.choose_partition(8, 8, 49152, context_lens=lens) == 1024
    assert lib.choose_partition(8, 8, 49152, context_lens=np.asarray(lens, np.int32)) == 1024
    assert lib.choose_partition(8, 8, 49152, context_lens=torch.tensor(lens)) == 1024
    # empty contexts add no CTAs: 8 x 48 = 384 at 1024 tokens, 8 x 96 = 768 > 729 at 512
    assert lib.choose_partition(8, 8, 49152, context_lens=[0] * 7 + [49152]) == 1024
