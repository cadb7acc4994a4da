"""Host-side logic of bench.py: algorithmic work, replica seeds, and the max-over-ranks
reduction with two gloo ranks on CPU (no GPU)."""
import os
import socket

import numpy as np
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from paged_kv_attention_18_gb300 import workloads as W


def test_step_work_by_hand():
    wl = W.simple_workload("w", seed=0, dtype="bf16", H_q=4, H_kv=2, D=64,
                           seqs=[(20, 1), (5, 5), (9, 0)])
    w = bench.step_work(wl, wl.steps[0])
    # KV: contexts 20 and 5 (the n = 0 sequence reads nothing), 2 heads, 64 dims, K and V
    assert w["kv_bytes"] == (20 + 5) * 2 * 64 * 2 * 2
    # pairs: decode at position 19 sees 20 keys; prefill rows see 1..5 keys
    assert w["flops"] == 4 * 64 * 4 * (20 + 15)
    assert w["tokens"] == 6


def test_replica_seeds_differ():
    a = bench.make_workload("tiny_decode", 0)
    b = bench.make_workload("tiny_decode", 1)
    assert not np.array_equal(a.steps[0].q, b.steps[0].q)
    assert a.steps[0].q.shape == b.steps[0].q.shape


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        results[rank] = bench.reduce_max(1.5 * (rank + 1), world)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        assert dict(results) == {0: 3.0, 1: 3.0}


def test_subset_keeps_values_and_relabels_blocks():
    wl = W.simple_workload("s", seed=1, dtype="f16", H_q=4, H_kv=2, D=64,
                           seqs=[(40, 1), (17, 2), (70, 3)])
    st = wl.steps[0]
    sub, sst = W.subset(wl, st, [2, 0])
    assert sst.T == 4 and sst.B == 2
    assert sub.num_blocks == 5 + 3
    for i, b in enumerate([2, 0]):
        for j in range(-(-int(st.seq_lens[b]) // 16)):
            assert np.array_equal(sub.k_pool[sst.block_tables[i, j]], wl.k_pool[st.block_tables[b, j]])


def test_traffic_records_follow_code_not_comments():
    # a kernel's committed DRAM counters are keyed to its code: comments and blank lines
    # may change, any code change drops the record
    src = b"""// header
__global__ void k(int* p) {  // trailing note
  /* block
     comment */
  p[0] = 1;

}
"""
    commented = src.replace(b"// header", b"// a new header, longer").replace(b"\n\n}", b"\n}")
    edited = src.replace(b"p[0] = 1;", b"p[0] = 2;")
    assert bench.code_only(src) == bench.code_only(commented)
    assert bench.code_only(src) != bench.code_only(edited)
    assert b"//" not in bench.code_only(src) and b"/*" not in bench.code_only(src)
