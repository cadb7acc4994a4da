"""The attention step captured in a CUDA graph and replayed.

The planner runs on the device, so a step needs no host synchronisation: capturing the
five launches (with their programmatic dependent launch edges) in a graph and replaying
it must give the eager result, and a replay after new inputs are written in place must
match the oracle on those inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_18_gb300 import binding
from paged_kv_attention_18_gb300 import workloads as W
from tests.gpu_util import TOL, DevicePools, dev, host_bits

pytestmark = pytest.mark.gpu


def _graph_workload(name):
    if name == "planned_both":
        # 39 sequences with contexts past 64 pages: the planned chain with both attention
        # kernels (the tile kernel reading the plan without a wait of its own)
        seqs = [(800 + 37 * i, 1) for i in range(37)] + [(1500, 200), (600, 150)]
        return W.simple_workload("planned_both", seed=91, dtype="bf16", H_q=12, H_kv=2,
                                 D=128, seqs=seqs)
    return W.named(name)


@pytest.mark.parametrize("name", ["qwen05b_mixed", "tiny_decode", "planned_both"])
def test_step_replayed_from_cuda_graph(name):
    wl = _graph_workload(name)
    st = wl.steps[0]
    pools = DevicePools(wl)
    dt = wl.dtype
    q, k, v = dev(st.q, dt), dev(st.k, dt), dev(st.v, dt)
    bt, sl, qs = dev(st.block_tables), dev(st.seq_lens), dev(st.query_start_loc)
    out = torch.empty_like(q)
    slots = torch.empty(st.T, dtype=torch.int32, device="cuda")
    ws = binding.alloc_workspace(st.T, st.B, wl.H_q, wl.H_kv, wl.D,
                                 int(st.block_tables.shape[1]) * 16)

    def step():
        binding.attention_step(q, k, v, pools.k, pools.v, bt, sl, qs, wl.scale, out=out,
                               workspace=ws, slot_buf=slots)

    step()  # eager (also sets up the library's per-device state)
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    assert torch.equal(out, eager)

    # new query and new-token K/V values in place, same batch layout: the replay must
    # follow them (pool rows at the same slots are overwritten)
    rng = np.random.default_rng(77)
    q2 = W.round_to_bits(rng.standard_normal(st.q.shape, dtype=np.float32), dt)
    k2 = W.round_to_bits(rng.standard_normal(st.k.shape, dtype=np.float32), dt)
    v2 = W.round_to_bits(rng.standard_normal(st.v.shape, dtype=np.float32), dt)
    q.copy_(dev(q2, dt))
    k.copy_(dev(k2, dt))
    v.copy_(dev(v2, dt))
    g.replay()
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    slots_ref = oracle.slot_mapping(st.block_tables, st.seq_lens, st.query_start_loc)
    np.testing.assert_array_equal(slots.cpu().numpy(), slots_ref)
    kref, vref = oracle.reshape_and_cache(st.k, st.v, slots_ref, wl.k_pool, wl.v_pool)
    kref, vref = oracle.reshape_and_cache(k2, v2, slots_ref, kref, vref)
    assert np.array_equal(host_bits(pools.k), kref)
    assert np.array_equal(host_bits(pools.v), vref)
    ref = oracle.paged_attention(q2, kref, vref, st.block_tables, st.seq_lens,
                                 st.query_start_loc, wl.scale, dt, acc=np.float32)
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err <= TOL[dt], err


def test_host_step_graph_follows_host_buffers():
    # ps_attention_step_host recorded in a graph: every launch copies the host buffers'
    # current contents in and the output out, so new tokens written into the same pinned
    # tensors between launches must show up in the pools and the output
    wl = W.named("qwen05b_mixed")
    st = wl.steps[0]
    pools = DevicePools(wl)
    dt = wl.dtype
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dt]

    def pin(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else a)
        return (t.view(dtype) if dtype is not None else t).pin_memory()

    q, k, v = pin(st.q, tdt), pin(st.k, tdt), pin(st.v, tdt)
    bt, sl, qs = pin(st.block_tables), pin(st.seq_lens), pin(st.query_start_loc)
    out = torch.empty(q.shape, dtype=tdt).pin_memory()
    n = binding.staging_size(st.T, st.B, st.max_blocks_per_seq, wl.H_q, wl.H_kv, wl.D,
                             int(st.seq_lens.max()))
    staging = torch.empty(n, dtype=torch.uint8, device="cuda")
    g = binding.HostStepGraph(q, k, v, bt, sl, qs, out, pools.k, pools.v, wl.scale, staging)
    try:
        assert np.array_equal(host_bits(pools.k), wl.k_pool)  # creation runs nothing
        slots_ref = oracle.slot_mapping(st.block_tables, st.seq_lens, st.query_start_loc)
        kref, vref = wl.k_pool, wl.v_pool
        rng = np.random.default_rng(78)
        for launch in range(2):
            if launch:
                for t, a in ((q, st.q), (k, st.k), (v, st.v)):
                    new = W.round_to_bits(rng.standard_normal(a.shape, dtype=np.float32), dt)
                    t.copy_(torch.from_numpy(new.view(np.int16)).view(tdt))
            qh, kh, vh = (t.view(torch.int16).numpy().view(np.uint16).copy() for t in (q, k, v))
            g.launch()
            torch.cuda.synchronize()
            assert binding.device_error() == 0
            kref, vref = oracle.reshape_and_cache(kh, vh, slots_ref, kref, vref)
            assert np.array_equal(host_bits(pools.k), kref)
            assert np.array_equal(host_bits(pools.v), vref)
            ref = oracle.paged_attention(qh, kref, vref, st.block_tables, st.seq_lens,
                                         st.query_start_loc, wl.scale, dt, acc=np.float32)
            err = np.abs(out.float().numpy() - ref).max()
            assert err <= TOL[dt], (launch, err)
    finally:
        g.close()


def _host_step_tensors(wl, st, pinned=True):
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]

    def host(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else a)
        t = (t.view(dtype) if dtype is not None else t).clone()
        return t.pin_memory() if pinned else t

    q, k, v = host(st.q, tdt), host(st.k, tdt), host(st.v, tdt)
    bt, sl, qs = host(st.block_tables), host(st.seq_lens), host(st.query_start_loc)
    out = torch.empty(q.shape, dtype=tdt)
    out = out.pin_memory() if pinned else out
    n = binding.staging_size(st.T, st.B, st.max_blocks_per_seq, wl.H_q, wl.H_kv, wl.D,
                             max(1, int(st.seq_lens.max())))
    return q, k, v, bt, sl, qs, out, torch.empty(n, dtype=torch.uint8, device="cuda")


def test_host_step_graph_empty_batch():
    # no query tokens: the recorded graph is empty and launching it does nothing
    wl = W.simple_workload("z", seed=4, dtype="f16", H_q=4, H_kv=2, D=64,
                           seqs=[(10, 0), (33, 0)])
    st = wl.steps[0]
    pools = DevicePools(wl)
    q, k, v, bt, sl, qs, out, staging = _host_step_tensors(wl, st)
    g = binding.HostStepGraph(q, k, v, bt, sl, qs, out, pools.k, pools.v, wl.scale, staging)
    g.launch()
    torch.cuda.synchronize()
    g.close()
    assert binding.device_error() == 0
    assert np.array_equal(host_bits(pools.k), wl.k_pool)


@pytest.mark.parametrize("name,batch", [("tiny_decode", None), ("qwen05b_mixed", None),
                                        ("qwen15b_decode", 64), ("prefix_chunked_prefill", None)])
def test_host_step_matches_device_step(name, batch):
    # Each path of the host step with page-locked buffers:
    #   - tiny decode: direct split mode, the query copy a gather kernel first;
    #   - mixed: the tile kernel's direct mode, likewise;
    #   - 64 decodes: the planner, with the query copy on its extra CTAs and the output
    #     written into the host buffer by the step's kernels;
    #   - chunked prefill: the planner, with a 25 MB output moved by a kernel after the step.
    # Each must be bit-identical to the device entry point's output on the same inputs, in
    # a fresh pool each, and leave the same pools.
    wl = W.named(name, batch=batch) if batch else W.named(name)
    st = wl.steps[0]
    dt = wl.dtype
    pools_d = DevicePools(wl)
    q, k, v = dev(st.q, dt), dev(st.k, dt), dev(st.v, dt)
    bt, sl, qs = dev(st.block_tables), dev(st.seq_lens), dev(st.query_start_loc)
    ref = binding.attention_step(q, k, v, pools_d.k, pools_d.v, bt, sl, qs, wl.scale)
    pools_h = DevicePools(wl)
    args = _host_step_tensors(wl, st, pinned=True)
    binding.attention_step_host(*args[:7], pools_h.k, pools_h.v, wl.scale, args[7])
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    assert torch.equal(args[6].view(torch.int16), ref.cpu().view(torch.int16))
    assert torch.equal(pools_h.k, pools_d.k) and torch.equal(pools_h.v, pools_d.v)


def test_host_step_graph_rejects_pageable_buffers():
    # the graph copies from and to page-locked host memory only: pageable buffers are
    # rejected before anything is recorded, and a graph over pinned buffers still works
    wl = W.named("tiny_decode")
    st = wl.steps[0]
    pools = DevicePools(wl)
    args = _host_step_tensors(wl, st, pinned=False)
    with pytest.raises(binding.PagedServeError):
        binding.HostStepGraph(*args[:7], pools.k, pools.v, wl.scale, args[7])
    assert np.array_equal(host_bits(pools.k), wl.k_pool)
    args = _host_step_tensors(wl, st, pinned=True)
    g = binding.HostStepGraph(*args[:7], pools.k, pools.v, wl.scale, args[7])
    g.launch()
    torch.cuda.synchronize()
    g.close()
    assert binding.device_error() == 0
    out = args[6]
    slots_ref = oracle.slot_mapping(st.block_tables, st.seq_lens, st.query_start_loc)
    kref, vref = oracle.reshape_and_cache(st.k, st.v, slots_ref, wl.k_pool, wl.v_pool)
    ref = oracle.paged_attention(st.q, kref, vref, st.block_tables, st.seq_lens,
                                 st.query_start_loc, wl.scale, wl.dtype, acc=np.float32)
    assert np.abs(out.float().numpy() - ref).max() <= TOL[wl.dtype]


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("name", ["qwen05b_mixed", "qwen15b_decode"])
def test_host_step_pinned_and_pageable(name, pinned):
    # ps_attention_step_host: page-locked inputs are gathered by one kernel reading them
    # across the host link, pageable ones copied one by one; the pools and the output must
    # match the oracle either way
    wl = W.named(name, batch=16) if name == "qwen15b_decode" else W.named(name)
    st = wl.steps[0]
    pools = DevicePools(wl)
    q, k, v, bt, sl, qs, out, staging = _host_step_tensors(wl, st, pinned=pinned)
    binding.attention_step_host(q, k, v, bt, sl, qs, out, pools.k, pools.v, wl.scale, staging)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    slots_ref = oracle.slot_mapping(st.block_tables, st.seq_lens, st.query_start_loc)
    kref, vref = oracle.reshape_and_cache(st.k, st.v, slots_ref, wl.k_pool, wl.v_pool)
    assert np.array_equal(host_bits(pools.k), kref)
    assert np.array_equal(host_bits(pools.v), vref)
    ref = oracle.paged_attention(st.q, kref, vref, st.block_tables, st.seq_lens,
                                 st.query_start_loc, wl.scale, wl.dtype, acc=np.float32)
    assert np.abs(out.float().numpy() - ref).max() <= TOL[wl.dtype]
