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


@pytest.mark.parametrize("name", ["qwen05b_mixed", "tiny_decode"])
def test_step_replayed_from_cuda_graph(name):
    wl = W.named(name)
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
