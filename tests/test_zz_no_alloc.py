"""ps_paged_attention_noalloc: the attention entry point for callers that cannot allocate.

Some callers are given only their input and output buffers and may not create device
memory (a plug-in whose host framework owns all device memory, a loop that must not
call cudaMalloc/cudaFree because they can synchronise the device). The no-allocation
entry point keeps its scratch in a fixed array inside the library. These tests call it
through the C ABI on two calls in a row and check each result against the ordinary
entry point (which takes a caller-allocated workspace) within the parity tolerance.
"""
import ctypes

import numpy as np
import pytest
import torch

from paged_kv_attention_18_gb300 import _lib, binding
from paged_kv_attention_18_gb300 import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"f16": 2e-3, "bf16": 1e-2}
DTYPE = {"f16": 0, "bf16": 1}


def _noalloc(lib, st, wl, q, kp, vp, bt, sl, qs, out):
    return lib.ps_paged_attention_noalloc(
        q.data_ptr(), kp.data_ptr(), vp.data_ptr(), bt.data_ptr(), bt.shape[1], sl.data_ptr(),
        qs.data_ptr(), st.B, st.T, wl.H_q, wl.H_kv, wl.D, wl.num_blocks,
        ctypes.c_float(wl.scale), out.data_ptr(), DTYPE[wl.dtype],
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _compare_one(lib, wl):
    st = wl.steps[0]
    dev = lambda a, dt=None: W.to_device(a, dt)  # noqa: E731
    q, kp, vp = dev(st.q, wl.dtype), dev(wl.k_pool, wl.dtype), dev(wl.v_pool, wl.dtype)
    bt, sl, qs = dev(st.block_tables), dev(st.seq_lens), dev(st.query_start_loc)
    ref = binding.paged_attention(q, kp, vp, bt, sl, qs, wl.scale)  # caller workspace
    out = torch.full_like(q, float("nan"))
    rc = _noalloc(lib, st, wl, q, kp, vp, bt, sl, qs, out)
    assert rc == 0, lib.ps_status_string(rc)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    got, want = out.float().cpu().numpy(), ref.float().cpu().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - want).max() <= TOL[wl.dtype]


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    lib = _lib.load()
    # first call: decodes, verify rows and a prefill chunk; long contexts split
    first = W.simple_workload("noalloc-a", seed=21, dtype="bf16", H_q=12, H_kv=2, D=128,
                              seqs=[(3000, 1), (700, 5), (300, 64), (1, 1), (5000, 1)])
    # second call: a smaller batch of another shape, so stale scratch from the first
    # call is left in the array and must not leak into the result
    second = W.simple_workload("noalloc-b", seed=22, dtype="f16", H_q=14, H_kv=2, D=64,
                               seqs=[(90, 1), (512, 256), (33, 2)])
    _compare_one(lib, first)
    _compare_one(lib, second)


def test_noalloc_rejects_a_batch_beyond_its_fixed_scratch():
    lib = _lib.load()
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = lib.ps_paged_attention_noalloc(fake, fake, fake, fake, 1, fake, fake, 1 << 20, 1 << 22,
                                        32, 1, 128, 64, ctypes.c_float(0.1), fake, 1, None)
    assert rc == -4  # PS_ERR_WORKSPACE
