"""ps_paged_attention_noalloc: the attention entry point for callers that cannot allocate.

Some callers are given only their input and output buffers and may not create device
memory (a plug-in whose host framework owns all device memory, a loop that must not
call cudaMalloc/cudaFree because they can synchronise the device). The no-allocation
entry point keeps its scratch in a fixed array inside the library. These tests call it
through the C ABI on two calls in a row and check each result against the CPU oracle
within the parity bound, and against the ordinary entry point (which takes a
caller-allocated workspace) within the same bound.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_18_gb300 import _lib, binding
from paged_kv_attention_18_gb300 import workloads as W
from tests.gpu_util import bound_check

pytestmark = pytest.mark.gpu

TOL = {"f16": 2e-3, "bf16": 1e-2}
DTYPE = {"f16": 0, "bf16": 1}


def _noalloc(lib, st, wl, q, kp, vp, bt, sl, qs, out):
    return lib.ps_paged_attention_noalloc(
        q.data_ptr(), kp.data_ptr(), vp.data_ptr(), bt.data_ptr(), bt.shape[1], sl.data_ptr(),
        qs.data_ptr(), st.B, st.T, wl.H_q, wl.H_kv, wl.D, wl.num_blocks,
        ctypes.c_float(wl.scale), out.data_ptr(), DTYPE[wl.dtype],
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _compare_one(lib, wl, rows=None):
    """One no-allocation call against the oracle (on `rows`, or every row) and against
    the workspace entry point."""
    st = wl.steps[0]
    dev = lambda a, dt=None: W.to_device(a, dt)  # noqa: E731
    q, kp, vp = dev(st.q, wl.dtype), dev(wl.k_pool, wl.dtype), dev(wl.v_pool, wl.dtype)
    bt, sl, qs = dev(st.block_tables), dev(st.seq_lens), dev(st.query_start_loc)
    out = torch.full_like(q, float("nan"))
    rc = _noalloc(lib, st, wl, q, kp, vp, bt, sl, qs, out)
    assert rc == 0, lib.ps_status_string(rc)
    torch.cuda.synchronize()
    assert binding.device_error() == 0  # no plan overflow, no bad index
    got = out.float().cpu().numpy()
    ref = oracle.paged_attention(st.q, wl.k_pool, wl.v_pool, st.block_tables, st.seq_lens,
                                 st.query_start_loc, wl.scale, wl.dtype, acc=np.float32,
                                 rows=rows)
    sel = slice(None) if rows is None else np.asarray(rows, dtype=np.int64)
    bound_check(got[sel], ref[sel], wl.dtype)
    ws_out = binding.paged_attention(q, kp, vp, bt, sl, qs, wl.scale).float().cpu().numpy()
    torch.cuda.synchronize()
    assert np.isfinite(got).all()
    assert np.abs(got - ws_out).max() <= TOL[wl.dtype]


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


def test_noalloc_batch_whose_split_room_does_not_fit():
    # 4096 one-token decodes: the work lists with room for splitting long contexts would
    # take about 65 MB, more than the fixed scratch, so the call lays out the unsplit lists
    # (under 1 MB). Half the sequences are long enough that the planner first splits them
    # in two, which overflows those lists; it must coarsen the splits until the plan fits,
    # and record no plan overflow.
    rng = np.random.default_rng(71)
    short = [(int(L), 1) for L in rng.integers(1, 17, size=2000)]
    long_ = [(int(L), 1) for L in rng.integers(600, 901, size=2096)]
    order = rng.permutation(len(short) + len(long_))
    seqs = [(short + long_)[i] for i in order]
    users = [i for i, (L, _) in enumerate(seqs) if L >= 600]
    wl = W.simple_workload("noalloc-wide", seed=71, dtype="f16", H_q=12, H_kv=2, D=64,
                           seqs=seqs, shared_prefix_blocks=37, prefix_users=users)
    lib = _lib.load()
    st = wl.steps[0]
    rows = sorted(rng.choice(st.T, size=300, replace=False).tolist())
    _compare_one(lib, wl, rows=rows)


def test_noalloc_rejects_a_batch_beyond_its_fixed_scratch():
    lib = _lib.load()
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = lib.ps_paged_attention_noalloc(fake, fake, fake, fake, 1, fake, fake, 1 << 20, 1 << 22,
                                        32, 1, 128, 64, ctypes.c_float(0.1), fake, 1, None)
    assert rc == -4  # PS_ERR_WORKSPACE
