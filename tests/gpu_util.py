"""Helpers for GPU parity tests: move seeded workloads to the device, run steps through
the C ABI, and compare with the CPU oracle."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from paged_kv_attention_18_gb300 import binding

TOL = {"f16": 2e-3, "bf16": 1e-2}  # max-abs error against the fp32 oracle
TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def dev(a: np.ndarray, dtype: str | None = None) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(TORCH_DT[dtype])
    else:
        t = torch.from_numpy(a)
    return t.cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


class DevicePools:
    def __init__(self, wl):
        self.wl = wl
        self.k = dev(wl.k_pool, wl.dtype)
        self.v = dev(wl.v_pool, wl.dtype)


def run_step(wl, st, pools: DevicePools, workspace=None, separate_calls=False):
    """Slot mapping, scatter and attention of one step on the GPU. Returns (out, slots)."""
    dt = wl.dtype
    q, k, v = dev(st.q, dt), dev(st.k, dt), dev(st.v, dt)
    bt, sl, qs = dev(st.block_tables), dev(st.seq_lens), dev(st.query_start_loc)
    if separate_calls:
        slots = binding.slot_mapping(bt, sl, qs, st.T, wl.num_blocks)
        binding.reshape_and_cache(k, v, slots, pools.k, pools.v)
        out = binding.paged_attention(q, pools.k, pools.v, bt, sl, qs, wl.scale,
                                      workspace=workspace)
    else:
        slots = torch.empty(st.T, dtype=torch.int32, device="cuda")
        out = binding.attention_step(q, k, v, pools.k, pools.v, bt, sl, qs, wl.scale,
                                     workspace=workspace, slot_buf=slots)
    torch.cuda.synchronize()
    return out, slots


def half_ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Half a unit in the last place of |x| in the output type (the output rounding)."""
    mant = {"f16": 10, "bf16": 7}[dtype]
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -14)))
    return 0.5 * 2.0 ** (e - mant)


def check_workload(wl, rows_for_step=None, check_pool=True, separate_calls=False,
                   workspace=None, output_rounding_slack=False):
    """Run every step of a workload on GPU and oracle; compare slots, pools and outputs.

    rows_for_step(step_index, step) -> list of packed rows to compare, or None for all.
    With output_rounding_slack the bound per element is the tolerance plus half an ulp of
    the reference value in the output type: an output of |o| >= 2 in bf16 is rounded by up
    to 2^-8, so for the short or sharply peaked contexts some tests build, the rounding of
    the result alone can approach the plain bound. Returns the largest max-abs error seen.
    """
    pools = DevicePools(wl)
    kref, vref = wl.k_pool, wl.v_pool
    worst = 0.0
    for si, st in enumerate(wl.steps):
        out, slots = run_step(wl, st, pools, workspace=workspace, separate_calls=separate_calls)
        assert binding.device_error() == 0
        slots_ref = oracle.slot_mapping(st.block_tables, st.seq_lens, st.query_start_loc)
        np.testing.assert_array_equal(slots.cpu().numpy(), slots_ref)
        kref, vref = oracle.reshape_and_cache(st.k, st.v, slots_ref, kref, vref)
        if check_pool:
            assert np.array_equal(host_bits(pools.k), kref), "K pool differs after scatter"
            assert np.array_equal(host_bits(pools.v), vref), "V pool differs after scatter"
        rows = None if rows_for_step is None else rows_for_step(si, st)
        ref = oracle.paged_attention(st.q, kref, vref, st.block_tables, st.seq_lens,
                                     st.query_start_loc, wl.scale, wl.dtype, acc=np.float32,
                                     rows=rows)
        got = out.float().cpu().numpy()
        sel = slice(None) if rows is None else np.asarray(rows, dtype=np.int64)
        err = np.abs(got[sel] - ref[sel])
        assert np.isfinite(got[sel]).all()
        if output_rounding_slack:
            err = err - half_ulp(ref[sel], wl.dtype)
        e = float(err.max()) if err.size else 0.0
        report = os.environ.get("PS_PARITY_REPORT")
        if report:
            with open(report, "a") as f:
                f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "?"),
                                    "workload": wl.name, "dtype": wl.dtype, "step": si,
                                    "max_abs_err": e, "tol": TOL[wl.dtype],
                                    "rows": int(got[sel].shape[0])}) + "\n")
        assert e <= TOL[wl.dtype], f"step {si}: max-abs error {e} > {TOL[wl.dtype]}"
        worst = max(worst, e)
    return worst
