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


# Magnitudes from which rounding the exact result to the output type can by itself use up
# most of the bound: a bf16 output in [4, 8) is rounded by up to 2^-6 (above 1e-2), an f16
# output in [2, 4) by up to 2^-10 (half of 2e-3). Only elements at or above these get half
# an output ulp added to the bound; every other element must meet the bound as it is.
SLACK_FROM = {"f16": 2.0, "bf16": 4.0}


def bound_stats(got: np.ndarray, ref: np.ndarray, dtype: str) -> dict:
    """Max-abs error of the output against the fp32 oracle, split by the rule above: the
    raw max over all elements, the max over elements with |ref| below SLACK_FROM (bound:
    TOL), and the largest excess over half an output ulp on the others (bound: TOL)."""
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    big = np.abs(ref) >= SLACK_FROM[dtype]
    return {"raw": float(err.max()) if err.size else 0.0,
            "plain": float(err[~big].max()) if (~big).any() else 0.0,
            "rounded_excess": (float((err[big] - half_ulp(ref[big], dtype)).max())
                               if big.any() else 0.0),
            "n_big": int(big.sum()), "finite": bool(np.isfinite(got).all())}


def assert_bound(stats: dict, dtype: str, where: str = "") -> None:
    tol = TOL[dtype]
    assert stats["finite"], f"{where}non-finite output"
    assert stats["plain"] <= tol, \
        f"{where}max-abs error {stats['plain']} > {tol} on outputs below {SLACK_FROM[dtype]}"
    assert stats["rounded_excess"] <= tol, \
        (f"{where}error beyond half an output ulp {stats['rounded_excess']} > {tol} on "
         f"outputs of |o| >= {SLACK_FROM[dtype]}")


def bound_check(got: np.ndarray, ref: np.ndarray, dtype: str) -> dict:
    """bound_stats, asserted."""
    stats = bound_stats(got, ref, dtype)
    assert_bound(stats, dtype)
    return stats


def check_workload(wl, rows_for_step=None, check_pool=True, separate_calls=False,
                   workspace=None):
    """Run every step of a workload on GPU and oracle; compare slots, pools and outputs.

    rows_for_step(step_index, step) -> list of packed rows to compare, or None for all.
    Outputs are checked with bound_check. Returns the largest raw max-abs error seen.
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
        res = bound_stats(got[sel], ref[sel], wl.dtype)
        report = os.environ.get("PS_PARITY_REPORT")
        if report:
            with open(report, "a") as f:
                f.write(json.dumps({"test": os.environ.get("PYTEST_CURRENT_TEST", "?"),
                                    "workload": wl.name, "dtype": wl.dtype, "step": si,
                                    "max_abs_err": res["raw"], "plain": res["plain"],
                                    "rounded_excess": res["rounded_excess"],
                                    "n_big": res["n_big"], "tol": TOL[wl.dtype],
                                    "rows": int(got[sel].shape[0])}) + "\n")
        assert_bound(res, wl.dtype, f"step {si}: ")
        worst = max(worst, res["raw"])
    return worst
