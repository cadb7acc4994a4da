#!/usr/bin/env python
"""Benchmark of one paged-KV attention step on GB300.

A step is the whole hot path over one packed batch: slot mapping, KV scatter and
paged attention (planner, split kernel, tile kernel, split combine), through the C ABI.

With no --workload, the run covers the five workloads the attention step is specified
on, each timed on its own:

    tiny_decode            4 decodes, 4/2 heads, D 64, f16
    qwen05b_mixed          8 decodes + 2 prefill chunks of 256, 14/2 heads, D 64, f16
    qwen15b_decode         256 decodes, contexts U[512, 4096], 12/2 heads, D 128, bf16
    prefix_chunked_prefill 64 prompts sharing a cached 1024-token prefix, chunked under an
                           8192-token budget with 32 decodes (4 engine steps), bf16
    spec_verify_long       132 sequences x 5 verify tokens, contexts up to 32768, bf16

``value`` is the decode workload's (qwen15b_decode) algorithmic HBM bytes / device time
(GB/s, whole job). ``workloads`` holds, for every workload, its GB/s, TFLOP/s and
tokens/s, the roofline of its dominant kernel and the CPU oracle's rate on the host
cores. The line also carries the end-to-end decode figure through the host-buffer entry
point and the SM clocks seen during the timed regions.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]
    python -m torch.distributed.run --nproc-per-node N bench.py --gpus N ...  (replicas)
"""
from __future__ import annotations

import os
import re

# the CPU oracle runs single-threaded (reported as cores = 1)
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import tempfile  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_attention_18_gb300 import workloads as W  # noqa: E402

METRIC = "decode paged-attn HBM GB/s (% of peak); mixed-batch attention tokens/s"
L2_BYTES = 129_000_000
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# committed ncu DRAM counters of the dominant kernels, with the sources they were taken on
TRAFFIC_FILES = {
    ("split_attention", "qwen15b_decode"): "split_attention_qwen15b_decode_traffic.json",
    ("split_attention", "spec_verify_long"): "split_attention_spec_verify_long_traffic.json",
    ("tile_attention", "prefix_chunked_prefill"): "tile_attention_prefix_chunked_prefill_traffic.json",
    ("tile_attention", "long_prefill"): "tile_attention_long_prefill_traffic.json",
}
# the source text each kernel is built from: a whole file, or (file, first line, line that
# ends the region) for a kernel that shares its file with others
KERNEL_SOURCES = {
    "split_attention": [("paged_kv_attention_18_gb300/csrc/ps_attention.cu",
                         "// split kernel: one warp = one work item at a time",
                         "// combine: one warp per (token, head) whose rows were split"),
                        "paged_kv_attention_18_gb300/csrc/ps_common.cuh"],
    "tile_attention": ["paged_kv_attention_18_gb300/csrc/ps_tile.cu",
                       "paged_kv_attention_18_gb300/csrc/ps_tc05.cuh",
                       "paged_kv_attention_18_gb300/csrc/ps_common.cuh"],
}


# ------------------------------------------------------------------------------------
# algorithmic work of a step
# ------------------------------------------------------------------------------------
def step_work(wl: W.Workload, st: W.Step) -> dict:
    """Algorithmic bytes and flops of one step (each context read once, no split partials).

    Also split by the kernel that serves each sequence: sequences with more than 64
    packed rows (n * G, four 16-row groups) go to the tile kernel, the others (decodes,
    verify rows) to the split kernel."""
    es = 2  # bytes per 16-bit element
    L = st.seq_lens.astype(np.int64)
    n = np.diff(st.query_start_loc).astype(np.int64)
    G = wl.H_q // wl.H_kv
    tile = (n * G > 64) & (G <= 16)
    live = n > 0
    kv_b = L * wl.H_kv * wl.D * es * 2
    qo_b = 2 * n * wl.H_q * wl.D * es
    bt_b = ((L + 15) // 16) * 4
    attn_b = np.where(live, kv_b + qo_b + bt_b, 0)
    pairs = np.zeros(st.B, dtype=np.int64)
    for b in range(st.B):
        if n[b]:
            p = L[b] - n[b] + np.arange(n[b])
            pairs[b] = int((p + 1).sum())  # row at position p sees p + 1 keys
    flops_b = 4 * wl.D * wl.H_q * pairs
    scatter = 2 * (st.T * wl.H_kv * wl.D * es * 2) + st.T * 4  # read k/v, write pool rows, slots
    return {"attn_bytes": int(attn_b.sum()), "kv_bytes": int(np.where(live, kv_b, 0).sum()),
            "step_bytes": int(attn_b.sum()) + scatter, "flops": int(flops_b.sum()),
            "tokens": st.T,
            "split_bytes": int(attn_b[~tile].sum()), "split_kv_bytes": int(np.where(live & ~tile, kv_b, 0).sum()),
            "tile_bytes": int(attn_b[tile].sum()), "tile_flops": int(flops_b[tile].sum())}


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_only(text: bytes) -> bytes:
    """Source text without comments and blank lines: editing a comment leaves the kernel,
    and so its committed counters, as they were."""
    text = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)
    text = re.sub(rb"//[^\n]*", b"", text)
    return b"\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for src in KERNEL_SOURCES[kernel]:
        rel, first, end = (src, None, None) if isinstance(src, str) else src
        with open(os.path.join(ROOT, rel), "rb") as f:
            text = f.read()
        if first is not None:
            a = text.index(first.encode())
            text = text[a:text.index(end.encode(), a)]
        h.update(code_only(text))
    return h.hexdigest()


def committed_traffic(kernel: str, workload: str, units: float) -> float | None:
    """DRAM bytes per launch of `kernel` from its committed ncu capture on `workload`,
    scaled to this launch by the units the record names (KV bytes for the split kernel,
    tile flops for the tile kernel), or None when there is no capture for the pair or the
    kernel's sources changed since it was taken."""
    name = TRAFFIC_FILES.get((kernel, workload))
    path = os.path.join(ROOT, "profiles", name) if name else None
    if not path or not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_sha256") != kernel_source_hash(kernel):
        return None
    return rec["dram_bytes_per_launch"] * units / rec["units_per_launch"]


# ------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.index)], stdout=self.file,
                stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        rows = [ln.split(",") for ln in self.file.read().splitlines() if ln.strip()]
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for nm, val in zip(names, r[5:9]):
                    if val.strip() == "Active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------------------------
# distributed plumbing (replicas: no collective on the data path)
# ------------------------------------------------------------------------------------
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity on one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------------------------
# CPU oracle timing (baseline and reference arm)
# ------------------------------------------------------------------------------------
def cpu_info() -> dict:
    """The host CPU: core count, model name (or, on Arm, implementer and part) and the
    BLAS threads each oracle process uses."""
    model = None
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k, v = k.strip(), v.strip()
                if k.lower() == "model name" and not model:
                    model = v
                elif k in ("CPU implementer", "CPU part") and k not in fields:
                    fields[k] = v
    except OSError:
        pass
    if not model:
        import platform
        model = platform.machine() + (" (" + ", ".join(f"{k} {v}" for k, v in fields.items())
                                      + ")" if fields else "")
    return {"cpu_count": os.cpu_count() or 1, "model": model,
            "blas_threads_per_process": int(os.environ.get("OPENBLAS_NUM_THREADS", "1"))}


def oracle_seconds(wl: W.Workload, st: W.Step, seqs: list[int]) -> tuple[float, int, int]:
    """Time the oracle (slot mapping, scatter, attention) on a subset of sequences.

    The subset keeps only the pool blocks its sequences use, so the oracle's copy of the
    pool in its scatter scales with the sample. Returns (seconds, algorithmic bytes,
    tokens)."""
    import oracle
    sub, sst = W.subset(wl, st, seqs)
    t0 = time.perf_counter()
    oracle.attention_step(sst, sub.k_pool, sub.v_pool, sub.scale, sub.dtype, acc=np.float32)
    dt = time.perf_counter() - t0
    return dt, step_work(sub, sst)["step_bytes"], sst.T


_SAMPLE_ARRAYS = ("k_pool", "v_pool", "q", "k", "v", "block_tables", "seq_lens",
                  "query_start_loc", "seq_ids")


def save_sample(wl: W.Workload, st: W.Step, seqs: list[int], path: str) -> None:
    """The sample's sequences of one step, with only the pool blocks they use, written as
    .npy files under `path` for the oracle worker processes to map read-only."""
    sub, sst = W.subset(wl, st, seqs)
    os.makedirs(path, exist_ok=True)
    for name in _SAMPLE_ARRAYS:
        np.save(os.path.join(path, name + ".npy"), getattr(sub if "pool" in name else sst, name))
    with open(os.path.join(path, "meta.json"), "w") as f:
        json.dump({"name": sub.name, "dtype": sub.dtype, "H_q": sub.H_q, "H_kv": sub.H_kv,
                   "D": sub.D, "num_blocks": sub.num_blocks}, f)


_SAMPLES: dict = {}


def _oracle_chunk(task) -> tuple[int, int]:
    """Worker process: run the oracle on sequences `seqs` of the sample stored at `path`
    (with no sequences, only map the sample and wait `pause` seconds, so that a round of
    such tasks reaches every worker). Returns (algorithmic bytes, tokens) of the chunk."""
    path, seqs, pause = task
    if not path:
        return 0, 0
    if path not in _SAMPLES:
        with open(os.path.join(path, "meta.json")) as f:
            m = json.load(f)
        a = {n: np.load(os.path.join(path, n + ".npy"), mmap_mode="r") for n in _SAMPLE_ARRAYS}
        wl = W.Workload(name=m["name"], dtype=m["dtype"], H_q=m["H_q"], H_kv=m["H_kv"], D=m["D"],
                        num_blocks=m["num_blocks"], k_pool=a["k_pool"], v_pool=a["v_pool"])
        st = W.Step(q=a["q"], k=a["k"], v=a["v"], block_tables=np.array(a["block_tables"]),
                    seq_lens=np.array(a["seq_lens"]),
                    query_start_loc=np.array(a["query_start_loc"]), seq_ids=np.array(a["seq_ids"]))
        _SAMPLES.clear()
        _SAMPLES[path] = (wl, st)
    if not seqs:
        time.sleep(pause)
        return 0, 0
    wl, st = _SAMPLES[path]
    _, nb, nt = oracle_seconds(wl, st, list(seqs))
    return nb, nt


class OraclePool:
    """One oracle process per host core (spawned, so no process is forked from one that
    has used the GPU), each with single-threaded BLAS."""

    def __init__(self, n: int | None = None):
        import multiprocessing as mp
        from concurrent.futures import ProcessPoolExecutor
        self.n = n or (os.cpu_count() or 1)
        self.ex = ProcessPoolExecutor(self.n, mp_context=mp.get_context("spawn"))
        list(self.ex.map(_oracle_chunk, [("", [], 0.0)] * self.n))  # start every worker

    def prepare(self, path: str) -> None:
        """Every worker maps the sample (untimed): each of 2n pausing tasks holds its
        worker, so the round reaches all of them."""
        list(self.ex.map(_oracle_chunk, [(path, [], 0.3)] * (2 * self.n)))

    def run(self, path: str, chunks: list[list[int]]) -> tuple[float, int, int]:
        """Wall seconds, bytes and tokens of the oracle over `chunks` in parallel (after
        prepare(path))."""
        t0 = time.perf_counter()
        res = list(self.ex.map(_oracle_chunk, [(path, c, 0.0) for c in chunks]))
        return time.perf_counter() - t0, sum(r[0] for r in res), sum(r[1] for r in res)

    def close(self):
        self.ex.shutdown()


def _rate(nbytes: int, tokens: int, sec: float, unit: str) -> float:
    return nbytes / sec / 1e9 if unit == "GB/s" else tokens / sec


def sample_sequences(wl: W.Workload, st: W.Step, budget_s: float, seed: int = 0) -> list[int]:
    """A seeded random order of step 0's sequences, cut to about budget_s of single-core
    oracle time (measured on a probe of the first few)."""
    order = [int(b) for b in np.random.default_rng(seed).permutation(st.B)]
    probe = order[:min(4, st.B)]
    dt, _, _ = oracle_seconds(wl, st, probe)
    per_seq = max(dt / max(1, len(probe)), 1e-5)
    n = int(max(1, min(st.B, budget_s / per_seq)))
    return sorted(order[:n])


def cpu_baseline(wl: W.Workload, unit: str, pool: OraclePool | None, budget_s: float = 3.0,
                 tmpdir: str | None = None) -> dict:
    """The oracle's rate on the same workload (its first engine step): on one core over a
    sample of about budget_s, and on every core (one process per core) over a sample
    about cores times larger, split by sequence. Rates are algorithmic bytes (or tokens)
    of the sample / time, in the workload's unit."""
    st = wl.steps[0]
    info = cpu_info()
    min_s = min(1.0, budget_s)  # a sample that runs shorter is repeated up to this time
    one = sample_sequences(wl, st, budget_s)
    dt1, nb1, nt1, reps = 0.0, 0, 0, 0
    while dt1 < min_s:
        dt, nb, nt = oracle_seconds(wl, st, one)
        dt1, nb1, nt1, reps = dt1 + dt, nb1 + nb, nt1 + nt, reps + 1
    single = {"value": _rate(nb1, nt1, dt1, unit), "unit": unit, "cores": 1, "kind": "oracle",
              "sample": f"{len(one)} of {st.B} sequences of engine step 0 "
                        f"({nt1 // reps} tokens) x {reps}, {dt1:.1f} s on one core"}
    if pool is None:
        single["cpu"] = info
        return single
    # every core: a sample of about cores x budget_s of single-core time (capped at the
    # whole step), split into chunks of about equal oracle work
    seqs = sample_sequences(wl, st, budget_s * pool.n, seed=1)
    n_b = np.diff(st.query_start_loc).astype(np.int64)
    cost = {b: int(st.seq_lens[b]) * max(1, int(n_b[b])) for b in seqs}  # oracle work ~ L * n
    chunks: list[list[int]] = [[] for _ in range(pool.n)]
    loads = [0] * pool.n
    for b in sorted(seqs, key=lambda x: -cost[x]):
        i = loads.index(min(loads))
        chunks[i].append(b)
        loads[i] += cost[b]
    path = tempfile.mkdtemp(prefix="oracle_sample_", dir=tmpdir)
    try:
        save_sample(wl, st, seqs, path)
        # sequence ids inside the saved sample are its positions
        pos = {b: i for i, b in enumerate(seqs)}
        chunks = [[pos[b] for b in c] for c in chunks if c]
        pool.prepare(path)
        dta, nba, nta, reps = 0.0, 0, 0, 0
        while dta < min_s:
            dt, nb, nt = pool.run(path, chunks)
            dta, nba, nta, reps = dta + dt, nba + nb, nta + nt, reps + 1
    finally:
        import shutil
        shutil.rmtree(path, ignore_errors=True)
    return {"value": _rate(nba, nta, dta, unit), "unit": unit, "cores": len(chunks),
            "kind": "oracle",
            "sample": f"{len(seqs)} of {st.B} sequences of engine step 0 ({nta // reps} "
                      f"tokens) x {reps}, split over {len(chunks)} single-threaded oracle "
                      f"processes (of {pool.n} host cores), {dta:.1f} s wall",
            "single_core": single, "cpu": info}


# ------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------
def make_workload(name: str, rank: int, batch: int | None = None) -> W.Workload:
    """The named workload; each replica rank draws its own batch (seed + 1000 * rank)."""
    base = {"qwen15b_decode": 2, "tiny_decode": 0, "qwen05b_mixed": 1,
            "prefix_chunked_prefill": 3, "spec_verify_long": 4, "long_prefill": 5}[name]
    kw = {"batch": batch} if (batch and name == "qwen15b_decode") else {}
    return W.named(name, seed=base + 1000 * rank, **kw)


class DeviceWorkload:
    """A workload's tensors resident on the GPU, ready to run steps."""

    def __init__(self, wl: W.Workload, device):
        import torch
        dev = lambda a, dt=None: W.to_device(a, dt, device)  # noqa: E731
        self.wl = wl
        self.k_pool = dev(wl.k_pool, wl.dtype)
        self.v_pool = dev(wl.v_pool, wl.dtype)
        self.steps = []
        max_len = max(int(st.seq_lens.max()) if st.B else 0 for st in wl.steps)
        from paged_kv_attention_18_gb300 import binding
        for st in wl.steps:
            d = {"q": dev(st.q, wl.dtype), "k": dev(st.k, wl.dtype), "v": dev(st.v, wl.dtype),
                 "bt": dev(st.block_tables), "sl": dev(st.seq_lens),
                 "qsl": dev(st.query_start_loc)}
            d["out"] = torch.empty_like(d["q"])
            d["slots"] = torch.empty(st.T, dtype=torch.int32, device=device)
            d["ws"] = binding.alloc_workspace(st.T, st.B, wl.H_q, wl.H_kv, wl.D, max_len,
                                              device=device)
            self.steps.append(d)

        # a pool smaller than twice the L2 would stay resident between steps: such a
        # workload writes a buffer larger than L2 before each step, outside the timing
        pool_bytes = 2 * wl.k_pool.nbytes
        self.flush_buf = (torch.empty(4 * L2_BYTES, dtype=torch.uint8, device=device)
                          if pool_bytes < 2 * L2_BYTES else None)
        self.graphs = None  # set by capture()

    def flush_l2(self):
        if self.flush_buf is not None:
            self.flush_buf.fill_(1)

    def run_one(self, d, eager=False):
        from paged_kv_attention_18_gb300 import binding
        if self.graphs is not None and not eager:
            d["graph"].replay()
            return
        binding.attention_step(d["q"], d["k"], d["v"], self.k_pool, self.v_pool, d["bt"],
                               d["sl"], d["qsl"], self.wl.scale, out=d["out"],
                               workspace=d["ws"], slot_buf=d["slots"])

    def capture(self):
        """Capture each engine step in its own CUDA graph (after one eager run)."""
        import torch
        self.run_eager()
        torch.cuda.synchronize()
        for d in self.steps:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, capture_error_mode="thread_local"):
                self.run_one(d, eager=True)
            d["graph"] = g
        self.graphs = True
        torch.cuda.synchronize()

    def run_eager(self):
        for d in self.steps:
            self.flush_l2()
            self.run_one(d, eager=True)

    def run(self):
        for d in self.steps:
            self.flush_l2()
            self.run_one(d)


def time_device(dw: DeviceWorkload, steps: int, warmup: int, world: int, device):
    """Time `steps` steps with CUDA events (max over ranks), then time each kernel.

    The per-kernel times come from a second pass over the same steps with the library's
    timing hook (CUDA events around every launch). The hook is kept out of the first pass
    because an event between two launches would undo their programmatic dependent launch.
    Returns (ms for the timed steps, {kernel: (ms, launches)} per hook step, hook steps).
    """
    import torch
    from paged_kv_attention_18_gb300 import binding
    for _ in range(warmup):
        dw.run()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    if dw.flush_buf is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            dw.run()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
    else:
        # L2 written over before every engine step; only the steps are timed
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps * len(dw.steps))]
        i = 0
        for _ in range(steps):
            for d in dw.steps:
                dw.flush_l2()
                ev[i][0].record(stream)
                dw.run_one(d)
                ev[i][1].record(stream)
                i += 1
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in ev)
    barrier(world)
    hook_steps = min(steps, 200)
    binding.profile_begin(hook_steps * len(dw.steps))
    for _ in range(hook_steps):
        dw.run_eager()  # the timing hook sees eager launches only
    torch.cuda.synchronize()
    prof = binding.profile_end()
    return reduce_max(ms, world, device), prof, hook_steps


def time_e2e(dw: DeviceWorkload, steps: int, warmup: int, world: int, device,
             eager: bool = False):
    """Same steps from pinned host buffers: each engine step replays its
    ps_attention_step_host graph (copies in, the step, copy out), or with ``eager`` calls
    ps_attention_step_host itself; the stream is synchronised after every engine step."""
    import torch
    from paged_kv_attention_18_gb300 import binding
    wl = dw.wl
    hosts, h2d, d2h = [], 0, 0
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]
    max_len = max(int(st.seq_lens.max()) if st.B else 0 for st in wl.steps)
    for st in wl.steps:
        def pin(a, dtype=None):
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else a)
            t = t.view(dtype) if dtype is not None else t
            return t.pin_memory()
        h = {"q": pin(st.q, dt), "k": pin(st.k, dt), "v": pin(st.v, dt),
             "bt": pin(st.block_tables), "sl": pin(st.seq_lens), "qsl": pin(st.query_start_loc)}
        h["out"] = torch.empty(h["q"].shape, dtype=dt).pin_memory()
        n = binding.staging_size(st.T, st.B, st.max_blocks_per_seq, wl.H_q, wl.H_kv, wl.D,
                                 max_len)
        h["staging"] = torch.empty(n, dtype=torch.uint8, device=device)
        h2d += sum(h[k].numel() * h[k].element_size() for k in ("q", "k", "v", "bt", "sl", "qsl"))
        d2h += h["out"].numel() * h["out"].element_size()
        if not eager:
            h["graph"] = binding.HostStepGraph(h["q"], h["k"], h["v"], h["bt"], h["sl"], h["qsl"],
                                               h["out"], dw.k_pool, dw.v_pool, wl.scale,
                                               h["staging"])
        hosts.append(h)
    stream = torch.cuda.current_stream()

    def one():
        for h in hosts:
            if eager:
                binding.attention_step_host(h["q"], h["k"], h["v"], h["bt"], h["sl"], h["qsl"],
                                            h["out"], dw.k_pool, dw.v_pool, wl.scale,
                                            h["staging"])
            else:
                h["graph"].launch()
            stream.synchronize()  # the caller reads the step's output

    for _ in range(warmup):
        one()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    sec = reduce_max(time.perf_counter() - t0, world, device)
    for h in hosts:
        if "graph" in h:
            h["graph"].close()
    return sec, h2d, d2h


def time_flushed(dw: DeviceWorkload, steps: int, world: int, device) -> float:
    """ms per step with the L2 written over before every engine step (outside the timed
    events), for a workload whose inputs are larger than L2 and so run unflushed in the main
    timing. Events around each engine step also stop the next step's planner from
    overlapping the previous step's last kernel."""
    import torch
    if dw.flush_buf is not None:
        raise ValueError("this workload is already timed with the L2 flushed")
    dw.flush_buf = torch.empty(4 * L2_BYTES, dtype=torch.uint8, device=device)
    try:
        stream = torch.cuda.current_stream()
        for _ in range(2):
            dw.run()
        torch.cuda.synchronize()
        barrier(world)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps * len(dw.steps))]
        i = 0
        for _ in range(steps):
            for d in dw.steps:
                dw.flush_l2()
                ev[i][0].record(stream)
                dw.run_one(d)
                ev[i][1].record(stream)
                i += 1
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in ev)
        return reduce_max(ms / 1e3, world, device) * 1e3 / steps
    finally:
        dw.flush_buf = None


# the five workloads the step is specified on; the decode one gives the headline value
ALL_WORKLOADS = ["tiny_decode", "qwen05b_mixed", "qwen15b_decode", "prefix_chunked_prefill",
                 "spec_verify_long"]
HEADLINE = "qwen15b_decode"
# each workload's own unit: HBM GB/s where every row is a decode or verify row (the
# split kernel streams the context), tokens/s where prefill chunks are mixed in
UNITS = {"tiny_decode": "GB/s", "qwen05b_mixed": "tokens/s", "qwen15b_decode": "GB/s",
         "prefix_chunked_prefill": "tokens/s", "spec_verify_long": "GB/s",
         "long_prefill": "tokens/s"}


def roofline_of(prof: dict, work: list[dict], name: str, peaks: dict, peaks_src: str,
                hook_steps: int) -> dict:
    """Roofline of the step's dominant attention kernel (split or tile, by summed time),
    from the library hook's per-launch CUDA-event times on the launching stream."""
    kernel_ms = {k: t for k, (t, n) in prof.items() if n > 0}
    nsteps = len(work)
    attn = {k: kernel_ms.get(k, 0.0) for k in ("split_attention", "tile_attention")}
    dom = max(attn, key=attn.get)
    dom_ms, dom_n = prof[dom]
    avg_s = dom_ms / 1e3 / max(1, dom_n)
    share = dom_ms / (sum(kernel_ms.values()) or 1)
    if dom == "tile_attention":
        flops_launch = sum(w["tile_flops"] for w in work) / nsteps
        peak = peaks["bf16_tflops"]
        achieved = flops_launch / avg_s / 1e12
        r = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
             "frac": achieved / peak,
             "traffic": committed_traffic("tile_attention", name, flops_launch),
             "kernel": "tile_attention_kernel (tcgen05)",
             "algorithmic_per_launch": {"flops": flops_launch},
             "peak_source": f"{peaks_src} bf16_tflops (burst: the kernel runs well under a "
                            "millisecond per launch; fp16 runs at the bf16 rate)"}
    else:
        bytes_launch = sum(w["split_bytes"] for w in work) / nsteps
        achieved = bytes_launch / avg_s / 1e9
        r = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
             "frac": achieved / peaks["hbm_gbs"],
             "traffic": committed_traffic("split_attention", name,
                                          sum(w["split_kv_bytes"] for w in work) / nsteps),
             "kernel": "split_attention_kernel",
             "algorithmic_per_launch": {"bytes": bytes_launch},
             "peak_source": f"{peaks_src} hbm_gbs"}
    r["kernel_share_of_step"] = share
    r["per_kernel_ms_per_step"] = {k: t / max(1, prof[k][1]) * nsteps for k, t in kernel_ms.items()}
    r["timing"] = (f"kernel times from a second pass of {hook_steps} steps with CUDA events "
                   "around every launch (library timing hook)")
    return r


def measure_workload(name: str, wl: W.Workload, args, world: int, device, peaks: dict,
                     peaks_src: str, keep: bool = False):
    """Device timing of one workload: the step rate, its GB/s, TFLOP/s and tokens/s, the
    L2-flushed companion for a workload larger than L2, and the dominant kernel's
    roofline. Returns (entry, the resident workload if `keep`)."""
    import torch
    from paged_kv_attention_18_gb300 import binding
    work = [step_work(wl, st) for st in wl.steps]
    step_bytes = sum(w["step_bytes"] for w in work)
    tokens = sum(w["tokens"] for w in work)
    flops = sum(w["flops"] for w in work)
    dw = DeviceWorkload(wl, device)
    if args.graph:
        dw.capture()
    ms, prof, hook_steps = time_device(dw, args.steps, args.warmup, world, device)
    if binding.device_error() != 0:
        raise RuntimeError(f"device error word set during the {name} benchmark")
    sec = ms / 1e3
    unit = UNITS[name]
    gbs = world * step_bytes * args.steps / sec / 1e9
    tok_s = world * tokens * args.steps / sec
    flushed = None
    if dw.flush_buf is None and not args.no_flushed:
        fsteps = max(3, min(args.steps, 100))
        fms = time_flushed(dw, fsteps, world, device)
        flushed = {"value": (world * step_bytes / (fms / 1e3) / 1e9 if unit == "GB/s"
                             else world * tokens / (fms / 1e3)),
                   "ms_per_step": fms, "steps": fsteps,
                   "note": "the same steps with the L2 written over (516 MB) before every "
                           "engine step, outside CUDA events around each step"}
    st0 = wl.steps[0]
    entry = {
        "workload": wl.name, "description": wl.description, "dtype": wl.dtype,
        "value": gbs if unit == "GB/s" else tok_s, "unit": unit,
        "ms_per_step": ms / args.steps, "steps": args.steps,
        "engine_steps_per_step": len(wl.steps),
        "gbs": gbs, "tflops": world * flops * args.steps / sec / 1e12, "tokens_per_s": tok_s,
        "B": [st.B for st in wl.steps] if len(wl.steps) > 1 else st0.B,
        "T_per_step": tokens, "H_q": wl.H_q, "H_kv": wl.H_kv, "head_dim": wl.D,
        "block_size": 16, "num_blocks": wl.num_blocks,
        "kv_bytes_per_step": sum(w["kv_bytes"] for w in work),
        "algorithmic_bytes_per_step": step_bytes, "flops_per_step": flops,
        "l2": (f"inputs larger than L2 ({2 * wl.k_pool.nbytes / 1e6:.0f} MB KV pool, "
               f"{sum(w['kv_bytes'] for w in work) / 1e6:.0f} MB of it read per step, vs "
               f"{L2_BYTES / 1e6:.0f} MB L2); no flush" if dw.flush_buf is None else
               f"L2 flushed before every engine step ({4 * L2_BYTES / 1e6:.0f} MB buffer "
               f"written, outside the timed events): the {2 * wl.k_pool.nbytes / 1e6:.0f} MB "
               "KV pool fits in L2"),
        "l2_flushed": flushed,
        "gpu_launches": int(sum(n for _, n in prof.values()) * args.steps // hook_steps),
        "roofline": roofline_of(prof, work, name, peaks, peaks_src, hook_steps),
    }
    if not keep:
        del dw
        torch.cuda.empty_cache()
        return entry, None
    return entry, dw


def run_ours(args, rank, world, local_rank) -> dict | None:
    import torch
    import __graft_entry__
    __graft_entry__.build()
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    peaks, peaks_src = load_peaks()
    names = [args.workload] if args.workload else list(ALL_WORKLOADS)
    head = args.workload or HEADLINE
    # the headline workload last, so that it stays resident for the end-to-end leg
    names = [n for n in names if n != head] + [head]
    wls = {n: make_workload(n, rank, args.batch) for n in names}
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 and not args.no_clocks \
        else None
    if clocks:
        clocks.start()
    t_load = time.perf_counter()
    entries, head_dw = {}, None
    for n in names:
        entries[n], dw = measure_workload(n, wls[n], args, world, device, peaks, peaks_src,
                                          keep=(n == head))
        if n == head:
            head_dw = dw
    # keep the same load running until the clock sampler has seen enough of it
    while clocks and time.perf_counter() - t_load < 1.5:
        head_dw.run()
        torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None

    hd = entries[head]
    e2e = None
    if not args.no_e2e:
        wl = wls[head]
        e2e_steps = max(3, min(args.steps, 200))
        e2e_s, h2d, d2h = time_e2e(head_dw, e2e_steps, 3, world, device, eager=args.e2e_eager)
        nbytes = hd["algorithmic_bytes_per_step"]
        e2e = {"value": (world * nbytes * e2e_steps / e2e_s / 1e9 if hd["unit"] == "GB/s"
                         else world * hd["T_per_step"] * e2e_steps / e2e_s),
               "unit": hd["unit"], "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps,
               "api": ("ps_attention_step_host (pinned host buffers, stream sync per step)"
                       if args.e2e_eager else
                       "ps_attention_step_host_graph_create once per engine step, then "
                       "ps_graph_launch each step: the inputs read from the pinned host "
                       "buffers (block tables, lengths and offsets by a gather kernel, the "
                       "queries by the planner's copy CTAs, the new K/V by the scatter), the "
                       "step, the output written into the pinned buffer by the step's "
                       "kernels; stream sync per step")}
        del wl
    del head_dw
    torch.cuda.empty_cache()

    if rank != 0:
        return None
    # the CPU oracle on the host cores, after all GPU work (its worker processes are
    # spawned, never forked from this process)
    if not args.no_cpu_baseline:
        pool = OraclePool() if (os.cpu_count() or 1) > 1 else None
        try:
            for n in names:
                entries[n]["cpu_baseline"] = cpu_baseline(wls[n], UNITS[n], pool)
        finally:
            if pool:
                pool.close()
    result = {
        "metric": METRIC, "value": hd["value"], "unit": hd["unit"], "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": hd["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": hd["dtype"],
        "data": "synthetic (seeded N(0,1) values, random block permutation)",
        "config": {"workload": hd["workload"], "description": hd["description"],
                   "B": hd["B"], "T": hd["T_per_step"], "H_q": hd["H_q"], "H_kv": hd["H_kv"],
                   "head_dim": hd["head_dim"], "block_size": 16,
                   "num_blocks": hd["num_blocks"], "kv_bytes_per_step": hd["kv_bytes_per_step"],
                   "algorithmic_bytes_per_step": hd["algorithmic_bytes_per_step"],
                   "flops_per_step": hd["flops_per_step"], "tflops": hd["tflops"],
                   "l2": hd["l2"], "l2_flushed": hd["l2_flushed"],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "launch": ("each engine step replayed from a CUDA graph (captured once)"
                              if args.graph else "eager launches through the C ABI")},
        "gpu_launches": hd["gpu_launches"],
        "roofline": hd["roofline"],
        "workloads": {n: entries[n] for n in ALL_WORKLOADS if n in entries} if len(names) > 1
        else None,
        "mixed_batch": ({"workload": entries["prefix_chunked_prefill"]["workload"],
                         "value": entries["prefix_chunked_prefill"]["tokens_per_s"],
                         "unit": "tokens/s",
                         "tflops": entries["prefix_chunked_prefill"]["tflops"]}
                        if "prefix_chunked_prefill" in entries else None),
        "e2e": e2e,
        "cpu_baseline": hd.get("cpu_baseline"),
        "clocks": clk,
    }
    return result


# ------------------------------------------------------------------------------------
# other operations on the pool: block copies (copy-on-write, swap out / in)
# ------------------------------------------------------------------------------------
def time_events(fn, steps: int, warmup: int, per_graph: int = 0) -> float:
    """Mean ms of fn() over `steps` calls, CUDA events on the current stream. With
    per_graph > 0 the calls are captured in a CUDA graph of per_graph calls and replayed,
    so the host's per-call cost (argument checks, ctypes) does not limit the rate."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if per_graph > 0:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            for _ in range(per_graph):
                fn()
        reps = max(1, steps // per_graph)
        g.replay()
        torch.cuda.synchronize()
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(reps):
            g.replay()
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * per_graph)
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_copy_blocks(args, rank, world, local_rank) -> dict | None:
    """Copy-on-write of 8192 blocks inside the decode workload's pool (device to device),
    and a swap of 4096 blocks out to a pinned host pool and back in."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_attention_18_gb300 import binding
    torch.cuda.set_device(local_rank)
    peaks, peaks_src = load_peaks()
    wl = make_workload("qwen15b_decode", rank)
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}[wl.dtype]
    k = W.to_device(wl.k_pool, wl.dtype, "cuda")
    v = W.to_device(wl.v_pool, wl.dtype, "cuda")
    nb = wl.num_blocks
    block_bytes = 16 * wl.H_kv * wl.D * 2
    rng = np.random.default_rng(90 + rank)
    n_cow = 8192
    perm = rng.permutation(nb)
    src = torch.tensor(perm[:n_cow].astype(np.int32), device="cuda")
    dst = torch.tensor(perm[n_cow:2 * n_cow].astype(np.int32), device="cuda")
    ms_cow = time_events(lambda: binding.copy_blocks(k, v, k, v, src, dst), args.steps,
                         args.warmup, per_graph=10)
    cow_bytes = 2 * 2 * n_cow * block_bytes  # read + write, K and V
    n_swap = 4096
    hk = torch.empty((n_swap, 16, wl.H_kv, wl.D), dtype=dt).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    host_ids = torch.arange(n_swap, dtype=torch.int32, device="cuda")
    dev_ids = torch.tensor(rng.choice(nb, n_swap, replace=False).astype(np.int32), device="cuda")
    swap_steps = max(3, min(args.steps, 50))
    ms_out = time_events(lambda: binding.copy_blocks(k, v, hk, hv, dev_ids, host_ids),
                         swap_steps, args.warmup, per_graph=5)
    ms_in = time_events(lambda: binding.copy_blocks(hk, hv, k, v, host_ids, dev_ids),
                        swap_steps, args.warmup, per_graph=5)
    if binding.device_error() != 0:
        raise RuntimeError("device error word set during the block-copy benchmark")
    ms_cow = reduce_max(ms_cow, world)
    swap_bytes = 2 * n_swap * block_bytes  # K and V moved once over the host link
    gbs = world * cow_bytes / (ms_cow / 1e3) / 1e9
    if rank != 0:
        return None
    return {
        "metric": "KV block copy-on-write GB/s (read + write)", "value": gbs, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_cow,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (the decode workload's pool; random block pairs)",
        "config": {"workload": f"copy {n_cow} blocks of {block_bytes} B (K and V) inside the "
                               f"{2 * nb * block_bytes / 1e6:.0f} MB decode pool",
                   "l2": "pool larger than L2; no flush"},
        "roofline": {"bound": "hbm", "achieved": gbs / world, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": gbs / world / peaks["hbm_gbs"], "traffic": None,
                     "kernel": "copy_blocks_kernel", "peak_source": f"{peaks_src} (hbm_gbs)"},
        "swap": {"blocks": n_swap, "bytes": swap_bytes,
                 "out_gbs": swap_bytes / (ms_out / 1e3) / 1e9,
                 "in_gbs": swap_bytes / (ms_in / 1e3) / 1e9,
                 "note": "device pool <-> pinned host pool in one kernel over the host link "
                         "(no measured link peak, so no roofline)"},
        "gpu_launches": args.steps,
    }


def run_rope_cache(args, rank, world, local_rank) -> dict | None:
    """Rotary embedding of q (in place) and k, fused with the KV scatter, for 32768 new
    tokens at Qwen2.5-1.5B attention shapes (12/2 heads, D 128, bf16, theta 10^6)."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_attention_18_gb300 import binding
    torch.cuda.set_device(local_rank)
    peaks, peaks_src = load_peaks()
    T, H_q, H_kv, D, nb = 32768, 12, 2, 128, 2304
    dev = torch.device("cuda", local_rank)
    g = torch.Generator(dev).manual_seed(97 + rank)
    q = torch.randn((T, H_q, D), device=dev, generator=g).to(torch.bfloat16)
    k = torch.randn((T, H_kv, D), device=dev, generator=g).to(torch.bfloat16)
    v = torch.randn((T, H_kv, D), device=dev, generator=g).to(torch.bfloat16)
    kp = torch.zeros((nb, 16, H_kv, D), device=dev, dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    rng = np.random.default_rng(97 + rank)
    pos = torch.tensor(rng.integers(0, 32768, T).astype(np.int32), device=dev)
    slots = torch.tensor(rng.permutation(nb * 16)[:T].astype(np.int32), device=dev)
    ms = reduce_max(time_events(lambda: binding.rope_reshape_and_cache(q, k, v, pos, slots, kp, vp, 1e6),
                                args.steps, args.warmup, per_graph=10), world)
    if binding.device_error() != 0:
        raise RuntimeError("device error word set during the rotary scatter benchmark")
    nbytes = T * (2 * H_q + 4 * H_kv) * D * 2 + 2 * T * 4  # q in and out, k, v in, pool rows out
    gbs = world * nbytes / (ms / 1e3) / 1e9
    if rank != 0:
        return None
    return {
        "metric": "rotary KV scatter GB/s (q rotated in place, k rotated into the pool)",
        "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (N(0,1) values, random slots)",
        "config": {"workload": f"T={T} tokens, {H_q}/{H_kv} heads, D {D}, theta 1e6",
                   "bytes_per_call": nbytes, "l2": f"{nbytes / 1e6:.0f} MB per call, larger than L2"},
        "roofline": {"bound": "hbm", "achieved": gbs / world, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": gbs / world / peaks["hbm_gbs"], "traffic": None,
                     "kernel": "rope_reshape_and_cache_kernel",
                     "peak_source": f"{peaks_src} (hbm_gbs)"},
        "gpu_launches": args.steps,
    }


def run_spec_accept(args, rank, world, local_rank) -> dict | None:
    """Acceptance of 4 drafts for 132 sequences over a 151936-token vocabulary: the
    rejection rule with draft-model probabilities (the headline), with one-hot n-gram
    drafts, and greedy."""
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from paged_kv_attention_18_gb300 import binding
    torch.cuda.set_device(local_rank)
    peaks, peaks_src = load_peaks()
    B, k, V = 132, 4, 151936
    dev = torch.device("cuda", local_rank)
    # three independent input sets used in turn, so no call re-reads rows the call before
    # it left in L2 (the one-hot mode reads 80 MB a call, less than the L2)
    sets = []
    for i in range(3):
        seed = 95 + 7 * rank + i
        rng = np.random.default_rng(seed)
        gen = torch.Generator(dev).manual_seed(seed)
        lt = torch.randn((B, k + 1, V), device=dev, generator=gen) * 2.0
        p = torch.softmax(lt, dim=-1).contiguous()
        q = torch.softmax(lt[:, :k] * 0.9 + torch.randn((B, k, V), device=dev, generator=gen),
                          dim=-1).contiguous()
        del lt
        drafts = torch.multinomial(q.reshape(B * k, V), 1, generator=gen).reshape(B, k)
        drafts = drafts.to(torch.int32).contiguous()
        rnd = torch.tensor(rng.integers(0, 2 ** 32, size=(B, k + 1), dtype=np.uint64)
                           .astype(np.uint32).view(np.int32), device=dev)
        sets.append((p, q, drafts, rnd))
    ws = torch.empty(max(int(binding.lib().ps_spec_accept_workspace_size(B, k, V)), 256),
                     dtype=torch.uint8, device=dev)
    turn = [0]

    def cycled(call):
        def fn():
            p, q, drafts, rnd = sets[turn[0] % len(sets)]
            turn[0] += 1
            return call(p, q, drafts, rnd)
        return fn

    # outputs preallocated by the first call are reused inside the captured graph
    runs = {
        "draft_model": (cycled(lambda p, q, d, r: binding.spec_accept(p, d, r, q, workspace=ws)),
                        2),
        "ngram": (cycled(lambda p, q, d, r: binding.spec_accept(p, d, r, None, workspace=ws)), 1),
        "greedy": (cycled(lambda p, q, d, r: binding.spec_accept(p, d, None, None, greedy=True,
                                                                  workspace=ws)), k + 1),
    }
    # rows each call reads: with draft rows q, the stopping row of p and of q, or p alone
    # for a sequence whose every draft survived (the bonus draw); averaged over the sets
    q_rows = []
    for p, q, drafts, rnd in sets:
        _, num = binding.spec_accept(p, drafts, rnd, q, workspace=ws)
        q_rows.append(float((num < k).float().mean().item()))
    runs["draft_model"] = (runs["draft_model"][0], 1 + sum(q_rows) / len(q_rows))
    res = {}
    for name, (fn, rows) in runs.items():
        ms = reduce_max(time_events(fn, args.steps, args.warmup, per_graph=10), world)
        nbytes = B * rows * V * 4  # probability rows the rule needs per call
        res[name] = {"ms": ms, "gbs": world * nbytes / (ms / 1e3) / 1e9,
                     "seq_per_s": world * B / (ms / 1e3),
                     "rows_read_per_sequence": round(rows, 4)}
    p, q, drafts, rnd = sets[0]
    _, num = binding.spec_accept(p, drafts, rnd, q, workspace=ws)
    torch.cuda.synchronize()
    if binding.device_error() != 0:
        raise RuntimeError("device error word set during the acceptance benchmark")
    if rank != 0:
        return None
    head = res["draft_model"]
    return {
        "metric": "speculative acceptance GB/s of probability rows (rejection rule)",
        "value": head["gbs"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (softmax of N(0, 4) logits; drafts drawn from q)",
        "config": {"workload": f"B={B} sequences, k={k} drafts, V={V}",
                   "mean_accepted": float(num.float().mean().item()),
                   "l2": "three input sets (400 MB target, 320 MB draft rows each) used in "
                         "turn: consecutive calls read different rows"},
        "roofline": {"bound": "hbm", "achieved": head["gbs"] / world, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": head["gbs"] / world / peaks["hbm_gbs"],
                     "traffic": None, "kernel": "spec_stream_kernel + spec_final_kernel",
                     "peak_source": f"{peaks_src} (hbm_gbs)"},
        "modes": res,
        "gpu_launches": 2 * args.steps,
    }


# ------------------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands
# ------------------------------------------------------------------------------------
def run_reference(args, rank, world) -> dict | None:
    """The CPU oracle as it stands, on the host cores (one single-threaded process per
    core), on the headline workload and unit; each step is one pass over a bounded sample
    of its sequences, sized so that warm-up and steps take about two minutes."""
    if rank != 0:
        return None
    name = args.workload or HEADLINE
    unit = UNITS[name]
    wl = make_workload(name, 0, args.batch)
    st = wl.steps[0]
    pool = OraclePool() if (os.cpu_count() or 1) > 1 else None
    ncores = pool.n if pool else 1
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    seqs = sample_sequences(wl, st, per_step_budget * ncores)
    path = tempfile.mkdtemp(prefix="oracle_ref_")
    total_t, total_b, total_tok = 0.0, 0, 0
    try:
        if pool:
            save_sample(wl, st, seqs, path)
            n_b = np.diff(st.query_start_loc).astype(np.int64)
            order = sorted(range(len(seqs)),
                           key=lambda i: -int(st.seq_lens[seqs[i]]) * max(1, int(n_b[seqs[i]])))
            chunks = [order[c::ncores] for c in range(ncores)]
            chunks = [c for c in chunks if c]
            pool.prepare(path)
            run = lambda: pool.run(path, chunks)  # noqa: E731
        else:
            run = lambda: oracle_seconds(wl, st, seqs)  # noqa: E731
        for _ in range(args.warmup):
            run()
        for _ in range(args.steps):
            dt, nb, nt = run()
            total_t += dt
            total_b += nb
            total_tok += nt
    finally:
        import shutil
        shutil.rmtree(path, ignore_errors=True)
        if pool:
            pool.close()
    value = _rate(total_b, total_tok, total_t, unit)
    sample = (f"{len(seqs)} of {st.B} sequences of engine step 0 per step, over {ncores} "
              "single-threaded CPU oracle processes")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic (seeded N(0,1) values, random block permutation)",
            "config": {"workload": wl.name, "description": wl.description},
            "cpu_baseline": {"value": value, "unit": unit, "cores": ncores, "kind": "oracle",
                             "sample": sample, "cpu": cpu_info()},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, choices=sorted(W.NAMED),
                    help="time this workload alone (default: the five specified workloads, "
                         "with the decode workload as the headline)")
    ap.add_argument("--batch", type=int, default=None,
                    help="decode batch size for qwen15b_decode (default 256); for small "
                         "profiling cases")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-flushed", action="store_true",
                    help="skip the L2-flushed companion timing of a workload larger than L2")
    ap.add_argument("--e2e-eager", action="store_true",
                    help="time the end-to-end leg with plain ps_attention_step_host calls "
                         "instead of its recorded graph")
    ap.add_argument("--op", choices=["step", "copy_blocks", "spec_accept", "rope_cache"],
                    default="step",
                    help="step: the attention step (default); copy_blocks: block copies; "
                         "spec_accept: speculative acceptance; rope_cache: rotary KV scatter")
    ap.add_argument("--graph", action="store_true",
                    help="capture each engine step in a CUDA graph and time its replays")
    ap.add_argument("--no-clocks", action="store_true",
                    help="no nvidia-smi sampling and no extra load after the timed steps")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" and torch.cuda.is_available() else "gloo"
        if args.impl == "reference":
            # only rank 0 works; the others leave at once
            if rank != 0:
                return 0
            world_eff = 1
        else:
            torch.cuda.set_device(local_rank)
            dist.init_process_group(backend=backend)
            world_eff = world
    else:
        world_eff = 1
    if args.impl == "reference":
        res = run_reference(args, 0 if world_eff == 1 else rank, world)
    elif args.op == "copy_blocks":
        res = run_copy_blocks(args, rank, world_eff, local_rank)
    elif args.op == "spec_accept":
        res = run_spec_accept(args, rank, world_eff, local_rank)
    elif args.op == "rope_cache":
        res = run_rope_cache(args, rank, world_eff, local_rank)
    else:
        res = run_ours(args, rank, world_eff, local_rank)
    if res is not None:
        print(json.dumps(res), flush=True)
    if world_eff > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
