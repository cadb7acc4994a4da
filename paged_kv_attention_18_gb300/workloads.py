"""Seeded synthetic inputs for one paged-KV attention step.

This module draws values, context lengths, query counts and block tables, and
nothing else: it holds no slot arithmetic and no attention arithmetic. The CUDA
path and the CPU oracle both consume what it makes, so it is the only code they
share.

Every array of 16-bit floating-point values is held as its raw bit pattern
(``numpy.uint16``) together with a dtype tag ("f16" or "bf16"). Values are drawn
as float32 N(0, 1) from ``numpy.random.default_rng(seed)`` and rounded to the
16-bit type with round-to-nearest-even, so both sides see identical inputs.

Block tables follow the paged pool the pages describe (PageServe, section 03
"Paged KV cache"; tinyserve, "How it works"): a pool of fixed 16-token blocks,
and per sequence a list of physical block ids taken from a random permutation of
the free ids. Entries past a sequence's last block are -1 and are never read.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK_SIZE = 16


# --------------------------------------------------------------------------- #
# value rounding (input preparation only)
# --------------------------------------------------------------------------- #
def round_to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to f16 or bf16 (nearest-even) and return the bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x.view(np.uint32).astype(np.uint64)
        u = u + 0x7FFF + ((u >> 16) & 1)
        return (u >> 16).astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def _normal_bits(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    return round_to_bits(rng.standard_normal(shape, dtype=np.float32), dtype)


# --------------------------------------------------------------------------- #
# containers
# --------------------------------------------------------------------------- #
@dataclass
class Step:
    """One packed [1, T] batch: the tokens scheduled in one engine step.

    ``seq_lens[b]`` is the context length of sequence b *after* this step's
    tokens, so its ``n_b = query_start_loc[b+1] - query_start_loc[b]`` query
    tokens are the last n_b positions of its context.
    """

    q: np.ndarray                # uint16 [T, H_q, D]
    k: np.ndarray                # uint16 [T, H_kv, D]
    v: np.ndarray                # uint16 [T, H_kv, D]
    block_tables: np.ndarray     # int32 [B, max_blocks_per_seq], -1 padded
    seq_lens: np.ndarray         # int32 [B]
    query_start_loc: np.ndarray  # int32 [B + 1]
    seq_ids: np.ndarray          # int32 [B]: which sequence of the workload each row is

    @property
    def T(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def B(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])


@dataclass
class Workload:
    name: str
    dtype: str                   # "f16" | "bf16"
    H_q: int
    H_kv: int
    D: int
    num_blocks: int
    k_pool: np.ndarray           # uint16 [num_blocks, 16, H_kv, D]: state before step 0
    v_pool: np.ndarray
    steps: list[Step] = field(default_factory=list)
    description: str = ""

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(D), rounded to float32 as a caller would pass it."""
        return float(np.float32(1.0) / np.sqrt(np.float32(self.D)))

    @property
    def G(self) -> int:
        return self.H_q // self.H_kv


# --------------------------------------------------------------------------- #
# generic builder
# --------------------------------------------------------------------------- #
def _blocks_for(tokens: int) -> int:
    return (tokens + BLOCK_SIZE - 1) // BLOCK_SIZE


def build_workload(
    name: str,
    *,
    seed: int,
    dtype: str,
    H_q: int,
    H_kv: int,
    D: int,
    capacities: list[int],
    steps: list[list[tuple[int, int, int]]],
    num_blocks: int | None = None,
    free_fraction: float = 0.10,
    shared_prefix_blocks: int = 0,
    prefix_users: list[int] | None = None,
    rng: np.random.Generator | None = None,
    description: str = "",
) -> Workload:
    """Build a workload from sequence capacities and per-step schedules.

    capacities[i]   -- tokens sequence i ever holds (sizes its block table).
    steps[s]        -- list of (seq index, context length after the step, n query tokens),
                       in packed order.
    shared_prefix_blocks / prefix_users -- the first ``shared_prefix_blocks`` entries of
                       every listed sequence's table point at the same physical blocks
                       (prefix caching: one copy, many tables).
    num_blocks      -- pool size; default ceil(blocks needed * (1 + free_fraction)).
    """
    if rng is None:
        rng = np.random.default_rng(seed)
    prefix_users = set(prefix_users or [])
    need = []
    for i, cap in enumerate(capacities):
        nb = _blocks_for(cap)
        if i in prefix_users:
            if nb < shared_prefix_blocks:
                raise ValueError("a prefix user is shorter than the shared prefix")
            nb -= shared_prefix_blocks
        need.append(nb)
    total = sum(need) + (shared_prefix_blocks if prefix_users else 0)
    if num_blocks is None:
        num_blocks = max(1, math.ceil(total * (1.0 + free_fraction)))
    if total > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {total}")

    perm = rng.permutation(num_blocks).astype(np.int32)
    cursor = 0
    prefix = perm[cursor:cursor + shared_prefix_blocks] if prefix_users else perm[:0]
    cursor += len(prefix)
    max_blk = max([_blocks_for(c) for c in capacities] + [1])
    tables = np.full((len(capacities), max_blk), -1, dtype=np.int32)
    for i, nb in enumerate(need):
        row = []
        if i in prefix_users:
            row.extend(prefix.tolist())
        row.extend(perm[cursor:cursor + nb].tolist())
        cursor += nb
        tables[i, :len(row)] = row

    k_pool = _normal_bits(rng, (num_blocks, BLOCK_SIZE, H_kv, D), dtype)
    v_pool = _normal_bits(rng, (num_blocks, BLOCK_SIZE, H_kv, D), dtype)

    wl = Workload(name=name, dtype=dtype, H_q=H_q, H_kv=H_kv, D=D,
                  num_blocks=num_blocks, k_pool=k_pool, v_pool=v_pool,
                  description=description)
    for sched in steps:
        ids = np.array([s for s, _, _ in sched], dtype=np.int32)
        lens = np.array([L for _, L, _ in sched], dtype=np.int32)
        ns = np.array([n for _, _, n in sched], dtype=np.int32)
        for (s, L, n) in sched:
            if not (0 <= n <= L <= capacities[s]):
                raise ValueError(f"bad schedule entry {(s, L, n)}")
        qsl = np.zeros(len(sched) + 1, dtype=np.int32)
        np.cumsum(ns, out=qsl[1:])
        T = int(qsl[-1])
        q = _normal_bits(rng, (T, H_q, D), dtype)
        k = _normal_bits(rng, (T, H_kv, D), dtype)
        v = _normal_bits(rng, (T, H_kv, D), dtype)
        bt = tables[ids] if len(ids) else np.zeros((0, max_blk), dtype=np.int32)
        wl.steps.append(Step(q=q, k=k, v=v, block_tables=np.ascontiguousarray(bt),
                             seq_lens=lens, query_start_loc=qsl, seq_ids=ids))
    return wl


def simple_workload(name: str, *, seed: int, dtype: str, H_q: int, H_kv: int, D: int,
                    seqs: list[tuple[int, int]], num_blocks: int | None = None,
                    shared_prefix_blocks: int = 0, prefix_users=None,
                    free_fraction: float = 0.10) -> Workload:
    """One-step workload from a list of (context length after the step, n query tokens)."""
    return build_workload(
        name, seed=seed, dtype=dtype, H_q=H_q, H_kv=H_kv, D=D,
        capacities=[max(L, 1) for L, _ in seqs],
        steps=[[(i, L, n) for i, (L, n) in enumerate(seqs)]],
        num_blocks=num_blocks, free_fraction=free_fraction,
        shared_prefix_blocks=shared_prefix_blocks, prefix_users=prefix_users)


# --------------------------------------------------------------------------- #
# the five named workloads
# --------------------------------------------------------------------------- #
def tiny_decode(seed: int = 0) -> Workload:
    """4 decodes, contexts U[1, 100]; 4/2 heads, D 64, f16, pool of 64 blocks."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 100, size=4, endpoint=True)
    return build_workload(
        "tiny_decode", seed=seed, rng=rng, dtype="f16", H_q=4, H_kv=2, D=64,
        capacities=[int(L) for L in lens],
        steps=[[(i, int(L), 1) for i, L in enumerate(lens)]],
        num_blocks=64,
        description="4 decode sequences, context U[1,100], GQA 4/2, D 64, f16, 64-block pool")


def qwen05b_mixed(seed: int = 1) -> Workload:
    """8 decodes (contexts U[64, 1024]) + 2 prefill chunks of 256 at offsets 0 and 512."""
    rng = np.random.default_rng(seed)
    dec = rng.integers(64, 1024, size=8, endpoint=True)
    caps = [int(L) for L in dec] + [256, 768]
    sched = [(i, int(L), 1) for i, L in enumerate(dec)] + [(8, 256, 256), (9, 768, 256)]
    return build_workload(
        "qwen2.5-0.5b_mixed_T520", seed=seed, rng=rng, dtype="f16", H_q=14, H_kv=2, D=64,
        capacities=caps, steps=[sched], num_blocks=2048,
        description="Qwen2.5-0.5B attention shapes 14/2, D 64, f16; T = 8 decodes + 2x256 "
                    "prefill chunks at offsets 0 and 512; 2048-block pool")


def qwen15b_decode(seed: int = 2, batch: int = 256, lo: int = 512, hi: int = 4096) -> Workload:
    """256 decodes, contexts U[512, 4096]; 12/2 heads, D 128, bf16; pool = need + 10%."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi, size=batch, endpoint=True)
    return build_workload(
        f"qwen2.5-1.5b_decode_B{batch}", seed=seed, rng=rng, dtype="bf16", H_q=12, H_kv=2,
        D=128, capacities=[int(L) for L in lens],
        steps=[[(i, int(L), 1) for i, L in enumerate(lens)]],
        description=f"Qwen2.5-1.5B attention shapes 12/2, D 128, bf16; {batch} decodes, "
                    f"context U[{lo},{hi}]; pool = blocks needed + 10% free")


def prefix_chunked_prefill(seed: int = 3, n_prefill: int = 64, prefix_tokens: int = 1024,
                           suffix_lo: int = 128, suffix_hi: int = 768, n_decode: int = 32,
                           dec_lo: int = 256, dec_hi: int = 2048, budget: int = 8192) -> Workload:
    """Prefix-cached chunked prefill packed with decodes, over several engine steps.

    64 sequences share a 1024-token prefix that is already in the pool (one set of
    physical blocks referenced by every table). Their distinct suffixes, U[128, 768],
    are prefilled first-come-first-served in chunks under a per-step budget of 8192
    new tokens, which also pays for 32 running decodes (contexts U[256, 2048], one
    token per step). Decodes are planned first, then prefill chunks (PageServe
    section 01 "Plan"; tinyserve "How it works"): the last admitted prompt is cut
    to fit the budget.
    """
    if prefix_tokens % BLOCK_SIZE:
        raise ValueError("the shared prefix must be block aligned")
    rng = np.random.default_rng(seed)
    suffix = rng.integers(suffix_lo, suffix_hi, size=n_prefill, endpoint=True)
    dec0 = rng.integers(dec_lo, dec_hi, size=n_decode, endpoint=True)
    # simulate the schedule
    done = [0] * n_prefill
    sched_steps = []
    step = 0
    while any(done[i] < suffix[i] for i in range(n_prefill)):
        sched = [(n_prefill + j, int(dec0[j]) + step, 1) for j in range(n_decode)]
        left = budget - n_decode
        for i in range(n_prefill):
            if left <= 0:
                break
            rem = int(suffix[i]) - done[i]
            if rem <= 0:
                continue
            chunk = min(rem, left)
            done[i] += chunk
            left -= chunk
            sched.append((i, prefix_tokens + done[i], chunk))
        sched_steps.append(sched)
        step += 1
    nsteps = len(sched_steps)
    caps = [prefix_tokens + int(s) for s in suffix] + [int(L) + nsteps - 1 for L in dec0]
    return build_workload(
        "qwen2.5-1.5b_prefix_chunked_prefill", seed=seed, rng=rng, dtype="bf16", H_q=12,
        H_kv=2, D=128, capacities=caps, steps=sched_steps,
        shared_prefix_blocks=prefix_tokens // BLOCK_SIZE, prefix_users=list(range(n_prefill)),
        description=f"{n_prefill} seqs share a {prefix_tokens}-token cached prefix; suffixes "
                    f"U[{suffix_lo},{suffix_hi}] chunk-prefilled under a {budget}-token step "
                    f"budget with {n_decode} decodes U[{dec_lo},{dec_hi}]; {nsteps} steps; "
                    "12/2 heads, D 128, bf16")


def spec_verify_long(seed: int = 4, n_seq: int = 128, lo: int = 1024, hi: int = 8192,
                     n_long: int = 4, long_len: int = 32768, k_plus_1: int = 5) -> Workload:
    """128 sequences with contexts U[1024, 8192] plus 4 at 32768, each scoring 5 tokens."""
    rng = np.random.default_rng(seed)
    lens = [int(L) for L in rng.integers(lo, hi, size=n_seq, endpoint=True)]
    lens += [long_len] * n_long
    return build_workload(
        "qwen2.5-1.5b_spec_verify_long", seed=seed, rng=rng, dtype="bf16", H_q=12, H_kv=2,
        D=128, capacities=lens, steps=[[(i, L, k_plus_1) for i, L in enumerate(lens)]],
        description=f"{n_seq} seqs U[{lo},{hi}] + {n_long} at {long_len}, each with "
                    f"{k_plus_1} verify tokens; 12/2 heads, D 128, bf16")


def long_prefill(seed: int = 5, n_seq: int = 4, prompt: int = 4096) -> Workload:
    """Whole prompts prefilled in one step (no cached prefix): a tensor-core stress case."""
    rng = np.random.default_rng(seed)
    return build_workload(
        f"qwen2.5-1.5b_prefill_{n_seq}x{prompt}", seed=seed, rng=rng, dtype="bf16", H_q=12,
        H_kv=2, D=128, capacities=[prompt] * n_seq,
        steps=[[(i, prompt, prompt) for i in range(n_seq)]],
        description=f"{n_seq} prompts of {prompt} tokens prefilled at once, causal; 12/2 "
                    "heads, D 128, bf16")


NAMED = {
    "tiny_decode": tiny_decode,
    "qwen05b_mixed": qwen05b_mixed,
    "qwen15b_decode": qwen15b_decode,
    "prefix_chunked_prefill": prefix_chunked_prefill,
    "spec_verify_long": spec_verify_long,
    "long_prefill": long_prefill,
}


def named(name: str, **kw) -> Workload:
    return NAMED[name](**kw)


# --------------------------------------------------------------------------- #
# device upload and sub-sampling (host plumbing)
# --------------------------------------------------------------------------- #
def to_device(a: np.ndarray, dtype: str | None = None, device="cuda"):
    """A torch tensor on ``device`` holding the array; uint16 bit patterns become f16/bf16."""
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).view(
            {"f16": torch.float16, "bf16": torch.bfloat16}[dtype])
    else:
        t = torch.from_numpy(a)
    return t.to(device)


def subset(wl: Workload, step: Step, seqs: list[int]) -> tuple[Workload, Step]:
    """The sequences ``seqs`` of one step, with a pool holding only the blocks they use.

    Physical block ids are relabelled 0..m-1 in order of first use; values are unchanged.
    """
    seqs = list(seqs)
    bt = step.block_tables[seqs]
    used = []
    seen = {}
    for row in bt:
        for blk in row:
            if blk >= 0 and int(blk) not in seen:
                seen[int(blk)] = len(used)
                used.append(int(blk))
    remap = np.vectorize(lambda x: seen.get(int(x), -1), otypes=[np.int32])
    new_bt = remap(bt) if bt.size else bt.astype(np.int32)
    n = np.diff(step.query_start_loc)[seqs]
    qsl = np.zeros(len(seqs) + 1, dtype=np.int32)
    np.cumsum(n, out=qsl[1:])
    rows = np.concatenate([np.arange(step.query_start_loc[b], step.query_start_loc[b + 1])
                           for b in seqs]).astype(np.int64) if seqs else np.zeros(0, np.int64)
    sub = Workload(name=wl.name + f"[{len(seqs)} seqs]", dtype=wl.dtype, H_q=wl.H_q,
                   H_kv=wl.H_kv, D=wl.D, num_blocks=max(1, len(used)),
                   k_pool=wl.k_pool[used] if used else wl.k_pool[:1],
                   v_pool=wl.v_pool[used] if used else wl.v_pool[:1], description=wl.description)
    st = Step(q=step.q[rows], k=step.k[rows], v=step.v[rows],
              block_tables=np.ascontiguousarray(new_bt, dtype=np.int32),
              seq_lens=step.seq_lens[seqs].copy(), query_start_loc=qsl,
              seq_ids=step.seq_ids[seqs].copy())
    sub.steps.append(st)
    return sub, st
