"""CPU oracle for one attention step over a paged KV cache.

TEST INFRASTRUCTURE. This module is the plain, slow, obviously-correct statement
of what the CUDA library computes. Only the test-suite, the package's smoke check
and the benchmark's CPU-baseline arm may import or run it; the library never does,
and it imports nothing from the library.

What it follows (the three pages on paged KV serving: "PageServe", "tinyserve",
"PagedServe"):

* Pool layout. One pre-allocated pool of fixed 16-token blocks, shaped
  [blocks, 16, H_kv, D] for one layer (PageServe, "System architecture" figure,
  PagedKVCache [layers, blocks, 16, H, D]; development-history phase 7). tinyserve
  ("How it works") holds the same memory as a slab [blocks x 16, H_kv, D], so
  ``pool.reshape(blocks * 16, H_kv, D)[slot]`` is the row a slot names.
* Slot formula. A token at position ``pos`` of a sequence lives at
  ``slot = block_table[pos // 16] * 16 + pos % 16`` (PageServe, section 01
  "Scheduler loop", closing paragraph, and the attention_wrapper.py code box in
  section 03 "Paged KV cache").
* Positions. Each sequence tracks the tokens that already have K/V in the pool; a
  prefill chunk, a decode and a recompute are the same operation over the tokens
  not yet computed (PageServe, section 01 "Scheduler loop"). With ``seq_lens`` the
  context length after this step, the step's n query tokens therefore sit at
  positions ``seq_len - n .. seq_len - 1``.
* Scatter then attend. The attention backend "writes K/V into the pool" and "reads
  context via block tables" in one packed [1, T] pass with explicit positions
  (PageServe, section 01 "Execute" / "Pack"; development-history phase 8).
* Attention. softmax(q K^T * scale) V with a causal mask (key j visible to the
  query at position p iff j <= p); grouped-query attention with query head h using
  KV head h // (H_q / H_kv) (tinyserve, "Highlights" table, forward-pass row;
  the "stepped causal mask" for k+1 verify tokens, tinyserve "How it works").

The arithmetic defaults to float64; ``acc=np.float32`` runs the same steps in
float32. Inputs of 16-bit types arrive as raw bit patterns (uint16) and are decoded
exactly.
"""
from __future__ import annotations

import numpy as np

BLOCK_SIZE = 16


# --------------------------------------------------------------------------- #
# 16-bit decoding (exact)
# --------------------------------------------------------------------------- #
def decode_bits(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of f16 / bf16 bit patterns."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# --------------------------------------------------------------------------- #
# slot mapping and scatter
# --------------------------------------------------------------------------- #
def slot_of(block_table_row: np.ndarray, pos: int) -> int:
    """Physical slot of logical position ``pos`` (PageServe section 01 / 03)."""
    return int(block_table_row[pos // BLOCK_SIZE]) * BLOCK_SIZE + pos % BLOCK_SIZE


def query_positions(seq_lens: np.ndarray, query_start_loc: np.ndarray) -> np.ndarray:
    """Position of every packed query token: the uncomputed tail of its sequence."""
    T = int(query_start_loc[-1])
    pos = np.full(T, -1, dtype=np.int64)
    for b in range(len(seq_lens)):
        start, end = int(query_start_loc[b]), int(query_start_loc[b + 1])
        n = end - start
        L = int(seq_lens[b])
        if n > L:
            raise ValueError(f"sequence {b}: {n} query tokens but context {L}")
        for i in range(n):
            pos[start + i] = L - n + i
    return pos


def slot_mapping(block_tables: np.ndarray, seq_lens: np.ndarray,
                 query_start_loc: np.ndarray) -> np.ndarray:
    """Slot of every packed token ("slot mapping per token", PageServe section 01)."""
    pos = query_positions(seq_lens, query_start_loc)
    out = np.full(pos.shape[0], -1, dtype=np.int64)
    for b in range(len(seq_lens)):
        for t in range(int(query_start_loc[b]), int(query_start_loc[b + 1])):
            out[t] = slot_of(block_tables[b], int(pos[t]))
    return out


def reshape_and_cache(k: np.ndarray, v: np.ndarray, slots: np.ndarray,
                      k_pool: np.ndarray, v_pool: np.ndarray):
    """Pools after writing each token's K/V row at its slot; a negative slot is skipped.

    Returns new arrays; the inputs are not modified. Works on any element type (the
    copy is of bit patterns).
    """
    nb, bs, h_kv, d = k_pool.shape
    kp = k_pool.copy().reshape(nb * bs, h_kv, d)
    vp = v_pool.copy().reshape(nb * bs, h_kv, d)
    for t in range(k.shape[0]):
        s = int(slots[t])
        if s < 0:
            continue
        kp[s] = k[t]
        vp[s] = v[t]
    return kp.reshape(nb, bs, h_kv, d), vp.reshape(nb, bs, h_kv, d)


# --------------------------------------------------------------------------- #
# block copies (copy-on-write, swap out / in)
# --------------------------------------------------------------------------- #
def copy_blocks(src_pool: np.ndarray, dst_pool: np.ndarray, src_ids, dst_ids) -> np.ndarray:
    """A copy of dst_pool in which block dst_ids[i] holds block src_ids[i] of src_pool.

    Every pair reads the source as it was before the call. This is the copy-on-write of
    a block shared by several tables before one of them writes into it (tinyserve "How
    it works"; "Highlights" table, paged KV-cache row) and the lossless swap of a
    preempted sequence's blocks to a pinned host pool and back (PageServe section 04
    "Phase 9 - Preemption"; tinyserve "How it works"). A pair with an id outside its
    pool is skipped.
    """
    src = np.asarray(src_pool)
    out = np.array(dst_pool, copy=True)
    for s, d in zip(np.asarray(src_ids).tolist(), np.asarray(dst_ids).tolist()):
        if 0 <= s < src.shape[0] and 0 <= d < out.shape[0]:
            out[d] = src[s]
    return out


# --------------------------------------------------------------------------- #
# rotary position embedding (fused with the scatter in the library)
# --------------------------------------------------------------------------- #
def rope(x_bits: np.ndarray, positions, theta: float, dtype: str) -> np.ndarray:
    """Rotary embedding of x [T, H, D] (16-bit bit patterns) by each token's position,
    exact in float64: for frequency i < D/2, with a = pos * theta^(-2i/D),
    x'[i] = x[i] cos a - x[i + D/2] sin a and x'[i + D/2] = x[i + D/2] cos a + x[i] sin a.

    The Qwen2 decoder's rotary embeddings (tinyserve "Highlights" table, forward-pass
    row) applied at the explicit position ids of the packed batch (PageServe section 01);
    the pairing of element i with i + D/2 (rotate-half) is the plainest reading of a
    Qwen2-style rotary embedding, which the pages name without a formula."""
    x = decode_bits(x_bits, dtype)
    D = x.shape[-1]
    half = D // 2
    inv_freq = float(theta) ** (-(2.0 * np.arange(half)) / D)
    a = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    c, s = np.cos(a)[:, None, :], np.sin(a)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_reshape_and_cache(q, k, v, positions, slots, k_pool, v_pool, theta, dtype):
    """The fused step: (rotated q, rotated k, v pool after the scatter) in float64 for q
    and k; the K pool rows at the slots hold the rotated keys rounded to the 16-bit type,
    which the caller compares within the rounding; the V pool is exact bits."""
    q_rot = rope(q, positions, theta, dtype)
    k_rot = rope(k, positions, theta, dtype)
    _, v_out = reshape_and_cache(k, v, slots, k_pool, v_pool)
    return q_rot, k_rot, v_out


# --------------------------------------------------------------------------- #
# attention
# --------------------------------------------------------------------------- #
def kv_head_of(h: int, H_q: int, H_kv: int) -> int:
    """KV head read by query head h: consecutive query heads share one KV head."""
    return h // (H_q // H_kv)


def gather_context(pool: np.ndarray, block_table_row: np.ndarray, L: int) -> np.ndarray:
    """The first L cached rows of a sequence, [L, H_kv, D], read through its table."""
    nb, bs, h_kv, d = pool.shape
    flat = pool.reshape(nb * bs, h_kv, d)
    rows = [flat[slot_of(block_table_row, j)] for j in range(L)]
    if not rows:
        return np.zeros((0, h_kv, d), dtype=pool.dtype)
    return np.stack(rows)


def causal_softmax_attention(Q: np.ndarray, K: np.ndarray, V: np.ndarray,
                             positions: np.ndarray, scale: float, acc=np.float64):
    """softmax(Q K^T * scale + causal mask) V for one head.

    Q [R, D] query rows at the given positions, K/V [L, D]. Key j is visible to row r
    iff j <= positions[r]. Returns (O [R, D], P [R, L]); masked entries of P are 0.
    """
    Q = Q.astype(acc)
    K = K.astype(acc)
    V = V.astype(acc)
    scale = acc(scale)
    L = K.shape[0]
    S = (Q @ K.T) * scale
    visible = np.arange(L)[None, :] <= np.asarray(positions)[:, None]
    if not visible.any(axis=1).all():
        raise ValueError("a query row sees no key")
    S = np.where(visible, S, acc(-np.inf))
    m = S.max(axis=1, keepdims=True)
    E = np.where(visible, np.exp(S - m), acc(0))
    P = E / E.sum(axis=1, keepdims=True)
    return P @ V, P


def paged_attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                    block_tables: np.ndarray, seq_lens: np.ndarray,
                    query_start_loc: np.ndarray, scale: float, dtype: str,
                    acc=np.float64, rows=None, return_probs: bool = False):
    """Attention output for every packed query token (or the ``rows`` subset).

    q [T, H_q, D] and the pools [blocks, 16, H_kv, D] are 16-bit bit patterns of
    ``dtype``. Returns float arrays in ``acc``: out [T, H_q, D] (rows not selected
    are NaN); with ``return_probs`` also a dict {(row, head): P over the context}.
    """
    T, H_q, D = q.shape
    H_kv = k_pool.shape[2]
    if H_q % H_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    qf = decode_bits(q, dtype)
    out = np.full((T, H_q, D), np.nan, dtype=acc)
    probs = {}
    pos = query_positions(seq_lens, query_start_loc)
    want = None if rows is None else set(int(r) for r in rows)
    for b in range(len(seq_lens)):
        start, end = int(query_start_loc[b]), int(query_start_loc[b + 1])
        rs = [r for r in range(start, end) if want is None or r in want]
        if not rs:
            continue
        L = int(seq_lens[b])
        Kb = decode_bits(gather_context(k_pool, block_tables[b], L), dtype)
        Vb = decode_bits(gather_context(v_pool, block_tables[b], L), dtype)
        for h in range(H_q):
            kv = kv_head_of(h, H_q, H_kv)
            O, P = causal_softmax_attention(qf[rs, h, :], Kb[:, kv, :], Vb[:, kv, :],
                                            pos[rs], scale, acc)
            out[rs, h, :] = O
            if return_probs:
                for i, r in enumerate(rs):
                    probs[(r, h)] = P[i]
    if return_probs:
        return out, probs
    return out


def attention_step(wl_step, k_pool, v_pool, scale, dtype, acc=np.float64, rows=None):
    """One engine step: scatter the step's K/V at their slots, then attend.

    Returns (out, k_pool_after, v_pool_after).
    """
    slots = slot_mapping(wl_step.block_tables, wl_step.seq_lens, wl_step.query_start_loc)
    kp, vp = reshape_and_cache(wl_step.k, wl_step.v, slots, k_pool, v_pool)
    out = paged_attention(wl_step.q, kp, vp, wl_step.block_tables, wl_step.seq_lens,
                          wl_step.query_start_loc, scale, dtype, acc=acc, rows=rows)
    return out, kp, vp
