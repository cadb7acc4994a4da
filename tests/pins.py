"""Checks that pin the CPU oracle to facts other than itself.

Each pin takes the oracle module and raises AssertionError when the oracle
disagrees with what the pages or the mathematics fix: the pages' worked block-table
figure, hand-worked cases, closed forms, a library attention routine, and the
invariances the pages state (paging and prefix sharing change no result). The
mutant tests run the same pins against copies of the oracle with planted mistakes
and require every mistake to be caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BS = 16


def f16(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def place_paged(ctx: np.ndarray, table: list[int], num_blocks: int, fill: np.ndarray | None = None):
    """Pool [num_blocks, 16, H, D] holding context row j in block table[j // 16], row j % 16.

    Test scaffolding: this is how a block table is defined to map positions (the pages'
    block tables map logical positions to physical blocks of 16).
    """
    L, H, D = ctx.shape
    pool = np.zeros((num_blocks, BS, H, D), dtype=ctx.dtype) if fill is None else fill.copy()
    for j in range(L):
        pool[table[j // BS], j % BS] = ctx[j]
    return pool


def enumerate_slots(table: list[int], L: int) -> list[int]:
    """Slots of positions 0..L-1 by walking the table's blocks in order (no division)."""
    out = []
    for blk in table:
        for off in range(BS):
            if len(out) == L:
                return out
            out.append(blk * BS + off)
    return out


# --------------------------------------------------------------------------- #
# slot formula and scatter
# --------------------------------------------------------------------------- #
def pin_slots_golden(o):
    fx = json.load(open(os.path.join(GOLDEN, "slots_tinyserve_figure.json")))
    for s in fx["sequences"]:
        L = s["length"]
        tables = np.array([s["block_table"]], dtype=np.int32)
        got = o.slot_mapping(tables, np.array([L]), np.array([0, L]))
        assert got.tolist() == s["expected_slots"], (s["name"], got.tolist())


def pin_slots_brute_force(o, seed=11):
    rng = np.random.default_rng(seed)
    nb = 40
    perm = rng.permutation(nb)
    lens = [1, 15, 16, 17, 33, 70]
    tables, cur = [], 0
    for L in lens:
        k = -(-L // BS)
        tables.append(list(perm[cur:cur + k]) + [-1] * (5 - k))
        cur += k
    tables = np.array(tables, dtype=np.int32)
    # every position of every sequence queried once (n = L)
    qsl = np.concatenate([[0], np.cumsum(lens)])
    got = o.slot_mapping(tables, np.array(lens), qsl)
    want = sum((enumerate_slots(list(t), L) for t, L in zip(tables, lens)), [])
    assert got.tolist() == want
    assert len(set(want)) == len(want)  # unshared blocks: every slot distinct
    # decode rows (n = 1): the last position only
    got = o.slot_mapping(tables, np.array(lens), np.arange(len(lens) + 1))
    assert got.tolist() == [enumerate_slots(list(t), L)[-1] for t, L in zip(tables, lens)]


def pin_scatter_roundtrip(o, seed=12):
    rng = np.random.default_rng(seed)
    nb, H, D = 24, 2, 8
    sentinel = np.uint16(0x7BFF)
    kp = np.full((nb, BS, H, D), sentinel, dtype=np.uint16)
    vp = np.full((nb, BS, H, D), sentinel, dtype=np.uint16)
    perm = rng.permutation(nb)
    lens, ns = [5, 40, 16], [5, 3, 1]
    tables = np.full((3, 3), -1, dtype=np.int32)
    cur = 0
    for b, L in enumerate(lens):
        k = -(-L // BS)
        tables[b, :k] = perm[cur:cur + k]
        cur += k
    qsl = np.concatenate([[0], np.cumsum(ns)])
    T = int(qsl[-1])
    k = rng.integers(0, 0x7000, size=(T, H, D)).astype(np.uint16)
    v = rng.integers(0, 0x7000, size=(T, H, D)).astype(np.uint16)
    slots = o.slot_mapping(tables, np.array(lens), qsl)
    kp2, vp2 = o.reshape_and_cache(k, v, slots, kp, vp)
    assert kp.flat[0] == sentinel  # inputs untouched
    written = set()
    for b, (L, n) in enumerate(zip(lens, ns)):
        for i in range(n):
            pos = L - n + i
            s = enumerate_slots(list(tables[b]), L)[pos]
            written.add(s)
            t = qsl[b] + i
            assert (kp2.reshape(-1, H, D)[s] == k[t]).all()
            assert (vp2.reshape(-1, H, D)[s] == v[t]).all()
    for s in range(nb * BS):
        if s not in written:
            assert (kp2.reshape(-1, H, D)[s] == sentinel).all()
            assert (vp2.reshape(-1, H, D)[s] == sentinel).all()
    # a negative slot is skipped
    kp3, _ = o.reshape_and_cache(k, v, np.full(T, -1), kp, vp)
    assert (kp3 == kp).all()
    # the first and the last slot of the pool are ordinary slots
    edge = np.full(T, -1)
    edge[0], edge[1] = 0, nb * BS - 1
    kp4, vp4 = o.reshape_and_cache(k, v, edge, kp, vp)
    assert (kp4[0, 0] == k[0]).all() and (vp4[0, 0] == v[0]).all()
    assert (kp4[-1, -1] == k[1]).all() and (vp4[-1, -1] == v[1]).all()
    assert (kp4.reshape(-1, H, D)[1:-1] == sentinel).all()


# --------------------------------------------------------------------------- #
# attention
# --------------------------------------------------------------------------- #
def _run_case(o, q, K, V, scale, n, table=(3, 1), nb=5, seed=0):
    """Attention of one sequence whose context K/V [L, H_kv, D] sits at ``table``."""
    rng = np.random.default_rng(seed)
    L = K.shape[0]
    noise = f16(rng.standard_normal((nb, BS) + K.shape[1:]))
    kp = place_paged(K, list(table), nb, noise)
    vp = place_paged(V, list(table), nb, noise)
    bt = np.array([list(table)], dtype=np.int32)
    return o.paged_attention(q, kp, vp, bt, np.array([L]), np.array([0, n]), scale, "f16")


def pin_golden_tiny(o):
    fx = json.load(open(os.path.join(GOLDEN, "tiny_attention_cases.json")))
    scales = {"ln3": math.log(3.0), "ln2": math.log(2.0), "1": 1.0}
    for c in fx["cases"]:
        q = f16(c["q"])[:, None, :]
        K = f16(c["K"])[:, None, :]
        V = f16(c["V"])[:, None, :]
        out = _run_case(o, q, K, V, scales[c["scale"]], c["n_query"])
        np.testing.assert_allclose(out[:, 0, :], np.array(c["expected"]), rtol=0, atol=1e-12,
                                   err_msg=c["name"])


def pin_closed_forms(o, seed=13):
    rng = np.random.default_rng(seed)
    D = 16
    # context of one: o = v0 exactly, for every head
    q = f16(rng.standard_normal((1, 4, D)))
    K = f16(rng.standard_normal((1, 2, D)))
    V = f16(rng.standard_normal((1, 2, D)))
    out = _run_case(o, q, K, V, 0.25, 1)
    vv = o.decode_bits(V, "f16")
    for h in range(4):
        assert (out[0, h] == vv[0, h // 2]).all()
    # all keys equal: uniform weights, o = mean of V over the visible keys
    L = 37
    K = np.repeat(f16(rng.standard_normal((1, 2, D))), L, axis=0)
    V = f16(rng.standard_normal((L, 2, D)))
    q = f16(rng.standard_normal((3, 4, D)))
    out = _run_case(o, q, K, V, 0.3, 3, table=(4, 0, 2))
    vv = o.decode_bits(V, "f16")
    for i in range(3):
        p = L - 3 + i
        for h in range(4):
            np.testing.assert_allclose(out[i, h], vv[:p + 1, h // 2].mean(axis=0), atol=1e-12)
    # q = 0: same uniform average whatever the keys are
    K = f16(rng.standard_normal((L, 2, D)))
    q = f16(np.zeros((2, 4, D)))
    out = _run_case(o, q, K, V, 0.3, 2, table=(4, 0, 2))
    for i in range(2):
        p = L - 2 + i
        for h in range(4):
            np.testing.assert_allclose(out[i, h], vv[:p + 1, h // 2].mean(axis=0), atol=1e-12)
    # one dominant logit: o is that key's value (other weights below e^-40)
    K = f16(np.zeros((L, 2, D)))
    K[5] = f16(np.full((2, D), 4.0))
    q = f16(np.full((1, 4, D), 4.0))
    out = _run_case(o, q, K, V, 1.0, 1, table=(4, 0, 2))
    for h in range(4):
        np.testing.assert_allclose(out[0, h], vv[5, h // 2], atol=1e-12)


def pin_gqa_mapping(o):
    """Query head h reads KV head h // G: make each KV head's values a constant."""
    D, L = 8, 20
    K = f16(np.zeros((L, 3, D)))
    V = f16(np.stack([np.full((L, D), c) for c in (1.0, 2.0, 3.0)], axis=1))
    q = f16(np.ones((1, 6, D)))
    out = _run_case(o, q, K, V, 0.5, 1, table=(0, 2))
    np.testing.assert_allclose(out[0, :, :], np.repeat([[1.0], [1.0], [2.0], [2.0], [3.0], [3.0]], D, 1),
                               rtol=0, atol=1e-12)


def pin_softmax_rows(o, seed=14):
    rng = np.random.default_rng(seed)
    L, n, D = 45, 4, 16
    K = f16(rng.standard_normal((L, 2, D)))
    V = f16(rng.standard_normal((L, 2, D)))
    q = f16(rng.standard_normal((n, 4, D)))
    kp = place_paged(K, [1, 0, 3], 4)
    vp = place_paged(V, [1, 0, 3], 4)
    _, P = o.paged_attention(q, kp, vp, np.array([[1, 0, 3]]), np.array([L]), np.array([0, n]),
                             0.25, "f16", return_probs=True)
    for (r, h), p in P.items():
        assert p.shape == (L,)
        assert abs(p.sum() - 1.0) < 1e-12
        pos = L - n + r
        assert (p[pos + 1:] == 0).all() and (p[:pos + 1] > 0).all()


def pin_matches_library_sdpa(o, seed=15):
    """Agreement with torch's scaled_dot_product_attention (float64, CPU, GQA)."""
    import torch
    rng = np.random.default_rng(seed)
    H_q, H_kv, D = 6, 2, 32
    seqs = [(1, 1), (23, 1), (40, 5), (70, 70), (53, 17)]
    nb = sum(-(-L // BS) for L, _ in seqs) + 3
    perm = rng.permutation(nb)
    kp = f16(rng.standard_normal((nb, BS, H_kv, D)))
    vp = f16(rng.standard_normal((nb, BS, H_kv, D)))
    tables = np.full((len(seqs), 5), -1, dtype=np.int32)
    cur = 0
    ctxK, ctxV = [], []
    for b, (L, n) in enumerate(seqs):
        k = -(-L // BS)
        tables[b, :k] = perm[cur:cur + k]
        cur += k
        Kc = f16(rng.standard_normal((L, H_kv, D)))
        Vc = f16(rng.standard_normal((L, H_kv, D)))
        kp = place_paged(Kc, list(tables[b, :k]), nb, kp)
        vp = place_paged(Vc, list(tables[b, :k]), nb, vp)
        ctxK.append(Kc)
        ctxV.append(Vc)
    ns = [n for _, n in seqs]
    qsl = np.concatenate([[0], np.cumsum(ns)])
    q = f16(rng.standard_normal((int(qsl[-1]), H_q, D)))
    scale = 1.0 / math.sqrt(D)
    out = o.paged_attention(q, kp, vp, tables, np.array([L for L, _ in seqs]), qsl, scale, "f16")
    qq = torch.from_numpy(q.view(np.float16).astype(np.float64))
    for b, (L, n) in enumerate(seqs):
        Kt = torch.from_numpy(ctxK[b].view(np.float16).astype(np.float64)).permute(1, 0, 2)
        Vt = torch.from_numpy(ctxV[b].view(np.float16).astype(np.float64)).permute(1, 0, 2)
        Qt = qq[qsl[b]:qsl[b + 1]].permute(1, 0, 2)
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            Qt[None], Kt[None], Vt[None], attn_mask=mask, scale=scale, enable_gqa=True)[0]
        np.testing.assert_allclose(out[qsl[b]:qsl[b + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=0, atol=1e-12)


def pin_block_permutation_invariance(o, seed=16):
    from paged_kv_attention_18_gb300 import workloads as W
    wl = W.simple_workload("perm", seed=seed, dtype="bf16", H_q=4, H_kv=2, D=16,
                           seqs=[(50, 1), (33, 4), (90, 20)])
    st = wl.steps[0]
    a = o.paged_attention(st.q, wl.k_pool, wl.v_pool, st.block_tables, st.seq_lens,
                          st.query_start_loc, wl.scale, wl.dtype)
    pi = np.random.default_rng(seed + 1).permutation(wl.num_blocks)
    kp = np.empty_like(wl.k_pool)
    vp = np.empty_like(wl.v_pool)
    kp[pi] = wl.k_pool
    vp[pi] = wl.v_pool
    bt = np.where(st.block_tables >= 0, pi[np.maximum(st.block_tables, 0)], -1)
    b = o.paged_attention(st.q, kp, vp, bt, st.seq_lens, st.query_start_loc, wl.scale, wl.dtype)
    assert np.array_equal(a, b)


def pin_prefix_sharing_invariance(o, seed=17):
    """Two sequences reading one shared copy of a prefix equal reading private copies."""
    rng = np.random.default_rng(seed)
    H_q, H_kv, D, P = 4, 2, 16, 32
    prefix_k = f16(rng.standard_normal((P, H_kv, D)))
    prefix_v = f16(rng.standard_normal((P, H_kv, D)))
    tails = [(f16(rng.standard_normal((t, H_kv, D))), f16(rng.standard_normal((t, H_kv, D))))
             for t in (7, 21)]
    q = f16(rng.standard_normal((2 + 5, H_q, D)))
    lens = np.array([P + 7, P + 21])
    qsl = np.array([0, 2, 7])
    nb = 12
    # shared: both tables start with blocks 9, 4
    shared_tables = [[9, 4, 1], [9, 4, 6, 2]]
    kp = np.zeros((nb, BS, H_kv, D), np.uint16)
    vp = np.zeros_like(kp)
    for (tk, tv), tab in zip(tails, shared_tables):
        kp = place_paged(np.concatenate([prefix_k, tk]), tab, nb, kp)
        vp = place_paged(np.concatenate([prefix_v, tv]), tab, nb, vp)
    bt = np.array([tab + [-1] * (4 - len(tab)) for tab in shared_tables], dtype=np.int32)
    a = o.paged_attention(q, kp, vp, bt, lens, qsl, 0.25, "f16")
    # private copies of the prefix
    priv_tables = [[0, 3, 1], [5, 7, 6, 2]]
    kp2 = np.zeros_like(kp)
    vp2 = np.zeros_like(kp)
    for (tk, tv), tab in zip(tails, priv_tables):
        kp2 = place_paged(np.concatenate([prefix_k, tk]), tab, nb, kp2)
        vp2 = place_paged(np.concatenate([prefix_v, tv]), tab, nb, vp2)
    bt2 = np.array([tab + [-1] * (4 - len(tab)) for tab in priv_tables], dtype=np.int32)
    b = o.paged_attention(q, kp2, vp2, bt2, lens, qsl, 0.25, "f16")
    assert np.array_equal(a, b)


def pin_ragged_equals_per_sequence(o, seed=18):
    from paged_kv_attention_18_gb300 import workloads as W
    wl = W.simple_workload("rag", seed=seed, dtype="f16", H_q=6, H_kv=2, D=16,
                           seqs=[(17, 1), (0, 0), (64, 5), (31, 31), (5, 2)])
    st = wl.steps[0]
    full = o.paged_attention(st.q, wl.k_pool, wl.v_pool, st.block_tables, st.seq_lens,
                             st.query_start_loc, wl.scale, wl.dtype)
    for b in range(st.B):
        s, e = st.query_start_loc[b], st.query_start_loc[b + 1]
        one = o.paged_attention(st.q[s:e], wl.k_pool, wl.v_pool, st.block_tables[b:b + 1],
                                st.seq_lens[b:b + 1], np.array([0, e - s]), wl.scale, wl.dtype)
        assert np.array_equal(one, full[s:e])


def pin_fp32_close_to_fp64(o, seed=19):
    from paged_kv_attention_18_gb300 import workloads as W
    wl = W.simple_workload("acc", seed=seed, dtype="bf16", H_q=12, H_kv=2, D=128,
                           seqs=[(600, 1), (300, 5), (129, 40)])
    st = wl.steps[0]
    args = (st.q, wl.k_pool, wl.v_pool, st.block_tables, st.seq_lens, st.query_start_loc,
            wl.scale, wl.dtype)
    a = o.paged_attention(*args, acc=np.float64)
    b = o.paged_attention(*args, acc=np.float32)
    assert np.abs(a - b).max() < 1e-5


# --------------------------------------------------------------------------- #
# block copies: copy-on-write and swap (contexts read through tables are unchanged)
# --------------------------------------------------------------------------- #
def pin_copy_on_write_keeps_contexts(o, seed=20):
    """tinyserve's figure: seq A [7, 2] and seq B [7, 5] share block 7. Copying block 7
    to a free block and pointing B's table at the copy must leave every sequence's
    context, read through its table, exactly as it was, and change no other block."""
    rng = np.random.default_rng(seed)
    nb, H, D = 10, 2, 4
    pool = f16(rng.standard_normal((nb, BS, H, D)))
    tables = {"A": [7, 2], "B": [7, 5]}
    before = {n: o.gather_context(pool, np.array(t), 2 * BS) for n, t in tables.items()}
    free = 9
    after_pool = o.copy_blocks(pool, pool, [7], [free])
    new_tables = {"A": [7, 2], "B": [free, 5]}
    for n, t in new_tables.items():
        assert np.array_equal(o.gather_context(after_pool, np.array(t), 2 * BS), before[n]), n
    others = [b for b in range(nb) if b != free]
    assert np.array_equal(after_pool[others], pool[others])
    # several pairs at once, one of them reading block 0, read the pool before the call
    pairs_src, pairs_dst = [0, 3, 7], [8, 9, 1]
    out = o.copy_blocks(pool, pool, pairs_src, pairs_dst)
    for s_, d_ in zip(pairs_src, pairs_dst):
        assert np.array_equal(out[d_], pool[s_])
    keep = [b for b in range(nb) if b not in pairs_dst]
    assert np.array_equal(out[keep], pool[keep])


def pin_swap_round_trip(o, seed=21):
    """A sequence's blocks swapped out to a host pool and back into other blocks: its
    context through the remapped table is bit-identical (the pages: swapped KV is
    lossless), and host blocks outside the swap keep their contents."""
    rng = np.random.default_rng(seed)
    H, D, L = 2, 8, 70
    ctx = f16(rng.standard_normal((L, H, D)))
    table = [4, 0, 11, 6, 2]
    dev = place_paged(ctx, table, 12, f16(rng.standard_normal((12, BS, H, D))))
    sentinel = np.full((6, BS, H, D), 0x7BFF, dtype=np.uint16)
    host_ids = [3, 0, 5, 1, 4]
    host = o.copy_blocks(dev, sentinel, table, host_ids)
    assert np.array_equal(host[2], sentinel[2])  # not part of the swap
    back_ids = [1, 7, 3, 9, 10]
    dev2 = o.copy_blocks(host, np.zeros_like(dev), host_ids, back_ids)
    assert np.array_equal(o.gather_context(dev2, np.array(back_ids), L), ctx)
    # a pair with an id outside its pool is skipped
    out = o.copy_blocks(dev, sentinel, [12, 0], [0, 6])
    assert np.array_equal(out, sentinel)


# --------------------------------------------------------------------------- #
# rotary embedding: identity at position 0, rotation (norm), relative positions, hand
# cases with the frequencies written out
# --------------------------------------------------------------------------- #
def _bf16_bits(x):
    from paged_kv_attention_18_gb300 import workloads as W
    return W.round_to_bits(np.asarray(x, np.float32), "bf16")


def pin_rope_identity_and_norm(o, seed=22):
    rng = np.random.default_rng(seed)
    x = _bf16_bits(rng.standard_normal((5, 3, 16)))
    xv = o.decode_bits(x, "bf16")
    r0 = o.rope(x, np.zeros(5, np.int32), 1e4, "bf16")
    assert np.array_equal(r0, xv)  # cos 0 = 1, sin 0 = 0
    r = o.rope(x, np.array([1, 7, 100, 4095, 32767]), 1e6, "bf16")
    assert np.allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(xv, axis=-1), rtol=1e-12)


def pin_rope_relative_position(o, seed=23):
    """<rope(q, m), rope(k, n)> depends on m - n only: RoPE's defining property."""
    rng = np.random.default_rng(seed)
    q = _bf16_bits(rng.standard_normal((1, 1, 32)))
    k = _bf16_bits(rng.standard_normal((1, 1, 32)))
    for m, n, shift in ((5, 2, 11), (40, 39, 1000), (3, 17, 250)):
        d0 = float(np.sum(o.rope(q, [m], 1e4, "bf16") * o.rope(k, [n], 1e4, "bf16")))
        d1 = float(np.sum(o.rope(q, [m + shift], 1e4, "bf16") * o.rope(k, [n + shift], 1e4, "bf16")))
        assert abs(d0 - d1) < 1e-9, (m, n, shift, d0, d1)


def pin_rope_hand_cases(o):
    """D = 4, theta = 10^4: frequencies 1 and 10^-2; element i pairs with i + 2."""
    e0 = _bf16_bits([[[1, 0, 0, 0]]])
    e1 = _bf16_bits([[[0, 1, 0, 0]]])
    r0 = o.rope(e0, [3], 1e4, "bf16")[0, 0]
    r1 = o.rope(e1, [3], 1e4, "bf16")[0, 0]
    assert np.allclose(r0, [math.cos(3), 0, math.sin(3), 0], atol=1e-15)
    assert np.allclose(r1, [0, math.cos(0.03), 0, math.sin(0.03)], atol=1e-15)
    e2 = _bf16_bits([[[0, 0, 1, 0]]])  # the second half rotates the other way round
    r2 = o.rope(e2, [3], 1e4, "bf16")[0, 0]
    assert np.allclose(r2, [-math.sin(3), 0, math.cos(3), 0], atol=1e-15)


ALL_PINS = [
    pin_slots_golden, pin_slots_brute_force, pin_scatter_roundtrip, pin_golden_tiny,
    pin_closed_forms, pin_gqa_mapping, pin_softmax_rows, pin_matches_library_sdpa,
    pin_block_permutation_invariance, pin_prefix_sharing_invariance,
    pin_ragged_equals_per_sequence, pin_fp32_close_to_fp64,
    pin_copy_on_write_keeps_contexts, pin_swap_round_trip,
    pin_rope_identity_and_norm, pin_rope_relative_position, pin_rope_hand_cases,
]
