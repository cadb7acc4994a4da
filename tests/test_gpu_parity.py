"""CUDA path vs the CPU oracle, element by element, through the C ABI.

Slot mapping and the pools after the KV scatter must be bit-exact; attention outputs
must agree within max-abs 2e-3 (fp16) / 1e-2 (bf16) of the fp32 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_18_gb300 import binding
from paged_kv_attention_18_gb300 import workloads as W
from tests.gpu_util import TOL, DevicePools, check_workload, dev, run_step

pytestmark = pytest.mark.gpu


def _sample_rows(st, n_seqs, rng, extra_rows=0):
    """All rows of a random subset of sequences (plus some random rows)."""
    qsl = st.query_start_loc
    seqs = rng.choice(st.B, size=min(n_seqs, st.B), replace=False)
    rows = [r for b in seqs for r in range(qsl[b], qsl[b + 1])]
    if extra_rows and st.T:
        rows += rng.choice(st.T, size=min(extra_rows, st.T), replace=False).tolist()
    return sorted(set(int(r) for r in rows))


# ------------------------------------------------------------------------------------
# the five named workloads
# ------------------------------------------------------------------------------------
def test_tiny_decode():
    check_workload(W.tiny_decode())


def test_qwen05b_mixed():
    check_workload(W.qwen05b_mixed())


def test_qwen05b_mixed_separate_calls():
    check_workload(W.qwen05b_mixed(), separate_calls=True)


def test_qwen15b_decode_full_size():
    wl = W.qwen15b_decode()
    rng = np.random.default_rng(100)
    check_workload(wl, rows_for_step=lambda i, st: _sample_rows(st, 48, rng))


def test_prefix_chunked_prefill_all_steps():
    wl = W.prefix_chunked_prefill()
    assert len(wl.steps) >= 3
    rng = np.random.default_rng(101)

    def rows(i, st):
        qsl = st.query_start_loc
        r = list(range(32))  # every decode row
        for b in range(32, st.B):  # first and last row of every prefill chunk
            r += [int(qsl[b]), int(qsl[b + 1]) - 1]
        r += rng.choice(st.T, size=200, replace=False).tolist()
        return sorted(set(r))

    check_workload(wl, rows_for_step=rows)


def test_spec_verify_long_full_size():
    wl = W.spec_verify_long()
    st = wl.steps[0]
    rng = np.random.default_rng(102)
    long_rows = list(range(int(st.query_start_loc[-5]), st.T))  # the four 32k sequences
    check_workload(wl, rows_for_step=lambda i, s: sorted(set(_sample_rows(s, 24, rng) +
                                                             long_rows)))


def test_long_prefill_sampled():
    # 16384 tokens in one step: the planner at its CTA cap, the scatter CTAs looping over
    # more tokens than they have warps (every pool row is still compared exactly)
    wl = W.long_prefill()
    st = wl.steps[0]
    assert st.T == 16384
    rng = np.random.default_rng(103)
    qsl = st.query_start_loc
    rows = [int(qsl[b]) for b in range(st.B)] + [int(qsl[b + 1]) - 1 for b in range(st.B)]
    rows = sorted(set(rows + rng.choice(st.T, size=60, replace=False).tolist()))
    check_workload(wl, rows_for_step=lambda i, s_: rows)


# ------------------------------------------------------------------------------------
# randomized small shapes: several tiles, splits and ragged tails, compared in full
# ------------------------------------------------------------------------------------
SWEEP = [
    ("f16", 64, 4, 2), ("bf16", 64, 14, 2), ("f16", 128, 12, 2), ("bf16", 128, 12, 2),
    ("bf16", 128, 8, 8), ("f16", 64, 16, 1), ("bf16", 128, 32, 4), ("f16", 128, 6, 3),
    ("bf16", 128, 32, 1),  # 32 query heads per KV head: every row on the split kernel
]


@pytest.mark.parametrize("dtype,D,H_q,H_kv", SWEEP)
@pytest.mark.parametrize("seed", [0, 1])
def test_random_mix(dtype, D, H_q, H_kv, seed):
    rng = np.random.default_rng(1000 + seed * 31 + D + H_q)
    seqs = []
    for _ in range(int(rng.integers(3, 9))):
        kind = rng.integers(0, 4)
        L = int(rng.integers(1, 1200))
        n = {0: 1, 1: min(L, int(rng.integers(2, 9))), 2: min(L, int(rng.integers(1, 300))),
             3: 0}[int(kind)]
        seqs.append((L, n))
    seqs.append((int(rng.integers(2000, 5000)), 1))  # a long decode that splits
    wl = W.simple_workload("mix", seed=seed, dtype=dtype, H_q=H_q, H_kv=H_kv, D=D, seqs=seqs)
    check_workload(wl)


def test_verify_rows_many_splits():
    seqs = [(int(L), 5) for L in np.random.default_rng(5).integers(1024, 8192, size=20)]
    seqs += [(32768, 5)]
    wl = W.simple_workload("verify", seed=5, dtype="bf16", H_q=12, H_kv=2, D=128, seqs=seqs)
    check_workload(wl)


def test_batch_larger_than_planner_staging():
    # more than 4096 sequences: the planner keeps its per-sequence offsets in global memory
    # (one CTA); a few long decodes split, so the combine's token list is exercised too
    rng = np.random.default_rng(41)
    seqs = [(int(L), 1) for L in rng.integers(1, 48, size=5000)]
    seqs += [(int(L), int(n)) for L, n in zip(rng.integers(3000, 6000, size=6),
                                              rng.integers(1, 4, size=6))]
    # three prefill chunks: tile items planned without the staged rank tables
    seqs += [(300, 40), (900, 100), (2000, 250)]
    wl = W.simple_workload("wide", seed=41, dtype="bf16", H_q=12, H_kv=2, D=128, seqs=seqs)
    rng_rows = np.random.default_rng(42)

    def rows(i, st):
        qsl = st.query_start_loc
        r = list(range(int(qsl[-10]), st.T))  # every row of the long sequences and chunks
        return sorted(set(r + _sample_rows(st, 200, rng_rows)))

    check_workload(wl, rows_for_step=rows)


def test_many_prefill_chunks():
    # more than 512 prefill chunks of different lengths: the tile items of the ranks past
    # the shortest chunk's are placed sequence by sequence instead of rank by rank
    rng = np.random.default_rng(61)
    seqs = [(int(L), int(n)) for L, n in zip(rng.integers(120, 400, size=600),
                                             rng.integers(11, 60, size=600))]
    seqs += [(int(L), 1) for L in rng.integers(500, 3000, size=20)]  # decodes among them
    wl = W.simple_workload("chunks", seed=61, dtype="f16", H_q=12, H_kv=2, D=64, seqs=seqs)
    rr = np.random.default_rng(62)
    check_workload(wl, rows_for_step=lambda i, st: _sample_rows(st, 80, rr, extra_rows=300))


def test_planner_grid_sizes():
    # batches that give the planner different grid sizes (a CTA per 8 sequences and per 1024
    # tokens, at most 64), with split decodes and a prefill chunk
    for B, seed in ((31, 51), (33, 52), (1025, 53)):
        rng = np.random.default_rng(seed)
        seqs = [(int(L), 1) for L in rng.integers(200, 2500, size=B)]
        seqs[0] = (seqs[0][0], min(seqs[0][0], 700))  # one prefill chunk among them
        wl = W.simple_workload(f"grid{B}", seed=seed, dtype="f16", H_q=8, H_kv=2, D=64,
                               seqs=seqs)
        rr = np.random.default_rng(seed + 100)
        check_workload(wl, rows_for_step=lambda i, st: _sample_rows(st, 64, rr, extra_rows=200))


# ------------------------------------------------------------------------------------
# edge cases
# ------------------------------------------------------------------------------------
def test_context_of_one_gives_v():
    wl = W.simple_workload("one", seed=3, dtype="bf16", H_q=12, H_kv=2, D=128,
                           seqs=[(1, 1), (1, 1), (17, 1)])
    pools = DevicePools(wl)
    st = wl.steps[0]
    out, _ = run_step(wl, st, pools)
    got = out.cpu()
    v = dev(st.v, "bf16").cpu()
    for t in range(2):
        for h in range(12):
            assert torch.equal(got[t, h], v[t, h // 6])  # softmax of one key is exactly 1


def test_empty_and_zero_query_batches():
    wl = W.simple_workload("z", seed=4, dtype="f16", H_q=4, H_kv=2, D=64,
                           seqs=[(10, 0), (33, 0)])
    pools = DevicePools(wl)
    st = wl.steps[0]
    assert st.T == 0
    out, slots = run_step(wl, st, pools)
    assert out.shape == (0, 4, 64) and slots.numel() == 0
    assert binding.device_error() == 0
    # zero-query sequences between real ones
    check_workload(W.simple_workload("z2", seed=4, dtype="f16", H_q=4, H_kv=2, D=64,
                                     seqs=[(10, 0), (50, 3), (0, 0), (20, 1), (7, 0)]))


def test_full_block_table_and_block_boundaries():
    # contexts ending exactly on, just before and just after block boundaries; the
    # longest uses every entry of its block table
    seqs = [(16, 1), (15, 1), (17, 1), (32, 16), (48, 17), (64, 64), (1, 1), (160, 2)]
    check_workload(W.simple_workload("edge", seed=9, dtype="bf16", H_q=12, H_kv=2, D=128,
                                     seqs=seqs, free_fraction=0.0))


def test_negative_slots_are_skipped():
    wl = W.simple_workload("neg", seed=11, dtype="f16", H_q=4, H_kv=2, D=64,
                           seqs=[(30, 3), (9, 1)])
    st = wl.steps[0]
    pools = DevicePools(wl)
    slots = torch.tensor([-1, 5, -1, -7], dtype=torch.int32, device="cuda")
    binding.reshape_and_cache(dev(st.k, "f16"), dev(st.v, "f16"), slots, pools.k, pools.v)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    kref, _ = oracle.reshape_and_cache(st.k, st.v, slots.cpu().numpy(), wl.k_pool, wl.v_pool)
    from tests.gpu_util import host_bits
    assert np.array_equal(host_bits(pools.k), kref)


def test_minimum_workspace_means_no_splits():
    wl = W.simple_workload("ws", seed=12, dtype="bf16", H_q=12, H_kv=2, D=128,
                           seqs=[(3000, 1), (2500, 5), (900, 1)])
    st = wl.steps[0]
    n = binding.workspace_size(st.T, st.B, 12, 2, 128, 0)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    check_workload(wl, workspace=ws)


def test_bad_block_id_sets_device_error_without_fault():
    wl = W.simple_workload("bad", seed=13, dtype="bf16", H_q=12, H_kv=2, D=128,
                           seqs=[(40, 1), (40, 1)])
    st = wl.steps[0]
    bt = st.block_tables.copy()
    bt[1, 1] = wl.num_blocks + 5  # out of the pool: checked on the device, never read
    pools = DevicePools(wl)
    q = dev(st.q, "bf16")
    out = binding.paged_attention(q, pools.k, pools.v, dev(bt), dev(st.seq_lens),
                                  dev(st.query_start_loc), wl.scale)
    torch.cuda.synchronize()
    assert binding.device_error() == 1
    assert binding.device_error() == 0  # reading clears it
    ref = oracle.paged_attention(st.q, wl.k_pool, wl.v_pool, st.block_tables, st.seq_lens,
                                 st.query_start_loc, wl.scale, "bf16", acc=np.float32)
    assert np.abs(out.float().cpu().numpy()[0] - ref[0]).max() <= TOL["bf16"]


def test_two_calls_share_a_workspace():
    wl = W.qwen05b_mixed()
    st = wl.steps[0]
    pools = DevicePools(wl)
    ws = binding.alloc_workspace(st.T, st.B, wl.H_q, wl.H_kv, wl.D, 1024)
    a, _ = run_step(wl, st, pools, workspace=ws)
    b = binding.paged_attention(dev(st.q, "f16"), pools.k, pools.v, dev(st.block_tables),
                                dev(st.seq_lens), dev(st.query_start_loc), wl.scale,
                                workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)  # deterministic: same plan, same order of accumulation


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_large_score_jumps_mid_context(dtype):
    # Keys of a few pool blocks are scaled up so the running max jumps by far more than
    # 2^8 (and often 2^64) in the middle of KV tiles: every rescale path of the kernels
    # must keep the result equal to the plain softmax.
    #
    # Such rows are sharply peaked: the output is a mix of one or two V rows. The kernels
    # multiply V by probabilities rounded to the 16-bit input type (the tensor core takes
    # both operands in one type), 2^-9 relative in bf16, and the reference is scaled
    # lazily, so even the largest weight carries that rounding. A near-even mix of two V
    # rows that lie d apart then moves by up to about d * 2^-10, and the output's own
    # rounding adds half an ulp (2^-8 for |o| in [2, 4)). With N(0, 1) values in bf16 the
    # two together can pass 1e-2 (0.0117 measured, equal bit for bit to a CPU model of
    # the kernel's steps), so the bf16 case draws V at 0.35 times that scale: outputs stay
    # below 2, where the plain bound holds, while the keys jump just as far. The f16 case
    # keeps N(0, 1) values (rounding 2^-11: within 2e-3 at |o| < 2, half an output ulp
    # more above).
    seqs = [(700, 300), (900, 5), (1500, 1), (400, 128), (2100, 40)]
    wl = W.simple_workload("jumps", seed=31, dtype=dtype, H_q=12, H_kv=2, D=128, seqs=seqs)
    vals = oracle.decode_bits(wl.k_pool, dtype)
    rng = np.random.default_rng(32)
    hot = rng.choice(wl.num_blocks, size=wl.num_blocks // 6, replace=False)
    vals[hot] *= 40.0
    wl.k_pool = W.round_to_bits(vals.astype(np.float32), dtype)
    if dtype == "bf16":
        wl.v_pool = W.round_to_bits((0.35 * oracle.decode_bits(wl.v_pool, dtype)).astype(np.float32),
                                    dtype)
        st = wl.steps[0]
        st.v = W.round_to_bits((0.35 * oracle.decode_bits(st.v, dtype)).astype(np.float32), dtype)
    check_workload(wl)


# ------------------------------------------------------------------------------------
# small batches: the whole step in one launch (no plan)
# ------------------------------------------------------------------------------------
SMALL_BATCHES = [
    # (dtype, H_q, H_kv, D, [(context after the step, query tokens), ...])
    ("f16", 4, 2, 64, [(1, 1), (15, 1), (16, 1), (17, 1), (100, 1), (31, 0), (64, 1)]),
    ("bf16", 8, 2, 128, [(40, 4), (0, 0), (16, 0)]),          # one 16-row group, G = 4
    ("bf16", 12, 2, 128, [(90, 2), (7, 0)]),                  # verify-like rows, G = 6
    ("f16", 8, 8, 64, [(1024, 1), (513, 1)]),                 # 64 pages, MHA (G = 1)
    ("bf16", 16, 1, 128, [(33, 1)]),                          # G = 16: one row group
    ("f16", 4, 2, 64, [(17, 2), (33, 2), (2, 2)]),            # two new rows across pages
]


@pytest.mark.parametrize("case", range(len(SMALL_BATCHES)))
@pytest.mark.parametrize("separate", [False, True])
def test_small_batches_in_one_launch(case, separate):
    dt, H_q, H_kv, D, seqs = SMALL_BATCHES[case]
    wl = W.simple_workload(f"small{case}", seed=40 + case, dtype=dt, H_q=H_q, H_kv=H_kv, D=D,
                           seqs=seqs)
    assert wl.steps[0].T * (H_q // H_kv) <= 16
    check_workload(wl, separate_calls=separate)


def test_small_batch_skips_the_plan():
    small = W.simple_workload("one_launch", seed=50, dtype="f16", H_q=4, H_kv=2, D=64,
                              seqs=[(30, 1), (70, 1), (5, 1)])
    large = W.simple_workload("planned", seed=51, dtype="f16", H_q=4, H_kv=2, D=64,
                              seqs=[(30, 1)] * 9)  # 9 tokens x G = 2: 18 rows
    launches = {}
    for wl in (small, large):
        pools = DevicePools(wl)
        binding.profile_begin(8)
        run_step(wl, wl.steps[0], pools)
        prof = binding.profile_end()
        launches[wl.name] = {k: n for k, (_, n) in prof.items()}
    assert launches["one_launch"]["plan"] == 0 and launches["one_launch"]["split_attention"] == 1
    assert launches["one_launch"]["reshape_and_cache"] == 0
    assert launches["planned"]["plan"] == 1
    check_workload(small)


# Batches for the tile kernel's direct mode: query tiles, at most 32 sequences, few enough
# that each could have its own tile items, no block table wider than 64 pages
DIRECT_TILE_BATCHES = [
    ("f16", 14, 2, 64, [(97, 1), (520, 1), (256, 256), (768, 256)]),   # decodes + chunks
    ("bf16", 12, 2, 128, [(1024, 1024)]),                                # a whole prompt
    ("bf16", 8, 8, 128, [(300, 150), (0, 0), (129, 129)]),               # G = 1, an empty one
    ("f16", 16, 1, 64, [(40, 9), (17, 17), (1000, 33)]),                 # G = 16: 8-token tiles
    ("bf16", 12, 2, 128, [(64 + 5 * i, 3 + i % 4) for i in range(32)]),  # 32 sequences
]


@pytest.mark.parametrize("case", range(len(DIRECT_TILE_BATCHES)))
@pytest.mark.parametrize("separate", [False, True])
def test_direct_tile_batches(case, separate):
    dt, H_q, H_kv, D, seqs = DIRECT_TILE_BATCHES[case]
    wl = W.simple_workload(f"dtile{case}", seed=70 + case, dtype=dt, H_q=H_q, H_kv=H_kv, D=D,
                           seqs=seqs)
    pools = DevicePools(wl)
    binding.profile_begin(8)
    run_step(wl, wl.steps[0], pools, separate_calls=separate)
    prof = binding.profile_end()
    # the tile kernel alone: no plan, no split kernel, nothing to combine
    assert prof["tile_attention"][1] == 1
    assert prof["plan"][1] == 0 and prof["split_attention"][1] == 0 and prof["combine"][1] == 0
    check_workload(wl, separate_calls=separate)


@pytest.mark.parametrize("separate", [False, True])
def test_split_rows_of_both_kernels_combined(separate):
    # 38 long decodes (the split kernel splits them) beside two short chunks of long
    # contexts (too few tile items: the planner splits those too); one combine after the
    # tile kernel merges the partials of both kernels' rows
    seqs = [(1000 + (53 * i) % 2000, 1) for i in range(38)] + [(3000, 64), (2500, 100)]
    wl = W.simple_workload("both_split", seed=90, dtype="bf16", H_q=12, H_kv=2, D=128,
                           seqs=seqs)
    pools = DevicePools(wl)
    binding.profile_begin(8)
    run_step(wl, wl.steps[0], pools, separate_calls=separate)
    prof = binding.profile_end()
    assert prof["split_attention"][1] == 1 and prof["tile_attention"][1] == 1
    assert prof["combine"][1] == 1
    check_workload(wl, separate_calls=separate)


def test_direct_tile_bad_sequence_sets_device_error():
    wl = W.simple_workload("dtile_bad", seed=80, dtype="bf16", H_q=12, H_kv=2, D=128,
                           seqs=[(200, 100), (300, 40)])
    st = wl.steps[0]
    sl = st.seq_lens.copy()
    sl[1] = 30  # 40 query tokens over a 30-token context: the sequence is skipped
    pools = DevicePools(wl)
    out = binding.paged_attention(dev(st.q, "bf16"), pools.k, pools.v, dev(st.block_tables),
                                  dev(sl), dev(st.query_start_loc), wl.scale)
    torch.cuda.synchronize()
    assert binding.device_error() == 3
    ref = oracle.paged_attention(st.q, wl.k_pool, wl.v_pool, st.block_tables, st.seq_lens,
                                 st.query_start_loc, wl.scale, "bf16", acc=np.float32)
    assert np.abs(out.float().cpu().numpy()[:100] - ref[:100]).max() <= TOL["bf16"]


def test_long_sequence_among_empty_ones_takes_the_split_kernel():
    # T = B: with a token in every sequence no sequence could reach a query tile, so the
    # tile kernel is not launched; here one sequence holds all 12 tokens (72 rows at G = 6)
    # and the others none, and the split kernel takes its rows
    seqs = [(0, 0)] * 5 + [(300, 12)] + [(40, 0)] * 6
    wl = W.simple_workload("one_long", seed=60, dtype="bf16", H_q=12, H_kv=2, D=128, seqs=seqs)
    st = wl.steps[0]
    assert st.T == st.B == 12
    pools = DevicePools(wl)
    binding.profile_begin(8)
    run_step(wl, st, pools)
    prof = binding.profile_end()
    assert prof["tile_attention"][1] == 0 and prof["split_attention"][1] == 1
    check_workload(wl)


def test_decode_batch_launches_no_tile_kernel():
    wl = W.simple_workload("decodes", seed=61, dtype="bf16", H_q=12, H_kv=2, D=128,
                           seqs=[(200 + 37 * i, 1) for i in range(40)])
    pools = DevicePools(wl)
    binding.profile_begin(8)
    run_step(wl, wl.steps[0], pools)
    prof = binding.profile_end()
    assert prof["tile_attention"][1] == 0 and prof["plan"][1] == 1
    check_workload(wl)


def test_output_aligned_to_16_bytes_only():
    # the tile kernel writes 32-byte pieces of each row when the output allows it, and
    # 16-byte pieces otherwise: both give the same bits
    wl = W.simple_workload("align", seed=70, dtype="bf16", H_q=12, H_kv=2, D=128,
                           seqs=[(400, 300), (90, 64), (700, 1)])
    st = wl.steps[0]
    pools = DevicePools(wl)
    q = dev(st.q, "bf16")
    bt, sl, qs = dev(st.block_tables), dev(st.seq_lens), dev(st.query_start_loc)
    ref = binding.paged_attention(q, pools.k, pools.v, bt, sl, qs, wl.scale)
    buf = torch.empty(q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(q.shape)  # 16 bytes past a 256-byte boundary
    assert out.data_ptr() % 32 == 16
    binding.paged_attention(q, pools.k, pools.v, bt, sl, qs, wl.scale, out=out)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
