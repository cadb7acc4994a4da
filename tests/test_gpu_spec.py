"""Speculative acceptance through the C ABI vs the CPU oracle: the accepted-draft counts
and every emitted token must be identical (the decisions are fixed to a precision)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import spec_oracle
from paged_kv_attention_18_gb300 import binding

pytestmark = pytest.mark.gpu
U32 = 2 ** 32


def _softmax(x):
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def make_case(B, k, V, seed, near=0.7, peak=2.0):
    """Target rows p, draft rows q near p, drafts drawn from q, random words."""
    rng = np.random.default_rng(seed)
    lt = rng.standard_normal((B, k + 1, V)).astype(np.float32) * peak
    p = _softmax(lt)
    q = _softmax(lt[:, :k] * near + rng.standard_normal((B, k, V)).astype(np.float32))
    cq = np.cumsum(q.astype(np.float64), axis=-1)
    u = rng.random((B, k, 1))
    drafts = np.minimum((cq <= u).sum(axis=-1), V - 1).astype(np.int32)
    rnd = rng.integers(0, U32, size=(B, k + 1), dtype=np.uint64).astype(np.uint32)
    return p, q, drafts, rnd


def run(p, drafts, rnd, q=None, greedy=False):
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    r = None if rnd is None else dev(rnd.view(np.int32))
    out, num = binding.spec_accept(dev(p), dev(drafts), r, None if q is None else dev(q),
                                   greedy=greedy)
    torch.cuda.synchronize()
    return out.cpu().numpy(), num.cpu().numpy()


# (512, 2, 200): two 128-token runs per row, so one CTA's share of runs spans many
# sequences and its warps decide many acceptances
@pytest.mark.parametrize("B,k,V", [(64, 4, 1000), (37, 3, 3001), (20, 4, 8197), (9, 1, 50000),
                                   (512, 2, 200)])
@pytest.mark.parametrize("mode", ["draft_model", "ngram", "greedy"])
def test_matches_oracle(B, k, V, mode):
    p, q, drafts, rnd = make_case(B, k, V, seed=B + k + V, peak=6.0 if mode == "ngram" else 2.0)
    if mode == "ngram":
        # a deterministic proposer: half of the drafts on the target's most likely token
        am = p.argmax(axis=-1)[:, :k]
        pick = np.random.default_rng(V).random((B, k)) < 0.5
        drafts = np.where(pick, am, drafts).astype(np.int32)
    if mode == "greedy":
        # plant argmax-equal drafts for part of the batch so acceptance runs vary
        am = p.argmax(axis=-1)[:, :k]
        drafts = np.where(np.arange(B)[:, None] % 3 == 0, am, drafts).astype(np.int32)
        got = run(p, drafts, None, greedy=True)
        ref = oracle.spec_accept(p, drafts, greedy=True)
    else:
        qq = q if mode == "draft_model" else None
        got = run(p, drafts, rnd, qq)
        ref = oracle.spec_accept(p, drafts, rnd, qq)
    assert binding.device_error() == 0
    np.testing.assert_array_equal(got[1], ref[1])
    np.testing.assert_array_equal(got[0], ref[0])
    if mode != "greedy":
        assert 0 < ref[1].mean() < k  # both accepting and rejecting paths ran


def test_modes_in_turn_share_one_workspace():
    # greedy, draft-model and one-hot calls in turn through one workspace: each call writes
    # every entry it later reads, so no mode sees another's stale sums or maxima
    B, k, V = 40, 3, 20000
    p, q, drafts, rnd = make_case(B, k, V, seed=321)
    am = p.argmax(axis=-1)[:, :k]
    gd = np.where(np.arange(B)[:, None] % 2 == 0, am, drafts).astype(np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    ws = torch.empty(max(int(binding.lib().ps_spec_accept_workspace_size(B, k, V)), 256),
                     dtype=torch.uint8, device="cuda")
    pd, qd, rd = dev(p), dev(q), dev(rnd.view(np.int32))
    cases = [
        (lambda: binding.spec_accept(pd, dev(gd), None, None, greedy=True, workspace=ws),
         oracle.spec_accept(p, gd, greedy=True)),
        (lambda: binding.spec_accept(pd, dev(drafts), rd, qd, workspace=ws),
         oracle.spec_accept(p, drafts, rnd, q)),
        (lambda: binding.spec_accept(pd, dev(drafts), rd, None, workspace=ws),
         oracle.spec_accept(p, drafts, rnd, None)),
    ]
    for _ in range(2):
        for call, ref in cases:
            out, num = call()
            torch.cuda.synchronize()
            assert binding.device_error() == 0
            np.testing.assert_array_equal(num.cpu().numpy(), ref[1])
            np.testing.assert_array_equal(out.cpu().numpy(), ref[0])


def test_full_vocabulary_batch():
    # 132 sequences x (4 drafts + bonus) over a 151936-token vocabulary
    B, k, V = 132, 4, 151936
    p, q, drafts, rnd = make_case(B, k, V, seed=5, near=0.9)
    got = run(p, drafts, rnd, q)
    ref = oracle.spec_accept(p, drafts, rnd, q)
    assert binding.device_error() == 0
    np.testing.assert_array_equal(got[1], ref[1])
    np.testing.assert_array_equal(got[0], ref[0])
    # greedy over the same rows, a third of the drafts on the target's argmax
    am = p.argmax(axis=-1)[:, :k]
    gd = np.where(np.arange(B)[:, None] % 3 == 0, am, drafts).astype(np.int32)
    got = run(p, gd, None, greedy=True)
    ref = oracle.spec_accept(p, gd, greedy=True)
    assert binding.device_error() == 0
    np.testing.assert_array_equal(got[1], ref[1])
    np.testing.assert_array_equal(got[0], ref[0])


@pytest.mark.parametrize("V", [4096, 3001])
@pytest.mark.parametrize("mode", ["draft_model", "ngram", "bonus"])
def test_draw_on_exact_boundaries(V, mode):
    """The fixed-point sums are exact. Residual mass below 2^-8 gives Z < 2^32, so the final
    word can put the target on any integer. Targets at C_v - 1 and at C_v (C the oracle's
    running sums) must pick token v and the next weighted token. An error of one unit in
    any weight before v would change the token. V = 4096 takes 16-byte rows, V = 3001
    4-byte ones."""
    B, k = 16, 2
    rng = np.random.default_rng(V + 7 * len(mode))
    p = _softmax(rng.standard_normal((B, k + 1, V)).astype(np.float32))
    drafts = rng.integers(0, V, (B, k)).astype(np.int32)
    rnd = np.zeros((B, k + 1), np.uint64)
    q = None
    if mode == "draft_model":
        # q a hair below p: residual mass about 2^-11; draft 0 rejected (q above p there)
        q = (p[:, :k] * np.float32(1 - 2.0 ** -11)).astype(np.float32)
        for b in range(B):
            q[b, 0, drafts[b, 0]] = p[b, 0, drafts[b, 0]] * np.float32(1.5)
        rnd[:, 0] = U32 - 1
        rows = [np.maximum(p[b, 0] - q[b, 0], np.float32(0)) for b in range(B)]
    elif mode == "ngram":
        # one-hot drafts on rows of mass 2^-10: draft 0 rejected, residual = p but 0 at it
        p = (p * np.float32(2.0 ** -10)).astype(np.float32)
        rnd[:, 0] = U32 - 1
        rows = []
        for b in range(B):
            w = p[b, 0].copy()
            w[drafts[b, 0]] = max(w[drafts[b, 0]] - np.float32(1), np.float32(0))
            rows.append(w)
    else:
        # every draft accepted (R = 0): the bonus draw from p_k, mass 2^-10
        p = (p * np.float32(2.0 ** -10)).astype(np.float32)
        rows = [p[b, k] for b in range(B)]
    expect = np.zeros(B, np.int64)
    for b in range(B):
        W = spec_oracle.weights(rows[b])
        C = np.cumsum(W)
        Z = int(C[-1])
        assert 0 < Z < 2 ** 32
        v = V // 3 + 37 * b
        while W[v] == 0:
            v += 1
        T = int(C[v]) - (1 if b % 2 == 0 else 0)
        R = (T * 2 ** 32 + Z - 1) // Z
        assert R < 2 ** 32 and (R * Z) >> 32 == T
        rnd[b, k] = R
        nxt = v + 1
        while W[nxt] == 0:
            nxt += 1
        expect[b] = v if b % 2 == 0 else nxt
    rnd = rnd.astype(np.uint32)
    got = run(p, drafts, rnd, q)
    ref = oracle.spec_accept(p, drafts, rnd, q)
    assert binding.device_error() == 0
    last = ref[0][np.arange(B), ref[1]]
    np.testing.assert_array_equal(last, expect)  # the case is set up as described
    np.testing.assert_array_equal(got[1], ref[1])
    np.testing.assert_array_equal(got[0], ref[0])


def test_unaligned_rows_take_word_loads():
    # V a multiple of 4 but p and q 4 bytes past a 16-byte boundary: rows read as 4-byte words
    B, k, V = 24, 3, 4096
    p, q, drafts, rnd = make_case(B, k, V, seed=77)
    flat_p = torch.zeros(p.size + 1, dtype=torch.float32, device="cuda")
    flat_q = torch.zeros(q.size + 1, dtype=torch.float32, device="cuda")
    pd = flat_p[1:].view(B, k + 1, V)
    qd = flat_q[1:].view(B, k, V)
    pd.copy_(torch.from_numpy(p))
    qd.copy_(torch.from_numpy(q))
    assert pd.data_ptr() % 16 == 4 and qd.data_ptr() % 16 == 4
    out, num = binding.spec_accept(pd, torch.from_numpy(drafts).cuda(),
                                   torch.from_numpy(rnd.view(np.int32)).cuda(), qd)
    torch.cuda.synchronize()
    ref = oracle.spec_accept(p, drafts, rnd, q)
    assert binding.device_error() == 0
    np.testing.assert_array_equal(num.cpu().numpy(), ref[1])
    np.testing.assert_array_equal(out.cpu().numpy(), ref[0])


def test_edges():
    # k = 0: one draw from p_0
    p, q, drafts, rnd = make_case(16, 0, 777, seed=8)
    got = run(p, np.zeros((16, 0), np.int32), rnd)
    ref = oracle.spec_accept(p, np.zeros((16, 0), np.int32), rnd)
    np.testing.assert_array_equal(got[0], ref[0])
    assert (got[1] == 0).all()
    # an invalid draft id: error code, counted as rejected, replacement drawn from p
    p, q, drafts, rnd = make_case(8, 3, 500, seed=9)
    drafts[3, 1] = 500
    drafts[5, 0] = -2
    rnd[:, :3] = 0  # every valid draft accepted
    got = run(p, drafts, rnd, q)
    assert binding.device_error() == 6  # PS_DEV_BAD_TOKEN
    ref = oracle.spec_accept(p, drafts, rnd, q)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])
    # no residual mass (every positive difference below 2^-40): the draw falls back to p
    V = 64
    p = np.full((4, 2, V), 1.0 / V, np.float32)
    p[:, 0, 5] = 0.0
    q = p[:, :1].copy()
    q[:, 0, 0] += np.float32(2.0 ** -27)   # q(d) > p(d): the draft can be rejected
    p[:, 0, 5] = np.float32(2.0 ** -45)    # the only positive residual, below 2^-40
    drafts = np.zeros((4, 1), np.int32)
    rnd = np.array([[U32 - 1, r] for r in (0, 2 ** 30, 2 ** 31, U32 - 1)], np.uint64).astype(np.uint32)
    got = run(p, drafts, rnd, q)
    ref = oracle.spec_accept(p, drafts, rnd, q)
    assert (ref[1] == 0).all()
    np.testing.assert_array_equal(got[0], ref[0])
