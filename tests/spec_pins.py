"""Checks that pin the speculative-acceptance oracle to facts other than itself: the
statistical law the pages state (the sampler reproduces the target distribution), exact
quadrature over evenly spread random words, and hand-worked greedy and residual cases."""
from __future__ import annotations

import numpy as np

U32 = 2 ** 32


def _probs(rng, shape):
    x = rng.standard_normal(shape).astype(np.float64) * 1.5
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def pin_sampler_reproduces_target_law(s, seed=30):
    """tinyserve ("How it works"; "Correctness & testing" table): verification by
    rejection sampling reproduces sampling from the target distribution. With drafts
    drawn from q and k = 2, the first emitted token follows p_0."""
    rng = np.random.default_rng(seed)
    V, N = 6, 40000
    p0 = _probs(rng, (V,))
    q0 = _probs(rng, (V,))
    p = np.broadcast_to(np.stack([p0, _probs(rng, (V,)), _probs(rng, (V,))]), (N, 3, V)).copy()
    q = np.broadcast_to(np.stack([q0, _probs(rng, (V,))]), (N, 2, V)).copy()
    cq = np.cumsum(q0.astype(np.float64))
    d0 = np.minimum(np.searchsorted(cq, rng.random(N), side="right"), V - 1)
    drafts = np.stack([d0, rng.integers(0, V, N)], axis=1).astype(np.int32)
    rnd = rng.integers(0, U32, size=(N, 3), dtype=np.uint64).astype(np.uint32)
    out, _ = s.spec_accept(p, drafts, rnd, q)
    freq = np.bincount(out[:, 0], minlength=V) / N
    tv = 0.5 * np.abs(freq - p0.astype(np.float64)).sum()
    assert tv < 0.015, (tv, freq, p0)


def pin_acceptance_rate_by_quadrature(s):
    """With R spread evenly over [0, 2^32), a draft with p(d) / q(d) = r is accepted for
    a fraction r of the words (to one word); with one-hot drafts, for a fraction p(d)."""
    N = 4096
    R = (np.arange(N, dtype=np.uint64) * (U32 // N)).astype(np.uint32)
    V = 4
    for pd, qd in ((0.25, 1.0), (0.2, 0.5), (0.9, 0.3)):
        p = np.zeros((N, 2, V), np.float32)
        p[:, :, 0] = pd
        p[:, :, 1] = 1 - pd
        q = np.zeros((N, 1, V), np.float32)
        q[:, 0, 0] = qd
        q[:, 0, 2] = 1 - qd
        drafts = np.zeros((N, 1), np.int32)
        rnd = np.stack([R, R], axis=1)
        _, num = s.spec_accept(p, drafts, rnd, q)
        want = min(1.0, pd / qd) * N
        assert abs(num.sum() - want) <= 1, (pd, qd, num.sum(), want)
        _, num1 = s.spec_accept(p, drafts, rnd, None)  # one-hot drafts: q(d) = 1
        assert abs(num1.sum() - pd * N) <= 1, (pd, num1.sum())


def pin_bonus_draw_by_quadrature(s):
    """All drafts accepted (q = p): the bonus token follows p_k; with R spread evenly the
    histogram is N * p_k to one word per token, and tokens come in increasing order."""
    N, V = 8192, 5
    pk = np.array([0.1, 0.0, 0.45, 0.25, 0.2], np.float32)
    p = np.zeros((N, 2, V), np.float32)
    p[:, 0, 3] = 1.0
    p[:, 1] = pk
    q = p[:, :1].copy()
    drafts = np.full((N, 1), 3, np.int32)
    R = (np.arange(N, dtype=np.uint64) * (U32 // N)).astype(np.uint32)
    out, num = s.spec_accept(p, drafts, np.stack([np.zeros(N, np.uint32), R], axis=1), q)
    assert (num == 1).all() and (out[:, 0] == 3).all()
    hist = np.bincount(out[:, 1], minlength=V)
    assert np.all(np.abs(hist - pk.astype(np.float64) * N) <= 1), hist
    assert np.all(np.diff(out[:, 1]) >= 0)


def pin_residual_hand_case(s):
    """p = [0.5, 0.5], q = [1, 0], draft 0 rejected: max(p - q, 0) = [0, 0.5], so the
    replacement is token 1 whatever the final word."""
    p = np.array([[[0.5, 0.5], [0.3, 0.7]]], np.float32).repeat(16, axis=0)
    q = np.array([[[1.0, 0.0]]], np.float32).repeat(16, axis=0)
    drafts = np.zeros((16, 1), np.int32)
    rnd = np.stack([np.full(16, U32 - 1, np.uint64),
                    np.arange(16, dtype=np.uint64) * (U32 // 16)], axis=1).astype(np.uint32)
    out, num = s.spec_accept(p, drafts, rnd, q)
    assert (num == 0).all() and (out[:, 0] == 1).all() and (out[:, 1] == -1).all()


def pin_greedy_hand_cases(s):
    p = np.zeros((4, 3, 5), np.float32)
    p[:, 0] = [0.1, 0.6, 0.1, 0.1, 0.1]   # argmax 1
    p[:, 1] = [0.3, 0.1, 0.3, 0.2, 0.1]   # tie between 0 and 2: the lowest, 0
    p[:, 2] = [0.0, 0.0, 0.0, 0.0, 1.0]   # argmax 4
    drafts = np.array([[1, 0], [1, 2], [3, 0], [1, 0]], np.int32)
    out, num = s.spec_accept(p, drafts, greedy=True)
    assert num.tolist() == [2, 1, 0, 2]
    assert out[0].tolist() == [1, 0, 4]  # both match, bonus argmax p_2
    assert out[1].tolist() == [1, 0, -1]  # second draft 2 loses the tie to 0
    assert out[2].tolist() == [1, -1, -1]  # first draft wrong: emit argmax p_0


SPEC_PINS = [pin_sampler_reproduces_target_law, pin_acceptance_rate_by_quadrature,
             pin_bonus_draw_by_quadrature, pin_residual_hand_case, pin_greedy_hand_cases]
