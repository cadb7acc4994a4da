"""CPU oracle for speculative-decoding acceptance: TEST INFRASTRUCTURE ONLY.

Only the test-suite, the package smoke check and the benchmark may import this module;
the CUDA library never does, and it imports nothing from the library.

The rule (tinyserve, "How it works", speculative decoding): draft d_i is accepted with
probability min(1, p_i(d_i) / q_i(d_i)); at the first rejection the replacement token is
drawn from normalize(max(p_i - q_i, 0)); if all k drafts survive, a bonus token is drawn
from the last target distribution. Greedy verification (temperature 0) accepts a draft
while it equals argmax p_i (tinyserve, "How it works": bit-identical greedy output).

The randomness is given: one uint32 word R per draft and one for the final draw. The
decisions are taken in the same fixed precision as the library states them:
acceptance is the fp64 comparison R * q < p * 2^32; residual weights are fp32
max(p - q, 0), made exact integers trunc(w * 2^40); the draw is the first token whose
running sum exceeds floor(R * Z / 2^32), Z the total; argmax ties go to the lowest token.
"""
from __future__ import annotations

import numpy as np

FIX = float(2 ** 40)


def accepts(R: int, pv: float, qv: float) -> bool:
    """Acceptance of a draft with target probability pv and draft probability qv, given
    the random word R: u < p / q with u = R / 2^32, as R * q < p * 2^32 (fp64 products)."""
    return float(R) * float(np.float32(qv)) < float(np.float32(pv)) * 4294967296.0


def weights(w: np.ndarray) -> np.ndarray:
    """fp32 weights as exact integers trunc(w * 2^40) (0 where w <= 0)."""
    w = np.asarray(w, dtype=np.float32)
    W = np.floor(w.astype(np.float64) * FIX)
    W[~(w > 0)] = 0
    return W.astype(np.int64)


def draw(W: np.ndarray, R: int) -> int:
    """First token whose running sum of W exceeds floor(R * Z / 2^32); -1 when Z = 0."""
    Z = int(W.sum())
    if Z == 0:
        return -1
    t = (int(R) * Z) >> 32
    return int(np.searchsorted(np.cumsum(W), t, side="right"))


def spec_accept(p: np.ndarray, drafts: np.ndarray, rnd: np.ndarray | None = None,
                q: np.ndarray | None = None, greedy: bool = False):
    """Accepted drafts and the replacement / bonus token of every sequence.

    p [B, k+1, V] float32 target probabilities; drafts [B, k] int; rnd [B, k+1] uint32;
    q [B, k, V] float32 draft probabilities, or None for one-hot drafts (a deterministic
    proposer). Returns (out [B, k+1] int32: accepted drafts, the final token, then -1;
    num [B] int32: accepted drafts)."""
    p = np.asarray(p, dtype=np.float32)
    B, k1, V = p.shape
    k = k1 - 1
    out = np.full((B, k1), -1, dtype=np.int32)
    num = np.zeros(B, dtype=np.int32)
    for b in range(B):
        a = 0
        if greedy:
            while True:
                tok = int(np.argmax(p[b, a]))  # the first maximum: lowest token on ties
                if a == k or int(drafts[b, a]) != tok:
                    break
                a += 1
        else:
            plain = True  # every draft survived (bonus draw from p_k), or an invalid draft
            for i in range(k):
                d = int(drafts[b, i])
                if d < 0 or d >= V:
                    break
                qv = 1.0 if q is None else q[b, i, d]
                if not accepts(int(rnd[b, i]), p[b, i, d], qv):
                    plain = False
                    break
                a += 1
            if plain:
                w = p[b, a]
            else:
                qr = np.zeros(V, np.float32) if q is None else np.asarray(q[b, a], np.float32)
                if q is None:
                    qr[int(drafts[b, a])] = 1.0
                w = np.maximum(p[b, a] - qr, np.float32(0))
            tok = draw(weights(w), int(rnd[b, k]))
            if tok < 0:  # no residual mass: the same draw from p itself
                tok = draw(weights(p[b, a]), int(rnd[b, k]))
            tok = max(tok, 0)
        out[b, :a] = drafts[b, :a]
        out[b, a] = tok
        num[b] = a
    return out, num
