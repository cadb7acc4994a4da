"""Plant plausible mistakes in the CPU oracle and check that the pins catch each one.

Each mutant rewrites one expression of one oracle function (a dropped term, a wrong
index or sign, an off-by-one, a swapped operand), installs it in place of the
original for the duration of the test, and runs every pin. At least one pin must
fail. Nothing here touches a GPU.
"""
import inspect
import textwrap

import pytest

import oracle.paged_kv_oracle as O
import oracle.spec_oracle as S
from tests import pins, spec_pins

MUTANTS = [
    ("slot_of", "* BLOCK_SIZE + pos % BLOCK_SIZE", "* (BLOCK_SIZE - 1) + pos % BLOCK_SIZE"),
    ("slot_of", "+ pos % BLOCK_SIZE", "+ (pos + 1) % BLOCK_SIZE"),
    ("slot_of", "block_table_row[pos // BLOCK_SIZE]", "block_table_row[-1 - pos // BLOCK_SIZE]"),
    ("query_positions", "pos[start + i] = L - n + i", "pos[start + i] = L - n + i - 1"),
    ("query_positions", "pos[start + i] = L - n + i", "pos[start + i] = n - 1 - i"),
    ("kv_head_of", "return h // (H_q // H_kv)", "return h % H_kv"),
    ("causal_softmax_attention", "<= np.asarray(positions)", "< np.asarray(positions)"),
    ("causal_softmax_attention", "S = (Q @ K.T) * scale", "S = (Q @ K.T)"),
    ("causal_softmax_attention", "S = (Q @ K.T) * scale", "S = (Q @ K.T) / scale"),
    ("causal_softmax_attention", "P = E / E.sum(axis=1, keepdims=True)", "P = E"),
    ("causal_softmax_attention", "return P @ V, P", "return P @ K, P"),
    ("causal_softmax_attention", "np.exp(S - m)", "np.exp(m - S)"),
    ("paged_attention", "Vb = decode_bits(gather_context(v_pool", "Vb = decode_bits(gather_context(k_pool"),
    ("paged_attention", "qf[rs, h, :]", "qf[rs, kv, :]"),
    ("gather_context", "flat[slot_of(block_table_row, j)]", "flat[slot_of(block_table_row, L - 1 - j)]"),
    ("reshape_and_cache", "vp[s] = v[t]", "vp[s] = k[t]"),
    ("reshape_and_cache", "if s < 0:", "if s <= 0:"),
    ("decode_bits", "<< 16", "<< 15"),
    ("copy_blocks", "out[d] = src[s]", "out[s] = src[d]"),
    ("copy_blocks", "out[d] = src[s]", "out[d] = out[s]"),
    ("copy_blocks", "if 0 <= s < src.shape[0]", "if 0 < s < src.shape[0]"),
    ("rope", "[x1 * c - x2 * s, x2 * c + x1 * s]", "[x1 * c + x2 * s, x2 * c - x1 * s]"),
    ("rope", "(-(2.0 * np.arange(half)) / D)", "(-(1.0 * np.arange(half)) / D)"),
    ("rope", "c, s = np.cos(a)[:, None, :], np.sin(a)[:, None, :]",
     "s, c = np.cos(a)[:, None, :], np.sin(a)[:, None, :]"),
    ("rope", "x1, x2 = x[..., :half], x[..., half:]", "x1, x2 = x[..., 0::2], x[..., 1::2]"),
]


SPEC_MUTANTS = [
    ("accepts", "float(R) * float(np.float32(qv)) < float(np.float32(pv)) * 4294967296.0",
     "float(R) * float(np.float32(pv)) < float(np.float32(qv)) * 4294967296.0"),
    ("spec_accept", "np.maximum(p[b, a] - qr, np.float32(0))",
     "np.maximum(qr - p[b, a], np.float32(0))"),
    ("spec_accept", "                w = p[b, a]\n", "                w = p[b, 0]\n"),
    ("spec_accept", "qv = 1.0 if q is None else q[b, i, d]", "qv = 1.0"),
    ("spec_accept", "if not accepts(int(rnd[b, i]), p[b, i, d], qv):",
     "if accepts(int(rnd[b, i]), p[b, i, d], qv):"),
    ("spec_accept", "int(np.argmax(p[b, a]))", "int(np.argmin(p[b, a]))"),
    ("draw", "t = (int(R) * Z) >> 32", "t = (int(R) * Z) >> 33"),
]


def _mutated(name, old, new, mod=O):
    src = textwrap.dedent(inspect.getsource(getattr(mod, name)))
    assert src.count(old) == 1, (name, old)
    ns = dict(vars(mod))
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), ns)
    return ns[name]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[f"{m[0]}:{m[2]}" for m in MUTANTS])
def test_mutant_is_caught(monkeypatch, name, old, new):
    monkeypatch.setattr(O, name, _mutated(name, old, new))
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(O)
        except Exception as e:  # an assertion or a crash both count as caught
            failed.append((pin.__name__, type(e).__name__))
    assert failed, f"no pin caught the mutant {name}: {old!r} -> {new!r}"


@pytest.mark.parametrize("name,old,new", SPEC_MUTANTS, ids=[f"{m[0]}:{m[2]}" for m in SPEC_MUTANTS])
def test_spec_mutant_is_caught(monkeypatch, name, old, new):
    monkeypatch.setattr(S, name, _mutated(name, old, new, S))
    failed = []
    for pin in spec_pins.SPEC_PINS:
        try:
            pin(S)
        except Exception as e:  # an assertion or a crash both count as caught
            failed.append((pin.__name__, type(e).__name__))
    assert failed, f"no pin caught the mutant {name}: {old!r} -> {new!r}"
