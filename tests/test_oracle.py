"""The CPU oracle against its pins (no GPU)."""
import numpy as np
import pytest

import oracle
import oracle.spec_oracle
from tests import pins, spec_pins


@pytest.mark.parametrize("pin", spec_pins.SPEC_PINS, ids=lambda p: p.__name__)
def test_spec_pin(pin):
    pin(oracle.spec_oracle)


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle)


def test_empty_batch():
    q = np.zeros((0, 4, 8), np.uint16)
    kp = np.zeros((2, 16, 2, 8), np.uint16)
    out = oracle.paged_attention(q, kp, kp, np.zeros((0, 1), np.int32), np.zeros(0, np.int32),
                                 np.zeros(1, np.int32), 0.5, "f16")
    assert out.shape == (0, 4, 8)
    assert oracle.slot_mapping(np.zeros((0, 1), np.int32), np.zeros(0), np.zeros(1)).shape == (0,)


def test_rejects_more_queries_than_context():
    with pytest.raises(ValueError):
        oracle.query_positions(np.array([2]), np.array([0, 3]))


def test_sampled_rows_match_full():
    from paged_kv_attention_18_gb300 import workloads as W
    wl = W.simple_workload("s", seed=3, dtype="bf16", H_q=4, H_kv=2, D=16,
                           seqs=[(40, 3), (17, 1), (60, 9)])
    st = wl.steps[0]
    args = (st.q, wl.k_pool, wl.v_pool, st.block_tables, st.seq_lens, st.query_start_loc,
            wl.scale, wl.dtype)
    full = oracle.paged_attention(*args)
    rows = [0, 4, 12]
    part = oracle.paged_attention(*args, rows=rows)
    np.testing.assert_allclose(part[rows], full[rows], rtol=0, atol=1e-12)
    assert np.isnan(part[[1, 2, 3]]).all()
