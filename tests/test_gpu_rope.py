"""Rotary embedding fused with the KV scatter, through the C ABI, vs the CPU oracle.

q (rotated in place) and the key rows written to the pool must lie within one unit in
the last place of the exact float64 rotation plus 2^-20 (|x[i]| + |x[i + D/2]|): the
output's own rounding is half a unit, and the kernel's fp32 cosine and sine of the reduced
angle (error about 2^-22 of the pair's size) add the rest, which can exceed a unit of a
result much smaller than its inputs. V rows and every untouched pool row are bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_18_gb300 import binding
from paged_kv_attention_18_gb300 import workloads as W
from tests.gpu_util import dev, host_bits

pytestmark = pytest.mark.gpu

MANT = {"f16": 10, "bf16": 7}
MIN_EXP = {"f16": -14, "bf16": -126}


def ulp(x, dtype):
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** MIN_EXP[dtype])))
    return 2.0 ** (e - MANT[dtype])


def within_bound(got_bits, exact, x_bits, dtype):
    got = oracle.decode_bits(got_bits, dtype)
    x = oracle.decode_bits(x_bits, dtype)
    half = x.shape[-1] // 2
    mag = np.abs(x[..., :half]) + np.abs(x[..., half:])
    mag = np.concatenate([mag, mag], axis=-1)
    return np.abs(got - exact) <= ulp(exact, dtype) + 2.0 ** -20 * mag


# the last case has 136 heads per token: nine rounds of 128 rows in each 8-token pass
@pytest.mark.parametrize("dtype,H_q,H_kv,D,theta", [("bf16", 12, 2, 128, 1e6),
                                                    ("f16", 14, 2, 64, 1e6),
                                                    ("bf16", 8, 8, 128, 1e4),
                                                    ("f16", 128, 8, 128, 1e6)])
def test_rope_scatter_matches_oracle(dtype, H_q, H_kv, D, theta):
    rng = np.random.default_rng(110 + D + H_q)
    T, nb = 700, 96
    q = W.round_to_bits(rng.standard_normal((T, H_q, D), dtype=np.float32) * 2, dtype)
    k = W.round_to_bits(rng.standard_normal((T, H_kv, D), dtype=np.float32) * 2, dtype)
    v = W.round_to_bits(rng.standard_normal((T, H_kv, D), dtype=np.float32), dtype)
    kp = W.round_to_bits(rng.standard_normal((nb, 16, H_kv, D), dtype=np.float32), dtype)
    vp = W.round_to_bits(rng.standard_normal((nb, 16, H_kv, D), dtype=np.float32), dtype)
    pos = rng.integers(0, 40000, size=T).astype(np.int32)
    pos[:5] = [0, 1, 2, 32767, 39999]
    slots = rng.permutation(nb * 16)[:T].astype(np.int32)
    slots[::50] = -1  # padding tokens: q rotated, nothing cached
    qd, kd, vd = dev(q, dtype), dev(k, dtype), dev(v, dtype)
    kpd, vpd = dev(kp, dtype), dev(vp, dtype)
    binding.rope_reshape_and_cache(qd, kd, vd, dev(pos), dev(slots), kpd, vpd, theta)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    q_rot, k_rot, v_ref = oracle.rope_reshape_and_cache(q, k, v, pos, slots, kp, vp, theta, dtype)
    assert within_bound(host_bits(qd), q_rot, q, dtype).all()
    assert np.array_equal(host_bits(kd), k)  # k itself is not modified
    assert np.array_equal(host_bits(vpd), v_ref)
    got_k = host_bits(kpd).reshape(nb * 16, H_kv, D)
    ref_k = kp.reshape(nb * 16, H_kv, D)
    live = slots >= 0
    assert within_bound(got_k[slots[live]], k_rot[live], k[live], dtype).all()
    untouched = np.setdiff1d(np.arange(nb * 16), slots[live])
    assert np.array_equal(got_k[untouched], ref_k[untouched])


def test_rope_bad_slot_is_recorded():
    dtype, H_q, H_kv, D = "bf16", 4, 2, 64
    rng = np.random.default_rng(120)
    T, nb = 8, 4
    q = W.round_to_bits(rng.standard_normal((T, H_q, D), dtype=np.float32), dtype)
    k = W.round_to_bits(rng.standard_normal((T, H_kv, D), dtype=np.float32), dtype)
    kp = np.zeros((nb, 16, H_kv, D), np.uint16)
    slots = np.arange(T, dtype=np.int32)
    slots[3] = nb * 16  # past the pool
    kpd, vpd = dev(kp, dtype), dev(kp, dtype)
    qd = dev(q, dtype)
    binding.rope_reshape_and_cache(qd, dev(k, dtype), dev(k, dtype), dev(np.arange(T, dtype=np.int32)),
                                   dev(slots), kpd, vpd, 1e4)
    torch.cuda.synchronize()
    assert binding.device_error() == 2  # PS_DEV_BAD_SLOT
    skip = np.where(slots >= nb * 16, -1, slots)  # the kernel skips the bad slot
    q_rot, _, _ = oracle.rope_reshape_and_cache(q, k, k, np.arange(T), skip, kp, kp, 1e4, dtype)
    assert within_bound(host_bits(qd), q_rot, q, dtype).all()  # every q rotated
