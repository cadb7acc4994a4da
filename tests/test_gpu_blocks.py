"""Block copies through the C ABI vs the CPU oracle, bit-exact: copy-on-write inside a
device pool, and a swap out to a pinned host pool and back in."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_18_gb300 import binding
from paged_kv_attention_18_gb300 import workloads as W
from tests.gpu_util import TORCH_DT, dev, host_bits

pytestmark = pytest.mark.gpu


def _pool(rng, nb, H_kv, D, dtype):
    return W.round_to_bits(rng.standard_normal((nb, 16, H_kv, D), dtype=np.float32), dtype)


def _pinned(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(TORCH_DT[dtype])
    return t.pin_memory()


def _ids(a) -> torch.Tensor:
    return torch.tensor(np.asarray(a, dtype=np.int32), device="cuda")


@pytest.mark.parametrize("dtype,H_kv,D", [("bf16", 2, 128), ("f16", 2, 64), ("bf16", 8, 128)])
def test_copy_on_write_in_device_pool(dtype, H_kv, D):
    rng = np.random.default_rng(60 + D + H_kv)
    nb = 700
    kp, vp = _pool(rng, nb, H_kv, D, dtype), _pool(rng, nb, H_kv, D, dtype)
    perm = rng.permutation(nb)
    src, dst = perm[:250], perm[250:500]  # disjoint, distinct destinations
    src[:3] = [perm[0], perm[1], perm[0]]  # a block copied twice
    k, v = dev(kp, dtype), dev(vp, dtype)
    binding.copy_blocks(k, v, k, v, _ids(src), _ids(dst))
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    assert np.array_equal(host_bits(k), oracle.copy_blocks(kp, kp, src, dst))
    assert np.array_equal(host_bits(v), oracle.copy_blocks(vp, vp, src, dst))


def test_swap_out_to_pinned_host_and_back():
    dtype, H_kv, D = "bf16", 2, 128
    rng = np.random.default_rng(70)
    nb, nh = 512, 200
    kp, vp = _pool(rng, nb, H_kv, D, dtype), _pool(rng, nb, H_kv, D, dtype)
    hk0, hv0 = _pool(rng, nh, H_kv, D, dtype), _pool(rng, nh, H_kv, D, dtype)
    k, v = dev(kp, dtype), dev(vp, dtype)
    hk, hv = _pinned(hk0, dtype), _pinned(hv0, dtype)
    out_src = rng.choice(nb, size=150, replace=False)
    out_dst = rng.choice(nh, size=150, replace=False)
    binding.copy_blocks(k, v, hk, hv, _ids(out_src), _ids(out_dst))  # swap out
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    hk_ref = oracle.copy_blocks(kp, hk0, out_src, out_dst)
    hv_ref = oracle.copy_blocks(vp, hv0, out_src, out_dst)
    assert np.array_equal(hk.view(torch.int16).numpy().view(np.uint16), hk_ref)
    assert np.array_equal(hv.view(torch.int16).numpy().view(np.uint16), hv_ref)
    # swap back in to other device blocks (ids held in pinned host memory this time)
    free = np.setdiff1d(np.arange(nb), out_src)
    in_dst = rng.choice(free, size=150, replace=False)
    ids_src = torch.tensor(out_dst.astype(np.int32)).pin_memory()
    ids_dst = torch.tensor(in_dst.astype(np.int32)).pin_memory()
    binding.copy_blocks(hk, hv, k, v, ids_src, ids_dst)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    assert np.array_equal(host_bits(k), oracle.copy_blocks(hk_ref, kp, out_dst, in_dst))
    assert np.array_equal(host_bits(v), oracle.copy_blocks(hv_ref, vp, out_dst, in_dst))
    # the blocks came back unchanged: each sequence block round-tripped bit-exact
    assert np.array_equal(host_bits(k)[in_dst], kp[out_src])


def test_copy_blocks_bad_ids_are_skipped():
    dtype, H_kv, D = "f16", 2, 64
    rng = np.random.default_rng(80)
    nb = 64
    kp, vp = _pool(rng, nb, H_kv, D, dtype), _pool(rng, nb, H_kv, D, dtype)
    k, v = dev(kp, dtype), dev(vp, dtype)
    src, dst = np.array([1, 70, 2, 3]), np.array([10, 11, -1, 12])
    binding.copy_blocks(k, v, k, v, _ids(src), _ids(dst))
    torch.cuda.synchronize()
    assert binding.device_error() == 1  # PS_DEV_BAD_BLOCK_ID
    assert np.array_equal(host_bits(k), oracle.copy_blocks(kp, kp, src, dst))
    assert np.array_equal(host_bits(v), oracle.copy_blocks(vp, vp, src, dst))
    # n = 0 is a no-op
    binding.copy_blocks(k, v, k, v, _ids([]), _ids([]))
    torch.cuda.synchronize()
    assert binding.device_error() == 0
