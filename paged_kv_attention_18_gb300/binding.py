"""Python binding of the C ABI: argument marshalling from torch tensors, nothing else.

Every function checks that its tensors live on the current CUDA device, are
contiguous and have the expected dtypes and shapes, passes their addresses and the
current stream to the matching ``ps_*`` entry point of include/pagedserve.h, and
raises :class:`PagedServeError` on a non-zero status. All arithmetic happens in the
library's CUDA kernels.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

DTYPE_CODE = {torch.float16: 0, torch.bfloat16: 1}
BLOCK_SIZE = 16

# kernel kinds of the timing hook
PROFILE_KINDS = {"slot_mapping": 0, "reshape_and_cache": 1, "plan": 2, "split_attention": 3,
                 "combine": 4, "tile_attention": 5, "copy_blocks": 6, "spec_accept": 7,
                 "rope_reshape_and_cache": 8}


class PagedServeError(RuntimeError):
    pass


def lib():
    return _lib.load()


def _check(rc: int, what: str) -> None:
    if rc != 0:
        msg = lib().ps_status_string(rc).decode()
        if rc == -5:
            msg += f" [{lib().ps_last_error_message().decode()}]"
        raise PagedServeError(f"{what} failed: {msg} ({rc})")


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dev(t: torch.Tensor, name: str, dtype=None, ndim=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise PagedServeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise PagedServeError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise PagedServeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if ndim is not None and t.dim() != ndim:
        raise PagedServeError(f"{name} must have {ndim} dimensions, has {t.dim()}")
    return t.data_ptr()


def _batch(block_tables, seq_lens, query_start_loc):
    bt = _dev(block_tables, "block_tables", torch.int32, 2)
    sl = _dev(seq_lens, "seq_lens", torch.int32, 1)
    qs = _dev(query_start_loc, "query_start_loc", torch.int32, 1)
    B = seq_lens.shape[0]
    if block_tables.shape[0] != B or query_start_loc.shape[0] != B + 1:
        raise PagedServeError("block_tables / query_start_loc do not match seq_lens")
    return bt, sl, qs, B, block_tables.shape[1]


def slot_mapping(block_tables, seq_lens, query_start_loc, T: int, num_blocks: int, out=None,
                 stream=None) -> torch.Tensor:
    """int32 [T]: pool slot of every packed query token (ps_slot_mapping)."""
    bt, sl, qs, B, maxblk = _batch(block_tables, seq_lens, query_start_loc)
    if out is None:
        out = torch.empty(T, dtype=torch.int32, device=seq_lens.device)
    o = _dev(out, "slot_mapping", torch.int32, 1)
    _check(lib().ps_slot_mapping(bt, maxblk, sl, qs, B, T, num_blocks, o, _stream(stream)),
           "ps_slot_mapping")
    return out


def reshape_and_cache(k, v, slot_mapping_t, k_pool, v_pool, stream=None) -> None:
    """Write k/v [T, H_kv, D] into the pools [NB, 16, H_kv, D] at the slots (in place)."""
    dt = tuple(DTYPE_CODE)
    kp = _dev(k, "k", dt, 3)
    vp = _dev(v, "v", k.dtype, 3)
    sp = _dev(slot_mapping_t, "slot_mapping", torch.int32, 1)
    kpp = _dev(k_pool, "k_pool", k.dtype, 4)
    vpp = _dev(v_pool, "v_pool", k.dtype, 4)
    T, H_kv, D = k.shape
    if v.shape != k.shape or slot_mapping_t.shape[0] != T or k_pool.shape != v_pool.shape \
            or tuple(k_pool.shape[1:]) != (BLOCK_SIZE, H_kv, D):
        raise PagedServeError("reshape_and_cache: inconsistent shapes")
    _check(lib().ps_reshape_and_cache(kp, vp, sp, kpp, vpp, T, H_kv, D, k_pool.shape[0],
                                      DTYPE_CODE[k.dtype], _stream(stream)),
           "ps_reshape_and_cache")


def _mem(t: torch.Tensor, name: str, dtype=None, ndim=None) -> int:
    """Pointer to a CUDA tensor or a pinned host tensor (device-addressable memory)."""
    if isinstance(t, torch.Tensor) and not t.is_cuda and t.is_pinned():
        if not t.is_contiguous():
            raise PagedServeError(f"{name} must be contiguous")
        if dtype is not None and t.dtype != dtype and not (isinstance(dtype, tuple) and t.dtype in dtype):
            raise PagedServeError(f"{name} has dtype {t.dtype}")
        if ndim is not None and t.dim() != ndim:
            raise PagedServeError(f"{name} must have {ndim} dimensions")
        return t.data_ptr()
    return _dev(t, name, dtype, ndim)


def copy_blocks(src_k, src_v, dst_k, dst_v, src_ids, dst_ids, stream=None) -> None:
    """Copy whole blocks between pools (ps_copy_blocks): block dst_ids[i] of (dst_k, dst_v)
    becomes block src_ids[i] of (src_k, src_v). Pools are CUDA or pinned host tensors
    [num_blocks, 16, H_kv, D]; ids are int32 CUDA (or pinned) tensors of equal length."""
    dt = tuple(DTYPE_CODE)
    skp = _mem(src_k, "src_k", dt, 4)
    svp = _mem(src_v, "src_v", src_k.dtype, 4)
    dkp = _mem(dst_k, "dst_k", src_k.dtype, 4)
    dvp = _mem(dst_v, "dst_v", src_k.dtype, 4)
    sip = _mem(src_ids, "src_ids", torch.int32, 1)
    dip = _mem(dst_ids, "dst_ids", torch.int32, 1)
    if src_k.shape != src_v.shape or dst_k.shape != dst_v.shape or \
            tuple(src_k.shape[1:]) != tuple(dst_k.shape[1:]) or src_ids.shape != dst_ids.shape:
        raise PagedServeError("copy_blocks: inconsistent shapes")
    _, bs, H_kv, D = src_k.shape
    if bs != BLOCK_SIZE:
        raise PagedServeError("copy_blocks: pools must have 16-row blocks")
    _check(lib().ps_copy_blocks(skp, svp, src_k.shape[0], dkp, dvp, dst_k.shape[0], sip, dip,
                                src_ids.shape[0], H_kv, D, DTYPE_CODE[src_k.dtype],
                                _stream(stream)),
           "ps_copy_blocks")


def rope_reshape_and_cache(q, k, v, positions, slot_mapping_t, k_pool, v_pool,
                           rope_theta: float, stream=None) -> None:
    """Rotate q [T, H_q, D] in place and k [T, H_kv, D] into the pools at the slots by each
    token's position, copying v too (ps_rope_reshape_and_cache)."""
    dt = tuple(DTYPE_CODE)
    qp = _dev(q, "q", dt, 3)
    kp = _dev(k, "k", q.dtype, 3)
    vp = _dev(v, "v", q.dtype, 3)
    pp = _dev(positions, "positions", torch.int32, 1)
    sp = _dev(slot_mapping_t, "slot_mapping", torch.int32, 1)
    kpp = _dev(k_pool, "k_pool", q.dtype, 4)
    vpp = _dev(v_pool, "v_pool", q.dtype, 4)
    T, H_q, D = q.shape
    H_kv = k.shape[1]
    if k.shape != (T, H_kv, D) or v.shape != k.shape or positions.shape[0] != T or \
            slot_mapping_t.shape[0] != T or tuple(k_pool.shape[1:]) != (BLOCK_SIZE, H_kv, D) \
            or k_pool.shape != v_pool.shape:
        raise PagedServeError("rope_reshape_and_cache: inconsistent shapes")
    _check(lib().ps_rope_reshape_and_cache(qp, kp, vp, pp, sp, kpp, vpp, T, H_q, H_kv, D,
                                           k_pool.shape[0], float(rope_theta),
                                           DTYPE_CODE[q.dtype], _stream(stream)),
           "ps_rope_reshape_and_cache")


def spec_accept(target_probs, draft_tokens, random_bits=None, draft_probs=None,
                greedy: bool = False, workspace=None, stream=None):
    """Speculative acceptance (ps_spec_accept). target_probs float32 [B, k+1, V];
    draft_tokens int32 [B, k]; random_bits int32 [B, k+1] holding uint32 words (or None
    when greedy); draft_probs float32 [B, k, V] or None. Returns (out_tokens [B, k+1],
    num_accepted [B]) as int32 CUDA tensors."""
    pp = _dev(target_probs, "target_probs", torch.float32, 3)
    B, k1, V = target_probs.shape
    k = k1 - 1
    if draft_tokens.shape != (B, k):
        raise PagedServeError("spec_accept: draft_tokens shape")
    dp = _dev(draft_tokens, "draft_tokens", torch.int32, 2) if k > 0 else None
    qp = None
    if draft_probs is not None:
        if draft_probs.shape != (B, k, V):
            raise PagedServeError("spec_accept: draft_probs shape")
        qp = _dev(draft_probs, "draft_probs", torch.float32, 3)
    rp = None
    if random_bits is not None:
        if random_bits.shape != (B, k + 1):
            raise PagedServeError("spec_accept: random_bits shape")
        rp = _dev(random_bits, "random_bits", torch.int32, 2)
    elif not greedy:
        raise PagedServeError("spec_accept: random_bits required unless greedy")
    out = torch.empty((B, k + 1), dtype=torch.int32, device=target_probs.device)
    num = torch.empty((B,), dtype=torch.int32, device=target_probs.device)
    if workspace is None:
        n = max(int(lib().ps_spec_accept_workspace_size(B, k, V)), 256)
        workspace = torch.empty(n, dtype=torch.uint8, device=target_probs.device)
    wp = _dev(workspace, "workspace", torch.uint8, 1)
    _check(lib().ps_spec_accept(pp, qp, dp, rp, B, k, V, 1 if greedy else 0, _dev(out, "out"),
                                _dev(num, "num"), wp, workspace.numel(), _stream(stream)),
           "ps_spec_accept")
    return out, num


def workspace_size(T: int, B: int, H_q: int, H_kv: int, D: int, max_seq_len: int) -> int:
    return int(lib().ps_paged_attention_workspace_size(T, B, H_q, H_kv, D, max_seq_len))


def alloc_workspace(T, B, H_q, H_kv, D, max_seq_len, device=None) -> torch.Tensor:
    n = max(workspace_size(T, B, H_q, H_kv, D, max_seq_len), 256)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def paged_attention(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc, scale: float,
                    out=None, workspace=None, max_seq_len: int | None = None,
                    stream=None) -> torch.Tensor:
    """Causal paged attention of every packed query row (ps_paged_attention)."""
    qp = _dev(q, "q", tuple(DTYPE_CODE), 3)
    kpp = _dev(k_pool, "k_pool", q.dtype, 4)
    vpp = _dev(v_pool, "v_pool", q.dtype, 4)
    bt, sl, qs, B, maxblk = _batch(block_tables, seq_lens, query_start_loc)
    T, H_q, D = q.shape
    NB, bs, H_kv, Dk = k_pool.shape
    if bs != BLOCK_SIZE or Dk != D or v_pool.shape != k_pool.shape:
        raise PagedServeError("paged_attention: inconsistent pool shape")
    if out is None:
        out = torch.empty_like(q)
    op = _dev(out, "out", q.dtype, 3)
    if tuple(out.shape) != tuple(q.shape):
        raise PagedServeError("out must have q's shape")
    if workspace is None:
        msl = max_seq_len if max_seq_len is not None else maxblk * BLOCK_SIZE
        workspace = alloc_workspace(T, B, H_q, H_kv, D, msl, device=q.device)
    wp = _dev(workspace, "workspace", torch.uint8, 1)
    _check(lib().ps_paged_attention(qp, kpp, vpp, bt, maxblk, sl, qs, B, T, H_q, H_kv, D, NB,
                                    float(scale), op, wp, workspace.numel(),
                                    DTYPE_CODE[q.dtype], _stream(stream)),
           "ps_paged_attention")
    return out


def attention_step(q, k, v, k_pool, v_pool, block_tables, seq_lens, query_start_loc,
                   scale: float, out=None, workspace=None, slot_buf=None,
                   max_seq_len: int | None = None, stream=None) -> torch.Tensor:
    """Slot mapping, KV scatter and paged attention of one step (ps_attention_step)."""
    qp = _dev(q, "q", tuple(DTYPE_CODE), 3)
    kp = _dev(k, "k", q.dtype, 3)
    vp = _dev(v, "v", q.dtype, 3)
    kpp = _dev(k_pool, "k_pool", q.dtype, 4)
    vpp = _dev(v_pool, "v_pool", q.dtype, 4)
    bt, sl, qs, B, maxblk = _batch(block_tables, seq_lens, query_start_loc)
    T, H_q, D = q.shape
    NB, _, H_kv, _ = k_pool.shape
    if k.shape != (T, H_kv, D) or v.shape != k.shape:
        raise PagedServeError("attention_step: k/v shape")
    if out is None:
        out = torch.empty_like(q)
    op = _dev(out, "out", q.dtype, 3)
    if slot_buf is None:
        slot_buf = torch.empty(T, dtype=torch.int32, device=q.device)
    sp = _dev(slot_buf, "slot_buf", torch.int32, 1)
    if workspace is None:
        msl = max_seq_len if max_seq_len is not None else maxblk * BLOCK_SIZE
        workspace = alloc_workspace(T, B, H_q, H_kv, D, msl, device=q.device)
    wp = _dev(workspace, "workspace", torch.uint8, 1)
    _check(lib().ps_attention_step(qp, kp, vp, kpp, vpp, bt, maxblk, sl, qs, B, T, H_q, H_kv, D,
                                   NB, float(scale), op, sp, wp, workspace.numel(),
                                   DTYPE_CODE[q.dtype], _stream(stream)),
           "ps_attention_step")
    return out


def device_error() -> int:
    """Read and clear the device error word (synchronises)."""
    code = ctypes.c_int(0)
    _check(lib().ps_get_device_error(ctypes.addressof(code)), "ps_get_device_error")
    return code.value


def profile_begin(max_launches_per_kind: int) -> None:
    _check(lib().ps_profile_begin(max_launches_per_kind), "ps_profile_begin")


def profile_end() -> dict:
    _check(lib().ps_profile_end(), "ps_profile_end")
    res = {}
    for name, kind in PROFILE_KINDS.items():
        ms, n = ctypes.c_float(0), ctypes.c_int(0)
        _check(lib().ps_profile_read(kind, ctypes.addressof(ms), ctypes.addressof(n)),
               "ps_profile_read")
        res[name] = (ms.value, n.value)
    return res


def staging_size(T: int, B: int, max_blocks: int, H_q: int, H_kv: int, D: int,
                 max_seq_len: int) -> int:
    return int(lib().ps_attention_step_host_staging_size(T, B, max_blocks, H_q, H_kv, D,
                                                         max_seq_len))


def _host_step_args(q, k, v, block_tables, seq_lens, query_start_loc, out, k_pool, v_pool,
                    scale, staging) -> tuple:
    """Checked arguments of ps_attention_step_host, up to (not including) the stream."""
    for name, t in (("q", q), ("k", k), ("v", v), ("block_tables", block_tables),
                    ("seq_lens", seq_lens), ("query_start_loc", query_start_loc), ("out", out)):
        if t.is_cuda or not t.is_contiguous():
            raise PagedServeError(f"{name} must be a contiguous host tensor")
    if q.dtype not in DTYPE_CODE or k.dtype != q.dtype or v.dtype != q.dtype or out.dtype != q.dtype:
        raise PagedServeError("q/k/v/out dtype")
    for name, t in (("block_tables", block_tables), ("seq_lens", seq_lens),
                    ("query_start_loc", query_start_loc)):
        if t.dtype != torch.int32:
            raise PagedServeError(f"{name} must be int32")
    kpp = _dev(k_pool, "k_pool", q.dtype, 4)
    vpp = _dev(v_pool, "v_pool", q.dtype, 4)
    sp = _dev(staging, "staging", torch.uint8, 1)
    T, H_q, D = q.shape
    NB, _, H_kv, _ = k_pool.shape
    B, maxblk = block_tables.shape
    return (q.data_ptr(), k.data_ptr(), v.data_ptr(), block_tables.data_ptr(),
            seq_lens.data_ptr(), query_start_loc.data_ptr(), out.data_ptr(), kpp, vpp, maxblk, B,
            T, H_q, H_kv, D, NB, float(scale), sp, staging.numel(), DTYPE_CODE[q.dtype])


def attention_step_host(q, k, v, block_tables, seq_lens, query_start_loc, out, k_pool, v_pool,
                        scale: float, staging, stream=None) -> None:
    """One step from host tensors (ps_attention_step_host); ``out`` is a host tensor.

    q/k/v/block_tables/seq_lens/query_start_loc/out live in host memory (pin them for
    asynchronous copies); k_pool/v_pool and staging live on the device. The call returns
    once everything is enqueued: synchronise the stream before reading ``out``.
    """
    args = _host_step_args(q, k, v, block_tables, seq_lens, query_start_loc, out, k_pool,
                           v_pool, scale, staging)
    _check(lib().ps_attention_step_host(*args, _stream(stream)), "ps_attention_step_host")


class HostStepGraph:
    """ps_attention_step_host recorded once in a CUDA graph (ps_attention_step_host_graph_create).

    Every launch() copies the current contents of the host tensors to the device, runs the
    step and copies the output back into ``out``: write a step's inputs into the same
    tensors, launch, synchronise the stream, read ``out``. Shapes are fixed at creation;
    the host tensors must be pinned. The object keeps every tensor alive until close().
    """

    def __init__(self, q, k, v, block_tables, seq_lens, query_start_loc, out, k_pool, v_pool,
                 scale: float, staging):
        args = _host_step_args(q, k, v, block_tables, seq_lens, query_start_loc, out, k_pool,
                               v_pool, scale, staging)
        handle = ctypes.c_void_p()
        _check(lib().ps_attention_step_host_graph_create(*args, ctypes.addressof(handle)),
               "ps_attention_step_host_graph_create")
        self._handle = handle.value
        self._keep = (q, k, v, block_tables, seq_lens, query_start_loc, out, k_pool, v_pool,
                      staging)

    def launch(self, stream=None) -> None:
        if not self._handle:
            raise PagedServeError("graph is closed")
        _check(lib().ps_graph_launch(self._handle, _stream(stream)), "ps_graph_launch")

    def close(self) -> None:
        """Release the graph; its last launch must have completed."""
        if self._handle:
            lib().ps_graph_destroy(self._handle)
            self._handle = None
            self._keep = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
