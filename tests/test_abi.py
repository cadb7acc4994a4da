"""The C ABI: the library loads, exports every declared symbol, and rejects bad
arguments on the host before touching a GPU (no compute calls here)."""
import ctypes
import os
import re

from paged_kv_attention_18_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pagedserve.h")


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ps_\w+)\s*\(", src)))


def test_header_declares_entry_points():
    names = declared_symbols()
    for n in ["ps_slot_mapping", "ps_reshape_and_cache", "ps_paged_attention",
              "ps_paged_attention_workspace_size", "ps_attention_step", "ps_get_device_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, name


def test_status_strings(lib):
    assert lib.ps_status_string(0) == b"PS_OK"
    for rc in (-1, -2, -3, -4, -5):
        assert lib.ps_status_string(rc).startswith(b"PS_ERR")


def test_workspace_size(lib):
    small = lib.ps_paged_attention_workspace_size(4, 4, 4, 2, 64, 0)
    big = lib.ps_paged_attention_workspace_size(256, 256, 12, 2, 128, 4096)
    assert 0 < small < big
    assert lib.ps_paged_attention_workspace_size(4, 4, 5, 2, 64, 100) == 0  # H_q % H_kv
    assert lib.ps_paged_attention_workspace_size(4, 4, 4, 2, 96, 100) == 0  # head_dim
    big = 2 ** 31 - 1  # sizes are taken in 64 bits: no wrapped (small) size comes back
    assert lib.ps_paged_attention_workspace_size(big, big, 12, 2, 128, 0) == 0


def test_batch_sizes_near_int_max_are_rejected_before_device_work(lib):
    big = 2 ** 31 - 1
    rc = lib.ps_paged_attention(FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, big, big, 12, 2, 128,
                                64, ctypes.c_float(0.1), FAKE, FAKE, 1 << 40, 1, None)
    assert rc == -4  # PS_ERR_WORKSPACE: the plan's lists cannot be laid out
    rc = lib.ps_paged_attention_noalloc(FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, big, big, 12,
                                        2, 128, 64, ctypes.c_float(0.1), FAKE, 1, None)
    assert rc == -4


FAKE = 1 << 20  # a 16-byte-aligned non-null address; never dereferenced by these calls


def test_reshape_and_cache_rejects(lib):
    f = lib.ps_reshape_and_cache
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 96, 8, 1, None) == -2      # head_dim
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 8, 7, None) == -2      # dtype
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, -1, 2, 64, 8, 1, None) == -1     # T
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 0, 1, None) == -1      # pool
    assert f(FAKE + 2, FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 8, 1, None) == -3  # alignment
    assert f(None, FAKE, FAKE, FAKE, FAKE, 4, 2, 64, 8, 1, None) == -1      # null
    assert f(None, None, None, None, None, 0, 2, 64, 8, 1, None) == 0       # empty: no-op


def test_slot_mapping_rejects(lib):
    f = lib.ps_slot_mapping
    assert f(FAKE, 4, FAKE, FAKE, 0, 3, 8, FAKE, None) == -1   # B = 0 with T > 0
    assert f(FAKE, 4, None, FAKE, 2, 3, 8, FAKE, None) == -1   # null seq_lens
    assert f(FAKE, 4, FAKE, FAKE, 2, 3, 8, None, None) == -1   # null output
    assert f(FAKE, 4, FAKE, FAKE, 2, 3, -1, FAKE, None) == -1  # pool
    assert f(None, 0, None, None, 0, 0, 8, None, None) == 0    # empty batch: no-op


def test_paged_attention_rejects(lib):
    f = lib.ps_paged_attention

    def call(**kw):
        a = dict(q=FAKE, kp=FAKE, vp=FAKE, bt=FAKE, maxblk=4, sl=FAKE, qsl=FAKE, B=2, T=3,
                 Hq=12, Hkv=2, D=128, NB=64, scale=0.1, out=FAKE, ws=FAKE, wsb=1 << 30,
                 dtype=1)
        a.update(kw)
        return f(a["q"], a["kp"], a["vp"], a["bt"], a["maxblk"], a["sl"], a["qsl"], a["B"],
                 a["T"], a["Hq"], a["Hkv"], a["D"], a["NB"], ctypes.c_float(a["scale"]),
                 a["out"], a["ws"], a["wsb"], a["dtype"], None)

    assert call(Hq=13) == -2
    assert call(D=80) == -2
    assert call(dtype=3) == -2
    assert call(q=FAKE + 8) == -3
    assert call(out=FAKE + 4) == -3
    assert call(ws=None) == -4
    assert call(ws=FAKE + 64) == -4          # workspace must be 256-byte aligned
    assert call(wsb=16) == -4                # too small
    assert call(B=0) == -1                   # T > 0 needs sequences
    assert call(maxblk=0) == -1
    assert call(T=0) == 0                    # nothing to do


def test_attention_step_rejects(lib):
    f = lib.ps_attention_step
    rc = f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 2, 3, 12, 2, 72, 64,
           ctypes.c_float(0.1), FAKE, FAKE, FAKE, 1 << 30, 1, None)
    assert rc == -2  # D = 72 unsupported, found before anything is enqueued
    rc = f(FAKE, FAKE + 4, FAKE, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 2, 3, 12, 2, 128, 64,
           ctypes.c_float(0.1), FAKE, FAKE, FAKE, 1 << 30, 1, None)
    assert rc == -3  # k misaligned


def test_profile_read_rejects(lib):
    ms, n = ctypes.c_float(), ctypes.c_int()
    assert lib.ps_profile_read(9, ctypes.addressof(ms), ctypes.addressof(n)) == -1
    assert lib.ps_profile_begin(0) == -1


def test_copy_blocks_rejects(lib):
    f = lib.ps_copy_blocks
    args = lambda **kw: [kw.get(n, d) for n, d in (  # noqa: E731
        ("sk", FAKE), ("sv", FAKE), ("snb", 8), ("dk", FAKE), ("dv", FAKE), ("dnb", 8),
        ("si", FAKE), ("di", FAKE), ("n", 4), ("hkv", 2), ("d", 64), ("dt", 1), ("s", None))]
    assert f(*args(d=96)) == -2              # head_dim
    assert f(*args(dt=7)) == -2              # dtype
    assert f(*args(n=-1)) == -1              # count
    assert f(*args(snb=0)) == -1             # source pool size
    assert f(*args(sk=FAKE + 2)) == -3       # alignment
    assert f(*args(si=None)) == -1           # ids
    assert f(*args(sk=None, sv=None, dk=None, dv=None, si=None, di=None, n=0)) == 0  # no-op


def test_rope_reshape_and_cache_rejects(lib):
    f = lib.ps_rope_reshape_and_cache
    args = lambda **kw: [kw.get(n, d) for n, d in (  # noqa: E731
        ("q", FAKE), ("k", FAKE), ("v", FAKE), ("pos", FAKE), ("slots", FAKE), ("kp", FAKE),
        ("vp", FAKE), ("T", 4), ("hq", 12), ("hkv", 2), ("d", 128), ("nb", 8),
        ("theta", ctypes.c_float(1e6)), ("dt", 1), ("s", None))]
    assert f(*args(d=96)) == -2                          # head_dim
    assert f(*args(hq=5)) == -2                          # H_q % H_kv
    assert f(*args(theta=ctypes.c_float(0.5))) == -1     # rotary base
    assert f(*args(T=-1)) == -1                          # count
    assert f(*args(q=FAKE + 4)) == -3                    # alignment
    assert f(*args(pos=None)) == -1                      # positions
    assert f(*args(q=None, k=None, v=None, pos=None, slots=None, kp=None, vp=None, T=0)) == 0


def test_spec_accept_rejects(lib):
    f = lib.ps_spec_accept
    need = lib.ps_spec_accept_workspace_size(4, 4, 1000)
    assert need > 0 and lib.ps_spec_accept_workspace_size(-1, 4, 1000) == 0
    args = lambda **kw: [kw.get(n, d) for n, d in (  # noqa: E731
        ("p", FAKE), ("q", None), ("dr", FAKE), ("r", FAKE), ("B", 4), ("k", 4), ("V", 1000),
        ("g", 0), ("out", FAKE), ("num", FAKE), ("ws", FAKE), ("wsb", need), ("s", None))]
    assert f(*args(B=-1)) == -1              # batch
    assert f(*args(V=0)) == -1               # vocabulary
    assert f(*args(k=32)) == -2              # one lane per draft: k <= 31
    assert f(*args(V=(1 << 30) + 1)) == -2   # token indices stay 32-bit
    assert f(*args(r=None)) == -1            # random words needed by the rejection rule
    assert f(*args(dr=None)) == -1           # drafts needed when k > 0
    assert f(*args(ws=FAKE + 16)) == -4      # workspace alignment (256 bytes)
    assert f(*args(wsb=need - 1)) == -4      # workspace size
    assert f(*args(p=None, dr=None, r=None, out=None, num=None, ws=None, B=0)) == 0


def test_graph_calls_reject_null_handles(lib):
    assert lib.ps_graph_launch(None, None) == -1
    assert lib.ps_graph_destroy(None) == -1
    # no place for the handle: rejected before any CUDA call
    f = lib.ps_attention_step_host_graph_create
    rc = f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 3, 12, 2, 128, 64,
           ctypes.c_float(0.1), FAKE, 1 << 30, 1, None)
    assert rc == -1
    # shape errors come back before any device work or recording
    handle = ctypes.c_void_p()
    rc = f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 3, 12, 2, 72, 64,
           ctypes.c_float(0.1), FAKE, 1 << 30, 1, ctypes.addressof(handle))
    assert rc == -2 and handle.value is None  # D = 72 unsupported; no handle
    rc = f(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 3, 12, 5, 128, 64,
           ctypes.c_float(0.1), FAKE, 1 << 30, 1, ctypes.addressof(handle))
    assert rc == -2 and handle.value is None  # 12 query heads over 5 KV heads
