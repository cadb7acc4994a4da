"""ctypes loader for the in-tree CUDA library ``libpagedserve.so``.

Declares the argument and result types of every entry point of include/pagedserve.h.
There is no fallback: if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedserve.so")

_lock = threading.Lock()
_lib = None

c_int, c_float, c_size_t, c_void_p, c_char_p = (ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                                                 ctypes.c_void_p, ctypes.c_char_p)
_p = c_void_p  # every pointer argument is passed as an address

SIGNATURES = {
    "ps_slot_mapping": (c_int, [_p, c_int, _p, _p, c_int, c_int, c_int, _p, _p]),
    "ps_reshape_and_cache": (c_int, [_p, _p, _p, _p, _p, c_int, c_int, c_int, c_int, c_int, _p]),
    "ps_copy_blocks": (c_int, [_p, _p, c_int, _p, _p, c_int, _p, _p, c_int, c_int, c_int, c_int,
                               _p]),
    "ps_rope_reshape_and_cache": (c_int, [_p, _p, _p, _p, _p, _p, _p, c_int, c_int, c_int, c_int,
                                          c_int, c_float, c_int, _p]),
    "ps_spec_accept_workspace_size": (c_size_t, [c_int, c_int, c_int]),
    "ps_spec_accept": (c_int, [_p, _p, _p, _p, c_int, c_int, c_int, c_int, _p, _p, _p, c_size_t,
                               _p]),
    "ps_paged_attention_workspace_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int, c_int]),
    "ps_paged_attention": (c_int, [_p, _p, _p, _p, c_int, _p, _p, c_int, c_int, c_int, c_int,
                                   c_int, c_int, c_float, _p, _p, c_size_t, c_int, _p]),
    "ps_paged_attention_noalloc": (c_int, [_p, _p, _p, _p, c_int, _p, _p, c_int, c_int, c_int,
                                           c_int, c_int, c_int, c_float, _p, c_int, _p]),
    "ps_attention_step": (c_int, [_p, _p, _p, _p, _p, _p, c_int, _p, _p, c_int, c_int, c_int,
                                  c_int, c_int, c_int, c_float, _p, _p, _p, c_size_t, c_int, _p]),
    "ps_attention_step_host_staging_size": (c_size_t, [c_int, c_int, c_int, c_int, c_int,
                                                        c_int, c_int]),
    "ps_attention_step_host": (c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _p, c_int, c_int, c_int,
                                       c_int, c_int, c_int, c_int, c_float, _p, c_size_t, c_int,
                                       _p]),
    "ps_attention_step_host_graph_create": (c_int, [_p, _p, _p, _p, _p, _p, _p, _p, _p, c_int,
                                                    c_int, c_int, c_int, c_int, c_int, c_int,
                                                    c_float, _p, c_size_t, c_int, _p]),
    "ps_graph_launch": (c_int, [_p, _p]),
    "ps_graph_destroy": (c_int, [_p]),
    "ps_get_device_error": (c_int, [_p]),
    "ps_status_string": (c_char_p, [c_int]),
    "ps_last_error_message": (c_char_p, []),
    "ps_profile_begin": (c_int, [c_int]),
    "ps_profile_end": (c_int, []),
    "ps_profile_read": (c_int, [c_int, _p, _p]),
}


def load(path: str = LIB_PATH):
    """Load the library once and declare its entry points. Raises if it is not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is not built; run __graft_entry__.build() "
                    "(nvcc, sm_103a). There is no CPU fallback.")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib
