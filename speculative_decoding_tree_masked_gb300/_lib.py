"""ctypes declarations of libtreeverify.so (the C ABI in include/treeverify.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtreeverify.so")

c_i32 = ctypes.c_int32
c_i64 = ctypes.c_int64
c_ptr = ctypes.c_void_p
c_size = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/treeverify.h one to one
SIGNATURES = {
    "tv_status_string": (ctypes.c_char_p, [c_i32]),
    "tv_version": (c_i32, []),
    "tv_checked_build": (c_i32, []),
    "tv_tree_mask": (c_i32, [c_ptr, c_i32, c_ptr, c_ptr, c_ptr]),
    "tv_attn_uses_tensor_cores": (c_i32, [c_i32]),
    "tv_attn_workspace_size": (c_size, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32]),
    "tv_attn_plan": (c_i32, [c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_ptr, c_ptr, c_ptr,
                             c_ptr]),
    "tv_tree_attn_verify": (c_i32, [c_ptr, c_ptr, c_ptr, c_i64, c_i32, c_i32, c_ptr, c_ptr,
                                    c_i32, c_i32, c_i32, c_i32, ctypes.c_float, c_ptr, c_size,
                                    c_ptr, c_ptr]),
    "tv_tree_attn_verify_static": (c_i32, [c_ptr, c_ptr, c_ptr, c_i64, c_i32, c_i32, c_ptr,
                                           c_ptr, c_i32, c_i32, c_i32, c_i32, ctypes.c_float,
                                           c_ptr, c_ptr]),
    "tv_attn_batched_workspace_size": (c_size, [c_i32, c_ptr, c_i32, c_i32, c_i32, c_i32]),
    "tv_tree_attn_verify_batched": (c_i32, [c_i32, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr,
                                            c_ptr, c_ptr, c_i32, c_i32, c_i32, c_i32,
                                            ctypes.c_float, c_ptr, c_size, c_ptr, c_ptr]),
    "tv_tree_attn_verify_paged": (c_i32, [c_ptr, c_ptr, c_ptr, c_i32, c_i32, c_ptr, c_i32, c_i32,
                                          c_ptr, c_ptr, c_i32, c_i32, c_i32, c_i32,
                                          ctypes.c_float, c_ptr, c_size, c_ptr, c_ptr]),
    "tv_tree_attn_verify_batched_paged": (c_i32, [c_i32, c_ptr, c_ptr, c_ptr, c_i32, c_i32, c_ptr,
                                                  c_ptr, c_ptr, c_ptr, c_ptr, c_i32, c_i32, c_i32,
                                                  c_i32, ctypes.c_float, c_ptr, c_size, c_ptr,
                                                  c_ptr]),
    "tv_kv_compact_paged": (c_i32, [c_ptr, c_ptr, c_i32, c_i64, c_i32, c_i32, c_i32, c_i32, c_i32,
                                    c_ptr, c_i32, c_i32, c_ptr, c_ptr, c_ptr]),
    "tv_tree_accept": (c_i32, [c_ptr, c_i32, c_ptr, c_ptr, c_i32, c_i32, c_ptr, c_ptr, c_ptr,
                               c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr]),
    "tv_kv_compact": (c_i32, [c_ptr, c_ptr, c_i32, c_i64, c_i32, c_i64, c_i32, c_i32, c_i32,
                              c_i32, c_ptr, c_ptr, c_ptr]),
    "tv_tree_accept_tokens": (c_i32, [c_ptr, c_i32, c_ptr, c_ptr, c_i32, c_i32, c_ptr, c_ptr,
                                      c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr]),
    "tv_tree_accept_sampled": (c_i32, [c_ptr, c_i32, c_ptr, c_ptr, c_i32, c_i32, ctypes.c_float,
                                       ctypes.c_uint64, ctypes.c_uint64, c_ptr, c_ptr, c_ptr,
                                       c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr]),
    "tv_tree_accept_batched": (c_i32, [c_i32, c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_ptr, c_ptr,
                                       c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr]),
    "tv_tree_accept_tokens_batched": (c_i32, [c_i32, c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_ptr,
                                              c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr,
                                              c_ptr]),
    "tv_tree_accept_sampled_batched": (c_i32, [c_i32, c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_ptr,
                                               c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr,
                                               c_ptr, c_ptr, c_ptr, c_ptr, c_ptr]),
    "tv_kv_compact_batched": (c_i32, [c_i32, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr,
                                      c_i32, c_i32, c_i32, c_i32, c_ptr, c_ptr]),
    "tv_kv_compact_batched_paged": (c_i32, [c_i32, c_ptr, c_ptr, c_i32, c_i64, c_i32, c_i32,
                                            c_i32, c_i32, c_i32, c_ptr, c_ptr, c_ptr, c_ptr,
                                            c_ptr, c_ptr]),
    "tv_expand_workspace_size": (c_size, [c_i32, c_i32, c_i32]),
    "tv_tree_expand": (c_i32, [c_ptr, c_i32, c_i32, c_ptr, c_ptr, c_i32, c_i32, c_ptr, c_ptr,
                               c_ptr, c_ptr, c_size, c_ptr, c_ptr]),
    "tv_draft_reroot": (c_i32, [c_ptr, c_ptr, c_ptr, c_i32, c_ptr, c_ptr, c_ptr, c_i32, c_ptr,
                                c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr]),
    "tv_lm_head_workspace_size": (c_size, [c_i32, c_i32]),
    "tv_lm_head_argmax": (c_i32, [c_ptr, c_ptr, c_i32, c_i32, c_i32, c_ptr, c_ptr, c_ptr, c_size,
                                  c_ptr, c_ptr]),
}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load (once) and return the library with every signature declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: the CUDA library has not been built "
            "(run speculative_decoding_tree_masked_gb300._build.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
