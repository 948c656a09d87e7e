"""ctypes binding of libpagedkv.so: argument marshalling only.

The library is loaded from this package directory (built by ``build.py`` or
``__graft_entry__.build()``).  A missing library raises: there is no fallback.
"""
import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_CUDA = -3
PKV_ERR_OUT_OF_BLOCKS = -4
PKV_ERR_BAD_INDEX = -5

PKV_DEV_OK = 0
PKV_DEV_BAD_BLOCK_ID = 1
PKV_DEV_BAD_CONTEXT_LEN = 2
PKV_DEV_BAD_SLOT = 3
PKV_DEV_WAIT_TIMEOUT = 4
PKV_DEV_BAD_POSITION = 5
PKV_DEV_BAD_GROUP = 6

# name -> (restype, argtypes); every symbol the header declares.
_P, _I, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [_I]),
    "pkv_version": (_I, []),
    "pkv_paged_attention_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I64, _I, _F,
                                        _P, _SZ, _P, _P]),
    "pkv_paged_attention_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "pkv_paged_attention_split_tokens": (_I, [_I, _I, _I, _I]),
    "pkv_paged_attention_decode_grouped": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                                _I, _I, _I, _I, _I64, _I, _F, _P, _SZ, _P, _P]),
    "pkv_paged_attention_grouped_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "pkv_paged_attention_decode_grouped_fused": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                                      _I, _I, _I, _I, _I, _I, _I, _I, _I64, _I,
                                                      _F, _P, _SZ, _P, _P]),
    "pkv_plan_shared_prefix_groups": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "pkv_paged_attention_decode_fused_cow": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I,
                                                  _I, _I, _I, _I64, _I, _F, _P, _SZ, _P, _P]),
    "pkv_paged_attention_decode_grouped_fused_cow": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                                          _P, _I, _I, _I, _P, _P, _I, _I, _I, _I,
                                                          _I, _I64, _I, _F, _P, _SZ, _P, _P]),
    "pkv_cow_targets": (_I, [_P, _I, _P, _I, _I, _P, _P]),
    "pkv_paged_attention_decode_fused": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                              _I64, _I, _F, _P, _SZ, _P, _P]),
    "pkv_paged_attention_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I64,
                                                _I, _F, _P, _P]),
    "pkv_reshape_and_cache": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I64, _P, _P]),
    "pkv_slot_mapping": (_I, [_P, _P, _I, _I, _I, _I64, _P, _P, _P]),
    "pkv_copy_blocks": (_I, [_P, _P, _I, _P, _I, _I64, _I64, _P, _P]),
    "pkv_selftest_bounded_wait": (_I, [_P, _P, _I, _P]),
    "pkv_fill_normal_f16": (_I, [_P, _I64, ctypes.c_uint64, ctypes.c_uint64, _P]),
    "pkv_swap_blocks": (_I, [_P, _P, _I, _P, _I, _I64, _I64, _I64, _P, _P]),
    "pkv_sched_create": (_P, [_P, _I, _I, _I, _I, _I64, ctypes.c_uint64, _I]),
    "pkv_sched_destroy": (None, [_P]),
    "pkv_sched_add_request": (_I, [_P, _I64, _P, _I64, _I64]),
    "pkv_sched_step": (_I, [_P, _P]),
    "pkv_sched_num_unfinished": (_I64, [_P]),
    "pkv_sched_meta_bytes": (_SZ, [_P]),
    "pkv_sched_launch_decode": (_I, [_P, _P, _P, _P]),
    "pkv_sched_stage_decode": (_I, [_P, _P, _P, _P]),
    "pkv_sched_request_tokens": (_I64, [_P, _I64, _P, _I64]),
    "pkv_bm_create": (_P, [_I64, _I, _I, _P]),
    "pkv_bm_destroy": (None, [_P]),
    "pkv_bm_allocate": (_I, [_P, _I64, _P, _I64, _P, _I64, _P, _P]),
    "pkv_bm_append_slot": (_I, [_P, _I64, ctypes.c_int32, _P]),
    "pkv_bm_append_slots": (_I, [_P, _P, _P, _I64, _P, _P]),
    "pkv_bm_fork": (_I, [_P, _I64, _I64]),
    "pkv_bm_free": (_I, [_P, _I64]),
    "pkv_bm_slot": (_I, [_P, _I64, _I64, _P]),
    "pkv_bm_num_free_blocks": (_I64, [_P]),
    "pkv_bm_can_allocate": (_I, [_P, _I64]),
    "pkv_bm_block_table": (_I64, [_P, _I64, _P, _I64]),
    "pkv_bm_num_tokens": (_I64, [_P, _I64]),
    "pkv_bm_num_cached_tokens": (_I64, [_P, _I64]),
    "pkv_bm_fill_block_tables": (_I, [_P, _P, _I64, _P, _I64, ctypes.c_int32, _P]),
    "pkv_bm_take_cow_pairs": (_I64, [_P, _P, _I64]),
    "pkv_bm_free_list": (_I64, [_P, _P, _I64]),
    "pkv_bm_evictable_list": (_I64, [_P, _P, _I64]),
    "pkv_bm_ref_counts": (_I64, [_P, _P, _I64]),
    "pkv_bm_check_invariants": (_I, [_P]),
}

_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        name = lib().pkv_status_string(status).decode() if _lib is not None else str(status)
        super().__init__("%s: %s (status %d)" % (what, name, status))


def lib():
    """Load libpagedkv.so once; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libpagedkv.so is not built (%s); run "
                              "`python -m paged_kv_cache_138_gb300.build`" % LIB_PATH)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def check(status, what):
    if status != PKV_OK:
        raise PagedKVError(status, what)
    return status
