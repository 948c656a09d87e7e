"""libpagedkv loads and exports every function include/pagedkv.h declares.

No CUDA call is made here: argument validation that fails before any launch is
exercised, nothing else.
"""
import ctypes
import os
import re

from conftest import ROOT


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pagedkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(native_lib):
    from paged_kv_cache_138_gb300._lib import LIB_PATH, SIGNATURES
    raw = ctypes.CDLL(LIB_PATH)
    names = declared_functions()
    assert len(names) >= 25
    for n in names:
        assert hasattr(raw, n), "missing export " + n
        assert n in SIGNATURES, "binding lacks " + n


def test_status_strings_and_version(native_lib):
    assert native_lib.pkv_version() >= 100
    assert native_lib.pkv_status_string(0) == b"ok"
    assert b"out of KV blocks" in native_lib.pkv_status_string(-4)


def test_host_side_validation_needs_no_gpu(native_lib):
    L = native_lib
    # unsupported head_dim / block size / GQA ratio are rejected before any launch
    args = [None] * 6
    assert L.pkv_paged_attention_decode(*args, 1, 8, 8, 64, 16, 10, 4, 0.1, None, 0, None,
                                        None) == -2
    assert L.pkv_paged_attention_decode(*args, 1, 8, 8, 128, 12, 10, 4, 0.1, None, 0, None,
                                        None) == -2
    assert L.pkv_paged_attention_decode(*args, 1, 12, 8, 128, 16, 10, 4, 0.1, None, 0, None,
                                        None) == -2
    assert L.pkv_paged_attention_decode(*args, 1, 24, 8, 128, 16, 10, 4, 0.1, None, 0, None,
                                        None) == -2     # G = 3 has no kernel
    # empty batch is a no-op
    assert L.pkv_paged_attention_decode(*args, 0, 8, 8, 128, 16, 10, 4, 0.1, None, 0, None,
                                        None) == 0
    # workspace sizing: one split per 512 tokens, (D + 2) floats per split
    assert L.pkv_paged_attention_workspace_bytes(4, 8, 32, 16, 128) == 0
    assert L.pkv_paged_attention_workspace_bytes(4, 8, 33, 16, 128) == 4 * 8 * 2 * 130 * 4
    assert L.pkv_paged_attention_workspace_bytes(4, 8, 64, 8, 128) == 0
    assert L.pkv_paged_attention_workspace_bytes(4, 8, 9, 64, 128) == 4 * 8 * 2 * 130 * 4
    # block sizes without a kernel
    assert L.pkv_paged_attention_decode(*args, 1, 8, 8, 128, 4, 10, 4, 0.1, None, 0, None,
                                        None) == -2
    assert L.pkv_paged_attention_decode_fused(*(args + [None, None]), 1, 8, 8, 128, 128, 10, 4,
                                              0.1, None, 0, None, None) == -2
    assert L.pkv_reshape_and_cache(None, None, None, None, None, 0, 8, 128, 16, 10, None,
                                   None) == 0
    assert L.pkv_reshape_and_cache(None, None, None, None, None, 3, 8, 128, 16, 10, None,
                                   None) == -1
    assert L.pkv_copy_blocks(None, None, 1, None, 0, 4096, 10, None, None) == 0
    assert L.pkv_copy_blocks(None, None, 1, None, 2, 4095, 10, None, None) == -1


def test_split_length_per_launch(native_lib):
    """The longest split (2048, 1024, 512 tokens) for which S x Hkv x
    ceil(table tokens / split) still reaches 1024 CTAs."""
    st = native_lib.pkv_paged_attention_split_tokens
    assert st(64, 40, 256, 16) == 2048        # the Llama-2-13B layer batch: 5120 CTAs
    assert st(256, 8, 256, 16) == 2048        # GQA 32/8
    assert st(64, 32, 256, 16) == 2048        # a Llama-2-7B layer
    assert st(256, 4, 256, 16) == 2048        # 1024 x 2 CTAs
    assert st(128, 4, 256, 16) == 2048        # 512 KV rows x 2 splits = 1024
    assert st(64, 4, 256, 16) == 1024         # 256 x 2 < 1024; 256 x 4 = 1024
    assert st(32, 8, 256, 16) == 1024         # 256 x 4 = 1024
    assert st(16, 8, 256, 16) == 512          # 128 x 8 = 1024 (1024-token splits give 512)
    assert st(8, 8, 256, 16) == 512           # too small for anything longer
    assert st(1, 1, 4096, 16) == 512          # one 64K-token context: 128 CTAs at best
    assert st(64, 40, 512, 8) == 2048         # the same tokens in 8-token blocks
    assert st(64, 40, 64, 64) == 2048
    assert st(5, 8, 4, 16) == 512             # the tiny batch
    assert st(0, 8, 4, 16) == -1 and st(4, 8, 4, 12) == -1
