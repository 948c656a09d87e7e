"""TEST INFRASTRUCTURE ONLY: fp64 paged decode attention, two independent forms.

``paged_attention_decode`` calls the C oracle (``paged_attention_ref.c``): the
plain definition, gathered through the block table and masked at the context
length, in fp64 with OpenMP over (sequence, head).

``paged_attention_gather_concat`` is a second, pure-NumPy form for tiny inputs.
It follows the gather-and-concatenate pseudocode of "qaqbuyan: vLLM
PagedAttention" (`paged_attention`): collect each logical block's physical block,
concatenate them, slice to the context length and apply dense softmax attention.
The two forms share no code; tests require them to agree to 1e-12.
"""
import ctypes

import numpy as np

from .build import build_oracle

_lib = None


def _load():
    global _lib
    if _lib is None:
        _lib = bind(ctypes.CDLL(build_oracle()))
    return _lib


def bind(lib):
    """Declare the C oracle's entry points on a loaded library (``_load``; the
    mutation tests bind deliberately broken copies the same way)."""
    P = ctypes.c_void_p
    lib.oracle_paged_attention_decode.argtypes = [
        P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_double]
    lib.oracle_paged_attention_decode.restype = ctypes.c_int
    lib.oracle_paged_attention_decode_rows.argtypes = [
        P, P, P, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_double, P, P, ctypes.c_int]
    lib.oracle_paged_attention_decode_rows.restype = ctypes.c_int
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_num_threads.restype = None
    return lib


class OracleError(RuntimeError):
    pass


def _half_bits(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    if a.dtype == np.uint16:
        return a
    raise TypeError("expected float16 (or its uint16 bits), got %s" % a.dtype)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def half_to_double(bits: int) -> float:
    """The C oracle's binary16 -> binary64 widening of one bit pattern."""
    return _load().oracle_half_to_double(int(bits) & 0xFFFF)


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Threads the oracle's later calls use (OpenMP)."""
    _load().oracle_set_num_threads(int(n))


def paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale):
    """fp64 out[S, Hq, D] = softmax(scale * q K^T) V over context_lens[s] tokens.

    q: fp16 [S, Hq, D]; k_cache/v_cache: fp16 [num_blocks, bs, Hkv, D];
    block_tables: int32 [S, max_blocks]; context_lens: int32 [S].
    """
    qb, kb, vb = _half_bits(q), _half_bits(k_cache), _half_bits(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, Hq, D = qb.shape
    num_blocks, bs, Hkv, D2 = kb.shape
    if D2 != D or vb.shape != kb.shape or bt.shape[0] != S or cl.shape != (S,):
        raise ValueError("shape mismatch")
    out = np.zeros((S, Hq, D), dtype=np.float64)
    rc = _load().oracle_paged_attention_decode(
        _ptr(out), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(bt), _ptr(cl), S, Hq, Hkv, D, bs,
        num_blocks, bt.shape[1], float(scale))
    if rc != 0:
        raise OracleError("oracle status %d" % rc)
    return out


def paged_attention_decode_rows(q, k_cache, v_cache, block_tables, context_lens, scale,
                                seq_idx, head_idx):
    """The same definition evaluated only at rows (seq_idx[i], head_idx[i])."""
    qb, kb, vb = _half_bits(q), _half_bits(k_cache), _half_bits(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    si = np.ascontiguousarray(seq_idx, dtype=np.int32)
    hi = np.ascontiguousarray(head_idx, dtype=np.int32)
    S, Hq, D = qb.shape
    num_blocks, bs, Hkv, _ = kb.shape
    out = np.zeros((len(si), D), dtype=np.float64)
    rc = _load().oracle_paged_attention_decode_rows(
        _ptr(out), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(bt), _ptr(cl), S, Hq, Hkv, D, bs,
        num_blocks, bt.shape[1], float(scale), _ptr(si), _ptr(hi), len(si))
    if rc != 0:
        raise OracleError("oracle status %d" % rc)
    return out


def paged_attention_gather_concat(q, k_cache, v_cache, block_tables, context_lens, scale):
    """Pure-NumPy fp64 form for tiny inputs (gather blocks, concatenate, attend)."""
    q = np.asarray(q, dtype=np.float16).astype(np.float64)
    kc = np.asarray(k_cache, dtype=np.float16)
    vc = np.asarray(v_cache, dtype=np.float16)
    S, Hq, D = q.shape
    _, bs, Hkv, _ = kc.shape
    group = Hq // Hkv
    out = np.zeros((S, Hq, D), dtype=np.float64)
    for s in range(S):
        L = int(context_lens[s])
        if L == 0:
            continue
        n_logical = -(-L // bs)
        keys = np.concatenate([kc[int(block_tables[s][i])] for i in range(n_logical)], axis=0)
        values = np.concatenate([vc[int(block_tables[s][i])] for i in range(n_logical)], axis=0)
        keys = keys[:L].astype(np.float64)      # [L, Hkv, D]
        values = values[:L].astype(np.float64)
        for h in range(Hq):
            g = h // group
            logits = scale * (keys[:, g, :] @ q[s, h])
            w = np.exp(logits - logits.max())
            w /= w.sum()
            out[s, h] = w @ values[:, g, :]
    return out
