"""The allocation-free attention entry point (pkv_paged_attention_decode_noalloc).

It serves callers that may not allocate device memory: a plugin inside a host
framework that owns the whole device memory pool, or a latency-critical path
that cannot afford an allocation's implicit device synchronisation.  Instead of
a caller workspace it uses a fixed 16 MiB scratch array inside the library.
These tests call it through the C ABI, twice in a row on different shapes (the
second call sees the first call's leftovers in the shared scratch), and require
its output to equal the workspace entry point's bit for bit (the same kernels
run the same split length over the same inputs) and to match the fp64 oracle
within the attention tolerance.  A call after a warm-up call must leave the
device's allocated memory unchanged.  This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import attention as oa
from parity_helpers import attention_tolerance
from paged_kv_cache_138_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
D = 128
SCRATCH_LIMIT = 16 << 20


def _case(seed, lengths, Hq, Hkv):
    rng = np.random.default_rng(seed)
    nb = sum(wl.blocks_for(L) for L in lengths) + 4
    tables = wl.handout_tables(lengths, rng.permutation(nb).astype(np.int32))
    q = wl.host_normal_fp16(rng, (len(lengths), Hq, D))
    kc = wl.host_normal_fp16(rng, (nb, 16, Hkv, D))
    vc = wl.host_normal_fp16(rng, (nb, 16, Hkv, D))
    dev = lambda a: torch.from_numpy(a).cuda()
    return dev(q), dev(kc), dev(vc), dev(tables), dev(np.array(lengths, np.int32))


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(lib, out, q, kc, vc, tables, lens, scale, err):
    S, Hq, _ = q.shape
    nb, bs, Hkv, _ = kc.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.pkv_paged_attention_decode_noalloc(
        _p(out), _p(q), _p(kc), _p(vc), _p(tables), _p(lens), S, Hq, Hkv, D, bs, nb,
        tables.shape[1], float(scale), _p(err), stream)


def test_noalloc_matches_workspace_entry_point(native_lib):
    from paged_kv_cache_138_gb300 import ops
    scale = 1.0 / np.sqrt(D)
    cases = [
        # long, ragged contexts so that several splits go through the scratch
        _case(1, [1, 700, 2049, 4096, 33, 1500], 32, 8),
        _case(2, [4096, 3000, 17, 512, 513, 999, 16], 40, 40),
    ]
    for q, kc, vc, tables, lens in cases:       # two calls in a row
        S, Hq, _ = q.shape
        assert ops.workspace_bytes(S, Hq, tables.shape[1]) > 0     # the scratch is used
        ref = torch.empty_like(q)
        ops.paged_attention_decode(ref, q, kc, vc, tables, lens, scale)
        out = torch.full_like(q, float("nan"))
        err = ops.new_error_word()
        rc = _noalloc(native_lib, out, q, kc, vc, tables, lens, scale, err)
        assert rc == 0
        assert ops.read_error_word(err) == 0
        # same kernels, same split length, same inputs: the same bits
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        oracle = oa.paged_attention_decode(q.cpu().numpy(), kc.cpu().numpy(), vc.cpu().numpy(),
                                           tables.cpu().numpy(), lens.cpu().numpy(), scale)
        diff = np.abs(out.cpu().numpy().astype(np.float64) - oracle).max()
        assert diff <= attention_tolerance(), diff


def test_noalloc_allocates_nothing(native_lib):
    from paged_kv_cache_138_gb300 import ops
    q, kc, vc, tables, lens = _case(3, [4096, 2500, 1, 700], 16, 4)
    out = torch.empty_like(q)
    err = ops.new_error_word()
    scale = 1.0 / np.sqrt(D)
    assert _noalloc(native_lib, out, q, kc, vc, tables, lens, scale, err) == 0   # warm-up
    torch.cuda.synchronize()
    torch_before = torch.cuda.memory_allocated()
    free_before = torch.cuda.mem_get_info()[0]
    assert _noalloc(native_lib, out, q, kc, vc, tables, lens, scale, err) == 0
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == torch_before
    assert torch.cuda.mem_get_info()[0] == free_before
    assert ops.read_error_word(err) == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(native_lib):
    from paged_kv_cache_138_gb300 import ops
    S, Hq, max_blocks = 4096, 64, 256          # needs far more than 16 MiB
    assert ops.workspace_bytes(S, Hq, max_blocks) > SCRATCH_LIMIT
    q = torch.zeros((S, Hq, D), dtype=torch.float16, device="cuda")
    kc = torch.zeros((4, 16, 8, D), dtype=torch.float16, device="cuda")
    tables = torch.zeros((S, max_blocks), dtype=torch.int32, device="cuda")
    lens = torch.zeros(S, dtype=torch.int32, device="cuda")
    rc = _noalloc(native_lib, q, q, kc, kc, tables, lens, 0.1, None)
    assert rc == -2                             # PKV_ERR_UNSUPPORTED, nothing launched
