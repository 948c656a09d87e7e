"""Python face of the libpagedkv kernels: torch tensors in, C-ABI call out.

Every function here only checks shapes and dtypes and marshals pointers; all
computation runs in the CUDA kernels of libpagedkv.so.  Device tensors must be
contiguous and live on the current CUDA device; work is enqueued on the current
torch stream unless ``stream`` (a torch.cuda.Stream or raw handle) is given.
"""
import ctypes

import torch

from ._lib import check, lib

HEAD_DIM = 128
BLOCK_SIZE = 16


def _stream_handle(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _dev(t, name, dtype, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if ndim is not None and t.dim() != ndim:
        raise ValueError("%s must have %d dims, got %s" % (name, ndim, tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


class PreparedLaunch:
    """One C-ABI launch whose arguments were checked and marshalled once.

    Calling it enqueues the same launch again: same tensors (their current
    contents), same stream.  It keeps those tensors alive.  The per-call cost
    is the C call alone, for loops that relaunch on fixed buffers (the
    ``prepare=True`` form of the launch functions below)."""

    __slots__ = ("_fn", "_args", "_what", "_keep")

    def __init__(self, fn, args, what, keep):
        self._fn, self._args, self._what, self._keep = fn, args, what, keep

    def __call__(self):
        rc = self._fn(*self._args)
        if rc != 0:
            check(rc, self._what)


def _issue(fn, args, what, keep, prepare, result):
    if prepare:
        return PreparedLaunch(fn, args, what, keep)
    check(fn(*args), what)
    return result


def fill_normal(t, seed, offset, stream=None):
    """Fill fp16 tensor ``t`` (contiguous, 16-byte aligned) with standard-normal
    values: elements offset .. offset + numel - 1 of the device stream keyed by
    ``seed`` (``pkv_fill_normal_f16``).  Returns the offset after them."""
    _dev(t, "t", torch.float16)
    n = t.numel()
    check(lib().pkv_fill_normal_f16(_ptr(t), n, ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF),
                                    ctypes.c_uint64(offset), _stream_handle(stream)),
          "pkv_fill_normal_f16")
    return offset + n


def new_error_word(device=None):
    """A zeroed device int32 for the kernels' first-error code."""
    return torch.zeros(1, dtype=torch.int32, device=device or torch.cuda.current_device())


def read_error_word(dev_err):
    """Synchronise and return the device error code (0 = none)."""
    torch.cuda.current_stream().synchronize()
    return int(dev_err.item())


def workspace_bytes(num_seqs, num_q_heads, max_blocks_per_seq, block_size=BLOCK_SIZE,
                    head_dim=HEAD_DIM):
    """Bytes of split-K partials paged_attention_decode may need (an upper
    bound over the split lengths a launch of these sizes can choose)."""
    return int(lib().pkv_paged_attention_workspace_bytes(num_seqs, num_q_heads,
                                                         max_blocks_per_seq, block_size,
                                                         head_dim))


def split_tokens(num_seqs, num_kv_heads, max_blocks_per_seq, block_size=BLOCK_SIZE):
    """Split length (tokens) the attention launches use for these sizes."""
    t = lib().pkv_paged_attention_split_tokens(num_seqs, num_kv_heads, max_blocks_per_seq,
                                               block_size)
    if t < 0:
        check(t, "pkv_paged_attention_split_tokens")
    return t


def alloc_workspace(num_seqs, num_q_heads, max_blocks_per_seq, device=None,
                    block_size=BLOCK_SIZE):
    """A device buffer of workspace_bytes (None when no split is possible)."""
    n = workspace_bytes(num_seqs, num_q_heads, max_blocks_per_seq, block_size)
    if n == 0:
        return None
    return torch.empty(n, dtype=torch.uint8, device=device or torch.cuda.current_device())


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                           workspace=None, dev_err=None, stream=None, prepare=False):
    """out[s,h] = softmax(scale * q[s,h] . K_s^T) V_s over context_lens[s] tokens.
    prepare=True returns a PreparedLaunch instead of launching."""
    _dev(q, "q", torch.float16, 3)
    _dev(out, "out", torch.float16, 3)
    _dev(k_cache, "k_cache", torch.float16, 4)
    _dev(v_cache, "v_cache", torch.float16, 4)
    _dev(block_tables, "block_tables", torch.int32, 2)
    _dev(context_lens, "context_lens", torch.int32, 1)
    S, Hq, D = q.shape
    nb, bs, Hkv, D2 = k_cache.shape
    if out.shape != q.shape or v_cache.shape != k_cache.shape or D2 != D:
        raise ValueError("shape mismatch")
    if block_tables.shape[0] != S or context_lens.shape[0] != S:
        raise ValueError("block_tables / context_lens must have num_seqs rows")
    max_blocks = block_tables.shape[1]
    need = workspace_bytes(S, Hq, max_blocks, bs, D)
    if need and workspace is None:
        workspace = alloc_workspace(S, Hq, max_blocks, q.device, bs)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = (_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
            _ptr(context_lens), S, Hq, Hkv, D, bs, nb, max_blocks, float(scale), _ptr(workspace),
            ws_bytes, _ptr(dev_err), _stream_handle(stream))
    keep = (out, q, k_cache, v_cache, block_tables, context_lens, workspace, dev_err, stream)
    return _issue(lib().pkv_paged_attention_decode, args, "paged_attention_decode", keep, prepare,
                  out)


def paged_attention_decode_fused(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                                 context_lens, scale, workspace=None, dev_err=None, stream=None,
                                 prepare=False, cow=None):
    """One launch: store k_new[s]/v_new[s] at position context_lens[s] - 1 of each
    sequence (slot from its block table) and attend over context_lens[s] tokens.
    cow=(cow_block, cow_src) (int32 [S] device tensors, see cow_targets) also
    makes each sequence's copy-on-write copy in the same launch.
    prepare=True returns a PreparedLaunch instead of launching."""
    _dev(q, "q", torch.float16, 3)
    _dev(out, "out", torch.float16, 3)
    _dev(k_new, "k_new", torch.float16, 3)
    _dev(v_new, "v_new", torch.float16, 3)
    _dev(k_cache, "k_cache", torch.float16, 4)
    _dev(v_cache, "v_cache", torch.float16, 4)
    _dev(block_tables, "block_tables", torch.int32, 2)
    _dev(context_lens, "context_lens", torch.int32, 1)
    S, Hq, D = q.shape
    nb, bs, Hkv, D2 = k_cache.shape
    if out.shape != q.shape or v_cache.shape != k_cache.shape or D2 != D:
        raise ValueError("shape mismatch")
    if k_new.shape != (S, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [num_seqs, num_kv_heads, head_dim]")
    max_blocks = block_tables.shape[1]
    need = workspace_bytes(S, Hq, max_blocks, bs, D)
    if need and workspace is None:
        workspace = alloc_workspace(S, Hq, max_blocks, q.device, bs)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if cow is not None:
        cb, cs = _cow_args(cow, S)
        args = (_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                _ptr(block_tables), _ptr(context_lens), _ptr(cb), _ptr(cs), S, Hq, Hkv, D, bs,
                nb, max_blocks, float(scale), _ptr(workspace), ws_bytes, _ptr(dev_err),
                _stream_handle(stream))
        keep = (out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, cb, cs,
                workspace, dev_err, stream)
        return _issue(lib().pkv_paged_attention_decode_fused_cow, args,
                      "paged_attention_decode_fused_cow", keep, prepare, out)
    args = (_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
            _ptr(block_tables), _ptr(context_lens), S, Hq, Hkv, D, bs, nb, max_blocks,
            float(scale), _ptr(workspace), ws_bytes, _ptr(dev_err), _stream_handle(stream))
    keep = (out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, workspace,
            dev_err, stream)
    return _issue(lib().pkv_paged_attention_decode_fused, args, "paged_attention_decode_fused",
                  keep, prepare, out)


def _cow_args(cow, S):
    cb, cs = cow
    _dev(cb, "cow_block", torch.int32, 1)
    _dev(cs, "cow_src", torch.int32, 1)
    if cb.shape[0] != S or cs.shape[0] != S:
        raise ValueError("cow_block / cow_src must be int32 [num_seqs]")
    return cb, cs


def cow_targets(pairs, block_tables):
    """Host (native): copy-on-write pairs (src, dst) -> (cow_block, cow_src),
    int32 [S] numpy arrays for the fused launches' ``cow`` argument: the logical
    block of each sequence whose table holds a pair's dst, and that pair's src
    (-1 where none).  Raises PagedKVError (UNSUPPORTED) if a sequence needs
    two copies in one step."""
    import numpy as np
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    S = tables.shape[0]
    cb = np.empty(max(S, 1), np.int32)
    cs = np.empty(max(S, 1), np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    rc = lib().pkv_cow_targets(p(pr), pr.shape[0], p(tables), S, tables.shape[1], p(cb), p(cs))
    check(rc, "cow_targets")
    return cb[:S], cs[:S]


def reshape_and_cache(k, v, slot_mapping, k_cache, v_cache, dev_err=None, stream=None,
                      prepare=False):
    """k_cache[slot // bs, slot % bs] = k[i] (and v) for slot = slot_mapping[i] >= 0.
    prepare=True returns a PreparedLaunch instead of launching."""
    _dev(k, "k", torch.float16, 3)
    _dev(v, "v", torch.float16, 3)
    _dev(slot_mapping, "slot_mapping", torch.int64, 1)
    _dev(k_cache, "k_cache", torch.float16, 4)
    _dev(v_cache, "v_cache", torch.float16, 4)
    T, Hkv, D = k.shape
    nb, bs, Hkv2, D2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or (Hkv2, D2) != (Hkv, D):
        raise ValueError("shape mismatch")
    if slot_mapping.shape[0] != T:
        raise ValueError("slot_mapping must have one entry per token")
    args = (_ptr(k), _ptr(v), _ptr(slot_mapping), _ptr(k_cache), _ptr(v_cache), T, Hkv, D, bs,
            nb, _ptr(dev_err), _stream_handle(stream))
    keep = (k, v, slot_mapping, k_cache, v_cache, dev_err, stream)
    return _issue(lib().pkv_reshape_and_cache, args, "reshape_and_cache", keep, prepare, None)


def slot_mapping(block_tables, positions, num_blocks, block_size=BLOCK_SIZE, out=None,
                 dev_err=None, stream=None):
    """slot[s] = table[s][p // bs] * bs + p % bs with p = positions[s] (device)."""
    _dev(block_tables, "block_tables", torch.int32, 2)
    _dev(positions, "positions", torch.int32, 1)
    S, mb = block_tables.shape
    if out is None:
        out = torch.empty(S, dtype=torch.int64, device=block_tables.device)
    _dev(out, "out", torch.int64, 1)
    rc = lib().pkv_slot_mapping(_ptr(block_tables), _ptr(positions), S, mb, block_size,
                                int(num_blocks), _ptr(out), _ptr(dev_err), _stream_handle(stream))
    check(rc, "slot_mapping")
    return out


def copy_blocks(k_caches, v_caches, block_pairs, dev_err=None, stream=None):
    """cache[dst] = cache[src] for every (src, dst) row of block_pairs, every layer."""
    if isinstance(k_caches, torch.Tensor):
        k_caches, v_caches = [k_caches], [v_caches]
    if len(k_caches) != len(v_caches) or not k_caches:
        raise ValueError("need matching, non-empty lists of K and V caches")
    _dev(block_pairs, "block_pairs", torch.int64, 2)
    ref = k_caches[0]
    for c in list(k_caches) + list(v_caches):
        _dev(c, "cache", ref.dtype)
        if c.shape != ref.shape:
            raise ValueError("all caches must share one shape")
    n = len(k_caches)
    kp = (ctypes.c_void_p * n)(*[c.data_ptr() for c in k_caches])
    vp = (ctypes.c_void_p * n)(*[c.data_ptr() for c in v_caches])
    block_bytes = ref[0].numel() * ref.element_size()
    rc = lib().pkv_copy_blocks(kp, vp, n, _ptr(block_pairs), block_pairs.shape[0], block_bytes,
                               ref.shape[0], _ptr(dev_err), _stream_handle(stream))
    check(rc, "copy_blocks")


def swap_blocks(src_pools, dst_pools, block_pairs, dev_err=None, stream=None):
    """dst_pools[i][dst] = src_pools[i][src] for every (src, dst) row of block_pairs.

    Pools are tensors of one shape per side ([num_blocks, ...]); either side may
    be pinned host memory (``tensor.is_pinned()``), which the kernel reads or
    writes over the host link.  block_pairs must be readable by the GPU (a CUDA
    tensor or pinned host memory)."""
    if isinstance(src_pools, torch.Tensor):
        src_pools, dst_pools = [src_pools], [dst_pools]
    if len(src_pools) != len(dst_pools) or not src_pools:
        raise ValueError("need matching, non-empty lists of source and destination pools")
    for side in (src_pools, dst_pools):
        for t in side:
            if not (t.is_cuda or t.is_pinned()):
                raise TypeError("pools must be CUDA tensors or pinned host tensors")
            if not t.is_contiguous() or t.shape[1:] != side[0].shape[1:]:
                raise ValueError("pools of one side must be contiguous with one shape")
    if src_pools[0][0].numel() * src_pools[0].element_size() != \
            dst_pools[0][0].numel() * dst_pools[0].element_size():
        raise ValueError("source and destination blocks differ in size")
    if block_pairs.dtype != torch.int64 or block_pairs.dim() != 2 or not \
            (block_pairs.is_cuda or block_pairs.is_pinned()):
        raise TypeError("block_pairs must be int64 [P, 2] on the GPU or pinned")
    n = len(src_pools)
    sp = (ctypes.c_void_p * n)(*[t.data_ptr() for t in src_pools])
    dp = (ctypes.c_void_p * n)(*[t.data_ptr() for t in dst_pools])
    block_bytes = src_pools[0][0].numel() * src_pools[0].element_size()
    rc = lib().pkv_swap_blocks(sp, dp, n, _ptr(block_pairs), block_pairs.shape[0], block_bytes,
                               src_pools[0].shape[0], dst_pools[0].shape[0], _ptr(dev_err),
                               _stream_handle(stream))
    check(rc, "swap_blocks")


def shared_prefix_groups(block_tables, context_lens, block_size=BLOCK_SIZE, group_size_limit=16):
    """Host planning of grouped attention (native): consecutive sequences whose
    tables start with the same physical block form a group (at most
    group_size_limit members); a group shares the longest run of leading blocks
    every member has in common with its first member, cut to a multiple of 16
    tokens and of the block size and to the shortest member's context.

    Returns (group_first int32 [G+1], seq_group int32 [S], group_shared int32
    [G], max_shared_tokens, max_own_tokens)."""
    import numpy as np
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    S = len(lens)
    first = np.empty(S + 1, np.int32)
    seq_group = np.empty(max(S, 1), np.int32)
    shared = np.empty(max(S, 1), np.int32)
    ng, ms, mo = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    rc = lib().pkv_plan_shared_prefix_groups(
        p(tables), p(lens), S, tables.shape[1] if tables.ndim == 2 else 1, int(block_size),
        int(group_size_limit), p(first), p(seq_group), p(shared), ctypes.byref(ng),
        ctypes.byref(ms), ctypes.byref(mo))
    check(rc, "plan_shared_prefix_groups")
    n = ng.value
    return first[:n + 1], seq_group[:S], shared[:n], ms.value, mo.value


def grouped_workspace_bytes(num_seqs, num_q_heads, max_blocks_per_seq, max_shared_tokens,
                            block_size=BLOCK_SIZE, head_dim=HEAD_DIM):
    """Workspace bytes of the grouped entry points: the split-K bound plus the
    partial slots of shared prefixes up to max_shared_tokens."""
    return int(lib().pkv_paged_attention_grouped_workspace_bytes(
        num_seqs, num_q_heads, max_blocks_per_seq, block_size, head_dim, max_shared_tokens))


def paged_attention_decode_grouped(out, q, k_cache, v_cache, block_tables, context_lens,
                                   group_first, seq_group, group_shared, max_shared_tokens,
                                   max_own_tokens, scale, workspace=None, dev_err=None,
                                   stream=None, prepare=False):
    """Same result as paged_attention_decode; each group's shared prefix is read
    once for all its members (see shared_prefix_groups).  prepare=True returns a
    PreparedLaunch instead of launching."""
    _dev(q, "q", torch.float16, 3)
    _dev(out, "out", torch.float16, 3)
    _dev(k_cache, "k_cache", torch.float16, 4)
    _dev(v_cache, "v_cache", torch.float16, 4)
    _dev(block_tables, "block_tables", torch.int32, 2)
    _dev(context_lens, "context_lens", torch.int32, 1)
    for name, t in (("group_first", group_first), ("seq_group", seq_group),
                    ("group_shared", group_shared)):
        _dev(t, name, torch.int32, 1)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    G = group_shared.shape[0]
    if group_first.shape[0] != G + 1 or seq_group.shape[0] != S:
        raise ValueError("group arrays do not match")
    max_blocks = block_tables.shape[1]
    need = grouped_workspace_bytes(S, Hq, max_blocks, int(max_shared_tokens), bs, D)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = (_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
            _ptr(context_lens), _ptr(group_first), _ptr(seq_group), _ptr(group_shared), G,
            int(max_shared_tokens), int(max_own_tokens), S, Hq, Hkv, D, bs, nb, max_blocks,
            float(scale), _ptr(workspace), ws_bytes, _ptr(dev_err), _stream_handle(stream))
    keep = (out, q, k_cache, v_cache, block_tables, context_lens, group_first, seq_group,
            group_shared, workspace, dev_err, stream)
    return _issue(lib().pkv_paged_attention_decode_grouped, args,
                  "paged_attention_decode_grouped", keep, prepare, out)


def paged_attention_decode_grouped_fused(out, q, k_new, v_new, k_cache, v_cache, block_tables,
                                         context_lens, group_first, seq_group, group_shared,
                                         max_shared_tokens, max_own_tokens, scale,
                                         workspace=None, dev_err=None, stream=None,
                                         prepare=False, cow=None):
    """One launch: store k_new[s]/v_new[s] at position context_lens[s] - 1 of each
    sequence (a block past its group's shared prefix) and attend as
    paged_attention_decode_grouped.  cow=(cow_block, cow_src) also makes the
    copy-on-write copies in the same launch (see paged_attention_decode_fused)."""
    _dev(q, "q", torch.float16, 3)
    _dev(out, "out", torch.float16, 3)
    _dev(k_new, "k_new", torch.float16, 3)
    _dev(v_new, "v_new", torch.float16, 3)
    _dev(k_cache, "k_cache", torch.float16, 4)
    _dev(v_cache, "v_cache", torch.float16, 4)
    _dev(block_tables, "block_tables", torch.int32, 2)
    _dev(context_lens, "context_lens", torch.int32, 1)
    for name, t in (("group_first", group_first), ("seq_group", seq_group),
                    ("group_shared", group_shared)):
        _dev(t, name, torch.int32, 1)
    S, Hq, D = q.shape
    nb, bs, Hkv, _ = k_cache.shape
    if k_new.shape != (S, Hkv, D) or v_new.shape != k_new.shape:
        raise ValueError("k_new / v_new must be [num_seqs, num_kv_heads, head_dim]")
    G = group_shared.shape[0]
    if group_first.shape[0] != G + 1 or seq_group.shape[0] != S:
        raise ValueError("group arrays do not match")
    max_blocks = block_tables.shape[1]
    need = grouped_workspace_bytes(S, Hq, max_blocks, int(max_shared_tokens), bs, D)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    if cow is not None:
        cb, cs = _cow_args(cow, S)
        args = (_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                _ptr(block_tables), _ptr(context_lens), _ptr(group_first), _ptr(seq_group),
                _ptr(group_shared), G, int(max_shared_tokens), int(max_own_tokens), _ptr(cb),
                _ptr(cs), S, Hq, Hkv, D, bs, nb, max_blocks, float(scale), _ptr(workspace),
                ws_bytes, _ptr(dev_err), _stream_handle(stream))
        keep = (out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, group_first,
                seq_group, group_shared, cb, cs, workspace, dev_err, stream)
        return _issue(lib().pkv_paged_attention_decode_grouped_fused_cow, args,
                      "paged_attention_decode_grouped_fused_cow", keep, prepare, out)
    args = (_ptr(out), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
            _ptr(block_tables), _ptr(context_lens), _ptr(group_first), _ptr(seq_group),
            _ptr(group_shared), G, int(max_shared_tokens), int(max_own_tokens), S, Hq, Hkv, D,
            bs, nb, max_blocks, float(scale), _ptr(workspace), ws_bytes, _ptr(dev_err),
            _stream_handle(stream))
    keep = (out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, group_first,
            seq_group, group_shared, workspace, dev_err, stream)
    return _issue(lib().pkv_paged_attention_decode_grouped_fused, args,
                  "paged_attention_decode_grouped_fused", keep, prepare, out)
