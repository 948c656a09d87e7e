"""Inputs that make the softmax bookkeeping of the attention kernels matter.

With q, K ~ N(0, 1) and scale 1/sqrt(128) the logits of a context differ by a
few units at most, so a kernel's running maximum settles on its first tile and
a lazy rescale, or a merge of splits whose maxima lie far apart, never has
anything to do.  The builders here place the logits on purpose instead:

  q[s, h] = gain[h] / (scale * log2 e) * u_g          (u_g: a unit vector per KV head)
  K[t, g] = sigma * z_t + r_s(t) * u_g                  (z_t ~ N(0, 1)^128)

so that query head h sees the base-2 logit  gain[h] * (r_s(t) + sigma * n_t)  at
token t, with n_t ~ N(0, 1).  The profile r_s(t) is a ramp (logits climbing or,
for a negative gain, falling through the whole context), a valley, or a few
spikes that dominate every other token.  Mistakes in the rescale (alpha applied
to o but not to l, a stale maximum), in the cross-warp or cross-split merge
(weights not taken relative to the common maximum, a split dropped) or in the
row a token lands in then move the output by O(|V|) instead of O(1e-3).

V ~ N(0, 0.4^2) by default: outputs stay below 2 in magnitude, where the fp16
output rounding (at most 2^-11 relative) keeps a correct kernel well inside
the 2e-3 tolerance even when one token dominates; v_scale = 1 gives |V| up to
~4.5, where a kernel whose softmax sum and P.V weights disagree by an fp16
rounding (2^-11 relative) misses a dominant token's row by up to ~2e-3.

``tile_loop_rescales`` is a CPU emulation of the kernels' tile schedule (16-token
tiles, warp w of a split taking tiles w, w + 4, ..., a running maximum that moves
only when a tile's maximum exceeds it by more than 8 in log2 units); the CPU
tests use it to show that these inputs reach the rescale branch.
"""
import numpy as np

from paged_kv_cache_138_gb300 import workloads as wl

D = 128
LOG2E = 1.4426950408889634
V_SCALE = 0.4


def gains_for(G, kind="mixed"):
    """Per-query-head gains within one KV head's group of G heads."""
    if kind == "mixed":    # rising, falling, half and double slopes
        base = [1.0, -1.0, 0.5, 2.0, -0.5, -2.0, 1.5, 0.25]
    else:                  # all positive: spikes stay maxima for every head
        base = [1.0, 2.0, 1.5, 3.0, 1.25, 2.5, 1.75, 1.0]
    return np.array([base[i % len(base)] for i in range(G)])


def ramp(slope):
    return lambda L, t: slope * t


def valley(slope, centre_frac=0.5):
    return lambda L, t: slope * np.abs(t - int(centre_frac * L))


def spikes(points, base=0.0):
    """points: (position, height) pairs; negative positions count from L."""
    def f(L, t):
        r = np.full(t.shape, base, dtype=np.float64)
        for p, h in points:
            p = p + L if p < 0 else p
            if 0 <= p < L:
                r[t == p] = h
        return r
    return f


def build(seed, tables, lens, profiles, Hq, Hkv, nb, bs=16, gain_kind="mixed", sigma=1.0,
          scale=1.0 / np.sqrt(D), seq_factor=None, v_scale=V_SCALE):
    """q [S, Hq, D], k_cache / v_cache [nb, bs, Hkv, D] (fp16) for the given
    block tables and lengths; profiles[s](L, t) is sequence s's base-2 logit
    profile; query head h of sequence s has gain gains_for(G)[h % G] *
    seq_factor[s].  A physical slot read by several sequences (a shared
    prefix) takes the profile of the first sequence that reaches it.  Slots no
    sequence reads hold NaN."""
    rng = np.random.default_rng(seed)
    S = len(lens)
    G = Hq // Hkv
    u = rng.standard_normal((Hkv, D))
    u /= np.linalg.norm(u, axis=1, keepdims=True)
    kc = np.full((nb, bs, Hkv, D), np.nan)
    vc = np.full((nb, bs, Hkv, D), np.nan)
    seen = np.zeros((nb, bs), dtype=bool)
    for s in range(S):
        L = int(lens[s])
        if L == 0:
            continue
        t = np.arange(L)
        blk = tables[s][t // bs].astype(np.int64)
        off = t % bs
        new = ~seen[blk, off]
        t, blk, off = t[new], blk[new], off[new]
        r = profiles[s](L, np.arange(L))[new]
        z = rng.standard_normal((len(t), Hkv, D)) * sigma
        kc[blk, off] = z + r[:, None, None] * u[None]
        vc[blk, off] = rng.standard_normal((len(t), Hkv, D)) * v_scale
        seen[blk, off] = True
    gain = np.tile(gains_for(G, gain_kind), Hkv)              # [Hq]
    f = np.ones(S) if seq_factor is None else np.asarray(seq_factor, dtype=np.float64)
    q = ((f[:, None] * gain[None, :]) / (scale * LOG2E))[:, :, None] * \
        u[np.arange(Hq) // G][None]
    return q.astype(np.float16), kc.astype(np.float16), vc.astype(np.float16)


def plain_tables(seed, lengths, bs=16, extra=3):
    """Each sequence its own randomly placed blocks (as the tests' plain cases)."""
    rng = np.random.default_rng(seed)
    need = [wl.blocks_for(L, bs) for L in lengths]
    nb = sum(need) + extra
    order = rng.permutation(nb).astype(np.int32)
    tables = wl.handout_tables(lengths, order, block_size=bs)
    return tables, np.array(lengths, dtype=np.int32), nb


def forked_tables(seed, groups, prefix_tokens, own_lengths, bs=16):
    """groups: members per group; member i of the batch holds the group's
    prefix_tokens through shared blocks, then own_lengths[i] private tokens."""
    rng = np.random.default_rng(seed)
    rows, lens, nxt, i = [], [], 0, 0
    pb = prefix_tokens // bs
    for members in groups:
        prefix = list(range(nxt, nxt + pb))
        nxt += pb
        for _ in range(members):
            L = prefix_tokens + int(own_lengths[i])
            i += 1
            extra = wl.blocks_for(L, bs) - pb
            rows.append(prefix + list(range(nxt, nxt + extra)))
            nxt += extra
            lens.append(L)
    nb = nxt + 2
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.full((len(rows), max(len(r) for r in rows)), -1, np.int32)
    for j, r in enumerate(rows):
        tables[j, :len(r)] = perm[r]
    return tables, np.array(lens, np.int32), nb


def logits_log2(q, kc, tables, lens, scale, s, h, bs=16):
    """fp64 base-2 logits of query head h of sequence s over its context."""
    L = int(lens[s])
    Hq, Hkv = q.shape[1], kc.shape[2]
    g = h // (Hq // Hkv)
    t = np.arange(L)
    K = kc[tables[s][t // bs], t % bs, g].astype(np.float64)
    return scale * LOG2E * (K @ q[s, h].astype(np.float64))


def tile_loop_rescales(x, split_tokens, tile=16, warps=4, threshold=8.0, first_tile=0):
    """Emulate the kernels' running maximum over logits x (base 2) of one row.

    The context from tile first_tile on is cut into splits of split_tokens;
    within a split warp w takes tiles w, w + warps, ...  Returns (rescales,
    split_maxima): how many times a warp's running maximum moved after that
    warp's first tile (the lazy-rescale branch), and each split's maximum."""
    L = len(x)
    ntiles = -(-L // tile)
    per_split = split_tokens // tile
    rescales, maxima = 0, []
    for sb in range(first_tile, ntiles, per_split):
        se = min(ntiles, sb + per_split)
        maxima.append(float(x[sb * tile:min(L, se * tile)].max()))
        for w in range(warps):
            m = -np.inf
            for k, tix in enumerate(range(sb + w, se, warps)):
                bm = x[tix * tile:min(L, (tix + 1) * tile)].max()
                if bm > m + threshold:
                    rescales += k > 0
                    m = bm
    return rescales, maxima


def emulated_row(x, v, split_tokens, mistake=None, tile=16, warps=4, threshold=8.0):
    """fp64 model of how the kernels combine one row: per split, per warp a
    running (m, l, o) over the warp's tiles with the lazy rescale; the warps'
    states merged against their common maximum, then the splits' states merged
    the same way.  x: base-2 logits [L], v: V rows [L, D].  ``mistake`` plants
    one error a kernel could make, for the tests that show these inputs catch
    it: "no_l_rescale", "no_o_rescale", "merge_first_max" (splits weighted
    against the first split's maximum instead of the largest),
    "drop_last_split", "drop_last_token", "row_shift" (a tile's rows read one
    position late)."""
    def exp2(d):    # the kernels keep (m, l, o) in fp32: 2^d overflows past 128
        with np.errstate(over="ignore"):
            return float(np.exp2(np.float32(d)))

    L = len(x)
    if mistake == "drop_last_token":
        L -= 1
    ntiles = -(-L // tile)
    per_split = split_tokens // tile
    splits = []
    for sb in range(0, ntiles, per_split):
        se = min(ntiles, sb + per_split)
        states = []
        for w in range(warps):
            m, l, o = -np.inf, 0.0, np.zeros(v.shape[1])
            for tix in range(sb + w, se, warps):
                lo, hi = tix * tile, min(L, (tix + 1) * tile)
                xs, vs = x[lo:hi], v[lo:hi]
                if mistake == "row_shift" and hi < len(x):
                    vs = v[lo + 1:hi + 1]
                bm = xs.max()
                if bm > m + threshold:
                    alpha = exp2(m - bm) if m > -np.inf else 0.0
                    if mistake != "no_l_rescale":
                        l *= alpha
                    if mistake != "no_o_rescale":
                        o = o * alpha
                    m = bm
                p = 2.0 ** (xs - m)
                l += p.sum()
                o = o + p @ vs
            states.append((m, l, o))
        M = max(s[0] for s in states)
        c = [exp2(s[0] - M) if s[0] > -np.inf else 0.0 for s in states]
        splits.append((M, sum(ci * s[1] for ci, s in zip(c, states)),
                       sum(ci * s[2] for ci, s in zip(c, states))))
    if mistake == "drop_last_split" and len(splits) > 1:
        splits = splits[:-1]
    M = splits[0][0] if mistake == "merge_first_max" else max(s[0] for s in splits)
    with np.errstate(over="ignore", invalid="ignore"):
        c = [exp2(s[0] - M) for s in splits]
        num = sum(ci * s[2] for ci, s in zip(c, splits))
        den = sum(ci * s[1] for ci, s in zip(c, splits))
        return num / den
