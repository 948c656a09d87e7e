"""Seeded synthetic inputs for the paged decode hot path.

This module draws random numbers and lays them out; it holds none of the
method's arithmetic (no slot formula, no hashing, no attention).  Both the CUDA
path and the CPU oracle take their inputs from here.

Workloads (sizes from the project's benchmark configurations; every value is
synthetic, there is no dataset):

  tiny               5 sequences, lengths [7, 16, 31, 48, 63] (the length list of
                     "ans20xx day 31", `allocate_requests`), 8 heads MHA, pool of
                     64 blocks handed out from a shuffled FIFO free list
  llama2-13b-layer   64 sequences, lengths ~ U{1..4096}, 40 heads MHA, pool =
                     ceil(1.1 * blocks needed), shuffled
  gqa-32-8           256 sequences of exactly 4096 tokens, 32 query / 8 KV heads,
                     pool = ceil(1.1 * 65536), shuffled
  prefix-sharing     8 prompts of 2048 tokens, each forked into 16 samples that
                     share the prompt blocks; 64..512 private tokens per sample;
                     32 heads MHA
  llama2-7b-32layer  32 layers x 64 sequences x 4096 tokens, 32 heads MHA, one
                     table shared by all layers over 16384 blocks per layer
  llama2-7b-layer    one layer of that step (same shapes, 4 GiB of K+V): small
                     enough to profile where the 128 GiB step is not

Common: head_dim 128, block_size 16, q/K/V ~ N(0, 1) rounded to fp16, the new
token counted in the context length L (it is written at position L - 1 before
attention runs), seed = 1000 + the workload's number.
"""
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np

HEAD_DIM = 128
BLOCK_SIZE = 16


@dataclass
class Workload:
    name: str
    number: int
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    num_layers: int = 1
    head_dim: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    description: str = ""
    replica: int = 0     # independent copy of the workload (one per rank)

    @property
    def seed(self) -> int:
        return 1000 + self.number + 7919 * self.replica

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.head_dim))


WORKLOADS = {
    "tiny": Workload("tiny", 1, 5, 8, 8, description="5 seqs, L=[7,16,31,48,63], 8 heads MHA"),
    "llama2-13b-layer": Workload("llama2-13b-layer", 2, 64, 40, 40,
                                 description="Llama-2-13B layer, batch 64, L~U[1,4096], 40 heads MHA"),
    "gqa-32-8": Workload("gqa-32-8", 3, 256, 32, 8,
                         description="GQA 32q/8kv, batch 256, L=4096"),
    "prefix-sharing": Workload("prefix-sharing", 4, 128, 32, 32,
                               description="8 prompts x 2048 tok forked x16, +64..512 private tok"),
    "llama2-7b-32layer": Workload("llama2-7b-32layer", 5, 64, 32, 32, num_layers=32,
                                  description="Llama-2-7B full step, 32 layers, batch 64 x 4096"),
    "llama2-7b-layer": Workload("llama2-7b-layer", 6, 64, 32, 32,
                                description="one layer of the Llama-2-7B step, batch 64 x 4096"),
}


def rng_for(w: Workload, stream: int = 0) -> np.random.Generator:
    return np.random.default_rng([w.seed, stream])


def blocks_for(length: int, block_size: int = BLOCK_SIZE) -> int:
    """Blocks that hold ``length`` tokens (ceiling division)."""
    return -(-int(length) // block_size)


def context_lengths(w: Workload) -> np.ndarray:
    """Context length per sequence, new token included (int32 [S])."""
    rng = rng_for(w, 1)
    if w.name == "tiny":
        return np.array([7, 16, 31, 48, 63], dtype=np.int32)
    if w.name == "llama2-13b-layer":
        return rng.integers(1, 4096, size=w.num_seqs, endpoint=True).astype(np.int32)
    if w.name in ("gqa-32-8", "llama2-7b-32layer", "llama2-7b-layer"):
        return np.full(w.num_seqs, 4096, dtype=np.int32)
    if w.name == "prefix-sharing":
        p = prefix_sharing_private_tokens(w)
        return (2048 + 1 + p).astype(np.int32)
    raise KeyError(w.name)


def pool_blocks(w: Workload, lengths: Optional[np.ndarray] = None) -> int:
    """Physical blocks in the pool for workload ``w``."""
    if w.name == "tiny" and w.block_size == BLOCK_SIZE:
        return 64
    if w.name in ("llama2-7b-32layer", "llama2-7b-layer"):
        return w.num_seqs * blocks_for(4096, w.block_size)
    if w.name == "prefix-sharing":
        p = prefix_sharing_private_tokens(w)
        unique = 8 * blocks_for(2048) + sum(blocks_for(1 + int(x)) for x in p)
        return int(np.ceil(1.1 * unique))
    if w.name == "tiny" and w.block_size != BLOCK_SIZE:
        return 64 * BLOCK_SIZE // w.block_size
    lengths = context_lengths(w) if lengths is None else lengths
    return int(np.ceil(1.1 * sum(blocks_for(int(L), w.block_size) for L in lengths)))


def free_order(w: Workload, num_blocks: Optional[int] = None) -> np.ndarray:
    """Seed-shuffled initial free list: random physical placement of blocks."""
    n = pool_blocks(w) if num_blocks is None else num_blocks
    return rng_for(w, 2).permutation(n).astype(np.int32)


def handout_tables(lengths, order, block_size: int = BLOCK_SIZE,
                   max_blocks: Optional[int] = None, pad: int = -1) -> np.ndarray:
    """Give sequence i the next blocks_for(L_i) entries of ``order`` (FIFO hand-out).

    Returns int32 [S, max_blocks]; entries past a sequence's blocks hold ``pad``.
    """
    need = [blocks_for(int(L), block_size) for L in lengths]
    mb = max(need + [1]) if max_blocks is None else max_blocks
    tables = np.full((len(lengths), mb), pad, dtype=np.int32)
    cursor = 0
    for i, n in enumerate(need):
        tables[i, :n] = order[cursor:cursor + n]
        cursor += n
    if cursor > len(order):
        raise ValueError("pool too small")
    return tables


def token_ids(w: Workload, count: int, stream: int = 3) -> np.ndarray:
    """Random token ids (int32) -- the content hashed by the prefix cache."""
    return rng_for(w, stream).integers(0, 32000, size=count).astype(np.int32)


def host_normal_fp16(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0, 1) samples rounded to fp16, on the host."""
    return rng.standard_normal(size=shape, dtype=np.float32).astype(np.float16)


def host_tensors(w: Workload, num_blocks: int, num_layers: int = 1):
    """q [S,Hq,D], k/v new tokens [S,Hkv,D] and caches [layers][nb,bs,Hkv,D] on host."""
    rng = rng_for(w, 4)
    S, Hq, Hkv, D, bs = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    q = host_normal_fp16(rng, (num_layers, S, Hq, D))
    k_new = host_normal_fp16(rng, (num_layers, S, Hkv, D))
    v_new = host_normal_fp16(rng, (num_layers, S, Hkv, D))
    k_cache = host_normal_fp16(rng, (num_layers, num_blocks, bs, Hkv, D))
    v_cache = host_normal_fp16(rng, (num_layers, num_blocks, bs, Hkv, D))
    return q, k_new, v_new, k_cache, v_cache


def device_normal_fp16_(t, seed: int, chunk_elems: int = 1 << 28):
    """Fill a CUDA fp16 tensor in place with N(0, 1) draws (torch generator)."""
    import torch
    g = torch.Generator(device=t.device)
    g.manual_seed(seed)
    flat = t.view(-1)
    for start in range(0, flat.numel(), chunk_elems):
        part = flat[start:start + chunk_elems]
        part.copy_(torch.randn(part.shape, generator=g, device=t.device, dtype=torch.float32))
    return t


# ---- prefix sharing / parallel sampling -------------------------------------------

PREFIX_PROMPTS = 8
PREFIX_PROMPT_TOKENS = 2048
PREFIX_SAMPLES = 16


def prefix_sharing_private_tokens(w: Workload) -> np.ndarray:
    """Private decoded tokens per sample after the fork, ~U{64..512}."""
    return rng_for(w, 5).integers(64, 512, size=PREFIX_PROMPTS * PREFIX_SAMPLES,
                                  endpoint=True).astype(np.int64)


@dataclass
class OpScript:
    """A sequence of BlockManager operations, as data.

    ``setup`` runs first; ``cow_step`` is the first post-fork append of every
    sample (the step whose copy-on-writes feed copy_blocks); ``fill`` appends the
    remaining private tokens but the last; ``step`` is the timed decode step (one
    append per sequence, in batch order).
    """
    setup: List[Tuple] = field(default_factory=list)
    cow_step: List[Tuple] = field(default_factory=list)
    fill: List[Tuple] = field(default_factory=list)
    step: List[Tuple] = field(default_factory=list)
    batch: List[int] = field(default_factory=list)


def prefix_sharing_script(w: Workload) -> OpScript:
    """8 prompts of 2048 random tokens; the parent of each appends one shared
    decoded token (opening a partial block), then is forked 15 times.  Each of the
    16 samples then decodes p_i private tokens; the first of those writes into
    the shared partial block.  Sequence id = prompt * 16 + sample; sample 0 is the
    parent."""
    p = prefix_sharing_private_tokens(w)
    toks = token_ids(w, PREFIX_PROMPTS * (PREFIX_PROMPT_TOKENS + 1) + int(p.sum()), stream=6)
    cur = 0
    sc = OpScript()
    for j in range(PREFIX_PROMPTS):
        parent = j * PREFIX_SAMPLES
        prompt = toks[cur:cur + PREFIX_PROMPT_TOKENS].tolist()
        cur += PREFIX_PROMPT_TOKENS
        sc.setup.append(("allocate", parent, prompt))
        sc.setup.append(("append", parent, int(toks[cur])))
        cur += 1
        for k in range(1, PREFIX_SAMPLES):
            sc.setup.append(("fork", parent, parent + k))
    seqs = list(range(PREFIX_PROMPTS * PREFIX_SAMPLES))
    sc.batch = seqs
    private = {}
    for s in seqs:
        private[s] = toks[cur:cur + int(p[s])].tolist()
        cur += int(p[s])
    sc.cow_step = [("append", s, private[s][0]) for s in seqs]
    for s in seqs:
        sc.fill.extend(("append", s, t) for t in private[s][1:-1])
    sc.step = [("append", s, private[s][-1]) for s in seqs]
    return sc


def decode_script(w: Workload, lengths) -> OpScript:
    """Plain decode batch: allocate L_i - 1 prompt tokens, then the timed step
    appends the new token of every sequence."""
    toks = token_ids(w, int(np.sum(lengths)), stream=3)
    sc = OpScript()
    cur = 0
    for s, L in enumerate(lengths):
        L = int(L)
        sc.setup.append(("allocate", s, toks[cur:cur + L - 1].tolist()))
        sc.step.append(("append", s, int(toks[cur + L - 1])))
        cur += L
    sc.batch = list(range(len(lengths)))
    return sc


# ---- content-keyed values for the multi-step driver ----------------------------------
# A decode step's K/V for a token must be a function of the tokens before it (as
# a model's would be), so that a block found again through the prefix cache
# holds the same values a fresh prefill would write.  Each prefix gets a 64-bit
# key (a multiply-xorshift chain over the token ids -- a random-number key, not
# the BlockManager's block hash) that seeds NumPy's generator.

_MIX = 0x9E3779B97F4A7C15
_MASK = (1 << 64) - 1


def prefix_keys(tokens, seed: int = 0) -> List[int]:
    """Key of every prefix tokens[:j + 1], j = 0 .. n - 1."""
    keys, h = [], (seed * _MIX + 0x632BE59BD9B4E019) & _MASK
    for t in tokens:
        h = ((h ^ (int(t) & 0xFFFFFFFF)) * _MIX) & _MASK
        h ^= h >> 29
        keys.append(h)
    return keys


def token_kv_host(keys, num_kv_heads: int, head_dim: int = HEAD_DIM):
    """fp16 K and V rows [n, Hkv, D] of the tokens whose prefix keys are given."""
    n = len(keys)
    k = np.empty((n, num_kv_heads, head_dim), dtype=np.float16)
    v = np.empty_like(k)
    for i, key in enumerate(keys):
        r = np.random.default_rng(key)
        k[i] = host_normal_fp16(r, (num_kv_heads, head_dim))
        v[i] = host_normal_fp16(r, (num_kv_heads, head_dim))
    return k, v


def step_query_host(seed: int, rid: int, pos: int, num_q_heads: int, head_dim: int = HEAD_DIM):
    """fp16 query [Hq, D] of request ``rid`` decoding position ``pos``."""
    return host_normal_fp16(np.random.default_rng([seed, rid, pos, 7]), (num_q_heads, head_dim))


def next_token_host(seed: int, rid: int, pos: int, vocab: int = 32000) -> int:
    """The token a request 'samples' at position ``pos`` (no model: random)."""
    return int(np.random.default_rng([seed, rid, pos, 11]).integers(0, vocab))


@dataclass
class RequestSpec:
    rid: int
    prompt: List[int]
    max_new_tokens: int
    arrival_step: int = 0


def serving_requests(seed: int, num_requests: int, num_system_prompts: int,
                     system_prompt_len: int, suffix_max: int, new_min: int, new_max: int,
                     arrivals_per_step: float = 0.0, vocab: int = 32000) -> List[RequestSpec]:
    """Synthetic serving trace: each prompt is one of a few shared system prompts
    followed by a private random suffix; output lengths ~U{new_min..new_max}."""
    rng = np.random.default_rng([seed, 21])
    systems = [rng.integers(0, vocab, size=system_prompt_len).tolist()
               for _ in range(num_system_prompts)]
    out = []
    for rid in range(num_requests):
        sys_p = systems[int(rng.integers(0, num_system_prompts))]
        suffix = rng.integers(0, vocab, size=int(rng.integers(1, suffix_max + 1))).tolist()
        arrive = int(rid / arrivals_per_step) if arrivals_per_step > 0 else 0
        out.append(RequestSpec(rid, sys_p + suffix, int(rng.integers(new_min, new_max + 1)),
                               arrive))
    return out
