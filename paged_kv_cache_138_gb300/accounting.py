"""Byte accounting for the roofline: what a decode step must move at minimum.

"qaqbuyan: KV cache size" gives the cache size as 2 x layers x heads x head_dim
x tokens x bytes-per-element (the 2 is K and V).  A decode step reads the K and
V of every valid token of every sequence once; the unread tail of a partial
last block is not credited.
"""


def kv_cache_bytes(layers: int, heads: int, head_dim: int, tokens: int,
                   bytes_per_elem: int = 2) -> int:
    return 2 * layers * heads * head_dim * tokens * bytes_per_elem


def prefix_sharing_bytes(num_requests: int, prefix_tokens: int, layers: int, heads: int,
                         head_dim: int, bytes_per_elem: int = 2):
    """KV bytes of a prompt prefix held by num_requests requests: stored once
    per request, and stored once for all of them through shared blocks
    ("qaqbuyan: vLLM PagedAttention", the prefix-sharing example)."""
    one = kv_cache_bytes(layers, heads, head_dim, prefix_tokens, bytes_per_elem)
    return num_requests * one, one


def slot_utilization(tokens: int, reserved_tokens: int) -> float:
    """Share of reserved KV slots that hold tokens: a contiguous reservation of
    the maximum length ("qaqbuyan: vLLM PagedAttention", the pre-allocation
    example) against paging, whose reservation is ceil(tokens / bs) * bs."""
    return tokens / reserved_tokens if reserved_tokens else 0.0


def paged_reserved_tokens(tokens: int, block_size: int) -> int:
    return -(-int(tokens) // block_size) * block_size


def step_kv_bytes(context_lens, num_kv_heads: int, head_dim: int, layers: int = 1,
                  bytes_per_elem: int = 2) -> int:
    """Algorithmic K+V bytes one decode step reads (valid tokens only)."""
    tokens = int(sum(int(L) for L in context_lens))
    return kv_cache_bytes(layers, num_kv_heads, head_dim, tokens, bytes_per_elem)


def unique_kv_bytes(tables, context_lens, block_size: int, num_kv_heads: int,
                    head_dim: int, bytes_per_elem: int = 2) -> int:
    """K+V bytes of the distinct (block, row) slots a step reads.

    With prefix sharing several tables name the same physical block; HBM only
    has to deliver each shared row once if the cache (L2) keeps it.
    """
    slots = set()
    for table, L in zip(tables, context_lens):
        for t in range(int(L)):
            slots.add((int(table[t // block_size]), t % block_size))
    return len(slots) * 2 * num_kv_heads * head_dim * bytes_per_elem
