"""Replays a golden BlockManager fixture against any manager with the common API.

The adapter protocol: allocate(seq, tokens) -> table (raises on OutOfBlocks),
append_slot(seq, token) -> slot, free(seq), slot(seq, pos), num_free_blocks,
num_cached_tokens(seq), block_table(seq), free_list(), evictable_list(),
ref_counts().
"""


class OracleAdapter:
    """Gives the oracle BlockManager the introspection calls of the protocol."""

    def __init__(self, bm):
        self.bm = bm

    def __getattr__(self, name):
        return getattr(self.bm, name)

    @property
    def num_free_blocks(self):
        return self.bm.num_free_blocks

    def free_list(self):
        return list(self.bm.free_blocks)

    def evictable_list(self):
        return list(self.bm.evictable)

    def ref_counts(self):
        return list(self.bm.ref)


def replay(fixture, bm, out_of_blocks_exc, seq_id=lambda s: s, check=None):
    for step in fixture["ops"]:
        op = step["op"]
        seq = seq_id(step["seq"]) if "seq" in step else None
        if op == "allocate":
            if step["expect"] == "OutOfBlocks":
                before = (bm.free_list(), bm.evictable_list(), bm.ref_counts())
                try:
                    bm.allocate(seq, step["tokens"])
                except out_of_blocks_exc:
                    pass
                else:
                    raise AssertionError("expected OutOfBlocks at %r" % (step,))
                after = (bm.free_list(), bm.evictable_list(), bm.ref_counts())
                assert before == after, "state changed by a failed allocate"
            else:
                table = bm.allocate(seq, step["tokens"])
                assert list(table) == step["expect"], (step, table)
        elif op == "append_slot":
            slot = bm.append_slot(seq, step["token"])
            assert slot == step["expect"], (step, slot)
        elif op == "slot":
            assert bm.slot(seq, step["pos"]) == step["expect"], step
        elif op == "free":
            bm.free(seq)
        elif op == "num_free_blocks":
            assert bm.num_free_blocks == step["expect"], step
        else:
            raise ValueError(op)
        if "cached" in step:
            assert bm.num_cached_tokens(seq) == step["cached"], step
        if "num_free_blocks" in step:
            assert bm.num_free_blocks == step["num_free_blocks"], step
        if "free_list" in step:
            assert bm.free_list() == step["free_list"], (step, bm.free_list())
        if "free_list_len" in step:
            assert len(bm.free_list()) == step["free_list_len"], step
        if "evictable" in step:
            assert bm.evictable_list() == step["evictable"], (step, bm.evictable_list())
        if "table" in step:
            assert list(bm.block_table(seq)) == step["table"], step
        if "ref" in step:
            refs = "".join(str(r) for r in bm.ref_counts())
            assert refs == step["ref"], (step, refs)
        if check is not None:
            check(bm)
