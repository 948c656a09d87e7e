"""The attention oracle's pins catch plausible mistakes.

Each mutant is a copy of the C oracle's source with one textual mistake of
the kind a restatement of the definition could contain (a dropped scale, an
off-by-one length, a wrong GQA head map, a wrong row inside a block, V read
from the K cache, a missing softmax normalisation, the wrong query head, a
wrong subnormal exponent).  It is compiled with the oracle's own flags into a
temporary directory and bound in place of the oracle for one test; that test
requires at least one pin of test_oracle_attention to fail on it.  The
unmodified copy, built the same way, must pass every pin.  The oracle's own
source and library are never modified.
"""
import ctypes
import os
import subprocess

import pytest

import test_oracle_attention as pins
from conftest import ROOT
from oracle import attention as oa

SRC = os.path.join(ROOT, "oracle", "paged_attention_ref.c")

MUTANTS = {
    "dropped scale": ("score[t] = scale * acc;", "score[t] = acc;"),
    "one token short": ("const int L = context_lens[s];", "const int L = context_lens[s] - 1;"),
    "GQA head map": ("const int g = h / group;", "const int g = h % Hkv;"),
    "K rows reversed in a block": (
        "const uint16_t* krow = k_cache + (((int64_t)b * bs + t % bs) * Hkv + g) * D;",
        "const uint16_t* krow = k_cache + (((int64_t)b * bs + (bs - 1 - t % bs)) * Hkv + g) * D;"),
    "V read from the K cache": ("const uint16_t* vrow = v_cache +",
                                "const uint16_t* vrow = k_cache +"),
    "unnormalised softmax": ("for (int t = 0; t < L; ++t) score[t] /= z;", ""),
    "wrong query head": ("const uint16_t* qrow = q + ((int64_t)s * Hq + h) * D;",
                         "const uint16_t* qrow = q + ((int64_t)s * Hq + (Hq - 1 - h)) * D;"),
    "subnormal widening": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
}

# the pins, with the arguments of one of their parametrised cases each
PINS = [
    ("binary16 widening", pins.test_half_widening_all_patterns, ()),
    ("torch sdpa, MHA", pins.test_identity_table_matches_torch_sdpa, (4, 4)),
    ("torch sdpa, GQA", pins.test_identity_table_matches_torch_sdpa, (8, 2)),
    ("gather-concat", pins.test_c_oracle_matches_gather_concat, (2, 4, 1, [1, 2, 17, 33])),
    ("gather-concat, GQA", pins.test_c_oracle_matches_gather_concat,
     (3, 8, 2, [0, 5, 64, 100])),
    ("closed forms", pins.test_closed_forms, ()),
]


def build_copy(tmp_path, mutation=None):
    src = open(SRC).read()
    if mutation is not None:
        old, new = mutation
        assert src.count(old) == 1, "mutation site not unique: %r" % old
        src = src.replace(old, new)
    path = tmp_path / "oracle_copy.c"
    path.write_text(src)
    lib = tmp_path / "liboracle_copy.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
                    "-ffp-contract=off", str(path), "-o", str(lib), "-lm"], check=True)
    return oa.bind(ctypes.CDLL(str(lib)))


def failing_pins(monkeypatch, lib):
    monkeypatch.setattr(oa, "_lib", lib)
    failed = []
    for name, fn, args in PINS:
        try:
            fn(*args)
        except (AssertionError, oa.OracleError):
            failed.append(name)
    return failed


def test_unmutated_copy_passes_every_pin(tmp_path, monkeypatch):
    assert failing_pins(monkeypatch, build_copy(tmp_path)) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_every_mutant_fails_a_pin(tmp_path, monkeypatch, name):
    failed = failing_pins(monkeypatch, build_copy(tmp_path, MUTANTS[name]))
    assert failed, "the mutant '%s' passed every pin" % name


# ---- the BlockManager oracle ----------------------------------------------------
import importlib.util  # noqa: E402

import test_oracle_block_manager as bm_pins  # noqa: E402

BM_SRC = os.path.join(ROOT, "oracle", "block_manager.py")

BM_MUTANTS = {
    "LIFO free list": ("b = self.free_blocks.popleft()", "b = self.free_blocks.pop()"),
    "forward-order free": ("for b in reversed(table):", "for b in table:"),
    "unconditional hash delete": (
        "            if self.hash_to_block.get(h) == b:\n                del self.hash_to_block[h]",
        "            self.hash_to_block.pop(h, None)"),
    "len // bs match limit": ("for h in chain[:(len(tokens) - 1) // bs]:",
                              "for h in chain[:len(tokens) // bs]:"),
    "evict the newest": ("b, _ = self.evictable.popitem(last=False)",
                         "b, _ = self.evictable.popitem(last=True)"),
    "no copy-on-write": ("        elif self.ref[table[-1]] > 1:", "        elif False:"),
    "a hit stays evictable": ("                del self.evictable[b]", "                pass"),
}

BM_PINS = [
    ("example 1", bm_pins.test_golden_replay, ("blockmanager_example1.json",)),
    ("example 2", bm_pins.test_golden_replay, ("blockmanager_example2.json",)),
    ("example 3", bm_pins.test_golden_replay, ("blockmanager_example3.json",)),
    ("eviction trace", bm_pins.test_golden_replay, ("blockmanager_eviction_trace.json",)),
    ("duplicate hash", bm_pins.test_golden_replay, ("blockmanager_duplicate_hash.json",)),
    ("key questions", bm_pins.test_key_questions, ()),
    ("allocate_requests tables", bm_pins.test_allocate_requests_tables, ()),
    ("self-check", bm_pins.test_self_check_shared_block_free_twice, ()),
    ("fork and copy-on-write", bm_pins.test_fork_and_copy_on_write, ()),
]


def load_bm_copy(tmp_path, mutation=None):
    src = open(BM_SRC).read()
    if mutation is not None:
        old, new = mutation
        assert src.count(old) == 1, "mutation site not unique: %r" % old
        src = src.replace(old, new)
    path = tmp_path / "bm_copy.py"
    path.write_text(src)
    spec = importlib.util.spec_from_file_location("bm_copy_%d" % id(tmp_path), path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def failing_bm_pins(monkeypatch, mod):
    monkeypatch.setattr(bm_pins, "BlockManager", mod.BlockManager)
    monkeypatch.setattr(bm_pins, "OutOfBlocks", mod.OutOfBlocks)
    failed = []
    for name, fn, args in BM_PINS:
        try:
            fn(*args)
        except Exception:        # a wrong state, a wrong table or an unexpected raise
            failed.append(name)
    return failed


def test_unmutated_block_manager_copy_passes_every_pin(tmp_path, monkeypatch):
    assert failing_bm_pins(monkeypatch, load_bm_copy(tmp_path)) == []


@pytest.mark.parametrize("name", sorted(BM_MUTANTS))
def test_every_block_manager_mutant_fails_a_pin(tmp_path, monkeypatch, name):
    failed = failing_bm_pins(monkeypatch, load_bm_copy(tmp_path, BM_MUTANTS[name]))
    assert failed, "the mutant '%s' passed every pin" % name
