"""Pins for the oracle's legal set and transition (CPU only).

The walk in ``oracle.grammar`` (live pointers below an edge, the owed-pointer
rule for separator and stop, the spent flag) is checked against the mask
taken literally from its definition over the enumerated language
("GLRMask", introduction), on every reachable prefix of tiny catalogs, and
against hand-derived fixtures in tests/golden/walk_examples.json."""
import json
import os

import numpy as np
import pytest

from oracle import grammar as G
from oracle import language as L
from trie_constrained_decoding_gb300 import inputs as I
from conftest import GOLDEN


def _check_against_definition(cat, sep, stop, V, k):
    trie = G.compile_catalog(cat, sep, stop, V)
    lang = L.language(trie.catalog, k, sep, stop)
    assert lang, "k <= K gives a non-empty language"
    for u in L.reachable_prefixes(lang):
        st = G.walk(trie, u, k)
        assert st is not None, f"walk rejects reachable prefix {u}"
        assert set(G.legal_tokens(trie, st, k)) == L.mask_by_definition(lang, u), (cat, k, u)
    # and the walk generates nothing outside the language
    assert G.all_walks(trie, k) == lang


@pytest.mark.parametrize("case", range(len(I.brute_catalogs())))
def test_walk_equals_definition_fixed(case):
    cat, sep, stop, V = I.brute_catalogs()[case]
    for k in range(1, min(3, len(cat)) + 1):
        _check_against_definition(cat, sep, stop, V, k)


def test_walk_equals_definition_random():
    rng = I.rng_for(9, extra=1)
    n = 0
    for _ in range(150):
        cat = I.random_small_catalog(rng, vocab=12, max_k=5, max_len=4)
        for k in range(1, min(3, len(cat)) + 1):
            _check_against_definition(cat, 10, 11, 12, k)
            n += 1
    assert n > 200


def test_unreachable_prefix_is_rejected():
    trie = G.compile_catalog([(1, 2), (3,)], 14, 15, 16)
    assert G.walk(trie, (2,), 1) is None            # 2 is no root edge
    assert G.walk(trie, (1, 2, 14), 1) is None      # separator when no pointer is owed
    assert G.walk(trie, (3, 15, 3), 1) is None      # nothing after stop


def test_golden_walks():
    with open(os.path.join(GOLDEN, "walk_examples.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        trie = G.compile_catalog([tuple(c) for c in case["catalog"]], gold["sep"], gold["stop"], gold["vocab"])
        lang = L.language(trie.catalog, case["k"], gold["sep"], gold["stop"])
        for step in case["steps"]:
            u = tuple(step["prefix"])
            st = G.walk(trie, u, case["k"])
            assert st is not None, (case["name"], u)
            assert G.legal_tokens(trie, st, case["k"]) == step["legal"], (case["name"], u, step["why"])
            assert sorted(L.mask_by_definition(lang, u)) == step["legal"], (case["name"], u)


def test_exactly_k_distinct_pointers():
    cat, sep, stop, V = I.brute_catalogs()[5]
    trie = G.compile_catalog(cat, sep, stop, V)
    for k in (1, 2, 3):
        for s in G.all_walks(trie, k):
            pieces = []
            cur = []
            for t in s:
                if t in (sep, stop):
                    pieces.append(tuple(cur))
                    cur = []
                else:
                    cur.append(t)
            assert s[-1] == stop and s.count(stop) == 1 and s.count(sep) == k - 1
            assert len(pieces) == k and len(set(pieces)) == k and all(p in cat for p in pieces)


@pytest.mark.parametrize("bad,reason", [
    ([(1,), ()], "empty_string"),
    ([(1, 2), (1, 2)], "duplicate"),
    ([(1, 14)], "control_collision"),
    ([(1, 15)], "control_collision"),
    ([(16,)], "token_range"),
    ([(-1,)], "token_range"),
])
def test_compile_refusals(bad, reason):
    with pytest.raises(G.CompileError) as e:
        G.compile_catalog(bad, 14, 15, 16)
    assert e.value.reason == reason


def test_fanout_cap_counts_control_edges():
    V = 1000
    # root with 256 children: allowed at cap 256, refused at 255
    cat = [(i,) for i in range(256)]
    G.compile_catalog(cat, V - 2, V - 1, V, max_fanout=256)
    with pytest.raises(G.CompileError):
        G.compile_catalog(cat, V - 2, V - 1, V, max_fanout=255)
    # a terminal node with 255 children has 257 edges (two control edges)
    cat = [(500,)] + [(500, i) for i in range(255)]
    assert G.compile_catalog(cat, V - 2, V - 1, V, max_fanout=257).max_fanout == 257
    with pytest.raises(G.CompileError):
        G.compile_catalog(cat, V - 2, V - 1, V, max_fanout=256)


def test_trie_sizes():
    trie = G.compile_catalog([(1, 2), (1, 3), (4,)], 14, 15, 16)
    # nodes: root, (1), (1,2), (1,3), (4)
    assert trie.n_nodes == 5
    # edges: root->1, root->4, (1)->2, (1)->3, + 2 control edges at each of 3 terminals
    assert trie.n_edges == 4 + 6
