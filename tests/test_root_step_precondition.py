"""The first decode step's legal set is the compiled root's token edges (CPU).

The tensor-core root step (TC_FLAG_ROOT_GEMM) gives every sequence of a fresh
decode the root's token edges as candidates, without filtering.  That rests on
two facts of the language ("Constraint made cheaper than no constraint",
section "The grammar as a trie over tokens"): the root is not a terminal (the
compiler refuses empty strings), so no separator or stop is legal there, and
every token edge has a pointer below it, none spent yet.  Here the oracle's
legal set at the empty prefix, for several k, is compared with the root edges
of the compiled CSR (token and character-level grammars), and with the flags
the library itself checks at bind (all root edges token edges with pointers)."""
import numpy as np
import pytest

from oracle import chars as C
from oracle import grammar as G
from trie_constrained_decoding_gb300 import inputs as I

TOKEN_WORKLOADS = ["tiny", "batched", "unstructured"]
CHAR_WORKLOADS = ["char_tiny", "char_tools"]


def _root_edges(exp):
    beg, end = int(exp["node_begin"][0]), int(exp["node_begin"][1])
    return exp["edge_tok"][beg:end], exp["edge_child"][beg:end], exp["static_cnt"][beg:end]


@pytest.mark.parametrize("name", TOKEN_WORKLOADS)
def test_token_grammar_root_is_the_first_legal_set(tcd, name):
    w = I.WORKLOADS[name]()
    trie = tcd.Trie.compile(w.catalog, w.sep_id, w.stop_id, w.vocab, w.max_fanout)
    toks, child, cnt = _root_edges(trie.export())
    trie.close()
    assert np.all(child >= 0) and np.all(cnt > 0)          # token edges only, each with pointers below
    assert np.all(np.diff(toks) > 0)                        # ascending: the GEMM's columns in token order
    oracle = G.compile_catalog(w.catalog, w.sep_id, w.stop_id, w.vocab, max_fanout=w.max_fanout)
    for k in sorted({1, 2, w.k, min(8, len(w.catalog))}):
        assert G.legal_tokens(oracle, G.WalkState(), k) == toks.tolist(), k


@pytest.mark.parametrize("name", CHAR_WORKLOADS)
def test_char_grammar_root_is_the_first_legal_set(tcd, name):
    w = I.WORKLOADS[name]()
    trie = tcd.Trie.compile_chars(w.char_strings, w.char_vocab, w.sep_id, w.stop_id, w.vocab, w.max_fanout)
    toks, child, cnt = _root_edges(trie.export())
    trie.close()
    assert np.all(child >= 0) and np.all(cnt > 0)
    assert np.all(np.diff(toks) > 0)
    g = C.CharGrammar(w.char_strings, w.char_vocab, w.sep_id, w.stop_id)
    for k in sorted({1, 2, w.k}):
        assert sorted(g.legal(g.start(), k)) == toks.tolist(), k


def test_a_prefix_pointer_never_makes_the_root_a_terminal(tcd):
    """Catalog strings that are prefixes of others end at inner nodes, never
    at the root; an empty string is refused outright."""
    sep, stop, V = 98, 99, 100
    catalog = [(1,), (1, 2), (3, 4, 5), (3,)]
    trie = tcd.Trie.compile(catalog, sep, stop, V)
    toks, child, _ = _root_edges(trie.export())
    trie.close()
    assert toks.tolist() == [1, 3] and np.all(child >= 0)
    oracle = G.compile_catalog(catalog, sep, stop, V)
    assert G.legal_tokens(oracle, G.WalkState(), 2) == [1, 3]
    with pytest.raises(tcd.TcError):
        tcd.Trie.compile([(1,), ()], sep, stop, V)
