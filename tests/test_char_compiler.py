"""The character-level grammar compiler (C ABI, CPU only) against the oracle.

The pith.science review of arXiv 2608.12574 (key machinery): a character trie
of the strings whose nodes carry every vocabulary token that walks from the
node without overshooting, found by Aho-Corasick matching along the trie.
Checked node by node against the oracle's definition (a token leads from
prefix p to p + bytes, which must be a prefix of some string)."""
import numpy as np
import pytest

from oracle import chars as C
from trie_constrained_decoding_gb300 import inputs as I

SEP, STOP, V = 98, 99, 100


def _prefixes(ex, vocab):
    """Prefix bytes of every CSR node, walking token edges from the root."""
    tb = dict(vocab)
    pre = {0: b""}
    order = [0]
    for n in order:
        for e in range(ex["node_begin"][n], ex["node_begin"][n + 1]):
            c = int(ex["edge_child"][e])
            if c >= 0:
                p = pre[n] + tb[int(ex["edge_tok"][e])]
                if c in pre:
                    assert pre[c] == p          # every path into a node spells the same prefix
                else:
                    pre[c] = p
                    order.append(c)
    return pre


def _check(tcd, strings, vocab, sep=SEP, stop=STOP, vsize=V, fan=4096):
    t = tcd.Trie.compile_chars(strings, vocab, sep, stop, vsize, fan)
    info, ex, rk = t.info(), t.export(), t.ranks()
    cg = C.CharGrammar(strings, vocab, sep, stop)
    pre = _prefixes(ex, vocab)
    all_prefixes = {s[:L] for s in strings for L in range(len(s) + 1)}
    assert set(pre.values()) == all_prefixes and info["n_nodes"] == len(all_prefixes)
    by_rank = np.empty(len(strings), dtype=np.int64)
    by_rank[rk["ptr_rank"]] = np.arange(len(strings))
    for n, p in pre.items():
        b, e = ex["node_begin"][n], ex["node_begin"][n + 1]
        toks = [int(x) for x in ex["edge_tok"][b:e]]
        assert toks == sorted(toks)
        got = {int(ex["edge_tok"][i]): pre[int(ex["edge_child"][i])] for i in range(b, e) if ex["edge_child"][i] >= 0}
        assert got == cg.token_edges(p)
        term = cg.index.get(p, -1)
        assert int(ex["node_ptr"][n]) == term
        ctl = {int(ex["edge_tok"][i]): int(ex["edge_child"][i]) for i in range(b, e) if ex["edge_child"][i] < 0}
        assert ctl == ({sep: -1, stop: -2} if term >= 0 else {})
        for i in range(b, e):
            c = int(ex["edge_child"][i])
            if c >= 0:
                below = {j for j, s in enumerate(strings) if s.startswith(pre[c])}
                lo, cnt = int(rk["edge_lo"][i]), int(ex["static_cnt"][i])
                assert cnt == len(below) and {int(by_rank[r]) for r in range(lo, lo + cnt)} == below
    assert info["max_depth"] == max(len(s) for s in strings)
    t.close()
    return info


def test_brute_catalogs(tcd):
    from test_oracle_chars import BRUTE
    for strings, vocab in BRUTE:
        _check(tcd, strings, vocab)


def test_random_catalogs(tcd):
    rng = np.random.default_rng(23)
    for rep in range(40):
        alpha = b"abc"
        strings = sorted({bytes(rng.choice(list(alpha), size=int(rng.integers(1, 7))).tolist())
                          for _ in range(int(rng.integers(1, 9)))})
        pieces = {bytes([c]) for c in alpha}
        for _ in range(int(rng.integers(0, 10))):
            s = strings[int(rng.integers(len(strings)))]
            L = int(rng.integers(1, len(s) + 1))
            i = int(rng.integers(0, len(s) - L + 1))
            pieces.add(s[i:i + L])
        pieces.add(b"cab")                      # may or may not occur in the strings
        vocab = [(j + 1, p) for j, p in enumerate(sorted(pieces))]
        _check(tcd, strings, vocab)


@pytest.mark.parametrize("name", ["char_tiny", "char_tools", "char_hex"])
def test_workload_grammars(tcd, name):
    w = I.WORKLOADS[name]()
    strings = w.char_strings if name != "char_hex" else w.char_strings[:150]
    info = _check(tcd, strings, w.char_vocab, w.sep_id, w.stop_id, w.vocab, w.max_fanout)
    assert info["n_strings"] == len(strings)


def test_refusals(tcd):
    with pytest.raises(tcd.TcError) as e:
        tcd.Trie.compile_chars([b"ab", b"ab"], [(1, b"a"), (2, b"b")], SEP, STOP, V)
    assert e.value.name == "TC_ERR_DUPLICATE"
    with pytest.raises(tcd.TcError) as e:
        tcd.Trie.compile_chars([b"ab"], [(1, b"a"), (1, b"b")], SEP, STOP, V)
    assert e.value.name == "TC_ERR_DUPLICATE"
    with pytest.raises(tcd.TcError) as e:
        tcd.Trie.compile_chars([b"ab"], [(1, b"a"), (2, b"a")], SEP, STOP, V)
    assert e.value.name == "TC_ERR_DUPLICATE"
    with pytest.raises(tcd.TcError) as e:
        tcd.Trie.compile_chars([b"ab"], [(SEP, b"a"), (2, b"b")], SEP, STOP, V)
    assert e.value.name == "TC_ERR_CONTROL_COLLISION"
    with pytest.raises(tcd.TcError) as e:
        tcd.Trie.compile_chars([b"ab"], [(1, b"a"), (200, b"b")], SEP, STOP, V)
    assert e.value.name == "TC_ERR_TOKEN_RANGE"
    with pytest.raises(tcd.TcError) as e:
        tcd.Trie.compile_chars([b""], [(1, b"a")], SEP, STOP, V)
    assert e.value.name == "TC_ERR_EMPTY_STRING"
    with pytest.raises(tcd.TcError) as e:      # root: a, b, ab, ba -> 4 edges
        tcd.Trie.compile_chars([b"ab", b"ba"], [(1, b"a"), (2, b"b"), (3, b"ab"), (4, b"ba")], SEP, STOP, V, 3)
    assert e.value.name == "TC_ERR_FANOUT"
