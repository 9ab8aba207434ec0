"""The host trie compiler (C ABI, CPU only) against the oracle's prefix trie.

"Constraint made cheaper than no constraint", section "The grammar as a trie
over tokens": an edge range per node, a token and a child per edge, sentinel
children for the separator and stop edges, each pointer's path of edges;
section "Masked sampling inside the sampler": per-edge live-pointer counts;
section "The sparse output layer": the fan-out cap."""

import numpy as np
import pytest

from oracle import grammar as G
from trie_constrained_decoding_gb300 import inputs as I


def _compare(tcd, cat, sep, stop, V, cap=256):
    ref = G.compile_catalog(cat, sep, stop, V, max_fanout=cap)
    tr = tcd.Trie.compile(cat, sep, stop, V, cap)
    info = tr.info()
    a = tr.export()
    assert info["n_nodes"] == ref.n_nodes
    assert info["n_edges"] == ref.n_edges
    assert info["n_strings"] == len(cat)
    assert info["max_fanout"] == ref.max_fanout
    assert info["root_fanout"] == ref.fanout(())
    assert info["max_depth"] == max(len(s) for s in cat)
    assert info["total_tokens"] == sum(len(s) for s in cat)
    nb, tok, child, nptr, cnt = a["node_begin"], a["edge_tok"], a["edge_child"], a["node_ptr"], a["static_cnt"]
    assert nb[0] == 0 and nb[-1] == info["n_edges"] and np.all(np.diff(nb) >= 0)
    # walk the CSR depth-first; node ids must come out in preorder, children by ascending token
    prefix_of = {0: ()}
    order = []
    q = [0]
    while q:
        n = q.pop()
        order.append(n)
        u = prefix_of[n]
        es = range(nb[n], nb[n + 1])
        toks = [int(tok[e]) for e in es]
        assert toks == sorted(toks)
        kids = sorted((int(tok[e]), int(child[e]), e) for e in es if child[e] >= 0)
        ctl = sorted((int(tok[e]), int(child[e])) for e in es if child[e] < 0)
        assert [t for t, _, _ in kids] == ref.children.get(u, [])
        if u in ref.terminal:
            assert ctl == sorted([(sep, -1), (stop, -2)])
            assert nptr[n] == ref.terminal[u]
        else:
            assert ctl == [] and nptr[n] == -1
        for t, c, e in kids:
            assert c not in prefix_of
            prefix_of[c] = u + (t,)
            assert cnt[e] == len(ref.below[u + (t,)])
        q.extend(c for _, c, _ in reversed(kids))
        for e in es:
            if child[e] < 0:
                assert cnt[e] == 0
    assert order == list(range(info["n_nodes"]))
    # per-pointer paths
    off, path = a["path_off"], a["path"]
    for p, s in enumerate(cat):
        es = path[off[p]:off[p + 1]]
        assert len(es) == len(s)
        n = 0
        for t, e in zip(s, es):
            assert nb[n] <= e < nb[n + 1] and tok[e] == t and child[e] >= 0
            n = child[e]
        assert nptr[n] == p
    tr.close()
    return info


@pytest.mark.parametrize("case", range(len(I.brute_catalogs())))
def test_compiler_matches_oracle_small(tcd, case):
    cat, sep, stop, V = I.brute_catalogs()[case]
    _compare(tcd, cat, sep, stop, V)


def test_compiler_matches_oracle_random(tcd):
    rng = I.rng_for(9, extra=7)
    for _ in range(100):
        cat = I.random_small_catalog(rng, vocab=12, max_k=8, max_len=5)
        _compare(tcd, cat, 10, 11, 12)


@pytest.mark.parametrize("name", ["tiny", "batched", "unstructured"])
def test_compiler_matches_oracle_workloads(tcd, name):
    w = I.WORKLOADS[name]()
    info = _compare(tcd, w.catalog, w.sep_id, w.stop_id, w.vocab, w.max_fanout)
    if name == "unstructured":
        assert info["root_fanout"] > 256


@pytest.mark.parametrize("bad,code", [
    ([(1,), ()], "TC_ERR_EMPTY_STRING"),
    ([(1, 2), (1, 2)], "TC_ERR_DUPLICATE"),
    ([(1, 14)], "TC_ERR_CONTROL_COLLISION"),
    ([(15,)], "TC_ERR_CONTROL_COLLISION"),
    ([(16,)], "TC_ERR_TOKEN_RANGE"),
    ([(-1,)], "TC_ERR_TOKEN_RANGE"),
])
def test_compiler_refusals(tcd, bad, code):
    with pytest.raises(tcd.TcError) as e:
        tcd.Trie.compile(bad, 14, 15, 16)
    assert e.value.name == code


def test_compiler_invalid_args(tcd):
    for args in [((1,), 14, 14, 16), ((1,), 16, 15, 16), ((1,), 14, 15, 1)]:
        with pytest.raises(tcd.TcError) as e:
            tcd.Trie.compile([args[0]], *args[1:])
        assert e.value.name == "TC_ERR_INVALID_ARG"
    with pytest.raises(tcd.TcError):
        tcd.Trie.compile([], 14, 15, 16)


def test_fanout_cap(tcd):
    V = 1000
    cat = [(i,) for i in range(256)]
    assert tcd.Trie.compile(cat, V - 2, V - 1, V, 256).info()["root_fanout"] == 256
    with pytest.raises(tcd.TcError) as e:
        tcd.Trie.compile(cat, V - 2, V - 1, V, 255)
    assert e.value.name == "TC_ERR_FANOUT"
    cat = [(500,)] + [(500, i) for i in range(255)]      # 255 children + 2 control edges
    assert tcd.Trie.compile(cat, V - 2, V - 1, V, 257).info()["max_fanout"] == 257
    with pytest.raises(tcd.TcError):
        tcd.Trie.compile(cat, V - 2, V - 1, V, 256)


def test_walk_image_size(tcd):
    """Header part: node ranges and pointer ranks (2N + 1 words, what constant
    residency copies); then 32-byte edge records from a 32-byte boundary."""
    w = I.tiny()
    info = tcd.Trie.compile(w.catalog, w.sep_id, w.stop_id, w.vocab).info()
    N, E = info["n_nodes"], info["n_edges"]
    assert info["header_bytes"] == 4 * (2 * N + 1)
    assert info["walk_image_bytes"] == 4 * (((2 * N + 1 + 7) & ~7) + 8 * E)
    assert info["header_bytes"] <= tcd.CONST_CAPACITY_BYTES
    u = I.unstructured()
    info = tcd.Trie.compile(u.catalog, u.sep_id, u.stop_id, u.vocab, u.max_fanout).info()
    assert info["header_bytes"] > tcd.CONST_CAPACITY_BYTES      # the hex catalog's headers need global memory


def _rank_catalogs():
    out = [(w.catalog, w.sep_id, w.stop_id, w.vocab, w.max_fanout) for w in (I.tiny(), I.batched(), I.unstructured())]
    for cat, sep, stop, V in I.brute_catalogs():
        out.append((cat, sep, stop, V, 256))
    for seed in range(6):
        cat = I.random_small_catalog(I.rng_for(40, extra=seed))
        out.append((cat, 10, 11, 12, 256))
    return out


def test_depth_first_ranks_give_each_subtree_one_range(tcd):
    """The read-only no-repeat state ("Constraint made cheaper than no
    constraint", section "The batched engine") needs the pointers below every
    edge as one range of ranks.  Checked against the oracle's own trie: the
    pointer ids whose rank lies in [edge_lo, edge_lo + static_cnt) are exactly
    the pointers at or below the edge's child, and a control edge's lo is the
    rank of the terminal's own pointer."""
    for cat, sep, stop, V, fan in _rank_catalogs():
        t = tcd.Trie.compile(cat, sep, stop, V, fan)
        ex, rk = t.export(), t.ranks()
        K = len(cat)
        assert sorted(rk["ptr_rank"].tolist()) == list(range(K))
        by_rank = np.empty(K, dtype=np.int64)
        by_rank[rk["ptr_rank"]] = np.arange(K)
        ot = G.compile_catalog(cat, sep, stop, V, max_fanout=fan)
        # prefix of every node: walk the CSR from the root
        prefix = {0: ()}
        order = [0]
        for n in order:
            for e in range(ex["node_begin"][n], ex["node_begin"][n + 1]):
                c = int(ex["edge_child"][e])
                if c >= 0:
                    prefix[c] = prefix[n] + (int(ex["edge_tok"][e]),)
                    order.append(c)
        for n in order:
            for e in range(ex["node_begin"][n], ex["node_begin"][n + 1]):
                c, lo = int(ex["edge_child"][e]), int(rk["edge_lo"][e])
                if c >= 0:
                    got = {int(by_rank[r]) for r in range(lo, lo + int(ex["static_cnt"][e]))}
                    want = set(ot.below[prefix[c]])
                    assert got == want
                else:
                    assert lo == rk["ptr_rank"][ex["node_ptr"][n]]
        t.close()


@pytest.mark.parametrize("name", ["tiny", "large_head", "batched", "unstructured"])
def test_single_edge_chains_have_consecutive_records(tcd, name):
    """Depth-first node numbers lay a chain of single-edge nodes out as
    consecutive edge records, which lets a forced continuation read a whole
    run at once: whenever a node's only edge leads to a child with a single
    edge, that edge is the next record.  (The device walk checks every link
    itself, so this pins the layout, not correctness.)"""
    w = I.WORKLOADS[name]()
    t = tcd.Trie.compile(w.catalog, w.sep_id, w.stop_id, w.vocab, w.max_fanout)
    ex = t.export()
    nb, child = ex["node_begin"], ex["edge_child"]
    links = 0
    for n in range(len(nb) - 1):
        if nb[n + 1] - nb[n] != 1 or child[nb[n]] < 0:
            continue
        c = int(child[nb[n]])
        if nb[c + 1] - nb[c] == 1:
            assert nb[c] == nb[n] + 1
            links += 1
    t.close()
    assert links > 0
