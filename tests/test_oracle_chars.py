"""Pins for the character-level oracle (CPU only).

Source: the pith.science review of arXiv 2608.12574 (key machinery): every
tokenization of a catalog string is accepted; a token is valid at a trie node
when its characters walk from the node without overshooting the strings.
Pinned against brute-force enumeration of the language (every segmentation of
every ordered choice of strings), the token-trie oracle on a one-byte
vocabulary (where tokenization is unique), and the generators' canonical
tokenizations."""
import itertools

import numpy as np

from oracle import chars as C
from oracle import decode as D
from oracle import grammar as G
from oracle import language as L
from trie_constrained_decoding_gb300 import inputs as I

SEP, STOP = 98, 99

BRUTE = [
    ([b"ab", b"b"], [(1, b"a"), (2, b"b"), (3, b"ab")]),
    ([b"aba", b"ab", b"bb"], [(1, b"a"), (2, b"b"), (3, b"ab"), (4, b"ba"), (5, b"bab")]),
    ([b"aaa", b"aab", b"b"], [(1, b"a"), (2, b"b"), (3, b"aa"), (4, b"aaa"), (5, b"ab")]),
    ([b"abc", b"bc", b"c", b"ca"], [(1, b"a"), (2, b"b"), (3, b"c"), (4, b"bc"), (5, b"abc"), (6, b"ca")]),
]


def test_legal_sets_equal_the_enumerated_language():
    """At every prefix of every member, the legal set is the mask taken from
    the enumerated language (all segmentations of all ordered choices)."""
    for strings, vocab in BRUTE:
        cg = C.CharGrammar(strings, vocab, SEP, STOP)
        for k in range(1, len(strings) + 1):
            lang = C.char_language(strings, vocab, k, SEP, STOP)
            assert lang
            for u in L.reachable_prefixes(lang):
                if u in lang:
                    continue
                st = cg.start()
                for t in u:
                    st = cg.advance(st, t, k)
                assert set(cg.legal(st, k)) == L.mask_by_definition(lang, u), (strings, k, u)


def test_one_byte_vocabulary_equals_the_token_trie():
    """With one token per byte, tokenization is unique and the character-level
    language is the token trie's language over those tokens."""
    rng = np.random.default_rng(17)
    for rep in range(20):
        n = int(rng.integers(1, 6))
        strings = sorted({bytes(rng.integers(97, 100, size=int(rng.integers(1, 5))).tolist()) for _ in range(n)})
        vocab = [(c - 97 + 1, bytes([c])) for c in range(97, 100)]
        cg = C.CharGrammar(strings, vocab, SEP, STOP)
        cat = [tuple(c - 97 + 1 for c in s) for s in strings]
        tt = G.compile_catalog(cat, SEP, STOP, 100)
        for k in range(1, len(strings) + 1):
            walks_c = set()
            stack = [((), cg.start())]
            while stack:
                seq, st = stack.pop()
                if st.done:
                    walks_c.add(seq)
                    continue
                for t in cg.legal(st, k):
                    stack.append((seq + (t,), cg.advance(st, t, k)))
            assert walks_c == G.all_walks(tt, k)


def test_canonical_and_other_tokenizations_are_accepted():
    w = I.char_tiny()
    cg = C.CharGrammar(w.char_strings, w.char_vocab, w.sep_id, w.stop_id)
    for s, canon in zip(w.char_strings, w.catalog):
        assert D.replay_ok(cg, list(canon) + [w.stop_id], 1)
        segs = C.segmentations(s, w.char_vocab)
        assert tuple(canon) in segs and len(segs) >= 1
        for seg in segs[:5]:
            assert D.replay_ok(cg, list(seg) + [w.stop_id], 1)
        assert cg.parse_pointers(list(segs[-1]) + [w.stop_id]) == [w.char_strings.index(s)]
    h = I.char_hex()
    ch = C.CharGrammar(h.char_strings, h.char_vocab, h.sep_id, h.stop_id)
    u = I.unstructured()        # the token-level workload's segmentation of the same strings
    for s, canon in zip(h.char_strings[:50], u.catalog[:50]):
        assert D.replay_ok(ch, list(canon) + [h.stop_id], 1)


def test_greedy_decode_emits_catalog_strings():
    w = I.char_tiny()
    cg = C.CharGrammar(w.char_strings, w.char_vocab, w.sep_id, w.stop_id)
    emb = w.embedding()
    hid = w.hidden_states(0, 6)
    for q in range(6):
        toks, logits, st = D.greedy_decode(cg, w.k, emb, hid[:, q], w.max_steps)
        assert st == "ok" and D.replay_ok(cg, toks, w.k)
        ptrs = cg.parse_pointers(toks)
        assert len(ptrs) == w.k and len(set(ptrs)) == w.k and min(ptrs) >= 0
