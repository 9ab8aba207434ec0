"""Pins for the oracle's forced-span decode (CPU only).

"Understanding Inference for Systems Engineers", section 7.5 (forced spans):
where the grammar admits exactly one continuation, the model's scores cannot
change the token, so it is taken without reading the head.  The oracle's
``greedy_decode(jump=True)`` reports such positions (from the second token on)
with a NaN logit.  Pinned here against hand-derived legal sets and against the
next-token mask taken from the enumerated language."""
import math

import numpy as np

from oracle import decode as D
from oracle import grammar as G
from oracle import language as L
from trie_constrained_decoding_gb300 import inputs as I

V, SEP, STOP = 32, 30, 31


def _emb(seed, rows=V, h=8):
    return I.integer_bf16(I.rng_for(seed, extra=11), (rows, h), lo=-3, hi=3)


def _nan_pattern(logits):
    return [math.isnan(x) for x in logits]


def test_single_string_is_one_decision_then_forced():
    # Legal sets along the only member: {5}, {6}, {7}, {STOP}.  The first comes
    # from the head; the other three are forced.
    trie = G.compile_catalog([(5, 6, 7)], SEP, STOP, V)
    emb = _emb(1)
    hid = I.integer_bf16(I.rng_for(2, extra=11), (8, 8), lo=-3, hi=3)
    toks, logits, status = D.greedy_decode(trie, 1, emb, hid, 8, jump=True)
    assert status == "ok" and toks == [5, 6, 7, STOP]
    assert _nan_pattern(logits) == [False, True, True, True]


def test_shared_prefix_pattern():
    # [(5,6,7), (5,6,8)], k=1: {5} head, {6} forced, {7,8} head, {STOP} forced.
    trie = G.compile_catalog([(5, 6, 7), (5, 6, 8)], SEP, STOP, V)
    emb = _emb(3)
    for q in range(6):
        hid = I.integer_bf16(I.rng_for(4, extra=q), (8, 8), lo=-3, hi=3)
        toks, logits, status = D.greedy_decode(trie, 1, emb, hid, 8, jump=True)
        assert status == "ok" and toks[:2] == [5, 6] and toks[2] in (7, 8) and toks[3] == STOP
        assert _nan_pattern(logits) == [False, True, False, True]


def test_pointer_completion_inside_a_span():
    # [(5,6), (9,)], k=2: after the first decision every remaining set is a
    # singleton - the separator, then the other pointer (the spent one has no
    # live pointer below it), then stop - so all later positions are forced.
    trie = G.compile_catalog([(5, 6), (9,)], SEP, STOP, V)
    seen = set()
    for q in range(12):
        emb = _emb(20 + q)
        hid = I.integer_bf16(I.rng_for(5, extra=q), (8, 8), lo=-3, hi=3)
        toks, logits, status = D.greedy_decode(trie, 2, emb, hid, 8, jump=True)
        assert status == "ok"
        assert toks in ([5, 6, SEP, 9, STOP], [9, SEP, 5, 6, STOP])
        assert _nan_pattern(logits) == [False] + [True] * (len(toks) - 1)
        seen.add(toks[0])
    assert seen == {5, 9}   # both orders occurred


def test_forced_positions_match_language_mask():
    """On the brute-force catalogs: the jump decode emits the same tokens as the
    plain decode, real logits equal, and NaN exactly where the mask taken from
    the enumerated language holds one token (second position on)."""
    for ci, (cat, sep, stop, vocab) in enumerate(I.brute_catalogs()):
        trie = G.compile_catalog(cat, sep, stop, vocab)
        emb = I.integer_bf16(I.rng_for(30, extra=ci), (vocab, 8), lo=-2, hi=2)
        for k in (1, 2, 3):
            if k > len(cat):
                continue
            lang = L.language(cat, k, sep, stop)
            for q in range(4):
                hid = I.integer_bf16(I.rng_for(31 + ci, extra=q * 7 + k), (k * 12, 8), lo=-2, hi=2)
                plain = D.greedy_decode(trie, k, emb, hid, k * 12)
                jump = D.greedy_decode(trie, k, emb, hid, k * 12, jump=True)
                assert jump[0] == plain[0] and jump[2] == plain[2] == "ok"
                toks = tuple(jump[0])
                want = [t > 0 and len(L.mask_by_definition(lang, toks[:t])) == 1 for t in range(len(toks))]
                assert _nan_pattern(jump[1]) == want
                for a, b, f in zip(jump[1], plain[1], want):
                    assert f or a == b
                assert D.forced_positions(trie, toks, k) == [t for t, f in enumerate(want) if f]


def test_teacher_force_jump_catches_a_missing_nan_and_a_stray_nan():
    trie = G.compile_catalog([(5, 6, 7), (5, 6, 8)], SEP, STOP, V)
    emb = _emb(3)
    hid = I.integer_bf16(I.rng_for(4, extra=0), (8, 8), lo=-3, hi=3)
    toks, logits, status = D.greedy_decode(trie, 1, emb, hid, 8, jump=True)
    assert D.teacher_force(trie, 1, emb, hid, toks, logits, status, 8, exact=True, jump=True).ok
    plain = D.greedy_decode(trie, 1, emb, hid, 8)
    # a real logit where the position is forced
    assert not D.teacher_force(trie, 1, emb, hid, plain[0], plain[1], status, 8, exact=True, jump=True).ok
    # a NaN where the head decides
    bad = list(logits)
    bad[2] = float("nan")
    assert not D.teacher_force(trie, 1, emb, hid, toks, bad, status, 8, exact=True, jump=True).ok
    assert np.isnan(logits[1]) and not np.isnan(logits[0])
