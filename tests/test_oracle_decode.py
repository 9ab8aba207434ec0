"""Pins for the oracle's decode loop, replay and teacher-forcing checker (CPU only)."""
import numpy as np
import pytest

from oracle import decode as D
from oracle import grammar as G
from oracle import language as L
from trie_constrained_decoding_gb300 import inputs as I


def _tiny_trie():
    w = I.tiny()
    return w, G.compile_catalog(w.catalog, w.sep_id, w.stop_id, w.vocab)


def test_greedy_outputs_are_language_members():
    w, trie = _tiny_trie()
    emb = w.embedding()
    hid = w.hidden_states(0, 16)
    for q in range(16):
        toks, logits, status = D.greedy_decode(trie, w.k, emb, hid[:, q], w.max_steps)
        assert status == "ok"
        assert D.replay_ok(trie, toks, w.k)
        ptrs = D.parse_pointers(trie, toks)
        assert len(ptrs) == w.k and len(set(ptrs)) == w.k and min(ptrs) >= 0


def test_greedy_brute_force_argmax_over_language():
    """On a tiny catalog, each greedy step's choice is the argmax (lower id on
    ties) over the mask taken from the enumerated language."""
    cat, sep, stop, V = I.brute_catalogs()[5]
    trie = G.compile_catalog(cat, sep, stop, V)
    rng = I.rng_for(9, extra=4)
    emb = I.integer_bf16(rng, (V, 8), lo=-1, hi=1)
    for k in (1, 2, 3):
        lang = L.language(cat, k, sep, stop)
        hid = I.integer_bf16(rng, (k * 4, 8), lo=-1, hi=1)
        toks, logits, status = D.greedy_decode(trie, k, emb, hid, k * 4)
        assert status == "ok" and tuple(toks) in lang
        for t in range(len(toks)):
            mask = sorted(L.mask_by_definition(lang, tuple(toks[:t])))
            emb_f = [sum(a * b for a, b in zip(
                [float(v) for v in (np.asarray(emb[m], np.uint32) << 16).view(np.float32)],
                [float(v) for v in (np.asarray(hid[t], np.uint32) << 16).view(np.float32)])) for m in mask]
            best = max(range(len(mask)), key=lambda i: (emb_f[i], -mask[i]))
            assert toks[t] == mask[best] and logits[t] == emb_f[best]


def test_dense_and_sparse_decode_agree():
    w, trie = _tiny_trie()
    emb = w.embedding()
    hid = w.hidden_states(0, 3)
    for q in range(3):
        a = D.greedy_decode(trie, w.k, emb, hid[:, q], w.max_steps, head="sparse")
        b = D.greedy_decode(trie, w.k, emb, hid[:, q], w.max_steps, head="dense")
        assert a == b


def test_max_steps_status():
    w, trie = _tiny_trie()
    emb = w.embedding()
    hid = w.hidden_states(0, 1)
    toks, logits, status = D.greedy_decode(trie, w.k, emb, hid[:, 0], 2)
    assert status == "max_steps" and len(toks) == 2


def test_empty_mask_when_more_pointers_owed_than_exist():
    # the walk, run unchecked with k > K, runs out of live edges after the
    # last pointer's separator (the language itself is empty: such k is refused up front)
    trie = G.compile_catalog([(1,)], 14, 15, 16)
    emb = np.zeros((16, 2), np.uint16)
    hid = np.zeros((5, 2), np.uint16)
    toks, logits, status = D.greedy_decode(trie, 2, emb, hid, 5)
    assert toks == [1, 14] and status == "empty_mask"
    assert L.language(trie.catalog, 2, 14, 15) == set()


def test_teacher_forcing_accepts_oracle_and_rejects_faults():
    w, trie = _tiny_trie()
    emb = w.embedding()
    hid = w.hidden_states(0, 1)[:, 0]
    toks, logits, status = D.greedy_decode(trie, w.k, emb, hid, w.max_steps)
    f32 = [float(np.float32(l)) for l in logits]
    assert D.teacher_force(trie, w.k, emb, hid, toks, f32, status, w.max_steps, exact=True).ok
    # a wrong logit in the last place
    bad = list(f32)
    bad[1] = float(np.nextafter(np.float32(bad[1]), np.float32(np.inf)))
    assert not D.teacher_force(trie, w.k, emb, hid, toks, bad, status, w.max_steps, exact=True).ok
    # an illegal token
    bad_t = list(toks)
    bad_t[0] = w.sep_id
    assert not D.teacher_force(trie, w.k, emb, hid, bad_t, f32, status, w.max_steps).ok
    # wrong status
    assert not D.teacher_force(trie, w.k, emb, hid, toks, f32, "max_steps", w.max_steps).ok
    # a non-argmax legal token with a clear margin
    legal = G.legal_tokens(trie, G.WalkState(), w.k)
    other = [t for t in legal if t != toks[0]][0]
    alt = [other] + list(toks[1:])
    rep = D.teacher_force(trie, w.k, emb, hid, alt[:1], f32[:1], "max_steps", 1)
    assert not rep.ok


def test_teacher_forcing_gaussian_tolerance():
    rng = I.rng_for(9, extra=5)
    trie = G.compile_catalog([(1,), (2,), (3,)], 14, 15, 16)
    emb = I.gaussian_bf16(rng, (16, 512), 0.02)
    hid = I.gaussian_bf16(rng, (2, 512), 1.0)
    toks, logits, status = D.greedy_decode(trie, 1, emb, hid, 2)
    ok = D.teacher_force(trie, 1, emb, hid, toks, [l * (1 + 5e-4) for l in logits], status, 2)
    assert ok.ok
    bad = D.teacher_force(trie, 1, emb, hid, toks, [l * (1 + 5e-3) for l in logits], status, 2)
    assert not bad.ok


def test_hidden_states_are_batch_independent():
    w = I.tiny()
    a = w.hidden_states(0, 4, steps=3)
    b = w.hidden_states(2, 2, steps=3)
    assert np.array_equal(a[:, 2:], b)
