"""Pins for the oracle's sampler (CPU only).

"Understanding Inference for Systems Engineers", section 3.8: softmax of the
logits over the temperature, optionally restricted to the top-k highest logits
(a value threshold: ties can keep more than k) and to the smallest set whose
probability exceeds top-p (an ascending prefix is removed; among equal
probabilities the highest id survives).  Pinned against hand-derived tie
cases, a library softmax, the greedy argmax (top-k = 1) and the limits of the
temperature."""
import math

import numpy as np
import pytest
from scipy.special import softmax

from oracle import decode as D
from oracle import grammar as G
from oracle import sample as S
from oracle.head import argmax_lower_id
from trie_constrained_decoding_gb300 import inputs as I


def _lengths(iv):
    return {t: hi - lo for t, (lo, hi) in iv.items()}


def test_plain_softmax_matches_library():
    rng = np.random.default_rng(5)
    for n in (1, 2, 7, 31):
        toks = sorted(rng.choice(1000, size=n, replace=False).tolist())
        lg = rng.normal(size=n).tolist()
        for T in (0.3, 1.0, 2.5):
            got = _lengths(S.token_intervals(toks, lg, T, 0, 1.0))
            want = softmax(np.array(lg) / T)
            assert np.allclose([got[t] for t in toks], want, rtol=1e-12, atol=1e-15)


def test_top_k_is_a_value_threshold():
    toks, lg = [10, 11, 12, 13], [3.0, 3.0, 2.0, 1.0]
    assert set(S.token_intervals(toks, lg, 1.0, 1, 1.0)) == {10, 11}      # both tied maxima kept
    assert set(S.token_intervals(toks, lg, 1.0, 2, 1.0)) == {10, 11}
    assert set(S.token_intervals(toks, lg, 1.0, 3, 1.0)) == {10, 11, 12}
    assert set(S.token_intervals(toks, lg, 1.0, 4, 1.0)) == {10, 11, 12, 13}
    assert S.kept_top_k([0.0, -0.0, -1.0], 1) == [True, True, False]      # -0 == +0


def test_top_p_removes_an_ascending_prefix_highest_tied_id_survives():
    toks, lg = [4, 7, 9, 20], [0.0, 0.0, 0.0, 0.0]                       # p = 1/4 each
    assert set(S.token_intervals(toks, lg, 1.0, 0, 0.5)) == {9, 20}       # masses .25, .5 <= .5 removed
    assert set(S.token_intervals(toks, lg, 1.0, 0, 0.3)) == {9, 20}       # <= .7: .25, .5 removed
    assert set(S.token_intervals(toks, lg, 1.0, 0, 0.2)) == {20}          # <= .8: three removed
    assert set(S.token_intervals(toks, lg, 1.0, 0, 0.76)) == {4, 7, 9, 20}  # <= .24: .25 is above, none removed
    # the largest is never removed, even at top_p = 0
    assert set(S.token_intervals(toks, lg, 1.0, 0, 0.0)) == {20}
    # unequal: p = [.1, .2, .3, .4] by logits; top_p = .65 removes .1 and .3 cumulative (<= .35)
    lg2 = [math.log(x) for x in (0.1, 0.2, 0.3, 0.4)]
    assert set(S.token_intervals(toks, lg2, 1.0, 0, 0.65)) == {9, 20}


def test_top_p_renormalises_over_the_top_k_set():
    toks, lg = [1, 2, 3], [math.log(0.5), math.log(0.3), math.log(0.2)]
    iv = _lengths(S.token_intervals(toks, lg, 1.0, 2, 0.6))
    # top-k keeps {1, 2} with probabilities 5/8, 3/8; top-p 0.6 removes the ascending prefix
    # with mass <= 0.4: 3/8 -> kept {1}
    assert set(iv) == {1} and iv[1] == pytest.approx(1.0)


def test_top_k_one_is_greedy():
    rng = np.random.default_rng(8)
    for _ in range(200):
        n = int(rng.integers(1, 12))
        toks = sorted(rng.choice(50, size=n, replace=False).tolist())
        lg = rng.integers(-3, 4, size=n).astype(float).tolist()           # frequent ties
        u = float(rng.random())
        tok, l = S.sample_token(toks, lg, 0.7, 1, 1.0, u)
        a_tok, a_l = argmax_lower_id(toks, lg)
        # ties at the maximum keep several tokens; the draw picks one of them
        assert l == a_l
        if lg.count(max(lg)) == 1:
            assert tok == a_tok


def test_temperature_limits():
    toks, lg = [3, 5, 8], [1.0, 0.0, -2.0]
    hot = _lengths(S.token_intervals(toks, lg, 1e9, 0, 1.0))
    assert all(abs(v - 1 / 3) < 1e-8 for v in hot.values())
    cold = _lengths(S.token_intervals(toks, lg, 1e-3, 0, 1.0))
    assert cold[3] > 1 - 1e-12


def test_inverse_cdf_in_ascending_token_order():
    toks, lg = [2, 4, 6], [0.0, 0.0, 0.0]
    assert S.sample_token(toks, lg, 1.0, 0, 1.0, 0.0)[0] == 2
    assert S.sample_token(toks, lg, 1.0, 0, 1.0, 0.34)[0] == 4
    assert S.sample_token(toks, lg, 1.0, 0, 1.0, 0.999999)[0] == 6
    # a fine grid of u draws each token in proportion to its probability
    lg2 = [0.5, -1.0, 2.0]
    iv = _lengths(S.token_intervals(toks, lg2, 0.8, 0, 1.0))
    N = 20000
    counts = {t: 0 for t in toks}
    for i in range(N):
        counts[S.sample_token(toks, lg2, 0.8, 0, 1.0, (i + 0.5) / N)[0]] += 1
    for t in toks:
        assert abs(counts[t] - N * iv[t]) <= 1.0


def test_sample_decode_language_and_greedy_special_case():
    w = I.tiny()
    trie = G.compile_catalog(w.catalog, w.sep_id, w.stop_id, w.vocab)
    emb = w.embedding()
    hid = w.hidden_states(0, 8)
    rng = np.random.default_rng(3)
    for q in range(8):
        u = rng.random(w.max_steps)
        toks, lg, st = S.sample_decode(trie, w.k, emb, hid[:, q], u, w.max_steps, 1.0, 0, 0.9)
        assert st == "ok" and D.replay_ok(trie, toks, w.k)
        ok, probs, exc = S.sample_teacher_force(trie, w.k, emb, hid[:, q], u, toks, lg, st, w.max_steps,
                                                1.0, 0, 0.9, exact_logits=True)
        assert ok and exc == 0, probs
        # top-k = 1 reproduces greedy decoding's logits at every position (ties at
        # the maximum may keep several tokens, all with the greedy logit)
        g = D.greedy_decode(trie, w.k, emb, hid[:, q], w.max_steps)
        s1 = S.sample_decode(trie, w.k, emb, hid[:, q], u, w.max_steps, 1.0, 1, 1.0)
        n = 0
        while n < min(len(g[0]), len(s1[0])) and g[0][n] == s1[0][n]:
            n += 1
        assert s1[1][:n] == g[1][:n]
        if n < min(len(g[0]), len(s1[0])):
            assert s1[1][n] == g[1][n]          # the first difference is a tie at the maximum


def test_checker_rejects_a_wrong_draw():
    toks, lg = [2, 4, 6], [0.0, 1.0, 2.0]
    iv = S.token_intervals(toks, lg, 1.0, 0, 1.0)
    u = (iv[4][0] + iv[4][1]) / 2
    assert not S.draw_excused(toks, lg, 1.0, 0, 1.0, u, 6)
    assert S.draw_excused(toks, lg, 1.0, 0, 1.0, iv[4][1] - 1e-7, 6)      # within rounding of the boundary
