"""Negative controls for the oracle's pins ("Understanding Inference for
Systems Engineers", section 8.4: a check that cannot fail proves nothing).

Each test plants one plausible mistake in a copy of an oracle function, on the
CPU, and shows that the pin meant to catch it does fail."""
import json
import os

import numpy as np

from oracle import grammar as G
from oracle import head as H
from oracle import language as L
from trie_constrained_decoding_gb300 import inputs as I
from conftest import GOLDEN


def _agrees_with_definition(legal_fn) -> bool:
    for cat, sep, stop, V in I.brute_catalogs():
        trie = G.compile_catalog(cat, sep, stop, V)
        for k in range(1, min(3, len(cat)) + 1):
            lang = L.language(trie.catalog, k, sep, stop)
            for u in sorted(L.reachable_prefixes(lang)):
                st = G.WalkState()
                for t in u:
                    if t in (sep, stop):
                        p = trie.terminal[st.prefix]
                        st = G.WalkState((), st.spent | {p}, t == stop)
                    else:
                        st = G.WalkState(st.prefix + (t,), st.spent, False)
                if set(legal_fn(trie, st, k)) != L.mask_by_definition(lang, u):
                    return False
    return True


def test_true_walk_passes():
    assert _agrees_with_definition(G.legal_tokens)


def test_catches_ignored_spent_flag():
    def bad(trie, st, k):
        if st.done:
            return []
        out = [c for c in trie.children.get(st.prefix, ())
               if any(p not in st.spent for p in trie.below[st.prefix + (c,)])]
        if st.prefix in trie.terminal:              # planted: spent flag not consulted
            j = len(st.spent)
            out += [trie.sep] if j + 1 < k else []
            out += [trie.stop] if j + 1 == k else []
        return sorted(out)
    assert not _agrees_with_definition(bad)


def test_catches_off_by_one_owed_rule():
    def bad(trie, st, k):
        if st.done:
            return []
        out = [c for c in trie.children.get(st.prefix, ())
               if any(p not in st.spent for p in trie.below[st.prefix + (c,)])]
        p = trie.terminal.get(st.prefix)
        if p is not None and p not in st.spent:
            j = len(st.spent)
            out += [trie.sep] if j < k else []        # planted: j < k instead of j + 1 < k
            out += [trie.stop] if j + 1 == k else []
        return sorted(out)
    assert not _agrees_with_definition(bad)


def test_catches_count_without_spent():
    def bad(trie, st, k):
        if st.done:
            return []
        out = [c for c in trie.children.get(st.prefix, ())
               if len(trie.below[st.prefix + (c,)]) > 0]    # planted: all pointers counted as live
        p = trie.terminal.get(st.prefix)
        if p is not None and p not in st.spent:
            j = len(st.spent)
            out += [trie.sep] if j + 1 < k else []
            out += [trie.stop] if j + 1 == k else []
        return sorted(out)
    assert not _agrees_with_definition(bad)


def test_catches_upper_id_tie_break():
    def bad_argmax(tokens, logits):
        best_t, best_l = None, None
        for t, l in zip(tokens, logits):
            if best_t is None or l > best_l or (l == best_l and t > best_t):   # planted
                best_t, best_l = int(t), float(l)
        return best_t, best_l
    with open(os.path.join(GOLDEN, "tie_examples.json")) as f:
        cases = json.load(f)["cases"]
    failures = 0
    for case in cases:
        V = 1 + max(int(r) for r in case["rows"])
        emb = np.zeros((V, len(case["x"])), np.uint16)
        for r, vals in case["rows"].items():
            emb[int(r)] = [int(v, 16) for v in vals]
        x = np.array([int(v, 16) for v in case["x"]], np.uint16)
        got = bad_argmax(case["legal"], H.candidate_logits(emb, x, case["legal"]))
        failures += got != (case["winner"], case["logit"])
    assert failures >= 3


def test_catches_dropped_term_in_dot():
    rng = I.rng_for(9, extra=6)
    emb = I.integer_bf16(rng, (50, 256))
    x = I.integer_bf16(rng, (256,))
    emb_i = np.rint(H.bf16_bits_to_f64(emb) * 16).astype(np.int64)
    x_i = np.rint(H.bf16_bits_to_f64(x) * 16).astype(np.int64)

    def bad_logits(e, xb, toks):   # planted: the last hidden element is dropped
        rows = H.bf16_bits_to_f64(e[np.asarray(toks)])[:, :-1]
        return rows @ H.bf16_bits_to_f64(xb)[:-1]
    toks = list(range(50))
    got = bad_logits(emb, x, toks)
    exact = emb_i[toks] @ x_i
    assert np.any(got * 256 != exact)
