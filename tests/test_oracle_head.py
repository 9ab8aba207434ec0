"""Pins for the oracle's logits and argmax (CPU only).

* bf16 decoding is checked on bit patterns whose values are known by hand.
* candidate logits are checked against exact integer arithmetic on the
  integer-valued workload (values k * 2**-4), which catches a transposed
  operand, a wrong row or a dropped term.
* the tie-break is checked on hand-built exact ties (tests/golden/tie_examples.json).
* the sparse argmax is checked against the dense logits-then-mask pipeline
  ("Understanding Inference for Systems Engineers", section 7.5).
"""
import json
import os

import numpy as np
import pytest

from oracle import head as H
from trie_constrained_decoding_gb300 import inputs as I
from conftest import GOLDEN


def test_bf16_decode_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3E80, 0x0000, 0x8000, 0x4120, 0x0001, 0x7F7F, 0x3DCC], dtype=np.uint16)
    want = [1.0, -2.0, 0.25, 0.0, -0.0, 10.0, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, 0.099609375]
    got = H.bf16_bits_to_f64(bits)
    for g, w in zip(got, want):
        assert g == w
    assert np.signbit(got[4])


def test_generator_rounding_matches_decode():
    # f32 -> bf16 rounding of the input generator, decoded back: exact on bf16-representable values
    vals = np.array([1.0, -2.5, 0.0625, -0.5, 3.0, 1.0 + 2 ** -7], dtype=np.float32)
    assert list(H.bf16_bits_to_f64(I.f32_to_bf16_bits(vals))) == [float(v) for v in vals]
    # ties to even: 1 + 2**-8 is halfway between 1 and 1 + 2**-7 -> 1.0
    assert H.bf16_bits_to_f64(I.f32_to_bf16_bits(np.array([1.0 + 2 ** -8], np.float32)))[0] == 1.0


def test_candidate_logits_exact_integers():
    rng = I.rng_for(9, extra=2)
    V, Hd = 300, 256
    emb = I.integer_bf16(rng, (V, Hd))
    x = I.integer_bf16(rng, (Hd,))
    # integer view: every value is an integer m * 2**-4 with |m| <= 8
    emb_i = np.rint(H.bf16_bits_to_f64(emb) * 16).astype(np.int64)
    x_i = np.rint(H.bf16_bits_to_f64(x) * 16).astype(np.int64)
    assert np.abs(emb_i).max() <= 8 and np.abs(x_i).max() <= 8
    toks = [0, 17, 299, 5, 5]
    got = H.candidate_logits(emb, x, toks)
    for t, g in zip(toks, got):
        exact = sum(int(a) * int(b) for a, b in zip(emb_i[t], x_i))   # python integers: exact
        assert g * 256 == exact
    # the abs-mass is the same sum over magnitudes
    mass = H.abs_mass(emb, x, [17])
    assert mass[0] * 256 == sum(abs(int(a) * int(b)) for a, b in zip(emb_i[17], x_i))


def test_logits_are_row_times_vector_not_column():
    # a non-square embedding: a transposed operand would not even index
    emb = I.f32_to_bf16_bits(np.array([[1, 2, 3], [4, 5, 6]], np.float32))
    x = I.f32_to_bf16_bits(np.array([1, 0, -1], np.float32))
    assert list(H.candidate_logits(emb, x, [1, 0])) == [-2.0, -2.0]
    x = I.f32_to_bf16_bits(np.array([0, 1, 0], np.float32))
    assert list(H.candidate_logits(emb, x, [0, 1])) == [2.0, 5.0]


def _golden_ties():
    with open(os.path.join(GOLDEN, "tie_examples.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _golden_ties(), ids=lambda c: c["name"])
def test_golden_ties(case):
    V = 1 + max(int(r) for r in case["rows"])
    Hd = len(case["x"])
    emb = np.zeros((V, Hd), dtype=np.uint16)
    for r, vals in case["rows"].items():
        emb[int(r)] = [int(v, 16) for v in vals]
    x = np.array([int(v, 16) for v in case["x"]], dtype=np.uint16)
    legal = case["legal"]
    tok, lg = H.argmax_lower_id(legal, H.candidate_logits(emb, x, legal))
    assert (tok, lg) == (case["winner"], case["logit"])
    dtok, dlg = H.dense_masked_argmax(emb, x, legal)
    assert (dtok, dlg) == (case["winner"], case["logit"])


def test_sparse_equals_dense_random():
    rng = I.rng_for(9, extra=3)
    V, Hd = 500, 64
    for trial in range(30):
        emb = I.integer_bf16(rng, (V, Hd), lo=-2, hi=2)     # small range: many exact ties
        x = I.integer_bf16(rng, (Hd,), lo=-1, hi=1)
        legal = sorted(set(int(t) for t in rng.integers(0, V, size=int(rng.integers(1, 40)))))
        s = H.argmax_lower_id(legal, H.candidate_logits(emb, x, legal))
        d = H.dense_masked_argmax(emb, x, legal)
        assert s == d


def test_empty_candidates_raise():
    with pytest.raises(ValueError):
        H.argmax_lower_id([], [])
