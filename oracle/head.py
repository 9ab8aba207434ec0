"""Logits and the greedy choice, in fp64.

Sources:

* "Constraint made cheaper than no constraint", section "The sparse output
  layer": one dot product of the tied embedding row with the hidden state per
  legal candidate; section "Masked sampling inside the sampler": argmax over
  the surviving tokens with ties broken toward the lower token id (ties are
  real: the smallest measured top-2 margin was zero).
* "Understanding Inference for Systems Engineers", section 3.8 (greedy takes
  the argmax, the lowest id on a tie) and section 7.5 (the production
  pipeline: logits for every token, minus infinity written into every
  disallowed logit, then the argmax).

bf16 inputs are carried as uint16 bit patterns.  A bf16 value has an 8-bit
significand, so a product of two bf16 values is exact in fp64 and the fp64
sum of H such products differs from the real sum by at most H * 2**-53
relative to the sum of magnitudes: the oracle's logits are the exact dot
products to far below any fp32 rounding.
"""
from __future__ import annotations

from typing import Iterable, Sequence, Tuple

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bit patterns: a bf16 value is the upper half of an fp32 value."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def candidate_logits(emb_bits: np.ndarray, x_bits: np.ndarray, tokens: Sequence[int]) -> np.ndarray:
    """logit[c] = sum_h E[tokens[c], h] * x[h] in fp64, one row per candidate."""
    if len(tokens) == 0:
        return np.zeros(0, dtype=np.float64)
    rows = bf16_bits_to_f64(emb_bits[np.asarray(tokens, dtype=np.int64)])
    x = bf16_bits_to_f64(x_bits)
    return rows @ x


def abs_mass(emb_bits: np.ndarray, x_bits: np.ndarray, tokens: Sequence[int]) -> np.ndarray:
    """sum_h |E[v, h] * x[h]| per candidate: the scale of a logit's rounding error."""
    if len(tokens) == 0:
        return np.zeros(0, dtype=np.float64)
    rows = np.abs(bf16_bits_to_f64(emb_bits[np.asarray(tokens, dtype=np.int64)]))
    return rows @ np.abs(bf16_bits_to_f64(x_bits))


def argmax_lower_id(tokens: Sequence[int], logits: Iterable[float]) -> Tuple[int, float]:
    """The candidate with the largest logit; among equal logits the lowest token id.

    Equality is IEEE equality, so -0.0 and +0.0 tie."""
    best_t, best_l = None, None
    for t, l in zip(tokens, logits):
        if best_t is None or l > best_l or (l == best_l and t < best_t):
            best_t, best_l = int(t), float(l)
    if best_t is None:
        raise ValueError("empty candidate set")
    return best_t, best_l


def dense_masked_argmax(emb_bits: np.ndarray, x_bits: np.ndarray, legal: Iterable[int]) -> Tuple[int, float]:
    """The post-logit pipeline taken literally: every vocabulary logit, minus
    infinity outside the legal set, then the first (lowest-id) maximum."""
    logits = bf16_bits_to_f64(emb_bits) @ bf16_bits_to_f64(x_bits)
    mask = np.zeros(logits.shape[0], dtype=bool)
    mask[np.asarray(list(legal), dtype=np.int64)] = True
    if not mask.any():
        raise ValueError("empty mask")
    logits[~mask] = -np.inf
    i = int(np.argmax(logits))          # numpy returns the first maximum: the lowest id
    return i, float(logits[i])
