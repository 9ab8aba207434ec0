"""The k-pointer output language and its next-token mask, by definition.

Sources:

* "GLRMask" (constrained decoding with weighted automata), introduction: the
  next-token mask at an emitted prefix u is the set of tokens v for which some
  continuation w makes u v w a member of the language L.  Here the language is
  over token ids directly (each token stands for itself), because the catalog
  is compiled over the model's own token ids ("Constraint made cheaper than no
  constraint", section "The grammar as a trie over tokens").
* "Constraint made cheaper than no constraint", section "Masked sampling inside
  the sampler": exactly k pointers come out, separated by the separator token
  and ended by the stop token, and no pointer repeats.

So, for a catalog P = {p_1..p_K} of distinct token-id strings,

    L_k = { p_i1 SEP p_i2 SEP ... p_ik STOP : i_1..i_k pairwise distinct }.

Everything here is brute force and only usable on tiny catalogs.
"""
from __future__ import annotations

from itertools import permutations
from typing import Iterable, Sequence, Set, Tuple

Str = Tuple[int, ...]


def language(catalog: Sequence[Str], k: int, sep: int, stop: int) -> Set[Str]:
    """All members of L_k, enumerated over ordered k-tuples of distinct pointers."""
    out: Set[Str] = set()
    if k <= 0 or k > len(catalog):
        return out
    for choice in permutations(range(len(catalog)), k):
        s: list = []
        for j, i in enumerate(choice):
            s.extend(catalog[i])
            s.append(stop if j == k - 1 else sep)
        out.add(tuple(s))
    return out


def mask_by_definition(lang: Iterable[Str], u: Str) -> Set[int]:
    """{v : exists w with u + (v,) + w in lang}, checked against every member."""
    n = len(u)
    return {s[n] for s in lang if len(s) > n and s[:n] == u}


def reachable_prefixes(lang: Iterable[Str]) -> Set[Str]:
    """Every prefix (including the empty one and the full strings) of a member."""
    out: Set[Str] = set()
    for s in lang:
        for i in range(len(s) + 1):
            out.add(s[:i])
    return out
