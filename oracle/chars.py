"""Character-level constraint over a byte vocabulary (test infrastructure only).

Source: the pith.science review of arXiv 2608.12574 (key machinery): a
character-level trie of the valid strings whose nodes carry the vocabulary
tokens that are valid continuations there, so that every tokenization of a
catalog string is accepted, not only the canonical one; a token is valid at a
node when its characters can be walked from that node without leaving the trie
(it must not overshoot the strings).  The review computes the per-node sets
with Aho-Corasick matching of the vocabulary over the trie; this module takes
the definition instead: at a state - the bytes emitted since the last
separator and the pointers completed - a token is legal when appending its
bytes still gives a prefix of some catalog string not yet emitted.  The
separator and stop tokens keep the tool-pointer rules ("Constraint made
cheaper than no constraint", section "Masked sampling inside the sampler"): at
a complete, unspent string, the separator while another pointer is owed after
it, stop when it is the last one.

A grammar object here provides start(), legal(state, k) and advance(state,
token, k), which oracle.decode and oracle.sample use in place of the token
trie's walk.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, FrozenSet, List, Sequence, Set, Tuple


@dataclass(frozen=True)
class CharState:
    partial: bytes = b""              # bytes since the last separator
    spent: FrozenSet[int] = frozenset()
    done: bool = False


class CharGrammar:
    def __init__(self, strings: Sequence[bytes], vocab: Sequence[Tuple[int, bytes]], sep: int, stop: int):
        if len(set(strings)) != len(strings) or any(len(s) == 0 for s in strings):
            raise ValueError("catalog strings must be distinct and non-empty")
        ids = [i for i, _ in vocab]
        if len(set(ids)) != len(ids) or sep in ids or stop in ids or sep == stop:
            raise ValueError("token ids must be distinct and differ from the control ids")
        if any(len(b) == 0 for _, b in vocab):
            raise ValueError("empty token")
        self.strings = list(strings)
        self.index: Dict[bytes, int] = {s: i for i, s in enumerate(self.strings)}
        self.vocab = sorted((int(i), bytes(b)) for i, b in vocab)
        self.tok_bytes: Dict[int, bytes] = dict(self.vocab)
        self.sep, self.stop = int(sep), int(stop)
        # every prefix of every string -> the strings that start with it
        self.below: Dict[bytes, Set[int]] = {}
        for i, s in enumerate(self.strings):
            for L in range(len(s) + 1):
                self.below.setdefault(s[:L], set()).add(i)

    def start(self) -> CharState:
        return CharState()

    def _live(self, prefix: bytes, spent: FrozenSet[int]) -> bool:
        return any(i not in spent for i in self.below.get(prefix, ()))

    def legal(self, st: CharState, k: int) -> List[int]:
        """Sorted legal next tokens for a query owing exactly k pointers."""
        if st.done:
            return []
        out = [i for i, b in self.vocab if self._live(st.partial + b, st.spent)]
        p = self.index.get(st.partial)
        if p is not None and p not in st.spent:
            j = len(st.spent)
            if j + 1 < k:
                out.append(self.sep)
            if j + 1 == k:
                out.append(self.stop)
        return sorted(out)

    def advance(self, st: CharState, tok: int, k: int) -> CharState:
        if tok not in self.legal(st, k):
            raise ValueError(f"token {tok} is not legal at {st}")
        if tok in (self.sep, self.stop):
            return CharState(b"", st.spent | {self.index[st.partial]}, tok == self.stop)
        return CharState(st.partial + self.tok_bytes[tok], st.spent, False)

    def parse_pointers(self, tokens: Sequence[int]) -> List[int]:
        """Split an output at control tokens; map each piece's bytes to its string id."""
        out, cur = [], b""
        for t in tokens:
            if t in (self.sep, self.stop):
                out.append(self.index.get(cur, -1))
                cur = b""
            else:
                cur += self.tok_bytes[int(t)]
        return out

    def token_edges(self, prefix: bytes) -> Dict[int, bytes]:
        """The tokens whose bytes can be walked from the trie node of `prefix`,
        each with the prefix it leads to (no-repeat state ignored)."""
        return {i: prefix + b for i, b in self.vocab if (prefix + b) in self.below}


def segmentations(s: bytes, vocab: Sequence[Tuple[int, bytes]]) -> List[Tuple[int, ...]]:
    """Every way of writing s as a sequence of vocabulary tokens (brute force)."""
    if not s:
        return [()]
    out = []
    for i, b in vocab:
        if s.startswith(b):
            out.extend((i,) + rest for rest in segmentations(s[len(b):], vocab))
    return out


def char_language(strings: Sequence[bytes], vocab: Sequence[Tuple[int, bytes]], k: int, sep: int,
                  stop: int) -> Set[Tuple[int, ...]]:
    """All token strings of the k-pointer language at character level: ordered
    k-tuples of distinct catalog strings, each written in every possible
    tokenization, joined by the separator and ended by stop."""
    from itertools import permutations
    segs = {s: segmentations(s, vocab) for s in strings}
    out: Set[Tuple[int, ...]] = set()
    for combo in permutations(range(len(strings)), k):
        parts: List[Tuple[int, ...]] = [()]
        for j, i in enumerate(combo):
            ctl = (stop,) if j == k - 1 else (sep,)
            parts = [p + seg + ctl for p in parts for seg in segs[strings[i]]]
        out.update(parts)
    return out
