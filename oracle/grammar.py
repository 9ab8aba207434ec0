"""The catalog as a prefix trie and the tool-pointer walk, written plainly.

Source: "Constraint made cheaper than no constraint" (coreyjames.ai):

* section "The grammar as a trie over tokens": the tool registry is a trie over
  the model's token ids; each node has outgoing edges, one per next token, and
  a node where a pointer ends also carries two control edges, "separator,
  another pointer follows" and "stop".
* section "Masked sampling inside the sampler": an edge is absent from the mask
  when no live (not yet emitted) pointer lies below it; the separator is legal
  only while another pointer is still owed and the stop edge only when none is;
  a per-pointer spent flag removes the control edges of a finished terminal
  while leaving its subtree walkable; completing a pointer walks its path.
* section "The sparse output layer": the compiler refuses a node with more
  than 256 edges (the cap is a parameter here).

This module does not use counts or a CSR layout: "live below an edge" is
computed by scanning the set of pointers whose string starts with the edge's
prefix, minus the spent set.  Readings of points the page leaves open:

* fan-out counts every edge of a node, control edges included;
* the compiler refuses empty strings, duplicate strings, strings that contain
  the separator or stop id, ids outside [0, vocab) and separator == stop;
* a pointer completes when its separator or stop edge is taken.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, FrozenSet, List, Optional, Sequence, Tuple

Str = Tuple[int, ...]


class CompileError(ValueError):
    """A catalog the compiler must refuse; ``reason`` names the rule."""

    def __init__(self, reason: str, detail: str = ""):
        super().__init__(f"{reason}: {detail}" if detail else reason)
        self.reason = reason


@dataclass
class PrefixTrie:
    catalog: List[Str]
    sep: int
    stop: int
    vocab: int
    below: Dict[Str, FrozenSet[int]] = field(default_factory=dict)     # prefix -> pointer ids below it (incl. ending there)
    children: Dict[Str, List[int]] = field(default_factory=dict)       # prefix -> sorted next tokens
    terminal: Dict[Str, int] = field(default_factory=dict)             # prefix -> pointer id ending there

    @property
    def n_nodes(self) -> int:
        return len(self.below)

    def fanout(self, prefix: Str) -> int:
        return len(self.children.get(prefix, ())) + (2 if prefix in self.terminal else 0)

    @property
    def n_edges(self) -> int:
        return sum(self.fanout(p) for p in self.below)

    @property
    def max_fanout(self) -> int:
        return max(self.fanout(p) for p in self.below)


def compile_catalog(catalog: Sequence[Sequence[int]], sep: int, stop: int, vocab: int,
                    max_fanout: int = 256) -> PrefixTrie:
    """Build the prefix trie, applying the compile-time refusals."""
    if vocab <= 0 or not (0 <= sep < vocab) or not (0 <= stop < vocab) or sep == stop:
        raise CompileError("invalid_arg", "control ids must be distinct ids in [0, vocab)")
    if len(catalog) == 0:
        raise CompileError("invalid_arg", "empty catalog")
    cat: List[Str] = []
    seen = set()
    for i, s in enumerate(catalog):
        s = tuple(int(t) for t in s)
        if len(s) == 0:
            raise CompileError("empty_string", f"entry {i}")
        for t in s:
            if t == sep or t == stop:
                raise CompileError("control_collision", f"entry {i}")
            if not (0 <= t < vocab):
                raise CompileError("token_range", f"entry {i}")
        if s in seen:
            raise CompileError("duplicate", f"entry {i}")
        seen.add(s)
        cat.append(s)
    below: Dict[Str, set] = {(): set()}
    children: Dict[Str, set] = {}
    terminal: Dict[Str, int] = {}
    for pid, s in enumerate(cat):
        below[()].add(pid)
        for d in range(1, len(s) + 1):
            below.setdefault(s[:d], set()).add(pid)
            children.setdefault(s[:d - 1], set()).add(s[d - 1])
        terminal[s] = pid
    trie = PrefixTrie(cat, sep, stop, vocab,
                      below={p: frozenset(v) for p, v in below.items()},
                      children={p: sorted(v) for p, v in children.items()},
                      terminal=terminal)
    for p in trie.below:
        if trie.fanout(p) > max_fanout:
            raise CompileError("fanout", f"node {p} has {trie.fanout(p)} edges > {max_fanout}")
    return trie


@dataclass(frozen=True)
class WalkState:
    """Where one sequence is: the prefix inside the current pointer, the set of
    pointers already emitted, and whether it has stopped."""
    prefix: Str = ()
    spent: FrozenSet[int] = frozenset()
    done: bool = False


def legal_tokens(trie: PrefixTrie, st: WalkState, k: int) -> List[int]:
    """Sorted legal next tokens at ``st`` for a query owing exactly ``k`` pointers."""
    if st.done:
        return []
    out = []
    for c in trie.children.get(st.prefix, ()):
        if any(p not in st.spent for p in trie.below[st.prefix + (c,)]):
            out.append(c)
    p = trie.terminal.get(st.prefix)
    if p is not None and p not in st.spent:
        j = len(st.spent)
        if j + 1 < k:
            out.append(trie.sep)
        if j + 1 == k:
            out.append(trie.stop)
    return sorted(out)


def advance(trie: PrefixTrie, st: WalkState, tok: int, k: int) -> WalkState:
    """The state after emitting ``tok`` (which must be legal)."""
    if tok not in legal_tokens(trie, st, k):
        raise ValueError(f"token {tok} is not legal at {st}")
    if tok == trie.sep or tok == trie.stop:
        p = trie.terminal[st.prefix]
        return WalkState((), st.spent | {p}, tok == trie.stop)
    return WalkState(st.prefix + (tok,), st.spent, False)


def walk(trie: PrefixTrie, tokens: Sequence[int], k: int) -> Optional[WalkState]:
    """Replay ``tokens`` from the start state; None if some token cannot be walked."""
    st = WalkState()
    for t in tokens:
        if t not in legal_tokens(trie, st, k):
            return None
        st = advance(trie, st, t, k)
    return st


def all_walks(trie: PrefixTrie, k: int, limit: int = 200000) -> set:
    """Every token string the walk can produce from the start state to a stop."""
    out = set()
    stack = [((), WalkState())]
    while stack:
        seq, st = stack.pop()
        if st.done:
            out.add(seq)
            if len(out) > limit:
                raise RuntimeError("too many walks")
            continue
        for t in legal_tokens(trie, st, k):
            stack.append((seq + (t,), advance(trie, st, t, k)))
    return out
