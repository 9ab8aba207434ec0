"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module only draws random numbers and arranges them into the shapes of the
workloads: catalogs of token-id strings, bf16 tied-embedding matrices and bf16
hidden states.  It holds none of the decoding method's arithmetic (no trie, no
mask, no dot product, no argmax), so that both the oracle and the CUDA path can
consume the same inputs without sharing any of the method.

bf16 values are carried as ``uint16`` bit patterns (numpy has no bf16 dtype).

Workload shapes follow the tool-pointer decoder described in "Constraint made
cheaper than no constraint" (sections "The grammar as a trie over tokens" and
"The sparse output layer": a 42-tool catalog, a 622 MB tied bf16 embedding
over a 151,936-token vocabulary) and the unstructured-enum falsifier of the
pith.science review of arXiv 2608.12574 (skeptic critique, concrete test:
1,000 random 32-character hex strings).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

MASTER_SEED = 20261202

# Sub-seed slots derived from the master seed with SeedSequence.spawn.
_SLOT_CATALOG, _SLOT_EMBEDDING, _SLOT_HIDDEN, _SLOT_ORDER, _SLOT_UNIFORM = range(5)


def sub_seed(slot: int, master: int = MASTER_SEED, extra: int = 0) -> np.random.SeedSequence:
    """Deterministic child seed ``slot`` of ``master`` (``extra`` selects a variant)."""
    return np.random.SeedSequence(entropy=master, spawn_key=(slot, extra))


def rng_for(slot: int, master: int = MASTER_SEED, extra: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(sub_seed(slot, master, extra)))


# ----------------------------------------------------------------------------
# bf16 bit patterns
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return uint16 bits.

    Inputs are finite by construction here; NaN handling is not needed."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def integer_bf16(rng: np.random.Generator, shape, lo: int = -8, hi: int = 8,
                 scale_log2: int = -4) -> np.ndarray:
    """bf16 bits of integers drawn uniformly from [lo, hi] times 2**scale_log2 (exact in bf16)."""
    ints = rng.integers(lo, hi + 1, size=shape, dtype=np.int32)
    return f32_to_bf16_bits(np.ldexp(ints.astype(np.float32), scale_log2))


def gaussian_bf16(rng: np.random.Generator, shape, std: float, chunk: int = 1 << 24) -> np.ndarray:
    """bf16 bits of N(0, std^2) samples, generated in chunks to bound host memory."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        out[s:e] = f32_to_bf16_bits(v)
    return out.reshape(shape)


# ----------------------------------------------------------------------------
# Catalog generators (token-id strings)
# ----------------------------------------------------------------------------

def tool_catalog(rng: np.random.Generator, n_names: int = 42, n_namespaces: int = 6,
                 vocab: int = 8192, min_len: int = 2, max_len: int = 8,
                 verbs_per_namespace: int = 4, suffix_pool: int = 512,
                 reserved: Sequence[int] = ()) -> List[Tuple[int, ...]]:
    """Tool names as token-id strings: a namespace prefix of 1-2 ids, a verb id
    drawn from a small per-namespace set (so names share sub-prefixes), then
    random suffix ids from a pool of ``suffix_pool`` ids.  Total length is
    ``min_len``..``max_len`` ids.  Ids in ``reserved`` never appear."""
    banned = set(int(r) for r in reserved)
    allowed = np.array([i for i in range(vocab) if i not in banned], dtype=np.int64)
    pick = rng.choice(allowed, size=suffix_pool + n_namespaces * (2 + verbs_per_namespace),
                      replace=False)
    pool = pick[:suffix_pool]
    rest = list(pick[suffix_pool:])
    namespaces = []
    for _ in range(n_namespaces):
        plen = int(rng.integers(1, 3))
        prefix = tuple(int(rest.pop()) for _ in range(plen))
        verbs = [int(rest.pop()) for _ in range(verbs_per_namespace)]
        namespaces.append((prefix, verbs))
    seen = set()
    out: List[Tuple[int, ...]] = []
    while len(out) < n_names:
        prefix, verbs = namespaces[int(rng.integers(n_namespaces))]
        length = int(rng.integers(max(min_len, len(prefix) + 1), max_len + 1))
        body = [verbs[int(rng.integers(len(verbs)))]]
        while len(prefix) + len(body) < length:
            body.append(int(pool[int(rng.integers(suffix_pool))]))
        name = tuple(prefix) + tuple(body[: length - len(prefix)])
        if name in seen:
            continue
        seen.add(name)
        out.append(name)
    return out


def hierarchical_catalog(rng: np.random.Generator, n_names: int = 1000, vocab: int = 151936,
                         min_len: int = 3, max_len: int = 10, n_namespaces: int = 16,
                         verbs_per_namespace: int = 4, groups_per_verb: int = 3,
                         subgroups_per_group: int = 2,
                         reserved: Sequence[int] = ()) -> List[Tuple[int, ...]]:
    """Prefix-structured tool names: namespace (1-2 ids) -> verb (1-2 ids) ->
    object group (1-2 ids) -> object subgroup (1 id) -> leaf suffix (the
    remaining ids), each level drawn from a small set under the level above so
    that names share prefixes.  The default parameters give
    (nodes-1)/total_tokens close to 0.40."""
    banned = set(int(r) for r in reserved)

    def fresh(n):
        out = []
        while len(out) < n:
            v = int(rng.integers(0, vocab))
            if v not in banned:
                out.append(v)
        return tuple(out)

    def level_item():
        return fresh(int(rng.integers(1, 3)))

    tree = []
    for _ in range(n_namespaces):
        ns = level_item()
        verbs = []
        for _ in range(verbs_per_namespace):
            vb = level_item()
            groups = [(level_item(), [fresh(1) for _ in range(subgroups_per_group)])
                      for _ in range(groups_per_verb)]
            verbs.append((vb, groups))
        tree.append((ns, verbs))
    seen = set()
    out: List[Tuple[int, ...]] = []
    while len(out) < n_names:
        ns, verbs = tree[int(rng.integers(len(tree)))]
        vb, groups = verbs[int(rng.integers(len(verbs)))]
        grp, subs = groups[int(rng.integers(len(groups)))]
        head = ns + vb + grp
        length = int(rng.integers(max(min_len, len(head) + 1), max_len + 1))
        name = head + subs[int(rng.integers(len(subs)))]
        if length > len(name):
            name = name + fresh(length - len(name))
        if name in seen:
            continue
        seen.add(name)
        out.append(name)
    return out


@dataclass
class HexVocab:
    """A 272-token hex subset of a larger vocabulary: 16 one-character and 256
    two-character hex tokens, each mapped to a distinct seeded token id."""
    one: dict
    two: dict

    @property
    def ids(self) -> List[int]:
        return sorted(list(self.one.values()) + list(self.two.values()))


def hex_vocab(rng: np.random.Generator, vocab: int = 151936, reserved: Sequence[int] = ()) -> HexVocab:
    banned = set(int(r) for r in reserved)
    allowed = np.array([i for i in range(vocab) if i not in banned], dtype=np.int64)
    ids = rng.choice(allowed, size=272, replace=False)
    digits = "0123456789abcdef"
    one = {d: int(ids[i]) for i, d in enumerate(digits)}
    two = {a + b: int(ids[16 + 16 * i + j]) for i, a in enumerate(digits) for j, b in enumerate(digits)}
    return HexVocab(one, two)


def hex_catalog(rng: np.random.Generator, hv: HexVocab, n_strings: int = 1000,
                n_chars: int = 32, p_one: float = 0.1) -> Tuple[List[str], List[Tuple[int, ...]]]:
    """Random ``n_chars``-character hex strings, each segmented into 1- or
    2-character hex tokens: at every position a 1-character token is taken
    with probability ``p_one`` (or when one character is left), else a
    2-character one.  Returns the strings and their token-id strings."""
    digits = np.array(list("0123456789abcdef"))
    seen = set()
    strings, toks = [], []
    while len(strings) < n_strings:
        s = "".join(digits[rng.integers(0, 16, size=n_chars)])
        if s in seen:
            continue
        seen.add(s)
        pos, ids = 0, []
        while pos < n_chars:
            if n_chars - pos == 1 or rng.random() < p_one:
                ids.append(hv.one[s[pos]])
                pos += 1
            else:
                ids.append(hv.two[s[pos:pos + 2]])
                pos += 2
        strings.append(s)
        toks.append(tuple(ids))
    # A segmentation may collide for different strings only if the strings are
    # equal, so the token strings are distinct as well.
    return strings, toks


# ----------------------------------------------------------------------------
# Character-level catalogs and byte vocabularies
# ----------------------------------------------------------------------------

def hex_byte_vocab(hv: HexVocab) -> List[Tuple[int, bytes]]:
    """The hex subset as (token id, bytes): 16 one-character and 256 two-character tokens."""
    out = [(i, d.encode()) for d, i in hv.one.items()] + [(i, d.encode()) for d, i in hv.two.items()]
    return sorted(out)


def char_tool_names(rng: np.random.Generator, n_names: int, n_namespaces: int = 8, verbs: int = 4,
                    objects: int = 3, max_suffix: int = 3) -> List[bytes]:
    """ASCII tool names ``namespace.verb_object[suffix]`` over a-z, '.' and '_':
    each level drawn from a small set under the level above (shared prefixes),
    then 0..max_suffix random letters."""
    letters = np.array(list("abcdefghijklmnopqrstuvwxyz"))

    def word(lo, hi):
        return "".join(letters[rng.integers(0, 26, size=int(rng.integers(lo, hi + 1)))])

    tree = [(word(2, 5), [(word(3, 6), [word(2, 6) for _ in range(objects)]) for _ in range(verbs)])
            for _ in range(n_namespaces)]
    seen, out = set(), []
    while len(out) < n_names:
        ns, vs = tree[int(rng.integers(len(tree)))]
        vb, obs = vs[int(rng.integers(len(vs)))]
        name = f"{ns}.{vb}_{obs[int(rng.integers(len(obs)))]}" + word(0, max_suffix)
        if name not in seen:
            seen.add(name)
            out.append(name.encode())
    return out


def char_bpe_vocab(rng: np.random.Generator, names: Sequence[bytes], vocab: int, n_pieces: int,
                   reserved: Sequence[int] = ()) -> List[Tuple[int, bytes]]:
    """A synthetic byte vocabulary for ``names``: every single character that
    occurs, the words between separators (also with their separator attached)
    and ``n_pieces`` random substrings of 2..4 characters, each given a distinct
    seeded token id."""
    pieces = set()
    for n in names:
        pieces.update(bytes([c]) for c in n)
        txt = n.decode()
        for part in txt.replace(".", " . ").replace("_", " _ ").split():
            pieces.add(part.encode())
        for sep in (".", "_"):
            for i, seg in enumerate(txt.split(sep)[:-1]):
                pieces.add((seg.split("." if sep == "_" else "_")[-1] + sep).encode())
    names = list(names)
    while len(pieces) < n_pieces + 40:
        n = names[int(rng.integers(len(names)))]
        L = int(rng.integers(2, 5))
        if len(n) >= L:
            i = int(rng.integers(0, len(n) - L + 1))
            pieces.add(n[i:i + L])
    banned = set(int(r) for r in reserved)
    allowed = np.array([i for i in range(vocab) if i not in banned], dtype=np.int64)
    ids = rng.choice(allowed, size=len(pieces), replace=False)
    return sorted(zip((int(i) for i in ids), sorted(pieces)))


def greedy_tokenize(s: bytes, vocab: Sequence[Tuple[int, bytes]]) -> Tuple[int, ...]:
    """Canonical tokenization: longest vocabulary match at each position."""
    by_bytes = {b: i for i, b in vocab}
    longest = max(len(b) for _, b in vocab)
    out, pos = [], 0
    while pos < len(s):
        for L in range(min(longest, len(s) - pos), 0, -1):
            i = by_bytes.get(s[pos:pos + L])
            if i is not None:
                out.append(i)
                pos += L
                break
        else:
            raise ValueError(f"{s!r} cannot be tokenized at {pos}")
    return tuple(out)


# ----------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------

@dataclass
class Workload:
    """One synthetic workload: a catalog, model shapes and query shape."""
    name: str
    vocab: int
    hidden: int
    catalog: List[Tuple[int, ...]]
    sep_id: int
    stop_id: int
    k: int
    batch: int
    n_queries: int
    max_fanout: int
    cand_cap: int
    residency: str                  # "const", "global" or "auto"
    emb_kind: str                   # "int" or "gauss"
    emb_std: float = 0.02
    hid_std: float = 1.0
    seed: int = MASTER_SEED
    notes: dict = field(default_factory=dict)
    # Character-level workloads: the catalog as byte strings and the byte
    # vocabulary as (token id, bytes); ``catalog`` then holds each string's
    # canonical (greedy longest-match) tokenization.
    char_strings: Optional[List[bytes]] = None
    char_vocab: Optional[List[Tuple[int, bytes]]] = None

    @property
    def max_depth(self) -> int:
        """Most tokens one pointer can take (characters, for a character-level catalog)."""
        if self.char_strings is not None:
            return max(len(p) for p in self.char_strings)
        return max(len(p) for p in self.catalog)

    @property
    def max_steps(self) -> int:
        # Each of the k pointers costs its tokens plus one control token.
        return self.k * (self.max_depth + 1)

    def embedding(self) -> np.ndarray:
        """bf16 bits [vocab, hidden] of the tied embedding."""
        rng = rng_for(_SLOT_EMBEDDING, self.seed, extra=self.vocab * 7919 + self.hidden)
        if self.emb_kind == "int":
            return integer_bf16(rng, (self.vocab, self.hidden))
        return gaussian_bf16(rng, (self.vocab, self.hidden), self.emb_std)

    def hidden_states(self, query0: int, n_queries: int, steps: Optional[int] = None) -> np.ndarray:
        """bf16 bits [steps, n_queries, hidden]: a fresh seeded state per (query, step).

        Query q's states depend only on q, so any batch split of the queries
        sees the same states."""
        steps = self.max_steps if steps is None else steps
        out = np.empty((steps, n_queries, self.hidden), dtype=np.uint16)
        for i in range(n_queries):
            rng = rng_for(_SLOT_HIDDEN, self.seed, extra=(query0 + i) * 16 + 1)
            if self.emb_kind == "int":
                out[:, i, :] = integer_bf16(rng, (steps, self.hidden))
            else:
                out[:, i, :] = gaussian_bf16(rng, (steps, self.hidden), self.hid_std)
        return out

    def uniforms(self, query0: int, n_queries: int, steps: Optional[int] = None) -> np.ndarray:
        """float32 [n_queries, steps] in [0, 1): the sampling draws of each
        (query, position), seeded per query like the hidden states."""
        steps = self.max_steps if steps is None else steps
        out = np.empty((n_queries, steps), dtype=np.float32)
        for i in range(n_queries):
            rng = rng_for(_SLOT_UNIFORM, self.seed, extra=(query0 + i) * 16 + 3)
            out[i] = rng.random(steps, dtype=np.float32)
        return out

    def order_rng(self, extra: int = 0) -> np.random.Generator:
        return rng_for(_SLOT_ORDER, self.seed, extra=extra)


def _tool42(vocab_for_ids: int = 8192) -> List[Tuple[int, ...]]:
    return tool_catalog(rng_for(_SLOT_CATALOG, extra=1), vocab=vocab_for_ids,
                        reserved=(vocab_for_ids - 2, vocab_for_ids - 1))


def tiny() -> Workload:
    """Vocab 8192, hidden 256, integer-valued bf16 (exact fp32 sums), 42 tools, k=3, B=1."""
    V = 8192
    return Workload("tiny", V, 256, _tool42(V), V - 2, V - 1, k=3, batch=1, n_queries=64,
                    max_fanout=256, cand_cap=256, residency="const", emb_kind="int")


def large_head() -> Workload:
    """Vocab 151936, hidden 2048 Gaussian bf16 (622 MB), the same 42 tools, k=5, B=1."""
    V = 151936
    return Workload("large_head", V, 2048, _tool42(8192), V - 2, V - 1, k=5, batch=1,
                    n_queries=1000, max_fanout=256, cand_cap=256, residency="const",
                    emb_kind="gauss")


def batched() -> Workload:
    """1000 prefix-structured tools (r~0.4), vocab 151936, hidden 4096, B=64, k=1."""
    V = 151936
    cat = hierarchical_catalog(rng_for(_SLOT_CATALOG, extra=3), vocab=V, reserved=(V - 2, V - 1))
    return Workload("batched", V, 4096, cat, V - 2, V - 1, k=1, batch=64, n_queries=4096,
                    max_fanout=256, cand_cap=256, residency="global", emb_kind="gauss")


def unstructured() -> Workload:
    """1000 random 32-char hex strings over a 272-token hex subset; B=16, k=2, C=4096."""
    V = 151936
    hv = hex_vocab(rng_for(_SLOT_CATALOG, extra=4), vocab=V, reserved=(V - 2, V - 1))
    strings, cat = hex_catalog(rng_for(_SLOT_CATALOG, extra=5), hv)
    return Workload("unstructured", V, 4096, cat, V - 2, V - 1, k=2, batch=16, n_queries=16,
                    max_fanout=4096, cand_cap=4096, residency="global", emb_kind="gauss",
                    notes={"hex_strings": strings, "hex_vocab": hv})


def tensor_batch() -> Workload:
    """The 1000-tool prefix catalog, vocab 151936, hidden 4096, B=256, k=3 (union GEMM path)."""
    w = batched()
    w.name = "tensor_batch"
    w.k, w.batch, w.n_queries = 3, 256, 4096
    return w


def _char_workload(name, V, H, names, cv, **kw) -> Workload:
    cat = [greedy_tokenize(n, cv) for n in names]
    return Workload(name, V, H, cat, V - 2, V - 1, char_strings=list(names), char_vocab=list(cv), **kw)


def char_tiny() -> Workload:
    """Character-level tool names (42, ASCII) over a synthetic byte vocabulary in
    vocab 8192, hidden 256, integer-valued bf16 (exact sums); k=3, B=1."""
    V = 8192
    names = char_tool_names(rng_for(_SLOT_CATALOG, extra=11), 42, n_namespaces=4, verbs=3, objects=3)
    cv = char_bpe_vocab(rng_for(_SLOT_CATALOG, extra=12), names, V, 120, reserved=(V - 2, V - 1))
    return _char_workload("char_tiny", V, 256, names, cv, k=3, batch=1, n_queries=64, max_fanout=256,
                          cand_cap=256, residency="const", emb_kind="int")


def char_tools() -> Workload:
    """200 character-level tool names over a 1200-piece byte vocabulary in vocab
    151936, hidden 2048 Gaussian (the large-head embedding); k=3, B=1."""
    V = 151936
    names = char_tool_names(rng_for(_SLOT_CATALOG, extra=13), 200)
    cv = char_bpe_vocab(rng_for(_SLOT_CATALOG, extra=14), names, V, 1200, reserved=(V - 2, V - 1))
    return _char_workload("char_tools", V, 2048, names, cv, k=3, batch=1, n_queries=1000, max_fanout=4096,
                          cand_cap=4096, residency="auto", emb_kind="gauss")


def char_hex() -> Workload:
    """The 1000 random 32-character hex strings at character level: any
    segmentation into the 272 hex tokens is legal; B=16, k=2."""
    V = 151936
    hv = hex_vocab(rng_for(_SLOT_CATALOG, extra=4), vocab=V, reserved=(V - 2, V - 1))
    strings, _ = hex_catalog(rng_for(_SLOT_CATALOG, extra=5), hv)
    return _char_workload("char_hex", V, 4096, [x.encode() for x in strings], hex_byte_vocab(hv), k=2, batch=16,
                          n_queries=16, max_fanout=4096, cand_cap=4096, residency="global", emb_kind="gauss")


WORKLOADS = {
    "tiny": tiny,
    "large_head": large_head,
    "batched": batched,
    "unstructured": unstructured,
    "tensor_batch": tensor_batch,
    "char_tiny": char_tiny,
    "char_tools": char_tools,
    "char_hex": char_hex,
}


def brute_catalogs() -> List[Tuple[List[Tuple[int, ...]], int, int, int]]:
    """Tiny catalogs for brute-force checks: (catalog, sep, stop, vocab).

    Includes prefix pairs ([a] and [a, b]), shared prefixes and a chain of
    three nested prefixes."""
    V = 16
    S, T = 14, 15
    return [
        ([(1,), (2,)], S, T, V),
        ([(1, 2), (1, 3), (4,)], S, T, V),
        ([(1,), (1, 2)], S, T, V),
        ([(1,), (1, 2), (1, 2, 3)], S, T, V),
        ([(3, 1), (3, 1, 2), (3, 4), (5, 6, 7)], S, T, V),
        ([(1, 2, 3), (1, 2, 4), (1, 5), (6,), (6, 7), (8, 9)], S, T, V),
    ]


def random_small_catalog(rng: np.random.Generator, vocab: int = 12, max_k: int = 6,
                         max_len: int = 4) -> List[Tuple[int, ...]]:
    """A random tiny catalog over ids [0, vocab-2) (the top two ids are reserved)."""
    n = int(rng.integers(1, max_k + 1))
    seen = set()
    out = []
    tries = 0
    while len(out) < n and tries < 1000:
        tries += 1
        L = int(rng.integers(1, max_len + 1))
        s = tuple(int(x) for x in rng.integers(0, 4, size=L))  # small alphabet: many shared prefixes
        if s not in seen:
            seen.add(s)
            out.append(s)
    return out
