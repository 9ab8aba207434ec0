"""Greedy constrained decoding, the host replay check and teacher forcing.

Sources:

* "Constraint made cheaper than no constraint", section "Masked sampling
  inside the sampler": each step filters the current node's edges, takes the
  argmax over the survivors (lower id on ties) and advances; an empty legal
  set is an error that stops the sequence.  Section "The whole loop on the
  device": the hidden state consumed at each step is the one the model
  produced for that step, so here it is indexed by (sequence, step) and does
  not depend on the path taken.  Section "The grammar as a trie over tokens":
  the host-side replay re-walks emitted tokens through the trie.
* "Understanding Inference for Systems Engineers", section 8.2 (teacher
  forcing: compare at every position while following the engine's own path,
  and judge a differing argmax by the oracle's own top-2 margin); section 7.5
  (forced spans: where the grammar admits exactly one continuation the
  model's scores are irrelevant, so that token is taken without a head read).

Status strings: "ok" (the stop token was emitted), "empty_mask" (no legal
token at some step) and "max_steps" (the step budget ran out first).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Sequence, Tuple

import numpy as np

from .grammar import PrefixTrie, WalkState, advance, legal_tokens, walk
from .head import abs_mass, argmax_lower_id, candidate_logits, dense_masked_argmax


def walk_fns(grammar):
    """(start, legal, advance) of a grammar: the token trie's walk, or the
    grammar object's own (oracle.chars.CharGrammar)."""
    if hasattr(grammar, "legal"):
        return grammar.start, grammar.legal, grammar.advance
    return (WalkState, lambda st, k: legal_tokens(grammar, st, k),
            lambda st, tok, k: advance(grammar, st, tok, k))

# Tolerances for Gaussian inputs: chosen logits within 1e-3 relative; a token
# may differ from the oracle's argmax only when the oracle's own top-2 margin
# is below 1e-5 relative.  Near zero, "relative" is taken against
# 2**-10 * sum_h |E[v,h] x[h]| so that a logit that cancels to almost nothing
# is judged at the scale of its own rounding error.
REL_TOL = 1e-3
MARGIN_TOL = 1e-5
FLOOR_SCALE = 2.0 ** -10


def greedy_decode(trie: PrefixTrie, k: int, emb_bits: np.ndarray, hidden_bits: np.ndarray,
                  max_steps: int, head: str = "sparse",
                  jump: bool = False) -> Tuple[List[int], List[float], str]:
    """Decode one sequence.  ``hidden_bits[t]`` is the bf16 hidden state of step t.

    ``head="dense"`` uses every vocabulary logit with the mask applied after
    (the post-logit pipeline); ``"sparse"`` computes only the legal rows.
    ``jump=True`` takes forced tokens without the head: from the second
    position on, a position whose legal set holds one token emits it with a
    NaN logit and computes nothing (the first token always comes from the head)."""
    start, legal_of, step = walk_fns(trie)
    st = start()
    toks: List[int] = []
    logits: List[float] = []
    for t in range(max_steps):
        legal = legal_of(st, k)
        if not legal:
            return toks, logits, "empty_mask"
        if jump and t > 0 and len(legal) == 1:
            toks.append(legal[0])
            logits.append(float("nan"))
            st = step(st, legal[0], k)
            if st.done:
                return toks, logits, "ok"
            continue
        if head == "dense":
            tok, lg = dense_masked_argmax(emb_bits, hidden_bits[t], legal)
        else:
            tok, lg = argmax_lower_id(legal, candidate_logits(emb_bits, hidden_bits[t], legal))
        toks.append(tok)
        logits.append(lg)
        st = step(st, tok, k)
        if st.done:
            return toks, logits, "ok"
    return toks, logits, "max_steps"


def forced_positions(trie: PrefixTrie, tokens: Sequence[int], k: int) -> List[int]:
    """Positions t >= 1 of a walkable output whose legal set holds exactly one
    token (where a forced-span decode emits without the head)."""
    start, legal_of, step = walk_fns(trie)
    st = start()
    out = []
    for t, tok in enumerate(tokens):
        if t > 0 and len(legal_of(st, k)) == 1:
            out.append(t)
        st = step(st, int(tok), k)
    return out


def replay_ok(trie: PrefixTrie, tokens: Sequence[int], k: int) -> bool:
    """Host replay: every token walkable and the string ends with the stop token."""
    start, legal_of, step = walk_fns(trie)
    st = start()
    for t in tokens:
        if int(t) not in legal_of(st, k):
            return False
        st = step(st, int(t), k)
    return st.done


def parse_pointers(trie: PrefixTrie, tokens: Sequence[int]) -> List[int]:
    """Split an output at separator/stop tokens and map each piece to its pointer id."""
    out, cur = [], []
    index = {s: i for i, s in enumerate(trie.catalog)}
    for t in tokens:
        if t == trie.sep or t == trie.stop:
            out.append(index.get(tuple(cur), -1))
            cur = []
        else:
            cur.append(t)
    return out


@dataclass
class ForcingReport:
    ok: bool = True
    problems: List[str] = field(default_factory=list)
    flips: int = 0                  # argmax differences excused by a sub-tolerance oracle margin
    steps: int = 0
    max_rel_err: float = 0.0

    def fail(self, msg: str):
        self.ok = False
        self.problems.append(msg)


def teacher_force(trie: PrefixTrie, k: int, emb_bits: np.ndarray, hidden_bits: np.ndarray,
                  toks: Sequence[int], logits: Sequence[float], status: str, max_steps: int,
                  exact: bool = False, jump: bool = False) -> ForcingReport:
    """Check an engine's emitted tokens/logits/status for one sequence.

    The oracle follows the engine's tokens.  At each step the token must be
    legal; with ``exact`` it must equal the oracle argmax and its logit must
    equal the exact dot product bit for bit (integer-valued inputs, where the
    fp32 sum is exact); otherwise the logit must be within ``REL_TOL`` and a
    differing token is excused only by an oracle top-2 margin under
    ``MARGIN_TOL``.  With ``jump`` a position t >= 1 whose legal set holds one
    token must carry a NaN logit (forced, no head read) and every other
    position a real one."""
    rep = ForcingReport()
    start, legal_of, step = walk_fns(trie)
    st = start()
    for t, (g_tok, g_log) in enumerate(zip(toks, logits)):
        rep.steps += 1
        legal = legal_of(st, k)
        if g_tok not in legal:
            rep.fail(f"step {t}: token {g_tok} not legal (legal={legal[:8]}...)")
            return rep
        if jump:
            forced = t > 0 and len(legal) == 1
            if forced != bool(np.isnan(g_log)):
                rep.fail(f"step {t}: forced={forced} but logit {float(g_log)!r}")
                return rep
            if forced:
                st = step(st, int(g_tok), k)
                if st.done and t != len(toks) - 1:
                    rep.fail(f"step {t}: tokens continue after stop")
                    return rep
                continue
        lg = candidate_logits(emb_bits, hidden_bits[t], legal)
        best_tok, best_l = argmax_lower_id(legal, lg)
        gi = legal.index(int(g_tok))
        r = float(lg[gi])
        if exact:
            if int(g_tok) != best_tok:
                rep.fail(f"step {t}: token {g_tok} != oracle {best_tok}")
            if float(np.float32(g_log)) != r:
                rep.fail(f"step {t}: logit {float(g_log)!r} != exact {r!r}")
        else:
            mass = abs_mass(emb_bits, hidden_bits[t], [int(g_tok), best_tok])
            scale = max(abs(r), FLOOR_SCALE * mass[0])
            err = abs(float(g_log) - r)
            rep.max_rel_err = max(rep.max_rel_err, err / scale if scale > 0 else 0.0)
            if err > REL_TOL * scale:
                rep.fail(f"step {t}: logit {float(g_log)} vs oracle {r} (tol {REL_TOL * scale:g})")
            if int(g_tok) != best_tok:
                bscale = max(abs(best_l), FLOOR_SCALE * mass[1])
                if best_l - r > MARGIN_TOL * bscale:
                    rep.fail(f"step {t}: token {g_tok} (logit {r}) != oracle {best_tok} "
                             f"(logit {best_l}); margin {best_l - r:g} above tolerance")
                else:
                    rep.flips += 1
        st = step(st, int(g_tok), k)
        if st.done and t != len(toks) - 1:
            rep.fail(f"step {t}: tokens continue after stop")
            return rep
    n = len(toks)
    if status == "ok":
        if not st.done:
            rep.fail("status ok but the output did not end with stop")
    elif status == "max_steps":
        if st.done or n != max_steps:
            rep.fail(f"status max_steps but done={st.done}, len={n}, max_steps={max_steps}")
    elif status == "empty_mask":
        if st.done or legal_of(st, k):
            rep.fail("status empty_mask but the oracle has legal tokens")
    else:
        rep.fail(f"unexpected status {status}")
    return rep
