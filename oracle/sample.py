"""Sampling over the legal candidates, in fp64 (test infrastructure only).

Source: "Understanding Inference for Systems Engineers", section 3.8: sampling
draws from softmax(logits / temperature) after optionally restricting to the
top-k highest logits and to the smallest set of tokens whose cumulative
probability exceeds top-p.  Each restriction has an exact tie rule: top-k is a
value threshold, so the kept set can hold more than k tokens when logits tie;
top-p removes an ascending prefix, and among equal probabilities the highest
token id survives.

Readings taken where the page is silent:

* Order: top-k first, then top-p over the probabilities renormalised on the
  top-k set (the order the page names them in).
* "Ascending prefix": the kept candidates ordered by (logit, token id)
  ascending; a candidate is removed when the probability mass up to and
  including it in that order is at most 1 - top_p; the last candidate in that
  order is never removed.
* The draw: one uniform u in [0, 1) per (sequence, position), supplied by the
  caller (random numbers are inputs, not generated here); the token is the
  first kept candidate, in ascending token-id order, whose cumulative
  renormalised probability exceeds u (the last kept candidate if rounding
  leaves none).
* temperature > 0; top_k <= 0 disables top-k; top_p >= 1 disables top-p.

Every function here takes the candidates in ascending token order, the order
the legal set comes in.
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence, Tuple

import numpy as np


def kept_top_k(logits: Sequence[float], top_k: int) -> List[bool]:
    """Value threshold: keep every candidate whose logit is at least the
    top_k-th largest, i.e. fewer than top_k logits are strictly larger."""
    n = len(logits)
    if top_k <= 0 or top_k >= n:
        return [True] * n
    return [sum(1 for m in logits if m > l) < top_k for l in logits]


def restrict(tokens: Sequence[int], logits: Sequence[float], temperature: float, top_k: int,
             top_p: float) -> Tuple[List[int], List[float]]:
    """The kept candidates (ascending token order) and their unnormalised
    weights exp((logit - max) / temperature) after top-k and top-p."""
    if not tokens:
        raise ValueError("empty candidate set")
    if not temperature > 0:
        raise ValueError("temperature must be positive")
    keep = kept_top_k(logits, top_k)
    idx = [i for i in range(len(tokens)) if keep[i]]
    m = max(logits[i] for i in idx)
    w = {i: math.exp((logits[i] - m) / temperature) for i in idx}
    if top_p < 1.0:
        total = sum(w.values())
        asc = sorted(idx, key=lambda i: (logits[i], tokens[i]))
        cut = 1.0 - top_p
        run = 0.0
        removed = set()
        for i in asc[:-1]:                      # the largest is never removed
            run += w[i] / total
            if run <= cut:
                removed.add(i)
            else:
                break
        idx = [i for i in idx if i not in removed]
    return [int(tokens[i]) for i in idx], [w[i] for i in idx]


def token_intervals(tokens: Sequence[int], logits: Sequence[float], temperature: float, top_k: int,
                    top_p: float) -> Dict[int, Tuple[float, float]]:
    """The sub-interval of [0, 1) of the uniform that draws each kept token."""
    kt, kw = restrict(tokens, logits, temperature, top_k, top_p)
    total = sum(kw)
    out, lo = {}, 0.0
    for t, wt in zip(kt, kw):
        hi = lo + wt / total
        out[t] = (lo, hi)
        lo = hi
    return out


def sample_token(tokens: Sequence[int], logits: Sequence[float], temperature: float, top_k: int,
                 top_p: float, u: float) -> Tuple[int, float]:
    """The drawn token and its logit."""
    kt, kw = restrict(tokens, logits, temperature, top_k, top_p)
    total = sum(kw)
    run = 0.0
    choice = kt[-1]
    for t, wt in zip(kt, kw):
        run += wt / total
        if run > u:
            choice = t
            break
    return choice, float(logits[list(tokens).index(choice)])


# ---------------------------------------------------------------- decode loop and checker

def sample_decode(trie, k: int, emb_bits: np.ndarray, hidden_bits: np.ndarray, uniforms: Sequence[float],
                  max_steps: int, temperature: float, top_k: int, top_p: float,
                  jump: bool = False) -> Tuple[List[int], List[float], str]:
    """Constrained decoding with sampling: greedy_decode with the argmax
    replaced by sample_token using uniforms[t] at position t (forced positions
    with ``jump`` draw nothing and report a NaN logit)."""
    from .decode import walk_fns
    from .head import candidate_logits
    start, legal_of, step = walk_fns(trie)
    st = start()
    toks: List[int] = []
    logits: List[float] = []
    for t in range(max_steps):
        legal = legal_of(st, k)
        if not legal:
            return toks, logits, "empty_mask"
        if jump and t > 0 and len(legal) == 1:
            tok, lg = legal[0], float("nan")
        else:
            lg_all = candidate_logits(emb_bits, hidden_bits[t], legal)
            tok, lg = sample_token(legal, list(lg_all), temperature, top_k, top_p, float(uniforms[t]))
        toks.append(tok)
        logits.append(lg)
        st = step(st, tok, k)
        if st.done:
            return toks, logits, "ok"
    return toks, logits, "max_steps"


def draw_excused(tokens: Sequence[int], logits: Sequence[float], temperature: float, top_k: int, top_p: float,
                 u: float, got: int, u_tol: float = 1e-5, logit_tol: float = 1e-6) -> bool:
    """Whether drawing `got` instead of the exact draw is explained by rounding:
    u lies within u_tol of got's interval, or got sits on a top-k or top-p
    boundary (its logit within logit_tol, relative, of the top-k threshold, or
    the ascending mass at it within u_tol of 1 - top_p)."""
    iv = token_intervals(tokens, logits, temperature, top_k, top_p)
    if got in iv:
        lo, hi = iv[got]
        return lo - u_tol <= u < hi + u_tol
    if got not in tokens:
        return False
    i = list(tokens).index(got)
    scale = max(1e-30, max(abs(float(x)) for x in logits))
    if 0 < top_k < len(tokens):
        tau = sorted(logits, reverse=True)[top_k - 1]
        if abs(float(logits[i]) - tau) <= logit_tol * scale:
            return True
    if top_p < 1.0:
        keep = kept_top_k(logits, top_k)
        idx = [j for j in range(len(tokens)) if keep[j]]
        m = max(logits[j] for j in idx)
        w = {j: math.exp((logits[j] - m) / temperature) for j in idx}
        total = sum(w.values())
        run = 0.0
        for j in sorted(idx, key=lambda j: (logits[j], tokens[j])):
            run += w[j] / total
            if j == i:
                return abs(run - (1.0 - top_p)) <= u_tol
    return False


def sample_teacher_force(trie, k: int, emb_bits: np.ndarray, hidden_bits: np.ndarray, uniforms: Sequence[float],
                         toks: Sequence[int], logits: Sequence[float], status: str, max_steps: int,
                         temperature: float, top_k: int, top_p: float, jump: bool = False,
                         exact_logits: bool = False):
    """Follow an engine's sampled output and check every position: the token
    is legal; it is the exact draw or its difference is excused by rounding
    (draw_excused); its logit equals the exact dot product (``exact_logits``)
    or is within the greedy checker's relative tolerance; forced positions
    (``jump``) carry NaN.  Returns (ok, problems, excused_draws)."""
    from .decode import FLOOR_SCALE, REL_TOL, walk_fns
    from .head import abs_mass, candidate_logits
    start, legal_of, step = walk_fns(trie)
    st = start()
    problems: List[str] = []
    excused = 0
    for t, (g_tok, g_log) in enumerate(zip(toks, logits)):
        legal = legal_of(st, k)
        g_tok = int(g_tok)
        if g_tok not in legal:
            return False, [f"step {t}: token {g_tok} not legal"], excused
        forced = jump and t > 0 and len(legal) == 1
        if forced != (jump and bool(np.isnan(g_log))):
            return False, [f"step {t}: forced={forced} but logit {g_log!r}"], excused
        if not forced:
            lg = list(candidate_logits(emb_bits, hidden_bits[t], legal))
            want, _ = sample_token(legal, lg, temperature, top_k, top_p, float(uniforms[t]))
            if want != g_tok:
                if draw_excused(legal, lg, temperature, top_k, top_p, float(uniforms[t]), g_tok):
                    excused += 1
                else:
                    problems.append(f"step {t}: drew {g_tok}, exact draw {want} (u={float(uniforms[t])!r})")
            r = lg[legal.index(g_tok)]
            if exact_logits:
                if float(np.float32(g_log)) != r:
                    problems.append(f"step {t}: logit {float(g_log)!r} != exact {r!r}")
            else:
                scale = max(abs(r), FLOOR_SCALE * float(abs_mass(emb_bits, hidden_bits[t], [g_tok])[0]))
                if abs(float(g_log) - r) > REL_TOL * scale:
                    problems.append(f"step {t}: logit {float(g_log)} vs exact {r}")
        st = step(st, g_tok, k)
        if st.done and t != len(toks) - 1:
            return False, problems + [f"step {t}: tokens continue after stop"], excused
    n = len(toks)
    if status == "ok" and not st.done:
        problems.append("status ok but no stop")
    if status == "max_steps" and (st.done or n != max_steps):
        problems.append("status max_steps inconsistent")
    return not problems, problems, excused
