"""Shared helpers of the GPU parity tests: workload fixtures and the oracle check.

Inputs come from trie_constrained_decoding_gb300.inputs (seeded); expected
values come only from the oracle."""
from __future__ import annotations

import functools

import numpy as np

from oracle import chars as C
from oracle import decode as D
from oracle import grammar as G
from trie_constrained_decoding_gb300 import inputs as I

STATUS_TO_ORACLE = {0: "ok", 16: "empty_mask", 18: "max_steps"}


def torch_mod():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch


def to_dev_bf16(bits: np.ndarray):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to("cuda").view(torch.bfloat16)


@functools.lru_cache(maxsize=None)
def workload(name: str):
    return I.WORKLOADS[name]()


@functools.lru_cache(maxsize=4)
def embedding(vocab: int, hidden: int, kind: str):
    """Host bits and device tensor of the tied embedding (shared by workloads of one shape)."""
    for name in I.WORKLOADS:
        w = workload(name)
        if (w.vocab, w.hidden, w.emb_kind) == (vocab, hidden, kind):
            bits = w.embedding()
            return bits, to_dev_bf16(bits)
    raise KeyError((vocab, hidden, kind))


@functools.lru_cache(maxsize=None)
def oracle_trie(name: str):
    """The oracle's grammar of a workload: the token trie, or the character-level grammar."""
    w = workload(name)
    if w.char_strings is not None:
        return C.CharGrammar(w.char_strings, w.char_vocab, w.sep_id, w.stop_id)
    return G.compile_catalog(w.catalog, w.sep_id, w.stop_id, w.vocab, max_fanout=w.max_fanout)


def compile_trie(tcd, w):
    if w.char_strings is not None:
        return tcd.Trie.compile_chars(w.char_strings, w.char_vocab, w.sep_id, w.stop_id, w.vocab, w.max_fanout)
    return tcd.Trie.compile(w.catalog, w.sep_id, w.stop_id, w.vocab, w.max_fanout)


def make_ctx(tcd, name: str, max_batch: int = None, residency=None):
    w = workload(name)
    _, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    ctx = tcd.Context(emb, max_batch=max_batch or w.batch, cand_cap=w.cand_cap)
    trie = compile_trie(tcd, w)
    res = {"const": tcd.RES_CONST, "global": tcd.RES_GLOBAL, "auto": tcd.RES_AUTO}[residency or w.residency]
    ctx.bind(trie, res)
    return ctx, trie


class DecodeBuffers:
    """Fixed device buffers for one (batch, max_steps) shape, so a captured graph replays."""

    def __init__(self, steps: int, batch: int, hidden: int, max_steps: int):
        torch = torch_mod()
        self.hid = torch.empty((steps, batch, hidden), dtype=torch.bfloat16, device="cuda")
        self.toks = torch.empty((batch, max_steps), dtype=torch.int32, device="cuda")
        self.logits = torch.empty((batch, max_steps), dtype=torch.float32, device="cuda")
        self.lens = torch.empty(batch, dtype=torch.int32, device="cuda")
        self.status = torch.empty(batch, dtype=torch.int32, device="cuda")
        self.max_steps = max_steps

    def load(self, hid_bits: np.ndarray):
        torch = torch_mod()
        self.hid.copy_(torch.from_numpy(np.ascontiguousarray(hid_bits).view(np.int16)).view(torch.bfloat16))

    def run(self, ctx, k: int, head: int = 0, mode: str = "graph"):
        torch = torch_mod()
        fn = ctx.decode if mode == "graph" else ctx.decode_host
        fn(self.hid, k, self.max_steps, self.toks, self.logits, self.lens, self.status, head=head)
        torch.cuda.synchronize()
        return (self.toks.cpu().numpy().copy(), self.logits.cpu().numpy().copy(),
                self.lens.cpu().numpy().copy(), self.status.cpu().numpy().copy())


def check_against_oracle(name: str, hid_bits: np.ndarray, out, k: int, max_steps: int, exact: bool,
                         seqs=None, jump: bool = False):
    """Teacher-force every sequence (or the listed ones); return the reports."""
    w = workload(name)
    trie = oracle_trie(name)
    emb_bits, _ = embedding(w.vocab, w.hidden, w.emb_kind)
    toks, logits, lens, status = out
    reports = []
    for b in (range(toks.shape[0]) if seqs is None else seqs):
        n = int(lens[b])
        assert np.all(toks[b, n:] == -1), f"seq {b}: tokens after the end"
        st = STATUS_TO_ORACLE.get(int(status[b]), f"code{int(status[b])}")
        rep = D.teacher_force(trie, k, emb_bits, hid_bits[:, b], list(map(int, toks[b, :n])),
                              list(map(float, logits[b, :n])), st, max_steps, exact=exact, jump=jump)
        assert rep.ok, f"seq {b}: {rep.problems[:3]}"
        reports.append(rep)
    return reports
