"""The two no-repeat state modes give identical decodes (through the C ABI).

"Constraint made cheaper than no constraint", section "Masked sampling inside
the sampler" (per-sequence live counts, decremented along a completed
pointer's path) and section "The batched engine" (a 16-byte per-sequence
banned set against read-only per-edge pointer sets).  The library uses the
read-only state for k <= 8; TC_BIND_LIVE_COUNTS forces the count arrays.  Bar:
tokens, logits, lengths and statuses bit-identical between the modes for every
head, loop form and forced-continuation setting, and equal to the oracle."""
import numpy as np
import pytest

from gpu_common import DecodeBuffers, check_against_oracle, embedding, make_ctx, torch_mod, workload
from oracle import decode as D
from oracle import grammar as G

pytestmark = pytest.mark.gpu


def _ctx(tcd, name, batch, counts, residency=None):
    w = workload(name)
    _, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    ctx = tcd.Context(emb, max_batch=batch, cand_cap=w.cand_cap)
    trie = tcd.Trie.compile(w.catalog, w.sep_id, w.stop_id, w.vocab, w.max_fanout)
    res = {"const": tcd.RES_CONST, "global": tcd.RES_GLOBAL, "auto": tcd.RES_AUTO}[residency or w.residency]
    ctx.bind(trie, res | (tcd.BIND_LIVE_COUNTS if counts else 0))
    return ctx


def _both(tcd, name, hid, batch, head, mode="graph", residency=None, k=None, max_steps=None):
    w = workload(name)
    ms = max_steps or w.max_steps
    outs = []
    for counts in (False, True):
        ctx = _ctx(tcd, name, batch, counts, residency)
        buf = DecodeBuffers(hid.shape[0], batch, w.hidden, ms)
        buf.load(hid)
        outs.append(buf.run(ctx, k or w.k, head=head, mode=mode))
        ctx.close()
    for a, b in zip(*outs):
        assert np.array_equal(a, b, equal_nan=True)
    return outs[0]


@pytest.mark.parametrize("residency", ["const", "global"])
@pytest.mark.parametrize("head", ["sparse", "dense", "union", "dense_gemm"])
def test_tiny_modes_identical_every_head(tcd, head, residency):
    w = workload("tiny")
    hid = w.hidden_states(0, 16)
    h = {"sparse": tcd.HEAD_SPARSE, "dense": tcd.HEAD_DENSE, "union": tcd.HEAD_UNION_GEMM,
         "dense_gemm": tcd.HEAD_DENSE_GEMM}[head]
    out = _both(tcd, "tiny", hid, 16, h, residency=residency)
    assert np.all(out[3] == 0)
    check_against_oracle("tiny", hid, out, w.k, w.max_steps, exact=True)


def test_tiny_modes_identical_host_loop_and_jump(tcd):
    w = workload("tiny")
    hid = w.hidden_states(20, 16)
    _both(tcd, "tiny", hid, 16, tcd.HEAD_SPARSE, mode="host")
    out = _both(tcd, "tiny", hid, 16, tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD)
    check_against_oracle("tiny", hid, out, w.k, w.max_steps, exact=True, jump=True)


def test_unstructured_modes_identical(tcd):
    """Multi-CTA sparse step (fan-out > 32) in both modes."""
    w = workload("unstructured")
    hid = w.hidden_states(0, w.batch)
    out = _both(tcd, "unstructured", hid, w.batch, tcd.HEAD_SPARSE)
    check_against_oracle("unstructured", hid, out, w.k, w.max_steps, exact=False)


def test_tensor_batch_union_modes_identical(tcd):
    w = workload("tensor_batch")
    hid = w.hidden_states(0, w.batch)
    out = _both(tcd, "tensor_batch", hid, w.batch, tcd.HEAD_UNION_GEMM)
    check_against_oracle("tensor_batch", hid, out, w.k, w.max_steps, exact=False, seqs=range(0, w.batch, 17))


def test_large_k_uses_counts_and_matches_oracle(tcd):
    """k = 10 > 8 falls back to the count arrays; both bindings then run the
    same mode and the decode still equals the oracle's."""
    w = workload("tiny")
    k = 10
    steps = k * 9
    hid = w.hidden_states(0, 8, steps=steps)
    out = _both(tcd, "tiny", hid, 8, tcd.HEAD_SPARSE, k=k, max_steps=steps)
    assert np.all(out[3] == 0)
    trie = G.compile_catalog(w.catalog, w.sep_id, w.stop_id, w.vocab)
    emb_bits, _ = embedding(w.vocab, w.hidden, w.emb_kind)
    for b in range(8):
        want_t, want_l, st = D.greedy_decode(trie, k, emb_bits, hid[:, b], steps)
        n = int(out[2][b])
        assert st == "ok" and out[0][b, :n].tolist() == want_t
        assert [float(x) for x in out[1][b, :n]] == want_l


def test_eight_pointers_fill_the_banned_set(tcd):
    """k = 8: the banned set's last slot is written at the final stop."""
    w = workload("tiny")
    k = 8
    steps = k * 9
    hid = w.hidden_states(40, 8, steps=steps)
    out = _both(tcd, "tiny", hid, 8, tcd.HEAD_SPARSE, k=k, max_steps=steps)
    trie = G.compile_catalog(w.catalog, w.sep_id, w.stop_id, w.vocab)
    emb_bits, _ = embedding(w.vocab, w.hidden, w.emb_kind)
    for b in range(8):
        want_t, _, st = D.greedy_decode(trie, k, emb_bits, hid[:, b], steps)
        assert st == "ok" and out[0][b, :int(out[2][b])].tolist() == want_t
