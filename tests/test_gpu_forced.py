"""GPU parity of forced continuations (TC_FLAG_JUMP_FORWARD) against the oracle.

"Understanding Inference for Systems Engineers", section 7.5 (forced spans):
after each head decision the kernels emit, in the same step, every token the
grammar forces, without a head read; those logit slots hold NaN.  Bar: the
tokens, lengths and statuses equal the plain decode's and the oracle's
(``greedy_decode(jump=True)``), real logits as in the plain decode, NaN exactly
at the positions the oracle finds forced, fewer decode steps."""
import math

import numpy as np
import pytest

from gpu_common import DecodeBuffers, check_against_oracle, embedding, make_ctx, oracle_trie, torch_mod, workload
from oracle import decode as D

pytestmark = pytest.mark.gpu


def _run(tcd, name, hid, batch, head, residency=None, max_steps=None):
    w = workload(name)
    ctx, _ = make_ctx(tcd, name, max_batch=batch, residency=residency)
    ms = max_steps or w.max_steps
    buf = DecodeBuffers(w.max_steps, batch, w.hidden, ms)
    buf.load(hid)
    ctx.stats(reset=True)
    out = buf.run(ctx, w.k, head=head)
    st = ctx.stats(reset=True)
    ctx.close()
    return out, st


@pytest.mark.parametrize("head", ["sparse", "dense"])
@pytest.mark.parametrize("residency", ["const", "global"])
def test_tiny_jump_bitexact(tcd, head, residency):
    """Integer inputs: tokens and real logits bit-exact against the oracle's jump decode."""
    w = workload("tiny")
    hid = w.hidden_states(0, w.n_queries)
    h = tcd.HEAD_SPARSE if head == "sparse" else tcd.HEAD_DENSE
    (toks, logits, lens, status), st = _run(tcd, "tiny", hid, w.n_queries, h | tcd.FLAG_JUMP_FORWARD, residency)
    plain, _ = _run(tcd, "tiny", hid, w.n_queries, h, residency)
    trie = oracle_trie("tiny")
    emb_bits, _ = embedding(w.vocab, w.hidden, w.emb_kind)
    n_forced = 0
    for b in range(w.n_queries):
        want_t, want_l, want_s = D.greedy_decode(trie, w.k, emb_bits, hid[:, b], w.max_steps, jump=True)
        n = int(lens[b])
        assert want_s == "ok" and status[b] == 0 and n == len(want_t)
        assert toks[b, :n].tolist() == want_t and np.all(toks[b, n:] == -1)
        for t in range(n):
            if math.isnan(want_l[t]):
                assert np.isnan(logits[b, t])
                n_forced += 1
            else:
                assert float(logits[b, t]) == want_l[t]
        # same tokens and lengths as the plain decode; real logits equal
        assert np.array_equal(toks[b], plain[0][b]) and lens[b] == plain[2][b]
        real = ~np.isnan(logits[b, :n])
        assert np.array_equal(logits[b, :n][real], plain[1][b, :n][real])
    assert n_forced > 0
    assert st["forced"] == n_forced
    assert st["seq_steps"] == int(lens.sum()) - n_forced


def test_tiny_jump_batch1_equals_batched(tcd):
    """Sequences stay independent when their lengths diverge inside one step."""
    w = workload("tiny")
    hid = w.hidden_states(0, 16)
    flag = tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD
    full, _ = _run(tcd, "tiny", hid, 16, flag)
    for b in range(0, 16, 5):
        one, _ = _run(tcd, "tiny", hid[:, b:b + 1], 1, flag)
        for i in range(4):
            assert np.array_equal(one[i][0], full[i][b], equal_nan=True)


def test_large_head_jump_teacher_forced(tcd):
    """One-CTA step with precomputed lists (fan-out <= 32), Gaussian inputs, B=1."""
    w = workload("large_head")
    n = 64
    hid = w.hidden_states(0, n)
    ctx, _ = make_ctx(tcd, "large_head", max_batch=1)
    buf = DecodeBuffers(w.max_steps, 1, w.hidden, w.max_steps)
    forced = steps = 0
    for q in range(n):
        buf.load(hid[:, q:q + 1])
        ctx.stats(reset=True)
        out = buf.run(ctx, w.k, head=tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD)
        st = ctx.stats(reset=True)
        assert out[3][0] == 0
        check_against_oracle("large_head", hid[:, q:q + 1], out, w.k, w.max_steps, exact=False, jump=True)
        forced += st["forced"]
        steps += st["seq_steps"]
        assert st["forced"] == int(np.isnan(out[1][0, :out[2][0]]).sum())
    ctx.close()
    assert forced > 0.3 * (forced + steps)


def test_unstructured_jump_teacher_forced(tcd):
    """Multi-CTA sparse step (hex catalog, fan-out > 32): forced spans after the root."""
    w = workload("unstructured")
    hid = w.hidden_states(0, w.batch)
    (toks, logits, lens, status), st = _run(tcd, "unstructured", hid, w.batch,
                                             tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD)
    plain, _ = _run(tcd, "unstructured", hid, w.batch, tcd.HEAD_SPARSE)
    assert np.all(status == 0)
    check_against_oracle("unstructured", hid, (toks, logits, lens, status), w.k, w.max_steps, exact=False, jump=True)
    assert np.array_equal(toks, plain[0]) and np.array_equal(lens, plain[2])
    assert st["forced"] > 0.5 * int(lens.sum())


@pytest.mark.parametrize("name", ["char_tools", "char_hex"])
def test_char_jump_teacher_forced(tcd, name):
    """Multi-CTA grammars whose narrow nodes take the one-CTA step: forced spans
    that start at a narrow node and cross into a wide one (a node wider than a
    precomputed list is counted by the chain itself)."""
    w = workload(name)
    B = 16
    hid = w.hidden_states(0, B)
    out, st = _run(tcd, name, hid, B, tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD)
    plain, _ = _run(tcd, name, hid, B, tcd.HEAD_SPARSE)
    assert np.all(out[3] == 0)
    check_against_oracle(name, hid, out, w.k, w.max_steps, exact=False, jump=True)
    assert np.array_equal(out[0], plain[0]) and np.array_equal(out[2], plain[2])
    assert st["forced"] == int(sum(np.isnan(out[1][b, :out[2][b]]).sum() for b in range(B)))
    assert st["forced"] > 0


def test_batched_jump_teacher_forced(tcd):
    w = workload("batched")
    hid = w.hidden_states(0, w.batch)
    out, st = _run(tcd, "batched", hid, w.batch, tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD)
    assert np.all(out[3] == 0)
    check_against_oracle("batched", hid, out, w.k, w.max_steps, exact=False, jump=True)
    assert st["forced"] == int(sum(np.isnan(out[1][b, :out[2][b]]).sum() for b in range(w.batch)))


def test_jump_respects_the_step_budget(tcd):
    """A forced span stops at max_steps; the sequence then fails with MAX_STEPS
    exactly as the plain decode does."""
    w = workload("tiny")
    hid = w.hidden_states(0, 8)
    for ms in (2, 3, 5):
        out, _ = _run(tcd, "tiny", hid, 8, tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD, max_steps=ms)
        plain, _ = _run(tcd, "tiny", hid, 8, tcd.HEAD_SPARSE, max_steps=ms)
        assert np.array_equal(out[0], plain[0]) and np.array_equal(out[2], plain[2])
        assert np.array_equal(out[3], plain[3])
        check_against_oracle("tiny", hid, out, w.k, ms, exact=True, jump=True)


def test_jump_rejected_where_unsupported(tcd):
    torch = torch_mod()
    w = workload("tiny")
    ctx, _ = make_ctx(tcd, "tiny", max_batch=2)
    buf = DecodeBuffers(w.max_steps, 2, w.hidden, w.max_steps)
    buf.load(w.hidden_states(0, 2))
    with pytest.raises(tcd.TcError) as e:
        buf.run(ctx, w.k, head=tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD, mode="host")
    assert e.value.name == "TC_ERR_UNSUPPORTED"
    with pytest.raises(tcd.TcError) as e:
        buf.run(ctx, w.k, head=tcd.HEAD_UNION_GEMM | tcd.FLAG_JUMP_FORWARD)
    assert e.value.name == "TC_ERR_UNSUPPORTED"
    ctx.reset(2, w.k)
    tok = torch.empty(2, dtype=torch.int32, device="cuda")
    with pytest.raises(tcd.TcError) as e:
        ctx.step(buf.hid[0], tok, head=tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD)
    assert e.value.name == "TC_ERR_INVALID_ARG"
    ctx.close()


@pytest.mark.parametrize("name", ["tiny", "large_head", "unstructured", "char_tools"])
def test_forced_logits_equal_the_plain_decode(tcd, name):
    """With TC_FLAG_FORCED_LOGITS forced positions still take no head decision
    but carry their logit: tokens and logits equal the plain decode's bit for
    bit (one-CTA and multi-CTA steps)."""
    w = workload(name)
    B = 8 if w.batch <= 8 else w.batch
    hid = w.hidden_states(0, B)
    flags = tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD | tcd.FLAG_FORCED_LOGITS
    out, st = _run(tcd, name, hid, B, flags)
    plain, _ = _run(tcd, name, hid, B, tcd.HEAD_SPARSE)
    for a, b in zip(out, plain):
        assert np.array_equal(a, b)
    assert st["forced"] > 0 and not np.isnan(out[1]).any()


def test_forced_logits_needs_jump(tcd):
    w = workload("tiny")
    with pytest.raises(tcd.TcError) as e:
        _run(tcd, "tiny", w.hidden_states(0, 2), 2, tcd.HEAD_SPARSE | tcd.FLAG_FORCED_LOGITS)
    assert e.value.name == "TC_ERR_INVALID_ARG"
