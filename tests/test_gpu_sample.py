"""GPU parity of sampling (tc_decode_sample / tc_step_sample) against the oracle,
on the one-CTA step (nodes of at most 32 edges) and the multi-CTA step.

"Understanding Inference for Systems Engineers", section 3.8: softmax of
logit / temperature over the legal candidates, restricted to the top-k highest
logits (a value threshold) and by top-p (an ascending prefix removed, highest
tied id survives); the uniforms are inputs.  Bar: every token legal and equal to
the oracle's exact draw, except where the oracle itself finds the draw within
rounding of a boundary (counted, and required rare); logits bit-exact on the
integer workload; on a grid of uniforms the tokens drawn match the oracle's
interval lengths."""
import numpy as np
import pytest

from gpu_common import embedding, make_ctx, oracle_trie, torch_mod, workload
from oracle import sample as S
from oracle import grammar as G
from oracle.head import candidate_logits

pytestmark = pytest.mark.gpu


class _Bufs:
    def __init__(self, S_, B, H, ms):
        torch = torch_mod()
        self.hid = torch.empty((S_, B, H), dtype=torch.bfloat16, device="cuda")
        self.u = torch.empty((B, ms), dtype=torch.float32, device="cuda")
        self.toks = torch.empty((B, ms), dtype=torch.int32, device="cuda")
        self.logits = torch.empty((B, ms), dtype=torch.float32, device="cuda")
        self.lens = torch.empty(B, dtype=torch.int32, device="cuda")
        self.status = torch.empty(B, dtype=torch.int32, device="cuda")
        self.ms = ms

    def run(self, ctx, hid, u, k, head=0, **sp):
        torch = torch_mod()
        self.hid.copy_(torch.from_numpy(np.ascontiguousarray(hid).view(np.int16)).view(torch.bfloat16))
        self.u.copy_(torch.from_numpy(np.ascontiguousarray(u)))
        ctx.decode_sample(self.hid, k, self.ms, self.u, self.toks, self.logits, self.lens, self.status, head=head, **sp)
        torch.cuda.synchronize()
        return (self.toks.cpu().numpy(), self.logits.cpu().numpy(), self.lens.cpu().numpy(),
                self.status.cpu().numpy())


def _check(name, hid, u, out, k, ms, T, top_k, top_p, jump=False, exact=False):
    w = workload(name)
    trie = oracle_trie(name)
    emb_bits, _ = embedding(w.vocab, w.hidden, w.emb_kind)
    toks, logits, lens, status = out
    steps = excused = 0
    for b in range(toks.shape[0]):
        n = int(lens[b])
        st = {0: "ok", 18: "max_steps", 16: "empty_mask"}.get(int(status[b]), "?")
        ok, problems, exc = S.sample_teacher_force(trie, k, emb_bits, hid[:, b], u[b], list(toks[b, :n]),
                                                   list(logits[b, :n]), st, ms, T, top_k, top_p, jump=jump,
                                                   exact_logits=exact)
        assert ok, (b, problems[:3])
        steps += n
        excused += exc
    assert excused <= max(1, steps // 200), (excused, steps)
    return steps, excused


@pytest.mark.parametrize("T,top_k,top_p", [(1.0, 0, 1.0), (0.7, 2, 1.0), (1.3, 0, 0.8), (0.5, 3, 0.6),
                                          (1.0, 1, 1.0)])
def test_tiny_sampling_matches_oracle(tcd, T, top_k, top_p):
    """Integer-valued inputs: exact fp32 logits, so ties at the top-k threshold are real."""
    w = workload("tiny")
    B = 64
    hid = w.hidden_states(0, B)
    u = w.uniforms(0, B)
    ctx, _ = make_ctx(tcd, "tiny", max_batch=B)
    out = _Bufs(w.max_steps, B, w.hidden, w.max_steps).run(ctx, hid, u, w.k, temperature=T, top_k=top_k,
                                                           top_p=top_p)
    ctx.close()
    assert np.all(out[3] == 0)
    _check("tiny", hid, u, out, w.k, w.max_steps, T, top_k, top_p, exact=True)


def test_large_head_sampling_matches_oracle(tcd):
    w = workload("large_head")
    B = 16
    hid = w.hidden_states(0, B)
    u = w.uniforms(0, B)
    ctx, _ = make_ctx(tcd, "large_head", max_batch=B)
    out = _Bufs(w.max_steps, B, w.hidden, w.max_steps).run(ctx, hid, u, w.k, temperature=1.0, top_k=0,
                                                           top_p=0.95)
    ctx.close()
    _check("large_head", hid, u, out, w.k, w.max_steps, 1.0, 0, 0.95)


def test_batched_sampling_with_forced_continuations(tcd):
    w = workload("batched")
    B = w.batch
    hid = w.hidden_states(0, B)
    u = w.uniforms(0, B)
    ctx, _ = make_ctx(tcd, "batched", max_batch=B)
    out = _Bufs(w.max_steps, B, w.hidden, w.max_steps).run(ctx, hid, u, w.k, head=tcd.FLAG_JUMP_FORWARD,
                                                           temperature=0.9, top_k=4, top_p=0.9)
    ctx.close()
    _check("batched", hid, u, out, w.k, w.max_steps, 0.9, 4, 0.9, jump=True)


def test_grid_of_uniforms_draws_in_proportion(tcd):
    """4096 sequences with the same hidden state and uniforms (i + 1/2) / 4096:
    the first tokens drawn follow the oracle's interval lengths."""
    w = workload("tiny")
    N = 4096
    one = w.hidden_states(5, 1)
    hid = np.repeat(one, N, axis=1)
    u = np.zeros((N, w.max_steps), dtype=np.float32)
    u[:, 0] = (np.arange(N, dtype=np.float64) + 0.5) / N
    u[:, 1:] = 0.5
    ctx, _ = make_ctx(tcd, "tiny", max_batch=N)
    T, top_k, top_p = 2.0, 0, 0.93
    out = _Bufs(w.max_steps, N, w.hidden, w.max_steps).run(ctx, hid, u, w.k, temperature=T, top_k=top_k,
                                                           top_p=top_p)
    ctx.close()
    trie = oracle_trie("tiny")
    emb_bits, _ = embedding(w.vocab, w.hidden, w.emb_kind)
    legal = G.legal_tokens(trie, G.WalkState(), w.k)
    lg = list(candidate_logits(emb_bits, one[0, 0], legal))
    iv = S.token_intervals(legal, lg, T, top_k, top_p)
    first = out[0][:, 0]
    assert set(np.unique(first).tolist()) <= set(iv)
    assert len(iv) >= 4
    for t, (lo, hi) in iv.items():
        assert abs(int((first == t).sum()) - N * (hi - lo)) <= 2.0


def test_draws_depend_only_on_the_sequence(tcd):
    w = workload("tiny")
    B = 16
    hid = w.hidden_states(30, B)
    u = w.uniforms(30, B)
    ctx, _ = make_ctx(tcd, "tiny", max_batch=B)
    full = _Bufs(w.max_steps, B, w.hidden, w.max_steps).run(ctx, hid, u, w.k, temperature=1.1, top_p=0.9)
    for b in (0, 7, 15):
        one = _Bufs(w.max_steps, 1, w.hidden, w.max_steps).run(ctx, hid[:, b:b + 1], u[b:b + 1], w.k,
                                                               temperature=1.1, top_p=0.9)
        for i in range(4):
            assert np.array_equal(one[i][0], full[i][b])
    ctx.close()


def test_step_sample_equals_decode_sample(tcd):
    torch = torch_mod()
    w = workload("tiny")
    B = 8
    hid = w.hidden_states(50, B)
    u = w.uniforms(50, B)
    ctx, _ = make_ctx(tcd, "tiny", max_batch=B)
    full = _Bufs(w.max_steps, B, w.hidden, w.max_steps).run(ctx, hid, u, w.k, temperature=0.8, top_k=3)
    ctx.reset(B, w.k)
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    lg = torch.empty(B, dtype=torch.float32, device="cuda")
    for t in range(w.max_steps):
        x = torch.from_numpy(np.ascontiguousarray(hid[t]).view(np.int16)).view(torch.bfloat16).cuda()
        ut = torch.from_numpy(np.ascontiguousarray(u[:, t])).cuda()
        ctx.step_sample(x, ut, tok, lg, temperature=0.8, top_k=3)
        tt = tok.cpu().numpy()
        live = tt >= 0
        assert np.array_equal(tt[live], full[0][live, t])
        assert np.array_equal(lg.cpu().numpy()[live], full[1][live, t])
    ctx.close()


def test_sampling_rejected_where_unsupported(tcd):
    w = workload("tiny")
    ctx, _ = make_ctx(tcd, "tiny", max_batch=2)
    bufs = _Bufs(w.max_steps, 2, w.hidden, w.max_steps)
    hid, u = w.hidden_states(0, 2), w.uniforms(0, 2)
    for kw, name in (({"head": tcd.HEAD_DENSE}, "TC_ERR_UNSUPPORTED"),
                     ({"temperature": 0.0}, "TC_ERR_INVALID_ARG"),
                     ({"top_p": 1.5}, "TC_ERR_INVALID_ARG"),
                     ({"top_k": -1}, "TC_ERR_INVALID_ARG")):
        with pytest.raises(tcd.TcError) as e:
            bufs.run(ctx, hid, u, w.k, **kw)
        assert e.value.name == name
    ctx.close()


@pytest.mark.parametrize("name,T,top_k,top_p", [("unstructured", 1.0, 0, 0.9), ("unstructured", 0.7, 20, 1.0),
                                                ("char_tools", 1.0, 0, 0.8), ("char_hex", 1.2, 50, 0.95)])
def test_multi_cta_sampling_matches_oracle(tcd, name, T, top_k, top_p):
    """Grammars with nodes of more than 32 edges: the multi-CTA step leaves every
    candidate's logit to the sequence's last CTA, which sorts and draws."""
    w = workload(name)
    B = 8
    hid = w.hidden_states(0, B)
    u = w.uniforms(0, B)
    ctx, _ = make_ctx(tcd, name, max_batch=B)
    out = _Bufs(w.max_steps, B, w.hidden, w.max_steps).run(ctx, hid, u, w.k, temperature=T, top_k=top_k,
                                                           top_p=top_p)
    ctx.close()
    assert np.all(out[3] == 0)
    _check(name, hid, u, out, w.k, w.max_steps, T, top_k, top_p)


def test_multi_cta_grid_of_uniforms(tcd):
    """The hex catalog's root (267 candidates), 2048 sequences with one hidden
    state and uniforms (i + 1/2) / 2048: the first tokens follow the oracle's
    interval lengths."""
    w = workload("unstructured")
    N = 2048
    one = w.hidden_states(3, 1)
    hid = np.repeat(one, N, axis=1)
    u = np.zeros((N, w.max_steps), dtype=np.float32)
    u[:, 0] = (np.arange(N, dtype=np.float64) + 0.5) / N
    u[:, 1:] = 0.5
    ctx, _ = make_ctx(tcd, "unstructured", max_batch=N)
    T, top_k, top_p = 0.5, 0, 0.9
    out = _Bufs(w.max_steps, N, w.hidden, w.max_steps).run(ctx, hid, u, w.k, temperature=T, top_k=top_k,
                                                           top_p=top_p)
    ctx.close()
    trie = oracle_trie("unstructured")
    emb_bits, _ = embedding(w.vocab, w.hidden, w.emb_kind)
    legal = G.legal_tokens(trie, G.WalkState(), w.k)
    lg = list(candidate_logits(emb_bits, one[0, 0], legal))
    iv = S.token_intervals(legal, lg, T, top_k, top_p)
    first = out[0][:, 0]
    assert set(np.unique(first).tolist()) <= set(iv)
    assert len(iv) >= 4
    for t, (lo, hi) in iv.items():
        assert abs(int((first == t).sum()) - N * (hi - lo)) <= 2.0
