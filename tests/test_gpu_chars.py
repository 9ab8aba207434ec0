"""GPU parity of character-level grammars (tc_compile_char_trie) against the oracle.

The pith.science review of arXiv 2608.12574 (key machinery): every tokenization
of a catalog string is legal.  The decode kernels walk the compiled token-level
CSR unchanged (several edges may lead to one node; the no-repeat state is the
read-only rank-range one).  Bar: bit-exact tokens and logits on the integer
workload, teacher forcing on the Gaussian ones, through every head path the
grammars reach (one-CTA sparse step for fan-out <= 32, multi-CTA above)."""
import numpy as np
import pytest

from gpu_common import (DecodeBuffers, check_against_oracle, compile_trie, embedding, make_ctx, oracle_trie,
                        torch_mod, workload)
from oracle import decode as D
from oracle import sample as S

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("head", ["sparse", "dense"])
def test_char_tiny_bitexact(tcd, head):
    w = workload("char_tiny")
    B = 64
    hid = w.hidden_states(0, B)
    ctx, _ = make_ctx(tcd, "char_tiny", max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(hid)
    out = buf.run(ctx, w.k, head=tcd.HEAD_SPARSE if head == "sparse" else tcd.HEAD_DENSE)
    ctx.close()
    assert np.all(out[3] == 0)
    check_against_oracle("char_tiny", hid, out, w.k, w.max_steps, exact=True)
    g = oracle_trie("char_tiny")
    multi = 0
    for b in range(B):
        toks = list(out[0][b, :out[2][b]])
        ptrs = g.parse_pointers(toks)
        assert len(set(ptrs)) == w.k and min(ptrs) >= 0
        canon = [tuple(w.catalog[i]) for i in ptrs]
        pieces, cur = [], []
        for t in toks:
            if t in (w.sep_id, w.stop_id):
                pieces.append(tuple(cur))
                cur = []
            else:
                cur.append(int(t))
        multi += sum(1 for p, c in zip(pieces, canon) if p != c)
    assert multi > 0        # the decoder used tokenizations other than the canonical one


def test_char_tiny_jump_and_sampling(tcd):
    torch = torch_mod()
    w = workload("char_tiny")
    B = 32
    hid = w.hidden_states(10, B)
    u = w.uniforms(10, B)
    ctx, _ = make_ctx(tcd, "char_tiny", max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(hid)
    out = buf.run(ctx, w.k, head=tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD)
    check_against_oracle("char_tiny", hid, out, w.k, w.max_steps, exact=True, jump=True)
    ud = torch.from_numpy(u).cuda()
    ctx.decode_sample(buf.hid, w.k, w.max_steps, ud, buf.toks, buf.logits, buf.lens, buf.status, temperature=2.0,
                      top_p=0.9)
    torch.cuda.synchronize()
    toks, logits, lens, status = (buf.toks.cpu().numpy(), buf.logits.cpu().numpy(), buf.lens.cpu().numpy(),
                                  buf.status.cpu().numpy())
    g = oracle_trie("char_tiny")
    emb_bits, _ = embedding(w.vocab, w.hidden, w.emb_kind)
    for b in range(B):
        n = int(lens[b])
        ok, probs, exc = S.sample_teacher_force(g, w.k, emb_bits, hid[:, b], u[b], list(toks[b, :n]),
                                                list(logits[b, :n]), "ok" if status[b] == 0 else "?", w.max_steps,
                                                2.0, 0, 0.9, exact_logits=True)
        assert ok, probs[:3]
    ctx.close()


def test_char_tools_multi_cta(tcd):
    """Fan-out 42: the multi-CTA sparse step; Gaussian inputs."""
    w = workload("char_tools")
    B = 16
    hid = w.hidden_states(0, B)
    ctx, _ = make_ctx(tcd, "char_tools", max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(hid)
    out = buf.run(ctx, w.k)
    assert np.all(out[3] == 0)
    check_against_oracle("char_tools", hid, out, w.k, w.max_steps, exact=False)
    jout = buf.run(ctx, w.k, head=tcd.HEAD_SPARSE | tcd.FLAG_JUMP_FORWARD)
    assert np.array_equal(jout[0], out[0])
    check_against_oracle("char_tools", hid, jout, w.k, w.max_steps, exact=False, jump=True)
    ctx.close()


def test_char_hex(tcd):
    """The unstructured falsifier at character level: root fan-out 270."""
    w = workload("char_hex")
    B = w.batch
    hid = w.hidden_states(0, B)
    ctx, _ = make_ctx(tcd, "char_hex", max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(hid)
    out = buf.run(ctx, w.k)
    assert np.all(out[3] == 0)
    check_against_oracle("char_hex", hid, out, w.k, w.max_steps, exact=False)
    ctx.close()


def test_char_grammar_refusals(tcd):
    w = workload("char_tiny")
    _, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    ctx = tcd.Context(emb, max_batch=2, cand_cap=w.cand_cap)
    trie = compile_trie(tcd, w)
    with pytest.raises(tcd.TcError) as e:
        ctx.bind(trie, tcd.RES_AUTO | tcd.BIND_LIVE_COUNTS)
    assert e.value.name == "TC_ERR_UNSUPPORTED"
    ctx.bind(trie)
    with pytest.raises(tcd.TcError) as e:       # k = 9 would need live-count arrays
        ctx.reset(2, 9)
    assert e.value.name == "TC_ERR_UNSUPPORTED"
    ctx.close()


@pytest.mark.parametrize("head", ["union", "dense_gemm"])
def test_char_tiny_gemm_heads_bitexact(tcd, head):
    """The GEMM heads walk the same compiled CSR: bit-exact on integer inputs."""
    w = workload("char_tiny")
    B = 32
    hid = w.hidden_states(100, B)
    ctx, _ = make_ctx(tcd, "char_tiny", max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(hid)
    h = tcd.HEAD_UNION_GEMM if head == "union" else tcd.HEAD_DENSE_GEMM
    out = buf.run(ctx, w.k, head=h)
    sparse = buf.run(ctx, w.k)
    ctx.close()
    assert np.all(out[3] == 0)
    check_against_oracle("char_tiny", hid, out, w.k, w.max_steps, exact=True)
    for a, b in zip(out, sparse):
        assert np.array_equal(a, b)
