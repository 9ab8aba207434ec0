"""Constant-memory re-binding and loud failures on the GPU (through the C ABI).

"Constraint made cheaper than no constraint", section "The grammar as a trie
over tokens": a one-pointer canary grammar once overwrote the product trie in
constant memory; residency is now owned by one grammar, re-bound on every
switch, and a captured graph re-binds at launch.  Section "Masked sampling
inside the sampler": a sequence that cannot continue sets an error and stops.
No test here faults the GPU: every failure is made by data or by arguments."""
import numpy as np
import pytest

from gpu_common import DecodeBuffers, check_against_oracle, embedding, make_ctx, torch_mod, workload
from oracle import decode as D
from oracle import grammar as G

pytestmark = pytest.mark.gpu

CANARY = [(11, 12, 13)]


def _oracle_single(name_or_trie, emb_bits, hid_bits, k, max_steps):
    return D.greedy_decode(name_or_trie, k, emb_bits, hid_bits, max_steps)


def test_graph_rebinds_constant_image_after_canary(tcd):
    torch = torch_mod()
    w = workload("tiny")
    emb_bits, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    ctx = tcd.Context(emb, max_batch=1)
    trie_a = tcd.Trie.compile(w.catalog, w.sep_id, w.stop_id, w.vocab)
    trie_b = tcd.Trie.compile(CANARY, w.sep_id, w.stop_id, w.vocab)
    ctx.bind(trie_a, tcd.RES_CONST)
    buf = DecodeBuffers(w.max_steps, 1, w.hidden, w.max_steps)
    hid = w.hidden_states(0, 1)
    buf.load(hid)
    graph_a = ctx.decode_graph(buf.hid, w.k, w.max_steps, buf.toks, buf.logits, buf.lens, buf.status)
    ctx.bind(trie_b, tcd.RES_CONST)            # the canary now holds the constant bank
    graph_a.launch()
    torch.cuda.synchronize()
    out = (buf.toks.cpu().numpy(), buf.logits.cpu().numpy(), buf.lens.cpu().numpy(), buf.status.cpu().numpy())
    assert out[3][0] == 0
    check_against_oracle("tiny", hid, out, w.k, w.max_steps, exact=True)
    # host-driven steps with the canary bound must walk the canary, not the graph's grammar
    ctx.reset(1, 1)
    tok = torch.empty(1, dtype=torch.int32, device="cuda")
    logit = torch.empty(1, dtype=torch.float32, device="cuda")
    got = []
    for t in range(5):
        x = torch.from_numpy(hid[t].view(np.int16)).view(torch.bfloat16).cuda()
        ctx.step(x, tok, logit)
        got.append(int(tok.item()))
    canary = G.compile_catalog(CANARY, w.sep_id, w.stop_id, w.vocab)
    want, _, st = D.greedy_decode(canary, 1, emb_bits, hid[:, 0], 4)
    assert st == "ok" and got == want + [-1]
    graph_a.close()
    ctx.close()


def test_two_contexts_share_the_constant_bank(tcd):
    """Each context re-binds its own grammar before a host-driven step."""
    torch = torch_mod()
    w = workload("tiny")
    emb_bits, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    c1, c2 = tcd.Context(emb, max_batch=1), tcd.Context(emb, max_batch=1)
    ta = tcd.Trie.compile(w.catalog, w.sep_id, w.stop_id, w.vocab)
    tb = tcd.Trie.compile(CANARY, w.sep_id, w.stop_id, w.vocab)
    c1.bind(ta, tcd.RES_CONST)
    c2.bind(tb, tcd.RES_CONST)
    hid = w.hidden_states(3, 1)
    c1.reset(1, w.k)
    tok = torch.empty(1, dtype=torch.int32, device="cuda")
    got = []
    for t in range(w.max_steps):
        x = torch.from_numpy(hid[t].view(np.int16)).view(torch.bfloat16).cuda()
        c1.step(x, tok)
        got.append(int(tok.item()))
    want, _, st = D.greedy_decode(G.compile_catalog(w.catalog, w.sep_id, w.stop_id, w.vocab), w.k, emb_bits,
                                  hid[:, 0], w.max_steps)
    assert got[:len(want)] == want and all(t == -1 for t in got[len(want):])
    c1.close()
    c2.close()


def test_step_api_matches_decode(tcd):
    """tc_step driven from Python equals tc_decode, token for token."""
    torch = torch_mod()
    w = workload("batched")
    ctx, _ = make_ctx(tcd, "batched", max_batch=8)
    hid = w.hidden_states(100, 8)
    buf = DecodeBuffers(w.max_steps, 8, w.hidden, w.max_steps)
    buf.load(hid)
    toks, logits, lens, status = buf.run(ctx, w.k)
    ctx.reset(8, w.k)
    tok = torch.empty(8, dtype=torch.int32, device="cuda")
    lg = torch.empty(8, dtype=torch.float32, device="cuda")
    st = torch.empty(8, dtype=torch.int32, device="cuda")
    for t in range(w.max_steps):
        ctx.step(buf.hid[t], tok, lg, st)
        tt, ll = tok.cpu().numpy(), lg.cpu().numpy()
        assert np.array_equal(tt, toks[:, t])
        assert np.array_equal(ll[tt >= 0], logits[tt >= 0, t])
    state = ctx.seq_state(8)
    assert np.array_equal(state["len"], lens) and np.all(state["done"] == 1)
    assert np.all(state["emitted"] == w.k)
    ctx.close()


def test_max_steps_budget(tcd):
    w = workload("tiny")
    ctx, _ = make_ctx(tcd, "tiny", max_batch=4)
    hid = w.hidden_states(0, 4)
    for mode in ("graph", "host"):
        buf = DecodeBuffers(w.max_steps, 4, w.hidden, 3)
        buf.load(hid)
        out = buf.run(ctx, w.k, mode=mode)
        assert np.all(out[3] == tcd.TC_ERR_MAX_STEPS) and np.all(out[2] == 3)
        check_against_oracle("tiny", hid, out, w.k, 3, exact=True)
        assert ctx.first_error() == (0, tcd.TC_ERR_MAX_STEPS)
    ctx.close()


def test_nan_hidden_fails_loudly_for_that_sequence_only(tcd):
    """A hidden state of NaNs leaves no comparable logit: that sequence stops
    with TC_ERR_BOUNDS at that step; its batch-mates are unaffected."""
    w = workload("tiny")
    ctx, _ = make_ctx(tcd, "tiny", max_batch=4)
    hid = w.hidden_states(0, 4).copy()
    hid[1, 2, :] = 0x7FC0          # bf16 quiet NaN, sequence 2, step 1
    buf = DecodeBuffers(w.max_steps, 4, w.hidden, w.max_steps)
    buf.load(hid)
    out = buf.run(ctx, w.k)
    assert out[3][2] == tcd.TC_ERR_BOUNDS and out[2][2] == 1
    assert ctx.first_error() == (2, tcd.TC_ERR_BOUNDS)
    check_against_oracle("tiny", hid, out, w.k, w.max_steps, exact=True, seqs=[0, 1, 3])
    with pytest.raises(tcd.TcError):
        ctx.raise_on_error()
    ctx.close()


def test_argument_errors(tcd):
    torch = torch_mod()
    w = workload("tiny")
    _, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    ctx = tcd.Context(emb, max_batch=2)
    tok = torch.empty(2, dtype=torch.int32, device="cuda")
    x = torch.zeros((2, w.hidden), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tcd.TcError) as e:
        ctx.step(x, tok)
    assert e.value.name == "TC_ERR_NOT_BOUND"
    trie = tcd.Trie.compile(w.catalog, w.sep_id, w.stop_id, w.vocab)
    ctx.bind(trie)
    assert ctx.residency() == tcd.RES_CONST
    with pytest.raises(tcd.TcError) as e:
        ctx.step(x, tok)                       # bound, but no reset yet
    assert e.value.name == "TC_ERR_NOT_BOUND"
    with pytest.raises(tcd.TcError) as e:
        ctx.reset(2, len(w.catalog) + 1)
    assert e.value.name == "TC_ERR_K_RANGE"
    with pytest.raises(tcd.TcError) as e:
        ctx.reset(2, 0)
    assert e.value.name == "TC_ERR_K_RANGE"
    with pytest.raises(tcd.TcError) as e:
        ctx.reset(3, 1)
    assert e.value.name == "TC_ERR_CAPACITY"
    buf = DecodeBuffers(4, 2, w.hidden, 5)
    with pytest.raises(tcd.TcError) as e:        # max_steps > hidden rows
        buf.run(ctx, 1)
    assert e.value.name == "TC_ERR_INVALID_ARG"
    ctx.close()


def test_residency_selection_and_capacity(tcd):
    b = workload("batched")
    _, emb = embedding(b.vocab, b.hidden, b.emb_kind)
    ctx = tcd.Context(emb, max_batch=1, cand_cap=4096)
    big = tcd.Trie.compile(b.catalog, b.sep_id, b.stop_id, b.vocab)
    ctx.bind(big, tcd.RES_AUTO)                 # 1000-tool headers fit the constant bank
    assert ctx.residency() == tcd.RES_CONST
    u = workload("unstructured")
    hexes = tcd.Trie.compile(u.catalog, u.sep_id, u.stop_id, u.vocab, 4096)
    with pytest.raises(tcd.TcError) as e:       # ~16k nodes: headers above the constant capacity
        ctx.bind(hexes, tcd.RES_CONST)
    assert e.value.name == "TC_ERR_CONST_CAPACITY"
    ctx.bind(hexes, tcd.RES_AUTO)
    assert ctx.residency() == tcd.RES_GLOBAL
    ctx.close()
    small = tcd.Context(emb, max_batch=1, cand_cap=256)
    with pytest.raises(tcd.TcError) as e:       # root fan-out above the 256-slot candidate buffer
        small.bind(hexes)
    assert e.value.name == "TC_ERR_CAPACITY"
    small.close()
