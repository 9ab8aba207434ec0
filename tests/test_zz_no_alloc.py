"""The allocation-free dense argmax (tc_dense_argmax_noalloc) against the dense
head of tc_step and against the oracle.

tc_dense_argmax_noalloc exists for callers that cannot allocate device memory:
code under a framework whose caching allocator owns the device budget, plugin
hosts that forbid allocation calls, and latency-critical paths where an
allocation or a free may synchronise the device.  Its scratch is one fixed
file-scope device array that every call shares.

Bar (its header's contract): tokens and logits equal tc_step's dense head bit
for bit (same lane map and shuffle tree); against the oracle, bit-exact on
integer-valued inputs, and on Gaussian inputs the chosen logit within 1e-3
relative with a differing token only below the oracle's 1e-5 top-2 margin.
An empty legal list gives -1 and 0.0; entries past n_legal are never read.

This file is collected last, so a run that stops at the first failure has
already run every other test; it passes alone in a fresh process and after
the other tests.
"""
import ctypes

import numpy as np
import pytest

from gpu_common import embedding, make_ctx, oracle_trie, to_dev_bf16, torch_mod, workload
from oracle import decode as D
from oracle import grammar as G
from oracle import head as OH

pytestmark = pytest.mark.gpu


def _noalloc_fn(tcd):
    f = tcd._lib.tc_dense_argmax_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p]
    return f


def _call(tcd, emb, x, legal_lists, stride=None, pad=None):
    """One call; list b is legal[b, :len] and the rest of its row is `pad[b]`
    (default -1), which the kernel must not read."""
    torch = torch_mod()
    B = len(legal_lists)
    stride = stride or max(1, max(len(l) for l in legal_lists))
    rows = np.full((B, stride), -1, dtype=np.int32)
    for b, l in enumerate(legal_lists):
        if pad is not None:
            rows[b, :] = pad[b]
        rows[b, :len(l)] = l
    legal = torch.from_numpy(rows).cuda()
    n = torch.tensor([len(l) for l in legal_lists], dtype=torch.int32).cuda()
    tok = torch.full((B,), 12345, dtype=torch.int32, device="cuda")
    lg = torch.full((B,), 7.0, dtype=torch.float32, device="cuda")
    V, H = emb.shape
    code = _noalloc_fn(tcd)(emb.data_ptr(), V, H, x.data_ptr(), B, legal.data_ptr(), stride, n.data_ptr(),
                            tok.data_ptr(), lg.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == 0, tcd.status_name(code)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), lg.cpu().numpy()


def _check_oracle(emb_bits, x_bits, legal_lists, got_t, got_l, exact):
    """Each sequence's result against the oracle's argmax over its legal list."""
    flips = 0
    for b, legal in enumerate(legal_lists):
        if len(legal) == 0:
            assert got_t[b] == -1 and got_l[b] == 0.0, (b, got_t[b], got_l[b])
            continue
        lg = OH.candidate_logits(emb_bits, x_bits[b], legal)
        best_t, best_l = OH.argmax_lower_id(legal, lg)
        assert int(got_t[b]) in legal, b
        r = float(lg[list(legal).index(int(got_t[b]))])
        if exact:
            assert int(got_t[b]) == best_t and float(got_l[b]) == r, (b, got_t[b], best_t, got_l[b], r)
            continue
        mass = OH.abs_mass(emb_bits, x_bits[b], [int(got_t[b]), best_t])
        scale = max(abs(r), D.FLOOR_SCALE * mass[0])
        assert abs(float(got_l[b]) - r) <= D.REL_TOL * scale, (b, got_l[b], r)
        if int(got_t[b]) != best_t:
            assert best_l - r <= D.MARGIN_TOL * max(abs(best_l), D.FLOOR_SCALE * mass[1]), b
            flips += 1
    return flips


@pytest.mark.parametrize("name", ["tiny", "large_head"])
def test_noalloc_matches_dense_head_on_two_calls(tcd, name):
    """Two calls in a row, each on the legal sets of a live decode: bitwise
    equal to tc_step's dense head, and within the oracle's bar."""
    torch = torch_mod()
    w = workload(name)
    emb_bits, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    B = 4
    ctx, _ = make_ctx(tcd, name, max_batch=B)
    ctx.reset(B, w.k)
    trie = oracle_trie(name)
    hid = w.hidden_states(0, B)
    states = [G.WalkState() for _ in range(B)]
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    lg = torch.empty(B, dtype=torch.float32, device="cuda")
    for step in range(2):
        x = to_dev_bf16(hid[step])
        ctx.step(x, tok, lg, head=tcd.HEAD_DENSE)
        torch.cuda.synchronize()
        want_t, want_l = tok.cpu().numpy(), lg.cpu().numpy()
        legal = [G.legal_tokens(trie, st, w.k) for st in states]
        got_t, got_l = _call(tcd, emb, x, legal)
        assert np.array_equal(got_t, want_t), (step, got_t, want_t)
        assert np.array_equal(got_l.view(np.uint32), want_l.view(np.uint32)), (step, got_l, want_l)
        assert _check_oracle(emb_bits, hid[step], legal, got_t, got_l, exact=w.emb_kind == "int") <= 1
        states = [G.advance(trie, st, int(t), w.k) for st, t in zip(states, want_t)]
    ctx.close()


def test_noalloc_empty_short_and_padded_lists(tcd):
    """Empty lists give -1 and 0.0; a list shorter than legal_stride is read
    only up to n_legal, even when the padding after it holds the row with the
    largest logit of the whole vocabulary."""
    w = workload("tiny")
    emb_bits, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    B = 8
    x_bits = w.hidden_states(0, B, steps=1)[0]
    rng = np.random.default_rng(7)
    full = OH.bf16_bits_to_f64(emb_bits) @ OH.bf16_bits_to_f64(x_bits).T      # [V, B]
    top = [int(np.argmax(full[:, b])) for b in range(B)]                       # lowest id among equal maxima
    lists = []
    for b in range(B):
        n = [0, 1, 2, 5, 0, 17, 40, 64][b]
        pool = np.setdiff1d(np.arange(w.vocab), [top[b]])
        lists.append(sorted(int(v) for v in rng.choice(pool, size=n, replace=False)))
    x = to_dev_bf16(x_bits)
    for _ in range(2):                               # the shared scratch keeps the last call's contents
        got_t, got_l = _call(tcd, emb, x, lists, stride=64, pad=top)
        _check_oracle(emb_bits, x_bits, lists, got_t, got_l, exact=True)
        for b in range(B):
            assert got_t[b] != top[b]


def test_noalloc_largest_batch(tcd):
    """At the largest batch (64 sequences, the fewest CTAs per sequence) with
    lists of every length up to the stride, on two calls with different hidden
    states: bit-exact against the oracle."""
    w = workload("tiny")
    emb_bits, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    B = 64
    rng = np.random.default_rng(11)
    hid = w.hidden_states(0, B, steps=2)
    for step in range(2):
        lists = [sorted(int(v) for v in rng.choice(w.vocab, size=int(rng.integers(0, 200)), replace=False))
                 for _ in range(B)]
        got_t, got_l = _call(tcd, emb, to_dev_bf16(hid[step]), lists, stride=200)
        _check_oracle(emb_bits, hid[step], lists, got_t, got_l, exact=True)


def test_noalloc_rejects_sizes_beyond_its_limits(tcd):
    torch = torch_mod()
    w = workload("tiny")
    _, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    f = _noalloc_fn(tcd)
    s = torch.cuda.current_stream().cuda_stream
    for B, H, stride in ((65, w.hidden, 1), (4, 8200, 1), (4, w.hidden, 4097)):
        x = torch.zeros((B, H), dtype=torch.bfloat16, device="cuda")
        legal = torch.zeros((B, stride), dtype=torch.int32, device="cuda")
        n = torch.ones(B, dtype=torch.int32, device="cuda")
        tok = torch.empty(B, dtype=torch.int32, device="cuda")
        lg = torch.empty(B, dtype=torch.float32, device="cuda")
        code = f(emb.data_ptr(), w.vocab, H, x.data_ptr(), B, legal.data_ptr(), stride, n.data_ptr(),
                 tok.data_ptr(), lg.data_ptr(), s)
        assert tcd.status_name(code) == "TC_ERR_CAPACITY", (B, H, stride)
