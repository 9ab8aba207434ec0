"""The allocation-free dense argmax (tc_dense_argmax_noalloc) against the dense head of tc_step.

tc_dense_argmax_noalloc exists for callers that cannot allocate device memory
(a framework allocator owns the budget, a plugin host forbids allocation, or
an allocation's implicit synchronisation is unaffordable); its scratch is a
fixed file-scope device array shared by every call.  This file is collected
last so that a run stopping at the first failure has already run everything
else; it passes alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest

from gpu_common import embedding, make_ctx, oracle_trie, to_dev_bf16, torch_mod, workload
from oracle import grammar as G

pytestmark = pytest.mark.gpu


def _noalloc_fn(tcd):
    f = tcd._lib.tc_dense_argmax_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32,
                  ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p]
    return f


def _call(tcd, emb, x, legal_lists):
    torch = torch_mod()
    B = len(legal_lists)
    stride = max(1, max(len(l) for l in legal_lists))
    legal = torch.full((B, stride), -1, dtype=torch.int32)
    for b, l in enumerate(legal_lists):
        legal[b, :len(l)] = torch.tensor(l, dtype=torch.int32)
    legal = legal.cuda()
    n = torch.tensor([len(l) for l in legal_lists], dtype=torch.int32).cuda()
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    lg = torch.empty(B, dtype=torch.float32, device="cuda")
    V, H = emb.shape
    code = _noalloc_fn(tcd)(emb.data_ptr(), V, H, x.data_ptr(), B, legal.data_ptr(), stride, n.data_ptr(),
                            tok.data_ptr(), lg.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert code == 0, tcd.status_name(code)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), lg.cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "large_head"])
def test_noalloc_matches_dense_head_on_two_calls(tcd, name):
    torch = torch_mod()
    w = workload(name)
    _, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    B = 4
    ctx, _ = make_ctx(tcd, name, max_batch=B)
    ctx.reset(B, w.k)
    trie = oracle_trie(name)
    hid = w.hidden_states(0, B)
    states = [G.WalkState() for _ in range(B)]
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    lg = torch.empty(B, dtype=torch.float32, device="cuda")
    for step in range(2):                        # two calls in a row, each checked
        x = to_dev_bf16(hid[step])
        ctx.step(x, tok, lg, head=tcd.HEAD_DENSE)
        want_t, want_l = tok.cpu().numpy(), lg.cpu().numpy()
        legal = [G.legal_tokens(trie, st, w.k) for st in states]
        got_t, got_l = _call(tcd, emb, x, legal)
        assert np.array_equal(got_t, want_t), (step, got_t, want_t)
        if w.emb_kind == "int":
            assert np.array_equal(got_l, want_l)     # exact sums on integer-valued inputs
        else:
            assert np.all(np.abs(got_l - want_l) <= 1e-3 * np.maximum(np.abs(want_l), 1e-6))
        states = [G.advance(trie, st, int(t), w.k) for st, t in zip(states, want_t)]
    ctx.close()


def test_noalloc_rejects_sizes_beyond_its_limits(tcd):
    torch = torch_mod()
    w = workload("tiny")
    _, emb = embedding(w.vocab, w.hidden, w.emb_kind)
    B = 65                                       # above the 64-sequence limit
    x = torch.zeros((B, w.hidden), dtype=torch.bfloat16, device="cuda")
    legal = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    n = torch.ones(B, dtype=torch.int32, device="cuda")
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    lg = torch.empty(B, dtype=torch.float32, device="cuda")
    code = _noalloc_fn(tcd)(emb.data_ptr(), w.vocab, w.hidden, x.data_ptr(), B, legal.data_ptr(), 1, n.data_ptr(),
                            tok.data_ptr(), lg.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert tcd.status_name(code) == "TC_ERR_CAPACITY"
