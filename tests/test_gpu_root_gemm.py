"""GPU parity of the tensor-core root step (TC_FLAG_ROOT_GEMM) against the oracle.

The first step of a decode, with every sequence at the root and nothing
emitted, runs as one tcgen05 GEMM over the root's token rows ("Constraint made
cheaper than no constraint", section "The sparse output layer"); the rest of
the decode is the sparse head.  Bar: tokens, lengths and statuses equal the
oracle's; logits bit-exact on integer-valued inputs (tensor-core fp32 sums of
those values are exact) and within the oracle's tolerance on Gaussian ones."""
import numpy as np
import pytest

from gpu_common import DecodeBuffers, check_against_oracle, make_ctx, to_dev_bf16, torch_mod, workload

pytestmark = pytest.mark.gpu


def _run(tcd, name, head, batch=None, mode="graph", start=0):
    w = workload(name)
    B = batch or w.batch
    ctx, _ = make_ctx(tcd, name, max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    hid = w.hidden_states(start, B)
    buf.load(hid)
    out = buf.run(ctx, w.k, head=head, mode=mode)
    ctx.close()
    return hid, out


def test_tiny_root_gemm_bitexact_and_equal_to_sparse(tcd):
    """Integer-valued inputs, hidden 256 (one K pass, the masked-argmax
    epilogue): the decode with the root step on the GEMM equals the sparse
    decode bit for bit, tokens and logits, and the oracle's."""
    w = workload("tiny")
    B = w.n_queries
    hid, root = _run(tcd, "tiny", tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM, batch=B)
    _, sparse = _run(tcd, "tiny", tcd.HEAD_SPARSE, batch=B)
    assert np.all(root[3] == 0)
    for x, y in zip(root, sparse):
        assert np.array_equal(x, y)
    check_against_oracle("tiny", hid, root, w.k, w.max_steps, exact=True)


def test_tiny_root_gemm_batch_of_one_and_host_loop(tcd):
    """Batch 1 (a single M row of the tile) and the host-driven loop give the
    graph loop's results."""
    w = workload("tiny")
    flag = tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM
    for q in range(8):
        hid, g = _run(tcd, "tiny", flag, batch=1, start=q)
        _, h = _run(tcd, "tiny", flag, batch=1, mode="host", start=q)
        for x, y in zip(g, h):
            assert np.array_equal(x, y)
        check_against_oracle("tiny", hid, g, w.k, w.max_steps, exact=True)


def test_tiny_root_gemm_two_m_tiles_bitexact(tcd):
    """200 sequences: two 128-sequence M tiles, the second ragged."""
    w = workload("tiny")
    hid, root = _run(tcd, "tiny", tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM, batch=200)
    _, sparse = _run(tcd, "tiny", tcd.HEAD_SPARSE, batch=200)
    for x, y in zip(root, sparse):
        assert np.array_equal(x, y)
    check_against_oracle("tiny", hid, root, w.k, w.max_steps, exact=True, seqs=range(0, 200, 7))


def test_char_tiny_root_gemm_bitexact(tcd):
    """A character-level grammar (several token edges may reach one node) on
    integer-valued inputs."""
    w = workload("char_tiny")
    B = 32
    hid, root = _run(tcd, "char_tiny", tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM, batch=B)
    _, sparse = _run(tcd, "char_tiny", tcd.HEAD_SPARSE, batch=B)
    for x, y in zip(root, sparse):
        assert np.array_equal(x, y)
    check_against_oracle("char_tiny", hid, root, w.k, w.max_steps, exact=True)


@pytest.mark.parametrize("batch", [16, 64, 256])
def test_hex_catalog_root_gemm(tcd, batch):
    """The unstructured hex catalog (root fan-out 267: three column tiles, the
    last ragged; hidden 4096: sixteen K splits summed in a fixed order) at
    B = 16, 64 and 256 (two M tiles), teacher-forced against the oracle."""
    w = workload("unstructured")
    hid, out = _run(tcd, "unstructured", tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM, batch=batch)
    assert np.all(out[3] == 0)
    seqs = range(batch) if batch <= 16 else range(0, batch, 8)
    check_against_oracle("unstructured", hid, out, w.k, w.max_steps, exact=False, seqs=seqs)


def test_large_head_root_gemm_teacher_forced(tcd):
    """Hidden 2048 (eight K splits), batch 1, Gaussian inputs: 64 queries."""
    w = workload("large_head")
    flag = tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM
    ctx, _ = make_ctx(tcd, "large_head", max_batch=1)
    buf = DecodeBuffers(w.max_steps, 1, w.hidden, w.max_steps)
    hid_all = w.hidden_states(0, 64)
    for q in range(64):
        buf.load(hid_all[:, q:q + 1])
        out = buf.run(ctx, w.k, head=flag)
        assert out[3][0] == 0
        check_against_oracle("large_head", hid_all[:, q:q + 1], out, w.k, w.max_steps, exact=False)
    ctx.close()


def test_root_gemm_rejections(tcd):
    """Forced continuations, sampling and other heads refuse the flag."""
    torch = torch_mod()
    w = workload("tiny")
    B = 4
    ctx, _ = make_ctx(tcd, "tiny", max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(w.hidden_states(0, B))
    for head in (tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM | tcd.FLAG_JUMP_FORWARD,
                 tcd.HEAD_DENSE | tcd.FLAG_ROOT_GEMM, tcd.HEAD_UNION_GEMM | tcd.FLAG_ROOT_GEMM):
        with pytest.raises(tcd.TcError) as ei:
            buf.run(ctx, w.k, head=head)
        assert ei.value.name == "TC_ERR_UNSUPPORTED"
    u = torch.full((B, w.max_steps), 0.5, dtype=torch.float32, device="cuda")
    with pytest.raises(tcd.TcError) as ei:
        ctx.decode_sample(buf.hid, w.k, w.max_steps, u, buf.toks, buf.logits, buf.lens, buf.status,
                          head=tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM)
    assert ei.value.name == "TC_ERR_UNSUPPORTED"
    # the context still decodes
    out = buf.run(ctx, w.k, head=tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM)
    assert np.all(out[3] == 0)
    ctx.close()


def test_tensor_batch_root_gemm_b256(tcd):
    """The 1000-tool catalog at B=256 (the bench's tensor_batch launch shape):
    every 8th sequence teacher-forced against the oracle, all finished."""
    w = workload("tensor_batch")
    hid, out = _run(tcd, "tensor_batch", tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM)
    assert np.all(out[3] == 0)
    check_against_oracle("tensor_batch", hid, out, w.k, w.max_steps, exact=False, seqs=range(0, w.batch, 8))


def test_host_steps_with_root_gemm_equal_decode(tcd):
    """tc_step with the flag on the first step after a reset, then sparse
    steps, gives the decode with the flag (integer inputs: and the all-sparse
    steps), bit for bit; the flag on a later step fails every live sequence
    with TC_ERR_BOUNDS (the device finds them away from a fresh root)."""
    torch = torch_mod()
    w = workload("tiny")
    B = 16
    hid_bits = w.hidden_states(0, B)
    S = hid_bits.shape[0]
    hid = to_dev_bf16(hid_bits)
    ctx, _ = make_ctx(tcd, "tiny", max_batch=B)
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    lg = torch.empty(B, dtype=torch.float32, device="cuda")
    st = torch.empty(B, dtype=torch.int32, device="cuda")

    def run(first_head):
        ctx.reset(B, w.k)
        toks, lgs = np.full((B, S), -1, np.int32), np.zeros((B, S), np.float32)
        for t in range(S):
            ctx.step(hid[t], tok, lg, st, head=first_head if t == 0 else tcd.HEAD_SPARSE)
            torch.cuda.synchronize()
            toks[:, t], lgs[:, t] = tok.cpu().numpy(), lg.cpu().numpy()
        return toks, lgs, st.cpu().numpy().copy()

    rt, rl, rs = run(tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM)
    pt, pl, ps = run(tcd.HEAD_SPARSE)
    assert np.array_equal(rt, pt) and np.array_equal(rl, pl) and np.array_equal(rs, ps)
    assert np.all(rs == 0)
    # the decode with the flag: the same tokens and logits
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(hid_bits)
    dt, dl, dn, ds = buf.run(ctx, w.k, head=tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM)
    for b in range(B):
        n = int(dn[b])
        assert np.array_equal(dt[b, :n], rt[b, :n]) and np.array_equal(dl[b, :n], rl[b, :n])
    # the flag on the second step: every sequence is away from a fresh root
    ctx.reset(B, w.k)
    ctx.step(hid[0], tok, lg, st, head=tcd.HEAD_SPARSE)
    ctx.step(hid[1], tok, lg, st, head=tcd.HEAD_SPARSE | tcd.FLAG_ROOT_GEMM)
    torch.cuda.synchronize()
    assert np.all(st.cpu().numpy() == tcd.TC_ERR_BOUNDS)
    assert np.all(tok.cpu().numpy() == -1)
    ctx.close()
