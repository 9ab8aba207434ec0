"""GPU parity of the constrained decode step against the oracle (through the C ABI).

Bar: tokens, lengths and statuses always equal the oracle's; logits bit-exact
on integer-valued inputs (where the fp32 sum is exact); on Gaussian inputs
chosen logits within 1e-3 relative and a differing token only where the
oracle's own top-2 margin is below 1e-5 relative (teacher forcing,
"Understanding Inference for Systems Engineers", section 8.2)."""
import numpy as np
import pytest

from gpu_common import (DecodeBuffers, check_against_oracle, embedding, make_ctx, to_dev_bf16, torch_mod,
                        workload)
from oracle import decode as D

pytestmark = pytest.mark.gpu


def _decode_queries_b1(tcd, name, n_queries, head=0, mode="graph", residency=None):
    """Decode queries one at a time at batch 1 (the workload's launch shape)."""
    w = workload(name)
    ctx, trie = make_ctx(tcd, name, max_batch=1, residency=residency)
    hid_all = w.hidden_states(0, n_queries)
    buf = DecodeBuffers(w.max_steps, 1, w.hidden, w.max_steps)
    outs = []
    for q in range(n_queries):
        buf.load(hid_all[:, q:q + 1])
        outs.append(buf.run(ctx, w.k, head=head, mode=mode))
    ctx.close()
    return hid_all, outs


def test_tiny_sparse_graph_bitexact(tcd):
    w = workload("tiny")
    hid, outs = _decode_queries_b1(tcd, "tiny", w.n_queries)
    for q, out in enumerate(outs):
        assert out[3][0] == 0
        check_against_oracle("tiny", hid[:, q:q + 1], out, w.k, w.max_steps, exact=True)


def test_tiny_dense_equals_sparse_bitwise(tcd):
    w = workload("tiny")
    _, sp = _decode_queries_b1(tcd, "tiny", 16, head=tcd.HEAD_SPARSE)
    _, de = _decode_queries_b1(tcd, "tiny", 16, head=tcd.HEAD_DENSE)
    for a, b in zip(sp, de):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_tiny_host_loop_equals_graph_loop(tcd):
    _, g = _decode_queries_b1(tcd, "tiny", 16, mode="graph")
    _, h = _decode_queries_b1(tcd, "tiny", 16, mode="host")
    for a, b in zip(g, h):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_tiny_global_residency_equals_const(tcd):
    _, c = _decode_queries_b1(tcd, "tiny", 16, residency="const")
    _, g = _decode_queries_b1(tcd, "tiny", 16, residency="global")
    for a, b in zip(c, g):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_tiny_batched_equals_batch1_and_shuffle_invariant(tcd):
    """Sequences are independent: a batch of all 64 queries, and the same batch
    shuffled, give each query exactly its batch-1 result ("Constraint made
    cheaper than no constraint": identical results across shuffled batches)."""
    w = workload("tiny")
    hid, outs = _decode_queries_b1(tcd, "tiny", w.n_queries)
    ctx, _ = make_ctx(tcd, "tiny", max_batch=w.n_queries)
    buf = DecodeBuffers(w.max_steps, w.n_queries, w.hidden, w.max_steps)
    buf.load(hid)
    full = buf.run(ctx, w.k)
    perm = w.order_rng(1).permutation(w.n_queries)
    buf.load(hid[:, perm])
    shuf = buf.run(ctx, w.k)
    for q in range(w.n_queries):
        for i in range(4):
            one = outs[q][i][0]
            assert np.array_equal(full[i][q], one)
        inv = int(np.where(perm == q)[0][0])
        for i in range(4):
            assert np.array_equal(shuf[i][inv], full[i][q])
    ctx.close()


def test_large_head_sparse_all_queries(tcd):
    """The 42-tool catalog in constant memory over the 622 MB head, 1000 queries at batch 1, k=5."""
    w = workload("large_head")
    hid, outs = _decode_queries_b1(tcd, "large_head", w.n_queries)
    flips = 0
    for q, out in enumerate(outs):
        reps = check_against_oracle("large_head", hid[:, q:q + 1], out, w.k, w.max_steps, exact=False)
        flips += sum(r.flips for r in reps)
        assert out[3][0] == 0
    assert flips <= 5, flips


def test_large_head_dense_equals_sparse(tcd):
    w = workload("large_head")
    _, sp = _decode_queries_b1(tcd, "large_head", 6, head=tcd.HEAD_SPARSE)
    _, de = _decode_queries_b1(tcd, "large_head", 6, head=tcd.HEAD_DENSE)
    for a, b in zip(sp, de):
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def _batched_run(tcd, name, n_batches, mode="graph"):
    w = workload(name)
    ctx, _ = make_ctx(tcd, name)
    buf = DecodeBuffers(w.max_steps, w.batch, w.hidden, w.max_steps)
    results = []
    for i in range(n_batches):
        hid = w.hidden_states(i * w.batch, w.batch)
        buf.load(hid)
        results.append((hid, buf.run(ctx, w.k, mode=mode)))
    ctx.close()
    return results


def test_batched_global_b64(tcd):
    """1000-tool prefix catalog in global memory, batches of 64, k=1 (two of the 64 batches)."""
    w = workload("batched")
    for hid, out in _batched_run(tcd, "batched", 2):
        assert np.all(out[3] == 0)
        check_against_oracle("batched", hid, out, w.k, w.max_steps, exact=False)


def test_unstructured_hex_b16(tcd):
    """Random hex catalog: root fan-out above 256, 4096-slot candidate buffer, B=16, k=2."""
    w = workload("unstructured")
    (hid, out), = _batched_run(tcd, "unstructured", 1)
    assert np.all(out[3] == 0)
    check_against_oracle("unstructured", hid, out, w.k, w.max_steps, exact=False)


def test_tensor_batch_sparse_b256(tcd):
    """B=256, k=3 over the 1000-tool catalog with the sparse head."""
    w = workload("tensor_batch")
    (hid, out), = _batched_run(tcd, "tensor_batch", 1)
    assert np.all(out[3] == 0)
    check_against_oracle("tensor_batch", hid, out, w.k, w.max_steps, exact=False)


def test_batched_host_equals_graph(tcd):
    (h1, g), = _batched_run(tcd, "unstructured", 1, mode="graph")
    (h2, h), = _batched_run(tcd, "unstructured", 1, mode="host")
    for x, y in zip(g, h):
        assert np.array_equal(x, y)


def _run_head(tcd, name, head, n_batches=1, batch=None, mode="graph"):
    w = workload(name)
    B = batch or w.batch
    ctx, _ = make_ctx(tcd, name, max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    out = []
    for i in range(n_batches):
        hid = w.hidden_states(i * B, B)
        buf.load(hid)
        out.append((hid, buf.run(ctx, w.k, head=head, mode=mode)))
    ctx.close()
    return out


def test_tiny_union_gemm_bitexact(tcd):
    """The union-of-legal-rows tcgen05 GEMM on integer-valued inputs: tensor-core
    fp32 sums of these values are exact, so tokens and logits equal the oracle's."""
    w = workload("tiny")
    (hid, out), = _run_head(tcd, "tiny", tcd.HEAD_UNION_GEMM, batch=w.n_queries)
    assert np.all(out[3] == 0)
    check_against_oracle("tiny", hid, out, w.k, w.max_steps, exact=True)


def test_tiny_gemm_heads_equal_sparse(tcd):
    w = workload("tiny")
    (_, sp), = _run_head(tcd, "tiny", tcd.HEAD_SPARSE, batch=w.n_queries)
    (_, un), = _run_head(tcd, "tiny", tcd.HEAD_UNION_GEMM, batch=w.n_queries)
    (_, dg), = _run_head(tcd, "tiny", tcd.HEAD_DENSE_GEMM, batch=w.n_queries)
    for x, y, z in zip(sp, un, dg):
        assert np.array_equal(x, y) and np.array_equal(x, z)


def test_tensor_batch_union_gemm_b256(tcd):
    """B=256, k=3 over the 1000-tool catalog with the union GEMM head."""
    w = workload("tensor_batch")
    (hid, out), = _run_head(tcd, "tensor_batch", tcd.HEAD_UNION_GEMM)
    assert np.all(out[3] == 0)
    check_against_oracle("tensor_batch", hid, out, w.k, w.max_steps, exact=False)


def test_union_and_dense_gemm_b64(tcd):
    """Both GEMM heads against the oracle at B=64, k=1 (the union head sums K in
    16 fixed splits, the dense GEMM in one pass: both within tolerance)."""
    w = workload("batched")
    for head in (tcd.HEAD_UNION_GEMM, tcd.HEAD_DENSE_GEMM):
        (hid, out), = _run_head(tcd, "batched", head)
        assert np.all(out[3] == 0)
        check_against_oracle("batched", hid, out, w.k, w.max_steps, exact=False)


def test_union_gemm_batch_invariant(tcd):
    """A sequence's union-GEMM result does not depend on its batch-mates: the
    same 64 queries decoded as one batch and in a shuffled order agree bitwise."""
    w = workload("batched")
    ctx, _ = make_ctx(tcd, "batched")
    buf = DecodeBuffers(w.max_steps, w.batch, w.hidden, w.max_steps)
    hid = w.hidden_states(0, w.batch)
    buf.load(hid)
    a = buf.run(ctx, w.k, head=tcd.HEAD_UNION_GEMM)
    perm = w.order_rng(2).permutation(w.batch)
    buf.load(hid[:, perm])
    b = buf.run(ctx, w.k, head=tcd.HEAD_UNION_GEMM)
    for x, y in zip(a, b):
        assert np.array_equal(x[perm], y)
    ctx.close()


def test_union_gemm_ragged_m_split_equals_narrow_batches(tcd):
    """Above 128 sequences the union GEMM runs each 128-sequence M tile as a
    task of its own (here a full tile and a ragged one of 72); every sequence's
    result equals the one it gets in batches of at most 128 (one M tile),
    bit for bit, and stays within the oracle's tolerance."""
    w = workload("batched")
    B = 200
    hid = w.hidden_states(0, B)
    ctx, _ = make_ctx(tcd, "batched", max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(hid)
    wide = buf.run(ctx, w.k, head=tcd.HEAD_UNION_GEMM)
    assert np.all(wide[3] == 0)
    for lo, hi in ((0, 128), (128, 200)):
        part = DecodeBuffers(w.max_steps, hi - lo, w.hidden, w.max_steps)
        part.load(hid[:, lo:hi])
        out = part.run(ctx, w.k, head=tcd.HEAD_UNION_GEMM)
        for i in range(4):
            assert np.array_equal(out[i], wide[i][lo:hi])
    ctx.close()
    check_against_oracle("batched", hid, wide, w.k, w.max_steps, exact=False, seqs=range(0, B, 8))


def test_tiny_union_gemm_m_split_bitexact(tcd):
    """Integer-valued inputs at B=200 (M-split union GEMM without a K split,
    the masked-argmax epilogue): tokens and logits equal the sparse head's."""
    w = workload("tiny")
    (_, sp), = _run_head(tcd, "tiny", tcd.HEAD_SPARSE, batch=200)
    (hid, un), = _run_head(tcd, "tiny", tcd.HEAD_UNION_GEMM, batch=200)
    assert np.all(un[3] == 0)
    for x, y in zip(sp, un):
        assert np.array_equal(x, y)
    check_against_oracle("tiny", hid, un, w.k, w.max_steps, exact=True, seqs=range(0, 200, 10))


def test_union_gemm_host_equals_graph(tcd):
    (_, g), = _run_head(tcd, "batched", tcd.HEAD_UNION_GEMM, mode="graph")
    (_, h), = _run_head(tcd, "batched", tcd.HEAD_UNION_GEMM, mode="host")
    for x, y in zip(g, h):
        assert np.array_equal(x, y)


def test_wide_batch_equals_two_narrow_batches(tcd):
    """Above the SM count the one-CTA step stages the hidden state in shared
    memory (two CTAs per SM); its results equal those of two smaller batches
    decoded with the register-resident variant, bit for bit."""
    w = workload("tensor_batch")
    B = 256
    hid = w.hidden_states(0, B)
    ctx, _ = make_ctx(tcd, "tensor_batch", max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(hid)
    wide = buf.run(ctx, w.k)
    half = DecodeBuffers(w.max_steps, B // 2, w.hidden, w.max_steps)
    for h in range(2):
        half.load(hid[:, h * (B // 2):(h + 1) * (B // 2)])
        out = half.run(ctx, w.k)
        for i in range(4):
            assert np.array_equal(out[i], wide[i][h * (B // 2):(h + 1) * (B // 2)])
    ctx.close()
    assert np.all(wide[3] == 0)


def test_host_steps_with_mixed_heads_equal_sparse_steps(tcd):
    """tc_step with a different head on every other step: the other heads move
    a sequence without refreshing the sparse step's precomputed candidate
    list, which the next sparse step must not use.  On integer inputs every
    head gives the same tokens and logits, so the mixed sequence of steps
    equals the all-sparse one bit for bit."""
    torch = torch_mod()
    w = workload("tiny")
    B = 16
    hid_bits = w.hidden_states(0, B)  # [S, B, H]
    S = hid_bits.shape[0]
    hid = to_dev_bf16(hid_bits)
    ctx, _ = make_ctx(tcd, "tiny", max_batch=B)
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    lg = torch.empty(B, dtype=torch.float32, device="cuda")
    st = torch.empty(B, dtype=torch.int32, device="cuda")
    others = [tcd.HEAD_DENSE, tcd.HEAD_UNION_GEMM, tcd.HEAD_DENSE_GEMM]

    def run(mixed):
        ctx.reset(B, w.k)
        out = []
        for t in range(S):
            head = others[(t // 2) % 3] if (mixed and t % 2 == 1) else tcd.HEAD_SPARSE
            ctx.step(hid[t], tok, lg, st, head=head)
            torch.cuda.synchronize()
            out.append((tok.cpu().numpy().copy(), lg.cpu().numpy().copy(), st.cpu().numpy().copy()))
        return out

    plain, mixed = run(False), run(True)
    ctx.close()
    for (a_t, a_l, a_s), (b_t, b_l, b_s) in zip(plain, mixed):
        assert np.array_equal(a_t, b_t) and np.array_equal(a_l, b_l) and np.array_equal(a_s, b_s)
    assert np.all(plain[-1][2] == 0)


def test_tiny_dense_gemm_two_m_tiles_bitexact(tcd):
    """The full-vocabulary tcgen05 GEMM above 128 sequences keeps both
    128-sequence M tiles in one CTA (every embedding tile read once, a
    three-stage ring, two 256-column TMEM accumulators).  On integer-valued
    inputs every fp32 sum is exact, so at B=256 (two full tiles) and B=200 (a
    ragged second tile of 72) tokens and logits equal the sparse head's bit for
    bit, and the oracle's ("Understanding Inference for Systems Engineers",
    section 7.5: every logit, then the mask, then the argmax)."""
    w = workload("tiny")
    for B in (256, 200):
        (_, sp), = _run_head(tcd, "tiny", tcd.HEAD_SPARSE, batch=B)
        (hid, dg), = _run_head(tcd, "tiny", tcd.HEAD_DENSE_GEMM, batch=B)
        assert np.all(dg[3] == 0)
        for x, y in zip(sp, dg):
            assert np.array_equal(x, y), B
        check_against_oracle("tiny", hid, dg, w.k, w.max_steps, exact=True)


def test_tensor_batch_dense_gemm_b256(tcd):
    """The dense comparator of the union head at its own shape: B=256, k=3,
    hidden 4096, every vocabulary row by the two-M-tile tcgen05 GEMM, then each
    sequence's mask and argmax; every sequence teacher-forced against the
    oracle (Gaussian inputs: chosen logits within 1e-3 relative, a differing
    token only below the oracle's 1e-5 top-2 margin)."""
    w = workload("tensor_batch")
    (hid, out), = _run_head(tcd, "tensor_batch", tcd.HEAD_DENSE_GEMM)
    assert np.all(out[3] == 0)
    reps = check_against_oracle("tensor_batch", hid, out, w.k, w.max_steps, exact=False)
    assert sum(r.flips for r in reps) <= 5


def test_dense_gemm_ragged_two_m_tiles_equal_narrow_batches(tcd):
    """A sequence's dense-GEMM result does not depend on which M tile, or
    which kernel configuration, computes it: B=200 in the two-M-tile kernel
    equals the batches of its first 128 and last 72 sequences (one M tile
    each) bit for bit, and stays within the oracle's tolerance."""
    w = workload("batched")
    B = 200
    hid = w.hidden_states(0, B)
    ctx, _ = make_ctx(tcd, "batched", max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(hid)
    wide = buf.run(ctx, w.k, head=tcd.HEAD_DENSE_GEMM)
    assert np.all(wide[3] == 0)
    for lo, hi in ((0, 128), (128, 200)):
        part = DecodeBuffers(w.max_steps, hi - lo, w.hidden, w.max_steps)
        part.load(hid[:, lo:hi])
        out = part.run(ctx, w.k, head=tcd.HEAD_DENSE_GEMM)
        for i in range(4):
            assert np.array_equal(out[i], wide[i][lo:hi]), (lo, i)
    ctx.close()
    check_against_oracle("batched", hid, wide, w.k, w.max_steps, exact=False)


def test_multi_cta_step_x_in_shared_memory_equals_register_variant(tcd):
    """The multi-CTA sparse step stages the hidden state in shared memory (two
    CTAs per SM) when one wave of its register variant cannot give every
    sequence the CTAs its widest node needs: the hex catalog (root fan-out
    267) at B=16 takes it, at B=4 it does not.  Both use the same lane map and
    reduction tree, so the 16 queries decoded as one batch equal the same
    queries in four batches of 4, bit for bit."""
    w = workload("unstructured")
    hid = w.hidden_states(0, 16)
    ctx, _ = make_ctx(tcd, "unstructured", max_batch=16)
    wide = DecodeBuffers(w.max_steps, 16, w.hidden, w.max_steps)
    wide.load(hid)
    a = wide.run(ctx, w.k)
    assert np.all(a[3] == 0)
    narrow = DecodeBuffers(w.max_steps, 4, w.hidden, w.max_steps)
    for q in range(0, 16, 4):
        narrow.load(hid[:, q:q + 4])
        b = narrow.run(ctx, w.k)
        for i in range(4):
            assert np.array_equal(b[i], a[i][q:q + 4]), (q, i)
    ctx.close()


def test_hex_catalog_b256_sparse_and_union(tcd):
    """The hex catalog (root fan-out 267) at B=256, the launch shape the bench
    reports beside the workload's own B=16: the multi-CTA step with the hidden
    state in shared memory and one CTA per sequence, and the union GEMM with
    two 128-sequence M tiles and wide union tiles; every 8th sequence
    teacher-forced against the oracle, all sequences finished."""
    w = workload("unstructured")
    B = 256
    hid = w.hidden_states(0, B)
    ctx, _ = make_ctx(tcd, "unstructured", max_batch=B)
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(hid)
    for head in (tcd.HEAD_SPARSE, tcd.HEAD_UNION_GEMM):
        out = buf.run(ctx, w.k, head=head)
        assert np.all(out[3] == 0), head
        check_against_oracle("unstructured", hid, out, w.k, w.max_steps, exact=False, seqs=range(0, B, 8))
    ctx.close()
