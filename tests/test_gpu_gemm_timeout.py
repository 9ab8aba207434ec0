"""The tcgen05 GEMM heads' bounded waits: a wait that runs out fails the step
loudly, without a fault or a hang, and the context works again after a reset
("Constraint made cheaper than no constraint", section "Masked sampling inside
the sampler": a step that cannot finish must stop with an error, not emit).

tc_gemm_wait_test makes the kernel's first CTA issue nothing for its first
pipeline stage and bounds every barrier wait by a small poll count, so the
MMA issuer's wait on that stage runs out: no copy is outstanding on it and
nothing is left running when the kernel returns.
"""
import numpy as np
import pytest

from gpu_common import DecodeBuffers, make_ctx, to_dev_bf16, torch_mod, workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("head_name,B", [("HEAD_UNION_GEMM", 64), ("HEAD_DENSE_GEMM", 200)])
def test_gemm_wait_timeout_fails_loudly_and_recovers(tcd, head_name, B):
    """The union head (row gathers, one M tile) at B=64 and the dense head
    (two M tiles in one CTA) at B=200."""
    torch = torch_mod()
    head = getattr(tcd, head_name)
    w = workload("tiny")
    ctx, _ = make_ctx(tcd, "tiny", max_batch=B)
    hid_bits = w.hidden_states(0, B)
    hid = to_dev_bf16(hid_bits)
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    lg = torch.empty(B, dtype=torch.float32, device="cuda")
    st = torch.empty(B, dtype=torch.int32, device="cuda")

    def one_step(h):
        ctx.reset(B, w.k)
        ctx.step(hid[0], tok, lg, st, head=h)
        torch.cuda.synchronize()
        return tok.cpu().numpy().copy(), lg.cpu().numpy().copy(), st.cpu().numpy().copy()

    want = one_step(tcd.HEAD_SPARSE)
    assert np.all(want[2] == 0)

    ctx.gemm_wait_test(True, 2000)
    t, _, s = one_step(head)
    assert np.all(s == tcd.TC_ERR_DEVICE_TIMEOUT), s
    assert np.all(t == -1)
    assert ctx.first_error() == (0, tcd.TC_ERR_DEVICE_TIMEOUT)
    # The device-resident loop fails its first step the same way.
    buf = DecodeBuffers(w.max_steps, B, w.hidden, w.max_steps)
    buf.load(hid_bits)
    out = buf.run(ctx, w.k, head=head)
    assert np.all(out[3] == tcd.TC_ERR_DEVICE_TIMEOUT) and np.all(out[2] == 0)

    ctx.gemm_wait_test(False, 0)
    got = one_step(head)
    assert ctx.first_error() == (-1, 0)
    for a, b in zip(got, want):
        assert np.array_equal(a, b)
    # A whole decode after recovery equals the sparse head's (integer inputs: exact).
    gemm = buf.run(ctx, w.k, head=head)
    sparse = buf.run(ctx, w.k, head=tcd.HEAD_SPARSE)
    for a, b in zip(gemm, sparse):
        assert np.array_equal(a, b)
    ctx.close()
