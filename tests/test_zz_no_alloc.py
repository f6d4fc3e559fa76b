"""GPU test of swa_attn_bwd_noalloc, the backward entry point that allocates nothing.

Some callers cannot allocate scratch device memory (their device heap is owned by a host
framework's allocator, or they must not allocate once running), so this entry point keeps the
backward's Delta scratch in a fixed device array inside the library instead of taking a workspace.
Called through the C ABI, it must give the same dQ, dK, dV as swa_attn_bwd (which takes a
caller-allocated workspace) bit for bit, on two calls in a row, since the array is shared and keeps
the previous call's contents.  The file name sorts last so that a stop-at-first-failure run has
already run every other test when it gets here.
"""
import pytest
import torch

import swa_inputs as si

pytestmark = pytest.mark.gpu


def _noalloc_bwd(lib, g, o, lse, case, stream):
    dq, dk, dv = torch.empty_like(g["q"]), torch.empty_like(g["k"]), torch.empty_like(g["v"])
    rc = lib.swa_attn_bwd_noalloc(
        g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(), o.data_ptr(), g["do"].data_ptr(),
        lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
        case.B, case.Hq, case.Hkv, case.N, case.D, case.W, case.softmax_scale, stream)
    assert rc == 0, lib.swa_strerror(rc)
    return dq, dk, dv


@pytest.mark.parametrize("case", [
    si.Case(B=2, Hq=4, Hkv=2, N=255, D=128, W=64, seed=3),
    si.Case(B=1, Hq=8, Hkv=2, N=1000, D=64, W=300, seed=4),
], ids=lambda c: c.name())
def test_noalloc_matches_workspace_backward(swa, case):
    lib = swa.load()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    # Two different problems back to back, then the first again: when each call starts, the shared
    # array holds the previous call's Delta rows.  Both entry points run the same kernels in the same
    # order on the same inputs, so their results must be equal bit for bit.
    other = si.Case(**{**case.__dict__, "seed": case.seed + 100})
    first = None
    for c in (case, other, case):
        g = {k: v.to(dev) for k, v in si.make_inputs(c).items()}
        o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], c.W, c.softmax_scale)
        ref = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, c.W, c.softmax_scale,
                               fused=False)
        for _ in range(2):
            got = _noalloc_bwd(lib, g, o, lse, c, stream)
            swa.swa_check_device()
            for name, a, b in zip(("dq", "dk", "dv"), got, ref):
                assert torch.isfinite(a.float()).all(), name
                assert torch.equal(a, b), name
        if first is None:
            first = got
        elif c is case:  # the repeated first problem gives the first call's gradients again
            for name, a, b in zip(("dq", "dk", "dv"), got, first):
                assert torch.equal(a, b), name


def test_noalloc_rejects_too_many_rows(swa):
    lib = swa.load()
    rows_max = 1 << 22
    fake = 0x10000
    # B*Hq*N one row above the array's capacity: refused on the host, nothing launched.
    rc = lib.swa_attn_bwd_noalloc(*([fake] * 9), 1, 4, 1, rows_max // 4 + 1, 128, 64, 0.1, None)
    assert rc == 6
