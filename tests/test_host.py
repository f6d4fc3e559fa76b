"""GPU: swa_attn_fwd_bwd_host (host tensors in and out, copies pipelined with the kernels over
chunks of (batch, kv head) groups) gives exactly the device-resident swa_attn_fwd / swa_attn_bwd
results, for chunk sizes that divide the group count, that do not, and that exceed it; one case
is also checked against the fp64 oracle at the usual bar."""
import numpy as np
import pytest
import torch

import swa_inputs as si
from oracle import swa_oracle as orc

pytestmark = pytest.mark.gpu


def _pinned(inp):
    return {k: v.contiguous().pin_memory() for k, v in inp.items()}


@pytest.mark.parametrize("case,U", [
    (si.Case(B=1, Hq=4, Hkv=2, N=700, D=128, W=200, seed=1), 1),
    (si.Case(B=2, Hq=4, Hkv=2, N=300, D=64, W=64, seed=2), 3),
    (si.Case(B=1, Hq=2, Hkv=1, N=256, D=256, W=64, seed=3), 5),
    (si.Case(B=3, Hq=8, Hkv=4, N=517, D=128, W=1000, seed=4), 4),
])
def test_host_pipeline_equals_device_path(swa, case, U):
    inp = _pinned(si.make_inputs(case))
    dev = torch.device("cuda:0")
    o_h, lse_h, dq_h, dk_h, dv_h = swa.swa_attn_fwd_bwd_host(
        inp["q"], inp["k"], inp["v"], inp["do"], case.W, case.softmax_scale, units_per_chunk=U)
    torch.cuda.synchronize(dev)
    swa.swa_check_device()
    g = {k: v.to(dev) for k, v in inp.items()}
    o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], case.W, case.softmax_scale)
    dq, dk, dv = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, case.W,
                                  case.softmax_scale, fused=False)
    swa.swa_check_device()
    for name, a, b in (("o", o_h, o), ("lse", lse_h, lse), ("dq", dq_h, dq), ("dk", dk_h, dk),
                       ("dv", dv_h, dv)):
        assert torch.equal(a, b.cpu()), name


def test_host_pipeline_against_oracle(swa):
    case = si.Case(B=2, Hq=4, Hkv=2, N=400, D=128, W=150, seed=5)
    inp = _pinned(si.make_inputs(case))
    outs = swa.swa_attn_fwd_bwd_host(inp["q"], inp["k"], inp["v"], inp["do"], case.W,
                                     case.softmax_scale, units_per_chunk=1)
    torch.cuda.synchronize()
    swa.swa_check_device()
    got = dict(zip(("o", "lse", "dq", "dk", "dv"), (t.double().numpy() for t in outs)))
    ref = orc.oracle_backward(inp["q"], inp["k"], inp["v"], inp["do"], case.W, case.softmax_scale)
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= 1e-3
    for n in ("o", "dq", "dk", "dv"):
        assert np.linalg.norm(got[n] - ref[n]) / np.linalg.norm(ref[n]) <= 1e-2, n


def test_host_pipeline_back_to_back_calls(swa):
    """Two calls in a row on one stream without a host synchronisation in between: the second
    call's copies wait for the first's (fork after join), so both results are intact."""
    c1 = si.Case(B=1, Hq=4, Hkv=2, N=300, D=128, W=100, seed=6)
    c2 = si.Case(B=1, Hq=4, Hkv=2, N=300, D=128, W=40, seed=7)
    i1, i2 = _pinned(si.make_inputs(c1)), _pinned(si.make_inputs(c2))
    r1 = swa.swa_attn_fwd_bwd_host(i1["q"], i1["k"], i1["v"], i1["do"], c1.W, c1.softmax_scale,
                                   units_per_chunk=1)
    r2 = swa.swa_attn_fwd_bwd_host(i2["q"], i2["k"], i2["v"], i2["do"], c2.W, c2.softmax_scale,
                                   units_per_chunk=1)
    torch.cuda.synchronize()
    swa.swa_check_device()
    for inp, case, r in ((i1, c1, r1), (i2, c2, r2)):
        s1 = swa.swa_attn_fwd_bwd_host(inp["q"], inp["k"], inp["v"], inp["do"], case.W,
                                       case.softmax_scale, units_per_chunk=2)
        torch.cuda.synchronize()
        for a, b in zip(r, s1):
            assert torch.equal(a, b)


def test_host_pipeline_from_two_host_threads(swa):
    """Calls from two host threads on one device (each on its own torch stream) are serialised
    while they enqueue on the library's shared streams: both results stay exact."""
    import threading

    cases = [si.Case(B=1, Hq=4, Hkv=2, N=300, D=128, W=80, seed=20 + i) for i in range(2)]
    inps = [_pinned(si.make_inputs(c)) for c in cases]
    dev = torch.device("cuda:0")
    expected = []
    for c, inp in zip(cases, inps):
        r = swa.swa_attn_fwd_bwd_host(inp["q"], inp["k"], inp["v"], inp["do"], c.W,
                                      c.softmax_scale, units_per_chunk=1)
        torch.cuda.synchronize(dev)
        expected.append([t.clone() for t in r])
    results = [None, None]

    def run(i):
        torch.cuda.set_device(dev)
        s = torch.cuda.Stream(dev)
        with torch.cuda.stream(s):
            for _ in range(3):
                r = swa.swa_attn_fwd_bwd_host(inps[i]["q"], inps[i]["k"], inps[i]["v"],
                                              inps[i]["do"], cases[i].W, cases[i].softmax_scale,
                                              units_per_chunk=1)
            s.synchronize()
        results[i] = r

    th = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    swa.swa_check_device()
    for i in range(2):
        for a, b in zip(results[i], expected[i]):
            assert torch.equal(a, b)
