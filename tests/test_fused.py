"""GPU parity of the fused backward (swa_attn_bwd_fused: one kernel for dK, dV and the dQ partials,
dQ summed in an fp32 accumulator) against the fp64 oracle, at the bar of every parity test: 1e-2
norm-wise for dQ, dK, dV (whole tensor and every head), zero gradients bounded as in the edge sweep.
Its dK and dV must equal the split backward's bit for bit (the same products in the same order);
its dQ, whose partials are added in a varying order, must agree with the split path's closely.

Cases: the edge sweep (ragged lengths, windows 1 / 7 / 64 / N, D 64 and 128), multi-tile shapes with
G = 1 ... 4, walks long enough to cycle the Q ring and the dQ staging several times, queries shorter
than keys (key blocks that no query sees), two-sided windows, fp16, and the phase entry points.
"""
import numpy as np
import pytest
import torch

import swa_inputs as si
from oracle import swa_oracle as orc
from test_parity import MULTI_TILE, _multi_case, check_against_oracle, check_per_head

pytestmark = pytest.mark.gpu


def _both(swa, g, W, scale, causal=True):
    o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], W, scale, causal=causal)
    fused = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, W, scale, causal=causal,
                             fused=True)
    split = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, W, scale, causal=causal,
                             fused=False)
    swa.swa_check_device()
    return o, lse, fused, split


def _np(t):
    return t.detach().float().cpu().double().numpy()


def _check(swa, case, inputs, W, causal=True, ref_w2=None):
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in inputs.items()}
    o, lse, (dq, dk, dv), (dq_s, dk_s, dv_s) = _both(swa, g, W, case.softmax_scale, causal)
    assert torch.equal(dk, dk_s) and torch.equal(dv, dv_s)
    ref = orc.oracle_backward(inputs["q"], inputs["k"], inputs["v"], inputs["do"], W,
                              case.softmax_scale, causal=causal)
    gpu = {"o": _np(o), "lse": _np(lse), "dq": _np(dq), "dk": _np(dk), "dv": _np(dv)}
    check_against_oracle(case, gpu, ref, ref_w2)
    n = np.linalg.norm(_np(dq_s))
    if n > 0:
        assert np.linalg.norm(_np(dq) - _np(dq_s)) <= 2e-3 * n
    return gpu


@pytest.mark.parametrize("case", si.edge_cases(), ids=lambda c: c.name())
def test_fused_edge_sweep(swa, case):
    inputs = si.make_inputs(case)
    ref_w2 = None
    if case.W == 1 or case.N == 1:
        c2 = si.Case(**{**case.__dict__, "W": 2})
        ref_w2 = orc.oracle_backward(inputs["q"], inputs["k"], inputs["v"], inputs["do"], 2,
                                     case.softmax_scale)
        if case.N == 1:
            ref_w2 = {k: np.ones_like(v) for k, v in ref_w2.items()}
    _check(swa, case, inputs, case.W, ref_w2=ref_w2)


@pytest.mark.parametrize("shape", MULTI_TILE + [(1, 2, 1, 2100, 128, 900), (2, 6, 2, 1500, 64, 700)])
def test_fused_multi_tile(swa, shape):
    case = _multi_case(shape)
    _check(swa, case, si.make_inputs(case), case.W)


@pytest.mark.parametrize("Lq,Lk,W,causal,D", [(200, 700, 150, False, 128), (17, 300, 7, True, 64),
                                              (300, 1000, 100, True, 128),
                                              (130, 900, 600, False, 64)])
def test_fused_queries_shorter_than_keys(swa, Lq, Lk, W, causal, D):
    case = si.Case(B=1, Hq=4, Hkv=2, N=Lk, D=D, W=W, seed=21)
    inp = si.make_inputs(case)
    for key in ("q", "do"):
        inp[key] = inp[key][:, :, Lk - Lq:].contiguous()
    _check(swa, case, inp, W, causal)


@pytest.mark.parametrize("D", [64, 128])
def test_fused_fp16(swa, D):
    case = si.Case(B=1, Hq=4, Hkv=2, N=777, D=D, W=200, seed=22)
    inp = si.make_inputs(case, dtype=torch.float16)
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in inp.items()}
    o, lse, (dq, dk, dv), (dq_s, dk_s, dv_s) = _both(swa, g, case.W, case.softmax_scale)
    assert dq.dtype == torch.float16
    assert torch.equal(dk, dk_s) and torch.equal(dv, dv_s)
    ref = orc.oracle_backward(inp["q"], inp["k"], inp["v"], inp["do"], case.W, case.softmax_scale)
    for key, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        x = _np(t)
        assert np.linalg.norm(x - ref[key]) <= 1e-2 * np.linalg.norm(ref[key]), key
        check_per_head(key, x, ref[key])


def test_fused_phases_equal_the_fused_call(swa):
    """The three phase entry points run the same kernels as swa_attn_bwd_fused: dK and dV equal
    bit for bit, dQ within the fused path's own run-to-run spread."""
    case = si.Case(B=1, Hq=8, Hkv=4, N=1500, D=128, W=500, seed=23)
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in si.make_inputs(case).items()}
    o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], case.W, case.softmax_scale)
    a = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, case.W, case.softmax_scale)
    marks = []
    b = swa.swa_attn_bwd_phases(g["q"], g["k"], g["v"], o, g["do"], lse, case.W,
                                case.softmax_scale, fused=True, between=marks.append)
    swa.swa_check_device()
    assert marks == [0, 1, 2, 3]
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    rel = (torch.linalg.vector_norm(a[0].float() - b[0].float()) /
           torch.linalg.vector_norm(a[0].float())).item()
    assert rel <= 2e-3


def test_fused_workspace_too_small_is_refused(swa):
    case = si.tiny_case()
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in si.make_inputs(case).items()}
    o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], case.W, case.softmax_scale)
    n = swa.swa_attn_bwd_fused_workspace_bytes(case.B, case.Hq, case.N, case.D)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, case.W, case.softmax_scale,
                     workspace=ws, fused=True)
    with pytest.raises(swa.SwaError):
        swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, case.W, case.softmax_scale,
                         workspace=ws[:n - 16], fused=True)
    swa.swa_check_device()
