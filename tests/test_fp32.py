"""GPU parity of fp32 tensors (swa_attn_fwd_f32 / swa_attn_bwd_f32 through the binding).

Every case is checked against the fp64 oracle on the unrounded fp32 draws, at the plain bars:
norm-wise relative error <= 1e-2 for O, dQ, dK, dV (whole tensor and every head) and max |LSE
difference| <= 1e-3.  The library rounds each input once to bf16 for the tensor cores and corrects
the forward's log-sum-exp for the rounding of q and k to first order (a split of q and k into bf16
high and low parts); without that correction the rounding alone moves LSE by up to ~6e-3 on these
draws.  Where the exact gradient is zero (W = 1) the GPU norm must stay within 1e-2 of the window-2
gradient's norm.  On inputs already representable in bf16 (low parts zero) the fp32 calls give
exactly the bf16 calls' results, widened.  The pages' gradient sweep runs fp32 inputs (Lab 28
record, numbers entry "Gradient parity, small shapes").
"""
import numpy as np
import pytest
import torch

import swa_inputs as si
from oracle import swa_oracle as orc
from test_parity import check_per_head, run_gpu

pytestmark = pytest.mark.gpu

F32 = torch.float32
REL_TOL = 1e-2
LSE_TOL = 1e-3


def _cases():
    cases = [c for c in si.edge_cases() if c.N in (17, 255, 512)]
    cases.append(si.Case(B=1, Hq=4, Hkv=2, N=1000, D=128, W=300, seed=6))
    return cases


def _oracle(case, inputs, W=None, causal=True):
    return orc.oracle_backward(inputs["q"], inputs["k"], inputs["v"], inputs["do"],
                               case.W if W is None else W, case.softmax_scale, causal=causal)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _check_unrounded(case, gpu, inputs, W, causal=True):
    """The fp32 outputs against the oracle on the same fp32 values, at the plain bars."""
    ref = _oracle(case, inputs, W=W, causal=causal)
    dl = np.abs(gpu["lse"] - ref["lse"])
    assert np.max(dl) <= LSE_TOL, ("lse", float(np.max(dl)))
    assert _rel(gpu["o"], ref["o"]) <= REL_TOL, ("o", _rel(gpu["o"], ref["o"]))
    check_per_head("o", gpu["o"], ref["o"])
    ref_w2 = _oracle(case, inputs, W=2, causal=causal) if W == 1 else None
    for key in ("dq", "dk", "dv"):
        if W == 1 and key in ("dq", "dk"):
            assert np.linalg.norm(gpu[key]) <= REL_TOL * np.linalg.norm(ref_w2[key]), key
        else:
            assert _rel(gpu[key], ref[key]) <= REL_TOL, (key, _rel(gpu[key], ref[key]))
            check_per_head(key, gpu[key], ref[key])
    return float(np.max(dl))


def _check_both(case, gpu, inputs, W=None, causal=True):
    return _check_unrounded(case, gpu, inputs, case.W if W is None else W, causal)


def test_tiny_fp32(swa):
    case = si.tiny_case()
    inputs = si.make_inputs(case, dtype=F32)
    _check_both(case, run_gpu(swa, case, inputs), inputs)


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c.name())
def test_fp32_sweep(swa, case):
    inputs = si.make_inputs(case, dtype=F32)
    _check_both(case, run_gpu(swa, case, inputs), inputs)


@pytest.mark.parametrize("Lq,Lk,W,causal", [(200, 700, 150, False), (17, 300, 7, True),
                                            (130, 900, 1, True)])
def test_fp32_queries_shorter_than_keys(swa, Lq, Lk, W, causal):
    case = si.Case(B=1, Hq=4, Hkv=2, N=Lk, D=128, W=W, seed=8)
    inp = si.make_inputs(case, dtype=F32)
    for key in ("q", "do"):
        inp[key] = inp[key][:, :, Lk - Lq:].contiguous()
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in inp.items()}
    o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], W, case.softmax_scale, causal=causal)
    dq, dk, dv = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, W, case.softmax_scale,
                                  causal=causal)
    swa.swa_check_device()
    got = {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
    got = {k: v.double().cpu().numpy() for k, v in got.items()}
    _check_unrounded(case, got, inp, W, causal)


def test_fp32_equals_bf16_path_on_rounded_inputs(swa):
    """Rounding happens once, to nearest even, as torch rounds: on unrounded fp32 inputs the fp32
    forward's O equals the bf16 forward's O on torch-rounded inputs bit for bit (widened), and its
    LSE differs only by the correction.  On bf16-representable inputs the low parts are zero, so
    every output, LSE and gradients included, equals the bf16 calls' bit for bit."""
    case = si.Case(B=1, Hq=4, Hkv=2, N=700, D=128, W=200, seed=9)
    dev = torch.device("cuda:0")
    raw = {k: v.to(dev) for k, v in si.make_inputs(case, dtype=F32).items()}
    bf = {k: v.to(torch.bfloat16) for k, v in raw.items()}
    o_b, l_b = swa.swa_attn_fwd(bf["q"], bf["k"], bf["v"], case.W, case.softmax_scale)
    g_b = swa.swa_attn_bwd(bf["q"], bf["k"], bf["v"], o_b, bf["do"], l_b, case.W,
                           case.softmax_scale, fused=False)  # the split path, as fp32 calls run
    o_f, l_f = swa.swa_attn_fwd(raw["q"], raw["k"], raw["v"], case.W, case.softmax_scale)
    rep = {k: v.float() for k, v in bf.items()}  # bf16-representable fp32 tensors
    o_r, l_r = swa.swa_attn_fwd(rep["q"], rep["k"], rep["v"], case.W, case.softmax_scale)
    g_r = swa.swa_attn_bwd(rep["q"], rep["k"], rep["v"], o_r, rep["do"], l_r, case.W,
                           case.softmax_scale)
    swa.swa_check_device()
    assert o_f.dtype == F32 and all(t.dtype == F32 for t in g_r)
    assert torch.equal(o_f, o_b.float())
    assert not torch.equal(l_f, l_b)  # the low parts of the raw draws are not zero
    assert torch.equal(o_r, o_b.float()) and torch.equal(l_r, l_b)
    for a, b in zip(g_r, g_b):
        assert torch.equal(a, b.float())


def test_fp32_lse_correction_is_second_order(swa):
    """The correction leaves only second-order terms: on the multi-tile case the LSE error is far
    below both the bar and the uncorrected error (the bf16 path on the rounded inputs)."""
    case = si.Case(B=1, Hq=4, Hkv=2, N=1000, D=128, W=300, seed=6)
    inputs = si.make_inputs(case, dtype=F32)
    ref = _oracle(case, inputs)
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in inputs.items()}
    _, l_f = swa.swa_attn_fwd(g["q"], g["k"], g["v"], case.W, case.softmax_scale)
    bf = {k: v.to(torch.bfloat16) for k, v in g.items()}
    _, l_b = swa.swa_attn_fwd(bf["q"], bf["k"], bf["v"], case.W, case.softmax_scale)
    swa.swa_check_device()
    e_f = float(np.max(np.abs(l_f.double().cpu().numpy() - ref["lse"])))
    e_b = float(np.max(np.abs(l_b.double().cpu().numpy() - ref["lse"])))
    assert e_f <= 2e-4 and e_f <= 0.1 * e_b, (e_f, e_b)


def test_fp32_caller_workspace_and_outputs(swa):
    case = si.tiny_case()
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in si.make_inputs(case, dtype=F32).items()}
    n = swa.swa_attn_f32_workspace_bytes(case.B, case.Hq, case.Hkv, case.N, case.N, case.D)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], case.W, case.softmax_scale, workspace=ws)
    dq, dk, dv = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, case.W,
                                  case.softmax_scale, workspace=ws)
    swa.swa_check_device()
    o2, lse2 = swa.swa_attn_fwd(g["q"], g["k"], g["v"], case.W, case.softmax_scale)
    swa.swa_check_device()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    with pytest.raises(swa.SwaError):
        swa.swa_attn_fwd(g["q"], g["k"], g["v"], case.W, case.softmax_scale, workspace=ws[:n - 1])
