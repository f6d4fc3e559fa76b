"""GPU parity of fp32 tensors (swa_attn_fwd_f32 / swa_attn_bwd_f32 through the binding).

The library rounds each fp32 input once to bf16 (nearest, ties to even) for the tensor cores, so
every case is checked twice against the fp64 oracle:
  1. on the inputs rounded to bf16 on the CPU by torch: the bf16 path's bar, norm-wise relative
     error <= 1e-2 for O, dQ, dK, dV and max |LSE difference| <= 1e-3 (the fp32 path computes
     exactly that problem);
  2. on the unrounded fp32 draws: relative error <= 1e-2 for O, dQ, dK, dV, and per row
     |LSE difference| <= 1e-3 + the input-rounding bound.  With u = 2^-8 (bf16's unit roundoff)
     each product q_d k_d moves by at most |q_d| |k_d| (2u + u^2), so score s_ij moves by at most
     scale * sum_d |q_id| |k_jd| (2u + u^2), and LSE_i, a smooth maximum of row i's scores, by at
     most the largest of those over the keys row i sees.
Where the exact gradient is zero (W = 1) the GPU norm must stay within 1e-2 of the window-2
gradient's norm.  On inputs already representable in bf16 the fp32 calls give exactly the bf16
calls' results, widened.  The pages' gradient sweep runs fp32 inputs (Lab 28 record, numbers entry
"Gradient parity, small shapes").
"""
import numpy as np
import pytest
import torch

import swa_inputs as si
from oracle import swa_oracle as orc
from test_parity import check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu

F32 = torch.float32
REL_TOL = 1e-2
LSE_TOL = 1e-3


def _cases():
    cases = [c for c in si.edge_cases() if c.N in (17, 255, 512)]
    cases.append(si.Case(B=1, Hq=4, Hkv=2, N=1000, D=128, W=300, seed=6))
    return cases


U_BF16 = 2.0 ** -8


def _oracle(case, inputs, W=None, causal=True):
    return orc.oracle_backward(inputs["q"], inputs["k"], inputs["v"], inputs["do"],
                               case.W if W is None else W, case.softmax_scale, causal=causal)


def _rounded(inputs):
    return {k: v.to(torch.bfloat16) for k, v in inputs.items()}


def _lse_rounding_bound(q, k, W, scale, causal=True):
    """Per query row, the largest score change that rounding q and k to bf16 can cause over the
    keys the row sees (fp64, [B, Hq, Lq])."""
    q = q.double().numpy()
    k = k.double().numpy()
    B, Hq, Lq, _ = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    out = np.zeros((B, Hq, Lq))
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    vis = orc.visible(i, j, W, Lk - Lq, causal)
    for b in range(B):
        for h in range(Hq):
            hk = orc.kv_head_of(h, Hq, Hkv)
            prod = np.abs(q[b, h]) @ np.abs(k[b, hk]).T
            out[b, h] = scale * (2 * U_BF16 + U_BF16 ** 2) * np.where(vis, prod, 0.0).max(axis=1)
    return out


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _check_unrounded(case, gpu, inputs, W, causal=True):
    """Check 2 of the module docstring."""
    ref = _oracle(case, inputs, W=W, causal=causal)
    bound = LSE_TOL + _lse_rounding_bound(inputs["q"], inputs["k"], W, case.softmax_scale, causal)
    assert np.all(np.abs(gpu["lse"] - ref["lse"]) <= bound)
    assert _rel(gpu["o"], ref["o"]) <= REL_TOL
    ref_w2 = _oracle(case, inputs, W=2, causal=causal) if W == 1 else None
    for key in ("dq", "dk", "dv"):
        if W == 1 and key in ("dq", "dk"):
            assert np.linalg.norm(gpu[key]) <= REL_TOL * np.linalg.norm(ref_w2[key]), key
        else:
            assert _rel(gpu[key], ref[key]) <= REL_TOL, (key, _rel(gpu[key], ref[key]))


def _check_both(case, gpu, inputs, W=None, causal=True):
    W = case.W if W is None else W
    r16 = _rounded(inputs)
    ref = _oracle(case, r16, W=W, causal=causal)
    ref_w2 = _oracle(case, r16, W=2, causal=causal) if W == 1 else None
    check_against_oracle(case, gpu, ref, ref_w2)
    _check_unrounded(case, gpu, inputs, W, causal)


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
    r16 = _rounded(inp)
    ref = _oracle(case, r16, W=W, causal=causal)
    assert _rel(got["o"], ref["o"]) <= REL_TOL
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= LSE_TOL
    for key in ("dv",) if W == 1 else ("dq", "dk", "dv"):
        assert _rel(got[key], ref[key]) <= REL_TOL, key
    _check_unrounded(case, got, inp, W, causal)


def test_fp32_equals_bf16_path_on_rounded_inputs(swa):
    """Rounding happens once, to nearest even, as torch rounds: on bf16-representable fp32 inputs
    the fp32 calls reproduce the bf16 calls bit for bit, widened to fp32."""
    case = si.Case(B=1, Hq=4, Hkv=2, N=700, D=128, W=200, seed=9)
    dev = torch.device("cuda:0")
    raw = {k: v.to(dev) for k, v in si.make_inputs(case, dtype=F32).items()}
    bf = {k: v.to(torch.bfloat16) for k, v in raw.items()}
    o_b, l_b = swa.swa_attn_fwd(bf["q"], bf["k"], bf["v"], case.W, case.softmax_scale)
    g_b = swa.swa_attn_bwd(bf["q"], bf["k"], bf["v"], o_b, bf["do"], l_b, case.W,
                           case.softmax_scale)
    # unrounded fp32 inputs: the library's own rounding must match torch's
    o_f, l_f = swa.swa_attn_fwd(raw["q"], raw["k"], raw["v"], case.W, case.softmax_scale)
    g_f = swa.swa_attn_bwd(raw["q"], raw["k"], raw["v"], o_f, raw["do"], l_f, case.W,
                           case.softmax_scale)
    swa.swa_check_device()
    assert o_f.dtype == F32 and all(t.dtype == F32 for t in g_f)
    assert torch.equal(o_f, o_b.float()) and torch.equal(l_f, l_b)
    for a, b in zip(g_f, g_b):
        assert torch.equal(a, b.float())


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
