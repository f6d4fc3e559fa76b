"""GPU parity of the fp16 entry points (swa_attn_fwd_f16 / swa_attn_bwd_f16) against the fp64
oracle on the same seeded inputs rounded to fp16.  Same bar as the bf16 path: norm-wise relative
error <= 1e-2 for O, dQ, dK, dV and max |LSE difference| <= 1e-3; zero-gradient cases (window 1)
are bounded by 1e-2 of the window-2 gradient.  The pages' gradient sweep covers fp16 as well as
bf16 inputs (Lab 28 record, numbers entry "Gradient parity, small shapes").
"""
import numpy as np
import pytest
import torch

import swa_inputs as si
from oracle import swa_oracle as orc
from test_parity import check_against_oracle, run_gpu

pytestmark = pytest.mark.gpu

F16 = torch.float16


def _case_id(c):
    return c.name()


def _fp16_cases():
    """A cross-section of the edge sweep (ragged lengths, both head dims, windows 1 / 7 / 64 / N)
    plus a multi-tile grouped-query case."""
    cases = [c for c in si.edge_cases() if c.N in (17, 255, 512)]
    cases.append(si.Case(B=1, Hq=4, Hkv=2, N=1000, D=128, W=300, seed=5))
    return cases


def _oracle(case, inputs, W=None):
    return orc.oracle_backward(inputs["q"], inputs["k"], inputs["v"], inputs["do"],
                               case.W if W is None else W, case.softmax_scale)


def test_tiny_fp16(swa):
    case = si.tiny_case()
    inputs = si.make_inputs(case, dtype=F16)
    gpu = run_gpu(swa, case, inputs)
    check_against_oracle(case, gpu, _oracle(case, inputs))


@pytest.mark.parametrize("case", _fp16_cases(), ids=_case_id)
def test_fp16_sweep(swa, case):
    inputs = si.make_inputs(case, dtype=F16)
    gpu = run_gpu(swa, case, inputs)
    ref = _oracle(case, inputs)
    ref_w2 = _oracle(case, inputs, W=2) if case.W == 1 else None
    check_against_oracle(case, gpu, ref, ref_w2)


def test_fp16_outputs_keep_dtype(swa):
    case = si.tiny_case()
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in si.make_inputs(case, dtype=F16).items()}
    o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], case.W, case.softmax_scale)
    dq, dk, dv = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, case.W,
                                  case.softmax_scale)
    swa.swa_check_device()
    assert o.dtype == dq.dtype == dk.dtype == dv.dtype == F16 and lse.dtype == torch.float32


def test_fp16_and_bf16_agree_on_shared_values(swa):
    """Inputs exactly representable in both types (8 significant bits, small exponents) give the
    same forward up to the two types' output rounding."""
    case = si.Case(B=1, Hq=2, Hkv=1, N=300, D=64, W=100, seed=3)
    # bf16 values, flushed to zero below fp16's normal range: the rest are exact in fp16 too.
    raw = {k: torch.where(v.abs() < 2.0 ** -14, torch.zeros_like(v), v)
           for k, v in si.make_inputs(case).items()}
    dev = torch.device("cuda:0")
    bf = {k: v.to(dev) for k, v in raw.items()}
    hf = {k: v.to(F16).to(dev) for k, v in raw.items()}
    assert all(torch.equal(bf[k].float(), hf[k].float()) for k in bf)
    o_b, l_b = swa.swa_attn_fwd(bf["q"], bf["k"], bf["v"], case.W, case.softmax_scale)
    o_h, l_h = swa.swa_attn_fwd(hf["q"], hf["k"], hf["v"], case.W, case.softmax_scale)
    swa.swa_check_device()
    # LSE is computed in fp32 from identical operands; O differs by P's rounding (bf16 vs fp16).
    assert torch.max(torch.abs(l_b - l_h)).item() <= 1e-3
    rel = (torch.linalg.norm(o_b.float() - o_h.float()) / torch.linalg.norm(o_h.float())).item()
    assert rel <= 1e-2


def test_fp16_rejects_mixed_dtypes(swa):
    case = si.tiny_case()
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in si.make_inputs(case, dtype=F16).items()}
    with pytest.raises(TypeError):
        swa.swa_attn_fwd(g["q"], g["k"].to(torch.bfloat16), g["v"], case.W)
