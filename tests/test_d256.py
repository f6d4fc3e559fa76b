"""GPU parity of head dimension 256 (Gemma 4's sliding layers; "Off NVIDIA, you fix the platform
yourself", Lab 28 record, numbers entry "Attention backward memory") against the fp64 oracle.

Same bar as the other head dims: norm-wise relative error <= 1e-2 for O, dQ, dK, dV and max |LSE
difference| <= 1e-3; where the exact gradient is zero (W = 1) the GPU norm must stay within 1e-2
of the window-2 gradient's norm.  The cases cover ragged lengths, windows 1 / 7 / 64 / N, grouped
heads, more query tiles than SMs (so a persistent CTA runs several tiles), queries shorter than
keys, two-sided windows, fp16 and fp32 tensors, and key blocks no query sees.
"""
import dataclasses

import numpy as np
import pytest
import torch

import swa_inputs as si
from oracle import swa_oracle as orc

pytestmark = pytest.mark.gpu

REL_TOL = 1e-2
LSE_TOL = 1e-3
U_BF16 = 2.0 ** -8


@dataclasses.dataclass(frozen=True)
class Shape:
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lk: int
    W: int
    causal: bool = True
    dtype: str = "bf16"
    seed: int = 0

    def name(self):
        kind = "causal" if self.causal else "twosided"
        return (f"B{self.B}_Hq{self.Hq}_Hkv{self.Hkv}_Lq{self.Lq}_Lk{self.Lk}_W{self.W}_{kind}_"
                f"{self.dtype}")


SHAPES = [
    Shape(1, 2, 1, 256, 256, 64),
    Shape(1, 2, 1, 17, 17, 7),
    Shape(2, 4, 2, 255, 255, 1),
    Shape(2, 4, 2, 300, 300, 300),
    Shape(1, 4, 1, 513, 513, 100),
    Shape(1, 4, 2, 700, 700, 200, causal=False),
    Shape(1, 2, 1, 200, 1000, 150),
    Shape(1, 2, 1, 130, 900, 64, causal=False),
    Shape(1, 2, 2, 1, 257, 5),
    Shape(1, 4, 2, 333, 333, 40, dtype="fp16"),
    Shape(1, 4, 2, 400, 600, 90, causal=False, dtype="fp16"),
    Shape(1, 2, 1, 300, 300, 64, dtype="fp32"),
    Shape(1, 2, 1, 150, 500, 64, causal=False, dtype="fp32"),
]

_DT = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


def _inputs(sh: Shape):
    case = si.Case(B=sh.B, Hq=sh.Hq, Hkv=sh.Hkv, N=sh.Lk, D=256, W=sh.W, seed=sh.seed)
    inp = si.make_inputs(case, dtype=_DT[sh.dtype])
    for key in ("q", "do"):
        inp[key] = inp[key][:, :, sh.Lk - sh.Lq:].contiguous()
    return inp, case.softmax_scale


def _run(swa, sh, inp, scale):
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in inp.items()}
    o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], sh.W, scale, causal=sh.causal)
    dq, dk, dv = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, sh.W, scale,
                                  causal=sh.causal)
    swa.swa_check_device()
    assert o.dtype == dq.dtype == dk.dtype == dv.dtype == g["q"].dtype
    return {k: v.detach().double().cpu().numpy()
            for k, v in {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}.items()}


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _check(gpu, ref, ref_w2, W, lse_bound=LSE_TOL):
    for key in gpu:
        assert np.all(np.isfinite(gpu[key])), key
    assert _rel(gpu["o"], ref["o"]) <= REL_TOL, _rel(gpu["o"], ref["o"])
    assert np.all(np.abs(gpu["lse"] - ref["lse"]) <= lse_bound)
    for key in ("dq", "dk", "dv"):
        if W == 1 and key in ("dq", "dk"):
            bound = REL_TOL * np.linalg.norm(ref_w2[key])
            assert np.linalg.norm(gpu[key]) <= bound, (key, np.linalg.norm(gpu[key]), bound)
        else:
            assert _rel(gpu[key], ref[key]) <= REL_TOL, (key, _rel(gpu[key], ref[key]))


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: s.name())
def test_d256_parity(swa, sh):
    inp, scale = _inputs(sh)
    gpu = _run(swa, sh, inp, scale)
    # fp32 tensors are checked against the oracle on the same unrounded fp32 values (the fp32
    # calls correct their log-sum-exp for the bf16 rounding of q and k)
    ref_in = inp
    ref = orc.oracle_backward(ref_in["q"], ref_in["k"], ref_in["v"], ref_in["do"], sh.W, scale,
                              causal=sh.causal)
    ref_w2 = None
    if sh.W == 1:
        ref_w2 = orc.oracle_backward(ref_in["q"], ref_in["k"], ref_in["v"], ref_in["do"], 2,
                                     scale, causal=sh.causal)
    _check(gpu, ref, ref_w2, sh.W)


def test_d256_more_tiles_than_sms(swa):
    """176 query tiles (B 2, Hq 8, 11 blocks) over at most 152 persistent CTAs: several CTAs run
    two tiles, so the Q reload, O / dQ hand-over and ring counters cross a tile boundary."""
    sh = Shape(2, 8, 4, 1300, 1300, 200, seed=4)
    inp, scale = _inputs(sh)
    gpu = _run(swa, sh, inp, scale)
    ref = orc.oracle_backward(inp["q"], inp["k"], inp["v"], inp["do"], sh.W, scale)
    _check(gpu, ref, None, sh.W)


@pytest.mark.parametrize("causal", [True, False])
def test_d256_unvisited_keys_get_exact_zeros(swa, causal):
    sh = Shape(1, 2, 1, 40, 700, 30, causal=causal, seed=3)
    inp, scale = _inputs(sh)
    gpu = _run(swa, sh, inp, scale)
    first_seen = (sh.Lk - sh.Lq) - (sh.W - 1)
    assert first_seen > 2 * 128
    assert np.all(gpu["dk"][:, :, :first_seen] == 0.0)
    assert np.all(gpu["dv"][:, :, :first_seen] == 0.0)
    assert np.abs(gpu["dv"][:, :, first_seen:]).max() > 0


@pytest.mark.parametrize("causal", [True, False])
def test_d256_key_block_pair_half_unvisited(swa, causal):
    """dK and dV run on CTA pairs over neighbouring key blocks, which walk the union of the two
    blocks' query blocks.  Here no query sees keys below 700, so of the pair (512..639, 640..767)
    the first block is unvisited while the second is partly visited: the first must come out as
    exact zeros and the second match the oracle."""
    sh = Shape(1, 2, 1, 100, 1000, 201, causal=causal, seed=6)
    inp, scale = _inputs(sh)
    gpu = _run(swa, sh, inp, scale)
    first_seen = (sh.Lk - sh.Lq) - (sh.W - 1)
    assert first_seen == 700 and 640 <= first_seen < 768  # inside key block 5, block 4 unseen
    assert np.all(gpu["dk"][:, :, :first_seen] == 0.0)
    assert np.all(gpu["dv"][:, :, :first_seen] == 0.0)
    ref = orc.oracle_backward(inp["q"], inp["k"], inp["v"], inp["do"], sh.W, scale,
                              causal=sh.causal)
    _check(gpu, ref, None, sh.W)


def test_d256_autograd(swa):
    """The autograd wrapper at D = 256 matches the explicit calls."""
    sh = Shape(1, 2, 1, 256, 256, 64, seed=5)
    inp, scale = _inputs(sh)
    dev = torch.device("cuda:0")
    q, k, v = (inp[n].to(dev).requires_grad_(True) for n in ("q", "k", "v"))
    o = swa.SlidingWindowAttention.apply(q, k, v, sh.W, scale)
    o.backward(inp["do"].to(dev))
    swa.swa_check_device()
    ref = _run(swa, sh, inp, scale)
    assert np.array_equal(o.detach().double().cpu().numpy(), ref["o"])
    assert np.array_equal(q.grad.double().cpu().numpy(), ref["dq"])
    assert np.array_equal(k.grad.double().cpu().numpy(), ref["dk"])
