"""GPU parity of queries shorter than keys (bottom-right alignment) and non-causal windows
(swa_attn_fwd_ex / swa_attn_bwd_ex through the binding) against the fp64 oracle.

Query i sits at key position i + Lk - Lq; a causal window sees keys with 0 <= pos - j < W, a
non-causal one keys with |pos - j| < W.  Bar as for the causal path: norm-wise relative error
<= 1e-2 for O, dQ, dK, dV, max |LSE difference| <= 1e-3; where the exact gradient is zero (W = 1)
the GPU norm must stay within 1e-2 of the window-2 gradient's norm.  Key blocks that no query
sees must come back exactly zero.  The pages' gradient sweep covers "queries shorter than keys"
and windows "causal and not" (Lab 28 record, numbers entry "Gradient parity, small shapes").
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


@dataclasses.dataclass(frozen=True)
class Shape:
    B: int
    Hq: int
    Hkv: int
    Lq: int
    Lk: int
    D: int
    W: int
    causal: bool
    f16: bool = False
    seed: int = 0

    def name(self):
        kind = "causal" if self.causal else "twosided"
        dt = "fp16" if self.f16 else "bf16"
        return (f"B{self.B}_Hq{self.Hq}_Hkv{self.Hkv}_Lq{self.Lq}_Lk{self.Lk}_D{self.D}_W{self.W}_"
                f"{kind}_{dt}")


SHAPES = [
    Shape(1, 2, 1, 17, 17, 64, 7, False),
    Shape(1, 2, 1, 255, 255, 128, 64, False),
    Shape(1, 4, 2, 512, 512, 64, 1, False),
    Shape(1, 2, 1, 512, 512, 128, 600, False),
    Shape(1, 2, 1, 17, 300, 64, 7, True),
    Shape(1, 2, 1, 17, 300, 64, 7, False),
    Shape(2, 4, 2, 200, 1000, 128, 100, True),
    Shape(2, 4, 2, 200, 1000, 128, 100, False),
    Shape(1, 2, 1, 128, 513, 64, 2000, True),
    Shape(1, 2, 1, 128, 513, 64, 2000, False),
    Shape(1, 2, 2, 1, 257, 128, 5, True),
    Shape(1, 2, 2, 1, 257, 128, 5, False),
    Shape(1, 2, 1, 300, 301, 64, 64, True),
    Shape(1, 2, 1, 130, 900, 128, 1, True),
    Shape(1, 4, 2, 200, 700, 128, 150, False, f16=True),
    Shape(1, 4, 2, 333, 333, 64, 40, False, f16=True),
]


def _inputs(sh: Shape):
    """Seeded draws of a length-Lk problem; the queries (and dO) are its last Lq rows."""
    case = si.Case(B=sh.B, Hq=sh.Hq, Hkv=sh.Hkv, N=sh.Lk, D=sh.D, W=sh.W, seed=sh.seed)
    dt = torch.float16 if sh.f16 else torch.bfloat16
    inp = si.make_inputs(case, dtype=dt)
    for key in ("q", "do"):
        inp[key] = inp[key][:, :, sh.Lk - sh.Lq:].contiguous()
    return inp, case.softmax_scale


def _np(t):
    return t.detach().float().cpu().double().numpy()


def _run_gpu(swa, sh, inp, scale):
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in inp.items()}
    o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], sh.W, scale, causal=sh.causal)
    dq, dk, dv = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, sh.W, scale,
                                  causal=sh.causal)
    swa.swa_check_device()
    assert o.dtype == dq.dtype == dk.dtype == dv.dtype == g["q"].dtype
    return {"o": _np(o), "lse": _np(lse), "dq": _np(dq), "dk": _np(dk), "dv": _np(dv)}


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: s.name())
def test_lq_lk_window_parity(swa, sh):
    inp, scale = _inputs(sh)
    gpu = _run_gpu(swa, sh, inp, scale)
    ref = orc.oracle_backward(inp["q"], inp["k"], inp["v"], inp["do"], sh.W, scale,
                              causal=sh.causal)
    assert np.all(np.isfinite(gpu["o"])) and np.all(np.isfinite(gpu["lse"]))
    assert _rel(gpu["o"], ref["o"]) <= REL_TOL
    assert np.max(np.abs(gpu["lse"] - ref["lse"])) <= LSE_TOL
    ref_w2 = None
    if sh.W == 1:
        ref_w2 = orc.oracle_backward(inp["q"], inp["k"], inp["v"], inp["do"], 2, scale,
                                     causal=sh.causal)
    for key in ("dq", "dk", "dv"):
        assert np.all(np.isfinite(gpu[key])), key
        if sh.W == 1 and key in ("dq", "dk"):
            bound = REL_TOL * max(np.linalg.norm(ref_w2[key]), 1e-30)
            assert np.linalg.norm(gpu[key]) <= bound, (key, np.linalg.norm(gpu[key]), bound)
        else:
            assert _rel(gpu[key], ref[key]) <= REL_TOL, (key, _rel(gpu[key], ref[key]))


@pytest.mark.parametrize("causal", [True, False])
def test_unvisited_keys_get_exact_zeros(swa, causal):
    """A short query suffix under a narrow window never sees the early keys: their dK, dV are 0."""
    sh = Shape(1, 2, 1, 40, 700, 64, 30, causal, seed=3)
    inp, scale = _inputs(sh)
    gpu = _run_gpu(swa, sh, inp, scale)
    first_seen = (sh.Lk - sh.Lq) - (sh.W - 1)  # earliest key any query sees
    assert first_seen > 2 * 128
    assert np.all(gpu["dk"][:, :, :first_seen] == 0.0)
    assert np.all(gpu["dv"][:, :, :first_seen] == 0.0)
    assert np.abs(gpu["dv"][:, :, first_seen:]).max() > 0


def test_equal_lengths_causal_match_the_plain_entry_points(swa):
    """Lq = Lk with causal=True through swa_attn_fwd_ex is bit-identical to swa_attn_fwd."""
    import ctypes

    sh = Shape(1, 4, 2, 300, 300, 128, 90, True, seed=7)
    inp, scale = _inputs(sh)
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in inp.items()}
    o1, l1 = swa.swa_attn_fwd(g["q"], g["k"], g["v"], sh.W, scale)
    o2, l2 = torch.empty_like(o1), torch.empty_like(l1)
    lib = swa.load()
    rc = lib.swa_attn_fwd_ex(g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(),
                             o2.data_ptr(), l2.data_ptr(), sh.B, sh.Hq, sh.Hkv, sh.Lq, sh.Lk,
                             sh.D, sh.W, 1, ctypes.c_float(scale), 0,
                             torch.cuda.current_stream(dev).cuda_stream)
    assert rc == 0
    swa.swa_check_device()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
