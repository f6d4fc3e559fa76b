"""GPU parity of the dK/dV kernel's shortest query walks against the fp64 oracle.

A key block's CTA walks T = G x (query blocks that see it) tiles.  The MMA warp issues the next
tile's S^T at the top of each step, so T = 1 (no next tile at all), T = 2 and T = 3 are the edge
cases of that schedule; a longer walk (T = 6) is the steady state.  Each case is chosen so that
the walk length of every key block is known:
  - G = 1, W = 1: every key block is seen only by its own query block (T = 1);
  - G = 2, W = 1: T = 2; G = 3, W = 1: T = 3; G = 1, W = 64: T = 2 (interior) and 1 (last);
  - G = 3, W = 64 over several blocks: interior key blocks are seen by two query blocks (T = 6)
    and the last one by one (T = 3).
Same bar as the other parity tests (norm-wise relative error <= 1e-2, |LSE difference| <= 1e-3;
zero exact gradients at W = 1 checked against the window-2 gradient's norm).
"""
import pytest

import swa_inputs as si
from oracle import swa_oracle as orc
from test_parity import check_against_oracle, run_gpu

CASES = [
    si.Case(B=1, Hq=1, Hkv=1, N=384, D=128, W=1, seed=21),
    si.Case(B=1, Hq=2, Hkv=1, N=300, D=128, W=1, seed=22),
    si.Case(B=2, Hq=3, Hkv=1, N=256, D=128, W=1, seed=23),
    si.Case(B=1, Hq=3, Hkv=1, N=640, D=128, W=64, seed=24),
    si.Case(B=1, Hq=2, Hkv=2, N=400, D=128, W=64, seed=27),
    si.Case(B=1, Hq=1, Hkv=1, N=200, D=64, W=1, seed=25),
    si.Case(B=1, Hq=6, Hkv=2, N=520, D=64, W=64, seed=26),
]


def walk_length(case: si.Case, key_block: int) -> int:
    """Tiles the dK/dV CTA of `key_block` walks: G x the query blocks that see any of its keys."""
    G = case.Hq // case.Hkv
    k0, k1 = 128 * key_block, min(128 * key_block + 127, case.N - 1)
    q_lo, q_hi = k0 // 128, min(k1 + case.W - 1, case.N - 1) // 128
    return G * (q_hi - q_lo + 1)


def test_walk_length_matches_brute_force():
    """walk_length agrees with counting, over the oracle's own visibility predicate, the query
    blocks holding at least one query that sees a key of the block."""
    import numpy as np
    for case in CASES:
        i = np.arange(case.N)[:, None]
        j = np.arange(case.N)[None, :]
        vis = orc.visible(i, j, case.W)
        for kb in range((case.N + 127) // 128):
            seen = vis[:, 128 * kb:128 * (kb + 1)].any(axis=1)
            qblocks = {q // 128 for q in np.nonzero(seen)[0]}
            assert walk_length(case, kb) == (case.Hq // case.Hkv) * len(qblocks), (case, kb)


def test_walk_lengths_cover_the_edge_cases():
    """The cases above reach walks of 1, 2, 3 and 6 tiles (a host-side check of the case list)."""
    lengths = {walk_length(c, kb) for c in CASES for kb in range((c.N + 127) // 128)}
    assert {1, 2, 3, 6} <= lengths


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name())
def test_short_walks_match_oracle(swa, case):
    inputs = si.make_inputs(case)
    gpu = run_gpu(swa, case, inputs)
    ref = orc.oracle_backward(inputs["q"], inputs["k"], inputs["v"], inputs["do"], case.W,
                              case.softmax_scale)
    ref_w2 = None
    if case.W == 1:
        ref_w2 = orc.oracle_backward(inputs["q"], inputs["k"], inputs["v"], inputs["do"], 2,
                                     case.softmax_scale)
    check_against_oracle(case, gpu, ref, ref_w2)
