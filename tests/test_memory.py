"""GPU: device memory of one sliding-window layer's forward + backward grows linearly in N.

The lab's criterion ("Off NVIDIA, you fix the platform yourself", section "What did fixing it
take?": memory now grows about in step with length) measured as peak allocated memory above the
inputs (Q, K, V, dO) for N = 8,192, 16,384, 32,768 at 32 q / 16 kv heads, D = 128, window 1,024:
each doubling of N must scale it by 1.9x to 2.1x, on both backward paths.  The library allocates
nothing itself; the outputs (O, LSE, dQ, dK, dV) and the workspace (Delta, and on the fused path the
fp32 dQ accumulator) are the only allocations.
"""
import pytest
import torch

import swa_inputs as si

pytestmark = pytest.mark.gpu


def _peak_above_inputs(swa, N, fused):
    dev = torch.device("cuda:0")
    case = si.long_swa_case(N)
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    inp = si.make_inputs(case, device="cuda:0")
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    o, lse = swa.swa_attn_fwd(inp["q"], inp["k"], inp["v"], case.W, case.softmax_scale)
    dq, dk, dv = swa.swa_attn_bwd(inp["q"], inp["k"], inp["v"], o, inp["do"], lse, case.W,
                                  case.softmax_scale, fused=fused)
    torch.cuda.synchronize(dev)
    peak = torch.cuda.max_memory_allocated(dev) - base
    del inp, o, lse, dq, dk, dv
    return peak


@pytest.mark.parametrize("fused,bound", [(False, 0.9e9), (True, 1.4e9)], ids=["split", "fused"])
def test_peak_memory_linear_in_length(swa, fused, bound):
    peaks = [_peak_above_inputs(swa, N, fused) for N in (8192, 16384, 32768)]
    ratios = [peaks[i + 1] / peaks[i] for i in range(2)]
    for r in ratios:
        assert 1.9 <= r <= 2.1, (peaks, ratios)
    # at N = 32,768: O + dQ (2 x 268 MB) + dK + dV (2 x 134 MB) + LSE + Delta (2 x 4 MB); the fused
    # path adds the fp32 dQ accumulator (537 MB)
    assert peaks[-1] < bound, peaks
