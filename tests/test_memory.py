"""GPU: device memory of one sliding-window layer's forward + backward grows linearly in N.

The lab's criterion ("Off NVIDIA, you fix the platform yourself", section "What did fixing it
take?": memory now grows about in step with length) measured as peak allocated memory above the
inputs (Q, K, V, dO) for N = 8,192, 16,384, 32,768 at 32 q / 16 kv heads, D = 128, window 1,024:
each doubling of N must scale it by 1.9x to 2.1x.  The library allocates nothing itself; the
outputs (O, LSE, dQ, dK, dV) and the Delta workspace are the only allocations.
"""
import pytest
import torch

import swa_inputs as si

pytestmark = pytest.mark.gpu


def _peak_above_inputs(swa, N):
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
                                  case.softmax_scale)
    torch.cuda.synchronize(dev)
    peak = torch.cuda.max_memory_allocated(dev) - base
    del inp, o, lse, dq, dk, dv
    return peak


def test_peak_memory_linear_in_length(swa):
    peaks = [_peak_above_inputs(swa, N) for N in (8192, 16384, 32768)]
    ratios = [peaks[i + 1] / peaks[i] for i in range(2)]
    for r in ratios:
        assert 1.9 <= r <= 2.1, (peaks, ratios)
    # O + dQ (2 x 268 MB) + dK + dV (2 x 134 MB) + LSE + Delta (2 x 4 MB) at N = 32,768
    assert peaks[-1] < 0.9e9
