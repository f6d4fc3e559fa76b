"""GPU: the entry points work inside CUDA graph capture (tensor maps are built on the host and
passed by value, so a captured launch replays with the same buffers).  A captured forward +
backward, replayed on new data written into the same input buffers, equals eager calls bit for
bit; likewise the fp32 entry points and the Lq < Lk / two-sided forms.  The fused backward is
captured too: its dK and dV replay bit for bit, its dQ (fp32 partials added in a varying order) to
within a few bf16 units."""
import pytest
import torch

import swa_inputs as si

pytestmark = pytest.mark.gpu


def _eager(swa, g, W, scale, causal, fused=False):
    o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], W, scale, causal=causal)
    dq, dk, dv = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, W, scale,
                                  causal=causal, fused=fused)
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("dtype,Lq,Lk,W,causal,fused", [
    (torch.bfloat16, 700, 700, 200, True, False),
    (torch.float16, 300, 900, 64, False, False),
    (torch.float32, 256, 256, 64, True, False),
    (torch.bfloat16, 700, 700, 200, True, True),
    (torch.float16, 300, 900, 64, False, True),
])
def test_captured_fwd_bwd_replays_exactly(swa, dtype, Lq, Lk, W, causal, fused):
    dev = torch.device("cuda:0")
    case = si.Case(B=1, Hq=4, Hkv=2, N=Lk, D=128, W=W, seed=30)
    sc = case.softmax_scale

    def inputs(seed):
        c = si.Case(B=1, Hq=4, Hkv=2, N=Lk, D=128, W=W, seed=seed)
        x = si.make_inputs(c, dtype=dtype)
        for key in ("q", "do"):
            x[key] = x[key][:, :, Lk - Lq:].contiguous()
        return {k: v.to(dev) for k, v in x.items()}

    g = inputs(30)
    static = {k: v.clone() for k, v in g.items()}
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):  # warm up outside the graph (kernel attributes, allocations)
        _eager(swa, static, W, sc, causal, fused)
    torch.cuda.current_stream(dev).wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        outs = _eager(swa, static, W, sc, causal, fused)
    for seed in (31, 32):
        fresh = inputs(seed)
        for k in static:
            static[k].copy_(fresh[k])
        graph.replay()
        torch.cuda.synchronize(dev)
        swa.swa_check_device()
        ref = _eager(swa, fresh, W, sc, causal, fused)
        torch.cuda.synchronize(dev)
        for i, (a, b) in enumerate(zip(outs, ref)):
            if fused and i == 2:  # dQ of the fused backward
                rel = (torch.linalg.vector_norm(a.float() - b.float()) /
                       torch.linalg.vector_norm(b.float())).item()
                assert rel <= 2e-3, rel
            else:
                assert torch.equal(a, b)
