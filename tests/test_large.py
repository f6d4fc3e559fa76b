"""GPU parity at the full workload sizes, in the launch configuration bench.py times.

The dense fp64 oracle cannot evaluate every output at N = 32,768 in seconds, so it evaluates
sampled outputs one by one: O / LSE / dQ rows of sampled (head, row) pairs need only those rows'
scores; dK / dV rows of sampled keys need the full forward (LSE, O, Delta) of their kv group's query
heads, which the oracle runs densely.  Each comparison is norm-wise relative error <= 1e-2 over the
sampled values of each head (|LSE difference| <= 1e-3).  Every 128-row query tile and every
128-key tile contributes at least one sampled row or key, so an error confined to one tile is seen.
"""
import numpy as np
import pytest
import torch

import swa_inputs as si
from oracle import swa_oracle as orc

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

REL_TOL = 1e-2
LSE_TOL = 1e-3


def _rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / np.linalg.norm(np.asarray(b)))


def _np(t):
    return t.detach().float().cpu().double().numpy()


def _run(swa, case, inp, causal=True):
    dev = torch.device("cuda:0")
    g = {k: v.to(dev) for k, v in inp.items()}
    o, lse = swa.swa_attn_fwd(g["q"], g["k"], g["v"], case.W, case.softmax_scale, causal=causal)
    dq, dk, dv = swa.swa_attn_bwd(g["q"], g["k"], g["v"], o, g["do"], lse, case.W, case.softmax_scale,
                                  causal=causal)
    swa.swa_check_device()
    return {"o": o.cpu(), "lse": lse.cpu(), "dq": dq.cpu(), "dk": dk.cpu(), "dv": dv.cpu()}


def _assert_rel(what, got, ref, tol=REL_TOL):
    """Norm-wise relative error <= tol; on failure the message names the worst sampled row."""
    got, ref = np.asarray(got), np.asarray(ref)
    e = _rel(got, ref)
    if e > tol:
        rows = np.linalg.norm(got - ref, axis=-1)
        raise AssertionError(f"{what}: relative error {e:.3e} > {tol}; worst sampled row "
                             f"{int(np.argmax(rows))} (error norm {float(np.max(rows)):.3e})")


def _check_sampled(case, inp, gpu, heads, rows, kv_heads, keys, causal=True):
    """Compare sampled rows of O, LSE, dQ (query heads `heads`) and sampled keys of dK, dV, head by
    head: each head's sampled rows (keys) must meet the bar on their own."""
    q, k, v, do = inp["q"], inp["k"], inp["v"], inp["do"]
    W, sc = case.W, case.softmax_scale
    for hq in heads:
        hk = orc.kv_head_of(hq, case.Hq, case.Hkv)
        o_r, l_r = orc.forward_rows(q[0, hq], k[0, hk], v[0, hk], rows, W, sc, causal)
        _assert_rel(f"o head {hq}", _np(gpu["o"][0, hq, rows]), o_r)
        dl = np.abs(_np(gpu["lse"][0, hq, rows]) - l_r)
        assert np.max(dl) <= LSE_TOL, (f"lse head {hq}", float(np.max(dl)),
                                       int(rows[int(np.argmax(dl))]))
        dq_r = orc.dq_rows(q[0, hq], k[0, hk], v[0, hk], do[0, hq], rows, W, sc, causal)
        _assert_rel(f"dq head {hq}", _np(gpu["dq"][0, hq, rows]), dq_r)
    for hk in kv_heads:
        group = [hq for hq in range(case.Hq) if orc.kv_head_of(hq, case.Hq, case.Hkv) == hk]
        dk_r, dv_r = orc.dkdv_rows([q[0, hq] for hq in group], k[0, hk], v[0, hk],
                                   [do[0, hq] for hq in group], keys, W, sc, causal=causal)
        _assert_rel(f"dk kv head {hk}", _np(gpu["dk"][0, hk, keys]), dk_r)
        _assert_rel(f"dv kv head {hk}", _np(gpu["dv"][0, hk, keys]), dv_r)


def _sample(rng, N, n, must=()):
    """One random position inside every 128-row tile of [0, N), so that an error confined to one
    tile is sampled, plus `n` more random positions and the ones in `must`."""
    s = set(int(t + rng.integers(0, min(128, N - t))) for t in range(0, N, 128))
    s.update(int(x) for x in rng.choice(N, size=min(n, N), replace=False))
    s.update(int(m) for m in must if 0 <= m < N)
    return np.array(sorted(s))


@pytest.mark.parametrize("N", [8192, 16384, 32768])
def test_long_swa_layer(swa, N):
    case = si.long_swa_case(N)
    inp = si.make_inputs(case)
    gpu = _run(swa, case, inp)
    for key, t in gpu.items():
        assert torch.isfinite(t.float()).all(), key
    rng = np.random.default_rng(1)
    N = case.N
    # first rows (window not yet full), block boundaries, the last row
    rows = _sample(rng, N, 24, must=(0, 1, 127, 128, 1023, 1024, 1151, N - 1))
    keys = _sample(rng, N, 24, must=(0, 127, 128, N - 129, N - 128, N - 1))
    _check_sampled(case, inp, gpu, heads=[0, 1, 17, 31], rows=rows, kv_heads=[0, 15], keys=keys)


def test_gqa_full_causal_n8192_group(swa):
    """Full causal, 4 query heads per kv head: one whole kv group exactly, plus sampled rows."""
    case = si.gqa_causal_case()
    inp = si.make_inputs(case)
    gpu = _run(swa, case, inp)
    ref = orc.group_backward(inp["q"], inp["k"], inp["v"], inp["do"], 0, 3, case.W, case.softmax_scale,
                             row_block=512)
    hq = list(ref["hq"])
    for i, h in enumerate(hq):  # each query head of the group on its own
        _assert_rel(f"o head {h}", _np(gpu["o"][0, h]), ref["o"][i])
        assert np.max(np.abs(_np(gpu["lse"][0, h]) - ref["lse"][i])) <= LSE_TOL, h
        _assert_rel(f"dq head {h}", _np(gpu["dq"][0, h]), ref["dq"][i])
    _assert_rel("dk kv head 3", _np(gpu["dk"][0, 3]), ref["dk"])
    _assert_rel("dv kv head 3", _np(gpu["dv"][0, 3]), ref["dv"])
    rng = np.random.default_rng(2)
    rows = _sample(rng, case.N, 16, must=(0, case.N - 1))
    _check_sampled(case, inp, gpu, heads=[5, 30], rows=rows, kv_heads=[], keys=[])


@pytest.mark.parametrize("layer", [0, 5])
def test_mixed_step_layers_n30553(swa, layer):
    """Layers of the mixed step (N = 30,553, not a tile multiple): a sliding and a full layer."""
    case = si.mixed_layer_cases()[layer]
    inp = si.make_inputs(case)
    gpu = _run(swa, case, inp)
    rng = np.random.default_rng(3 + layer)
    N = case.N
    rows = _sample(rng, N, 16, must=(0, N - 89, N - 1))
    keys = _sample(rng, N, 16, must=(N - 89, N - 1))
    _check_sampled(case, inp, gpu, heads=[0, 31], rows=rows, kv_heads=[15], keys=keys)


def test_two_sided_window_n32768(swa):
    """The headline layer's shapes with a two-sided window (|i - j| < 1024), as bench.py times it."""
    case = si.long_swa_case(32768)
    inp = si.make_inputs(case)
    gpu = _run(swa, case, inp, causal=False)
    for key, t in gpu.items():
        assert torch.isfinite(t.float()).all(), key
    rng = np.random.default_rng(4)
    N = case.N
    rows = _sample(rng, N, 16, must=(0, 127, 128, 1023, N - 1024, N - 129, N - 1))
    keys = _sample(rng, N, 16, must=(0, 1023, 1024, N - 1025, N - 1))
    _check_sampled(case, inp, gpu, heads=[0, 31], rows=rows, kv_heads=[7], keys=keys,
                   causal=False)


def test_query_suffix_8192_of_32768(swa):
    """8,192 queries at the last key positions of a 32,768-key layer (causal, W = 1024), as bench.py
    times it: keys no query reaches get exact zeros, the rest match the oracle."""
    case = si.long_swa_case(32768)
    Lq = 8192
    inp = si.make_inputs(case)
    for key in ("q", "do"):
        inp[key] = inp[key][:, :, case.N - Lq:].contiguous()
    gpu = _run(swa, case, inp)
    assert gpu["o"].shape[2] == Lq and gpu["dk"].shape[2] == case.N
    first_seen = case.N - Lq - (case.W - 1)
    assert torch.count_nonzero(gpu["dk"][:, :, :first_seen]) == 0
    assert torch.count_nonzero(gpu["dv"][:, :, :first_seen]) == 0
    rng = np.random.default_rng(5)
    rows = _sample(rng, Lq, 16, must=(0, 127, 128, Lq - 1))
    keys = _sample(rng, case.N - first_seen, 16, must=(0, 1023, 1024, case.N - first_seen - 1))
    keys = keys + first_seen
    _check_sampled(case, inp, gpu, heads=[3, 30], rows=rows, kv_heads=[1], keys=keys)


def test_d256_layer_n32768(swa):
    """The long sliding-window layer with 256-wide heads, as bench.py times it."""
    import dataclasses

    case = dataclasses.replace(si.long_swa_case(32768), D=256)
    inp = si.make_inputs(case)
    gpu = _run(swa, case, inp)
    for key, t in gpu.items():
        assert torch.isfinite(t.float()).all(), key
    rng = np.random.default_rng(6)
    N = case.N
    rows = _sample(rng, N, 16, must=(0, 127, 128, 1023, 1024, N - 1))
    keys = _sample(rng, N, 16, must=(0, 128, N - 129, N - 1))
    _check_sampled(case, inp, gpu, heads=[0, 31], rows=rows, kv_heads=[9], keys=keys)


def test_d64_layer_n32768(swa):
    """The long sliding-window layer with 64-wide heads, as bench.py times it."""
    import dataclasses

    case = dataclasses.replace(si.long_swa_case(32768), D=64)
    inp = si.make_inputs(case)
    gpu = _run(swa, case, inp)
    for key, t in gpu.items():
        assert torch.isfinite(t.float()).all(), key
    rng = np.random.default_rng(7)
    N = case.N
    rows = _sample(rng, N, 16, must=(0, 127, 128, 1023, 1024, N - 1))
    keys = _sample(rng, N, 16, must=(0, 128, N - 129, N - 1))
    _check_sampled(case, inp, gpu, heads=[1, 30], rows=rows, kv_heads=[4], keys=keys)
