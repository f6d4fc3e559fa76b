"""CPU pins for the fp64 oracle: each test checks it against something other than itself.

Pins (what they fix and why a plausible mistake fails one of them):
  * window >= N  ->  torch's causal scaled_dot_product_attention + autograd (a library routine).
  * general W    ->  torch SDPA with a boolean band mask built by a different route (tril minus
                     tril), again with autograd for the gradients.
  * W = 1        ->  closed form: O = V row, LSE = scale <q_i, k_i>, dV = group sum of dO, dQ = dK = 0
                     (the lab states the exact gradient vanishes at window 1).
  * finite differences of L = sum(dO * O) on tiny shapes.
  * brute force with Python loops on N <= 8.
  * structural invariants: softmax rows sum to 1, sum_j dS[i, j] = 0, dK/dV support in [i-W+1, i].
  * planted mistakes: an off-by-one window, a wrong GQA mapping, a dropped Delta, a transposed dS
    are each caught by the pins above.
  * queries shorter than keys and non-causal windows: torch SDPA without a mask (non-causal, full
    window) and with triu / tril-built masks (bottom-right causal band, two-sided band); the
    short-query problem equals the suffix of the full-length one whose extra rows carry dO = 0;
    reversal symmetry of the two-sided window; finite differences; brute-force loops; planted
    top-left alignment and one-sided "non-causal" windows are rejected.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import swa_oracle as orc


def _rand(shape, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape)


def _torch_reference(q, k, v, do, W, scale, use_is_causal=False):
    """torch SDPA on float64 CPU, grouped heads expanded with repeat_interleave, autograd backward."""
    G = q.shape[1] // k.shape[1]
    N = q.shape[2]
    tq = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    ke = tk.repeat_interleave(G, dim=1)
    ve = tv.repeat_interleave(G, dim=1)
    if use_is_causal:
        o = F.scaled_dot_product_attention(tq, ke, ve, is_causal=True, scale=scale)
    else:
        ones = torch.ones(N, N, dtype=torch.float64)
        band = (torch.tril(ones) - torch.tril(ones, diagonal=-W)) > 0.5
        o = F.scaled_dot_product_attention(tq, ke, ve, attn_mask=band, scale=scale)
    (o * torch.tensor(do)).sum().backward()
    return {"o": o.detach().numpy(), "dq": tq.grad.numpy(), "dk": tk.grad.numpy(), "dv": tv.grad.numpy()}


def _rel(a, b):
    """Norm-wise relative difference; an all-zero reference (N = 1 or W = 1 gradients) is
    compared absolutely, against unit scale."""
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1.0)


SHAPES = [
    # B, Hq, Hkv, N, D
    (1, 1, 1, 1, 8),
    (1, 2, 1, 5, 8),
    (2, 4, 2, 33, 16),
    (1, 4, 1, 70, 8),
    (1, 3, 3, 19, 4),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_full_window_is_plain_causal(shape):
    B, Hq, Hkv, N, D = shape
    q, k, v, do = (_rand((B, h, N, D), s) for h, s in ((Hq, 1), (Hkv, 2), (Hkv, 3), (Hq, 4)))
    scale = 1.0 / math.sqrt(D)
    ref = _torch_reference(q, k, v, do, N, scale, use_is_causal=True)
    for W in (N, N + 1, 10 * N + 7):
        out = orc.oracle_backward(q, k, v, do, W, scale)
        for key in ("o", "dq", "dk", "dv"):
            assert _rel(out[key], ref[key]) < 1e-12, (key, W)


@pytest.mark.parametrize("shape", SHAPES[1:])
@pytest.mark.parametrize("W", [1, 2, 3, 7])
def test_band_mask_matches_library_sdpa(shape, W):
    B, Hq, Hkv, N, D = shape
    q, k, v, do = (_rand((B, h, N, D), 10 + s) for h, s in ((Hq, 1), (Hkv, 2), (Hkv, 3), (Hq, 4)))
    scale = 0.37
    ref = _torch_reference(q, k, v, do, W, scale)
    out = orc.oracle_backward(q, k, v, do, W, scale, row_block=7)
    for key in ("o", "dq", "dk", "dv"):
        assert _rel(out[key], ref[key]) < 1e-12, key


def test_lse_matches_library_logsumexp():
    N, D, W = 40, 8, 9
    q, k = _rand((N, D), 5), _rand((N, D), 6)
    scale = 0.5
    _, lse = orc.head_forward(q, k, _rand((N, D), 7), W, scale)
    s = torch.tensor(scale * q @ k.T)
    i = torch.arange(N)[:, None]
    j = torch.arange(N)[None, :]
    s = s.masked_fill(~((j <= i) & (j > i - W)), float("-inf"))
    assert np.max(np.abs(lse - torch.logsumexp(s, dim=1).numpy())) < 1e-12


@pytest.mark.parametrize("G", [1, 2, 4])
def test_window_one_closed_form(G):
    B, Hkv, N, D = 2, 2, 23, 8
    Hq = G * Hkv
    q, k, v, do = (_rand((B, h, N, D), 20 + s) for h, s in ((Hq, 1), (Hkv, 2), (Hkv, 3), (Hq, 4)))
    scale = 0.25
    out = orc.oracle_backward(q, k, v, do, 1, scale)
    for b in range(B):
        for hq in range(Hq):
            hk = hq // G
            assert np.array_equal(out["o"][b, hq], v[b, hk])
            assert np.allclose(out["lse"][b, hq], scale * np.sum(q[b, hq] * k[b, hk], axis=1), atol=1e-13)
            assert np.max(np.abs(out["dq"][b, hq])) <= 1e-12
        assert np.max(np.abs(out["dk"][b])) <= 1e-12
        for hk in range(Hkv):
            assert np.allclose(out["dv"][b, hk], do[b, hk * G:(hk + 1) * G].sum(axis=0), atol=1e-13)


@pytest.mark.parametrize("G,W", [(1, 1), (1, 2), (2, 3), (2, 12), (1, 5)])
def test_finite_differences(G, W):
    B, Hkv, N, D = 1, 1, 12, 4
    Hq = G * Hkv
    q, k, v, do = (_rand((B, h, N, D), 40 + s) for h, s in ((Hq, 1), (Hkv, 2), (Hkv, 3), (Hq, 4)))
    scale = 0.6
    out = orc.oracle_backward(q, k, v, do, W, scale)
    h = 1e-6

    def loss(qq, kk, vv):
        o, _ = orc.oracle_forward(qq, kk, vv, W, scale)
        return float(np.sum(do * o))

    for name, arr, grad in (("q", q, out["dq"]), ("k", k, out["dk"]), ("v", v, out["dv"])):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = arr.copy(), arr.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (loss(args_p["q"], args_p["k"], args_p["v"])
                       - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        scale_ref = max(np.linalg.norm(fd), 1e-3)
        assert np.linalg.norm(fd - grad) / scale_ref < 1e-6, name


def _brute_force_forward(q, k, v, W, scale):
    """Triple loop with math.exp: no NumPy vector ops."""
    N, D = len(q), len(q[0])
    o = [[0.0] * len(v[0]) for _ in range(N)]
    lse = [0.0] * N
    for i in range(N):
        scores = []
        for j in range(N):
            if 0 <= i - j < W:
                scores.append((j, scale * sum(q[i][d] * k[j][d] for d in range(D))))
        m = max(s for _, s in scores)
        z = sum(math.exp(s - m) for _, s in scores)
        lse[i] = m + math.log(z)
        for j, s in scores:
            p = math.exp(s - lse[i])
            for d in range(len(v[0])):
                o[i][d] += p * v[j][d]
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("N,W", [(1, 1), (4, 2), (8, 3), (8, 8), (7, 100)])
def test_brute_force_loops(N, W):
    D = 3
    q, k, v = _rand((N, D), 60), _rand((N, D), 61), _rand((N, D), 62)
    o, lse = orc.head_forward(q, k, v, W, 0.9)
    o2, lse2 = _brute_force_forward(q.tolist(), k.tolist(), v.tolist(), W, 0.9)
    assert np.max(np.abs(o - o2)) < 1e-12
    assert np.max(np.abs(lse - lse2)) < 1e-12


def test_invariants():
    N, D, W = 30, 6, 5
    q, k, v, do = _rand((N, D), 70), _rand((N, D), 71), _rand((N, D), 72), _rand((N, D), 73)
    scale = 0.4
    p = orc.probabilities(q, k, W, scale)
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-14)
    i, j = np.meshgrid(np.arange(N), np.arange(N), indexing="ij")
    assert np.all(p[~((i - j >= 0) & (i - j < W))] == 0.0)
    # sum_j dS[i, j] = 0: dS = P * (dP - Delta) with Delta the row's <dO, O>.
    r = orc.head_backward(q, k, v, do, W, scale)
    dp = do @ v.T
    ds = p * (dp - r["delta"][:, None])
    assert np.max(np.abs(ds.sum(axis=1))) < 1e-12
    # dK/dV support: a single nonzero dO row i0 reaches keys i0-W+1 .. i0 only.
    i0 = 17
    do1 = np.zeros_like(do)
    do1[i0] = do[i0]
    r1 = orc.head_backward(q, k, v, do1, W, scale)
    support = np.nonzero(np.abs(r1["dv"]).sum(axis=1) > 0)[0]
    assert support.min() == i0 - W + 1 and support.max() == i0
    assert np.all(np.abs(r1["dk"][: i0 - W + 1]) == 0) and np.all(np.abs(r1["dk"][i0 + 1:]) == 0)


def test_sampled_rows_agree_with_dense():
    B, Hq, Hkv, N, D, W = 1, 4, 2, 50, 8, 9
    q, k, v, do = (_rand((B, h, N, D), 80 + s) for h, s in ((Hq, 1), (Hkv, 2), (Hkv, 3), (Hq, 4)))
    scale = 0.3
    full = orc.oracle_backward(q, k, v, do, W, scale)
    rows = [0, 3, 8, 9, 49]
    o_r, lse_r = orc.forward_rows(q[0, 3], k[0, 1], v[0, 1], rows, W, scale)
    assert np.allclose(o_r, full["o"][0, 3, rows], atol=1e-13)
    assert np.allclose(lse_r, full["lse"][0, 3, rows], atol=1e-13)
    dq_r = orc.dq_rows(q[0, 2], k[0, 1], v[0, 1], do[0, 2], rows, W, scale)
    assert np.allclose(dq_r, full["dq"][0, 2, rows], atol=1e-13)
    dk_r, dv_r = orc.dkdv_rows([q[0, 2], q[0, 3]], k[0, 1], v[0, 1], [do[0, 2], do[0, 3]], rows, W, scale)
    assert np.allclose(dk_r, full["dk"][0, 1, rows], atol=1e-13)
    assert np.allclose(dv_r, full["dv"][0, 1, rows], atol=1e-13)


# ---------------------------------------------------------------------------------------------
# Planted mistakes: each variant of the oracle below is wrong in one plausible way, and at least
# one pin must reject it.  The plant goes into the oracle module, on the CPU.
# ---------------------------------------------------------------------------------------------

def _pins_pass():
    """Run the library-SDPA and W=1 pins on one GQA case; True iff all agree."""
    B, Hq, Hkv, N, D, W = 1, 4, 2, 21, 8, 5
    q, k, v, do = (_rand((B, h, N, D), 90 + s) for h, s in ((Hq, 1), (Hkv, 2), (Hkv, 3), (Hq, 4)))
    scale = 0.45
    ref = _torch_reference(q, k, v, do, W, scale)
    out = orc.oracle_backward(q, k, v, do, W, scale)
    ok = all(_rel(out[key], ref[key]) < 1e-12 for key in ("o", "dq", "dk", "dv"))
    out1 = orc.oracle_backward(q, k, v, do, 1, scale)
    ok = ok and np.max(np.abs(out1["dq"])) <= 1e-12 and np.max(np.abs(out1["dk"])) <= 1e-12
    return ok


def test_pins_accept_the_oracle():
    assert _pins_pass()


def test_pins_reject_off_by_one_window(monkeypatch):
    monkeypatch.setattr(orc, "visible",
                        lambda i, j, W, off=0, causal=True: ((i + off - j) >= 0) & ((i + off - j) <= W))
    assert not _pins_pass()


def test_pins_reject_window_excluding_self(monkeypatch):
    monkeypatch.setattr(orc, "visible",
                        lambda i, j, W, off=0, causal=True: ((i + off - j) > 0) & ((i + off - j) <= W)
                        | ((i + off == 0) & (j == 0)))
    assert not _pins_pass()


def test_pins_reject_strided_gqa_mapping(monkeypatch):
    monkeypatch.setattr(orc, "kv_head_of", lambda hq, Hq, Hkv: hq % Hkv)
    assert not _pins_pass()


def test_pins_reject_dropped_delta(monkeypatch):
    real = orc.head_backward

    def no_delta(qh, kh, vh, doh, W, scale, row_block=1024, causal=True):
        r = real(qh, kh, vh, np.asarray(doh), W, scale, row_block, causal)
        # Recompute dQ/dK as if Delta were zero.
        p = orc.probabilities(qh, kh, W, scale)
        ds = p * (np.asarray(doh) @ np.asarray(vh).T)
        r["dq"] = scale * ds @ np.asarray(kh)
        r["dk"] = scale * ds.T @ np.asarray(qh)
        return r

    monkeypatch.setattr(orc, "head_backward", no_delta)
    assert not _pins_pass()


def test_pins_reject_transposed_ds(monkeypatch):
    real = orc.head_backward

    def transposed(qh, kh, vh, doh, W, scale, row_block=1024, causal=True):
        r = real(qh, kh, vh, doh, W, scale, row_block, causal)
        p = orc.probabilities(qh, kh, W, scale)
        ds = p * (np.asarray(doh) @ np.asarray(vh).T - r["delta"][:, None])
        r["dk"] = scale * ds @ np.asarray(qh)  # should be ds.T @ q
        return r

    monkeypatch.setattr(orc, "head_backward", transposed)
    assert not _pins_pass()


def test_golden_fixture_reproduces():
    """tests/golden/oracle_tiny.json was written by tests/golden/make_golden.py from the oracle."""
    import json
    import os

    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_tiny.json")
    rec = json.load(open(path))
    inp = {k: np.array(v) for k, v in rec["inputs"].items()}
    out = orc.oracle_backward(inp["q"], inp["k"], inp["v"], inp["do"], rec["window"], rec["scale"])
    for key, val in rec["outputs"].items():
        assert np.max(np.abs(out[key] - np.array(val))) < 1e-12, key


# ---------------------------------------------------------------------------------------------
# Queries shorter than keys (bottom-right alignment: query i at key position i + Lk - Lq) and
# non-causal windows (|pos(i) - j| < W).
# ---------------------------------------------------------------------------------------------

def _torch_masked(q, k, v, do, mask, scale):
    """torch SDPA (float64, CPU) with an explicit boolean mask [Lq, Lk] and autograd gradients."""
    G = q.shape[1] // k.shape[1]
    tq = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    o = F.scaled_dot_product_attention(tq, tk.repeat_interleave(G, dim=1),
                                       tv.repeat_interleave(G, dim=1), attn_mask=mask, scale=scale)
    (o * torch.tensor(do)).sum().backward()
    return {"o": o.detach().numpy(), "dq": tq.grad.numpy(), "dk": tk.grad.numpy(), "dv": tv.grad.numpy()}


def _lq_lk_inputs(B, Hq, Hkv, Lq, Lk, D, seed):
    return (_rand((B, Hq, Lq, D), seed + 1), _rand((B, Hkv, Lk, D), seed + 2),
            _rand((B, Hkv, Lk, D), seed + 3), _rand((B, Hq, Lq, D), seed + 4))


@pytest.mark.parametrize("shape", [(1, 2, 1, 9, 8), (2, 4, 2, 33, 16), (1, 3, 3, 1, 4)])
def test_noncausal_full_window_is_plain_sdpa(shape):
    B, Hq, Hkv, N, D = shape
    q, k, v, do = _lq_lk_inputs(B, Hq, Hkv, N, N, D, 100)
    scale = 1.0 / math.sqrt(D)
    G = Hq // Hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    o = F.scaled_dot_product_attention(tq, tk.repeat_interleave(G, dim=1),
                                       tv.repeat_interleave(G, dim=1), scale=scale)
    (o * torch.tensor(do)).sum().backward()
    ref = {"o": o.detach().numpy(), "dq": tq.grad.numpy(), "dk": tk.grad.numpy(), "dv": tv.grad.numpy()}
    for W in (N, N + 3):
        out = orc.oracle_backward(q, k, v, do, W, scale, causal=False)
        for key in ref:
            assert _rel(out[key], ref[key]) < 1e-12, (key, W)


@pytest.mark.parametrize("Lq,Lk", [(1, 1), (5, 5), (7, 20), (20, 20), (13, 40)])
@pytest.mark.parametrize("W", [1, 2, 6])
@pytest.mark.parametrize("causal", [True, False])
def test_windows_match_library_sdpa_with_masks(Lq, Lk, W, causal):
    """Masks for torch's SDPA built from torch.triu / torch.tril diagonals: the band of a
    bottom-right-aligned (Lk - Lq) causal window, or its two-sided form."""
    B, Hq, Hkv, D = 1, 4, 2, 8
    q, k, v, do = _lq_lk_inputs(B, Hq, Hkv, Lq, Lk, D, 110)
    scale = 0.5
    ones = torch.ones(Lq, Lk, dtype=torch.float64)
    off = Lk - Lq
    upper = torch.tril(ones, diagonal=off)  # keys at or before the query's position
    lower = torch.triu(ones, diagonal=off - (W - 1))  # keys within W - 1 before it
    if causal:
        mask = (upper * lower) > 0.5
    else:
        mask = (torch.tril(ones, diagonal=off + (W - 1)) * lower) > 0.5
    ref = _torch_masked(q, k, v, do, mask, scale)
    out = orc.oracle_backward(q, k, v, do, W, scale, causal=causal)
    for key in ref:
        assert _rel(out[key], ref[key]) < 1e-12, key


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("W", [1, 4, 100])
def test_shorter_queries_are_the_suffix_of_the_full_problem(causal, W):
    """Lq < Lk equals the last Lq query rows of the Lq = Lk problem whose first Lk - Lq query rows
    carry dO = 0 (those rows then add nothing to dK or dV)."""
    B, Hq, Hkv, Lq, Lk, D = 1, 2, 1, 9, 25, 6
    q, k, v, do = _lq_lk_inputs(B, Hq, Hkv, Lq, Lk, D, 120)
    pre = _rand((B, Hq, Lk - Lq, D), 129)
    q_full = np.concatenate([pre, q], axis=2)
    do_full = np.concatenate([np.zeros_like(pre), do], axis=2)
    scale = 0.7
    short = orc.oracle_backward(q, k, v, do, W, scale, causal=causal)
    full = orc.oracle_backward(q_full, k, v, do_full, W, scale, causal=causal)
    for key in ("o", "lse", "delta", "dq"):
        assert np.max(np.abs(short[key] - full[key][:, :, Lk - Lq:])) < 1e-12, key
    for key in ("dk", "dv"):
        assert np.max(np.abs(short[key] - full[key])) < 1e-12, key


def test_noncausal_window_is_symmetric_under_reversal():
    """Reversing the sequence maps a two-sided window onto itself."""
    B, Hq, Hkv, N, D, W = 1, 2, 1, 17, 5, 4
    q, k, v, do = _lq_lk_inputs(B, Hq, Hkv, N, N, D, 130)
    scale = 0.6
    a = orc.oracle_backward(q, k, v, do, W, scale, causal=False)
    flip = lambda x: x[:, :, ::-1].copy()  # noqa: E731
    b = orc.oracle_backward(flip(q), flip(k), flip(v), flip(do), W, scale, causal=False)
    for key in ("o", "dq", "dk", "dv"):
        assert np.max(np.abs(a[key] - flip(b[key]))) < 1e-12, key


@pytest.mark.parametrize("Lq,Lk,W,causal", [(5, 9, 3, True), (6, 6, 3, False), (4, 10, 4, False)])
def test_finite_differences_lq_lk(Lq, Lk, W, causal):
    B, Hq, Hkv, D = 1, 2, 1, 3
    q, k, v, do = _lq_lk_inputs(B, Hq, Hkv, Lq, Lk, D, 140)
    scale = 0.8
    out = orc.oracle_backward(q, k, v, do, W, scale, causal=causal)
    h = 1e-6

    def loss(qq, kk, vv):
        o, _ = orc.oracle_forward(qq, kk, vv, W, scale, causal=causal)
        return float(np.sum(do * o))

    for name, arr, grad in (("q", q, out["dq"]), ("k", k, out["dk"]), ("v", v, out["dv"])):
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args_p = {"q": q, "k": k, "v": v}
            args_m = {"q": q, "k": k, "v": v}
            args_p[name] = arr.copy()
            args_m[name] = arr.copy()
            args_p[name][idx] += h
            args_m[name][idx] -= h
            fd[idx] = (loss(args_p["q"], args_p["k"], args_p["v"])
                       - loss(args_m["q"], args_m["k"], args_m["v"])) / (2 * h)
        assert np.linalg.norm(fd - grad) / max(np.linalg.norm(fd), 1e-3) < 1e-6, name


def _brute_force_forward_general(q, k, v, W, scale, causal):
    """Loops with math.exp; query i at key position i + len(k) - len(q)."""
    Lq, Lk, D = len(q), len(k), len(q[0])
    off = Lk - Lq
    o = [[0.0] * len(v[0]) for _ in range(Lq)]
    lse = [0.0] * Lq
    for i in range(Lq):
        scores = []
        for j in range(Lk):
            d = i + off - j
            if (0 <= d < W) if causal else (-W < d < W):
                scores.append((j, scale * sum(q[i][c] * k[j][c] for c in range(D))))
        m = max(sc for _, sc in scores)
        lse[i] = m + math.log(sum(math.exp(sc - m) for _, sc in scores))
        for j, sc in scores:
            p = math.exp(sc - lse[i])
            for c in range(len(v[0])):
                o[i][c] += p * v[j][c]
    return np.array(o), np.array(lse)


@pytest.mark.parametrize("Lq,Lk,W,causal", [(3, 8, 2, True), (8, 8, 3, False), (2, 7, 9, False),
                                            (1, 6, 1, True)])
def test_brute_force_loops_lq_lk(Lq, Lk, W, causal):
    D = 3
    q, k, v = _rand((Lq, D), 150), _rand((Lk, D), 151), _rand((Lk, D), 152)
    o, lse = orc.head_forward(q, k, v, W, 0.9, causal=causal)
    o2, lse2 = _brute_force_forward_general(q.tolist(), k.tolist(), v.tolist(), W, 0.9, causal)
    assert np.max(np.abs(o - o2)) < 1e-12
    assert np.max(np.abs(lse - lse2)) < 1e-12


def _lq_lk_pins_pass():
    """The masked-SDPA pin on a short-query case, causal and not; True iff both agree."""
    B, Hq, Hkv, Lq, Lk, D, W = 1, 2, 1, 6, 15, 4, 5
    q, k, v, do = _lq_lk_inputs(B, Hq, Hkv, Lq, Lk, D, 160)
    ones = torch.ones(Lq, Lk, dtype=torch.float64)
    off = Lk - Lq
    lower = torch.triu(ones, diagonal=off - (W - 1))
    ok = True
    for causal, upper in ((True, torch.tril(ones, diagonal=off)),
                          (False, torch.tril(ones, diagonal=off + W - 1))):
        ref = _torch_masked(q, k, v, do, (upper * lower) > 0.5, 0.5)
        out = orc.oracle_backward(q, k, v, do, W, 0.5, causal=causal)
        ok = ok and all(_rel(out[key], ref[key]) < 1e-12 for key in ref)
    return ok


def test_lq_lk_pins_accept_the_oracle():
    assert _lq_lk_pins_pass()


def test_lq_lk_pins_reject_top_left_alignment(monkeypatch):
    monkeypatch.setattr(orc, "_offset", lambda qh, kh: 0)
    assert not _lq_lk_pins_pass()


def test_lq_lk_pins_reject_one_sided_noncausal_window(monkeypatch):
    real = orc.visible
    monkeypatch.setattr(orc, "visible", lambda i, j, W, off=0, causal=True: real(i, j, W, off, True))
    assert not _lq_lk_pins_pass()
