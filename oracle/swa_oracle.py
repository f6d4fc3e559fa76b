"""fp64 CPU oracle for sliding-window attention with grouped-query heads, forward and backward.

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import or run this module.  It shares no code with the CUDA library: it is the
plain definition written out with NumPy in float64, materialising the score matrix and the explicit
window mask, so that a reader can check it by eye.

What is computed (per batch b and query head hq; kv head hk = hq // (Hq / Hkv)); queries i in
[0, Lq), keys j in [0, Lk), Lq <= Lk, query i at key position pos(i) = i + (Lk - Lq):

    visible(i, j)  <=>  0 <= pos(i) - j < W        causal sliding window (self included), or
                   <=>  |pos(i) - j| < W           non-causal window (causal=False)
    S[i, j]  = scale * <Q[i], K[j]>   if visible(i, j), else -inf
    LSE[i]   = ln sum_j exp(S[i, j])                           (natural log, over scaled scores)
    P[i, j]  = exp(S[i, j] - LSE[i])
    O[i]     = sum_j P[i, j] V[j]
  backward of the loss L = sum(dO * O):
    dV[j]   += sum_i P[i, j] dO[i]              (summed over the query heads that share hk)
    dP[i, j] = <dO[i], V[j]>
    Delta[i] = <dO[i], O[i]>
    dS[i, j] = P[i, j] (dP[i, j] - Delta[i])
    dQ[i]    = scale * sum_j dS[i, j] K[j]
    dK[j]   += scale * sum_i dS[i, j] Q[i]      (summed over the query heads that share hk)

Where these come from:
  * "Off NVIDIA, you fix the platform yourself" (Layer2C Lab 28), section "What was broken?":
    the attention scores form a matrix with a row per query token and a column per key token, and
    a 1,024-token sliding window limits each row to the preceding 1,024 tokens.  The dense path
    that builds the whole matrix is the one the lab measured at 198 GB (lab record, numbers entry
    "Attention backward memory").
  * Same lab, section "What did fixing it take?" and the record's numbers entry "Gradient parity":
    the exact gradient vanishes at a one-token window.  That fixes the reading that the window
    includes the query itself (W = 1 leaves exactly one visible key, so the softmax is the constant
    1 and dQ = dK = 0).
  * mlx-train-perf README, flash-attention section: the saved state is the attention output and
    the log-sum-exp, and the backward recomputes what it needs.  LSE here is that saved quantity.
  * The pages print no formulas; the lines above are the standard scaled-dot-product attention and
    its hand-derived gradient.  Delta is the usual row-sum identity sum_j P[i,j] dP[i,j] = <dO[i], O[i]>.
  * Grouped-query mapping (the pages name grouped-query ratios but not the mapping): consecutive
    query heads share a kv head, hk = hq // G.
  * Lab 28's gradient sweep also includes query sequences shorter than the key sequence, and both
    causal and non-causal windows (record, numbers entry "Gradient parity, small shapes"), without
    defining either.  Readings:
    shorter queries are the last Lq positions of the key sequence (bottom-right alignment, the
    usual convention for a query suffix attending to a longer context), and a non-causal window of
    size W sees the keys within W - 1 positions on either side, |pos(i) - j| < W, so that W = 1 is
    still the query's own key and a window covering both sequences is full attention.  With
    Lq = Lk and causal=True everything reduces to the formulas above with pos(i) = i.

Row blocks: for long sequences S is materialised ``row_block`` query rows at a time (all N columns).
That only splits the sums over i in dK and dV into partial sums; nothing else changes.
"""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np

__all__ = [
    "visible",
    "kv_head_of",
    "head_forward",
    "head_backward",
    "rows_backward",
    "oracle_forward",
    "oracle_backward",
    "group_backward",
    "forward_rows",
    "dq_rows",
    "dkdv_rows",
    "probabilities",
]


def visible(i, j, W, off: int = 0, causal: bool = True):
    """Window visibility of query i (at key position i + off) and key j: 0 <= i + off - j < W
    (causal) or |i + off - j| < W (non-causal)."""
    d = i + off - j
    if causal:
        return (d >= 0) & (d < W)
    return (d > -W) & (d < W)


def kv_head_of(hq: int, Hq: int, Hkv: int) -> int:
    """Consecutive query heads share a kv head (G = Hq / Hkv query heads per kv head)."""
    return hq // (Hq // Hkv)


def _as64(x) -> np.ndarray:
    """Exact upcast of a bf16 torch tensor (or any array) to a float64 NumPy array."""
    if hasattr(x, "detach"):
        import torch  # local import: torch only as a container here

        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _offset(qh: np.ndarray, kh: np.ndarray) -> int:
    """Key position of query 0: the queries are the last Lq positions of the Lk keys."""
    off = kh.shape[0] - qh.shape[0]
    assert off >= 0, "queries may not outnumber keys"
    return off


def _scores(qh: np.ndarray, kh: np.ndarray, rows: np.ndarray, W: int, scale: float,
            causal: bool = True) -> np.ndarray:
    """Masked scaled scores S[rows, :] for one head (invisible cells are -inf)."""
    Lk = kh.shape[0]
    s = scale * (qh[rows] @ kh.T)
    mask = visible(rows[:, None], np.arange(Lk)[None, :], W, _offset(qh, kh), causal)
    return np.where(mask, s, -np.inf)


def _logsumexp_rows(s: np.ndarray) -> np.ndarray:
    """ln sum_j exp(s[i, j]) per row, with the row max taken out first."""
    m = np.max(s, axis=1)
    assert np.all(np.isfinite(m)), "every row sees at least the key at its own position"
    return m + np.log(np.sum(np.exp(s - m[:, None]), axis=1))


def _row_blocks(n: int, row_block: int):
    for r0 in range(0, n, row_block):
        yield np.arange(r0, min(n, r0 + row_block))


def probabilities(qh, kh, W: int, scale: float, causal: bool = True) -> np.ndarray:
    """The full softmax matrix P [Lq, Lk] of one head (small sizes only)."""
    qh, kh = _as64(qh), _as64(kh)
    rows = np.arange(qh.shape[0])
    s = _scores(qh, kh, rows, W, scale, causal)
    lse = _logsumexp_rows(s)
    return np.exp(s - lse[:, None])


def head_forward(qh, kh, vh, W: int, scale: float, row_block: int = 1024, causal: bool = True):
    """Forward for one (b, hq): returns (O [Lq, D], LSE [Lq]) in float64."""
    qh, kh, vh = _as64(qh), _as64(kh), _as64(vh)
    Lq, D = qh.shape
    o = np.empty((Lq, vh.shape[1]))
    lse = np.empty(Lq)
    for rows in _row_blocks(Lq, row_block):
        s = _scores(qh, kh, rows, W, scale, causal)
        l_r = _logsumexp_rows(s)
        p = np.exp(s - l_r[:, None])
        o[rows] = p @ vh
        lse[rows] = l_r
    return o, lse


def head_backward(qh, kh, vh, doh, W: int, scale: float, row_block: int = 1024,
                  causal: bool = True) -> Dict[str, np.ndarray]:
    """Forward and backward for one (b, hq).

    Returns a dict with o, lse, delta, dq for this query head and dk, dv = this head's contribution
    to its kv head's gradients (the caller sums them over the group).
    """
    qh, kh, vh, doh = _as64(qh), _as64(kh), _as64(vh), _as64(doh)
    Lq, D = qh.shape
    Lk = kh.shape[0]
    out = {
        "o": np.empty((Lq, vh.shape[1])),
        "lse": np.empty(Lq),
        "delta": np.empty(Lq),
        "dq": np.empty((Lq, D)),
        "dk": np.zeros((Lk, D)),
        "dv": np.zeros((Lk, vh.shape[1])),
    }
    for rows in _row_blocks(Lq, row_block):
        r = rows_backward(qh, kh, vh, doh, rows, W, scale, causal)
        for key in ("o", "lse", "delta", "dq"):
            out[key][rows] = r[key]
        out["dk"] += r["dk"]
        out["dv"] += r["dv"]
    return out


def rows_backward(qh, kh, vh, doh, rows, W: int, scale: float,
                  causal: bool = True) -> Dict[str, np.ndarray]:
    """Forward and backward restricted to the query rows `rows` of one head.

    Returns o, lse, delta, dq for those rows and dk, dv [Lk, D] = those rows' contribution to the
    kv head's gradients (dK[j] and dV[j] are sums over query rows i).
    """
    qh, kh, vh, doh = _as64(qh), _as64(kh), _as64(vh), _as64(doh)
    rows = np.asarray(rows, dtype=np.int64)
    s = _scores(qh, kh, rows, W, scale, causal)
    lse = _logsumexp_rows(s)
    p = np.exp(s - lse[:, None])
    o_r = p @ vh
    do_r = doh[rows]
    dp = do_r @ vh.T
    delta = np.sum(do_r * o_r, axis=1)
    ds = p * (dp - delta[:, None])
    return {
        "o": o_r,
        "lse": lse,
        "delta": delta,
        "dq": scale * (ds @ kh),
        "dk": scale * (ds.T @ qh[rows]),
        "dv": p.T @ do_r,
    }


def oracle_forward(q, k, v, window: int, scale: float, row_block: int = 1024,
                   causal: bool = True):
    """Forward over whole tensors q [B,Hq,Lq,D], k, v [B,Hkv,Lk,D]: returns (O [B,Hq,Lq,D],
    LSE [B,Hq,Lq]) in float64."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    B, Hq, Lq, D = q.shape
    Hkv = k.shape[1]
    o = np.empty(q.shape[:3] + (v.shape[3],))
    lse = np.empty((B, Hq, Lq))
    for b in range(B):
        for hq in range(Hq):
            hk = kv_head_of(hq, Hq, Hkv)
            o[b, hq], lse[b, hq] = head_forward(q[b, hq], k[b, hk], v[b, hk], window, scale,
                                                row_block, causal)
    return o, lse


def group_backward(q, k, v, do, b: int, hk: int, window: int, scale: float, row_block: int = 1024,
                   causal: bool = True):
    """Forward + backward of one kv group (kv head hk of batch b and its G query heads).

    Every gradient of a group depends only on that group, so this is exact for those heads.
    Returns dict: hq (list of query heads), o/lse/delta/dq stacked over the group's query heads,
    dk/dv for kv head hk.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    heads = [hq for hq in range(Hq) if kv_head_of(hq, Hq, Hkv) == hk]
    assert len(heads) == G
    res = {"hq": heads, "o": [], "lse": [], "delta": [], "dq": []}
    dk = np.zeros(k.shape[2:])
    dv = np.zeros(v.shape[2:])
    for hq in heads:
        r = head_backward(q[b, hq], k[b, hk], v[b, hk], do[b, hq], window, scale, row_block, causal)
        for key in ("o", "lse", "delta", "dq"):
            res[key].append(r[key])
        dk += r["dk"]
        dv += r["dv"]
    for key in ("o", "lse", "delta", "dq"):
        res[key] = np.stack(res[key])
    res["dk"], res["dv"] = dk, dv
    return res


def oracle_backward(q, k, v, do, window: int, scale: float, row_block: int = 1024,
                    causal: bool = True):
    """Full forward + backward over whole tensors.

    Returns dict with o, lse, delta [B,Hq,Lq(,D)], dq [B,Hq,Lq,D], dk, dv [B,Hkv,Lk,D], float64.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    out = {
        "o": np.empty((B, Hq, Lq, v.shape[3])),
        "lse": np.empty((B, Hq, Lq)),
        "delta": np.empty((B, Hq, Lq)),
        "dq": np.empty((B, Hq, Lq, D)),
        "dk": np.empty((B, Hkv, Lk, D)),
        "dv": np.empty((B, Hkv, Lk, v.shape[3])),
    }
    for b in range(B):
        for hk in range(Hkv):
            r = group_backward(q, k, v, do, b, hk, window, scale, row_block, causal)
            for idx, hq in enumerate(r["hq"]):
                for key in ("o", "lse", "delta", "dq"):
                    out[key][b, hq] = r[key][idx]
            out["dk"][b, hk] = r["dk"]
            out["dv"][b, hk] = r["dv"]
    return out


# ---------------------------------------------------------------------------------------------
# Sampled outputs for sizes where the dense oracle over every head is too slow.  Each value is
# the same definition evaluated for the requested rows only.
# ---------------------------------------------------------------------------------------------

def forward_rows(qh, kh, vh, rows: Sequence[int], W: int, scale: float, causal: bool = True):
    """O[rows] and LSE[rows] of one head; each row only needs its own scores against all keys."""
    qh, kh, vh = _as64(qh), _as64(kh), _as64(vh)
    rows = np.asarray(rows, dtype=np.int64)
    s = _scores(qh, kh, rows, W, scale, causal)
    lse = _logsumexp_rows(s)
    p = np.exp(s - lse[:, None])
    return p @ vh, lse


def dq_rows(qh, kh, vh, doh, rows: Sequence[int], W: int, scale: float, causal: bool = True):
    """dQ[rows] of one head (needs only those rows' P, dP and Delta)."""
    qh, kh, vh, doh = _as64(qh), _as64(kh), _as64(vh), _as64(doh)
    rows = np.asarray(rows, dtype=np.int64)
    s = _scores(qh, kh, rows, W, scale, causal)
    lse = _logsumexp_rows(s)
    p = np.exp(s - lse[:, None])
    o_r = p @ vh
    dp = doh[rows] @ vh.T
    delta = np.sum(doh[rows] * o_r, axis=1)
    ds = p * (dp - delta[:, None])
    return scale * (ds @ kh)


def dkdv_rows(q_heads, kh, vh, do_heads, keys: Sequence[int], W: int, scale: float,
              row_block: int = 1024, fwd: Optional[list] = None, causal: bool = True):
    """dK[keys], dV[keys] of one kv head, summed over the query heads given.

    q_heads, do_heads: sequences of [Lq, D] arrays (the group's query heads).  Column j of P and dS
    needs LSE and Delta of every row, so each head's full forward runs first (or is passed in
    ``fwd`` as a list of (O, LSE) pairs).
    """
    kh, vh = _as64(kh), _as64(vh)
    keys = np.asarray(keys, dtype=np.int64)
    dk = np.zeros((len(keys), kh.shape[1]))
    dv = np.zeros((len(keys), vh.shape[1]))
    for g, (qh, doh) in enumerate(zip(q_heads, do_heads)):
        qh, doh = _as64(qh), _as64(doh)
        if fwd is not None:
            o, lse = fwd[g]
        else:
            o, lse = head_forward(qh, kh, vh, W, scale, row_block, causal)
        delta = np.sum(doh * o, axis=1)
        rows = np.arange(qh.shape[0])
        # Columns `keys` of S for every row: S[:, keys] = scale * Q K[keys]^T, masked.
        s = scale * (qh @ kh[keys].T)
        s = np.where(visible(rows[:, None], keys[None, :], W, _offset(qh, kh), causal), s, -np.inf)
        p = np.exp(s - lse[:, None])
        dp = doh @ vh[keys].T
        ds = p * (dp - delta[:, None])
        dv += p.T @ doh
        dk += scale * (ds.T @ qh)
    return dk, dv
