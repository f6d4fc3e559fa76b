"""Sequence-sharded causal sliding-window attention over a torch.distributed process group.

Rank r of P holds positions [r L, (r + 1) L) of every head: q, k, v, dO chunks [B, H, L, D].  A
query at global position p sees keys p - W + 1 .. p, so rank r needs, besides its own chunk, the
h = min(W - 1, r L) keys and values just before it (a halo owned by the ranks before it).  With
the halo prepended, rank r's problem is the single-GPU library's "queries shorter than keys" form:
Lq = L queries that are the last L of Lk = h + L keys (bottom-right alignment), computed by the
same kernels.  The backward produces dK, dV for the halo rows too; those go back to the ranks
that own the rows and are added there (the exchange step of the sharding: one point-to-point
round before the forward, one after the backward).  Every gradient of a kv head depends only on
that head's group, so nothing else is exchanged.

The exchange plan is a pure function of (rank, world, L, W), so every rank derives the same
matching sends and receives.  Transfers go through batch_isend_irecv (16-bit tensors as raw int16
words); NCCL on GPUs, gloo on the CPU.  Halo gradients are added in fp32 (or wider) and rounded
once.  Only causal windows shard this way (a two-sided window would put the queries in the middle
of the keys, which the kernels' bottom-right alignment does not express).

The compute functions default to the library's kernels (swa_attn_fwd / swa_attn_bwd); `fwd_fn` /
`bwd_fn` replace them, which is how the CPU tests drive this exchange logic with a reference.
"""
from __future__ import annotations

from typing import Callable, List, Optional, Tuple

Plan = List[Tuple[int, int, int]]  # (peer rank, first global row, one past the last)


def halo_plan(rank: int, L: int, W: int) -> Plan:
    """Rows rank `rank` receives: the h = min(W - 1, rank L) positions before its chunk, as
    (source rank, start, stop) segments in position order."""
    h = min(W - 1, rank * L)
    lo = rank * L - h
    segs = []
    for src in range(lo // L if L > 0 else 0, rank):
        a, b = max(lo, src * L), (src + 1) * L
        if a < b:
            segs.append((src, a, b))
    return segs


def send_plan(rank: int, world: int, L: int, W: int) -> Plan:
    """Rows of rank `rank`'s chunk that later ranks need: (destination rank, start, stop)."""
    out = []
    for dst in range(rank + 1, world):
        for src, a, b in halo_plan(dst, L, W):
            if src == rank:
                out.append((dst, a, b))
    return out


def _wire_dtype(dtype):
    """16-bit tensors travel as int16 words (gloo has no bf16 type); others as they are."""
    import torch

    return torch.int16 if torch.empty((), dtype=dtype).element_size() == 2 else dtype


def _words(t):
    return t.contiguous().view(_wire_dtype(t.dtype))


def _exchange(sends, recvs, group):
    """Posts every send and receive of one round and waits for all of them."""
    import torch.distributed as dist

    def glob(peer):  # plans number ranks inside `group`; P2POp's peer is a global rank
        return peer if group is None else dist.get_global_rank(group, peer)

    ops = [dist.P2POp(dist.isend, buf, glob(peer), group) for peer, buf in sends]
    ops += [dist.P2POp(dist.irecv, buf, glob(peer), group) for peer, buf in recvs]
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()


def _rank_world(group):
    import torch.distributed as dist

    return dist.get_rank(group), dist.get_world_size(group)


def gather_halo(k, v, window: int, group=None):
    """K and V of this rank's chunk with the halo before it prepended: (k_ext, v_ext, h)."""
    import torch

    rank, world = _rank_world(group)
    L = k.shape[2]
    base = rank * L
    kv = torch.stack([k, v])  # [2, B, Hkv, L, D]
    sends = [(dst, _words(kv[:, :, :, a - base:b - base])) for dst, a, b in
             send_plan(rank, world, L, window)]
    segs = halo_plan(rank, L, window)
    bufs = [torch.empty((2,) + tuple(k.shape[:2]) + (b - a, k.shape[3]),
                        dtype=_wire_dtype(k.dtype), device=k.device) for _, a, b in segs]
    _exchange(sends, [(src, buf) for (src, _, _), buf in zip(segs, bufs)], group)
    halo = [buf.view(k.dtype) for buf in bufs]
    k_ext = torch.cat([x[0] for x in halo] + [k], dim=2)
    v_ext = torch.cat([x[1] for x in halo] + [v], dim=2)
    return k_ext, v_ext, k_ext.shape[2] - L


def _default_fwd(q, k_ext, v_ext, window, scale):
    from . import swa_attn_fwd

    return swa_attn_fwd(q, k_ext, v_ext, window, scale, causal=True)


def _default_bwd(q, k_ext, v_ext, o, do, lse, window, scale):
    from . import swa_attn_bwd

    return swa_attn_bwd(q, k_ext, v_ext, o, do, lse, window, scale, causal=True)


def seq_fwd(q, k, v, window: int, scale: Optional[float] = None, group=None,
            fwd_fn: Optional[Callable] = None):
    """Forward of this rank's query chunk: returns (o, lse, k_ext, v_ext).  k_ext / v_ext (the
    chunk's keys and values with the halo prepended) are what seq_bwd needs."""
    if q.shape[2] != k.shape[2]:
        raise ValueError("every rank holds the same positions of q, k and v")
    k_ext, v_ext, _ = gather_halo(k, v, window, group)
    o, lse = (fwd_fn or _default_fwd)(q, k_ext, v_ext, window, scale)
    return o, lse, k_ext, v_ext


def seq_bwd(q, k_ext, v_ext, o, do, lse, window: int, scale: Optional[float] = None, group=None,
            bwd_fn: Optional[Callable] = None):
    """Backward of this rank's chunk: returns (dq, dk, dv) for the positions this rank owns, with
    the halo contributions of later ranks added."""
    import torch

    rank, world = _rank_world(group)
    L = q.shape[2]
    h = k_ext.shape[2] - L
    dq, dk_ext, dv_ext = (bwd_fn or _default_bwd)(q, k_ext, v_ext, o, do, lse, window, scale)
    dkv = torch.stack([dk_ext, dv_ext])  # [2, B, Hkv, h + L, D]
    # halo rows go back to their owners, segment by segment (the forward's receive plan)
    first = rank * L - h
    sends = [(src, _words(dkv[:, :, :, a - first:b - first])) for src, a, b in
             halo_plan(rank, L, window)]
    mine = send_plan(rank, world, L, window)
    bufs = [torch.empty((2,) + tuple(dk_ext.shape[:2]) + (b - a, dk_ext.shape[3]),
                        dtype=_wire_dtype(dk_ext.dtype), device=dk_ext.device) for _, a, b in mine]
    _exchange(sends, [(dst, buf) for (dst, _, _), buf in zip(mine, bufs)], group)
    acc = dkv[:, :, :, h:].to(torch.promote_types(dkv.dtype, torch.float32))
    base = rank * L
    for (_, a, b), buf in zip(mine, bufs):
        acc[:, :, :, a - base:b - base] += buf.view(dk_ext.dtype).to(acc.dtype)
    out = acc.to(dk_ext.dtype)
    return dq, out[0], out[1]


def _make_autograd():
    import torch

    class SequenceShardedAttention(torch.autograd.Function):
        """o = attention over this rank's chunk of a sequence sharded across `group` (causal
        window); the backward returns this rank's dq and its owned rows of dk, dv."""

        @staticmethod
        def forward(ctx, q, k, v, window: int, scale: Optional[float] = None, group=None,
                    fwd_fn: Optional[Callable] = None, bwd_fn: Optional[Callable] = None):
            o, lse, k_ext, v_ext = seq_fwd(q, k, v, window, scale, group, fwd_fn)
            ctx.save_for_backward(q, k_ext, v_ext, o, lse)
            ctx.window, ctx.scale, ctx.group, ctx.bwd_fn = window, scale, group, bwd_fn
            return o

        @staticmethod
        def backward(ctx, do):
            q, k_ext, v_ext, o, lse = ctx.saved_tensors
            dq, dk, dv = seq_bwd(q, k_ext, v_ext, o, do.contiguous(), lse, ctx.window, ctx.scale,
                                 ctx.group, ctx.bwd_fn)
            return dq, dk, dv, None, None, None, None, None

    return SequenceShardedAttention


class _LazyAutograd:
    _cls = None

    def __getattr__(self, name):
        if _LazyAutograd._cls is None:
            _LazyAutograd._cls = _make_autograd()
        return getattr(_LazyAutograd._cls, name)


SequenceShardedAttention = _LazyAutograd()
