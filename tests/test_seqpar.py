"""Sequence sharding (sliding_window_flash_gb300.seqpar) on the CPU over gloo: the halo exchange
and the return of halo gradients, with the fp64 oracle as each rank's compute, must reproduce the
unsharded oracle on the whole sequence.  World sizes 2 and 3; windows shorter than a chunk, equal
to it, and spanning several ranks (so a rank's halo comes from more than one rank).  A rank that
dies before the exchange makes the other rank's exchange raise rather than hang."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import swa_inputs as si
from sliding_window_flash_gb300 import seqpar

L = 24  # positions per rank


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_fwd(q, k, v, W, scale):
    from oracle import swa_oracle as orc

    o, lse = orc.oracle_forward(q, k, v, W, scale)
    return torch.from_numpy(o), torch.from_numpy(lse)


def _oracle_bwd(q, k, v, o, do, lse, W, scale):
    from oracle import swa_oracle as orc

    r = orc.oracle_backward(q, k, v, do, W, scale)
    return torch.from_numpy(r["dq"]), torch.from_numpy(r["dk"]), torch.from_numpy(r["dv"])


def _case(world, W):
    return si.Case(B=1, Hq=4, Hkv=2, N=world * L, D=16, W=W, seed=world * 100 + W)


def _worker(rank, world, W, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case = _case(world, W)
    full = si.make_inputs(case)
    sl = slice(rank * L, (rank + 1) * L)
    q, k, v, do = (full[n][:, :, sl].contiguous() for n in ("q", "k", "v", "do"))
    o, lse, k_ext, v_ext = seqpar.seq_fwd(q, k, v, W, case.softmax_scale, fwd_fn=_oracle_fwd)
    assert k_ext.shape[2] == L + min(W - 1, rank * L)
    dq, dk, dv = seqpar.seq_bwd(q, k_ext, v_ext, o, do, lse, W, case.softmax_scale,
                                bwd_fn=_oracle_bwd)
    out[rank] = {n: t.numpy() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
    dist.destroy_process_group()


@pytest.mark.parametrize("world,W", [(2, 7), (2, 24), (2, 25), (3, 10), (3, 40), (3, 60)])
def test_sharded_equals_unsharded(world, W):
    from oracle import swa_oracle as orc

    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, W, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    case = _case(world, W)
    full = si.make_inputs(case)
    ref = orc.oracle_backward(full["q"], full["k"], full["v"], full["do"], W, case.softmax_scale)
    for name in ("o", "lse", "dq", "dk", "dv"):
        got = np.concatenate([out[r][name] for r in range(world)], axis=2)
        np.testing.assert_allclose(got, ref[name], rtol=1e-10, atol=1e-12, err_msg=name)


def _autograd_worker(rank, world, W, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    case = _case(world, W)
    full = si.make_inputs(case)
    sl = slice(rank * L, (rank + 1) * L)
    q, k, v, do = (full[n][:, :, sl].double().contiguous() for n in ("q", "k", "v", "do"))
    for t in (q, k, v):
        t.requires_grad_(True)
    o = seqpar.SequenceShardedAttention.apply(q, k, v, W, case.softmax_scale, None, _oracle_fwd,
                                              _oracle_bwd)
    o.backward(do)
    out[rank] = {"o": o.detach().numpy(), "dq": q.grad.numpy(), "dk": k.grad.numpy(),
                 "dv": v.grad.numpy()}
    dist.destroy_process_group()


def test_autograd_wrapper_two_ranks():
    """SequenceShardedAttention through torch autograd reproduces the unsharded gradients."""
    from oracle import swa_oracle as orc

    world, W = 2, 30
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_autograd_worker, args=(r, world, W, port, out))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    case = _case(world, W)
    full = si.make_inputs(case)
    ref = orc.oracle_backward(full["q"], full["k"], full["v"], full["do"], W, case.softmax_scale)
    for name in ("o", "dq", "dk", "dv"):
        got = np.concatenate([out[r][name] for r in range(world)], axis=2)
        np.testing.assert_allclose(got, ref[name], rtol=1e-10, atol=1e-12, err_msg=name)


def _subgroup_worker(rank, world, members, W, port, out):
    """A sequence-parallel subgroup inside a larger job: the ranks in `members` shard one sequence
    among themselves (group rank g, which torch assigns in order of global rank, holds chunk g);
    the others take no part in the exchange."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    group = dist.new_group(members)  # every rank takes part in creating the group
    if rank in members:
        g = dist.get_rank(group)
        case = _case(len(members), W)
        full = si.make_inputs(case)
        sl = slice(g * L, (g + 1) * L)
        q, k, v, do = (full[n][:, :, sl].contiguous() for n in ("q", "k", "v", "do"))
        o, lse, k_ext, v_ext = seqpar.seq_fwd(q, k, v, W, case.softmax_scale, group=group,
                                              fwd_fn=_oracle_fwd)
        dq, dk, dv = seqpar.seq_bwd(q, k_ext, v_ext, o, do, lse, W, case.softmax_scale,
                                    group=group, bwd_fn=_oracle_bwd)
        out[g] = {n: t.numpy() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("members,W", [([1, 3], 30), ([3, 0, 2], 40)])
def test_sharded_over_a_subgroup(members, W):
    """Sharding over a subgroup of a 4-rank job (group ranks differ from global ranks) reproduces
    the unsharded oracle: the exchange addresses the global ranks of the group's members."""
    from oracle import swa_oracle as orc

    world = 4
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_subgroup_worker, args=(r, world, members, W, port, out))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    n = len(members)
    case = _case(n, W)
    full = si.make_inputs(case)
    ref = orc.oracle_backward(full["q"], full["k"], full["v"], full["do"], W, case.softmax_scale)
    for name in ("o", "lse", "dq", "dk", "dv"):
        got = np.concatenate([out[g][name] for g in range(n)], axis=2)
        np.testing.assert_allclose(got, ref[name], rtol=1e-10, atol=1e-12, err_msg=name)


@pytest.mark.parametrize("world,W", [(2, 1), (4, 30), (4, 200), (3, 48)])
def test_plans_match_and_cover(world, W):
    """Every receive has the matching send, and a rank's halo is exactly the min(W - 1, r L)
    positions before its chunk, in order."""
    sends = {(r, dst, a, b) for r in range(world) for dst, a, b in seqpar.send_plan(r, world, L, W)}
    recvs = {(src, r, a, b) for r in range(world) for src, a, b in seqpar.halo_plan(r, L, W)}
    assert sends == recvs
    for r in range(world):
        rows = [i for _, a, b in seqpar.halo_plan(r, L, W) for i in range(a, b)]
        h = min(W - 1, r * L)
        assert rows == list(range(r * L - h, r * L))


@pytest.mark.gpu
@pytest.mark.parametrize("world,L_rank,W,D", [(2, 384, 100, 128), (4, 256, 600, 128),
                                              (3, 300, 300, 64), (2, 256, 200, 256)])
def test_sharded_kernels_rank_by_rank(swa, world, L_rank, W, D):
    """The CUDA path of each rank of a sharded layer (queries = its chunk, keys = halo + chunk),
    run rank after rank on one GPU with the halo gradients added at their owners' positions as
    seq_bwd does, reproduces the oracle on the whole sequence (bar: 1e-2 norm-wise, LSE 1e-3)."""
    from oracle import swa_oracle as orc

    case = si.Case(B=1, Hq=4, Hkv=2, N=world * L_rank, D=D, W=W, seed=11)
    full = si.make_inputs(case)
    dev = torch.device("cuda:0")
    g = {k_: v_.to(dev) for k_, v_ in full.items()}
    outs = {n: [] for n in ("o", "lse", "dq")}
    dk = torch.zeros(full["k"].shape, dtype=torch.float32, device=dev)
    dv = torch.zeros_like(dk)
    for r in range(world):
        lo = r * L_rank - min(W - 1, r * L_rank)
        sl = slice(r * L_rank, (r + 1) * L_rank)
        q, do = g["q"][:, :, sl].contiguous(), g["do"][:, :, sl].contiguous()
        k_ext = g["k"][:, :, lo:(r + 1) * L_rank].contiguous()
        v_ext = g["v"][:, :, lo:(r + 1) * L_rank].contiguous()
        o, lse = swa.swa_attn_fwd(q, k_ext, v_ext, W, case.softmax_scale)
        dq, dk_e, dv_e = swa.swa_attn_bwd(q, k_ext, v_ext, o, do, lse, W, case.softmax_scale)
        swa.swa_check_device()
        outs["o"].append(o.float())
        outs["lse"].append(lse)
        outs["dq"].append(dq.float())
        dk[:, :, lo:(r + 1) * L_rank] += dk_e.float()
        dv[:, :, lo:(r + 1) * L_rank] += dv_e.float()
    got = {n: torch.cat(t, dim=2).double().cpu().numpy() for n, t in outs.items()}
    got["dk"], got["dv"] = dk.double().cpu().numpy(), dv.double().cpu().numpy()
    ref = orc.oracle_backward(full["q"], full["k"], full["v"], full["do"], W, case.softmax_scale)
    assert np.max(np.abs(got["lse"] - ref["lse"])) <= 1e-3
    for n in ("o", "dq", "dk", "dv"):
        rel = np.linalg.norm(got[n] - ref[n]) / np.linalg.norm(ref[n])
        assert rel <= 1e-2, (n, rel)


def _failing_worker(rank, world, port, out):
    """Rank 0 fails right after joining the group and leaves; rank 1 then needs its halo from
    rank 0 and must end the exchange with an error, not wait forever."""
    import datetime

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=10))
    if rank == 0:
        os._exit(3)  # a rank that dies between steps, with nothing of its own in flight
    case = _case(world, 7)
    full = si.make_inputs(case)
    sl = slice(rank * L, (rank + 1) * L)
    q, k, v = (full[n][:, :, sl].contiguous() for n in ("q", "k", "v"))
    try:
        seqpar.seq_fwd(q, k, v, 7, case.softmax_scale, fwd_fn=_oracle_fwd)
        out[rank] = ("returned", False, "")
    except Exception as e:  # the peer is gone: gloo reports it as a RuntimeError
        out[rank] = ("raised", isinstance(e, RuntimeError), f"{type(e).__name__}: {e}")


def test_dead_peer_ends_the_halo_exchange_with_an_error():
    """Failure is made on the host: one rank exits before the halo exchange.  The surviving rank's
    exchange raises (connection closed or the group's 10 s timeout) instead of hanging."""
    port = _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_failing_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        for p in procs:
            p.join(timeout=120)
        assert procs[0].exitcode == 3
        assert procs[1].exitcode == 0, "the surviving rank hung or crashed"
        assert 1 in out and out[1][0] == "raised" and out[1][1], out.get(1)
    finally:
        for p in procs:
            if p.is_alive():
                p.kill()
