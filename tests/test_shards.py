"""The layer over several ranks on the CPU ("Keeping each expert's batch large":
data parallelism for the gate and expert parallelism for the experts), with
world_size-2 gloo ranks and no GPU.

* The expert-parallel exchange plan (``moe_ep_plan``, host-only, through the C ABI)
  on a case worked by hand, and its argument checks.
* Data parallel: two ranks each gate their half of a batch, add their Importance
  and Load vectors with the package's all-reduce, and the losses formed from the
  totals equal the one-process oracle's losses of the whole batch (1e-5), while
  each half's own losses do not.
* Expert parallel: two ranks, each holding half of the experts, gate and dispatch
  their tokens, exchange the offsets and the routed rows with the package's
  collectives and the library's plan, run their experts on the rows that arrived
  (regrouped expert-major as the plan says) and send the outputs back; each rank's
  combined output equals the one-process oracle's layer output on its tokens.
The per-rank arithmetic here is the oracle's (the library's kernels need a GPU;
tests/test_gpu_shards.py runs them); what is tested is the plan and the exchange.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT

import sparsely_gated_mixture_03_b300 as moe
from oracle import moe_oracle as O


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_ep_plan_by_hand():
    """world 2, n 4 (rank 0 holds experts 0-1, rank 1 holds 2-3).
    rank 0 routes 2, 1, 3, 0 rows to experts 0..3; rank 1 routes 1, 2, 0, 4."""
    offs = np.array([[0, 2, 3, 6, 6], [0, 1, 3, 3, 7]], dtype=np.int32)
    send, recv, plan = moe.moe_ep_plan(2, 1, 4, offs)
    assert send.tolist() == [3, 4]        # its rows for experts 0-1, then 2-3
    assert recv.tolist() == [3, 4]        # rank 0 sends 3 + 0 rows, rank 1 sends 0 + 4
    # arrival order: [rank 0: expert 2 (3 rows), expert 3 (0)] [rank 1: expert 2 (0), expert 3 (4)]
    # expert-major:  [expert 2: rank 0 (3), rank 1 (0)] [expert 3: rank 0 (0), rank 1 (4)]
    B = 4
    assert plan[:B].tolist() == [0, 3, 3, 3]           # arrival start of (e, s), e * 2 + s
    assert plan[B:2 * B + 1].tolist() == [0, 3, 3, 3, 7]
    assert plan[2 * B + 1:].tolist() == [0, 3, 7]      # local expert offsets
    send, recv, plan = moe.moe_ep_plan(2, 0, 4, offs)
    assert send.tolist() == [3, 3] and recv.tolist() == [3, 3]
    # arrival: [rank 0: e0 2, e1 1] [rank 1: e0 1, e1 2]; expert-major: e0: 2 + 1, e1: 1 + 2
    assert plan[:B].tolist() == [0, 3, 2, 4]
    assert plan[B:2 * B + 1].tolist() == [0, 2, 3, 4, 6]
    assert plan[2 * B + 1:].tolist() == [0, 3, 6]
    # one rank holding everything: the plan is the identity
    send, recv, plan = moe.moe_ep_plan(1, 0, 4, offs[:1])
    assert plan[:4].tolist() == [0, 2, 3, 6] and plan[4:9].tolist() == [0, 2, 3, 6, 6]


def test_ep_plan_checks():
    offs = np.array([[0, 2, 3, 6, 6], [0, 1, 3, 3, 7]], dtype=np.int32)
    moe.moe_ep_plan(3, 0, 3, np.zeros((3, 4), np.int32) + np.arange(4))      # one expert a rank
    with pytest.raises(moe.MoeError, match="UNSUPPORTED"):
        moe.moe_ep_plan(2, 0, 3, np.zeros((2, 4), np.int32))                  # 3 % 2 != 0
    with pytest.raises(moe.MoeError, match="INVALID_ARG"):
        bad = offs.copy()
        bad[1, 2] = 0                       # decreasing offsets
        moe.moe_ep_plan(2, 0, 4, bad)
    with pytest.raises(moe.MoeError, match="INVALID_ARG"):
        moe.moe_ep_plan(2, 2, 4, offs)      # rank outside the world


def _batch(seed, T, d, n, h):
    rng = np.random.default_rng(seed)
    return dict(x=rng.normal(size=(T, d)), W_g=rng.normal(size=(d, n)) / np.sqrt(d),
                W_noise=rng.normal(size=(d, n)) / np.sqrt(d), eps=rng.normal(size=(T, n)),
                W_in=rng.normal(size=(n, d, h)) / np.sqrt(d),
                W_out=rng.normal(size=(n, h, d)) / np.sqrt(h))


T_ALL, D, N, H, K = 96, 6, 8, 5, 2


def _regroup(plan, world, nl, rows_in, to_expert_major):
    """The row permutation moe_ep_regroup performs, written out from its contract."""
    B = world * nl
    src, dst = plan[:B], plan[B:2 * B + 1]
    out = np.empty_like(rows_in)
    for q in range(B):
        cnt = dst[q + 1] - dst[q]
        if to_expert_major:
            out[dst[q]:dst[q] + cnt] = rows_in[src[q]:src[q] + cnt]
        else:
            out[src[q]:src[q] + cnt] = rows_in[dst[q]:dst[q] + cnt]
    return out


def _rank_main(rank, world, port, errfile):
    import sys
    sys.path.insert(0, ROOT)
    from sparsely_gated_mixture_03_b300 import shards
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        a = _batch(5, T_ALL, D, N, H)
        Tr = T_ALL // world
        mine = slice(rank * Tr, (rank + 1) * Tr)
        full = O.moe_forward(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"], a["W_out"], K)
        g = O.gating(a["x"][mine], a["W_g"], a["W_noise"], a["eps"][mine], K)

        # data parallel: the batch's losses from the all-reduced sums
        imp = O.importance_of(g["idx"], g["gates"], N)
        load = g["P"].sum(axis=0)
        sums = torch.tensor(np.concatenate([imp, load]), dtype=torch.float32)
        shards.allreduce_sums(sums)
        ci, cl, aux = O.balance_losses(sums[:N].double().numpy(), sums[N:].double().numpy())
        ref = full["losses"]
        assert abs(ci - ref[0]) <= 1e-5 * abs(ref[0]) and abs(cl - ref[1]) <= 1e-5 * abs(ref[1])
        assert abs(aux - ref[2]) <= 1e-5 * abs(ref[2])
        own = O.balance_losses(imp, load)
        assert abs(own[0] - ref[0]) > 1e-3 * abs(ref[0])   # a half's CV^2 is not the batch's

        # expert parallel: rank r holds experts [r nl, (r+1) nl)
        nl = N // world
        offsets, perm, inv = O.dispatch(g["idx"], N)
        x_perm = a["x"][mine][perm // K]
        send, recv, plan = shards.exchange_plan(torch.from_numpy(offsets.astype(np.int32)),
                                                world, rank, N)
        x_recv = shards.exchange_rows(torch.from_numpy(x_perm), send, recv).numpy()
        x_local = _regroup(plan, world, nl, x_recv, True)
        loc = plan[2 * world * nl + 1:]
        y_local = np.zeros_like(x_local)
        for e in range(nl):
            p0, p1 = loc[e], loc[e + 1]
            if p1 > p0:
                ge = rank * nl + e
                y_local[p0:p1] = O.expert_ffn(x_local[p0:p1], a["W_in"][ge], a["W_out"][ge])
        y_recv = _regroup(plan, world, nl, y_local, False)
        y_perm = shards.exchange_rows(torch.from_numpy(y_recv), recv, send).numpy()
        y = O.combine_gathered(y_perm, inv, g["gates"])
        assert np.allclose(y, full["y"][mine], rtol=1e-12, atol=1e-12)
        assert int(recv.sum()) == int(np.isin(full["idx"], range(rank * nl, (rank + 1) * nl)).sum())
    except BaseException as e:          # report the failure to the parent
        with open(errfile + str(rank), "w") as f:
            f.write(repr(e))
        raise
    finally:
        dist.destroy_process_group()


def test_data_and_expert_parallel_two_gloo_ranks(tmp_path):
    world, port = 2, _free_port()
    errfile = str(tmp_path / "err")
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, errfile)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    errs = [open(errfile + str(r)).read() for r in range(world) if os.path.exists(errfile + str(r))]
    assert not errs, errs
    assert all(p.exitcode == 0 for p in procs)
