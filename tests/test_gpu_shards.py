"""The sharded layer's kernels on one GPU ("Keeping each expert's batch large":
data-parallel ranks, experts spread over ranks).  Needs a B300; ``pytest -m gpu``.

The ranks are emulated one after another in this process: every collective is a
plain data movement done here by the test (the sum an all-reduce would form, the
slices an all-to-all would deliver), so no kernel waits on another.

* Data parallel: the batch split in shards, each shard's forward pass giving its
  Importance and Load vectors, their sum formed here, and ``moe_losses_from_sums``
  giving the whole batch's losses: against the oracle on the whole batch (run with
  the GPU's kept experts, 1e-5) and the one-GPU forward pass.  Also the Switch gate.
* Expert parallel: each emulated rank gates and dispatches its tokens; the plan of
  ``moe_ep_plan``, the row regroup of ``moe_ep_regroup`` around an all-to-all
  emulated by slicing, each rank's experts on its rows, and the combine; the output
  is bit-identical to the one-GPU forward pass of the whole batch (the same rows reach
  each expert in the same order) and matches the oracle.
"""
import numpy as np
import pytest
import torch

import sparsely_gated_mixture_03_b300 as moe
from sparsely_gated_mixture_03_b300 import synthetic as S
from oracle import moe_oracle as O
from gpu_helpers import assert_rel, assert_y, kept_of, np64, oracle_arrays

pytestmark = pytest.mark.gpu

DEV = "cuda"
F32, BF16 = torch.float32, torch.bfloat16
ROW = moe.FLAG_FFN_ROW_TILES


def _forward(cfg, inp, rows=slice(None), sums=None):
    T, n, k, d = cfg.T, cfg.n, cfg.k, cfg.d
    out = dict(y=torch.empty((T, d), dtype=F32, device=DEV), losses=torch.empty(3, device=DEV),
               idx=torch.empty(T * k, dtype=torch.int32, device=DEV),
               gates=torch.empty(T * k, dtype=F32, device=DEV))
    if sums is None:
        sums = torch.empty(2 * n, dtype=F32, device=DEV)
    moe.moe_forward(cfg, inp["x"][rows].contiguous(), inp["W_g"], inp["W_noise"],
                    inp["eps"][rows].contiguous(), inp["b_g"], inp["W_in"], inp["W_out"],
                    out["y"], out["losses"], out["idx"], out["gates"], None, sums[:n], sums[n:],
                    moe.alloc_workspace(cfg))
    assert moe.moe_get_device_error() == 0
    out["sums"] = sums
    return out


def _cfg(shape, T, flags=0):
    return moe.make_config(T, shape.d, shape.n, shape.h, shape.k, shape.x_dtype,
                           shape.expert_dtype, flags=flags)


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("shape,flags", [
    (S.FlatShape("dp-bf16", 4096, 512, 64, 1024, 4), ROW),
    (S.FlatShape("dp-ragged-fp32", 1000, 64, 12, 128, 3, F32, F32), 0),
    (S.FlatShape("dp-switch", 2048, 128, 32, 256, 1), ROW | moe.FLAG_SWITCH_GATE)],
    ids=["bf16", "fp32", "switch"])
def test_data_parallel_losses(shape, flags, world):
    inp = S.make_flat_inputs(shape, seed=61, device=DEV)
    T, n, k = shape.T, shape.n, shape.k
    bounds = np.linspace(0, T, world + 1).astype(int)       # uneven shards when T % world
    total = torch.zeros(2 * n, dtype=F32, device=DEV)
    idx = []
    for r in range(world):
        part = _forward(_cfg(shape, int(bounds[r + 1] - bounds[r]), flags), inp,
                        slice(bounds[r], bounds[r + 1]))
        total += part["sums"]                               # the all-reduce's sum
        idx.append(part["idx"])
    losses = torch.empty(3, device=DEV)
    cfg_all = _cfg(shape, T, flags)
    moe.moe_losses_from_sums(cfg_all, total[:n].contiguous(), total[n:].contiguous(), losses)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    whole = _forward(cfg_all, inp)
    assert_rel(np64(losses), np64(whole["losses"]), "losses against the one-GPU forward")
    a = oracle_arrays(inp)
    kept = kept_of(torch.cat(idx).cpu().numpy(), k)
    ref = O.moe_forward(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"], a["W_out"], k, 0.0,
                        a["b_g"], switch=bool(flags & moe.FLAG_SWITCH_GATE),
                        kept=None if flags & moe.FLAG_SWITCH_GATE else kept)
    if flags & moe.FLAG_SWITCH_GATE:
        assert np.array_equal(ref["idx"], kept)
    assert_rel(np64(losses), list(ref["losses"]), "losses against the oracle")


def _ep_forward(shape, inp, world, flags):
    """Every emulated rank's part of the expert-parallel layer; returns y [T, d]."""
    T, n, k, d = shape.T, shape.n, shape.k, shape.d
    nl, Tr = n // world, T // world
    ranks = []
    for r in range(world):
        cfg = _cfg(shape, Tr, flags)
        ws = moe.alloc_workspace(cfg)
        rows = slice(r * Tr, (r + 1) * Tr)
        x = inp["x"][rows].contiguous()
        st = dict(cfg=cfg, idx=torch.empty(Tr * k, dtype=torch.int32, device=DEV),
                  gates=torch.empty(Tr * k, dtype=F32, device=DEV),
                  offsets=torch.empty(n + 1, dtype=torch.int32, device=DEV),
                  perm=torch.empty(Tr * k, dtype=torch.int32, device=DEV),
                  inv=torch.empty(Tr * k, dtype=torch.int32, device=DEV),
                  x_perm=torch.empty((Tr * k, d), dtype=shape.expert_dtype, device=DEV))
        load = torch.empty(n, dtype=F32, device=DEV)
        moe.moe_gate(cfg, x, inp["W_g"], inp["W_noise"], inp["eps"][rows].contiguous(), inp["b_g"],
                     st["idx"], st["gates"], torch.empty(Tr, dtype=torch.uint8, device=DEV), load,
                     None, ws)
        moe.moe_dispatch(cfg, st["idx"], x, st["offsets"], st["perm"], st["inv"], st["x_perm"], ws)
        ranks.append(st)
    all_offsets = torch.stack([st["offsets"] for st in ranks]).cpu().numpy()
    plans = [moe.moe_ep_plan(world, r, n, all_offsets) for r in range(world)]
    ydt = moe.expert_rows_dtype(ranks[0]["cfg"])
    y_back = [[None] * world for _ in range(world)]         # [source][expert rank]
    for q in range(world):                                  # the rank holding experts of q
        send_q, recv_q, plan = plans[q]
        parts = []
        for s in range(world):                              # the all-to-all: s's block for q
            o = all_offsets[s]
            parts.append(ranks[s]["x_perm"][o[q * nl]:o[(q + 1) * nl]])
        x_recv = torch.cat(parts)
        rows = x_recv.shape[0]
        assert rows == int(recv_q.sum())
        y_recv = torch.empty((rows, d), dtype=ydt, device=DEV)
        if rows:                                            # a rank whose experts got no row
            plan_dev = torch.from_numpy(plan).to(DEV)
            x_local = torch.empty_like(x_recv)
            moe.moe_ep_regroup(world, nl, plan_dev, x_recv, x_local, True)
            B2 = 2 * world * nl + 1
            fc = moe.make_config(rows, d, nl, shape.h, 1, shape.x_dtype, shape.expert_dtype,
                                 flags=flags & 3)
            y_local = torch.empty((rows, d), dtype=ydt, device=DEV)
            moe.moe_expert_ffn(fc, x_local, plan_dev[B2:B2 + nl + 1].contiguous(),
                               inp["W_in"][q * nl:(q + 1) * nl].contiguous(),
                               inp["W_out"][q * nl:(q + 1) * nl].contiguous(), y_local,
                               moe.alloc_workspace(fc))
            moe.moe_ep_regroup(world, nl, plan_dev, y_local, y_recv, False)
        starts = np.concatenate([[0], np.cumsum(recv_q)])
        for s in range(world):
            y_back[s][q] = y_recv[starts[s]:starts[s + 1]]
    ys = []
    for r, st in enumerate(ranks):
        y_perm = torch.cat(y_back[r])                       # the return all-to-all
        assert y_perm.shape[0] == Tr * k
        y = torch.empty((Tr, d), dtype=F32, device=DEV)
        moe.moe_combine(st["cfg"], y_perm, st["inv"], st["gates"], y)
        ys.append(y)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    return torch.cat(ys), torch.cat([st["idx"] for st in ranks])


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("shape,flags", [
    (S.FlatShape("ep-bf16", 4096, 512, 64, 1024, 4), ROW),
    (S.FlatShape("ep-fp32", 1024, 64, 16, 128, 2, F32, F32), 0),
    (S.FlatShape("ep-skewed-empty", 2048, 256, 32, 256, 2), ROW)],
    ids=["bf16", "fp32", "sparse"])
def test_expert_parallel_forward(shape, flags, world):
    inp = S.make_flat_inputs(shape, seed=67, device=DEV)
    if shape.name == "ep-skewed-empty":                     # whole ranks' experts left empty
        inp["b_g"] = torch.zeros(shape.n, device=DEV)
        inp["b_g"][: shape.n // 2] = -30.0
    y_ep, idx = _ep_forward(shape, inp, world, flags)
    if shape.name == "ep-skewed-empty":
        assert (idx.cpu() >= shape.n // 2).all()            # ranks holding the first half idle
    whole = _forward(_cfg(shape, shape.T, flags), inp)
    assert torch.equal(idx, whole["idx"])
    assert torch.equal(y_ep, whole["y"])
    a = oracle_arrays(inp)
    ref = O.moe_forward(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"], a["W_out"],
                        shape.k, 0.0, a["b_g"], kept=kept_of(idx.cpu().numpy(), shape.k))
    assert_y(np64(y_ep), ref["y"], shape.expert_dtype == BF16)


def test_ep_regroup_round_trip_and_checks():
    """Regrouping there and back restores every row; misaligned rows are refused."""
    world, n = 3, 9
    offs = np.array([[0, 5, 5, 9, 30, 31, 40, 41, 41, 50],
                     [0, 0, 7, 8, 8, 20, 21, 22, 40, 44],
                     [0, 1, 2, 3, 4, 5, 6, 7, 8, 9]], dtype=np.int32)
    for rank in range(world):
        send, recv, plan = moe.moe_ep_plan(world, rank, n, offs)
        rows = int(recv.sum())
        x = torch.randn((rows, 24), device=DEV).to(torch.bfloat16)     # 48-byte rows
        mid, back = torch.empty_like(x), torch.empty_like(x)
        p = torch.from_numpy(plan).to(DEV)
        moe.moe_ep_regroup(world, n // world, p, x, mid, True)
        moe.moe_ep_regroup(world, n // world, p, mid, back, False)
        torch.cuda.synchronize()
        assert torch.equal(back, x)
        # expert-major order: each local expert's rows from every source, sources ascending
        B = world * (n // world)
        src, dst = plan[:B], plan[B:2 * B + 1]
        for q in range(B):
            c = dst[q + 1] - dst[q]
            assert torch.equal(mid[dst[q]:dst[q] + c], x[src[q]:src[q] + c])
    odd = torch.empty((4, 3), dtype=torch.bfloat16, device=DEV)        # 6-byte rows
    with pytest.raises(moe.MoeError, match="UNSUPPORTED"):
        moe.moe_ep_regroup(world, 3, torch.zeros(moe.ep_plan_size(3, 3), dtype=torch.int32,
                                                  device=DEV), odd, torch.empty_like(odd), True)
