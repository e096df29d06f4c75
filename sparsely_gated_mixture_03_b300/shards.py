"""The layer over several GPUs, one process per GPU ("Keeping each expert's batch
large" of "Mixture of Experts: Outrageously Large Neural Networks", intuitivepapers.ai:
the gate and the other layers replicated data-parallel, the experts spread over the
devices, every routed row sent to the device that holds its expert).

Only the collectives live here (torch.distributed: NCCL between GPUs, gloo in the
CPU tests) and the host bookkeeping around them; every step of the layer itself is a
library kernel behind the C ABI (include/moe.h).

* Data parallel: each rank runs the whole layer on its own tokens; the balancing
  losses are batch quantities, so the ranks add their Importance and Load vectors
  (one all-reduce of 2n floats) and form the losses from the totals
  (``global_losses``).
* Expert parallel: rank r holds experts [r n/world, (r+1) n/world).  Each rank gates
  and dispatches its own tokens; the ranks all-gather their dispatch offsets, plan
  the exchange on the host (``moe_ep_plan``), send every routed row to its expert's
  rank (all-to-all), regroup the arrivals expert-major, run their experts, regroup
  back, return the outputs (all-to-all) and combine locally
  (``ExpertParallelLayer``).
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import binding as B


def allreduce_sums(sums: torch.Tensor, group=None) -> None:
    """Add every rank's [importance; load] buffer (2n floats) in place."""
    dist.all_reduce(sums, op=dist.ReduceOp.SUM, group=group)


def global_losses(cfg_global, sums: torch.Tensor, losses: torch.Tensor, group=None,
                  stream=None) -> None:
    """The whole batch's balancing losses from every rank's sums.  ``sums`` is the
    rank's [importance; load] buffer of 2n floats (moe_forward's importance and load
    outputs as its two halves); it holds the totals afterwards.  ``cfg_global.T`` is
    the whole batch's token count (read by the Switch gate's loss only)."""
    allreduce_sums(sums, group)
    n = cfg_global.n
    B.moe_losses_from_sums(cfg_global, sums[:n], sums[n:], losses, stream)


def gather_offsets(offsets: torch.Tensor, world: int, group=None) -> np.ndarray:
    """Every rank's dispatch offsets [world, n+1] on the host: one all-gather of
    n+1 int32 per rank, then one copy to the host (a synchronisation: the
    all-to-all split sizes are host numbers)."""
    out = offsets.new_empty(world * offsets.numel())
    dist.all_gather_into_tensor(out, offsets, group=group)
    return out.cpu().numpy().reshape(world, offsets.numel())


def exchange_plan(offsets: torch.Tensor, world: int, rank: int, n: int, group=None):
    """(send_rows, recv_rows, plan) of this rank: numpy int32 (``moe_ep_plan``)."""
    return B.moe_ep_plan(world, rank, n, gather_offsets(offsets, world, group))


def exchange_rows(send: torch.Tensor, send_rows, recv_rows, group=None,
                  out: torch.Tensor | None = None) -> torch.Tensor:
    """All-to-all of row blocks: rank r's rows [sum of send_rows[:q], + send_rows[q])
    go to rank q; returns the rows received, source rank major (into ``out`` when
    given: sum(recv_rows) rows)."""
    recv = out if out is not None else \
        send.new_empty((int(np.sum(recv_rows)),) + tuple(send.shape[1:]))
    dist.all_to_all_single(recv, send, output_split_sizes=[int(v) for v in recv_rows],
                           input_split_sizes=[int(v) for v in send_rows], group=group)
    return recv


class ExpertParallelLayer:
    """One rank of the expert-parallel layer.

    cfg: this rank's moe_config (T = its tokens, n = every expert of the layer,
    bf16 or fp32 as usual); W_in_local [n/world, d, h] and W_out_local
    [n/world, h, d]: the weights of the experts this rank holds.  The gate's weights
    are replicated.  ``forward`` writes y [T, d] for this rank's tokens and the
    whole batch's losses (every rank must call it, in the same order)."""

    def __init__(self, cfg, world: int, rank: int, W_in_local, W_out_local, group=None):
        if cfg.n % world:
            raise ValueError("the expert count must be a multiple of the world size")
        if cfg.flags & B.FLAG_SWITCH_GATE:
            raise ValueError("the expert-parallel layer takes the noisy top-k gate")
        self.cfg, self.world, self.rank, self.group = cfg, world, rank, group
        self.n_local = cfg.n // world
        self.W_in, self.W_out = W_in_local, W_out_local
        dev = W_in_local.device
        T, d, n, k = cfg.T, cfg.d, cfg.n, cfg.k
        self.ws = B.alloc_workspace(cfg)
        self.idx = torch.empty(T * k, dtype=torch.int32, device=dev)
        self.gates = torch.empty(T * k, dtype=torch.float32, device=dev)
        self.tie = torch.empty(T, dtype=torch.uint8, device=dev)
        self.offsets = torch.empty(n + 1, dtype=torch.int32, device=dev)
        self.perm = torch.empty(T * k, dtype=torch.int32, device=dev)
        self.inv = torch.empty(T * k, dtype=torch.int32, device=dev)
        self.x_perm = torch.empty((T * k, d), dtype=W_in_local.dtype, device=dev)
        self.sums = torch.empty(2 * n, dtype=torch.float32, device=dev)
        self.local_losses = torch.empty(3, dtype=torch.float32, device=dev)
        self.ffn_ws = None
        self.ffn_rows = 0

    def _ffn_workspace(self, rows: int):
        if self.ffn_ws is None or rows > self.ffn_rows:
            c = self.cfg
            self.ffn_rows = max(rows, 2 * self.ffn_rows)
            fc = B.make_config(self.ffn_rows, c.d, self.n_local, c.h, 1,
                               B._xdt(c), B._edt(c), flags=c.flags & 3)
            self.ffn_ws = B.alloc_workspace(fc)
        return self.ffn_ws

    def forward(self, x, W_g, W_noise, eps, b_g, y, losses, stream=None):
        c, world, nl = self.cfg, self.world, self.n_local
        n, d = c.n, c.d
        imp, load = self.sums[:n], self.sums[n:]
        B.moe_gate(c, x, W_g, W_noise, eps, b_g, self.idx, self.gates, self.tie, load, None,
                   self.ws, stream)
        B.moe_dispatch(c, self.idx, x, self.offsets, self.perm, self.inv, self.x_perm, self.ws,
                       stream)
        B.moe_balance_losses(c, self.gates, self.perm, self.offsets, load, imp,
                             self.local_losses, stream)
        send, recv, plan = exchange_plan(self.offsets, world, self.rank, n, self.group)
        plan_dev = torch.from_numpy(plan).to(x.device)
        x_recv = exchange_rows(self.x_perm[:int(send.sum())], send, recv, self.group)
        rows = int(recv.sum())
        ydt = B.expert_rows_dtype(c)
        y_recv = torch.empty((rows, d), dtype=ydt, device=x.device)
        if rows:
            x_local = torch.empty_like(x_recv)
            B.moe_ep_regroup(world, nl, plan_dev, x_recv, x_local, True, stream)
            fc = B.make_config(rows, d, nl, c.h, 1, B._xdt(c), B._edt(c), flags=c.flags & 3)
            y_local = torch.empty((rows, d), dtype=ydt, device=x.device)
            B2 = 2 * world * nl + 1
            B.moe_expert_ffn(fc, x_local, plan_dev[B2:B2 + nl + 1], self.W_in, self.W_out,
                             y_local, self._ffn_workspace(rows), stream)
            B.moe_ep_regroup(world, nl, plan_dev, y_local, y_recv, False, stream)
        y_perm = torch.empty((c.T * c.k, d), dtype=ydt, device=x.device)
        exchange_rows(y_recv, recv, send, self.group, out=y_perm[:int(send.sum())])
        B.moe_combine(c, y_perm, self.inv, self.gates, y, stream)
        cg = B.make_config(c.T * world, c.d, c.n, c.h, c.k, B._xdt(c), B._edt(c), c.std_floor,
                           c.w_importance, c.w_load, c.flags, c.capacity)
        global_losses(cg, self.sums, losses, self.group, stream)
