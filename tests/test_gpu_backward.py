"""The backward pass (moe_backward, through the C ABI) against the fp64 oracle's
backward, which is pinned by finite differences of the forward pass.

Tolerances: the all-fp32 workload runs fp32 arithmetic throughout, so every gradient
is held to max-abs <= 1e-4 RMS of the oracle's (the layer output's fp32 bound).  With
bf16 experts every gradient is linear in quantities that carry the forward's bf16
rounding (the bf16 hidden layer, the fp16 expert outputs in the gate gradient), so
they are held to the layer output's bf16 bound, max-abs <= 2e-2 RMS, and the expert
weight gradients also elementwise: dW_out[e] = a_e^T dE_e and dW_in[e] = x_e^T dU_e
multiply operands of which at most two carry a bf16 rounding of 2^-9 relative (the
hidden layer a; dE and dU, which the tensor-core data gradients keep in bf16), so each
element is held to 2^-7 (|a_e|^T |dE_e|), resp. 2^-7 (|x_e|^T |dU_e|) (twice that),
which also holds where an expert has one or two rows and the products are heavy-tailed
against the tensor's RMS.

ReLU'(u) is a branch that floating point decides: where |u| is within the fp32
accumulation error of the forward's first product, tau = d 2^-22 (|x| |W_in|) (the
bound for a d-term dot product whose additions truncate to fp32, 2^-23 each, as the
tensor core's do, doubled), the GPU and the oracle may legitimately take
different branches.  The oracle marks those (row, hidden) elements and each element of
dW_in, dx and dW_out gets, on top of its rounding bound, the absolute value of those
elements' contributions (|x|^T |dA| on them, |dA| |W_in|^T, tau |dE|), so exactly the
ambiguous terms are excused and nothing else.  The seeds have no near tie at the k-th
place (checked through moe_forward's selection), so the kept experts, which the
gradient depends on, are the oracle's.
"""
import numpy as np
import pytest
import torch

import sparsely_gated_mixture_03_b300 as moe
from sparsely_gated_mixture_03_b300 import synthetic as S
from oracle import moe_oracle as O
from gpu_helpers import check_selection, np64, oracle_arrays

pytestmark = pytest.mark.gpu

DEV = "cuda"
F32, BF16 = torch.float32, torch.bfloat16

SHAPES = [
    S.WORKLOADS["tiny-fp32"],
    S.FlatShape("k-equals-n", 77, 64, 6, 64, 6, F32, F32),
    S.FlatShape("ragged-bf16", 1000, 128, 40, 192, 3),
    S.FlatShape("k1-bf16", 300, 64, 16, 128, 1),
    S.FlatShape("big-600", 600, 64, 600, 64, 2),
    S.FlatShape("tc-256x256", 2000, 256, 64, 256, 2),
    S.WORKLOADS["moe256"],
]


def _run(shape, inp, floor=0.0, w_imp=0.1, w_load=0.1, seed=5):
    T, d, n, h, k = shape.T, shape.d, shape.n, shape.h, shape.k
    cfg = moe.make_config(T, d, n, h, k, shape.x_dtype, shape.expert_dtype, std_floor=floor,
                          w_importance=w_imp, w_load=w_load)
    dy = torch.randn((T, d), generator=torch.Generator().manual_seed(seed)).to(DEV)
    out = dict(dx=torch.full((T, d), float("nan"), device=DEV),
               dW_g=torch.full((d, n), float("nan"), device=DEV),
               dW_noise=torch.full((d, n), float("nan"), device=DEV),
               db_g=torch.full((n,), float("nan"), device=DEV),
               dW_in=torch.full((n, d, h), float("nan"), device=DEV),
               dW_out=torch.full((n, h, d), float("nan"), device=DEV))
    ws = moe.alloc_backward_workspace(cfg)
    moe.moe_backward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], inp["b_g"], inp["W_in"],
                     inp["W_out"], dy, out["dx"], out["dW_g"], out["dW_noise"], out["db_g"],
                     out["dW_in"], out["dW_out"], ws)
    # the kept experts of this input, for the no-near-tie precondition
    fws = moe.alloc_workspace(cfg)
    idx = torch.empty(T * k, dtype=torch.int32, device=DEV)
    gates = torch.empty(T * k, dtype=F32, device=DEV)
    moe.moe_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], inp["b_g"], inp["W_in"],
                    inp["W_out"], torch.empty((T, d), device=DEV), torch.empty(3, device=DEV),
                    idx=idx, gates=gates, workspace=fws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    return out, dy, idx, gates


def _check(shape, inp, out, dy, idx, gates, floor=0.0, w_imp=0.1, w_load=0.1):
    a = oracle_arrays(inp)
    ref_g = O.gating(a["x"], a["W_g"], a["W_noise"], a["eps"], shape.k, floor, a["b_g"])
    same = check_selection(idx.cpu().numpy(), np64(gates), ref_g, shape.k)
    assert same.all(), "a near tie: the seed must keep the oracle's experts"
    ref = O.moe_backward(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"], a["W_out"], shape.k,
                         np64(dy), floor, a["b_g"], w_imp, w_load)
    bf16 = shape.expert_dtype == BF16
    bound = 2e-2 if bf16 else 1e-4
    # the ReLU-branch slack of every element (see the module docstring) and the bf16
    # bound of dW_out, per expert from the oracle's own routing
    idx_r, G = ref_g["idx"], ref_g["gates"]
    dyn = np64(dy)
    x, W_in, W_out = a["x"], a["W_in"], a["W_out"]
    slack = dict(dx=np.zeros_like(ref["dx"]), dW_in=np.zeros_like(ref["dW_in"]),
                 dW_out=np.zeros_like(ref["dW_out"]))
    out_lim = np.zeros_like(ref["dW_out"])
    in_lim = np.zeros_like(ref["dW_in"])
    for e in np.unique(idx_r):
        tt, jj = np.nonzero(idx_r == e)
        xe = x[tt]
        u = xe @ W_in[e]
        tau = shape.d * 2.0 ** -22 * (np.abs(xe) @ np.abs(W_in[e]))
        amb = np.abs(u) <= tau
        dE = G[tt, jj][:, None] * dyn[tt]
        dA = np.abs(dE @ W_out[e].T) * amb
        slack["dW_in"][e] = np.abs(xe).T @ dA
        np.add.at(slack["dx"], tt, dA @ np.abs(W_in[e]).T)
        slack["dW_out"][e] = (tau * amb).T @ np.abs(dE)
        out_lim[e] = 2.0 ** -7 * (np.abs(np.maximum(u, 0.0)).T @ np.abs(dE))
        dU_ref = (dE @ W_out[e].T) * (u > 0.0)
        in_lim[e] = 2.0 ** -7 * (np.abs(xe).T @ np.abs(dU_ref))
    names = ["dx", "dW_g", "dW_noise", "dW_in", "dW_out"] + (["db_g"] if a["b_g"] is not None else [])
    for name in names:
        got, r = np64(out[name]), ref[name]
        rms = float(np.sqrt(np.mean(r * r)))
        if name == "dW_out" and bf16:
            lim = out_lim + slack["dW_out"] + 1e-7
        elif name == "dW_in" and bf16:
            lim = np.maximum(bound * rms, in_lim) + slack["dW_in"]
        else:
            lim = bound * rms + slack.get(name, 0.0)
        bad = np.abs(got - r) > lim
        assert not bad.any(), (f"{name}: {int(bad.sum())} elements beyond the bound, worst "
                               f"{float(np.max(np.abs(got - r) - lim)):.3e} over (RMS {rms:.3e})")
    empty = np.setdiff1d(np.arange(shape.n), np.unique(idx_r))
    assert not np64(out["dW_out"])[empty].any() and not np64(out["dW_in"])[empty].any()


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_backward(shape):
    inp = S.make_flat_inputs(shape, seed=51, device=DEV)
    inp["b_g"] = torch.randn(shape.n, generator=torch.Generator().manual_seed(52)).to(DEV) * 0.1
    out, dy, idx, gates = _run(shape, inp)
    _check(shape, inp, out, dy, idx, gates)


def test_backward_floor_weights_and_no_noise():
    """The noise floor, other loss weights, and the noiseless gate (eps = NULL)."""
    shape = S.FlatShape("ragged-bf16", 1000, 128, 40, 192, 3)
    inp = S.make_flat_inputs(shape, seed=53, device=DEV)
    out, dy, idx, gates = _run(shape, inp, floor=0.01, w_imp=0.3, w_load=0.7)
    _check(shape, inp, out, dy, idx, gates, floor=0.01, w_imp=0.3, w_load=0.7)
    inp0 = dict(inp, eps=None)
    out, dy, idx, gates = _run(shape, inp0)
    inp0z = dict(inp, eps=torch.zeros_like(inp["eps"]))
    _check(shape, inp0z, out, dy, idx, gates)


def test_backward_refuses_capacity_and_switch():
    cfg = moe.make_config(64, 64, 8, 64, 2, capacity=4)
    with pytest.raises(moe.MoeError, match="UNSUPPORTED"):
        z = lambda *s: torch.zeros(*s, device=DEV)
        moe.moe_backward(cfg, z(64, 64).to(BF16), z(64, 8), z(64, 8), z(64, 8), None,
                         z(8, 64, 64).to(BF16), z(8, 64, 64).to(BF16), z(64, 64), z(64, 64),
                         z(64, 8), z(64, 8), None, z(8, 64, 64), z(8, 64, 64),
                         torch.empty(moe.backward_workspace_size(cfg), dtype=torch.uint8,
                                     device=DEV))


def test_backward_timed_matches_backward():
    """moe_backward_timed gives the same gradients and records its six events."""
    shape = S.FlatShape("ragged-bf16", 1000, 128, 40, 192, 3)
    inp = S.make_flat_inputs(shape, seed=57, device=DEV)
    cfg = moe.make_config(shape.T, shape.d, shape.n, shape.h, shape.k)
    ws = moe.alloc_backward_workspace(cfg)
    dy = torch.randn((shape.T, shape.d), generator=torch.Generator().manual_seed(9)).to(DEV)
    outs = []
    for timed in (False, True):
        f = dict(device=DEV, dtype=F32)
        o = [torch.empty((shape.T, shape.d), **f), torch.empty((shape.d, shape.n), **f),
             torch.empty((shape.d, shape.n), **f), None,
             torch.empty((shape.n, shape.d, shape.h), **f),
             torch.empty((shape.n, shape.h, shape.d), **f)]
        a = (cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], None, inp["W_in"],
             inp["W_out"], dy, *o, ws)
        if timed:
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
            moe.moe_backward_timed(*a, ev)
        else:
            moe.moe_backward(*a)
        torch.cuda.synchronize()
        outs.append(o)
    for g0, g1 in zip(outs[0], outs[1]):
        if g0 is not None:
            assert torch.equal(g0, g1)
    assert all(ev[i].elapsed_time(ev[i + 1]) >= 0.0 for i in range(5))


def test_backward_empty_experts_tensor_cores():
    """Skewed routing on the tensor-core weight-gradient path (d = h = 256): a bias of
    -30 keeps a quarter of the experts, spread over the expert range, from ever being
    chosen, so their weight-gradient units load nothing and must store exact zeros,
    while their neighbours' gradients stay within the bounds."""
    shape = S.FlatShape("tc-256x256-empty", 2000, 256, 64, 256, 2)
    inp = S.make_flat_inputs(shape, seed=59, device=DEV)
    b = torch.zeros(shape.n)
    b[::4] = -30.0
    inp["b_g"] = b.to(DEV)
    out, dy, idx, gates = _run(shape, inp)
    chosen = np.unique(idx.cpu().numpy())
    assert not np.isin(np.arange(0, shape.n, 4), chosen).any()
    _check(shape, inp, out, dy, idx, gates)
