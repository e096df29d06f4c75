"""Hierarchical MoE ("Hierarchical MoE" section of "Mixture of Experts: Outrageously
Large Neural Networks", intuitivepapers.ai) through the C ABI against the fp64 oracle.
Needs a B300; run with ``pytest -m gpu``.

Element by element at sizes the oracle finishes in seconds (several 128-row tiles
per group and ragged group sizes), the reductions a = 1 (a flat layer over b
experts) and b = 1 (a flat layer over the a groups) bit-exactly against the flat
entry point, and the 128 x 128 workload at full size on sampled tokens plus its
batch sums.

Tolerances as for the flat layer: kept experts exact except on rows where a gate
has a near tie at its k-th place (there the oracle checks that the GPU's choice is
a valid tie-break and is rerun with it), product gates, the Importance / Load
vectors and the losses within 1e-5 relative, y within 2e-2 RMS(y), on every row.
"""
import numpy as np
import pytest
import torch

import sparsely_gated_mixture_03_b300 as moe
from sparsely_gated_mixture_03_b300 import synthetic as S
from oracle import moe_oracle as O
from gpu_helpers import assert_rel, assert_y, np64, scaled_err

pytestmark = pytest.mark.gpu

DEV = "cuda"
F32 = torch.float32


class LazyExperts:
    """Expert weights read one expert at a time from the device copy."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        return np64(self.t[int(e)])


def _run(shape, inp, std_floor=0.0):
    cfg = moe.make_hier_config(shape.T, shape.d, shape.a, shape.b, shape.h, shape.k1, shape.k2,
                               std_floor=std_floor)
    ws = moe.alloc_hier_workspace(cfg)
    T, a, b, K = shape.T, shape.a, shape.b, shape.k1 * shape.k2
    out = dict(y=torch.empty((T, shape.d), dtype=F32, device=DEV),
               losses=torch.empty(3, dtype=F32, device=DEV),
               idx=torch.empty(T * K, dtype=torch.int32, device=DEV),
               gates=torch.empty(T * K, dtype=F32, device=DEV),
               tie1=torch.empty(T, dtype=torch.uint8, device=DEV),
               tie2=torch.empty(T * shape.k1, dtype=torch.uint8, device=DEV),
               importance1=torch.empty(a, dtype=F32, device=DEV),
               load1=torch.empty(a, dtype=F32, device=DEV),
               importance=torch.empty(a * b, dtype=F32, device=DEV),
               load2=torch.empty(a * b, dtype=F32, device=DEV))
    moe.moe_hier_forward(cfg, inp["x"], inp["W_g1"], inp["W_noise1"], inp["eps1"], inp["W_g2"],
                         inp["W_noise2"], inp["eps2"], inp["W_in"], inp["W_out"], out["y"],
                         out["losses"], out["idx"], out["gates"], out["tie1"], out["tie2"],
                         out["importance1"], out["load1"], out["importance"], out["load2"],
                         workspace=ws)
    assert moe.moe_get_device_error() == 0
    return out


def _check_rows(got_idx, got_gates, own, ref, K):
    """Per row: the kept (expert, product gate) pairs.  Rows without a near tie in
    either gate keep exactly the oracle's own experts (``own``); every row's
    product gates match, within 1e-5, those the oracle forms over the GPU's kept
    experts (``ref``, which it accepts only as a valid tie-break of its own
    logits).  Returns the mask of rows whose kept set equals the oracle's own."""
    gi = np.asarray(got_idx).reshape(-1, K)
    gg = np.asarray(got_gates, np.float64).reshape(-1, K)
    tie = own["tie1"] | own["tie2"].any(axis=1)
    same = np.array([set(gi[t]) == set(own["idx"][t]) for t in range(gi.shape[0])])
    bad = np.nonzero(~tie & ~same)[0]
    assert bad.size == 0, f"{bad.size} rows without a near tie keep other experts: {bad[:5]}"
    assert np.array_equal(ref["idx"], gi)
    assert_rel(gg, ref["gates"], "product gates")
    assert np.allclose(gg.sum(axis=1), 1.0, atol=1e-5)
    return same


def _oracle(inp, shape, rows=None, with_y=True, kept=None, std_floor=0.0):
    a = {k: (np64(v) if k not in ("W_in", "W_out") else LazyExperts(v)) for k, v in inp.items()}
    return O.hier_forward(a["x"], a["W_g1"], a["W_noise1"], a["eps1"], a["W_g2"], a["W_noise2"],
                          a["eps2"], a["W_in"], a["W_out"], shape.k1, shape.k2, std_floor,
                          rows=rows, with_y=with_y, kept=kept)


def _check_sums(got, ref, what=""):
    """The four reported vectors and the losses (the primary gate's CV^2 pair)."""
    for name, key in (("importance1", "importance1"), ("load1", "load1"),
                      ("importance", "importance_flat"), ("load2", "load2")):
        assert_rel(np64(got[name]), ref[key], what + name)
    ci, cl, aux = O.balance_losses(ref["importance1"], ref["load1"], 0.1, 0.1)
    assert_rel(np64(got["losses"]), [ci, cl, aux], what + "losses")


SMALL = [
    S.HierShape("hier-8x16", 1000, 128, 8, 16, 192, 2, 2),
    S.HierShape("hier-3x40-k1x3", 700, 64, 3, 40, 128, 1, 3),
    S.HierShape("hier-5x9-k2x1", 333, 64, 5, 9, 64, 2, 1),
    S.HierShape("hier-single-token", 1, 64, 2, 4, 64, 2, 2),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_hier_forward(shape):
    inp = S.make_hier_inputs(shape, seed=31, device=DEV)
    got = _run(shape, inp)
    K = shape.k1 * shape.k2
    gi = got["idx"].cpu().numpy().reshape(-1, K).astype(np.int64)
    own = _oracle(inp, shape, with_y=False)
    ref = _oracle(inp, shape, kept=gi)
    _check_rows(gi, np64(got["gates"]), own, ref, K)
    assert_y(np64(got["y"]), ref["y"], True)
    # the GPU's primary near-tie flag agrees with the oracle's except within fp32 noise of 1e-5
    dis = np.nonzero(got["tie1"].cpu().numpy().astype(bool) != own["tie1"])[0]
    assert all(abs(own["gap1"][t] - O.TIE_GAP) < 2e-6 for t in dis)
    _check_sums(got, ref)
    # invariants of the product gates: Importance sums to T
    assert abs(np64(got["importance"]).sum() - shape.T) < 1e-3 * max(1, shape.T) ** 0.5


def test_hier_one_group_equals_flat():
    """a = 1, k1 = 1: every token goes to group 0 with gate 1 and the secondary gate
    is the flat gate over b experts: bit-identical to moe_forward's outputs."""
    shape = S.HierShape("hier-1x24", 900, 128, 1, 24, 128, 1, 3)
    inp = S.make_hier_inputs(shape, seed=41, device=DEV)
    got = _run(shape, inp)
    flat = S.FlatShape("flat-24", shape.T, shape.d, shape.b, shape.h, shape.k2)
    cfg = moe.make_config(flat.T, flat.d, flat.n, flat.h, flat.k)
    ws = moe.alloc_workspace(cfg)
    T, K = shape.T, shape.k2
    y = torch.empty((T, shape.d), dtype=F32, device=DEV)
    losses = torch.empty(3, dtype=F32, device=DEV)
    idx = torch.empty(T * K, dtype=torch.int32, device=DEV)
    gates = torch.empty(T * K, dtype=F32, device=DEV)
    imp = torch.empty(shape.b, dtype=F32, device=DEV)
    load = torch.empty(shape.b, dtype=F32, device=DEV)
    moe.moe_forward(cfg, inp["x"], inp["W_g2"][0].contiguous(), inp["W_noise2"][0].contiguous(),
                    inp["eps2"].reshape(T, shape.b).contiguous(), None, inp["W_in"], inp["W_out"],
                    y, losses, idx, gates, None, imp, load, ws)
    assert moe.moe_get_device_error() == 0
    assert torch.equal(got["idx"], idx)
    assert torch.equal(got["gates"], gates)
    assert torch.equal(got["y"], y)
    # Load and Importance: the same tile sums, added over tiles in another fixed order
    assert_rel(np64(got["load2"]), np64(load), "load")
    assert_rel(np64(got["importance"]), np64(imp), "importance")
    assert float(got["importance1"][0]) == T and float(got["load1"][0]) == T


def test_hier_one_expert_per_group_equals_flat_over_groups():
    """b = 1, k2 = 1: the layer is a flat layer over the a groups; the product gate
    is the primary gate (times exactly 1)."""
    shape = S.HierShape("hier-20x1", 1200, 64, 20, 1, 128, 3, 1)
    inp = S.make_hier_inputs(shape, seed=43, device=DEV)
    got = _run(shape, inp)
    cfg = moe.make_config(shape.T, shape.d, shape.a, shape.h, shape.k1)
    ws = moe.alloc_workspace(cfg)
    T, K = shape.T, shape.k1
    y = torch.empty((T, shape.d), dtype=F32, device=DEV)
    losses = torch.empty(3, dtype=F32, device=DEV)
    idx = torch.empty(T * K, dtype=torch.int32, device=DEV)
    gates = torch.empty(T * K, dtype=F32, device=DEV)
    imp = torch.empty(shape.a, dtype=F32, device=DEV)
    load = torch.empty(shape.a, dtype=F32, device=DEV)
    moe.moe_forward(cfg, inp["x"], inp["W_g1"], inp["W_noise1"], inp["eps1"], None, inp["W_in"],
                    inp["W_out"], y, losses, idx, gates, None, imp, load, ws)
    assert moe.moe_get_device_error() == 0
    assert torch.equal(got["idx"], idx)
    assert torch.equal(got["gates"], gates)
    assert torch.equal(got["y"], y)
    assert torch.equal(got["losses"], losses)
    assert torch.equal(got["importance1"], imp) and torch.equal(got["load1"], load)
    # one expert per group: its secondary load is the group's row count (P = 1, k = n)
    counts = np.bincount(idx.cpu().numpy(), minlength=shape.a)
    assert np.array_equal(np64(got["load2"]), counts.astype(np.float64))


def test_hier_noise_floor_and_determinism():
    shape = S.HierShape("hier-6x32", 800, 64, 6, 32, 64, 2, 2)
    inp = S.make_hier_inputs(shape, seed=47, device=DEV)
    a = _run(shape, inp, std_floor=0.01)
    b = _run(shape, inp, std_floor=0.01)
    for k in a:
        assert torch.equal(a[k], b[k]), k
    gi = a["idx"].cpu().numpy().reshape(-1, 4).astype(np.int64)
    own = _oracle(inp, shape, with_y=False, std_floor=0.01)
    ref = _oracle(inp, shape, kept=gi, std_floor=0.01)
    _check_rows(gi, np64(a["gates"]), own, ref, 4)
    assert_y(np64(a["y"]), ref["y"], True)
    _check_sums(a, ref)


@pytest.mark.slow
def test_hier128x128_full_size_sampled():
    """128 groups x 128 experts, T = 65536 (about 34 GB of bf16 expert weights):
    kept experts, product gates and y on 512 sampled tokens; the Importance and
    Load vectors against the oracle's full-batch sums."""
    shape = S.WORKLOADS["hier128x128"]
    inp = S.make_hier_inputs(shape, seed=53, device=DEV)
    got = _run(shape, inp)
    K = shape.k1 * shape.k2
    kept = got["idx"].cpu().numpy().reshape(-1, K).astype(np.int64)
    rows = np.sort(np.random.default_rng(1).choice(shape.T, 512, replace=False))
    own = _oracle(inp, shape, rows=rows, with_y=False)
    ref = _oracle(inp, shape, rows=rows, kept=kept[rows])
    gg = np64(got["gates"]).reshape(-1, K)[rows]
    _check_rows(kept[rows], gg, own, ref, K)
    assert_y(np64(got["y"])[rows], ref["y"], True)
    # batch sums over all T tokens, with the GPU's kept set on any near-tie row
    full = _oracle(inp, shape, with_y=False, kept=kept)
    _check_sums(got, full, "full batch: ")
    assert scaled_err(np64(got["importance"]).sum(), shape.T) < 1e-5
    counts = np.bincount(got["idx"].cpu().numpy(), minlength=shape.a * shape.b)
    assert counts.sum() == shape.T * K
