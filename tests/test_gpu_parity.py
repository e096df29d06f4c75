"""CUDA path (through the C ABI) against the fp64 oracle, stage by stage and
for the whole layer.  Needs a B300; run with ``pytest -m gpu``.

Element-by-element comparisons at sizes the oracle finishes in seconds
(several tiles and a ragged tail), the full 32- and 256-expert workloads in
full, and the 4096-expert Zipf workload on sampled tokens plus its batch sums.
"""
import numpy as np
import pytest
import torch

import sparsely_gated_mixture_03_b300 as moe
from sparsely_gated_mixture_03_b300 import synthetic as S
from oracle import moe_oracle as O
from gpu_helpers import (assert_rel, assert_y, check_selection, config_for, kept_of, np64,
                         oracle_arrays, own_selection, run_gate)

pytestmark = pytest.mark.gpu

DEV = "cuda"
F32, BF16 = torch.float32, torch.bfloat16

SMALL = [
    S.WORKLOADS["tiny-fp32"],
    S.FlatShape("ragged-bf16", 1000, 128, 40, 192, 3),
    S.FlatShape("k-equals-n", 77, 64, 6, 64, 6, F32, F32),
    S.FlatShape("k1-bf16", 300, 64, 16, 128, 1),
    S.FlatShape("single-token", 1, 64, 1, 64, 1, F32, F32),
    S.FlatShape("k8-bf16", 513, 64, 70, 128, 8),
    # 250 experts: the column scan's cluster of eight CTAs with a partial last CTA
    S.FlatShape("n250-bf16", 1500, 64, 250, 64, 3),
]
FULL = [S.WORKLOADS["moe32"], S.WORKLOADS["moe256"]]


class LazyExperts:
    """Expert weights read one expert at a time from the device copy (the full
    fp64 host copy of the large workloads would not fit in host memory)."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, e):
        return np64(self.t[int(e)])


def _inputs(shape, seed, **kw):
    return S.make_flat_inputs(shape, seed=seed, device=DEV, **kw)


def _gate_check(shape, inp, std_floor=0.0):
    cfg = config_for(shape, std_floor)
    ws = moe.alloc_workspace(cfg)
    got = run_gate(cfg, inp, ws)
    assert moe.moe_get_device_error() == 0
    a = oracle_arrays(inp)
    ref = O.gating(a["x"], a["W_g"], a["W_noise"], a["eps"], shape.k, std_floor, a["b_g"])
    T, n = shape.T, shape.n
    lg = np64(got["logits"]).reshape(3, T, n)
    assert_rel(lg[0], ref["clean"], "clean logits")
    assert_rel(lg[1], ref["std"], "noise std")
    assert_rel(lg[2], ref["H"], "noisy logits H")
    same = check_selection(got["idx"].cpu().numpy(), np64(got["gates"]), ref, shape.k)
    assert_rel(np64(got["load"]), ref["P"].sum(axis=0), "load")
    # the GPU's own near-tie flag agrees with the oracle's except within fp32 noise of 1e-5
    tie = got["tie"].cpu().numpy().astype(bool)
    dis = np.nonzero(tie != ref["tie"])[0]
    assert all(abs(ref["gap"][t] - O.TIE_GAP) < 2e-6 * max(1.0, abs(ref["H"][t]).max()) for t in dis)
    return got, ref, same


@pytest.mark.parametrize("shape", SMALL + FULL, ids=lambda s: s.name)
def test_gate(shape):
    _gate_check(shape, _inputs(shape, 1))


FUSABLE = [s for s in SMALL + FULL if s.x_dtype == BF16 and s.n <= 256]


@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("shape", FUSABLE, ids=lambda s: s.name)
def test_gate_fused(shape, bias):
    """moe_gate without the debug logits runs the fused gate (selection, softmax
    and Load partials inside the GEMM's epilogue).  idx, gates and tie must be
    bit-identical to the unfused path, which selects from the same fp32 logits,
    and match the oracle; Load within 1e-5."""
    inp = _inputs(shape, 21)
    if bias:
        inp["b_g"] = torch.randn(shape.n, generator=torch.Generator().manual_seed(3)).to(DEV)
    floor = 0.01 if bias else 0.0
    cfg = config_for(shape, floor)
    ws = moe.alloc_workspace(cfg)
    fused = run_gate(cfg, inp, ws, logits=False)
    plain = run_gate(cfg, inp, ws, logits=True)
    assert moe.moe_get_device_error() == 0
    for key in ("idx", "gates", "tie"):
        assert torch.equal(fused[key], plain[key]), key
    a = oracle_arrays(inp)
    ref = O.gating(a["x"], a["W_g"], a["W_noise"], a["eps"], shape.k, floor, a["b_g"])
    check_selection(fused["idx"].cpu().numpy(), np64(fused["gates"]), ref, shape.k)
    assert_rel(np64(fused["load"]), ref["P"].sum(axis=0), "load")


BIG = [S.FlatShape("big-600", 1000, 128, 600, 64, 4),
       # d = 1024: x streams beside the split weights instead of staying resident
       S.FlatShape("big-600-d1024", 1000, 1024, 600, 64, 4),
       # d = 512 (all eight resident x slots), k = 5, and a last pair tile whose upper
       # 128 rows lie past T
       S.FlatShape("big-300-d512-k5", 1300, 512, 300, 64, 5),
       S.FlatShape("big-400-k8", 700, 256, 400, 64, 8)]


@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("shape", BIG, ids=lambda s: s.name)
def test_gate_big(shape, bias):
    """More than 256 experts without the debug logits runs the chunked gate (selection
    in the GEMM's epilogue over 128-expert chunks, clean and std through memory for the
    Load): idx, gates and tie bit-identical to the debug path, which selects from the
    same fp32 logits, and the oracle matched."""
    inp = _inputs(shape, 22)
    if bias:
        inp["b_g"] = torch.randn(shape.n, generator=torch.Generator().manual_seed(4)).to(DEV)
    floor = 0.01 if bias else 0.0
    cfg = config_for(shape, floor)
    ws = moe.alloc_workspace(cfg)
    chunked = run_gate(cfg, inp, ws, logits=False)
    plain = run_gate(cfg, inp, ws, logits=True)
    assert moe.moe_get_device_error() == 0
    for key in ("idx", "gates", "tie"):
        assert torch.equal(chunked[key], plain[key]), key
    a = oracle_arrays(inp)
    got_idx = chunked["idx"].cpu().numpy()
    # the oracle rerun with the GPU's kept experts (validated as a near-tie choice)
    ref = O.gating(a["x"], a["W_g"], a["W_noise"], a["eps"], shape.k, floor, a["b_g"],
                   kept=kept_of(got_idx, shape.k))
    check_selection(got_idx, np64(chunked["gates"]), own_selection(ref, shape.k), shape.k)
    assert_rel(np64(chunked["gates"]).reshape(-1, shape.k), ref["gates"], "gates")
    assert_rel(np64(chunked["load"]), ref["P"].sum(axis=0), "load")


def test_gate_noise_floor_and_inference():
    shape = S.FlatShape("floor", 700, 64, 24, 64, 2)
    _gate_check(shape, _inputs(shape, 2), std_floor=0.01)
    _gate_check(shape, _inputs(shape, 3, noise=False), std_floor=0.01)   # eps = 0 (inference)


def test_gate_zero_init_uniform():
    """W_g = W_noise = 0: std = ln 2 everywhere and selection uniformly random."""
    shape = S.FlatShape("zero-init", 8192, 64, 8, 64, 2)
    got, ref, _ = _gate_check(shape, _inputs(shape, 4, zero_gate=True))
    std = np64(got["logits"]).reshape(3, shape.T, shape.n)[1]
    assert np.allclose(std, np.log(2.0), rtol=1e-6, atol=0)
    counts = np.bincount(got["idx"].cpu().numpy(), minlength=8)
    expect = shape.T * shape.k / 8
    assert ((counts - expect) ** 2 / expect).sum() < 30.0


def test_gate_ties_lower_index_first():
    """Duplicate W_g columns, no noise: equal logits rank the lower index first."""
    shape = S.FlatShape("ties", 200, 64, 12, 64, 3, F32, F32)
    inp = _inputs(shape, 5, noise=False)
    inp["W_g"][:, 7] = inp["W_g"][:, 2]
    inp["W_g"][:, 9] = inp["W_g"][:, 2]
    inp["W_noise"].zero_()
    _gate_check(shape, inp)


@pytest.mark.parametrize("T,n,k,skew,empty", [
    (1, 1, 1, 0.0, 0), (5, 3, 2, 0.0, 0), (1000, 40, 3, 0.0, 5), (4097, 256, 4, 1.1, 17),
    (32768, 256, 4, 0.0, 0), (65536, 4096, 4, 1.1, 100), (20000, 16384, 2, 0.5, 0)])
def test_dispatch(T, n, k, skew, empty):
    d = 64
    idx, _ = S.make_routing(T, n, k, seed=T + n, skew=skew, empty_experts=empty)
    x = torch.randn((T, d), generator=torch.Generator().manual_seed(7)).to(BF16)
    cfg = moe.make_config(T, d, n, 64, k)
    ws = moe.alloc_workspace(cfg)
    R = T * k
    offsets = torch.empty(n + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(R, dtype=torch.int32, device=DEV)
    inv = torch.empty(R, dtype=torch.int32, device=DEV)
    x_perm = torch.empty((R, d), dtype=BF16, device=DEV)
    moe.moe_dispatch(cfg, idx.to(DEV), x.to(DEV), offsets, perm, inv, x_perm, ws)
    assert moe.moe_get_device_error() == 0
    r_off, r_perm, r_inv = O.dispatch(idx.numpy(), n)
    assert np.array_equal(offsets.cpu().numpy(), r_off)
    assert np.array_equal(perm.cpu().numpy(), r_perm)
    assert np.array_equal(inv.cpu().numpy(), r_inv)
    assert torch.equal(x_perm.cpu(), x[torch.from_numpy(r_perm // k)])


@pytest.mark.parametrize("T,n,k,skew,cap", [
    (5, 3, 2, 0.0, 1), (1000, 40, 3, 0.0, 1), (1000, 40, 3, 0.0, 75), (4097, 256, 4, 1.1, 65),
    (32768, 256, 4, 0.0, 512), (65536, 4096, 4, 1.1, 64)])
def test_dispatch_capacity(T, n, k, skew, cap):
    """A per-expert capacity: each expert keeps its first `cap` routed rows,
    bit-exact against the oracle (offsets, perm, inv with -1 for dropped rows)."""
    d = 64
    idx, _ = S.make_routing(T, n, k, seed=T + n + cap, skew=skew)
    x = torch.randn((T, d), generator=torch.Generator().manual_seed(8)).to(BF16)
    cfg = moe.make_config(T, d, n, 64, k, capacity=cap)
    ws = moe.alloc_workspace(cfg)
    R = T * k
    offsets = torch.empty(n + 1, dtype=torch.int32, device=DEV)
    perm = torch.full((R,), -7, dtype=torch.int32, device=DEV)
    inv = torch.empty(R, dtype=torch.int32, device=DEV)
    x_perm = torch.empty((R, d), dtype=BF16, device=DEV)
    moe.moe_dispatch(cfg, idx.to(DEV), x.to(DEV), offsets, perm, inv, x_perm, ws)
    assert moe.moe_get_device_error() == 0
    r_off, r_perm, r_inv = O.dispatch(idx.numpy(), n, cap)
    kept = int(r_off[n])
    assert kept < R                               # the capacity drops rows in every case
    assert np.array_equal(offsets.cpu().numpy(), r_off)
    assert np.array_equal(perm.cpu().numpy()[:kept], r_perm)
    assert np.array_equal(inv.cpu().numpy(), r_inv)
    assert torch.equal(x_perm.cpu()[:kept], x[torch.from_numpy(r_perm // k)])


def test_dispatch_bad_index_reported():
    T, n, k, d = 64, 8, 2, 64
    idx, _ = S.make_routing(T, n, k, seed=1)
    idx[10, 1] = n + 3
    cfg = moe.make_config(T, d, n, 64, k)
    ws = moe.alloc_workspace(cfg)
    offsets = torch.empty(n + 1, dtype=torch.int32, device=DEV)
    perm = torch.full((T * k,), -1, dtype=torch.int32, device=DEV)
    inv = torch.full((T * k,), -1, dtype=torch.int32, device=DEV)
    x_perm = torch.empty((T * k, d), dtype=BF16, device=DEV)
    moe.moe_dispatch(cfg, idx.to(DEV), torch.zeros((T, d), dtype=BF16, device=DEV), offsets, perm,
                     inv, x_perm, ws)
    assert moe.moe_get_device_error() == 1          # MOE_ERR_INVALID_ARG, then cleared
    assert moe.moe_get_device_error() == 0
    assert int(offsets[n]) == T * k - 1


ROW_TILES, SIZED_TILES = moe.FLAG_FFN_ROW_TILES, moe.FLAG_FFN_SIZED_TILES


@pytest.mark.parametrize("R,n,d,h,dtype,empty,skew,flags", [
    (300, 5, 64, 128, F32, 1, 0.0, 0), (1000, 12, 128, 192, BF16, 3, 0.0, 0),
    (5000, 40, 512, 1024, BF16, 4, 1.1, SIZED_TILES), (5000, 40, 512, 1024, BF16, 4, 1.1, ROW_TILES),
    (2048, 8, 512, 1024, BF16, 0, 0.0, SIZED_TILES), (2048, 8, 512, 1024, BF16, 0, 0.0, ROW_TILES),
    (7, 4, 64, 64, BF16, 1, 0.0, 0)])
def test_expert_ffn(R, n, d, h, dtype, empty, skew, flags):
    x_rows, offsets = S.make_expert_rows(R, n, d, dtype, seed=R, empty_experts=empty, skew=skew)
    g = torch.Generator().manual_seed(R + 1)
    W_in = (torch.randn((n, d, h), generator=g) / d ** 0.5).to(dtype)
    W_out = (torch.randn((n, h, d), generator=g) / h ** 0.5).to(dtype)
    cfg = moe.make_config(R, d, n, h, 1, dtype, dtype, flags=flags)     # T = R rows, k = 1
    ws = moe.alloc_workspace(cfg)
    ydt = torch.float16 if dtype == BF16 else F32
    y = torch.full((R, d), float("nan"), dtype=ydt, device=DEV)
    moe.moe_expert_ffn(cfg, x_rows.to(DEV), offsets.to(DEV), W_in.to(DEV), W_out.to(DEV), y, ws)
    torch.cuda.synchronize()
    got = np64(y)
    xr, wi, wo, off = np64(x_rows), np64(W_in), np64(W_out), offsets.numpy()
    for e in range(n):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        assert_y(got[a:b], O.expert_ffn(xr[a:b], wi[e], wo[e]), dtype == BF16, f"expert {e}")


# Expert row counts around every tile edge of both bf16 FFN kernels (32-row steps of
# the tiles sized to the rows, 128-row halves and 256-row blocks), with an empty
# expert; d = h = 256 gives two items per unit, the tightest reuse of the hidden-ready
# barriers.
TILE_EDGE_ROWS = [1, 17, 31, 32, 33, 100, 127, 128, 129, 200, 255, 256, 257, 300, 511, 512, 513,
                  0, 640]


@pytest.mark.parametrize("d,h", [(256, 512), (256, 256), (512, 1024)])
@pytest.mark.parametrize("flags", [SIZED_TILES, ROW_TILES])
def test_expert_ffn_tile_edges(d, h, flags):
    counts = torch.tensor(TILE_EDGE_ROWS, dtype=torch.int64)
    n, R = len(TILE_EDGE_ROWS), int(counts.sum())
    offsets = torch.zeros(n + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
    g = torch.Generator().manual_seed(d + h)
    x_rows = torch.randn((R, d), generator=g).to(BF16)
    W_in = (torch.randn((n, d, h), generator=g) / d ** 0.5).to(BF16)
    W_out = (torch.randn((n, h, d), generator=g) / h ** 0.5).to(BF16)
    cfg = moe.make_config(R, d, n, h, 1, BF16, BF16, flags=flags)
    ws = moe.alloc_workspace(cfg)
    y = torch.full((R, d), float("nan"), dtype=torch.float16, device=DEV)
    moe.moe_expert_ffn(cfg, x_rows.to(DEV), offsets.to(DEV), W_in.to(DEV), W_out.to(DEV), y, ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    got = np64(y)
    xr, wi, wo, off = np64(x_rows), np64(W_in), np64(W_out), offsets.numpy()
    for e in range(n):
        a, b = off[e], off[e + 1]
        if a < b:
            assert_y(got[a:b], O.expert_ffn(xr[a:b], wi[e], wo[e]), True, f"expert {e} ({b - a} rows)")


@pytest.mark.parametrize("shape", [S.WORKLOADS["moe256"]], ids=lambda s: s.name)
def test_forward_row_tiles_flag(shape):
    """Both bf16 FFN kernels give the same layer output within the fp32 summation
    order (and the flag changes nothing else)."""
    inp = _inputs(shape, 21)
    outs = []
    for flags in (SIZED_TILES, ROW_TILES):
        cfg = moe.make_config(shape.T, shape.d, shape.n, shape.h, shape.k, shape.x_dtype,
                              shape.expert_dtype, flags=flags)
        ws = moe.alloc_workspace(cfg)
        y = torch.empty((shape.T, shape.d), dtype=F32, device=DEV)
        losses = torch.empty(3, dtype=F32, device=DEV)
        idx = torch.empty((shape.T, shape.k), dtype=torch.int32, device=DEV)
        moe.moe_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], None, inp["W_in"],
                        inp["W_out"], y, losses, idx=idx, workspace=ws)
        torch.cuda.synchronize()
        assert moe.moe_get_device_error() == 0
        outs.append((y.clone(), losses.clone(), idx.clone()))
    assert torch.equal(outs[0][2], outs[1][2])
    assert torch.equal(outs[0][1], outs[1][1])
    rms = outs[1][0].pow(2).mean().sqrt().item()
    assert (outs[0][0] - outs[1][0]).abs().max().item() <= 1e-2 * rms


@pytest.mark.parametrize("T,k,d,dtype", [(1, 1, 64, F32), (333, 3, 128, BF16), (4096, 4, 512, BF16),
                                          (100, 8, 64, F32)])
def test_combine(T, k, d, dtype):
    g = torch.Generator().manual_seed(T)
    R = T * k
    y_perm = torch.randn((R, d), generator=g).to(torch.float16 if dtype == BF16 else F32)
    inv = torch.randperm(R, generator=g).to(torch.int32)
    _, gates = S.make_routing(T, max(k, 2), k, seed=T)
    cfg = moe.make_config(T, d, max(k, 2), 64, k, dtype, dtype)
    y = torch.empty((T, d), dtype=F32, device=DEV)
    moe.moe_combine(cfg, y_perm.to(DEV), inv.to(DEV), gates.to(DEV), y)
    ref = O.combine_gathered(np64(y_perm), inv.numpy(), np64(gates))
    got = np64(y)
    # fp32 accumulation of k products of exact inputs: well inside 1e-6 relative to RMS
    assert np.max(np.abs(got - ref)) <= 1e-6 * np.sqrt(np.mean(ref ** 2))


@pytest.mark.parametrize("T,n,k,skew", [(1, 1, 1, 0.0), (1000, 40, 3, 0.0), (32768, 256, 4, 0.0),
                                        (65536, 4096, 4, 1.1)])
def test_balance_losses(T, n, k, skew):
    idx, gates = S.make_routing(T, n, k, seed=T + 3, skew=skew)
    load = torch.rand(n, generator=torch.Generator().manual_seed(n)) * T * k / n
    r_off, r_perm, _ = O.dispatch(idx.numpy(), n)
    cfg = moe.make_config(T, 64, n, 64, k)
    imp = torch.empty(n, dtype=F32, device=DEV)
    losses = torch.empty(3, dtype=F32, device=DEV)
    moe.moe_balance_losses(cfg, gates.to(DEV), torch.from_numpy(r_perm).to(torch.int32).to(DEV),
                           torch.from_numpy(r_off).to(torch.int32).to(DEV), load.to(DEV), imp, losses)
    ref_imp = O.importance_of(idx.numpy(), np64(gates), n)
    assert_rel(np64(imp), ref_imp, "importance")
    ci, cl, aux = O.balance_losses(ref_imp, np64(load), 0.1, 0.1)
    got = np64(losses)
    assert_rel(got, [ci, cl, aux], "losses")


def _forward(shape, inp, std_floor=0.0):
    cfg = config_for(shape, std_floor)
    ws = moe.alloc_workspace(cfg)
    T, n, k, d = shape.T, shape.n, shape.k, shape.d
    out = dict(y=torch.empty((T, d), dtype=F32, device=DEV),
               losses=torch.empty(3, dtype=F32, device=DEV),
               idx=torch.empty(T * k, dtype=torch.int32, device=DEV),
               gates=torch.empty(T * k, dtype=F32, device=DEV),
               tie=torch.empty(T, dtype=torch.uint8, device=DEV),
               importance=torch.empty(n, dtype=F32, device=DEV),
               load=torch.empty(n, dtype=F32, device=DEV))
    moe.moe_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], inp["b_g"],
                    inp["W_in"], inp["W_out"], out["y"], out["losses"], out["idx"], out["gates"],
                    out["tie"], out["importance"], out["load"], ws)
    assert moe.moe_get_device_error() == 0
    return out


def check_forward(shape, got, ref, bf16):
    """The whole layer against the oracle run with the GPU's kept set: selection
    (bit-exact outside near ties, against the oracle's own choice), gates, y on
    every row, Importance, Load and the three losses, all at their tolerances."""
    k = shape.k
    check_selection(got["idx"].cpu().numpy(), np64(got["gates"]), own_selection(ref, k), k)
    assert_rel(np64(got["gates"]).reshape(-1, k), ref["gates"], "gates")
    assert_y(np64(got["y"]), ref["y"], bf16)
    assert_rel(np64(got["importance"]), ref["importance"], "importance")
    assert_rel(np64(got["load"]), ref["load"], "load")
    assert_rel(np64(got["losses"]), list(ref["losses"]), "losses")


@pytest.mark.parametrize("shape", SMALL + FULL, ids=lambda s: s.name)
def test_forward(shape):
    inp = _inputs(shape, 11)
    got = _forward(shape, inp)
    a = oracle_arrays(inp)
    ref = O.moe_forward(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"], a["W_out"], shape.k,
                        0.0, a["b_g"], kept=kept_of(got["idx"].cpu().numpy(), shape.k))
    check_forward(shape, got, ref, shape.expert_dtype == BF16)


CAPACITY_SHAPES = [S.WORKLOADS["tiny-fp32"], S.FlatShape("ragged-bf16", 1000, 128, 40, 192, 3),
                   S.FlatShape("k8-bf16", 513, 64, 70, 128, 8),
                   S.FlatShape("n250-bf16", 1500, 64, 250, 64, 3), S.WORKLOADS["moe256"]]


@pytest.mark.parametrize("shape", CAPACITY_SHAPES, ids=lambda s: s.name)
def test_forward_capacity(shape):
    """The layer with a per-expert capacity of T k / n rows (capacity factor 1):
    dropped rows add nothing to y; the gate and the losses are those of the
    layer without a capacity."""
    cap = max(1, shape.T * shape.k // shape.n)
    inp = _inputs(shape, 23)
    cfg = moe.make_config(shape.T, shape.d, shape.n, shape.h, shape.k, shape.x_dtype,
                          shape.expert_dtype, capacity=cap)
    ws = moe.alloc_workspace(cfg)
    T, n, k, d = shape.T, shape.n, shape.k, shape.d
    y = torch.empty((T, d), dtype=F32, device=DEV)
    losses = torch.empty(3, dtype=F32, device=DEV)
    idx = torch.empty(T * k, dtype=torch.int32, device=DEV)
    gates = torch.empty(T * k, dtype=F32, device=DEV)
    moe.moe_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], inp["b_g"], inp["W_in"],
                    inp["W_out"], y, losses, idx=idx, gates=gates, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    a = oracle_arrays(inp)
    ref = O.moe_forward(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"], a["W_out"], k, 0.0,
                        a["b_g"], capacity=cap, kept=kept_of(idx.cpu().numpy(), k))
    check_selection(idx.cpu().numpy(), np64(gates), own_selection(ref, k), k)
    assert_rel(np64(gates).reshape(-1, k), ref["gates"], "gates")
    assert not ref["keep"].all()
    assert_y(np64(y), ref["y"], shape.expert_dtype == BF16)
    assert_rel(np64(losses), list(ref["losses"]), "losses")


@pytest.mark.parametrize("shape", [S.WORKLOADS["tiny-fp32"],
                                   S.FlatShape("ragged-bf16", 1000, 128, 40, 192, 3),
                                   S.FlatShape("big-600", 1000, 128, 600, 64, 4)],
                         ids=lambda s: s.name)
def test_no_noise_pointer(shape):
    """eps = NULL is the noiseless gate: the same results, bit for bit, as an
    all-zero noise tensor (gate and whole layer)."""
    inp = _inputs(shape, 24)
    inp["eps"] = torch.zeros_like(inp["eps"])
    cfg = config_for(shape)
    ws = moe.alloc_workspace(cfg)
    for logits in (False, True):        # the fused / large-n gates, and the logits path
        zero = run_gate(cfg, inp, ws, logits=logits)
        none = run_gate(cfg, dict(inp, eps=None), ws, logits=logits)
        torch.cuda.synchronize()
        for key in ("idx", "gates", "tie", "load") + (("logits",) if logits else ()):
            assert torch.equal(zero[key], none[key]), key
    outs = []
    for eps in (inp["eps"], None):
        y = torch.empty((shape.T, shape.d), dtype=F32, device=DEV)
        losses = torch.empty(3, dtype=F32, device=DEV)
        moe.moe_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], eps, inp["b_g"], inp["W_in"],
                        inp["W_out"], y, losses, workspace=ws)
        outs.append((y, losses))
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    # and the noiseless gate is the oracle's with eps = 0
    a = oracle_arrays(inp)
    ref = O.gating(a["x"], a["W_g"], a["W_noise"], a["eps"], shape.k, 0.0, a["b_g"])
    check_selection(none["idx"].cpu().numpy(), np64(none["gates"]), ref, shape.k)


SWITCH = moe.FLAG_SWITCH_GATE
SWITCH_SHAPES = [S.WORKLOADS["tiny-fp32"], S.FlatShape("switch-k1-bf16", 1000, 128, 40, 192, 1),
                 S.FlatShape("switch-k2-bf16", 777, 64, 256, 128, 2),
                 S.FlatShape("switch-big-600", 1000, 128, 600, 64, 1),
                 S.FlatShape("moe256-switch", 32768, 512, 256, 1024, 1)]


@pytest.mark.parametrize("shape", SWITCH_SHAPES, ids=lambda s: s.name)
def test_switch_forward(shape):
    """The Switch gate: the softmax over all n logits at the kept experts, the
    routed-row counts as load, the summed probabilities as importance, and the
    single loss n sum_i f_i P_i; the whole layer against the oracle."""
    inp = _inputs(shape, 31)
    cfg = moe.make_config(shape.T, shape.d, shape.n, shape.h, shape.k, shape.x_dtype,
                          shape.expert_dtype, flags=SWITCH)
    ws = moe.alloc_workspace(cfg)
    T, n, k, d = shape.T, shape.n, shape.k, shape.d
    out = dict(y=torch.empty((T, d), dtype=F32, device=DEV), losses=torch.empty(3, dtype=F32, device=DEV),
               idx=torch.empty(T * k, dtype=torch.int32, device=DEV),
               gates=torch.empty(T * k, dtype=F32, device=DEV),
               importance=torch.empty(n, dtype=F32, device=DEV), load=torch.empty(n, dtype=F32, device=DEV))
    moe.moe_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], inp["b_g"], inp["W_in"],
                    inp["W_out"], out["y"], out["losses"], idx=out["idx"], gates=out["gates"],
                    importance=out["importance"], load=out["load"], workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    a = oracle_arrays(inp)
    ref = O.moe_forward(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"], a["W_out"], k, 0.0,
                        a["b_g"], switch=True)
    same = check_selection(out["idx"].cpu().numpy(), np64(out["gates"]), ref, k, "switch gate")
    assert same.all()
    assert np.array_equal(np64(out["load"]), ref["load"])          # integer counts
    assert_rel(np64(out["importance"]), ref["importance"], "importance (summed probabilities)")
    assert_rel(np64(out["losses"]), list(ref["losses"]), "switch loss")
    # y_t = sum_j g_tj E_j(x_t) with gates that no longer sum to 1 and vary by orders of
    # magnitude between tokens; the expert and combine arithmetic is the default path's,
    # so the bf16 bound applies to y_t divided by the token's (oracle) gate mass, the
    # convex combination that the default gate's y is.
    mass = ref["gates"].sum(axis=1, keepdims=True)
    assert_y(np64(out["y"]) / mass, ref["y"] / mass, shape.expert_dtype == BF16)
    # moe_gate gives the same gates and counts
    g = run_gate(cfg, inp, ws, logits=False)
    torch.cuda.synchronize()
    assert torch.equal(g["idx"], out["idx"]) and torch.equal(g["gates"], out["gates"])
    assert torch.equal(g["load"], out["load"])


def test_balance_losses_refuses_capacity():
    T, n, k = 64, 8, 2
    cfg = moe.make_config(T, 64, n, 64, k, capacity=4)
    dev = dict(device=DEV)
    with pytest.raises(moe.MoeError, match="UNSUPPORTED"):
        moe.moe_balance_losses(cfg, torch.zeros(T * k, **dev), torch.zeros(T * k, dtype=torch.int32, **dev),
                               torch.zeros(n + 1, dtype=torch.int32, **dev), torch.zeros(n, **dev),
                               torch.zeros(n, **dev), torch.zeros(3, **dev))


def test_forward_timed_matches_forward():
    """moe_forward_timed runs the same forward pass and records its six stage events."""
    shape = S.WORKLOADS["moe32"]
    inp = _inputs(shape, 14)
    ref = _forward(shape, inp)
    cfg = config_for(shape)
    ws = moe.alloc_workspace(cfg)
    y = torch.empty_like(ref["y"])
    losses = torch.empty_like(ref["losses"])
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    moe.moe_forward_timed(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], inp["b_g"],
                          inp["W_in"], inp["W_out"], y, losses, ev, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    assert torch.equal(y, ref["y"]) and torch.equal(losses, ref["losses"])
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(5)]
    assert all(t >= 0.0 for t in times) and times[2] > 0.0      # the experts take time


def test_forward_deterministic():
    shape = S.WORKLOADS["moe256"]
    inp = _inputs(shape, 12)
    outs = [_forward(shape, inp) for _ in range(3)]
    for o in outs[1:]:
        for key in ("y", "losses", "idx", "gates", "importance", "load"):
            assert torch.equal(o[key], outs[0][key]), key


@pytest.mark.slow
def test_forward_zipf4096_sampled():
    """The 4096-expert Zipf workload at full size: gate and layer output on 512
    sampled tokens, Load and Importance against the oracle's full batch sums."""
    shape = S.WORKLOADS["moe4096-zipf"]
    k = shape.k
    inp = _inputs(shape, 13)
    got = _forward(shape, inp)
    counts = np.bincount(got["idx"].cpu().numpy(), minlength=shape.n)
    assert (counts == 0).sum() >= 1                  # the skew leaves some experts without tokens
    a = {key: np64(v) for key, v in inp.items() if key not in ("W_in", "W_out") and v is not None}
    kept = kept_of(got["idx"].cpu().numpy(), k)
    rows = np.sort(np.random.default_rng(0).choice(shape.T, 512, replace=False))
    ref = O.moe_forward_rows(a["x"], a["W_g"], a["W_noise"], a["eps"], LazyExperts(inp["W_in"]),
                             LazyExperts(inp["W_out"]), k, rows, 0.0, a["b_g"], kept=kept[rows])
    ref["order"] = np.argsort(-ref["H"], axis=1, kind="stable")
    g_rows = np64(got["gates"]).reshape(-1, k)[rows]
    check_selection(kept[rows], g_rows, own_selection(ref, k), k)
    assert_rel(g_rows, ref["gates"], "gates")
    assert_y(np64(got["y"])[rows], ref["y"], True)
    # batch sums over all T tokens, with the GPU's kept set on any near-tie row
    sums = O.gating_sums(a["x"], a["W_g"], a["W_noise"], a["eps"], k, 0.0, a["b_g"], kept=kept)
    assert_rel(np64(got["load"]), sums["load"], "load")
    assert_rel(np64(got["importance"]), sums["importance"], "importance")
    assert_rel(np64(got["losses"]), list(O.balance_losses(sums["importance"], sums["load"])),
               "losses")


def test_failure_detection_timeout_path():
    """The kernels' bounded waits, run out on purpose on a barrier nothing completes:
    the device error word reports MOE_ERR_TIMEOUT (read once, then cleared), nothing
    faults or hangs, and the context still runs a forward pass afterwards."""
    moe.moe_selftest_timeout(2_000_000)          # about 1 ms of SM cycles
    assert moe.moe_get_device_error() == 5       # MOE_ERR_TIMEOUT
    assert moe.moe_get_device_error() == 0
    shape = S.FlatShape("after-timeout", 300, 64, 16, 128, 2)
    inp = _inputs(shape, 15)
    got = _forward(shape, inp)
    a = oracle_arrays(inp)
    ref = O.moe_forward(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"], a["W_out"], shape.k,
                        kept=kept_of(got["idx"].cpu().numpy(), shape.k))
    check_forward(shape, got, ref, True)


def test_forward_max_experts():
    """n = 16384 experts (the largest flat layer), k = 2: the unfused tensor-core gate
    (logits through memory, 128 expert chunks), a dispatch over 16384 bins, and
    experts that mostly own no row."""
    shape = S.FlatShape("n16384", 700, 64, 16384, 64, 2)
    inp = _inputs(shape, 16)
    got = _forward(shape, inp)
    a = oracle_arrays(inp)
    ref = O.moe_forward(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"], a["W_out"], shape.k,
                        kept=kept_of(got["idx"].cpu().numpy(), shape.k))
    check_forward(shape, got, ref, True)


@pytest.mark.parametrize("d,h,flags", [(256, 256, ROW_TILES), (256, 256, SIZED_TILES),
                                        (128, 192, 0)],
                         ids=["pair", "sized", "one-cta"])
def test_fp16_output_range_reported(d, h, flags):
    """bf16 experts write fp16 outputs: with W_out scaled so that expert outputs reach
    about 1e6 (beyond fp16's 65504) every tensor-core FFN kernel reports MOE_ERR_RANGE
    through the device error word (no trap), which reads once and then clears; the
    call itself succeeds and in-range outputs stay exact."""
    n, R = 4, 700
    x_rows, offsets = S.make_expert_rows(R, n, d, BF16, seed=9)
    g = torch.Generator().manual_seed(10)
    W_in = (torch.randn((n, d, h), generator=g) / d ** 0.5).to(BF16)
    W_out = (torch.randn((n, h, d), generator=g) / h ** 0.5)
    W_out[2] *= 1e6                                  # only expert 2 leaves the range
    W_out = W_out.to(BF16)
    cfg = moe.make_config(R, d, n, h, 1, BF16, BF16, flags=flags)
    ws = moe.alloc_workspace(cfg)
    y = torch.empty((R, d), dtype=torch.float16, device=DEV)
    assert moe.moe_get_device_error() == 0
    moe.moe_expert_ffn(cfg, x_rows.to(DEV), offsets.to(DEV), W_in.to(DEV), W_out.to(DEV), y, ws)
    assert moe.moe_get_device_error() == 6           # MOE_ERR_RANGE
    assert moe.moe_get_device_error() == 0           # read and cleared
    got, off = np64(y), offsets.numpy()
    assert np.isinf(got[off[2]:off[3]]).any()
    xr, wi, wo = np64(x_rows), np64(W_in), np64(W_out)
    for e in (0, 1, 3):
        a, b = off[e], off[e + 1]
        if a < b:
            assert_y(got[a:b], O.expert_ffn(xr[a:b], wi[e], wo[e]), True, f"expert {e}")
