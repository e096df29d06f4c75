"""The batchwise top-m gate (moe_batchwise_forward, through the C ABI) against the fp64
oracle: each expert's token set bit-exact except where its m-th and (m+1)-th logits are
a near tie (there the oracle checks that the GPU's set is a valid choice and is rerun
with it), the layer output on every token within the layer's bf16 / fp32 bound, tokens
no expert took at exactly 0, and the losses within 1e-5.  And its inference mode
(moe_batchwise_threshold_forward): a learned per-expert threshold.
"""
import numpy as np
import pytest
import torch

import sparsely_gated_mixture_03_b300 as moe
from sparsely_gated_mixture_03_b300 import synthetic as S
from oracle import moe_oracle as O
from gpu_helpers import assert_rel, assert_y, np64, oracle_arrays

pytestmark = pytest.mark.gpu

DEV = "cuda"
F32, BF16 = torch.float32, torch.bfloat16

SHAPES = [
    S.WORKLOADS["tiny-fp32"],
    S.FlatShape("ragged-bf16", 1000, 128, 40, 192, 3),
    S.FlatShape("bw-600-experts", 2048, 64, 600, 64, 2),
    S.WORKLOADS["moe256"],
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_batchwise_forward(shape):
    T, d, n, h, k = shape.T, shape.d, shape.n, shape.h, shape.k
    m = k * T // n
    inp = S.make_flat_inputs(shape, seed=71, device=DEV)
    cfg = moe.make_config(T, d, n, h, k, shape.x_dtype, shape.expert_dtype)
    y = torch.full((T, d), float("nan"), dtype=F32, device=DEV)
    losses = torch.empty(3, dtype=F32, device=DEV)
    sel = torch.full((n, m), -1, dtype=torch.int32, device=DEV)
    moe.moe_batchwise_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], inp["b_g"],
                              inp["W_in"], inp["W_out"], y, losses, sel=sel)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    a = oracle_arrays(inp)
    got_sel = sel.cpu().numpy()
    assert np.all(np.diff(got_sel, axis=1) > 0)          # ascending, distinct tokens
    own = O.batchwise_gating(a["x"], a["W_g"], a["W_noise"], a["eps"], k, 0.0, a["b_g"])
    # each expert's set is the oracle's, except on a near tie at its m-th place, where the
    # oracle checks that the GPU's set is a valid choice and is rerun with it
    for i in range(n):
        if not np.array_equal(got_sel[i], own["sel"][i]):
            mth = np.sort(own["H"][:, i])[::-1][m - 1]
            assert own["mgap"][i] < O.TIE_GAP * max(1.0, abs(mth)), f"expert {i} differs"
    ref = O.moe_forward_batchwise(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"],
                                  a["W_out"], k, 0.0, a["b_g"], sel=got_sel)
    got_y = np64(y)
    assert_y(got_y, ref["y"], shape.expert_dtype == BF16)
    assert not got_y[~ref["taken"].any(axis=1)].any()    # tokens no expert took: exactly 0
    assert_rel(np64(losses), list(ref["losses"]), "losses")


def _separated_thresholds(H, quantile, rng):
    """Per expert a threshold between two adjacent logits of its column that lie at
    least 1e-3 apart near the given quantile, so that fp32 and fp64 logits take the
    same tokens."""
    T, n = H.shape
    thr = np.empty(n)
    for i in range(n):
        col = np.sort(H[:, i])[::-1]
        j = int(np.clip(round(quantile * T + rng.integers(-3, 4)), 1, T - 1))
        while j < T - 1 and col[j - 1] - col[j] < 1e-3:
            j += 1
        thr[i] = 0.5 * (col[j - 1] + col[j])
    return thr


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_batchwise_threshold_forward(shape):
    """The inference mode: thresholds well away from every logit (so the selection is
    unambiguous), counts exact, y on every token and the losses against the oracle; a
    threshold between each expert's m-th and (m+1)-th logits gives the training-time
    layer; +inf gives y = 0; thresholds admitting more than k T pairs report
    MOE_ERR_RANGE without a fault."""
    T, d, n, h, k = shape.T, shape.d, shape.n, shape.h, shape.k
    inp = S.make_flat_inputs(shape, seed=73, device=DEV)
    cfg = moe.make_config(T, d, n, h, k, shape.x_dtype, shape.expert_dtype)
    ws = moe.alloc_batchwise_workspace(cfg)
    a = oracle_arrays(inp)
    H = O.noisy_logits(a["x"], a["W_g"], a["W_noise"], a["eps"], 0.0, a["b_g"])[2]
    rng = np.random.default_rng(5)
    # about k/2 experts a token
    thr = _separated_thresholds(H, 0.5 * k / n * rng.uniform(0.5, 1.5), rng)
    y = torch.full((T, d), float("nan"), dtype=F32, device=DEV)
    losses = torch.empty(3, dtype=F32, device=DEV)
    counts = torch.full((n,), -1, dtype=torch.int32, device=DEV)
    thr_dev = torch.from_numpy(thr).float().to(DEV)
    moe.moe_batchwise_threshold_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"],
                                        inp["b_g"], thr_dev, inp["W_in"], inp["W_out"], y,
                                        losses, counts=counts, workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    ref = O.moe_forward_batchwise(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"],
                                  a["W_out"], k, 0.0, a["b_g"],
                                  threshold=thr_dev.double().cpu().numpy())
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    assert_y(np64(y), ref["y"], shape.expert_dtype == BF16)
    assert not np64(y)[~ref["taken"].any(axis=1)].any()
    assert_rel(np64(losses), list(ref["losses"]), "losses")

    # +inf: no expert takes anything
    moe.moe_batchwise_threshold_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"],
                                        inp["b_g"], torch.full((n,), float("inf"), device=DEV),
                                        inp["W_in"], inp["W_out"], y, losses, counts=counts,
                                        workspace=ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    assert not y.any() and not counts.any()
    # -inf: every expert takes every token, more than the k T pairs the workspace holds
    if n > k:
        moe.moe_batchwise_threshold_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"],
                                            inp["eps"], inp["b_g"],
                                            torch.full((n,), float("-inf"), device=DEV),
                                            inp["W_in"], inp["W_out"], y, losses, counts=counts,
                                            workspace=ws)
        assert moe.moe_get_device_error() == 6          # MOE_ERR_RANGE, then cleared
        assert moe.moe_get_device_error() == 0
        assert (counts.cpu().numpy() == T).all()


def test_batchwise_threshold_reproduces_training():
    """Thresholds between each expert's m-th and (m+1)-th largest logits take exactly
    the training-time sets: the same layer output, bit for bit, and the same losses."""
    shape = S.FlatShape("bw-thr", 4096, 256, 32, 256, 2)
    T, d, n, h, k = shape.T, shape.d, shape.n, shape.h, shape.k
    m = k * T // n
    # the first seed whose every expert has its m-th and (m+1)-th logits at least 1e-4
    # apart (the fp32 logits then fall on the same side of the midpoint threshold)
    for seed in range(79, 400):
        inp = S.make_flat_inputs(shape, seed=seed, device="cpu")
        a = oracle_arrays(inp)
        H = O.noisy_logits(a["x"], a["W_g"], a["W_noise"], a["eps"], 0.0, a["b_g"])[2]
        col = -np.sort(-H, axis=0)
        if (col[m - 1] - col[m] > 1e-4).all():
            break
    assert (col[m - 1] - col[m] > 1e-4).all()
    inp = {key: (None if v is None else v.to(DEV)) for key, v in inp.items()}
    cfg = moe.make_config(T, d, n, h, k, shape.x_dtype, shape.expert_dtype)
    y_tr = torch.empty((T, d), dtype=F32, device=DEV)
    l_tr = torch.empty(3, dtype=F32, device=DEV)
    moe.moe_batchwise_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], inp["b_g"],
                              inp["W_in"], inp["W_out"], y_tr, l_tr)
    thr = torch.from_numpy(0.5 * (col[m - 1] + col[m])).float().to(DEV)
    y = torch.empty_like(y_tr)
    losses = torch.empty_like(l_tr)
    counts = torch.empty(n, dtype=torch.int32, device=DEV)
    moe.moe_batchwise_threshold_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"],
                                        inp["b_g"], thr, inp["W_in"], inp["W_out"], y, losses,
                                        counts=counts)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    assert (counts.cpu() == m).all()
    assert torch.equal(y, y_tr)
    assert torch.equal(losses, l_tr)
