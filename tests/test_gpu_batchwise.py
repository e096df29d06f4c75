"""The batchwise top-m gate (moe_batchwise_forward, through the C ABI) against the fp64
oracle: each expert's token set bit-exact except where its m-th and (m+1)-th logits are
a near tie (there any valid choice), the gates within 1e-5, the layer output within the
layer's bf16 / fp32 bound on the tokens whose experts agree, tokens no expert took at
exactly 0, and the losses.
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
    ref = O.moe_forward_batchwise(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"],
                                  a["W_out"], k, 0.0, a["b_g"])
    got_sel = sel.cpu().numpy()
    assert np.all(np.diff(got_sel, axis=1) > 0)          # ascending, distinct tokens
    Hh = ref["H"]
    agree = np.ones(n, dtype=bool)
    for i in range(n):
        if np.array_equal(got_sel[i], ref["sel"][i]):
            continue
        agree[i] = False
        # a near tie at the m-th place: every token taken is within the tie gap of it
        mth = np.sort(Hh[:, i])[::-1][m - 1]
        assert ref["mgap"][i] < O.TIE_GAP * max(1.0, abs(mth)), f"expert {i} differs"
        assert np.all(Hh[got_sel[i], i] >= mth - O.TIE_GAP * max(1.0, abs(mth)))
    taken = np.zeros((T, n), dtype=bool)
    for i in range(n):
        taken[got_sel[i], i] = True
    same_tok = (taken == ref["taken"]).all(axis=1)     # the token's experts agree
    got_y = np64(y)
    assert_y(got_y[same_tok], ref["y"][same_tok], shape.expert_dtype == BF16)
    none = ~taken.any(axis=1)
    assert not got_y[none].any()
    if agree.all():
        assert_rel(np64(losses), list(ref["losses"]), "losses")
