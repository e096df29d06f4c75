"""The layer's own noise draws (MOE_FLAG_DEVICE_NOISE, moe_draw_noise) against the
oracle's draw_noise ("Noisy top-k gating", eq (4): one standard normal draw per token
and expert).  Needs a B300; ``pytest -m gpu``.

* moe_draw_noise against the oracle element by element (fp32 logf / sqrtf / cospif
  against fp64: within 4e-6 absolute, |eps| <= 5.77), for counts with and without a
  tail that is not a multiple of four.
* The whole forward pass with the flag and eps = None: bit-identical to the same call
  with eps = moe_draw_noise's draws passed in, and matching the oracle run on the
  oracle's own draws (with the GPU's kept experts on near-tie rows).
* The backward pass with the flag: bit-identical to the call with the draws passed in.
* Misuse: eps given with the flag, and the batchwise gate with the flag, are refused.
"""
import numpy as np
import pytest
import torch

import sparsely_gated_mixture_03_b300 as moe
from sparsely_gated_mixture_03_b300 import synthetic as S
from oracle import moe_oracle as O
from gpu_helpers import assert_rel, assert_y, check_selection, kept_of, np64, own_selection

pytestmark = pytest.mark.gpu

DEV = "cuda"
F32, BF16 = torch.float32, torch.bfloat16
NOISE = moe.FLAG_DEVICE_NOISE


@pytest.mark.parametrize("count", [1, 3, 4, 1000003, 1 << 22])
def test_draw_noise_matches_oracle(count):
    seed = 0x5EED0000 + count
    got = torch.empty(count, dtype=F32, device=DEV)
    moe.moe_draw_noise(seed, got)
    torch.cuda.synchronize()
    ref = O.draw_noise(seed, count)
    g = got.cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all()
    err = np.abs(g - ref).max()
    assert err < 4e-6, f"max |eps_gpu - eps_oracle| = {err}"


def _cfg(shape, flags=0, seed=0):
    return moe.make_config(shape.T, shape.d, shape.n, shape.h, shape.k, shape.x_dtype,
                           shape.expert_dtype, flags=flags, noise_seed=seed)


def _forward(cfg, inp, eps):
    T, n, k, d = cfg.T, cfg.n, cfg.k, cfg.d
    out = dict(y=torch.empty((T, d), dtype=F32, device=DEV),
               losses=torch.empty(3, dtype=F32, device=DEV),
               idx=torch.empty(T * k, dtype=torch.int32, device=DEV),
               gates=torch.empty(T * k, dtype=F32, device=DEV),
               importance=torch.empty(n, dtype=F32, device=DEV),
               load=torch.empty(n, dtype=F32, device=DEV))
    moe.moe_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], eps, inp["b_g"], inp["W_in"],
                    inp["W_out"], out["y"], out["losses"], out["idx"], out["gates"], None,
                    out["importance"], out["load"], moe.alloc_workspace(cfg))
    assert moe.moe_get_device_error() == 0
    return out


@pytest.mark.parametrize("shape", [S.FlatShape("noise-bf16", 3000, 128, 64, 256, 4),
                                   S.FlatShape("noise-big", 700, 64, 600, 64, 2),
                                   S.FlatShape("noise-fp32", 500, 64, 24, 64, 3, F32, F32)],
                         ids=lambda s: s.name)
def test_forward_device_noise(shape):
    seed = 987654321
    inp = S.make_flat_inputs(shape, seed=71, device=DEV)
    T, n, k = shape.T, shape.n, shape.k
    drawn = _forward(_cfg(shape, NOISE, seed), inp, None)
    eps = torch.empty((T, n), dtype=F32, device=DEV)
    moe.moe_draw_noise(seed, eps)
    given = _forward(_cfg(shape), inp, eps)
    for key in drawn:
        assert torch.equal(drawn[key], given[key]), key
    a = {key: (None if v is None else np64(v)) for key, v in inp.items()}
    eps_ref = O.draw_noise(seed, T * n).reshape(T, n)
    got_idx = drawn["idx"].cpu().numpy()
    ref = O.moe_forward(a["x"], a["W_g"], a["W_noise"], eps_ref, a["W_in"], a["W_out"], k, 0.0,
                        a["b_g"], kept=kept_of(got_idx, k))
    check_selection(got_idx, np64(drawn["gates"]), own_selection(ref, k), k)
    assert_rel(np64(drawn["gates"]).reshape(-1, k), ref["gates"], "gates")
    assert_y(np64(drawn["y"]), ref["y"], shape.expert_dtype == BF16)
    assert_rel(np64(drawn["importance"]), ref["importance"], "importance")
    assert_rel(np64(drawn["load"]), ref["load"], "load")
    assert_rel(np64(drawn["losses"]), list(ref["losses"]), "losses")


@pytest.mark.parametrize("shape,flags", [
    (S.FlatShape("gate-noise-bf16", 1000, 128, 40, 64, 3), 0),
    (S.FlatShape("gate-noise-switch", 777, 64, 256, 64, 1), moe.FLAG_SWITCH_GATE),
    (S.FlatShape("gate-noise-big", 600, 64, 600, 64, 4), 0)],
    ids=["bf16", "switch", "big"])
@pytest.mark.parametrize("logits", [False, True])
def test_gate_device_noise(shape, flags, logits):
    """moe_gate with the flag: every output (and the debug logits) bit-identical to the
    call with moe_draw_noise's draws passed in, for the fused, Switch and large-n gates."""
    from gpu_helpers import run_gate
    seed = 4242
    inp = S.make_flat_inputs(shape, seed=75, device=DEV)
    T, n = shape.T, shape.n
    cfg = _cfg(shape, flags | NOISE, seed)
    drawn = run_gate(cfg, dict(inp, eps=None), moe.alloc_workspace(cfg), logits=logits)
    eps = torch.empty((T, n), dtype=F32, device=DEV)
    moe.moe_draw_noise(seed, eps)
    cfg2 = _cfg(shape, flags)
    given = run_gate(cfg2, dict(inp, eps=eps), moe.alloc_workspace(cfg2), logits=logits)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error() == 0
    for key in drawn:
        if drawn[key] is not None:
            assert torch.equal(drawn[key], given[key]), key


def test_backward_device_noise():
    shape = S.FlatShape("noise-bwd", 1024, 256, 64, 256, 2)
    seed = 31337
    inp = S.make_flat_inputs(shape, seed=72, device=DEV)
    T, d, n, h = shape.T, shape.d, shape.n, shape.h
    dy = torch.randn((T, d), generator=torch.Generator().manual_seed(73)).to(DEV)

    def run(cfg, eps):
        f = dict(device=DEV, dtype=F32)
        out = [torch.empty((T, d), **f), torch.empty((d, n), **f), torch.empty((d, n), **f),
               torch.empty(n, **f), torch.empty((n, d, h), **f), torch.empty((n, h, d), **f)]
        b_g = torch.zeros(n, **f)
        moe.moe_backward(cfg, inp["x"], inp["W_g"], inp["W_noise"], eps, b_g, inp["W_in"],
                         inp["W_out"], dy, *out, moe.alloc_backward_workspace(cfg))
        assert moe.moe_get_device_error() == 0
        return out

    drawn = run(_cfg(shape, NOISE, seed), None)
    eps = torch.empty((T, n), dtype=F32, device=DEV)
    moe.moe_draw_noise(seed, eps)
    given = run(_cfg(shape), eps)
    for a, b in zip(drawn, given):
        assert torch.equal(a, b)


def test_device_noise_misuse_refused():
    shape = S.FlatShape("noise-misuse", 512, 64, 16, 64, 2)
    inp = S.make_flat_inputs(shape, seed=74, device=DEV)
    cfg = _cfg(shape, NOISE, 1)
    with pytest.raises(moe.MoeError, match="INVALID"):
        _forward(cfg, inp, inp["eps"])
    y = torch.empty((shape.T, shape.d), dtype=F32, device=DEV)
    with pytest.raises(moe.MoeError, match="UNSUPPORTED"):
        moe.moe_batchwise_forward(cfg, inp["x"], inp["W_g"], inp["W_noise"], None, inp["b_g"],
                                  inp["W_in"], inp["W_out"], y, torch.empty(3, device=DEV),
                                  workspace=moe.alloc_batchwise_workspace(cfg))
