"""moe_dispatch_noalloc: the dispatch for callers that cannot allocate device
memory (a plugin whose host framework owns all of the GPU's memory, a serving
loop that must not let cudaFree synchronise the device).  It keeps the counting
sort's scratch in the library's own 1 MiB device array instead of a caller
workspace.

Checked through the C ABI against moe_dispatch on the same inputs: dispatch is
integer work, so the outputs must be bit-identical, on two calls in a row (the
second with different routing, so stale contents of the shared array would
show); the permutation is also checked against the oracle's counting sort.  This file is collected last so a run stopping at the first failure has
run every other test already; it also passes alone in a fresh process.
"""
import pytest
import torch

import numpy as np

import sparsely_gated_mixture_03_b300 as moe
from sparsely_gated_mixture_03_b300 import synthetic as S
from oracle import moe_oracle as O

DEV = "cuda"


def _outputs(T, n, k, d):
    R = T * k
    return (torch.full((n + 1,), -1, dtype=torch.int32, device=DEV),
            torch.full((R,), -1, dtype=torch.int32, device=DEV),
            torch.full((R,), -1, dtype=torch.int32, device=DEV),
            torch.zeros((R, d), dtype=torch.bfloat16, device=DEV))


@pytest.mark.gpu
def test_noalloc_dispatch_matches_dispatch_on_two_calls():
    T, n, k, d = 32768, 256, 4, 512            # the 256-expert workload's routing size
    cfg = moe.make_config(T, d, n, 1024, k)
    ws = moe.alloc_workspace(cfg)
    x = torch.randn((T, d), generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).to(DEV)
    for call, skew in enumerate((0.0, 1.1)):
        idx, _ = S.make_routing(T, n, k, seed=40 + call, skew=skew,
                                empty_experts=3 if call else 0)
        idx = idx.to(DEV)
        ref = _outputs(T, n, k, d)
        moe.moe_dispatch(cfg, idx, x, *ref, ws)
        got = _outputs(T, n, k, d)
        moe.moe_dispatch_noalloc(cfg, idx, x, *got)
        assert moe.moe_get_device_error() == 0
        for name, a, b in zip(("offsets", "perm", "inv", "x_perm"), got, ref):
            assert torch.equal(a, b), f"call {call}: {name} differs from moe_dispatch"
        for name, a, b in zip(("offsets", "perm", "inv"), got, O.dispatch(idx.cpu().numpy(), n)):
            assert np.array_equal(a.cpu().numpy(), b), f"call {call}: {name} differs from the oracle"


@pytest.mark.gpu
def test_noalloc_dispatch_rejects_shapes_beyond_its_scratch():
    # n = 4096 fits up to T*k = 64512 routed rows; one 1024-row tile more does not
    d = 64
    ok = moe.make_config(64512 // 4, d, 4096, 64, 4)
    big = moe.make_config(65536 // 4, d, 4096, 64, 4)
    for cfg, expect_ok in ((ok, True), (big, False)):
        R = cfg.T * cfg.k
        idx, _ = S.make_routing(cfg.T, cfg.n, cfg.k, seed=3)
        x = torch.zeros((cfg.T, d), dtype=torch.bfloat16, device=DEV)
        out = _outputs(cfg.T, cfg.n, cfg.k, d)
        if expect_ok:
            moe.moe_dispatch_noalloc(cfg, idx.to(DEV), x, *out)
            assert moe.moe_get_device_error() == 0
            assert int(out[0][cfg.n]) == R
        else:
            with pytest.raises(moe.MoeError) as e:
                moe.moe_dispatch_noalloc(cfg, idx.to(DEV), x, *out)
            assert e.value.status == 3          # MOE_ERR_WORKSPACE, nothing enqueued
