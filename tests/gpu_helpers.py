"""Shared helpers of the GPU parity tests: run the library's entry points on
seeded inputs and compare with the fp64 oracle under the stated tolerances.

Tolerances (the layer's correctness criteria):
* expert indices and dispatch permutations: bit-exact, except rows whose k-th
  and (k+1)-th noisy logits differ by less than 1e-5 in the oracle (a near tie,
  where either choice is correct; only its validity is checked);
* logits, gates, Importance, Load and the losses: relative 1e-5, read as
  |got - ref| <= 1e-5 * max(|ref|, RMS(ref)) (a pure relative test is ill-posed
  for entries near 0);
* layer outputs: max |got - ref| <= 2e-2 * RMS(ref) with bf16 experts,
  <= 1e-4 * RMS(ref) with fp32 experts.

Where a near-tie row kept another valid expert set, every downstream quantity
(the row's gates and output, Importance, the losses) is still checked in full:
the oracle is rerun with the GPU's kept set (``kept=``), which it accepts only
as a valid tie-break of its own fp64 logits, and the results are compared at
the tolerances above, never with a slack that grows with the number of ties.
"""
from __future__ import annotations

import numpy as np
import torch

import sparsely_gated_mixture_03_b300 as moe
from oracle import moe_oracle as O

REL = 1e-5


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def scaled_err(got, ref):
    """max |got - ref| / max(|ref|, RMS(ref)) over all entries."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), rms)
    den = np.where(den == 0, 1.0, den)
    return float(np.max(np.abs(got - ref) / den))


def assert_rel(got, ref, what, rel=REL):
    e = scaled_err(got, ref)
    assert e <= rel, f"{what}: scaled error {e:.3e} > {rel:.0e}"


def assert_y(got, ref, bf16, what="y"):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    if ref.size == 0:
        return
    rms = float(np.sqrt(np.mean(ref * ref)))
    tol = (2e-2 if bf16 else 1e-4) * rms
    err = float(np.max(np.abs(got - ref)))
    assert err <= tol, f"{what}: max-abs {err:.3e} > {tol:.3e} (RMS {rms:.3e})"


def config_for(shape, std_floor=0.0):
    return moe.make_config(shape.T, shape.d, shape.n, shape.h, shape.k, shape.x_dtype,
                           shape.expert_dtype, std_floor=std_floor)


def oracle_arrays(inp: dict) -> dict:
    """Host fp64 copies of the generated inputs (bf16 values decoded exactly)."""
    return {k: (None if v is None else np64(v)) for k, v in inp.items()}


def run_gate(cfg, inp, ws, logits=True):
    T, n, k = cfg.T, cfg.n, cfg.k
    dev = inp["x"].device
    out = dict(idx=torch.empty(T * k, dtype=torch.int32, device=dev),
               gates=torch.empty(T * k, dtype=torch.float32, device=dev),
               tie=torch.empty(T, dtype=torch.uint8, device=dev),
               load=torch.empty(n, dtype=torch.float32, device=dev),
               logits=torch.empty(3 * T * n, dtype=torch.float32, device=dev) if logits else None)
    moe.moe_gate(cfg, inp["x"], inp["W_g"], inp["W_noise"], inp["eps"], inp["b_g"], out["idx"],
                 out["gates"], out["tie"], out["load"], out["logits"], ws)
    return out


def check_selection(idx_gpu, gates_gpu, ref, k, what="gate"):
    """idx/gates of the GPU against the oracle gating dict ``ref``.

    Rows without a near tie at the k-th place: the kept set and its order are
    bit-exact (order compared up to near ties inside the kept set), gates
    within REL.  Near-tie rows: every kept expert's oracle logit must be within
    the tie gap of the oracle's k-th logit (a valid choice).
    Returns the boolean mask of rows whose kept set equals the oracle's.
    """
    idx_gpu = np.asarray(idx_gpu).reshape(-1, k)
    gates_gpu = np.asarray(gates_gpu, np.float64).reshape(-1, k)
    T = idx_gpu.shape[0]
    ref_idx, ref_g, H = ref["idx"], ref["gates"], ref["H"]
    same_set = np.array([set(idx_gpu[t]) == set(ref_idx[t]) for t in range(T)])
    tie = ref["tie"]
    bad = np.nonzero(~tie & ~same_set)[0]
    assert bad.size == 0, f"{what}: {bad.size} unflagged rows keep other experts, e.g. row {bad[:5]}"
    # order inside the kept set: exact unless two kept logits are within the tie gap
    Hk = np.take_along_axis(H, ref_idx, axis=1)
    inner_tie = (np.abs(np.diff(Hk, axis=1)) < O.TIE_GAP).any(axis=1) if k > 1 else np.zeros(T, bool)
    strict = same_set & ~inner_tie
    assert np.array_equal(idx_gpu[strict], ref_idx[strict]), f"{what}: kept order differs"
    # gates matched by expert id on rows with the same set
    rows = np.nonzero(same_set)[0]
    if rows.size:
        o_gpu = np.argsort(idx_gpu[rows], axis=1)
        o_ref = np.argsort(ref_idx[rows], axis=1)
        g1 = np.take_along_axis(gates_gpu[rows], o_gpu, axis=1)
        g2 = np.take_along_axis(ref_g[rows], o_ref, axis=1)
        assert_rel(g1, g2, f"{what}: gates")
    # near-tie rows that chose differently: each chosen logit within the gap of the k-th
    for t in np.nonzero(~same_set)[0]:
        kth = H[t, ref["order"][t, k - 1]] if "order" in ref else np.sort(H[t])[::-1][k - 1]
        assert all(H[t, e] >= kth - 2 * O.TIE_GAP for e in idx_gpu[t]), f"{what}: row {t} invalid"
        assert len(set(idx_gpu[t])) == k
    return same_set


def own_selection(ref, k):
    """The oracle's own top-k choice from a gating dict computed with ``kept=``
    (its order and logits are its own; idx and gates are recomputed from them),
    for ``check_selection``."""
    idx = ref["order"][:, :k]
    return dict(idx=idx, gates=O.keep_top_k_softmax(ref["H"], idx), H=ref["H"], tie=ref["tie"],
                order=ref["order"])


def kept_of(idx_gpu, k):
    """The GPU's kept experts as an int64 [T, k] array (the oracle's ``kept=``)."""
    return np.asarray(idx_gpu).astype(np.int64).reshape(-1, k)
