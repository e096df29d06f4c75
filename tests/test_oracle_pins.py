"""The fp64 oracle against what the pages and the mathematics fix (CPU only).

Every pin runs on the real oracle.  Then a set of plausible mistakes is
planted into fresh copies of the oracle module (on the CPU, never in the CUDA
path), and each planted mistake must fail at least one pin: evidence that the
pins constrain every step of the oracle.
"""
import importlib.util
import os

import numpy as np
import pytest

import oracle_pins
from conftest import ROOT

ORACLE_PATH = os.path.join(ROOT, "oracle", "moe_oracle.py")


def fresh_oracle(tag="clean"):
    spec = importlib.util.spec_from_file_location(f"_oracle_copy_{tag}", ORACLE_PATH)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(fresh_oracle())


# ---------------------------------------------------------------- planted mistakes

def _mut_kth_always_kth(O):
    orig = O.kth_excluding

    def kth(H, k, order=None):
        H = np.asarray(H, dtype=np.float64)
        if order is None:
            order = O.top_k_order(H, k)
        v = H[np.arange(H.shape[0]), order[:, k - 1]]
        return np.repeat(v[:, None], H.shape[1], axis=1)
    O.kth_excluding = kth
    return orig


def _mut_dense_softmax(O):
    def f(H, idx):
        H = np.asarray(H, dtype=np.float64)
        e = np.exp(H - H.max(axis=1, keepdims=True))
        p = e / e.sum(axis=1, keepdims=True)
        return np.take_along_axis(p, np.asarray(idx), axis=1)
    O.keep_top_k_softmax = f


def _mut_sample_variance(O):
    def f(v):
        v = np.asarray(v, dtype=np.float64)
        if v.size <= 1 or v.mean() == 0:
            return 0.0
        return float(v.var(ddof=1) / v.mean() ** 2)
    O.cv_squared = f


def _mut_softplus_is_exp(O):
    O.softplus = lambda z: np.exp(np.asarray(z, dtype=np.float64))


def _mut_no_relu(O):
    O.expert_ffn = lambda X, Wi, Wo: (np.asarray(X, float) @ np.asarray(Wi, float)) @ np.asarray(Wo, float)


def _mut_noise_dropped(O):
    orig = O.noisy_logits

    def f(x, W_g, W_noise, eps, std_floor=0.0, b_g=None):
        clean, std, H = orig(x, W_g, W_noise, eps, std_floor, b_g)
        return clean, std, clean.copy()
    O.noisy_logits = f


def _mut_P_uses_noisy_logit(O):
    def f(clean, std, H, k, order=None):
        thr = O.kth_excluding(H, k, order)
        return O.normal_cdf((np.asarray(H) - thr) / np.asarray(std))
    O.load_probability = f


def _mut_ties_to_high_index(O):
    def f(H, k):
        H = np.asarray(H, dtype=np.float64)
        n = H.shape[1]
        rev = np.argsort(-H[:, ::-1], axis=1, kind="stable")
        return (n - 1) - rev
    O.top_k_order = f


def _mut_gate_not_applied(O):
    orig = O.combine_by_expert

    def f(x, idx, gates, W_in, W_out, rows=None, keep=None):
        return orig(x, idx, np.ones_like(np.asarray(gates, float)), W_in, W_out, rows, keep)
    O.combine_by_expert = f


def _mut_dispatch_unstable(O):
    def f(idx, n, capacity=0):
        flat = np.asarray(idx).reshape(-1).astype(np.int64)
        counts = np.bincount(flat, minlength=n)
        offsets = np.concatenate([[0], np.cumsum(counts)])
        perm = np.lexsort((-np.arange(flat.size), flat))
        inv = np.empty_like(perm)
        inv[perm] = np.arange(perm.size)
        return offsets, perm, inv
    O.dispatch = f


def _mut_importance_counts(O):
    def f(idx, gates, n):
        return np.bincount(np.asarray(idx).ravel(), minlength=n).astype(np.float64)
    O.importance_of = f


def _mut_floor_dropped(O):
    orig = O.noisy_logits

    def f(x, W_g, W_noise, eps, std_floor=0.0, b_g=None):
        return orig(x, W_g, W_noise, eps, 0.0, b_g)
    O.noisy_logits = f


def _mut_bias_not_in_clean(O):
    orig = O.noisy_logits

    def f(x, W_g, W_noise, eps, std_floor=0.0, b_g=None):
        clean, std, H = orig(x, W_g, W_noise, eps, std_floor, None)
        if b_g is not None:
            H = H + np.asarray(b_g, float)[None, :]
        return clean, std, H
    O.noisy_logits = f


def _mut_product_gate_missing(O):
    orig = O.keep_top_k_softmax
    state = {"calls": 0}

    def f(H, idx):
        return orig(H, idx)
    O.keep_top_k_softmax = f
    orig_h = O.hier_forward

    def h(*a, **kw):
        out = orig_h(*a, **kw)
        # secondary gates only (primary factor dropped), a plausible slip
        k1 = a[9]
        k2 = a[10]
        g1 = out["gates1"]
        out["gates"] = out["gates"] / np.repeat(g1, k2, axis=1)
        out["y"] = O.combine_by_expert(np.asarray(a[0], float), out["idx"], out["gates"], a[7], a[8])
        return out
    O.hier_forward = h


def _mut_capacity_keeps_last(O):
    orig = O.capacity_keep

    def keep_last(idx, n, capacity=0):
        # an expert keeps its last rows instead of its first: a plausible slip
        idx = np.asarray(idx)
        rev = orig(idx.reshape(-1)[::-1].reshape(idx.shape), n, capacity)
        return rev.reshape(-1)[::-1].reshape(idx.shape)
    O.capacity_keep = keep_last


def _mut_capacity_off_by_one(O):
    orig = O.capacity_keep

    def one_more(idx, n, capacity=0):
        return orig(idx, n, capacity + 1 if capacity > 0 else 0)
    O.capacity_keep = one_more


def _mut_switch_renormalised(O):
    orig = O.switch_gating

    def f(*a, **kw):
        g = orig(*a, **kw)
        # gates renormalised over the kept experts: the noisy top-k softmax again
        g["gates"] = O.keep_top_k_softmax(g["H"], g["idx"])
        return g
    O.switch_gating = f


def _mut_switch_loss_unscaled(O):
    orig = O.switch_balance_loss

    def f(idx, p, n):
        loss, load, imp = orig(idx, p, n)
        return loss / n, load, imp          # the factor n forgotten
    O.switch_balance_loss = f


def _mut_backward_threshold_constant(O):
    orig = O.kth_excluding
    orig_bwd = O.moe_backward

    def f(*a, **kw):
        # the load thresholds treated as constants: their logits get no gradient
        saved = O.np.add.at
        calls = []

        def add_at(arr, ind, val):
            calls.append(1)
            if len(calls) > 1:     # the first add.at is the softmax's, the rest the thresholds'
                return None
            return saved(arr, ind, val)
        O.np.add.at = add_at
        try:
            return orig_bwd(*a, **kw)
        finally:
            O.np.add.at = saved
    O.moe_backward = f


def _mut_backward_relu_passes_all(O):
    orig_np = O.np

    class Shim:
        def __getattr__(self, name):
            return getattr(orig_np, name)

        @staticmethod
        def outer(a, b):
            return orig_np.outer(a, b)

    def f(x, W_g, W_noise, eps, W_in, W_out, k, dy, std_floor=0.0, b_g=None,
          w_importance=0.1, w_load=0.1):
        # ReLU'(u) taken as 1 everywhere: the expert input gradients ignore the clamp
        g = orig_bwd(x, W_g, W_noise, eps, W_in, W_out, k, dy, std_floor, b_g, w_importance, w_load)
        gates = O.gating(x, W_g, W_noise, eps, k, std_floor, b_g)
        for t in range(x.shape[0]):
            for j in range(k):
                e = gates["idx"][t, j]
                u = x[t] @ W_in[e]
                dE = gates["gates"][t, j] * dy[t]
                da = dE @ W_out[e].T
                g["dW_in"][e] += orig_np.outer(x[t], da * (u <= 0.0))
        return g
    orig_bwd = O.moe_backward
    O.moe_backward = f


def _mut_batchwise_ties_high(O):
    orig = O.batchwise_gating

    def f(x, W_g, W_noise, eps, k, std_floor=0.0, b_g=None, sel=None):
        # equal logits rank the higher token index first
        g = orig(x[::-1], W_g, W_noise, eps[::-1], k, std_floor, b_g)
        T = x.shape[0]
        g["sel"] = np.sort(T - 1 - g["sel"], axis=1)
        g["taken"] = g["taken"][::-1]
        g["G"] = g["G"][::-1]
        g["H"] = g["H"][::-1]
        return g
    O.batchwise_gating = f


def _mut_batchwise_softmax_over_all(O):
    orig = O.batchwise_gating

    def f(*a, **kw):
        g = orig(*a, **kw)
        # the softmax over every expert, masked afterwards: gates no longer sum to 1
        e = np.exp(g["H"] - g["H"].max(axis=1, keepdims=True))
        g["G"] = np.where(g["taken"], e / e.sum(axis=1, keepdims=True), 0.0)
        return g
    O.batchwise_gating = f


MUTATIONS = [
    _mut_kth_always_kth,
    _mut_dense_softmax,
    _mut_sample_variance,
    _mut_softplus_is_exp,
    _mut_no_relu,
    _mut_noise_dropped,
    _mut_P_uses_noisy_logit,
    _mut_ties_to_high_index,
    _mut_gate_not_applied,
    _mut_dispatch_unstable,
    _mut_importance_counts,
    _mut_floor_dropped,
    _mut_bias_not_in_clean,
    _mut_product_gate_missing,
    _mut_capacity_keeps_last,
    _mut_capacity_off_by_one,
    _mut_switch_renormalised,
    _mut_switch_loss_unscaled,
    _mut_backward_threshold_constant,
    _mut_backward_relu_passes_all,
    _mut_batchwise_ties_high,
    _mut_batchwise_softmax_over_all,
]


@pytest.mark.parametrize("mutate", MUTATIONS, ids=lambda f: f.__name__)
def test_planted_mistake_is_caught(mutate):
    O = fresh_oracle(mutate.__name__)
    mutate(O)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(O)
        except (AssertionError, ValueError, IndexError, KeyError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches {mutate.__name__}"


# Mistakes planted in the oracle's source text (for slips inside a function body):
# (name, the exact text replaced, its replacement).
SOURCE_MUTATIONS = [
    ("noise_radius_halved",
     "np.sqrt(-2.0 * np.log(u1))",
     "np.sqrt(-1.0 * np.log(u1))"),
    ("noise_counter_from_zero",
     "(j + np.uint64(1)) * np.uint64(0x9E3779B97F4A7C15)",
     "j * np.uint64(0x9E3779B97F4A7C15) * np.uint64(0)"),
    ("noise_pair_halves_equal",
     "out[1::2] = r * np.sin(2.0 * np.pi * u2)",
     "out[1::2] = r * np.cos(2.0 * np.pi * u2)"),
    ("sums_drop_last_chunk",
     "    for s in range(0, T, chunk):\n        e = min(T, s + chunk)",
     "    for s in range(0, T - T % chunk if T > chunk else T, chunk):\n        e = min(T, s + chunk)"),
    ("sums_eps_misaligned",
     "eps[s:e], k, std_floor, b_g,",
     "eps[(np.arange(s, e) + 1) % T], k, std_floor, b_g,"),
    ("sums_load_not_accumulated",
     '        load += g["P"].sum(axis=0)',
     '        load = g["P"].sum(axis=0)'),
    ("rows_eps_sorted",
     "g = gating(x[rows], W_g, W_noise, eps[rows], k, std_floor, b_g, kept)",
     "g = gating(x[rows], W_g, W_noise, eps[np.sort(rows)], k, std_floor, b_g, kept)"),
    ("rows_y_from_sorted_rows",
     'y = combine_by_expert(x[rows], g["idx"], g["gates"], W_in, W_out)',
     'y = combine_by_expert(x[np.sort(rows)], g["idx"], g["gates"], W_in, W_out)'),
    ("hier_load2_by_slot",
     'load2[gi * b:(gi + 1) * b] += g2["P"].sum(axis=0)',
     'load2[s * b:(s + 1) * b] += g2["P"].sum(axis=0)'),
    ("hier_eps2_first_slot",
     "_f64(eps2)[tt, s, :], k2, std_floor,",
     "_f64(eps2)[tt, 0, :], k2, std_floor,"),
    ("hier_flat_id_by_k2",
     'idx[tt, s * k2:(s + 1) * k2] = gi * b + g2["idx"]',
     'idx[tt, s * k2:(s + 1) * k2] = gi * k2 + g2["idx"]'),
    ("threshold_not_strict",
     "    taken = H > thr\n",
     "    taken = H >= thr\n"),
    ("threshold_softmax_over_all",
     "    return dict(taken=taken, G=_batchwise_gates(H, taken), H=H, sel=sel,",
     "    return dict(taken=taken, G=_batchwise_gates(H, np.ones_like(taken)) * taken, H=H, sel=sel,"),
    ("batch_sel_ignored",
     "        own = given\n",
     "        given = own\n"),
    ("kept_ignored",
     "idx = order[:, :k] if kept is None else check_kept(H, k, order, kept)",
     "idx = order[:, :k]"),
    ("kept_unchecked",
     "    T, n = H.shape\n    kept = np.asarray(kept).astype(np.int64).reshape(T, k)\n    if T == 0:",
     "    T, n = H.shape\n    kept = np.asarray(kept).astype(np.int64).reshape(T, k)\n    if True:"),
]


def oracle_from_source(tag, old, new):
    src = open(ORACLE_PATH).read()
    assert src.count(old) == 1, f"planted mistake {tag}: the text to replace is not unique"
    mod = type(importlib)("_oracle_src_" + tag)
    mod.__file__ = ORACLE_PATH
    exec(compile(src.replace(old, new), ORACLE_PATH, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("tag,old,new", SOURCE_MUTATIONS, ids=[m[0] for m in SOURCE_MUTATIONS])
def test_planted_source_mistake_is_caught(tag, old, new):
    O = oracle_from_source(tag, old, new)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(O)
        except (AssertionError, ValueError, IndexError, KeyError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches {tag}"
