"""Pins for the fp64 oracle, written as functions of the oracle module ``O``.

Each pin checks the oracle against something other than itself: a value the
page prints (fixtures under tests/golden/, each with its citation), a closed
form, brute force on tiny inputs, a Monte-Carlo estimate of a probability,
or an invariant.  ``tests/test_oracle_pins.py`` runs them on the real oracle
and on mutated copies (planted mistakes) to show that each plausible mistake
fails at least one pin.
"""
import itertools
import math

import numpy as np

from conftest import golden


def _x_is_logits(logits):
    """Inputs for which the gate's noisy logits equal ``logits`` exactly:
    d = 1, x = 1, W_g = logits, W_noise = 0, eps = 0."""
    logits = np.asarray(logits, dtype=np.float64)[None, :]
    n = logits.shape[1]
    return np.ones((1, 1)), logits, np.zeros((1, n)), np.zeros((1, n))


def pin_worked_example_gates(O):
    g = golden("worked_example_gates.txt")
    n, k = int(g["n"]), int(g["k"])
    logits = np.array([0.0] * n)
    fill = iter([1.0, 0.3, -0.2, 0.9, -1.1])          # the five lost entries, all < 1.4
    named = {int(e): v for e, v in g["logit"]}
    for i in range(n):
        logits[i] = named.get(i + 1, None) if (i + 1) in named else next(fill)
    x, W_g, W_noise, eps = _x_is_logits(logits)
    out = O.gating(x, W_g, W_noise, eps, k)
    kept = [int(v) - 1 for v in g["kept"]]
    assert list(out["idx"][0]) == kept
    gates = dict(zip(out["idx"][0], out["gates"][0]))
    dec = int(g["decimals"])
    for e, val in g["gate"]:
        assert round(gates[int(e) - 1], dec) == val
    assert abs(out["gates"][0].sum() - 1.0) < 1e-15
    # d G_4 / d logit_4 = G(1 - G) = 0.25 (central difference through the gate)
    h = 1e-6
    up, dn = logits.copy(), logits.copy()
    up[kept[0]] += h
    dn[kept[0]] -= h
    gu = O.gating(*_x_is_logits(up), k)["gates"][0][0]
    gd = O.gating(*_x_is_logits(dn), k)["gates"][0][0]
    assert round((gu - gd) / (2 * h), dec) == g["dgate"]
    # expert 1 "missed by 0.1": 0.11 more and it replaces expert 5
    bumped = logits.copy()
    bumped[0] += 0.11
    out2 = O.gating(*_x_is_logits(bumped), k)
    assert sorted(out2["idx"][0]) == sorted([kept[0], 0])


def pin_importance_cv2(O):
    g = golden("importance_cv2.txt")
    imp = np.array(g["importance"])
    assert abs(imp.sum() - g["batch"]) < 1e-12
    cv2 = O.cv_squared(imp)
    assert abs(cv2 - g["cv2"]) < 1e-12
    assert abs(g["w"] * cv2 - g["loss"]) < 1e-12
    # gradient with the mean held fixed: derivative along e_i - (1/n) sum e_j
    n = imp.size
    h = 1e-6
    grads = []
    for i in range(n):
        dv = -np.full(n, 1.0 / n)
        dv[i] += 1.0
        grads.append((O.cv_squared(imp + h * dv) - O.cv_squared(imp - h * dv)) / (2 * h))
    assert abs(grads[0] - g["grad_first"]) < 1e-6
    assert abs(grads[-1] - g["grad_last"]) < 1e-6
    # Importance through eq (6): a batch of 8 rows of top-2 gates whose column sums are imp
    idx = np.array([[0, 1]] * 4 + [[0, 2]] * 2 + [[0, 3]] * 2)
    gates = np.array([[0.4, 0.6]] * 4      # e0 += 1.6, e1 += 2.4
                     + [[0.4, 0.6]] * 2    # e0 += 0.8, e2 += 1.2
                     + [[0.6, 0.4]] * 2)   # e0 += 1.2, e3 += 0.8
    got = O.importance_of(idx, gates, n)
    assert np.allclose(got, imp, atol=1e-12, rtol=0)
    # scale invariance and the balanced case
    assert abs(O.cv_squared(3.7 * imp) - cv2) < 1e-12
    assert O.cv_squared(np.full(7, 2.5)) == 0.0


def pin_load_probability_example(O):
    g = golden("load_probability.txt")
    clean, sigma, thr = g["clean"], g["sigma"], g["threshold"]
    raw = math.log(math.expm1(sigma))                 # Softplus(raw) = sigma
    dec = int(g["decimals"])
    # n = 3, k = 1; expert 1 carries the threshold (H = 1.3, no noise), expert 2 is far below.
    for eps0 in (0.0, 2.0):                           # expert 0 out of / in the top 1
        x = np.ones((1, 1))
        W_g = np.array([[clean, thr, -5.0]])
        W_noise = np.array([[raw, -40.0, -40.0]])
        eps = np.array([[eps0, 0.0, 0.0]])
        out = O.gating(x, W_g, W_noise, eps, 1)
        assert (out["idx"][0, 0] == 0) == (eps0 > 0)
        P = out["P"][0, 0]
        assert abs(P - 0.2742531177500736) < 1e-12
        assert round(P, dec) == g["P"]
        h = 1e-6
        Pu = O.gating(x, W_g + [[h, 0, 0]], W_noise, eps, 1)["P"][0, 0]
        Pd = O.gating(x, W_g - [[h, 0, 0]], W_noise, eps, 1)["P"][0, 0]
        slope = (Pu - Pd) / (2 * h)
        assert abs(slope - math.exp(-0.18) / math.sqrt(2 * math.pi) / sigma) < 1e-6
        assert round(slope, dec) == g["dP_dclean"]


def pin_kth_excluding_brute_force(O):
    rng = np.random.default_rng(11)
    for n, k in [(5, 1), (6, 2), (8, 3), (7, 6), (4, 4)]:
        for trial in range(30):
            if trial % 3 == 0:
                H = rng.integers(-2, 3, size=(3, n)).astype(np.float64)  # many ties
            else:
                H = rng.normal(size=(3, n))
            thr = O.kth_excluding(H, k)
            for t in range(3):
                for i in range(n):
                    others = sorted((H[t, j] for j in range(n) if j != i), reverse=True)
                    want = others[k - 1] if k - 1 < len(others) else -np.inf
                    assert thr[t, i] == want, (n, k, t, i)


def pin_topk_brute_force(O):
    """eps = 0 and W_noise = 0: KeepTopK equals a brute-force sort of the clean
    logits (ties to the lower index)."""
    rng = np.random.default_rng(3)
    for n, k, d in [(8, 2, 5), (16, 4, 7), (5, 5, 3), (9, 1, 4)]:
        x = rng.normal(size=(20, d))
        W_g = rng.normal(size=(d, n))
        if n == 16:
            W_g[:, 7] = W_g[:, 3]                      # exact ties between experts 3 and 7
        out = O.gating(x, W_g, np.zeros((d, n)), np.zeros((20, n)), k)
        clean = x @ W_g
        for t in range(20):
            want = sorted(range(n), key=lambda i: (-clean[t, i], i))[:k]
            assert list(out["idx"][t]) == want
            e = [math.exp(clean[t, i]) for i in want]
            assert np.allclose(out["gates"][t], [v / sum(e) for v in e], rtol=1e-13, atol=0)


def pin_gate_invariants(O):
    rng = np.random.default_rng(5)
    T, d, n = 64, 6, 10
    x = rng.normal(size=(T, d))
    W_g, W_noise = rng.normal(size=(d, n)), rng.normal(size=(d, n))
    eps = rng.normal(size=(T, n))
    for k in (1, 2, 4, n):
        out = O.gating(x, W_g, W_noise, eps, k)
        G = np.zeros((T, n))
        np.put_along_axis(G, out["idx"], out["gates"], axis=1)
        assert ((G > 0).sum(axis=1) == k).all()            # exactly k nonzero gates
        assert np.allclose(G.sum(axis=1), 1.0, atol=1e-14)  # each row sums to 1
        if k == 1:
            assert (out["gates"] == 1.0).all()              # a single kept logit gives exactly 1
        imp = O.importance_of(out["idx"], out["gates"], n)
        assert abs(imp.sum() - T) < 1e-10                   # importances sum to the batch size
        assert ((out["P"] >= 0) & (out["P"] <= 1)).all()


def pin_noisy_logits_closed_form(O):
    """H = x W_g + eps * (log(1 + e^{x W_noise}) + floor) entry by entry."""
    rng = np.random.default_rng(8)
    T, d, n = 4, 3, 5
    x, W_g, W_noise = rng.normal(size=(T, d)), rng.normal(size=(d, n)), rng.normal(size=(d, n))
    W_noise[0, 0] = 60.0                                    # a large softplus argument
    eps = rng.normal(size=(T, n))
    b = rng.normal(size=n)
    for floor in (0.0, 0.01):
        clean, std, H = O.noisy_logits(x, W_g, W_noise, eps, floor, b)
        for t in range(T):
            for i in range(n):
                c = sum(x[t, j] * W_g[j, i] for j in range(d)) + b[i]
                z = sum(x[t, j] * W_noise[j, i] for j in range(d))
                s = (z + math.log1p(math.exp(-z)) if z > 0 else math.log1p(math.exp(z))) + floor
                assert abs(clean[t, i] - c) < 1e-12
                assert abs(std[t, i] - s) < 1e-12 * max(1, abs(s))
                assert abs(H[t, i] - (c + eps[t, i] * s)) < 1e-11 * max(1, abs(s))


def pin_load_monte_carlo(O):
    """P(x, i) is the probability that a fresh noise draw for expert i alone
    puts i in the top k (eq (8)): resample eps_i, count selections."""
    rng = np.random.default_rng(21)
    d, n, k = 4, 6, 2
    x = rng.normal(size=(1, d))
    W_g, W_noise = 0.6 * rng.normal(size=(d, n)), 0.6 * rng.normal(size=(d, n))
    eps = rng.normal(size=(1, n))
    base = O.gating(x, W_g, W_noise, eps, k)
    draws = 40000
    for i in range(n):
        E = np.repeat(eps, draws, axis=0)
        E[:, i] = rng.normal(size=draws)
        out = O.gating(np.repeat(x, draws, axis=0), W_g, W_noise, E, k)
        freq = (out["idx"] == i).any(axis=1).mean()
        p = base["P"][0, i]
        assert abs(freq - p) < 5 * math.sqrt(max(p * (1 - p), 1e-4) / draws) + 1e-3, (i, freq, p)


def pin_zero_init(O):
    g = golden("zero_init.txt")
    rng = np.random.default_rng(9)
    T, d, n, k = 20000, 8, 8, 2
    x = rng.normal(size=(T, d))
    eps = rng.normal(size=(T, n))
    out = O.gating(x, np.zeros((d, n)), np.zeros((d, n)), eps, k)
    assert np.all(out["std"] == math.log(2.0))
    assert round(out["std"][0, 0], int(g["decimals"])) == g["softplus0"]
    counts = np.bincount(out["idx"].ravel(), minlength=n)
    expect = T * k / n
    chi2 = ((counts - expect) ** 2 / expect).sum()
    assert chi2 < 30.0                                      # dof 7: p ~ 1e-4 at 30


def pin_expert_ffn_brute_force(O):
    rng = np.random.default_rng(4)
    m, d, h = 3, 4, 5
    X, Wi, Wo = rng.normal(size=(m, d)), rng.normal(size=(d, h)), rng.normal(size=(h, d))
    got = O.expert_ffn(X, Wi, Wo)
    for r in range(m):
        hid = [max(0.0, sum(X[r, a] * Wi[a, c] for a in range(d))) for c in range(h)]
        for c in range(d):
            assert abs(got[r, c] - sum(hid[q] * Wo[q, c] for q in range(h))) < 1e-12
    # identity experts: n = 1, k = 1, W_in = W_out = I -> y = ReLU(x) * 1
    x = rng.normal(size=(6, d))
    I = np.eye(d)[None]
    y = O.combine_by_expert(x, np.zeros((6, 1), dtype=np.int64), np.ones((6, 1)), I, I)
    assert np.array_equal(y, np.maximum(x, 0.0))


def pin_dense_equals_sparse(O):
    """k = n: the sparse combine equals the dense all-experts sum, the load
    probability is 1 everywhere and CV^2(Load) = 0."""
    rng = np.random.default_rng(6)
    T, d, n, h = 5, 3, 4, 6
    x = rng.normal(size=(T, d))
    W_g, W_noise = rng.normal(size=(d, n)), rng.normal(size=(d, n))
    eps = rng.normal(size=(T, n))
    W_in, W_out = rng.normal(size=(n, d, h)), rng.normal(size=(n, h, d))
    out = O.moe_forward(x, W_g, W_noise, eps, W_in, W_out, n)
    clean = x @ W_g
    raw = x @ W_noise
    for t in range(T):
        Hs = [clean[t, i] + eps[t, i] * math.log1p(math.exp(raw[t, i])) for i in range(n)]
        den = sum(math.exp(v) for v in Hs)
        y = np.zeros(d)
        for i in range(n):
            hid = np.maximum(x[t] @ W_in[i], 0.0)
            y += math.exp(Hs[i]) / den * (hid @ W_out[i])
        assert np.allclose(out["y"][t], y, rtol=1e-12, atol=1e-12)
    assert np.all(out["P"] == 1.0)
    assert np.allclose(out["load"], T)
    assert out["losses"][1] == 0.0


def pin_combine_gathered_matches_by_expert(O):
    """Eq (1) evaluated from expert-grouped outputs (dispatch, run each expert
    on its rows, gather back) equals the per-expert loop of the listing."""
    rng = np.random.default_rng(14)
    T, d, n, h, k = 9, 3, 5, 4, 2
    x = rng.normal(size=(T, d))
    idx = np.array([rng.choice(n, size=k, replace=False) for _ in range(T)])
    gates = rng.uniform(0.1, 1.0, size=(T, k))
    W_in, W_out = rng.normal(size=(n, d, h)), rng.normal(size=(n, h, d))
    offsets, perm, inv = O.dispatch(idx, n)
    y_perm = np.zeros((T * k, d))
    for e in range(n):
        p = perm[offsets[e]:offsets[e + 1]]
        y_perm[offsets[e]:offsets[e + 1]] = O.expert_ffn(x[p // k], W_in[e], W_out[e])
    got = O.combine_gathered(y_perm, inv, gates)
    want = O.combine_by_expert(x, idx, gates, W_in, W_out)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)


def pin_dispatch_brute_force(O):
    rng = np.random.default_rng(12)
    for T, n, k in [(1, 3, 1), (7, 5, 2), (13, 4, 3), (9, 9, 4)]:
        idx = np.array([rng.choice(n, size=k, replace=False) for _ in range(T)])
        offsets, perm, inv = O.dispatch(idx, n)
        rows = []
        for e in range(n):
            start = len(rows)
            for t in range(T):
                for j in range(k):
                    if idx[t, j] == e:
                        rows.append(t * k + j)
            assert offsets[e] == start
        assert offsets[n] == T * k
        assert list(perm) == rows
        for p, r in enumerate(rows):
            assert inv[r] == p


def pin_capacity(O):
    """Fixed per-expert capacity ("From LSTMs to Switch and Mixtral": inputs
    beyond an expert's capacity skip it).  A case worked by hand; a capacity at
    or above every expert's count (or 0) changes nothing; an expert keeps
    min(count, C) rows, all before any row it drops; and the capped layer
    output equals the uncapped gathered combine with the dropped rows' gates
    set to zero."""
    # worked by hand: routed rows r = 0..7 go to experts 0 1 0 2 0 1 1 0
    idx = np.array([[0, 1], [0, 2], [0, 1], [1, 0]])
    keep = O.capacity_keep(idx, 3, 2)
    assert keep.tolist() == [[True, True], [True, True], [False, True], [False, False]]
    offsets, perm, inv = O.dispatch(idx, 3, 2)
    assert offsets.tolist() == [0, 2, 4, 5]
    assert perm.tolist() == [0, 2, 1, 5, 3]
    assert inv.tolist() == [0, 2, 1, 4, -1, 3, -1, -1]

    rng = np.random.default_rng(21)
    T, n, k, d, h = 40, 6, 3, 4, 5
    idx = np.array([rng.choice(n, size=k, replace=False) for _ in range(T)])
    counts = np.bincount(idx.reshape(-1), minlength=n)
    full = O.dispatch(idx, n)
    for C in (0, int(counts.max()), int(counts.max()) + 3):
        for a, b in zip(O.dispatch(idx, n, C), full):
            assert np.array_equal(a, b)
    x = rng.normal(size=(T, d))
    W_in, W_out = rng.normal(size=(n, d, h)), rng.normal(size=(n, h, d))
    gates = rng.uniform(0.1, 1.0, size=(T, k))
    off_f, perm_f, inv_f = full
    y_perm = np.zeros((T * k, d))
    for e in range(n):
        for p in range(off_f[e], off_f[e + 1]):
            y_perm[p] = O.expert_ffn(x[perm_f[p] // k][None], W_in[e], W_out[e])[0]
    for C in (1, 2, 5):
        offsets, perm, inv = O.dispatch(idx, n, C)
        assert np.array_equal(np.diff(offsets), np.minimum(counts, C))
        keep = O.capacity_keep(idx, n, C).reshape(-1)
        flat = idx.reshape(-1)
        for e in range(n):
            r_keep = np.nonzero((flat == e) & keep)[0]
            r_drop = np.nonzero((flat == e) & ~keep)[0]
            assert r_keep.size == min(counts[e], C)
            if r_keep.size and r_drop.size:
                assert r_keep.max() < r_drop.min()
        assert np.array_equal(inv[perm], np.arange(perm.size))
        assert np.all(inv[~keep] == -1)
        y_cap = O.combine_by_expert(x, idx, gates, W_in, W_out, keep=keep.reshape(T, k))
        y_ref = O.combine_gathered(y_perm, inv_f, gates * keep.reshape(T, k))
        assert np.allclose(y_cap, y_ref, rtol=1e-12, atol=1e-12)


def pin_switch_gate(O):
    """The Switch gate and loss ("From LSTMs to Switch and Mixtral").  Worked by
    hand: logits 1.7, 1.5, 1.4, 0 (three of them the page's worked example) give
    the kept expert the probability e^1.7 / (e^1.7 + e^1.5 + e^1.4 + 1) =
    0.364666, below the noisy top-1 gate of exactly 1.  k = n gives the full
    softmax (the noisy top-k gates).  A Switch gate over the k kept is the
    top-k gate times the kept probability mass.  The loss: uniform
    probabilities give exactly 1 whatever the routing; two hand cases give 1.0
    and 1.4."""
    H = np.array([[1.7, 1.5, 1.4, 0.0]])
    d = 4
    x = np.eye(d)[:1]                     # x = e_0, so clean = W_g[0]
    W_g = np.zeros((d, 4))
    W_g[0] = H[0]
    g = O.switch_gating(x, W_g, np.zeros((d, 4)), np.zeros((1, 4)), 1)
    assert g["idx"].tolist() == [[0]]
    assert abs(g["gates"][0, 0] - 0.364666) < 5e-7
    assert O.gating(x, W_g, np.zeros((d, 4)), np.zeros((1, 4)), 1)["gates"][0, 0] == 1.0

    rng = np.random.default_rng(31)
    T, n, dd = 12, 6, 5
    x = rng.normal(size=(T, dd))
    W_g, W_n = rng.normal(size=(dd, n)), rng.normal(size=(dd, n))
    eps = rng.normal(size=(T, n))
    full = O.switch_gating(x, W_g, W_n, eps, n)
    top = O.gating(x, W_g, W_n, eps, n)
    assert np.allclose(full["gates"], top["gates"], rtol=1e-13, atol=0)
    assert np.allclose(full["gates"].sum(axis=1), 1.0, rtol=1e-13)
    for k in (1, 2, 3):
        sg = O.switch_gating(x, W_g, W_n, eps, k)
        tg = O.gating(x, W_g, W_n, eps, k)
        assert np.array_equal(sg["idx"], tg["idx"])
        mass = np.take_along_axis(sg["p"], sg["idx"], axis=1).sum(axis=1, keepdims=True)
        assert np.allclose(sg["gates"], tg["gates"] * mass, rtol=1e-12)
        assert np.all(sg["gates"] < tg["gates"])

    # the loss
    for idx in ([[0], [3]], [[1], [1]], [[2, 0], [1, 0]]):
        loss, load, imp = O.switch_balance_loss(np.array(idx), np.full((2, 4), 0.25), 4)
        assert abs(loss - 1.0) < 1e-15
    p = np.array([[0.8, 0.2], [0.3, 0.7]])
    assert abs(O.switch_balance_loss(np.array([[0], [1]]), p, 2)[0] - 1.0) < 1e-15
    p = np.array([[0.8, 0.2], [0.6, 0.4]])
    loss, load, imp = O.switch_balance_loss(np.array([[0], [0]]), p, 2)
    assert abs(loss - 1.4) < 1e-15
    assert load.tolist() == [2.0, 0.0] and np.allclose(imp, [1.4, 0.6])


def _fd_grad(O, args, name, k, dy, floor, w_imp, w_load, h=1e-6):
    """Central differences of the oracle's scalar loss in one argument."""
    arr = args[name]
    num = np.zeros_like(arr)
    for i in np.ndindex(arr.shape):
        vals = []
        for sgn in (1.0, -1.0):
            a = dict(args)
            a[name] = arr.copy()
            a[name][i] += sgn * h
            vals.append(O.moe_loss(a["x"], a["W_g"], a["W_noise"], a["eps"], a["W_in"],
                                   a["W_out"], k, dy, floor, a["b_g"], w_imp, w_load))
        num[i] = (vals[0] - vals[1]) / (2.0 * h)
    return num


def pin_backward_finite_differences(O):
    """The backward ("Implementation notes": which parameters get gradient and by
    which path) against central finite differences of the forward pass's loss
    sum(dy * y) + w_imp CV^2(I) + w_load CV^2(L), for every parameter, on tiny
    inputs with k = 1, 2 and n (k = n: the load is constant); and the page's
    remark that W_g gets no task gradient when k = 1 (the gate is exactly 1)."""
    rng = np.random.default_rng(41)
    T, d, n, h = 5, 4, 4, 6
    for k, floor, w_imp, w_load, bias in [(2, 0.01, 0.3, 0.7, True), (1, 0.0, 0.2, 0.5, False),
                                          (4, 0.0, 0.4, 0.6, True)]:
        args = dict(x=rng.normal(size=(T, d)), W_g=rng.normal(size=(d, n)),
                    W_noise=0.5 * rng.normal(size=(d, n)), eps=rng.normal(size=(T, n)),
                    W_in=rng.normal(size=(n, d, h)), W_out=rng.normal(size=(n, h, d)),
                    b_g=rng.normal(size=n) if bias else None)
        dy = rng.normal(size=(T, d))
        gr = O.moe_backward(args["x"], args["W_g"], args["W_noise"], args["eps"], args["W_in"],
                            args["W_out"], k, dy, floor, args["b_g"], w_imp, w_load)
        names = ["x", "W_g", "W_noise", "W_in", "W_out"] + (["b_g"] if bias else [])
        for name in names:
            num = _fd_grad(O, args, name, k, dy, floor, w_imp, w_load)
            got = gr["d" + name]
            scale = max(1e-12, float(np.max(np.abs(num))))
            assert float(np.max(np.abs(got - num))) <= 1e-6 * scale, (k, name)
    # k = 1 and no load loss: the gate is 1, so W_g and W_noise get nothing from the task
    args = dict(x=rng.normal(size=(T, d)), W_g=rng.normal(size=(d, n)),
                W_noise=rng.normal(size=(d, n)), eps=rng.normal(size=(T, n)),
                W_in=rng.normal(size=(n, d, h)), W_out=rng.normal(size=(n, h, d)))
    gr = O.moe_backward(args["x"], args["W_g"], args["W_noise"], args["eps"], args["W_in"],
                        args["W_out"], 1, rng.normal(size=(T, d)), 0.0, None, 0.0, 0.0)
    assert not gr["dW_g"].any() and not gr["dW_noise"].any()


def pin_batchwise(O):
    """The batchwise top-m gate (the Appendix F gate the page describes): a case
    worked by hand (each expert takes the two tokens with its largest logits), ties
    going to the lower token index, brute force against a Python sort on tiny inputs,
    every expert taking exactly m tokens, a token's gates summing to 1 (0 when no
    expert took it), and k = n reducing to the flat layer with k = n."""
    d = 2
    x = np.eye(d)[[0, 0, 0, 0]]
    H = np.array([[3.0, 0.0], [2.0, 1.0], [1.0, 2.0], [0.0, 3.0]])
    # clean = x W_g = W_g[0] for every token; build per-token logits through eps instead
    W_g = np.zeros((d, 2))
    W_n = np.full((d, 2), 50.0)            # std = softplus(50) = 50 (to 1e-20)
    eps = H / 50.0
    g = O.batchwise_gating(x, W_g, W_n, eps, 1)
    assert g["m"] == 2 and g["sel"].tolist() == [[0, 1], [2, 3]]
    assert np.allclose(g["G"], [[1, 0], [1, 0], [0, 1], [0, 1]])
    # a near tie at the m-th place: another valid choice is accepted and its gates
    # follow it; a far one is refused
    Hn = np.array([[3.0, 0.0], [2.0 + 4e-6, 1.0], [2.0, 2.0], [0.0, 3.0]])
    gn = O.batchwise_gating(x, W_g, W_n, Hn / 50.0, 1)
    assert gn["sel"].tolist() == [[0, 1], [2, 3]]
    alt = O.batchwise_gating(x, W_g, W_n, Hn / 50.0, 1, sel=[[0, 2], [2, 3]])
    assert alt["sel"].tolist() == [[0, 2], [2, 3]]
    assert np.allclose(alt["G"][2], [0.5, 0.5], atol=1e-9) and not alt["G"][1].any()
    try:
        O.batchwise_gating(x, W_g, W_n, Hn / 50.0, 1, sel=[[0, 3], [2, 3]])
    except ValueError:
        pass
    else:
        raise AssertionError("a token far below the m-th logit was accepted")
    # ties: equal logits, the lower token index first
    g = O.batchwise_gating(x, W_g, W_n, np.zeros((4, 2)), 1)
    assert g["sel"].tolist() == [[0, 1], [0, 1]]
    assert np.allclose(g["G"][:2], 0.5) and not g["G"][2:].any()

    rng = np.random.default_rng(61)
    for T, n, k in [(9, 3, 1), (16, 4, 2), (13, 5, 3)]:
        dd = 3
        x = rng.normal(size=(T, dd))
        W_g, W_n = rng.normal(size=(dd, n)), rng.normal(size=(dd, n))
        eps = rng.normal(size=(T, n))
        g = O.batchwise_gating(x, W_g, W_n, eps, k)
        m = (k * T) // n
        Hh = g["H"]
        for i in range(n):
            ranked = sorted(range(T), key=lambda t: (-Hh[t, i], t))
            assert sorted(ranked[:m]) == g["sel"][i].tolist()
        assert np.all(g["taken"].sum(axis=0) == m)
        sums = g["G"].sum(axis=1)
        assert np.allclose(sums[g["taken"].any(axis=1)], 1.0)
        assert not sums[~g["taken"].any(axis=1)].any()
    T, dd, n, h = 7, 3, 4, 5
    x = rng.normal(size=(T, dd))
    W_g, W_n = rng.normal(size=(dd, n)), rng.normal(size=(dd, n))
    eps = rng.normal(size=(T, n))
    W_in, W_out = rng.normal(size=(n, dd, h)), rng.normal(size=(n, h, dd))
    flat = O.moe_forward(x, W_g, W_n, eps, W_in, W_out, n)
    bw = O.moe_forward_batchwise(x, W_g, W_n, eps, W_in, W_out, n)      # m = T
    assert np.allclose(bw["y"], flat["y"], rtol=1e-12, atol=1e-12)


def pin_hierarchical_reductions(O):
    """a = 1: one group holding all b experts is the flat MoE over b experts.
    b = 1: one expert per group is the flat MoE over the a groups.  Product
    gates sum to 1 per token."""
    rng = np.random.default_rng(13)
    T, d, h = 6, 4, 5
    # a = 1, flat over b = 5 experts with k2 = 2
    b = 5
    W_g2, W_n2 = rng.normal(size=(1, d, b)), rng.normal(size=(1, d, b))
    W_in, W_out = rng.normal(size=(b, d, h)), rng.normal(size=(b, h, d))
    x = rng.normal(size=(T, d))
    eps2 = rng.normal(size=(T, 1, b))
    hier = O.hier_forward(x, np.zeros((d, 1)), np.zeros((d, 1)), np.zeros((T, 1)),
                          W_g2, W_n2, eps2, W_in, W_out, 1, 2)
    flat = O.moe_forward(x, W_g2[0], W_n2[0], eps2[:, 0, :], W_in, W_out, 2)
    assert np.array_equal(hier["idx"], flat["idx"])
    assert np.allclose(hier["y"], flat["y"], rtol=1e-13, atol=1e-13)
    assert np.allclose(hier["importance_flat"], flat["importance"], atol=1e-13)
    assert np.allclose(hier["load2"], flat["load"], atol=1e-13)
    # b = 1, flat over a = 5 groups with k1 = 2
    a = 5
    W_g1, W_n1 = rng.normal(size=(d, a)), rng.normal(size=(d, a))
    eps1 = rng.normal(size=(T, a))
    W_in, W_out = rng.normal(size=(a, d, h)), rng.normal(size=(a, h, d))
    hier = O.hier_forward(x, W_g1, W_n1, eps1, np.zeros((a, d, 1)), np.zeros((a, d, 1)),
                          np.zeros((T, 2, 1)), W_in, W_out, 2, 1)
    flat = O.moe_forward(x, W_g1, W_n1, eps1, W_in, W_out, 2)
    assert np.array_equal(hier["idx"], flat["idx"])
    assert np.allclose(hier["y"], flat["y"], rtol=1e-13, atol=1e-13)
    assert np.allclose(hier["importance1"], flat["importance"], atol=1e-13)
    assert np.allclose(hier["load1"], flat["load"], atol=1e-13)
    # product gates
    a, b = 3, 4
    hier = O.hier_forward(x, rng.normal(size=(d, a)), rng.normal(size=(d, a)), rng.normal(size=(T, a)),
                          rng.normal(size=(a, d, b)), rng.normal(size=(a, d, b)),
                          rng.normal(size=(T, 2, b)), rng.normal(size=(a * b, d, h)),
                          rng.normal(size=(a * b, h, d)), 2, 2)
    assert np.allclose(hier["gates"].sum(axis=1), 1.0, atol=1e-14)
    assert abs(hier["importance_flat"].sum() - T) < 1e-12
    for t in range(T):
        assert len(set(hier["idx"][t])) == 4
        assert set(hier["idx"][t] // b) == set(hier["idx1"][t])


def pin_expert_size(O):
    g = golden("expert_size.txt")
    d, h = int(g["d"]), int(g["h"])
    assert d * h * 2 == int(g["weights"])
    assert round(g["k"] * d * h * 2 / 1e6, 1) == g["macs_per_input_millions"]


def _softplus_bf(z):
    return z + math.log1p(math.exp(-z)) if z > 0 else math.log1p(math.exp(z))


def _phi_bf(z):
    return 0.5 * math.erfc(-z / math.sqrt(2.0))


def _gate_row_bf(xrow, Wg, Wn, erow, k):
    """One token's noisy top-k gate by plain loops over the definition (eq (4),
    KeepTopK and softmax, eq (9) with kth_excluding as the k-th largest logit
    among the other experts).  Returns (kept ids, gates, P per expert)."""
    d, n = Wg.shape
    clean = [sum(xrow[j] * Wg[j, i] for j in range(d)) for i in range(n)]
    std = [_softplus_bf(sum(xrow[j] * Wn[j, i] for j in range(d))) for i in range(n)]
    H = [clean[i] + erow[i] * std[i] for i in range(n)]
    kept = sorted(range(n), key=lambda i: (-H[i], i))[:k]
    m = max(H[i] for i in kept)
    e = [math.exp(H[i] - m) for i in kept]
    gates = [v / sum(e) for v in e]
    P = []
    for i in range(n):
        others = sorted((H[j] for j in range(n) if j != i), reverse=True)
        thr = others[k - 1] if k - 1 < len(others) else -math.inf
        P.append(_phi_bf((clean[i] - thr) / std[i]))
    return kept, gates, P


def _ffn_bf(xrow, Wi, Wo):
    d, h = Wi.shape
    hid = [max(0.0, sum(xrow[a] * Wi[a, c] for a in range(d))) for c in range(h)]
    return np.array([sum(hid[q] * Wo[q, c] for q in range(h)) for c in range(Wo.shape[1])])


def pin_gating_sums_chunks(O):
    """``gating_sums`` (the batch taken in token chunks) gives, for chunk sizes
    that do and do not divide T (1, 5, 16, T - 1, T, more than T), the per-row
    outputs of the one-pass gate and the batch sums of eq (6) (Importance, the
    kept gates added per expert) and of eq (10) (Load, P added over the batch),
    the sums formed here by plain loops."""
    rng = np.random.default_rng(71)
    T, d, n, k = 37, 5, 7, 2
    x = rng.normal(size=(T, d))
    W_g, W_noise = rng.normal(size=(d, n)), rng.normal(size=(d, n))
    eps = rng.normal(size=(T, n))
    b_g = rng.normal(size=n)
    full = O.gating(x, W_g, W_noise, eps, k, 0.01, b_g)
    imp = [0.0] * n
    load = [0.0] * n
    for t in range(T):
        for j in range(k):
            imp[full["idx"][t, j]] += full["gates"][t, j]
        for i in range(n):
            load[i] += full["P"][t, i]
    for chunk in (1, 5, 16, T - 1, T, 100):
        s = O.gating_sums(x, W_g, W_noise, eps, k, 0.01, b_g, chunk=chunk)
        assert np.array_equal(s["idx"], full["idx"]), chunk
        assert np.allclose(s["gates"], full["gates"], rtol=1e-13, atol=0), chunk
        assert np.allclose(s["gap"], full["gap"], rtol=1e-12, atol=1e-13), chunk
        assert np.array_equal(s["tie"], full["tie"]), chunk
        assert np.allclose(s["importance"], imp, rtol=1e-12, atol=0), chunk
        assert np.allclose(s["load"], load, rtol=1e-12, atol=0), chunk
    assert abs(sum(imp) - T) < 1e-12


def pin_forward_rows_subset(O):
    """``moe_forward_rows`` on an unsorted, non-contiguous row set with a repeat
    gives those rows of the whole layer (eq (1)), and each output row equals the
    gate-weighted sum of its kept experts' outputs formed by plain loops."""
    rng = np.random.default_rng(72)
    T, d, n, h, k = 23, 4, 6, 5, 2
    x = rng.normal(size=(T, d))
    W_g, W_noise = rng.normal(size=(d, n)), rng.normal(size=(d, n))
    eps = rng.normal(size=(T, n))
    W_in, W_out = rng.normal(size=(n, d, h)), rng.normal(size=(n, h, d))
    rows = np.array([17, 3, 9, 22, 0, 3])
    full = O.moe_forward(x, W_g, W_noise, eps, W_in, W_out, k)
    got = O.moe_forward_rows(x, W_g, W_noise, eps, W_in, W_out, k, rows)
    assert np.array_equal(got["idx"], full["idx"][rows])
    assert np.allclose(got["gates"], full["gates"][rows], rtol=1e-13, atol=0)
    assert np.allclose(got["y"], full["y"][rows], rtol=1e-12, atol=1e-12)
    for r, t in enumerate(rows):
        kept, gates, _ = _gate_row_bf(x[t], W_g, W_noise, eps[t], k)
        assert list(got["idx"][r]) == kept
        want = sum(g * _ffn_bf(x[t], W_in[e], W_out[e]) for e, g in zip(kept, gates))
        assert np.allclose(got["y"][r], want, rtol=1e-12, atol=1e-12)


def pin_hierarchical_brute_force(O):
    """The two-level layer at a = 3 groups, b = 4 experts, k1 = k2 = 2, every token
    worked by plain loops: the primary gate over groups, the secondary gate of each
    kept group with that slot's noise, flat ids g b + j with product gates, the
    output, and the reported vectors (primary Importance and Load over groups, the
    flat Importance of the product gates, and the secondary Load of group g summed
    over the rows routed to g)."""
    rng = np.random.default_rng(73)
    T, d, h, a, b, k1, k2 = 9, 3, 4, 3, 4, 2, 2
    x = rng.normal(size=(T, d))
    W_g1, W_n1 = rng.normal(size=(d, a)), rng.normal(size=(d, a))
    eps1 = rng.normal(size=(T, a))
    W_g2, W_n2 = rng.normal(size=(a, d, b)), rng.normal(size=(a, d, b))
    eps2 = rng.normal(size=(T, k1, b))
    W_in, W_out = rng.normal(size=(a * b, d, h)), rng.normal(size=(a * b, h, d))
    got = O.hier_forward(x, W_g1, W_n1, eps1, W_g2, W_n2, eps2, W_in, W_out, k1, k2)
    imp1, load1 = np.zeros(a), np.zeros(a)
    impf, load2 = np.zeros(a * b), np.zeros(a * b)
    for t in range(T):
        kept1, g1, P1 = _gate_row_bf(x[t], W_g1, W_n1, eps1[t], k1)
        load1 += P1
        y = np.zeros(d)
        ids, gates = [], []
        for s, (gi, gg) in enumerate(zip(kept1, g1)):
            imp1[gi] += gg
            kept2, g2, P2 = _gate_row_bf(x[t], W_g2[gi], W_n2[gi], eps2[t, s], k2)
            load2[gi * b:(gi + 1) * b] += P2
            for j, gj in zip(kept2, g2):
                e = gi * b + j
                ids.append(e)
                gates.append(gg * gj)
                impf[e] += gg * gj
                y += gg * gj * _ffn_bf(x[t], W_in[e], W_out[e])
        assert list(got["idx"][t]) == ids, t
        assert np.allclose(got["gates"][t], gates, rtol=1e-12, atol=0)
        assert np.allclose(got["y"][t], y, rtol=1e-11, atol=1e-12)
    for key, want in (("importance1", imp1), ("load1", load1), ("importance_flat", impf),
                      ("load2", load2)):
        assert np.allclose(got[key], want, rtol=1e-12, atol=1e-14), key


def pin_kept_tie_break(O):
    """A kept set that another tie-break chose on a near tie: with logits 2,
    1 + 4e-6, 1, 0 and k = 2 the oracle keeps experts 0 and 1 and flags the row;
    keeping 0 and 2 instead is valid, its gates are the softmax over logits 2 and 1
    (e^2 / (e^2 + e), e / (e^2 + e)), and the load probabilities are unchanged
    (kth_excluding depends on the logits only).  The oracle's own set reproduces
    the plain gate; a set with an expert far below the k-th logit, a repeated
    expert or a kept order against the logits is refused.  The layer output of
    the chosen set is the plain-loop sum over experts 0 and 2."""
    logits = [2.0, 1.0 + 4e-6, 1.0, 0.0]
    x, W_g, W_noise, eps = _x_is_logits(logits)
    own = O.gating(x, W_g, W_noise, eps, 2)
    assert own["idx"].tolist() == [[0, 1]] and bool(own["tie"][0])
    alt = O.gating(x, W_g, W_noise, eps, 2, kept=[[0, 2]])
    assert alt["idx"].tolist() == [[0, 2]]
    e2, e1 = math.exp(2.0), math.exp(1.0)
    assert np.allclose(alt["gates"][0], [e2 / (e2 + e1), e1 / (e2 + e1)], rtol=1e-15, atol=0)
    assert np.array_equal(alt["P"], own["P"])
    same = O.gating(x, W_g, W_noise, eps, 2, kept=own["idx"])
    assert np.array_equal(same["gates"], own["gates"])
    for bad in ([[0, 3]], [[0, 0]], [[2, 0]]):
        try:
            O.gating(x, W_g, W_noise, eps, 2, kept=bad)
        except ValueError:
            continue
        raise AssertionError(f"kept set {bad} accepted")
    # an inner near tie: the kept order may swap
    x2, W_g2, W_n2, eps2 = _x_is_logits([1.0 + 3e-6, 1.0, 0.5, 0.0])
    sw = O.gating(x2, W_g2, W_n2, eps2, 2, kept=[[1, 0]])
    assert abs(sw["gates"][0, 0] - 1.0 / (1.0 + math.exp(3e-6))) < 1e-15
    # the layer with the chosen set
    rng = np.random.default_rng(74)
    h = 3
    W_in, W_out = rng.normal(size=(4, 1, h)), rng.normal(size=(4, h, 1))
    f = O.moe_forward(x, W_g, W_noise, eps, W_in, W_out, 2, kept=[[0, 2]])
    want = sum(g * _ffn_bf(x[0], W_in[ei], W_out[ei]) for ei, g in zip((0, 2), alt["gates"][0]))
    assert np.allclose(f["y"][0], want, rtol=1e-13, atol=1e-15)
    assert np.allclose(f["importance"], [alt["gates"][0, 0], 0.0, alt["gates"][0, 1], 0.0],
                       rtol=1e-15, atol=0)


def pin_batchwise_threshold(O):
    """The batchwise gate's inference mode (a learned per-expert threshold replaces
    the batch-wise top-m choice, as "What the paper measured" describes the Appendix F
    gate): a case worked by hand; a logit equal to its threshold is not taken; a
    threshold just under each expert's m-th largest logit and above its (m+1)-th
    reproduces the training-time choice on that batch; thresholds of -inf give every
    expert every token (the flat layer with k = n) and +inf gives y = 0."""
    d = 2
    x = np.eye(d)[[0, 0, 0, 0]]
    H = np.array([[3.0, 0.0], [2.0, 1.0], [1.0, 2.0], [0.0, 3.0]])
    W_g, W_n = np.zeros((d, 2)), np.full((d, 2), 50.0)       # std = 50, clean = 0
    eps = H / 50.0
    g = O.batchwise_threshold_gating(x, W_g, W_n, eps, [1.5, 1.0])
    assert [v.tolist() for v in g["sel"]] == [[0, 1], [2, 3]]  # H = 1.0 at (1, 1) not taken
    assert g["counts"].tolist() == [2, 2]
    assert np.allclose(g["G"], [[1, 0], [1, 0], [0, 1], [0, 1]], atol=1e-12)
    g = O.batchwise_threshold_gating(x, W_g, W_n, eps, [1.5, 0.5])
    assert [v.tolist() for v in g["sel"]] == [[0, 1], [1, 2, 3]]
    e = 1.0 / (1.0 + math.exp(-1.0))                         # token 1: logits 2 and 1
    assert np.allclose(g["G"][1], [e, 1.0 - e], atol=1e-9)

    rng = np.random.default_rng(62)
    T, dd, n, h, k = 24, 3, 4, 5, 2
    x = rng.normal(size=(T, dd))
    W_g, W_n = rng.normal(size=(dd, n)), rng.normal(size=(dd, n))
    eps = rng.normal(size=(T, n))
    W_in, W_out = rng.normal(size=(n, dd, h)), rng.normal(size=(n, h, dd))
    tr = O.moe_forward_batchwise(x, W_g, W_n, eps, W_in, W_out, k)
    m = tr["m"]
    Hs = -np.sort(-tr["H"], axis=0)
    thr = 0.5 * (Hs[m - 1] + Hs[m])                           # between the m-th and (m+1)-th
    inf = O.moe_forward_batchwise(x, W_g, W_n, eps, W_in, W_out, k, threshold=thr)
    assert [v.tolist() for v in inf["sel"]] == tr["sel"].tolist()
    assert np.allclose(inf["y"], tr["y"], rtol=1e-12, atol=1e-12)
    assert np.allclose(inf["losses"], tr["losses"], rtol=1e-12, atol=1e-15)
    dense = O.moe_forward(x, W_g, W_n, eps, W_in, W_out, n)
    allk = O.moe_forward_batchwise(x, W_g, W_n, eps, W_in, W_out, k, threshold=[-np.inf] * n)
    assert np.allclose(allk["y"], dense["y"], rtol=1e-12, atol=1e-12)
    assert allk["counts"].tolist() == [T] * n
    none = O.moe_forward_batchwise(x, W_g, W_n, eps, W_in, W_out, k, threshold=[np.inf] * n)
    assert not none["y"].any() and not none["G"].any() and none["counts"].sum() == 0


def pin_draw_noise(O):
    """The layer's own noise draws ("Noisy top-k gating", eq (4): standard normal):
    for several seeds, 2^20 draws have mean 0 and variance 1 within 5 standard errors,
    no lag-1 correlation beyond 5 standard errors, a Kolmogorov-Smirnov distance to
    the standard normal CDF with p > 1e-4 (scipy.stats.kstest), and |eps| at most
    sqrt(2 ln 2^24) (the smallest u1 is 2^-24); the two normals of a Box-Muller pair are
    uncorrelated; draw i does not depend on how many are drawn (counter-based); equal
    seeds repeat and different seeds differ."""
    from scipy import stats
    N = 1 << 20
    for seed in (0, 1, 7, 2 ** 63 + 5):
        e = O.draw_noise(seed, N)
        assert e.shape == (N,) and np.isfinite(e).all()
        assert abs(e.mean()) * math.sqrt(N) < 5.0
        assert abs(e.var() - 1.0) / math.sqrt(2.0 / N) < 5.0
        assert abs(np.corrcoef(e[:-1], e[1:])[0, 1]) * math.sqrt(N) < 5.0
        assert stats.kstest(e, "norm").pvalue > 1e-4
        assert np.abs(e).max() <= math.sqrt(2.0 * 24.0 * math.log(2.0)) + 1e-12
    # the two normals of a pair are uncorrelated (a cos / sin pair, not a repeat)
    e = O.draw_noise(5, N)
    assert abs(np.corrcoef(e[0::2], e[1::2])[0, 1]) * math.sqrt(N // 2) < 5.0
    a = O.draw_noise(123, 1000)
    assert np.array_equal(a[:10], O.draw_noise(123, 10))
    assert np.array_equal(a[:7], O.draw_noise(123, 7))
    assert np.array_equal(a, O.draw_noise(123, 1000))
    assert not np.allclose(a, O.draw_noise(124, 1000))


ALL_PINS = [
    pin_worked_example_gates,
    pin_importance_cv2,
    pin_load_probability_example,
    pin_kth_excluding_brute_force,
    pin_topk_brute_force,
    pin_gate_invariants,
    pin_noisy_logits_closed_form,
    pin_load_monte_carlo,
    pin_zero_init,
    pin_expert_ffn_brute_force,
    pin_dense_equals_sparse,
    pin_dispatch_brute_force,
    pin_capacity,
    pin_switch_gate,
    pin_backward_finite_differences,
    pin_batchwise,
    pin_combine_gathered_matches_by_expert,
    pin_hierarchical_reductions,
    pin_expert_size,
    pin_gating_sums_chunks,
    pin_forward_rows_subset,
    pin_hierarchical_brute_force,
    pin_kept_tie_break,
    pin_batchwise_threshold,
    pin_draw_noise,
]
