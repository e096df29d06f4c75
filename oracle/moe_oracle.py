"""fp64 CPU oracle for the noisy top-k Mixture-of-Experts forward pass.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The library's CUDA path never calls it, and it shares no code with
that path: it is a plain, slow restatement of what the layer computes, used
to check the kernels.

Source: "Mixture of Experts: Outrageously Large Neural Networks"
(intuitivepapers.ai), the explainer of Shazeer et al. 2017.  Every display
equation on that page was lost in extraction; each function below states the
equation from the prose that surrounds it, and cites the section it follows.
Where the page is silent the reading taken is stated in the function's
docstring.

Everything is numpy float64.  Library primitives used as single steps: matrix
products (``@``), ``argsort(kind="stable")``, ``np.logaddexp`` (for
log(1 + e^z)) and ``scipy.special.ndtr`` (the standard normal CDF).  There is
no blocking or fusion beyond a loop over token chunks in ``gating_sums`` (the
rows of the batch are independent, so only the order of a float64 sum over
tokens changes).

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
values printed on the page, closed forms, brute force on tiny inputs, and
invariants; ``draw_noise`` (a generator the pages do not fix) against the
statistics of a standard normal and the uniformity of its two 24-bit parts.
"""
from __future__ import annotations

import numpy as np
from scipy.special import ndtr

__all__ = [
    "softplus",
    "normal_cdf",
    "noisy_logits",
    "draw_noise",
    "top_k_order",
    "keep_top_k_softmax",
    "check_kept",
    "kth_excluding",
    "load_probability",
    "capacity_keep",
    "gating",
    "switch_gating",
    "switch_balance_loss",
    "gating_sums",
    "cv_squared",
    "balance_losses",
    "dispatch",
    "expert_ffn",
    "combine_by_expert",
    "combine_gathered",
    "moe_forward",
    "moe_forward_rows",
    "hier_forward",
    "cv_squared_grad",
    "normal_pdf",
    "moe_backward",
    "moe_loss",
    "batchwise_gating",
    "batchwise_threshold_gating",
    "moe_forward_batchwise",
    "TIE_GAP",
]

# Gap below which the k-th and (k+1)-th noisy logits count as a near tie;
# the selected set of such a row is compared only for validity.
TIE_GAP = 1e-5


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def softplus(z):
    """Softplus(z) = log(1 + e^z), the positive map from (x W_noise)_i to the
    noise standard deviation ("Noisy top-k gating", eq (4)).  Evaluated as
    log(e^0 + e^z) with numpy's logaddexp."""
    return np.logaddexp(0.0, _f64(z))


def normal_cdf(z):
    """Phi, the standard normal cumulative distribution function used by the
    smooth load ("A differentiable count of examples", eq (9))."""
    return ndtr(_f64(z))


def noisy_logits(x, W_g, W_noise, eps, std_floor=0.0, b_g=None):
    """Noisy logits, eq (4) of "Noisy top-k gating".

    clean_i = (x . W_g)_i            (+ b_g[i], an optional per-expert logit bias)
    std_i   = Softplus((x . W_noise)_i) + std_floor
    H_i     = clean_i + eps_i * std_i

    eps is supplied by the caller (one standard normal draw per token and
    expert).  ``std_floor`` = 0 is the formula as written; 0.01 is the floor of
    the official implementation that the page mentions.  Reading: a bias is
    part of the clean logit (the per-expert score of "Mixture of Experts:
    Sparse Activation for Scaling Language Models" (mbrenndoerfer.com), which
    adds b_i to W_i h), so it also enters the load probability's numerator.
    Returns (clean, std, H), each [T, n] float64.
    """
    x = _f64(x)
    clean = x @ _f64(W_g)
    if b_g is not None:
        clean = clean + _f64(b_g)[None, :]
    std = softplus(x @ _f64(W_noise)) + float(std_floor)
    H = clean + _f64(eps) * std
    return clean, std, H


def draw_noise(seed, count):
    """The standard normal draws of "Noisy top-k gating", eq (4) (one per token and
    expert), as the layer draws them itself (its device-noise mode): element i of a
    counter-based generator for a 64-bit seed, in float64.

    Steps, from their published definitions: for pair j = i // 2, the 64-bit state
    seed + (j + 1) g with the golden-ratio increment g = 0x9E3779B97F4A7C15, mixed by the
    finaliser of SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014: xor-shift 30, multiply by 0xBF58476D1CE4E5B9, xor-shift 27,
    multiply by 0x94D049BB133111EB, xor-shift 31, all mod 2^64); two 24-bit uniforms
    from it, u1 = (top 24 bits + 1) / 2^24 in (0, 1] and u2 = (low 24 bits) / 2^24 in
    [0, 1); then Box and Muller's transform: element 2j is sqrt(-2 ln u1) cos(2 pi u2)
    and element 2j + 1 is sqrt(-2 ln u1) sin(2 pi u2).  Reading: the pages only say
    "standard normal"; any generator meets that, this one is chosen so that any element
    can be drawn on its own.  Returns float64 [count].
    """
    pairs = (count + 1) // 2
    j = np.arange(pairs, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed) + (j + np.uint64(1)) * np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    u1 = ((z >> np.uint64(40)) + np.uint64(1)).astype(np.float64) / 2.0 ** 24
    u2 = (z & np.uint64(0xFFFFFF)).astype(np.float64) / 2.0 ** 24
    r = np.sqrt(-2.0 * np.log(u1))
    out = np.empty(2 * pairs)
    out[0::2] = r * np.cos(2.0 * np.pi * u2)
    out[1::2] = r * np.sin(2.0 * np.pi * u2)
    return out[:count]


def top_k_order(H, k):
    """Order of experts per row by noisy logit, largest first.

    Reading (the page is silent on ties): equal logits are ranked by the
    lower expert index first, which a stable sort of -H gives.  Returns the
    full order [T, n]; its first k columns are KeepTopK's survivors
    ("Noisy top-k gating", eq (3)/(5)) and column k is the extra (k+1)-th
    logit the forward pass takes for the load threshold.
    """
    H = _f64(H)
    return np.argsort(-H, axis=1, kind="stable")


def keep_top_k_softmax(H, idx):
    """KeepTopK then softmax ("Noisy top-k gating"): logits outside the kept
    set are -inf, so the softmax runs over the kept logits only and gives
    exactly 0 elsewhere.  ``idx`` [T, k] names the kept experts; returns their
    gate values [T, k] (each row sums to 1)."""
    Hk = np.take_along_axis(_f64(H), np.asarray(idx), axis=1)
    m = Hk.max(axis=1, keepdims=True)
    e = np.exp(Hk - m)
    return e / e.sum(axis=1, keepdims=True)


def kth_excluding(H, k, order=None):
    """kth_excluding(H, k, i) for every expert i ("A differentiable count of
    examples"): the k-th largest noisy logit among the experts other than i.

    By the official rule the page states: if i is in the top k it is the
    (k+1)-th largest overall, otherwise the k-th largest overall.
    Reading for k = n (no (k+1)-th logit exists): -inf, so an expert in the
    top n is kept with probability 1.
    Returns thr [T, n].
    """
    H = _f64(H)
    T, n = H.shape
    if order is None:
        order = top_k_order(H, k)
    rows = np.arange(T)
    kth = H[rows, order[:, k - 1]]
    k1th = H[rows, order[:, k]] if k < n else np.full(T, -np.inf)
    in_top = np.zeros((T, n), dtype=bool)
    in_top[rows[:, None], order[:, :k]] = True
    return np.where(in_top, k1th[:, None], kth[:, None])


def load_probability(clean, std, H, k, order=None):
    """P(x, i) = Phi((clean_i - kth_excluding(H, k, i)) / std_i), eqs (8)-(9)
    of "A differentiable count of examples": the probability that a fresh
    noise draw for expert i alone puts it in the top k."""
    thr = kth_excluding(H, k, order)
    return normal_cdf((_f64(clean) - thr) / _f64(std))


def check_kept(H, k, order, kept):
    """Validate a kept set chosen by another tie-break than ``top_k_order``'s.

    Where two noisy logits lie within TIE_GAP of each other either ranking is a
    correct top k (the page fixes no tie rule), so a kept set that differs from
    this oracle's is valid exactly when it holds k distinct experts and each of
    them has a logit no more than TIE_GAP below the oracle's k-th largest.  On
    rows without a near tie that forces the same set; its order may differ only
    where two kept logits are within TIE_GAP.  Raises ValueError otherwise.
    Returns ``kept`` as int64 [T, k].
    """
    T, n = H.shape
    kept = np.asarray(kept).astype(np.int64).reshape(T, k)
    if T == 0:
        return kept
    if kept.min() < 0 or kept.max() >= n:
        raise ValueError("kept expert id out of range")
    srt = np.sort(kept, axis=1)
    if k > 1 and (srt[:, 1:] == srt[:, :-1]).any():
        raise ValueError("a kept set repeats an expert")
    kth = H[np.arange(T), order[:, k - 1]]
    Hk = np.take_along_axis(H, kept, axis=1)
    low = np.nonzero(Hk.min(axis=1) < kth - TIE_GAP)[0]
    if low.size:
        raise ValueError(f"rows {low[:5]}: a kept expert lies below the k-th logit by more "
                         "than the tie gap")
    if k > 1 and (Hk[:, 1:] > Hk[:, :-1] + TIE_GAP).any():
        raise ValueError("kept experts out of logit order")
    return kept


def gating(x, W_g, W_noise, eps, k, std_floor=0.0, b_g=None, kept=None):
    """The whole noisy top-k gate for a batch ("Noisy top-k gating" and "A
    differentiable count of examples").

    ``kept`` [T, k] (optional): a kept set picked by another valid tie-break on
    near-tie rows (validated by ``check_kept``).  The gates are then the softmax
    over those experts' logits (eq (5) with that KeepTopK choice).  The load
    probability does not depend on it: kth_excluding(H, k, i) is the k-th
    largest logit among the experts other than i, a function of H alone.

    Returns a dict:
      idx [T,k] int64    kept experts, largest noisy logit first (or ``kept``)
      gates [T,k]        softmax over the kept logits
      clean, std, H, P   [T,n] float64
      gap [T]            H_(k) - H_(k+1) (inf when k = n)
      tie [T] bool       gap < TIE_GAP (a near tie at the k-th place)
    """
    clean, std, H = noisy_logits(x, W_g, W_noise, eps, std_floor, b_g)
    T, n = H.shape
    if not 1 <= k <= n:
        raise ValueError("k must be in [1, n]")
    order = top_k_order(H, k)
    idx = order[:, :k] if kept is None else check_kept(H, k, order, kept)
    gates = keep_top_k_softmax(H, idx)
    P = load_probability(clean, std, H, k, order)
    rows = np.arange(T)
    if k < n:
        gap = H[rows, order[:, k - 1]] - H[rows, order[:, k]]
    else:
        gap = np.full(T, np.inf)
    return dict(idx=idx, gates=gates, clean=clean, std=std, H=H, P=P, gap=gap,
                tie=gap < TIE_GAP, order=order)


def switch_gating(x, W_g, W_noise, eps, k, std_floor=0.0, b_g=None):
    """The Switch gate ("From LSTMs to Switch and Mixtral"): Switch Transformers
    run the softmax over all n logits first and multiply the chosen expert's
    output by its probability, a number below 1.

    Reading: the logits are this layer's noisy H (eq (4); eps = 0 is the
    noiseless gate), the kept experts are the k largest H as in ``gating``
    (k = 1 in Switch), and a kept expert's gate is its probability under the
    softmax over all n, not renormalised over the kept ones.
    Returns ``gating``'s dict with these gates and p [T, n], the probabilities.
    """
    g = gating(x, W_g, W_noise, eps, k, std_floor, b_g)
    H = g["H"]
    e = np.exp(H - H.max(axis=1, keepdims=True))
    p = e / e.sum(axis=1, keepdims=True)
    g.update(gates=np.take_along_axis(p, g["idx"], axis=1), p=p)
    return g


def switch_balance_loss(idx, p, n):
    """The single Switch balancing loss ("From LSTMs to Switch and Mixtral": a
    loss on the product of each expert's token fraction and mean gate
    probability): n * sum_i f_i P_i with f_i the fraction of routed rows sent
    to expert i and P_i the batch mean of expert i's probability.  Reading:
    the page gives no constant; the factor n (the one Switch Transformers use)
    makes perfectly uniform routing score exactly 1.
    Returns (loss, load [n] = routed rows per expert, importance [n] = summed p)."""
    idx = np.asarray(idx)
    T = idx.shape[0]
    load = np.bincount(idx.ravel(), minlength=n).astype(np.float64)
    importance = _f64(p).sum(axis=0)
    f = load / idx.size
    P = importance / T
    return n * float(np.sum(f * P)), load, importance


def gating_sums(x, W_g, W_noise, eps, k, std_floor=0.0, b_g=None, chunk=4096, kept=None):
    """Gating over a large batch in token chunks, keeping only per-row
    outputs and the batch sums the losses need (the [T, n] tensors of one
    chunk at a time).  Rows are independent, so this is ``gating`` with the
    float64 sums over tokens taken chunk by chunk.  ``kept`` as in ``gating``.

    Returns idx, gates, gap, tie ([T, ...]), importance [n], load [n].
    """
    T = x.shape[0]
    n = W_g.shape[1]
    idx = np.empty((T, k), dtype=np.int64)
    gates = np.empty((T, k))
    gap = np.empty(T)
    importance = np.zeros(n)
    load = np.zeros(n)
    for s in range(0, T, chunk):
        e = min(T, s + chunk)
        g = gating(x[s:e], W_g, W_noise, eps[s:e], k, std_floor, b_g,
                   None if kept is None else np.asarray(kept).reshape(T, k)[s:e])
        idx[s:e], gates[s:e], gap[s:e] = g["idx"], g["gates"], g["gap"]
        importance += importance_of(g["idx"], g["gates"], n)
        load += g["P"].sum(axis=0)
    return dict(idx=idx, gates=gates, gap=gap, tie=gap < TIE_GAP,
                importance=importance, load=load)


def importance_of(idx, gates, n):
    """Importance(X)_i = sum over the batch of G(x)_i, eq (6) of "Why experts
    collapse, and the balancing losses".  G(x) is zero outside the kept set,
    so only the kept (expert, gate) pairs contribute."""
    imp = np.zeros(n)
    np.add.at(imp, np.asarray(idx).ravel(), _f64(gates).ravel())
    return imp


def cv_squared(v):
    """CV(v)^2 = (population variance of v) / mean(v)^2, eq (7) of "Why
    experts collapse, and the balancing losses" (the worked example divides
    the squared deviations by the number of experts).  Reading (no epsilon on
    the page): a zero mean, or a single entry, gives 0."""
    v = _f64(v)
    if v.size <= 1:
        return 0.0
    mu = v.mean()
    if mu == 0.0:
        return 0.0
    return float(((v - mu) ** 2).mean() / (mu * mu))


def balance_losses(importance, load, w_importance=0.1, w_load=0.1):
    """L_importance = w_importance CV(Importance)^2 (eq (7)) and
    L_load = w_load CV(Load)^2 (eq (10)); Load_i is the batch sum of P(x, i).
    Weights 0.1 are the 1 Billion Word setting the page gives.
    Returns (cv2_importance, cv2_load, aux = weighted sum)."""
    ci = cv_squared(importance)
    cl = cv_squared(load)
    return ci, cl, w_importance * ci + w_load * cl


def capacity_keep(idx, n, capacity=0):
    """Which routed rows their expert processes under a fixed per-expert
    capacity ("From LSTMs to Switch and Mixtral": GShard gives each expert a
    fixed capacity, and inputs beyond it skip the expert and pass through the
    residual connection; the paper's own layer has no limit).

    Reading (the page gives no order): expert e takes its routed rows in
    ascending routed-row order r = t*k + j and keeps the first ``capacity`` of
    them; capacity 0 means no limit.  Returns a bool array shaped like idx.
    """
    idx = np.asarray(idx)
    keep = np.ones(idx.shape, dtype=bool)
    if capacity <= 0:
        return keep
    flat_keep = keep.reshape(-1)
    seen = np.zeros(n, dtype=np.int64)
    for r, e in enumerate(idx.reshape(-1)):
        flat_keep[r] = seen[e] < capacity
        seen[e] += 1
    return keep


def dispatch(idx, n, capacity=0):
    """Per-expert row lists for the forward pass: the inputs routed to expert
    i are the rows where G(x)_i is nonzero ("Implementation notes", the
    forward-pass listing's per-expert loop).

    Routed row r = t*k + j is token t's j-th kept slot.  Rows are grouped by
    expert, ascending expert id, and kept in ascending r inside a group (a
    stable counting sort).  With a capacity (``capacity_keep``) the rows an
    expert drops get no position.  Returns
      offsets [n+1]  start of expert e's rows (offsets[n] = rows kept, T*k
                     without a capacity)
      perm [kept]    perm[p] = r, the routed row stored at position p
      inv [T*k]      inv[r] = p, the position of routed row r (-1: dropped)
    """
    flat = np.asarray(idx).reshape(-1).astype(np.int64)
    keep = capacity_keep(idx, n, capacity).reshape(-1)
    counts = np.bincount(flat[keep], minlength=n)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    order = np.argsort(flat, kind="stable").astype(np.int64)
    perm = order[keep[order]]
    inv = np.full(flat.size, -1, dtype=np.int64)
    inv[perm] = np.arange(perm.size)
    return offsets, perm, inv


def expert_ffn(x_rows, W_in_e, W_out_e):
    """One expert, "How a mixture-of-experts layer works": an input layer,
    one hidden layer of ReLU units and an output layer, with separate weights
    and no biases: E(x) = ReLU(x W_in) W_out."""
    u = np.maximum(_f64(x_rows) @ _f64(W_in_e), 0.0)
    return u @ _f64(W_out_e)


def combine_by_expert(x, idx, gates, W_in, W_out, rows=None, keep=None):
    """y = sum_i G(x)_i E_i(x), eq (1) of "How a mixture-of-experts layer
    works", evaluated the way the forward-pass listing does: loop over
    experts, run each on the rows routed to it, and add gate * output into
    those rows.  Experts with no row are never run.

    ``rows`` restricts the computation to a subset of tokens (each output row
    depends only on its own token); y has one row per entry of ``rows``.
    ``keep`` (bool, shaped like idx; ``capacity_keep``) leaves out the routed
    rows an expert dropped.
    """
    x = _f64(x)
    idx = np.asarray(idx)
    gates = _f64(gates)
    n = W_in.shape[0]
    if rows is None:
        rows = np.arange(x.shape[0])
    rows = np.asarray(rows)
    sub_idx = idx[rows]
    sub_g = gates[rows]
    sub_keep = np.ones(sub_idx.shape, dtype=bool) if keep is None else np.asarray(keep)[rows]
    y = np.zeros((rows.size, W_out.shape[2]))
    for e in np.unique(sub_idx[sub_keep]):
        tt, jj = np.nonzero((sub_idx == e) & sub_keep)
        order = np.argsort(tt, kind="stable")
        tt, jj = tt[order], jj[order]
        y[tt] += sub_g[tt, jj][:, None] * expert_ffn(x[rows[tt]], W_in[e], W_out[e])
    return y


def combine_gathered(y_perm, inv, gates):
    """Eq (1) given every kept expert's output already computed: routed row
    r = t*k + j of token t sits at position inv[r] of the expert-grouped
    outputs y_perm, and y[t] = sum_j gates[t, j] * y_perm[inv[t*k + j]]."""
    gates = _f64(gates)
    T, k = gates.shape
    yp = _f64(y_perm)
    rows = np.asarray(inv).reshape(T, k)
    y = np.zeros((T, yp.shape[1]))
    for j in range(k):
        live = rows[:, j] >= 0          # -1: the expert dropped this row (capacity)
        y[live] += gates[live, j:j + 1] * yp[rows[live, j]]
    return y


def moe_forward(x, W_g, W_noise, eps, W_in, W_out, k, std_floor=0.0, b_g=None,
                w_importance=0.1, w_load=0.1, capacity=0, switch=False, kept=None):
    """The whole layer's forward pass in the order of the forward-pass listing
    ("Implementation notes"): gate, per-expert FFN on routed rows, combine,
    Importance and Load, and the two CV^2 losses.  ``capacity`` > 0 limits the
    rows each expert processes (``capacity_keep``); the gate and the losses do
    not depend on it.  ``switch``: the Switch gate and its single loss
    (``switch_gating``, ``switch_balance_loss``); losses = (L, 0, w_importance L).
    ``kept``: another valid tie-break's kept set (``gating``); not with ``switch``.
    Returns the gating dict extended with y, importance, load, losses, keep."""
    if switch:
        if kept is not None:
            raise ValueError("kept is not taken with the Switch gate")
        g = switch_gating(x, W_g, W_noise, eps, k, std_floor, b_g)
    else:
        g = gating(x, W_g, W_noise, eps, k, std_floor, b_g, kept)
    n = W_g.shape[1]
    keep = capacity_keep(g["idx"], n, capacity)
    y = combine_by_expert(x, g["idx"], g["gates"], W_in, W_out, keep=keep)
    if switch:
        L, load, importance = switch_balance_loss(g["idx"], g["p"], n)
        g.update(y=y, importance=importance, load=load, keep=keep,
                 losses=np.array([L, 0.0, w_importance * L]))
        return g
    importance = importance_of(g["idx"], g["gates"], n)
    load = g["P"].sum(axis=0)
    g.update(y=y, importance=importance, load=load, keep=keep,
             losses=balance_losses(importance, load, w_importance, w_load))
    return g


def moe_forward_rows(x, W_g, W_noise, eps, W_in, W_out, k, rows, std_floor=0.0, b_g=None,
                     kept=None):
    """Gate and layer output for a subset of tokens only (a sampled check at
    sizes where the whole batch is too slow); the batch losses are not
    formed.  ``kept`` [len(rows), k]: as in ``gating``, for those rows.
    Returns idx, gates, gap, tie, H for ``rows`` and y [len(rows), d]."""
    rows = np.asarray(rows)
    g = gating(x[rows], W_g, W_noise, eps[rows], k, std_floor, b_g, kept)
    y = combine_by_expert(x[rows], g["idx"], g["gates"], W_in, W_out)
    return dict(idx=g["idx"], gates=g["gates"], gap=g["gap"], tie=g["tie"], H=g["H"],
                clean=g["clean"], std=g["std"], y=y)


def hier_forward(x, W_g1, W_noise1, eps1, W_g2, W_noise2, eps2, W_in, W_out, k1, k2,
                 std_floor=0.0, rows=None, with_losses=True, with_y=True, kept=None):
    """Two-level MoE of "Hierarchical MoE": a primary noisy top-k1 gate over a
    groups, then, inside each kept group i, a secondary noisy top-k2 gate over
    that group's b experts; the final gate of expert (i, j) is the product
    G_primary(x)_i * G_i(x)_j, and the output is the sum of the products times
    the experts' outputs.

    Readings (the hierarchical formula is lost on the page):
      * the secondary gate of group i uses its own W_g2[i], W_noise2[i]; its
        noise is eps2[t, s, :] for the s-th kept group slot of token t;
      * expert (i, j) is flat expert i*b + j of W_in / W_out;
      * the page gives no hierarchical balancing loss.  The losses returned
        are the primary gate's Importance and Load over groups and the flat
        Importance over the a*b experts from the product gates
        (parity unpinned: only invariants are tested).
    ``kept`` [T, k1*k2] flat expert ids (of ``rows`` when given): kept sets that
    another valid tie-break chose, slot s*k2 + j holding expert j of the s-th kept
    group; each gate validates its part as ``gating`` does (so they may differ
    from this oracle's only on near-tie rows), and the rows then go to the groups
    it names.
    Returns idx [T, k1*k2] (flat expert ids, slot s*k2 + j), gates [T, k1*k2],
    y (None when ``with_y`` is false: gating and batch sums only), and the loss
    vectors.
    """
    x = _f64(x)
    if rows is not None:
        rows = np.asarray(rows)
        x, eps1, eps2 = x[rows], _f64(eps1)[rows], _f64(eps2)[rows]
    T = x.shape[0]
    a = W_g1.shape[1]
    b = W_g2.shape[2]
    kept1 = kept2 = None
    if kept is not None:
        kept = np.asarray(kept).astype(np.int64).reshape(T, k1, k2)
        kept1 = kept[:, :, 0] // b
        if (kept // b != kept1[:, :, None]).any():
            raise ValueError("a kept group slot mixes experts of two groups")
        kept2 = kept % b
    g1 = gating(x, W_g1, W_noise1, eps1, k1, std_floor, kept=kept1)
    idx = np.empty((T, k1 * k2), dtype=np.int64)
    gates = np.empty((T, k1 * k2))
    gap2 = np.empty((T, k1))
    load2 = np.zeros(a * b)
    for s in range(k1):
        grp = g1["idx"][:, s]
        for gi in np.unique(grp):
            tt = np.nonzero(grp == gi)[0]
            g2 = gating(x[tt], W_g2[gi], W_noise2[gi], _f64(eps2)[tt, s, :], k2, std_floor,
                        kept=None if kept2 is None else kept2[tt, s, :])
            idx[tt, s * k2:(s + 1) * k2] = gi * b + g2["idx"]
            gates[tt, s * k2:(s + 1) * k2] = g1["gates"][tt, s][:, None] * g2["gates"]
            gap2[tt, s] = g2["gap"]
            load2[gi * b:(gi + 1) * b] += g2["P"].sum(axis=0)
    y = combine_by_expert(x, idx, gates, W_in, W_out) if with_y else None
    out = dict(idx=idx, gates=gates, y=y, idx1=g1["idx"], gates1=g1["gates"],
               tie1=g1["tie"], tie2=gap2 < TIE_GAP, gap1=g1["gap"], gap2=gap2)
    if with_losses:
        out.update(importance1=importance_of(g1["idx"], g1["gates"], a),
                   load1=g1["P"].sum(axis=0),
                   importance_flat=importance_of(idx, gates, a * b),
                   load2=load2)
    return out


# ---- backward ------------------------------------------------------------------------
#
# "Implementation notes" of the intuitivepapers.ai page lists what receives gradient:
# each expert only from the rows routed to it, scaled by their gate values; W_g from the
# task loss through the softmax over the kept logits, from the importance loss by the
# same path, and from the load loss through the numerator of eq (9), also for experts
# that were not kept; W_noise through the noise term inside the kept logits and through
# the denominator of eq (9); the selection itself passes no gradient.  The functions
# below take the exact derivative of the forward pass as defined above for the loss
#   L = sum(dy * y) + w_importance CV(Importance)^2 + w_load CV(Load)^2,
# with the kept set (and the order that picks the load thresholds) held fixed.
# Reading: the threshold kth_excluding(H, k, i) is the noisy logit H_m of the expert m
# that sits at the k-th or (k+1)-th place, so its gradient reaches clean_m and std_m of
# that expert (the derivative of eq (9) as written; the page's summary is silent on the
# (k+1)-th logit's noise term).  ReLU'(0) = 0.


def cv_squared_grad(v):
    """d CV(v)^2 / d v_i with CV^2 = population variance / mean^2 (eq (7)):
    (2 / (n mean^2)) (v_i - mean - var / mean); 0 where CV^2 is defined as 0."""
    v = _f64(v)
    n = v.size
    mu = v.mean()
    if n <= 1 or mu == 0.0:
        return np.zeros(n)
    var = ((v - mu) ** 2).mean()
    return (2.0 / (n * mu * mu)) * (v - mu - var / mu)


def normal_pdf(z):
    """phi(z) = exp(-z^2 / 2) / sqrt(2 pi), the derivative of Phi (eq (9))."""
    z = _f64(z)
    return np.exp(-0.5 * z * z) / np.sqrt(2.0 * np.pi)


def moe_backward(x, W_g, W_noise, eps, W_in, W_out, k, dy, std_floor=0.0, b_g=None,
                 w_importance=0.1, w_load=0.1):
    """Gradients of L (see above) with respect to x, W_g, W_noise, b_g, W_in, W_out.

    Steps, each the chain rule through one forward step:
      dG_tj   = <dy_t, E_e(x_t)> + w_imp dCV^2(I)/dI_e          (e = idx[t, j])
      dH_t,e += G_tj (dG_tj - sum_l G_tl dG_tl)                 (softmax over the kept)
      for every (t, i), z = (clean - thr) / std, a = w_load dCV^2(L)/dL_i phi(z) / std:
        dclean_ti += a,  dstd_ti -= a z,  dH_t,m(t,i) -= a      (eq (9); m = threshold expert)
      dclean += dH,  dstd += eps dH,  dnz = dstd sigmoid(nz)    (eq (4))
      dW_g = x^T dclean, db_g = sum_t dclean, dW_noise = x^T dnz, dx = dclean W_g^T + dnz W_noise^T
      per routed (t, j): dE = G_tj dy_t, u = x_t W_in[e], du = (dE W_out[e]^T) [u > 0],
        dW_out[e] += ReLU(u)^T dE, dW_in[e] += x_t^T du, dx_t += du W_in[e]^T
    Returns a dict dx, dW_g, dW_noise, db_g, dW_in, dW_out (float64).
    """
    x = _f64(x)
    dy = _f64(dy)
    W_g, W_noise, W_in, W_out = _f64(W_g), _f64(W_noise), _f64(W_in), _f64(W_out)
    T, d = x.shape
    n = W_g.shape[1]
    g = gating(x, W_g, W_noise, eps, k, std_floor, b_g)
    idx, G, H, clean, std, order = g["idx"], g["gates"], g["H"], g["clean"], g["std"], g["order"]
    importance = importance_of(idx, G, n)
    load = g["P"].sum(axis=0)
    gI = w_importance * cv_squared_grad(importance)
    gL = w_load * cv_squared_grad(load)

    dx = np.zeros((T, d))
    dW_in = np.zeros_like(W_in)
    dW_out = np.zeros_like(W_out)
    dG = np.zeros((T, k))
    for e in np.unique(idx):                    # each expert on the rows routed to it
        tt, jj = np.nonzero(idx == e)
        u = x[tt] @ W_in[e]
        a = np.maximum(u, 0.0)
        E = a @ W_out[e]
        dG[tt, jj] = (dy[tt] * E).sum(axis=1) + gI[e]
        dE = G[tt, jj][:, None] * dy[tt]
        du = (dE @ W_out[e].T) * (u > 0.0)
        dW_out[e] += a.T @ dE
        dW_in[e] += x[tt].T @ du
        np.add.at(dx, tt, du @ W_in[e].T)

    dH = np.zeros((T, n))
    rows = np.arange(T)
    s = (G * dG).sum(axis=1, keepdims=True)
    np.add.at(dH, (rows[:, None].repeat(k, 1), idx), G * (dG - s))

    thr = kth_excluding(H, k, order)
    finite = np.isfinite(thr)                        # k = n: P = 1, no gradient
    z = np.where(finite, (clean - np.where(finite, thr, 0.0)) / std, 0.0)
    a = np.where(finite, gL[None, :] * normal_pdf(z) / std, 0.0)
    dclean = a.copy()
    dstd = -a * z
    in_top = np.zeros((T, n), dtype=bool)
    in_top[rows[:, None], order[:, :k]] = True
    m_kept = order[:, k] if k < n else order[:, k - 1]   # threshold expert of a kept i
    m_out = order[:, k - 1]                                # ... of an expert not kept
    to_kept = np.where(in_top, a, 0.0).sum(axis=1)
    to_out = np.where(~in_top, a, 0.0).sum(axis=1)
    if k < n:
        np.add.at(dH, (rows, m_kept), -to_kept)
    np.add.at(dH, (rows, m_out), -to_out)

    dclean += dH
    dstd += _f64(eps) * dH
    nz = x @ W_noise
    dnz = dstd / (1.0 + np.exp(-nz))
    dW_g = x.T @ dclean
    dW_noise = x.T @ dnz
    db_g = dclean.sum(axis=0)
    dx += dclean @ W_g.T + dnz @ W_noise.T
    return dict(dx=dx, dW_g=dW_g, dW_noise=dW_noise, db_g=db_g, dW_in=dW_in, dW_out=dW_out)


def moe_loss(x, W_g, W_noise, eps, W_in, W_out, k, dy, std_floor=0.0, b_g=None,
             w_importance=0.1, w_load=0.1):
    """The scalar L = sum(dy * y) + w_importance CV(I)^2 + w_load CV(L)^2 whose
    gradient ``moe_backward`` returns (for finite-difference checks)."""
    f = moe_forward(x, W_g, W_noise, eps, W_in, W_out, k, std_floor, b_g, w_importance, w_load)
    return float((_f64(dy) * f["y"]).sum()) + float(f["losses"][2])


# ---- batchwise top-m gate -------------------------------------------------------------
#
# The single-pair translation models of the intuitivepapers.ai page ("What the paper
# measured", the Appendix F gate) use a different gate: during training each expert takes
# exactly the top m = k |X| / n inputs of the batch, so every expert gets the same batch
# size.  Readings (the page gives no more): the score is the noisy logit H of eq (4);
# m = floor(k T / n); an expert ranks the tokens by H, larger first, equal H -> lower
# token index; a token's gate over the experts that took it is the softmax of their H
# (the KeepTopK softmax with the batchwise choice of experts), a token no expert took
# gets y = 0; the balancing losses report CV^2 of the Importance (the gates summed per
# expert) and of the exact counts, which are all m (so 0).
#
# At inference the page says a learned per-expert threshold replaces the batch-wise
# choice.  Readings: expert i takes token t when H_ti > threshold_i (strictly), so the
# counts vary; the gates and the output are formed as in training (softmax over the
# experts that took the token, y = 0 for a token none took); the losses report CV^2 of
# the Importance and of the counts, and w_importance CV^2(I) + w_load CV^2(counts).


def _batchwise_gates(H, taken):
    """Gates of the batchwise gate: for each token the softmax of H over the experts
    that took it; 0 elsewhere and for a token no expert took."""
    Hm = np.where(taken, H, -np.inf)
    mx = Hm.max(axis=1, keepdims=True)
    e = np.where(taken, np.exp(Hm - np.where(np.isfinite(mx), mx, 0.0)), 0.0)
    s = e.sum(axis=1, keepdims=True)
    return np.where(s > 0, e / np.where(s > 0, s, 1.0), 0.0)


def batchwise_threshold_gating(x, W_g, W_noise, eps, threshold, std_floor=0.0, b_g=None):
    """Inference mode of the batchwise gate: expert i takes token t when
    H_ti > threshold_i.  Returns a dict:
      taken [T, n] bool, G [T, n] (as ``batchwise_gating``), H [T, n],
      sel: list of n ascending int64 arrays (the tokens each expert took),
      counts [n] int64."""
    clean, std, H = noisy_logits(x, W_g, W_noise, eps, std_floor, b_g)
    thr = _f64(threshold).reshape(1, -1)
    if thr.shape[1] != H.shape[1]:
        raise ValueError("one threshold per expert")
    taken = H > thr
    sel = [np.nonzero(taken[:, i])[0].astype(np.int64) for i in range(H.shape[1])]
    return dict(taken=taken, G=_batchwise_gates(H, taken), H=H, sel=sel,
                counts=taken.sum(axis=0).astype(np.int64))


def batchwise_gating(x, W_g, W_noise, eps, k, std_floor=0.0, b_g=None, sel=None):
    """The batchwise top-m gate.  ``sel`` [n, m] (optional): token sets that another
    tie-break chose; accepted only where an expert's set differs from this oracle's on
    a near tie (every token taken has a logit within TIE_GAP max(1, |H_(m)|) of the
    expert's m-th largest), ascending and distinct; the gates and output then follow
    it.  Returns a dict:
      m                   rows per expert
      sel [n, m] int64    the tokens each expert takes, ascending token order
      taken [T, n] bool   token t taken by expert i
      G [T, n]            gate of (t, i), 0 where not taken
      H [T, n]            noisy logits;  mgap [n]  H_(m) - H_(m+1) of each expert's column
    """
    clean, std, H = noisy_logits(x, W_g, W_noise, eps, std_floor, b_g)
    T, n = H.shape
    m = (k * T) // n
    if not 1 <= m <= T:
        raise ValueError("k T / n must be in [1, T]")
    own = np.empty((n, m), dtype=np.int64)
    mth = np.empty(n)
    mgap = np.full(n, np.inf)
    for i in range(n):
        order = np.argsort(-H[:, i], kind="stable")
        own[i] = np.sort(order[:m])
        mth[i] = H[order[m - 1], i]
        if m < T:
            mgap[i] = H[order[m - 1], i] - H[order[m], i]
    if sel is not None:
        given = np.asarray(sel).astype(np.int64).reshape(n, m)
        for i in range(n):
            if np.array_equal(given[i], own[i]):
                continue
            tol = TIE_GAP * max(1.0, abs(mth[i]))
            if (given[i].min() < 0 or given[i].max() >= T or np.any(np.diff(given[i]) <= 0)
                    or H[given[i], i].min() < mth[i] - tol):
                raise ValueError(f"expert {i}: the given token set is not a valid top m")
        own = given
    taken = np.zeros((T, n), dtype=bool)
    for i in range(n):
        taken[own[i], i] = True
    return dict(m=m, sel=own, taken=taken, G=_batchwise_gates(H, taken), H=H, mgap=mgap)


def moe_forward_batchwise(x, W_g, W_noise, eps, W_in, W_out, k, std_floor=0.0, b_g=None,
                          w_importance=0.1, w_load=0.1, threshold=None, sel=None):
    """The layer with the batchwise top-m gate: y_t = sum over the experts i that took
    t of G_ti E_i(x_t).  ``threshold`` [n]: the inference mode (expert i takes the
    tokens with H_ti > threshold_i; k is then unused).  ``sel``: another valid
    tie-break's token sets in training (``batchwise_gating``).  Returns the gating dict with y,
    importance, load (the counts) and losses = (CV^2(importance), CV^2(load),
    w_importance CV^2(importance) + w_load CV^2(load)); in training CV^2(load) = 0."""
    if threshold is None:
        g = batchwise_gating(x, W_g, W_noise, eps, k, std_floor, b_g, sel)
    else:
        g = batchwise_threshold_gating(x, W_g, W_noise, eps, threshold, std_floor, b_g)
    x = _f64(x)
    T = x.shape[0]
    n = len(g["sel"])
    y = np.zeros((T, W_out.shape[2]))
    for i in range(n):
        rows = g["sel"][i]
        if len(rows):
            y[rows] += g["G"][rows, i][:, None] * expert_ffn(x[rows], W_in[i], W_out[i])
    importance = g["G"].sum(axis=0)
    load = g["taken"].sum(axis=0).astype(np.float64)
    ci, cl = cv_squared(importance), cv_squared(load)
    g.update(y=y, importance=importance, load=load,
             losses=np.array([ci, cl, w_importance * ci + w_load * cl]))
    return g
