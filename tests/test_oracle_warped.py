"""Pins of the oracle's top-k / top-p verification ("Speculative decoding."
lesson, "Why the output is exactly p": top-k and top-p are applied to p
before the rule; "Speculative Decoding: Draft, Verify, Accept", "The
rejection-sampling correctness argument": the rule reproduces whatever p it
is given).  The readings of top-k and top-p are ours (the pages name them
only): top-k keeps the K largest logits, lower index first on ties; top-p
keeps the shortest prefix of those, in the same order, whose renormalised
mass reaches top_p."""
import math

import numpy as np

import oracle
from helpers import first_token_tv
from speculative_decoding_verification_57_gb300 import workloads as W


def warped_p(logits_row, T, K, top_p):
    """p' by the definition, with numpy's sort (ties: lower index first)."""
    l = np.asarray(logits_row, np.float64)
    order = np.lexsort((np.arange(len(l)), -l))[:K]
    e = np.exp((l[order] - l[order[0]]) / T)
    n = len(order)
    if top_p < 1.0:
        c = np.cumsum(e) / e.sum()
        n = int(np.searchsorted(c, np.float64(np.float32(top_p)) - 0.0, side="left")) + 1
        n = min(n, len(order))
    pp = np.zeros(len(l))
    pp[order[:n]] = e[:n] / e[:n].sum()
    return pp


def test_no_filter_is_the_plain_rule():
    """K >= V and top_p = 1 give every output of the unwarped oracle."""
    w = W.make_random(name="nofilter", B=300, k=4, V=300, dtype="bf16", seed=21, logit_sigma=2.5, draft_sigma=1.0,
                      temperature=0.9, spike=4.0, spike_mode="position", greedy_rows=20)
    a = oracle.verify_warped(w.logits, w.q, w.x, w.u, w.T, np.full(w.B, 300), np.ones(w.B, np.float32))
    b = oracle.verify(w.logits, w.q, w.x, w.u, w.T)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_top1_is_greedy():
    """top_k = 1 makes p' the point mass at the argmax: the greedy outcome."""
    w = W.make_random(name="top1", B=400, k=5, V=64, dtype="f32", seed=22, logit_sigma=1.5, draft_sigma=0.5,
                      temperature=1.0)
    a = oracle.verify_warped(w.logits, w.q, w.x, w.u, w.T, np.ones(w.B), np.ones(w.B, np.float32))
    g = oracle.verify(w.logits, None, w.x, None, None)
    np.testing.assert_array_equal(a["num_accepted"], g["num_accepted"])
    np.testing.assert_array_equal(a["out_tokens"], g["out_tokens"])


def test_first_token_law_is_the_warped_p():
    """200k rounds on a 12-token alphabet: the first emitted token follows p'
    (top_k = 7, top_p = 0.8), not p; acceptance of the draft is
    sum min(p', q)."""
    rng = np.random.default_rng(23)
    V, B = 12, 200_000
    p = rng.dirichlet(np.ones(V))
    q = rng.dirichlet(np.ones(V))
    w = W.make_from_distributions(p, q, B=B, k=2, seed=24)
    K, tp = 7, 0.8
    r = oracle.verify_warped(w.logits, w.q, w.x, w.u, w.T, np.full(B, K), np.full(B, tp, np.float32))
    # every row has its own logits shift but the same law
    pp = warped_p(w.logits[0, 0].astype(np.float64), 1.0, K, tp)
    assert abs(pp.sum() - 1) < 1e-12 and np.count_nonzero(pp) <= K
    tv, _ = first_token_tv(r["out_tokens"][:, 0], pp)
    assert tv < 0.01
    alpha = np.minimum(pp, q).sum()
    keep = (r["num_accepted"] >= 1).mean()
    assert abs(keep - alpha) < 4 * math.sqrt(alpha * (1 - alpha) / B)
    assert np.all(pp[r["out_tokens"][:, 0]] > 0)


def test_nucleus_boundaries():
    """top_p picks the shortest prefix reaching the mass; ties in logits keep
    the lower index first."""
    T = np.array([1.0], np.float32)
    L = np.log(np.array([[[0.1, 0.4, 0.1, 0.3, 0.1], [0.1, 0.4, 0.1, 0.3, 0.1]]])).astype(np.float32)
    x = np.array([[2]], np.int32)
    q = np.full((1, 1, 5), 0.2, np.float32)
    for tp, kept in ((0.35, [1]), (0.65, [1, 3]), (0.75, [1, 3, 0]), (0.85, [1, 3, 0, 2]), (1.0, [1, 3, 0, 2, 4])):
        # equal logits at 0, 2, 4: the lower index enters the nucleus first
        for uu in (0.0, 0.999):
            u = np.array([[[uu, 0.5], [0.3, 0.5]]], np.float32)
            r = oracle.verify_warped(L, q, x, u, T, [5], [tp])
            pp = warped_p(L[0, 0], 1.0, 5, tp)
            assert sorted(np.nonzero(pp)[0].tolist()) == sorted(kept), (tp, pp)
            if 2 not in kept:
                assert r["num_accepted"][0] == 0 and r["out_tokens"][0, 0] in kept


def test_filter_errors():
    w = W.make_random(name="bad", B=4, k=2, V=50, dtype="f32", seed=25, logit_sigma=1.0, draft_sigma=1.0,
                      temperature=1.0)
    r = oracle.verify_warped(w.logits, w.q, w.x, w.u, w.T, [0, 3, 3, 3], np.array([1, 0, 1.5, 0.5], np.float32))
    assert r["row_status"].tolist()[:3] == [1024, 1024, 1024]
    assert r["row_status"][3] in (0, 16)


def _inverse_cdf(w, uu):
    """The smallest index whose prefix of w exceeds uu * sum(w) (vocabulary
    order); the last positive entry if rounding leaves none."""
    c = np.cumsum(w)
    i = int(np.searchsorted(c, uu * c[-1], side="right"))
    return i if i < len(w) else int(np.nonzero(w > 0)[0][-1])


def test_large_top_k_and_ties_match_the_definition():
    """top_k up to 4096 on rows with many equal logits (the K-th value tied
    across the cut): one-draft rows verified by a numpy restatement of the
    warped rule (lexsort ranks, p' on the kept prefix, accept test, residual
    or bonus by inverse CDF) give the oracle's outputs on every row the
    oracle does not flag as within 1e-6 of a decision edge."""
    rng = np.random.default_rng(31)
    B, V = 240, 5000
    w = W.make_random(name="bigk", B=B, k=1, V=V, dtype="f32", seed=32, logit_sigma=2.0, draft_sigma=0.3,
                      temperature=1.0)
    L = (np.round(w.logits * 4.0) / 4.0).astype(np.float32)  # values on a 0.25 grid: ties everywhere
    K = rng.choice([65, 100, 1000, 4096], size=B).astype(np.int32)
    P = rng.choice([1.0, 0.9, 0.5], size=B).astype(np.float32)
    r = oracle.verify_warped(L, w.q, w.x, w.u, w.T, K, P)
    checked = 0
    for b in range(B):
        if r["boundary"][b] or r["row_status"][b] & ~16:
            continue
        T = float(w.T[b])
        p0 = warped_p(L[b, 0], T, int(K[b]), float(P[b]))
        x0 = int(w.x[b, 0])
        rho = min(1.0, p0[x0] / max(float(w.q[b, 0, x0]), 1e-12))
        if float(w.u[b, 0, 0]) < rho:
            n_acc, tok = 1, _inverse_cdf(warped_p(L[b, 1], T, int(K[b]), float(P[b])), float(w.u[b, 1, 1]))
        else:
            res = np.where(p0 > 0, np.maximum(p0 - w.q[b, 0].astype(np.float64), 0.0), 0.0)
            n_acc, tok = 0, _inverse_cdf(res if res.sum() > 0 else p0, float(w.u[b, 0, 1]))
        assert r["num_accepted"][b] == n_acc, b
        assert r["out_tokens"][b, n_acc] == tok, (b, K[b], P[b])
        checked += 1
    assert checked >= B * 0.9
