"""Pins of the float64 oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden, each with its citation), closed forms, library
routines (scipy softmax, numpy argmax/searchsorted, scipy chi-square
quantiles) and exact enumeration on tiny inputs.
"""
import math
import random

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from conftest import read_golden
from helpers import (chi2_against, exact_outcome_distribution, expected_tokens, first_token_tv,
                     lattice_distribution, max_outcome_gap, montecarlo_distribution, prepare_tables,
                     random_simplex, tiny_tables)
from speculative_decoding_verification_57_gb300 import workloads as W


# --------------------------------------------------------------- closed form


def test_expected_tokens_matches_printed_tables():
    g = read_golden("expected_tokens.txt")
    ks = [int(v) for v in g["table_k"]]
    for key, vals in g.items():
        if key.startswith("table_alpha_"):
            a = float(key.split("_")[2])
            for kk, printed in zip(ks, vals):
                assert round(expected_tokens(a, kk), 3) == pytest.approx(printed, abs=1e-9), (a, kk)
    assert round(expected_tokens(0.8, 5), 3) == pytest.approx(g["beta_0.8_gamma_5"][0])
    assert round(expected_tokens(0.8, 5), 2) == pytest.approx(g["alpha_0.8_gamma_5_two_decimals"][0])


# --------------------------------------------------------------- step pins


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [0.25, 0.8, 1.0, 3.0])
def test_softmax_stats_match_scipy(dtype, T):
    rng = np.random.default_rng(1)
    raw = (rng.standard_normal(5003) * 4).astype(np.float32)
    row = W.f32_to_bf16_bits(raw) if dtype == "bf16" else raw
    vals = W.bf16_bits_to_f32(row).astype(np.float64) if dtype == "bf16" else raw.astype(np.float64)
    st, M, s, e = oracle.softmax_stats(row, T)
    assert st == 0
    assert M == vals.max()
    ref = scipy.special.softmax(vals / T)
    np.testing.assert_allclose(e / s, ref, rtol=1e-12, atol=0)


def test_softmax_stats_nonfinite():
    base = np.zeros(7, np.float32)
    for bad in (np.nan, np.inf):
        r = base.copy()
        r[3] = bad
        assert oracle.softmax_stats(r, 1.0)[0] == oracle.ST_NONFINITE
    assert oracle.softmax_stats(np.full(7, -np.inf, np.float32), 1.0)[0] == oracle.ST_NONFINITE
    r = base.copy()
    r[2] = -np.inf  # a masked entry is fine
    st, M, s, e = oracle.softmax_stats(r, 1.0)
    assert st == 0 and e[2] == 0.0 and s == pytest.approx(6.0)


def test_argmax_lowest_index_on_ties():
    rng = np.random.default_rng(2)
    for _ in range(200):
        V = int(rng.integers(1, 60))
        row = rng.integers(-3, 3, size=V).astype(np.float32)  # many ties
        st, a, m = oracle.argmax(row)
        assert st == 0 and a == int(np.argmax(row)) and m == row.max()
    r = np.array([0.0, -0.0, -1.0], np.float32)
    assert oracle.argmax(r)[1] == 0
    r = np.array([1.0, np.nan, 2.0], np.float32)
    assert oracle.argmax(r)[0] == oracle.ST_NONFINITE


def test_residual_pointwise_identity_and_mass():
    """min(q,p) + max(0,p-q) = p pointwise ("LLM Inference & Speculative
    Decoding ...", s.2 proof; "Speculative Decoding: Draft, Verify, Accept",
    correctness argument) and sum max(0,p-q) = 1 - sum min(p,q) ("Speculative
    Decoding: Mathematical Foundations, ...", proof, identity for 1 - beta)."""
    rng = np.random.default_rng(3)
    for V in (1, 2, 7, 1000):
        p = random_simplex(rng, V)
        q = random_simplex(rng, V, np.float32)
        st, r, S = oracle.residual(p, q)
        assert st == 0
        mn = np.minimum(p, q.astype(np.float64))
        np.testing.assert_allclose(mn + r, p, rtol=2.3e-16, atol=1e-300)
        assert S == pytest.approx(1.0 - mn.sum(), abs=1e-12)
        assert np.all(r >= 0)


def test_residual_printed_toy():
    """Residual of the demo's toy pair is printed as [0, 1/3, 2/3, 0]
    ("Speculative Decoding: Draft, Verify, Accept", demo output part B)."""
    g = read_golden("p4_toy.txt")
    p = np.array(g["p"]) / np.sum(g["p"])
    q = (np.array(g["q"]) / np.sum(g["q"])).astype(np.float32)
    st, r, S = oracle.residual(p, q)
    # q is stored as fp32, so the pin holds to fp32 rounding of q
    np.testing.assert_allclose(r / S, g["residual_printed"], atol=2e-7)
    # in pure float64 (q as double) the printed values are reached exactly
    exact = np.maximum(0, p - np.array(g["q"]) / np.sum(g["q"]))
    np.testing.assert_allclose(exact / exact.sum(), g["residual_printed"], rtol=1e-15, atol=1e-16)


def test_residual_flags_invalid_q():
    p = np.array([0.5, 0.5])
    for bad in (-0.1, np.nan, np.inf):
        assert oracle.residual(p, np.array([0.5, bad], np.float32))[0] == oracle.ST_Q_INVALID


def test_inverse_cdf_matches_searchsorted():
    """Smallest v with u*W < C(v) equals numpy.searchsorted(C, u*W, 'right')."""
    rng = np.random.default_rng(4)
    for _ in range(300):
        V = int(rng.integers(1, 50))
        w = rng.gamma(0.5, size=V)
        w[rng.random(V) < 0.3] = 0.0
        if w.sum() == 0:
            w[-1] = 1.0
        u = float(np.float32(rng.random()))
        t, lo, hi = oracle.inverse_cdf(w, u)
        C = np.cumsum(w)
        assert t == int(np.searchsorted(C, u * C[-1], side="right"))
        assert w[t] > 0 and lo <= u < hi
    # u = 0 never selects a leading zero-mass token
    assert oracle.inverse_cdf(np.array([0.0, 0.0, 1.0, 2.0]), 0.0)[0] == 2


# --------------------------------------------------------------- batch pins


def test_p1_vectors_distribution_and_mean_length():
    """The runnable verification script's p_true / q_skew ("LLM Inference &
    Speculative Decoding ...", s.5), at 200,000 trials: first emitted token
    and every emitted token follow p (TV < 0.01 as in the demo of "Speculative
    Decoding: Draft, Verify, Accept"; chi-square below the 5% quantile as in
    the "Speculative decoding." lesson), alpha prints as 0.80 and the mean
    emitted length matches (1 - alpha^(k+1)) / (1 - alpha) within 4 SE."""
    g = read_golden("p1_tv_vectors.txt")
    p, q = np.array(g["p_true"]), np.array(g["q_skew"])
    k = int(g["gamma"][0])
    alpha = np.minimum(p, q).sum()
    assert f"{alpha:.2f}" == f"{g['alpha_printed'][0]:.2f}"
    w = W.make_from_distributions(p, q, B=200_000, k=k, seed=11)
    r = oracle.verify(w.logits, w.q, w.x, w.u, w.T, nthreads=8)
    assert np.all(r["row_status"] == 0)
    tv, counts = first_token_tv(r["out_tokens"][:, 0], p)
    assert tv < 0.01
    chi2 = ((counts - p * counts.sum()) ** 2 / (p * counts.sum())).sum()
    assert chi2 < scipy.stats.chi2.ppf(0.95, len(p) - 1)
    emitted = r["out_tokens"][r["out_tokens"] >= 0]
    tv_all, _ = first_token_tv(emitted, p)
    assert tv_all < 0.01
    n = r["num_accepted"] + 1
    E = expected_tokens(alpha, k)
    assert abs(n.mean() - E) < 4 * n.std() / math.sqrt(len(n))
    assert abs(E - 3.3616) < 1e-12


def test_truncated_geometric_acceptance_counts():
    """P(num_accepted = m) = a^m (1-a) for m < k and a^k for m = k under iid
    acceptance ("Speculative Decoding: Mathematical Foundations, ...",
    "Expected Accepted Tokens per Speculative Round")."""
    rng = np.random.default_rng(5)
    for k in (2, 4, 8):
        V = 6
        p = random_simplex(rng, V)
        q = random_simplex(rng, V)
        a = np.minimum(p, q).sum()
        w = W.make_from_distributions(p, q, B=60_000, k=k, seed=100 + k)
        r = oracle.verify(w.logits, w.q, w.x, w.u, w.T, nthreads=8)
        probs = np.array([a ** m * (1 - a) for m in range(k)] + [a ** k])
        obs = np.bincount(r["num_accepted"], minlength=k + 1)
        exp = probs * len(r["num_accepted"])
        keep = exp > 5
        chi2 = (((obs - exp) ** 2 / exp)[keep]).sum()
        assert chi2 < scipy.stats.chi2.ppf(0.999, keep.sum() - 1), (k, obs, exp)
        n = r["num_accepted"] + 1
        assert abs(n.mean() - expected_tokens(a, k)) < 4 * n.std() / math.sqrt(len(n))


def _replay_p4(lib=None):
    """Replay the demo of "Speculative Decoding: Draft, Verify, Accept", part
    B: Python's random.Random(42) feeds, per trial and in this order, the
    draft proposal (inverse CDF with u <= running sum, the demo's own
    convention), the accept uniform and, only on rejection, the residual
    uniform.  The oracle makes the accept/residual decision (k = 1)."""
    g = read_golden("p4_toy.txt")
    p = np.array(g["p"]) / np.sum(g["p"])
    qd = np.array(g["q"]) / np.sum(g["q"])
    logits = np.log(p).astype(np.float32).reshape(1, 1, -1).repeat(2, axis=1)
    qrow = qd.astype(np.float32).reshape(1, 1, -1)
    T = np.ones(1, np.float32)
    lib = lib or oracle.load()
    rng = random.Random(int(g["seed"][0]))
    trials = int(g["trials"][0])
    counts = np.zeros(4, np.int64)

    def propose(u):
        acc = 0.0
        for i, v in enumerate(qd.tolist()):
            acc += v
            if u <= acc:
                return i
        return len(qd) - 1

    # the oracle is called in blocks: the residual uniform is drawn only on
    # rejection, so each trial's accept decision is needed before the next
    # draw; an accepted draw needs no residual uniform
    for _ in range(trials):
        x = propose(rng.random())
        ua = rng.random()
        u = np.array([[[ua, 0.5], [0.0, 0.5]]], np.float32)
        r = oracle.verify(logits, qrow, np.array([[x]], np.int32), u, T, lib=lib)
        if r["num_accepted"][0] == 1:
            counts[x] += 1
        else:
            ur = rng.random()
            u[0, 0, 1] = ur
            r = oracle.verify(logits, qrow, np.array([[x]], np.int32), u, T, lib=lib)
            assert r["num_accepted"][0] == 0
            counts[r["out_tokens"][0, 0]] += 1
    return counts, trials, p, g


def test_p4_exact_replay_reproduces_printed_output():
    counts, trials, p, g = _replay_p4()
    emp = counts / trials
    assert [round(v, 4) for v in emp.tolist()] == g["empirical_printed"]
    tv = 0.5 * np.abs(emp - p).sum()
    assert round(tv, 4) == g["tv_printed"][0]
    assert tv < g["tv_bound"][0]


def test_q_equals_p_always_accepts_and_bonus_is_textbook_sample():
    """q <= p everywhere gives min(1, p/q) = 1: every draft is kept and the
    bonus token is the inverse-CDF sample of p_k (numpy searchsorted on the
    float64 cumulative sum of scipy's softmax)."""
    rng = np.random.default_rng(6)
    B, k, V = 300, 3, 50
    L = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    P = scipy.special.softmax(L.astype(np.float64), axis=-1)
    q = P[:, :k].astype(np.float32)
    q = np.where(q.astype(np.float64) > P[:, :k], np.nextafter(q, np.float32(0)), q).astype(np.float32)
    x = rng.integers(0, V, size=(B, k)).astype(np.int32)
    u = rng.random((B, k + 1, 2), dtype=np.float32)
    T = np.ones(B, np.float32)
    r = oracle.verify(L, q, x, u, T)
    assert np.all(r["num_accepted"] == k)
    np.testing.assert_array_equal(r["out_tokens"][:, :k], x)
    for b in range(B):
        C = np.cumsum(P[b, k])
        assert r["out_tokens"][b, k] == int(np.searchsorted(C, u[b, k, 1] * C[-1], side="right"))


def test_one_hot_draft():
    """A one-hot q (prompt lookup) keeps its token with probability p(x) and
    otherwise samples p with x removed ("Speculative decoding." lesson, "One
    guess (lookup)" and "Where drafts come from")."""
    rng = np.random.default_rng(7)
    V, B = 12, 100_000
    p = random_simplex(rng, V)
    x0 = int(np.argmax(p))
    q = np.zeros(V)
    q[x0] = 1.0
    st, r_, S = oracle.residual(p, q.astype(np.float32))
    expect = p.copy()
    expect[x0] = 0.0
    np.testing.assert_allclose(r_ / S, expect / expect.sum(), rtol=1e-12)
    w = W.make_from_distributions(p, q, B=B, k=1, seed=8)
    assert np.all(w.x == x0)
    r = oracle.verify(w.logits, w.q, w.x, w.u, w.T, nthreads=8)
    keep = (r["num_accepted"] == 1).mean()
    assert abs(keep - p[x0]) < 4 * math.sqrt(p[x0] * (1 - p[x0]) / B)
    tv, _ = first_token_tv(r["out_tokens"][:, 0], p)
    assert tv < 0.01
    assert np.all(r["out_tokens"][r["num_accepted"] == 0, 0] != x0)


def test_one_hot_draft_without_q():
    """q = None means one-hot drafts ("Speculative decoding." lesson, "N-gram
    and prompt lookup": q is one-hot, so acceptance is just p(x)).  It must
    equal the explicit one-hot q in every output, and on one draft token it
    keeps x with probability p(x), otherwise samples p with x removed."""
    rng = np.random.default_rng(17)
    V, B = 10, 60_000
    p = random_simplex(rng, V)
    x0 = int(np.argsort(p)[-2])  # not the mode: the residual keeps the mode
    q = np.zeros(V)
    q[x0] = 1.0
    w = W.make_from_distributions(p, q, B=B, k=1, seed=18)
    assert np.all(w.x == x0)
    r_null = oracle.verify(w.logits, None, w.x, w.u, w.T, debug=True, nthreads=8)
    r_hot = oracle.verify(w.logits, w.q, w.x, w.u, w.T, debug=True, nthreads=8)
    for key in r_hot:
        np.testing.assert_array_equal(r_null[key], r_hot[key], err_msg=key)
    keep = (r_null["num_accepted"] == 1).mean()
    assert abs(keep - p[x0]) < 4 * math.sqrt(p[x0] * (1 - p[x0]) / B)
    fix = r_null["out_tokens"][r_null["num_accepted"] == 0, 0]
    assert np.all(fix != x0)
    expect = p.copy()
    expect[x0] = 0.0
    expect /= expect.sum()
    freq = np.bincount(fix, minlength=V) / len(fix)
    assert 0.5 * np.abs(freq - expect).sum() < 0.01
    # residual mass 1 - p(x) on the rejected rows
    rej = r_null["num_accepted"] == 0
    np.testing.assert_allclose(r_null["residual_mass"][rej], 1.0 - p[x0], rtol=1e-6)
    # many draft tokens and positions: still identical to the explicit form
    w2 = W.make_random(name="onehot", B=64, k=4, V=300, dtype="bf16", seed=19, logit_sigma=2.0, draft_sigma=1.0,
                       temperature=0.9)
    hot = np.zeros_like(w2.q)
    np.put_along_axis(hot, w2.x[:, :, None], 1.0, axis=2)
    a = oracle.verify(w2.logits, None, w2.x, w2.u, w2.T, debug=True)
    b = oracle.verify(w2.logits, hot, w2.x, w2.u, w2.T, debug=True)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_greedy_rows_match_textbook_argmax():
    rng = np.random.default_rng(9)
    B, k, V = 400, 4, 37
    L = rng.integers(-2, 2, size=(B, k + 1, V)).astype(np.float32)  # tie heavy
    A = np.argmax(L, axis=-1)
    x = A[:, :k].copy().astype(np.int32)
    # plant a first mismatch at a random position for most rows
    cut = rng.integers(0, k + 1, size=B)
    for b in range(B):
        if cut[b] < k:
            x[b, cut[b]] = (A[b, cut[b]] + 1 + rng.integers(0, V - 1)) % V
    r = oracle.verify(L, None, x, None, None)
    for b in range(B):
        j = int(cut[b])
        assert r["num_accepted"][b] == j
        assert list(r["out_tokens"][b, :j]) == list(x[b, :j])
        assert r["out_tokens"][b, j] == A[b, j]
        assert np.all(r["out_tokens"][b, j + 1:] == -1)
    # temperature 0 in a sampled call takes the same rule, q and u ignored
    q = np.full((B, k, V), 1.0 / V, np.float32)
    u = np.full((B, k + 1, 2), 0.5, np.float32)
    r2 = oracle.verify(L, q, x, u, np.zeros(B, np.float32))
    np.testing.assert_array_equal(r2["out_tokens"], r["out_tokens"])


def test_temperature_sharpens_and_debug_values():
    rng = np.random.default_rng(10)
    B, k, V = 20, 2, 64
    L = (rng.standard_normal((B, k + 1, V)) * 3).astype(np.float32)
    q = scipy.special.softmax(rng.standard_normal((B, k, V)), axis=-1).astype(np.float32)
    x = rng.integers(0, V, size=(B, k)).astype(np.int32)
    u = rng.random((B, k + 1, 2), dtype=np.float32)
    for T in (0.3, 1.0, 2.5):
        r = oracle.verify(L, q, x, u, np.full(B, T, np.float32), debug=True)
        T = float(np.float32(T))  # the temperature the oracle sees
        P = scipy.special.softmax(L.astype(np.float64) / T, axis=-1)
        np.testing.assert_array_equal(r["row_max"], L.max(-1))
        pa = np.take_along_axis(P[:, :k], x[..., None], -1)[..., 0]
        np.testing.assert_allclose(r["p_at_draft"], pa, rtol=1e-12)
        np.testing.assert_allclose(r["row_sumexp"] * np.exp(L.max(-1).astype(np.float64) / T),
                                   np.exp(L.astype(np.float64) / T).sum(-1), rtol=1e-12)
        rej = (r["num_accepted"] < k)
        for b in np.nonzero(rej)[0]:
            j = r["num_accepted"][b]
            S = np.maximum(0, P[b, j] - q[b, j].astype(np.float64)).sum()
            assert r["residual_mass"][b] == pytest.approx(S, rel=1e-12)


def test_status_bits_and_walk_order():
    V, k = 6, 3
    base_L = np.log(np.array([0.3, 0.2, 0.2, 0.1, 0.1, 0.1], np.float64)).astype(np.float32)
    L = np.tile(base_L, (1, k + 1, 1))
    q = np.tile(np.full(V, 1.0 / V, np.float32), (1, k, 1))
    x = np.array([[0, 0, 0]], np.int32)
    u = np.zeros((1, k + 1, 2), np.float32)
    T = np.ones(1, np.float32)

    def run(L=L, q=q, x=x, u=u, T=T):
        r = oracle.verify(L, q, x, u, T)
        return r["row_status"][0], r["num_accepted"][0], r["out_tokens"][0]

    st, n, out = run()
    assert st == 0 and n == k  # p(0)=0.3 > q=1/6 and u = 0 < 1: all kept
    for Tbad in (-1.0, np.nan, np.inf, 1e-40):
        st, n, out = run(T=np.array([Tbad], np.float32))
        assert st == oracle.ST_TEMPERATURE and n == 0 and np.all(out == -1)
    st, n, out = run(x=np.array([[0, V, 0]], np.int32))
    assert st == oracle.ST_TOKEN_RANGE and n == 0 and np.all(out == -1)
    uu = u.copy()
    uu[0, 1, 0] = 1.0
    assert run(u=uu)[0] == oracle.ST_UNIFORM_RANGE
    uu = u.copy()
    uu[0, k, 1] = -0.5  # bonus uniform
    assert run(u=uu)[0] == oracle.ST_UNIFORM_RANGE
    LL = L.copy()
    LL[0, 2, 4] = np.nan
    assert run(L=LL)[0] == oracle.ST_NONFINITE
    LL = L.copy()
    LL[0, 3, 1] = np.inf  # the bonus row is examined too
    assert run(L=LL)[0] == oracle.ST_NONFINITE
    qq = q.copy()
    qq[0, 1, 0] = -1e-3
    assert run(q=qq)[0] == oracle.ST_Q_INVALID
    # an error past the stop position is never examined
    uu = u.copy()
    uu[0, 0, 0] = 0.99  # reject at position 0 (rho = 1 there, so force via x)
    xx = np.array([[5, 0, 0]], np.int32)  # p=0.1 < q=1/6: rho = 0.6
    LL = L.copy()
    LL[0, 2, 0] = np.nan
    st, n, out = run(L=LL, x=xx, u=uu)
    assert st == 0 and n == 0 and out[0] >= 0 and out[0] != 5
    # q summing to 2: the residual is empty, the token comes from p (bit 16)
    qq = np.tile((2 * np.exp(base_L.astype(np.float64)) / np.exp(base_L.astype(np.float64)).sum()).astype(np.float32), (1, k, 1))
    st, n, out = run(q=qq, x=xx, u=uu)
    assert st == oracle.ST_ZERO_RESIDUAL and n == 0 and 0 <= out[0] < V


def test_boundary_flag_marks_close_uniforms():
    V, k = 4, 1
    p = np.array([0.1, 0.2, 0.3, 0.4])
    L = np.log(p).astype(np.float32).reshape(1, 1, V).repeat(k + 1, axis=1)
    q = np.array([[[0.4, 0.2, 0.2, 0.2]]], np.float32)
    x = np.array([[0]], np.int32)
    T = np.ones(1, np.float32)
    st, M, s, e = oracle.softmax_stats(L[0, 0], 1.0)
    rho = (e[0] / s) / np.float64(np.float32(0.4))
    for du, flagged in ((0.0, True), (5e-7, True), (-5e-7, True), (3e-6, False)):
        u = np.array([[[np.float32(rho + du), 0.5], [0.5, 0.5]]], np.float32)
        r = oracle.verify(L, q, x, u, T, boundary_eps=1e-6)
        assert (r["boundary"][0] == 1) == flagged, du


# --------------------------------------------------------------- brute force


@pytest.mark.parametrize("V,k,seed", [(2, 1, 0), (3, 1, 1), (3, 2, 2), (2, 2, 3)])
def test_brute_force_output_distribution(V, k, seed):
    """(a) The enumerated distribution obeys the sequence-level theorem of the
    "Speculative decoding." lesson ("From one token to a whole sequence"):
    the first token follows p(.|prefix) and, given the round continued past
    position t, token t+1 follows p(.|tokens so far).  (b) The oracle, driven
    by every draft sequence (weighted by its draft probability) and a midpoint
    lattice of uniforms, reproduces that distribution within the lattice's
    resolution."""
    import itertools

    rng = np.random.default_rng(seed)
    tabs = prepare_tables(tiny_tables(rng, V, k))
    exact = exact_outcome_distribution(tabs, V, k)
    assert sum(exact.values()) == pytest.approx(1.0, abs=1e-6)
    # (a) first token marginal and continuation conditionals
    first = np.zeros(V)
    for key, pr in exact.items():
        first[key[0]] += pr
    np.testing.assert_allclose(first, tabs[()][3], atol=2e-6)
    for t in range(k):
        for pre in itertools.product(range(V), repeat=t + 1):
            cont = np.zeros(V)
            for key, pr in exact.items():
                if len(key) > t + 1 and key[: t + 1] == pre:
                    cont[key[t + 1]] += pr
            if cont.sum() > 1e-9:
                np.testing.assert_allclose(cont / cont.sum(), tabs[pre][3], atol=2e-5)
    # (b) oracle on a lattice of uniforms (every outcome within the lattice's
    # resolution) and on simulated rounds (chi-square at the 1e-6 level)
    got, N = lattice_distribution(tabs, V, k)
    worst = max_outcome_gap(exact, got)
    assert worst < (k + 2) / N, worst
    counts = montecarlo_distribution(tabs, V, k, 400_000, seed=seed + 40)
    chi2, dof = chi2_against(exact, counts)
    assert chi2 < scipy.stats.chi2.ppf(1 - 1e-6, dof), (chi2, dof)
