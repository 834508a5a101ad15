"""Shared helpers of the oracle tests: closed forms, statistics and the
brute-force enumeration of one verify round on a toy language model."""
import itertools

import numpy as np
import scipy.special

import oracle


def expected_tokens(alpha, k):
    """E[tokens per round] = (1 - alpha^(k+1)) / (1 - alpha) under iid
    acceptance ("Speculative Decoding: Mathematical Foundations, ...",
    "Expected Accepted Tokens per Speculative Round"; the same closed form
    appears on the other pages)."""
    if abs(1 - alpha) < 1e-12:
        return k + 1
    return (1 - alpha ** (k + 1)) / (1 - alpha)


def first_token_tv(tokens, p):
    """Total-variation distance between the empirical law of ``tokens`` and
    ``p``, plus the counts."""
    counts = np.bincount(tokens, minlength=len(p)).astype(np.float64)
    return 0.5 * np.abs(counts / counts.sum() - p).sum(), counts


def random_simplex(rng, V, dtype=np.float64):
    a = rng.gamma(0.3, size=V)
    return (a / a.sum()).astype(dtype)


def tiny_tables(rng, V, k):
    """Target p(.|prefix) and draft q(.|prefix) for every prefix of length
    0..k over a V-token vocabulary (a toy language model)."""
    tabs = {}
    for n in range(k + 1):
        for pre in itertools.product(range(V), repeat=n):
            tabs[pre] = (random_simplex(rng, V), random_simplex(rng, V))
    return tabs


def prepare_tables(tabs):
    """Attach the view of each table that a verify call sees: fp32 logits
    log p + shift, fp32 q, and the float64 softmax of those fp32 logits.
    Entries: (p, q, q_fp32, p_seen, logits_fp32)."""
    for pre, (p, q) in list(tabs.items()):
        # a prefix-dependent shift: the softmax ignores it, but it keeps the
        # rows' maxima and sums distinct, so mixing rows up shows
        shift = 1.7 * len(pre) - 0.9 * sum(pre) + 0.3
        logit = (np.log(p) + shift).astype(np.float32)
        tabs[pre] = (p, q, q.astype(np.float32), scipy.special.softmax(logit.astype(np.float64)), logit)
    return tabs


def _draft_weight(tabs, d):
    w = 1.0
    for i in range(len(d)):
        qd = tabs[d[:i]][2].astype(np.float64)
        w *= qd[d[i]] / qd.sum()
    return w


def exact_outcome_distribution(tabs, V, k):
    """Probability of every emitted token sequence of one round, by
    enumeration of the draft tokens and of the accept / reject branches: a
    draft x at prefix h is proposed with q(x|h) and kept with min(1, p/q); a
    rejection emits from max(0, p - q) normalised; k keeps are followed by
    the bonus token from p(.|h)."""
    out = {}
    for d in itertools.product(range(V), repeat=k):
        w = _draft_weight(tabs, d)
        keep = 1.0
        for i in range(k + 1):
            p = tabs[d[:i]][3]
            if i == k:
                for y in range(V):
                    key = d + (y,)
                    out[key] = out.get(key, 0.0) + w * keep * p[y]
                break
            qv = tabs[d[:i]][2].astype(np.float64)
            rho = min(1.0, p[d[i]] / max(qv[d[i]], 1e-12))
            res = np.maximum(0.0, p - qv)
            if rho < 1.0:
                assert res.sum() > 0
                for y in range(V):
                    key = d[:i] + (y,)
                    out[key] = out.get(key, 0.0) + w * keep * (1 - rho) * res[y] / res.sum()
            keep *= rho
    return out


def lattice_distribution(tabs, V, k, lib=None):
    """Outcome distribution of the oracle over every draft sequence (weighted
    by its draft probability) and a midpoint lattice of uniforms: one N-point
    axis per accept uniform U[i,0] and one for the draw uniform (the same
    value serves U[j,1] at whatever position j the walk stops, since only one
    of them is ever read).  Returns (distribution, N)."""
    N = 400 if k == 1 else 60
    grid = (np.arange(N) + 0.5) / N
    mesh = np.stack(np.meshgrid(*([grid] * (k + 1)), indexing="ij"), -1).reshape(-1, k + 1).astype(np.float32)
    R = mesh.shape[0]
    got = {}
    for d in itertools.product(range(V), repeat=k):
        w = _draft_weight(tabs, d)
        logits = np.stack([tabs[d[:i]][4] for i in range(k + 1)])[None].repeat(R, 0)
        q = np.stack([tabs[d[:i]][2] for i in range(k)])[None].repeat(R, 0)
        u = np.empty((R, k + 1, 2), np.float32)
        u[:, :k, 0] = mesh[:, :k]
        u[:, k, 0] = 0.5
        u[:, :, 1] = mesh[:, k:k + 1]
        x = np.array(d, np.int32)[None].repeat(R, 0)
        r = oracle.verify(logits, q, x, u, np.ones(R, np.float32), nthreads=8, lib=lib)
        assert np.all(r["row_status"] == 0)
        rows, counts = np.unique(r["out_tokens"], axis=0, return_counts=True)
        for row, c in zip(rows, counts):
            key = tuple(int(t) for t in row if t >= 0)
            got[key] = got.get(key, 0.0) + w * c / R
    return got, N


def max_outcome_gap(a, b):
    keys = set(a) | set(b)
    return max(abs(a.get(kk, 0.0) - b.get(kk, 0.0)) for kk in keys)


def montecarlo_distribution(tabs, V, k, n, seed, lib=None):
    """Outcome counts of the oracle over ``n`` simulated rounds: drafts drawn
    from q(.|prefix) (fp32 q, inverse CDF), uniforms seeded.  Returns a dict
    outcome -> count."""
    rng = np.random.default_rng(seed)
    prefixes = sorted(tabs, key=lambda t: (len(t), t))
    index = {pre: i for i, pre in enumerate(prefixes)}
    logit_tab = np.stack([tabs[pre][4] for pre in prefixes])
    q_tab = np.stack([tabs[pre][2] for pre in prefixes])
    d = np.zeros((n, k), np.int32)
    rows = np.zeros((n, k + 1), np.int64)  # table index of every position
    for i in range(k + 1):
        if i == 0:
            rows[:, 0] = index[()]
        else:
            keys = [index[tuple(r)] for r in d[:, :i].tolist()]
            rows[:, i] = keys
        if i == k:
            break
        u = rng.random(n)
        for t in np.unique(rows[:, i]):
            sel = rows[:, i] == t
            c = np.cumsum(q_tab[t].astype(np.float64))
            d[sel, i] = np.minimum(np.searchsorted(c, u[sel] * c[-1], side="right"), V - 1)
    logits = logit_tab[rows]
    q = q_tab[rows[:, :k]]
    uu = rng.random((n, k + 1, 2), dtype=np.float32)
    r = oracle.verify(logits, q, d, uu, np.ones(n, np.float32), nthreads=8, lib=lib)
    assert np.all(r["row_status"] == 0)
    out_rows, counts = np.unique(r["out_tokens"], axis=0, return_counts=True)
    return {tuple(int(t) for t in row if t >= 0): int(c) for row, c in zip(out_rows, counts)}


def chi2_against(exact, counts):
    """Pearson chi-square of ``counts`` against the probabilities ``exact``
    (outcomes with expected count below 5 pooled), with its degrees of
    freedom."""
    n = sum(counts.values())
    keys = sorted(set(exact) | set(counts))
    obs = np.array([counts.get(kk, 0) for kk in keys], np.float64)
    exp = np.array([exact.get(kk, 0.0) * n for kk in keys])
    small = exp < 5
    o = np.append(obs[~small], obs[small].sum())
    e = np.append(exp[~small], exp[small].sum())
    if e[-1] == 0:
        if o[-1] > 0:
            return np.inf, len(o) - 2
        o, e = o[:-1], e[:-1]
    return float(((o - e) ** 2 / e).sum()), len(o) - 1
