"""Power of the oracle pins: plausible mistakes planted in a copy of the
oracle (compiled to a temporary shared object, on the CPU) must each fail at
least one pin, while the unmodified oracle passes them all.

The first two mistakes are the ones the "Speculative decoding." lesson warns
about under "Break It" (resample from p on rejection; a greedy draft passed
with its softmax q); the others are slips of sign, index or normalisation.
"""
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from conftest import ROOT, read_golden
from helpers import (chi2_against, exact_outcome_distribution, first_token_tv, lattice_distribution,
                     max_outcome_gap, montecarlo_distribution, prepare_tables, random_simplex, tiny_tables)
from speculative_decoding_verification_57_gb300 import workloads as W

SRC = os.path.join(ROOT, "oracle", "specv_oracle.c")


def check_tv(lib):
    """First-token law on the vectors of "LLM Inference & Speculative
    Decoding ...", s.5 (100,000 rows): TV < 0.01 and chi-square below the
    0.1% quantile."""
    g = read_golden("p1_tv_vectors.txt")
    p, q = np.array(g["p_true"]), np.array(g["q_skew"])
    w = W.make_from_distributions(p, q, B=100_000, k=4, seed=21)
    r = oracle.verify(w.logits, w.q, w.x, w.u, w.T, nthreads=8, lib=lib)
    if np.any(r["row_status"] & oracle.ST_ERROR_MASK):
        return False
    tv, counts = first_token_tv(r["out_tokens"][:, 0], p)
    chi2 = ((counts - p * counts.sum()) ** 2 / (p * counts.sum())).sum()
    return tv < 0.01 and chi2 < scipy.stats.chi2.ppf(0.999, len(p) - 1)


def check_brute(lib):
    """Exact enumeration against the oracle: a lattice of uniforms at V = 3,
    k = 1, and 400,000 simulated rounds (chi-square at the 1e-6 level) at
    V = 3, k = 2."""
    rng = np.random.default_rng(1)
    tabs = prepare_tables(tiny_tables(rng, 3, 1))
    got, N = lattice_distribution(tabs, 3, 1, lib=lib)
    if max_outcome_gap(exact_outcome_distribution(tabs, 3, 1), got) >= 3 / N:
        return False
    rng = np.random.default_rng(2)
    tabs = prepare_tables(tiny_tables(rng, 3, 2))
    counts = montecarlo_distribution(tabs, 3, 2, 400_000, seed=5, lib=lib)
    chi2, dof = chi2_against(exact_outcome_distribution(tabs, 3, 2), counts)
    return chi2 < scipy.stats.chi2.ppf(1 - 1e-6, dof)


def check_identity(lib):
    """min(q,p) + max(0, p-q) = p and S = 1 - sum min(p,q)."""
    rng = np.random.default_rng(3)
    p = random_simplex(rng, 500)
    q = random_simplex(rng, 500, np.float32)
    st, r, S = oracle.residual(p, q, lib=lib)
    mn = np.minimum(p, q.astype(np.float64))
    return st == 0 and np.allclose(mn + r, p, rtol=1e-15, atol=0) and abs(S - (1 - mn.sum())) < 1e-12


def check_softmax(lib):
    rng = np.random.default_rng(1)
    row = (rng.standard_normal(300) * 3).astype(np.float32)
    st, M, s, e = oracle.softmax_stats(row, 0.5, lib=lib)
    return st == 0 and np.allclose(e / s, scipy.special.softmax(row.astype(np.float64) / 0.5), rtol=1e-12)


CHECKS = {"tv": check_tv, "brute": check_brute, "identity": check_identity, "softmax": check_softmax}

MUTANTS = {
    # "Break It": on rejection, sample the target p again instead of the residual
    "resample_from_p": (
        "            token = specv_oracle_inverse_cdf(buf_w, V, (double)u1, &lo, &hi);\n        } else {",
        "            token = specv_oracle_inverse_cdf(buf_p, V, (double)u1, &lo, &hi);\n        } else {",
    ),
    # residual without the max(0, .)
    "no_clamp": ("        double r = p[v] - qv;\n        if (r < 0.0) r = 0.0;\n", "        double r = p[v] - qv;\n"),
    # acceptance ratio upside down
    "ratio_inverted": ("double rho = p / (q > 1e-12 ? q : 1e-12);", "double rho = q / (p > 1e-12 ? p : 1e-12);"),
    # accept test at position i reads the target row of position i+1
    "accept_next_row": (
        "        st |= specv_oracle_softmax_stats(J->dtype, row_ptr(J, b, i), V, T, &M, &s, NULL);",
        "        st |= specv_oracle_softmax_stats(J->dtype, row_ptr(J, b, i + 1), V, T, &M, &s, NULL);",
    ),
    # bonus drawn from the last draft position instead of position k
    "bonus_wrong_row": (
        "int st = specv_oracle_softmax_stats(J->dtype, row_ptr(J, b, j), V, T, &M, &s, buf_w);",
        "int st = specv_oracle_softmax_stats(J->dtype, row_ptr(J, b, j == k ? k - 1 : j), V, T, &M, &s, buf_w);",
    ),
    # residual built from the draft row of the next position
    "residual_next_q": (
        "specv_oracle_residual(buf_p, J->q + (b * k + j) * V, V, buf_w, &S)",
        "specv_oracle_residual(buf_p, J->q + (b * k + (j + 1) % k) * V, V, buf_w, &S)",
    ),
    # inverse CDF compares u with the unnormalised running sum
    "unnormalised_cdf": ("    double target = u * W;\n", "    double target = u;\n"),
    # temperature multiplies the logits
    "temperature_multiplies": (
        "        double e = exp((logit_at(dtype, row, v) - M) / T);",
        "        double e = exp((logit_at(dtype, row, v) - M) * T);",
    ),
}


@pytest.fixture(scope="module")
def base_results():
    lib = oracle.load()
    return {name: fn(lib) for name, fn in CHECKS.items()}


def test_unmodified_oracle_passes_every_check(base_results):
    assert all(base_results.values()), base_results


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"patch for {name} no longer applies"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = oracle.compile_oracle(str(path), str(tmp_path / f"lib{name}.so"))
    lib = oracle.load(so)
    failed = []
    for c, fn in CHECKS.items():
        try:
            ok = fn(lib)
        except AssertionError:
            ok = False
        if not ok:
            failed.append(c)
    assert failed, f"mutant {name} passed every pin"


def test_greedy_draft_with_softmax_q_is_caught():
    """ "Speculative decoding." lesson, "Break It", third item: drafting with
    argmax but passing the softmax q into the rule breaks the output law."""
    g = read_golden("p1_tv_vectors.txt")
    p, q = np.array(g["p_true"]), np.array(g["q_skew"])
    w = W.make_from_distributions(p, q, B=100_000, k=4, seed=22)
    w.x[:] = int(np.argmax(q))  # greedy draft
    r = oracle.verify(w.logits, w.q, w.x, w.u, w.T, nthreads=8)
    tv, _ = first_token_tv(r["out_tokens"][:, 0], p)
    assert tv > 0.05


def test_resample_from_p_matches_stated_law(tmp_path):
    """The resample-from-p bug yields min(p,q) + (1 - alpha) p (the law the
    "Break It" section states); checked on the s.5 vectors of "LLM Inference
    & Speculative Decoding ...", where it sits at TV 0.12 from p."""
    old, new = MUTANTS["resample_from_p"]
    path = tmp_path / "m.c"
    path.write_text(open(SRC).read().replace(old, new))
    lib = oracle.load(oracle.compile_oracle(str(path), str(tmp_path / "libm.so")))
    g = read_golden("p1_tv_vectors.txt")
    p, q = np.array(g["p_true"]), np.array(g["q_skew"])
    law = np.minimum(p, q) + (1 - np.minimum(p, q).sum()) * p
    assert 0.5 * np.abs(law - p).sum() == pytest.approx(0.12, abs=1e-12)
    w = W.make_from_distributions(p, q, B=200_000, k=4, seed=23)
    r = oracle.verify(w.logits, w.q, w.x, w.u, w.T, nthreads=8, lib=lib)
    tv_law, _ = first_token_tv(r["out_tokens"][:, 0], law)
    assert tv_law < 0.01
