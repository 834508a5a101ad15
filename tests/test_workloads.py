"""The seeded input recipe: shapes, types and distributions of the named
workloads as the configurations state them, and determinism.  The
generators serve both the GPU path and the oracle, and hold none of the
method's arithmetic, so these checks pin only what goes in."""
import numpy as np
import pytest

from speculative_decoding_verification_57_gb300 import workloads as W

SPECS = {
    # name: (B, k, V, dtype, T of sampled rows, logit sigma, greedy rows)
    "toy": (1, 4, 1000, "f32", 1.0, 2.0, 0),
    "zipf": (8, 4, 32000, "bf16", 0.8, 3.0, 0),
    "benchmark": (64, 5, 128256, "bf16", 1.0, 3.0, 0),
    "mixed": (256, 8, 128256, "bf16", 0.7, 3.0, 128),
    "split_v": (16, 16, 151936, "f32", 1.0, 4.0, 0),
}


def _logits_f32(w):
    return W.bf16_bits_to_f32(w.logits) if w.dtype == "bf16" else w.logits


@pytest.mark.parametrize("name", ["toy", "zipf", "benchmark", "split_v"])
def test_shapes_types_and_distributions(name):
    B, k, V, dtype, T, sigma, greedy = SPECS[name]
    w = W.make_workload(name)
    assert (w.B, w.k, w.V, w.dtype) == (B, k, V, dtype)
    assert w.logits.shape == (B, k + 1, V) and w.logits.dtype == (np.uint16 if dtype == "bf16" else np.float32)
    assert w.q.shape == (B, k, V) and w.q.dtype == np.float32
    assert w.x.shape == (B, k) and w.x.dtype == np.int32 and w.x.min() >= 0 and w.x.max() < V
    assert w.u.shape == (B, k + 1, 2) and w.u.dtype == np.float32 and w.u.min() >= 0 and w.u.max() < 1
    assert np.all(w.T[greedy:] == np.float32(T)) and np.all(w.T[:greedy] == 0)
    L = _logits_f32(w).astype(np.float64)
    # the bulk of every row is N(0, sigma^2): median absolute value sigma * 0.6745
    mad = np.median(np.abs(L), axis=-1)
    assert np.allclose(mad, sigma * 0.6745, rtol=0.1)
    # q is a probability distribution in fp32 at every draft position
    assert np.all(w.q >= 0) and np.allclose(w.q.sum(-1, dtype=np.float64), 1.0, atol=1e-4)


def test_spike_per_position():
    """spike_mode "position" (the benchmark's +8): exactly one token per
    (row, position) is lifted, a different random token at each position."""
    w = W.make_random(name="s", B=50, k=5, V=1000, dtype="f32", seed=5, logit_sigma=0.5, draft_sigma=1.0,
                      temperature=1.0, spike=8.0, spike_mode="position")
    high = w.logits > 5.0
    assert np.all(high.sum(-1) == 1)
    idx = np.argmax(w.logits, axis=-1)
    assert len(np.unique(idx)) > 200  # spread over the vocabulary, not one token


def test_zipf_boost_is_one_token_per_row():
    """spike_mode "zipf" (the zipf workload's +6): one token per row, the
    same at every position, its vocabulary index r - 1 with r ~ Zipf(1.1)
    restricted to r <= V."""
    w = W.make_random(name="z", B=3000, k=4, V=1000, dtype="f32", seed=6, logit_sigma=0.5, draft_sigma=1.0,
                      temperature=1.0, spike=6.0, spike_mode="zipf")
    high = w.logits > 3.0  # the lift is 6 sigma above the bulk's largest and 6 sigma below the spike
    assert np.all(high.sum(-1) == 1)
    idx = np.argmax(w.logits, axis=-1)
    assert np.all(idx == idx[:, :1])  # the same token at every position
    # draws above V are redrawn, so the law is Zipf truncated at V:
    # P(rank 1) = 1 / sum_{r <= V} r^-1.1 (0.179 at V = 1000)
    p1 = 1.0 / np.sum(np.arange(1, w.V + 1, dtype=np.float64) ** -1.1)
    frac0 = np.mean(idx[:, 0] == 0)
    assert abs(frac0 - p1) < 0.02  # 3 standard errors at 3000 rows


def test_mixed_half_greedy_and_draft_sigmas():
    w = W.make_workload("mixed")
    assert np.all(w.T[:128] == 0) and np.all(w.T[128:] == np.float32(0.7))


def test_greedy_rows_draft_the_argmax():
    w = W.make_random(name="g", B=6, k=3, V=500, dtype="f32", seed=4, logit_sigma=2.0, draft_sigma=1.0,
                      temperature=1.0, greedy_rows=3)
    # greedy drafts are the argmax of the draft logits, i.e. of q
    assert np.array_equal(w.x[:3], np.argmax(w.q[:3], axis=-1).astype(np.int32))


def test_drafts_follow_q():
    """Draft tokens are drawn from q: over many rows the empirical law of
    the first draft matches q (V = 5, one shared q)."""
    p = np.array([0.1, 0.2, 0.3, 0.25, 0.15])
    w = W.make_from_distributions(p, p, B=40000, k=1, seed=9)
    freq = np.bincount(w.x[:, 0], minlength=5) / w.B
    assert np.abs(freq - p).max() < 0.01


def test_seeded_and_deterministic():
    a, b = W.make_workload("zipf"), W.make_workload("zipf")
    for f in ("logits", "q", "x", "u", "T"):
        assert np.array_equal(getattr(a, f), getattr(b, f))
    c = W.make_workload("zipf", seed=1)
    assert not np.array_equal(a.logits, c.logits)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38, np.inf, -np.inf], dtype=np.float32)
    h = W.f32_to_bf16_bits(x)
    back = W.bf16_bits_to_f32(h)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: to even (1.0); 1 + 3 * 2^-8 ties up to 1 + 2^-6
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == np.float32(1.015625)
    assert back[3] == -2.5 and np.isinf(back[5]) and back[5] > 0 and np.isinf(back[6]) and back[6] < 0
