"""GPU parity of top-k / top-p verification with the oracle ("Speculative
decoding." lesson, "Why the output is exactly p": the filters are applied to
p before the rule).  Integer outputs must match the oracle's on every row;
a row whose uniform lies within 1e-6 of a decision edge of the oracle may
differ only as parity.compare allows: its outcome must be the oracle's
outcome for that uniform moved by at most 1e-6."""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    import speculative_decoding_verification_57_gb300 as sv

    handle = sv.specv_create(0, max_batch=4096, max_k=31, vocab=262_144)
    yield handle
    sv.specv_destroy(handle)


def _run(h, w, top_k, top_p, onehot=False):
    import torch

    import speculative_decoding_verification_57_gb300 as sv
    from parity import to_device

    L, q, x, u, T = to_device(w, "cuda:0")
    out = sv.specv_verify_sample_filtered(h, L, None if onehot else q, x, u, T,
                                          torch.from_numpy(np.asarray(top_k, np.int32)).cuda(),
                                          torch.from_numpy(np.asarray(top_p, np.float32)).cuda())
    torch.cuda.synchronize()
    return {kk: v.cpu().numpy() for kk, v in out.items()}


def _check(w, got, top_k, top_p, onehot=False):
    from parity import compare

    if onehot:
        w = W.Workload(w.name, w.dtype, w.logits, None, w.x, w.u, w.T)
    tk = np.asarray(top_k, np.int32)
    tp = np.asarray(top_p, np.float32)

    def rows(sl, u):
        return oracle.verify_warped(w.logits[sl], None if w.q is None else w.q[sl], w.x[sl], u, w.T[sl], tk[sl],
                                    tp[sl])

    ref = rows(slice(None), w.u)
    stats = compare(w, got, ref, oracle_rows=rows)
    return stats["mismatched"], ref


@pytest.mark.parametrize("B,k,V,dtype,K,p", [(64, 5, 128256, "bf16", 50, 0.9), (16, 4, 32000, "bf16", 20, 1.0),
                                             (24, 3, 1000, "f32", 64, 0.7), (32, 6, 40003, "f32", 7, 0.5),
                                             (12, 16, 151936, "f32", 1, 1.0), (9, 2, 300, "bf16", 64, 1.0)])
def test_filtered_matches_oracle(h, B, k, V, dtype, K, p):
    w = W.make_random(name="filtered", B=B, k=k, V=V, dtype=dtype, seed=V + K, logit_sigma=3.0, draft_sigma=0.7,
                      temperature=0.9, spike=4.0, spike_mode="position", greedy_rows=2)
    mism, ref = _check(w, _run(h, w, [K] * B, [p] * B), [K] * B, [p] * B)
    assert mism <= 1
    assert (ref["row_status"] == 0).sum() >= B // 2


def test_filtered_one_hot_and_mixed_filters(h):
    rng = np.random.default_rng(4)
    w = W.make_random(name="filtered1h", B=48, k=4, V=50000, dtype="bf16", seed=5, logit_sigma=2.5, draft_sigma=0.5,
                      temperature=1.1, spike=6.0, spike_mode="position", greedy_rows=4)
    K = rng.integers(1, 65, size=48)
    P = rng.choice([1.0, 0.95, 0.8, 0.3], size=48).astype(np.float32)
    assert _check(w, _run(h, w, K, P, onehot=True), K, P, onehot=True)[0] <= 1
    assert _check(w, _run(h, w, K, P), K, P)[0] <= 1


def test_filtered_many_uniforms(h):
    """The benchmark logits, top_k 40 and top_p 0.95, 20 uniform sets."""
    base = W.make_workload("benchmark")
    rng = np.random.default_rng(6)
    mism = 0
    for r in range(20):
        w = W.Workload(base.name, base.dtype, base.logits, base.q, base.x,
                       rng.random(base.u.shape, dtype=np.float32), base.T)
        mism += _check(w, _run(h, w, [40] * 64, [0.95] * 64), [40] * 64, [0.95] * 64)[0]
    assert mism <= 1


def test_filter_errors_and_bad_rows(h):
    w = W.make_random(name="ferr", B=8, k=3, V=5000, dtype="f32", seed=9, logit_sigma=1.0, draft_sigma=0.5,
                      temperature=1.0)
    w.logits[5, 0, 17] = np.nan
    w.logits[6, 1, 3] = np.inf
    w.x[7, 0] = 5000
    K = [0, 4097, 10, 10, 10, 10, 10, 10]
    P = np.array([1, 1, 0, 1.5, 1, 1, 1, 1], np.float32)
    got = _run(h, w, K, P)
    _, ref = _check(w, got, K, P)
    assert ref["row_status"][[0, 1, 2, 3, 5, 7]].tolist() == [1024, 1024, 1024, 1024, 1, 2]
    # the same bad rows with top_k above 64 (the wide kernel's)
    K = [0, 4097, 100, 100, 3000, 4096, 200, 65]
    assert _check(w, _run(h, w, K, P), K, P)[1]["row_status"][[0, 1, 2, 3, 5, 7]].tolist() == [1024, 1024, 1024,
                                                                                               1024, 1, 2]


@pytest.mark.parametrize("B,k,V,dtype,K,p", [(16, 5, 128256, "bf16", 4096, 1.0), (16, 5, 128256, "bf16", 4096, 0.9),
                                             (24, 4, 32000, "bf16", 1000, 0.95), (8, 16, 151936, "f32", 300, 0.8),
                                             (12, 3, 40003, "f32", 65, 1.0), (10, 2, 1000, "f32", 2000, 0.7),
                                             (6, 31, 5001, "bf16", 100, 0.5)])
def test_wide_top_k_matches_oracle(h, B, k, V, dtype, K, p):
    """top_k above 64 (the radix-select kernel): up to the 4096 the oracle
    takes, top-p alone within the 4096 at the full Llama-3 vocabulary, top_k
    above V, 16 positions (two on one CTA) and 31."""
    w = W.make_random(name="wide", B=B, k=k, V=V, dtype=dtype, seed=V + K + k, logit_sigma=3.0, draft_sigma=0.4,
                      temperature=0.9, spike=4.0, spike_mode="position", greedy_rows=2)
    mism, ref = _check(w, _run(h, w, [K] * B, [p] * B), [K] * B, [p] * B)
    assert mism <= 1
    assert (ref["row_status"] == 0).sum() >= B // 2
    assert ref["num_accepted"].max() >= 1  # some rows get past position 0


def test_wide_mixed_with_narrow_rows(h):
    """One call whose rows go to both kernels (top_k up to 64 and above),
    one-hot and full q, many uniform sets at the benchmark's shape."""
    rng = np.random.default_rng(11)
    w = W.make_random(name="wmix", B=48, k=4, V=50000, dtype="bf16", seed=12, logit_sigma=2.5, draft_sigma=0.5,
                      temperature=1.1, spike=6.0, spike_mode="position", greedy_rows=4)
    K = rng.choice([5, 64, 65, 300, 4096], size=48)
    P = rng.choice([1.0, 0.95, 0.5], size=48).astype(np.float32)
    assert _check(w, _run(h, w, K, P, onehot=True), K, P, onehot=True)[0] <= 1
    assert _check(w, _run(h, w, K, P), K, P)[0] <= 1
    base = W.make_workload("benchmark")
    mism = 0
    for r in range(3):
        wr = W.Workload(base.name, base.dtype, base.logits[:16], base.q[:16], base.x[:16],
                        rng.random(base.u[:16].shape, dtype=np.float32), base.T[:16])
        mism += _check(wr, _run(h, wr, [1000] * 16, [0.95] * 16), [1000] * 16, [0.95] * 16)[0]
    assert mism <= 1


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_filtered_ties_and_degenerate_rows(h, dtype):
    """Equal logits (the lower index first), -0 beside +0, an all -inf
    position, +inf, and many positions (k = 31, several per CTA)."""
    B, k, V = 10, 31, 3001
    w = W.make_random(name="fties", B=B, k=k, V=V, dtype=dtype, seed=77, logit_sigma=2.0, draft_sigma=0.6,
                      temperature=1.0, greedy_rows=2)
    L = W.bf16_bits_to_f32(w.logits) if dtype == "bf16" else w.logits.copy()
    rng = np.random.default_rng(78)
    L[0] = 0.0                                    # flat: every entry ties
    L[1] = np.round(L[1] * 2.0) / 2.0             # few distinct values
    L[2] = np.where(rng.random(L[2].shape) < 0.5, -0.0, 0.0)
    L[2, :, 5] = 0.25
    L[3, 0] = -np.inf                              # an all -inf position
    L[4, 0, 17] = np.inf
    L[5] = np.round(L[5]) - 3.0                    # ties around the 64th entry
    w.x[0] = rng.integers(0, 64, size=k)           # inside the flat row's kept set
    logits = W.f32_to_bf16_bits(L.astype(np.float32)) if dtype == "bf16" else L.astype(np.float32)
    w = W.Workload(w.name, w.dtype, logits, w.q, w.x, w.u, w.T)
    for K, p in [(64, 1.0), (13, 0.8), (1, 1.0), (100, 0.8), (3001, 1.0), (2000, 0.3), (65, 0.99)]:
        _check(w, _run(h, w, [K] * B, [p] * B), [K] * B, [p] * B)


def test_filtered_pinned_host_q(h):
    """q in page-locked host memory is read in place (by both kernels)."""
    import torch

    import speculative_decoding_verification_57_gb300 as sv
    from parity import to_device

    w = W.make_random(name="fpin", B=16, k=4, V=32000, dtype="bf16", seed=21, logit_sigma=3.0, draft_sigma=0.7,
                      temperature=0.9, spike=4.0, spike_mode="position", greedy_rows=2)
    L, _, x, u, T = to_device(w, "cuda:0")
    K, P = [40] * 8 + [500] * 8, [0.9] * 16
    out = sv.specv_verify_sample_filtered(h, L, torch.from_numpy(w.q).pin_memory(), x, u, T,
                                          torch.tensor(K, dtype=torch.int32, device="cuda:0"),
                                          torch.tensor(P, dtype=torch.float32, device="cuda:0"))
    torch.cuda.synchronize()
    assert _check(w, {kk: v.cpu().numpy() for kk, v in out.items()}, K, P)[0] <= 1


@pytest.mark.parametrize("V,dtype,K,p,k", [(50, "f32", 64, 1.0, 3), (37, "bf16", 40, 0.5, 2), (2049, "bf16", 64, 0.05, 1),
                                           (8, "f32", 3, 1.0, 6), (50, "f32", 100, 1.0, 3), (37, "bf16", 4096, 0.5, 2),
                                           (2049, "bf16", 700, 0.05, 1), (8, "f32", 65, 0.9, 6)])
def test_filtered_small_vocabularies(h, V, dtype, K, p, k):
    """V below the 64 kept entries (padded lists), top-p cutting to a single
    entry, one draft, tiny vocabularies."""
    w = W.make_random(name="fsmall", B=20, k=k, V=V, dtype=dtype, seed=V * 7 + K, logit_sigma=2.0, draft_sigma=0.8,
                      temperature=1.0, greedy_rows=2)
    assert _check(w, _run(h, w, [K] * 20, [p] * 20), [K] * 20, [p] * 20)[0] <= 1


def test_filtered_refuses_pageable_q(h):
    """A pageable CPU q is refused before launch (the kernel never sees it)."""
    import ctypes

    import torch

    import speculative_decoding_verification_57_gb300 as sv
    from speculative_decoding_verification_57_gb300 import _lib
    from parity import to_device

    w = W.make_random(name="fpage", B=4, k=2, V=4096, dtype="bf16", seed=5, logit_sigma=2.0, draft_sigma=0.5,
                      temperature=1.0)
    L, _, x, u, T = to_device(w, "cuda:0")
    q = torch.from_numpy(w.q)  # pageable
    tk = torch.full((4,), 10, dtype=torch.int32, device="cuda:0")
    tp = torch.full((4,), 1.0, dtype=torch.float32, device="cuda:0")
    outs = [torch.empty(4, dtype=torch.int32, device="cuda:0"), torch.empty((4, 3), dtype=torch.int32, device="cuda:0"),
            torch.empty(4, dtype=torch.int32, device="cuda:0")]
    st = _lib.load().specv_verify_sample_filtered(
        h.ptr, sv.SPECV_BF16, ctypes.c_void_p(L.data_ptr()), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(x.data_ptr()),
        ctypes.c_void_p(u.data_ptr()), ctypes.c_void_p(T.data_ptr()), ctypes.c_void_p(tk.data_ptr()),
        ctypes.c_void_p(tp.data_ptr()), 4, 2, 4096, ctypes.c_void_p(outs[0].data_ptr()),
        ctypes.c_void_p(outs[1].data_ptr()), ctypes.c_void_p(outs[2].data_ptr()), None)
    assert st == 1  # SPECV_ERR_INVALID_ARGUMENT
    with pytest.raises(ValueError):
        sv.specv_verify_sample_filtered(h, L, q, x, u, T, tk, tp)
