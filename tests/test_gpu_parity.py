"""GPU parity: the CUDA verify path through the C ABI against the float64
oracle on the same seeded inputs and uniforms."""
import os

import numpy as np
import pytest

import oracle
from conftest import read_golden
from helpers import first_token_tv
from parity import compare, run_gpu, to_device
from speculative_decoding_verification_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    import speculative_decoding_verification_57_gb300 as sv

    handle = sv.specv_create(0, max_batch=300_000, max_k=31, vocab=262_144)
    yield handle
    sv.specv_destroy(handle)


TOTALS = {"rows": 0, "flagged": 0, "mismatched": 0}


def _acc(stats):
    for key in TOTALS:
        TOTALS[key] += stats[key]
    return stats


@pytest.mark.parametrize("debug", [False, True])
@pytest.mark.parametrize("name", ["zipf", "benchmark", "mixed", "split_v"])
def test_named_workload_parity(h, name, debug):
    """Without debug outputs the split-vocabulary kernel reads no position
    past a row's first stop; with them it reads every position."""
    w = W.make_workload(name)
    got = run_gpu(h, w, debug=debug)
    stats = _acc(compare(w, got, check_debug=debug))
    print(name, debug, stats)


def test_toy_config_2000_rounds(h):
    """The toy workload: 2000 independent rounds of B=1, V=1000, fp32."""
    mism = 0
    for r in range(2000):
        w = W.make_workload("toy", seed=57001 + 1000 * r)
        got = run_gpu(h, w)
        mism += compare(w, got)["mismatched"]
    assert mism <= 1


def test_p1_vectors_200k_trials_on_gpu(h):
    """V = 8 alphabet of "LLM Inference & Speculative Decoding ...", s.5, at
    200,000 trials: parity with the oracle and the first-token law (TV < 0.01)."""
    g = read_golden("p1_tv_vectors.txt")
    p, q = np.array(g["p_true"]), np.array(g["q_skew"])
    w = W.make_from_distributions(p, q, B=200_000, k=4, seed=31)
    got = run_gpu(h, w)
    _acc(compare(w, got))
    tv, _ = first_token_tv(got["out_tokens"][:, 0], p)
    assert tv < 0.01


ODD = [
    # (V, k, B, dtype)
    (1, 1, 3, "f32"), (7, 2, 3, "bf16"), (8, 4, 2, "f32"), (13, 16, 3, "bf16"), (1001, 5, 3, "f32"),
    (2047, 3, 2, "bf16"), (2048, 31, 2, "f32"), (2049, 2, 3, "bf16"), (4099, 1, 3, "f32"),
    (32003, 16, 3, "bf16"), (65537, 2, 2, "f32"), (128257, 3, 2, "bf16"), (262144, 2, 2, "bf16"),
    (50000, 31, 3, "bf16"), (20000, 31, 2, "f32"),
]


@pytest.mark.parametrize("V,k,B,dtype", ODD)
def test_odd_sizes(h, V, k, B, dtype):
    w = W.make_random(name="odd", B=B, k=k, V=V, dtype=dtype, seed=V + 97 * k, logit_sigma=2.5,
                      draft_sigma=0.7, temperature=0.9, spike=5.0, spike_mode="position",
                      greedy_rows=1 if B > 2 else 0)
    for debug in (False, True):
        got = run_gpu(h, w, debug=debug)
        _acc(compare(w, got, check_debug=debug))


@pytest.mark.parametrize("offset,T", [(-40.0, 1.0), (0.0, 4.0), (40.0, 4.0), (40.0, 0.25), (200.0, 1.0)])
def test_bf16_logit_offsets(h, offset, T):
    """Softmax does not see a common offset, but the bf16 grid does: shifted
    logits put the stop row's large entries in a positive range (their exact
    e read from a per-row table), in a range reaching zero or below it (e
    evaluated directly), or on a coarse grid with many equal logits (+200:
    spacing 1)."""
    base = W.make_random(name="offset", B=6, k=4, V=50000, dtype="bf16", seed=int(offset) + 1000,
                         logit_sigma=3.0, draft_sigma=1.0, temperature=T, spike=6.0, spike_mode="position")
    lf = W.bf16_bits_to_f32(base.logits) + np.float32(offset)
    rng = np.random.default_rng(int(1000 + offset * 10 + T * 100))
    for _ in range(10):
        w = W.Workload("offset", "bf16", W.f32_to_bf16_bits(lf), base.q, base.x,
                       rng.random(base.u.shape, dtype=np.float32), base.T)
        debug = bool(_ % 2)
        got = run_gpu(h, w, debug=debug)
        _acc(compare(w, got, check_debug=debug))


@pytest.mark.parametrize("C", [None, 11, 16])
def test_cluster_sizes_agree(h, C, monkeypatch):
    """Every split of the vocabulary over a cluster gives the same result."""
    if C is not None:
        monkeypatch.setenv("SPECV_CLUSTER", str(C))
    w = W.make_random(name="split", B=4, k=3, V=151936, dtype="f32", seed=5, logit_sigma=4.0, draft_sigma=2.0,
                      temperature=1.0)
    for debug in (False, True):
        got = run_gpu(h, w, debug=debug)
        _acc(compare(w, got, check_debug=debug))


def test_unaligned_buffers(h):
    """Tensors starting one element past an aligned address exercise the
    unaligned head and tail of every slice."""
    import torch

    import speculative_decoding_verification_57_gb300 as sv

    for V, dtype in ((40001, "bf16"), (40003, "f32"), (1500, "bf16")):
        w = W.make_random(name="unaligned", B=3, k=4, V=V, dtype=dtype, seed=3, logit_sigma=3.0,
                          draft_sigma=1.0, temperature=1.0, spike=6.0, spike_mode="position")
        L, q, x, u, T = to_device(w, "cuda:0")
        Lb = torch.empty(L.numel() + 1, dtype=L.dtype, device="cuda:0")
        Lb[1:].copy_(L.reshape(-1))
        qb = torch.empty(q.numel() + 1, dtype=q.dtype, device="cuda:0")
        qb[1:].copy_(q.reshape(-1))
        out = sv.specv_verify_sample(h, Lb[1:].view(L.shape), qb[1:].view(q.shape), x, u, T)
        torch.cuda.synchronize()
        _acc(compare(w, {kk: v.cpu().numpy() for kk, v in out.items()}))


def test_greedy_entry_and_ties(h):
    import torch

    import speculative_decoding_verification_57_gb300 as sv

    rng = np.random.default_rng(4)
    for V, dtype in ((50, "bf16"), (5000, "bf16"), (70000, "f32")):
        B, k = 5, 6
        L = rng.integers(-3, 3, size=(B, k + 1, V)).astype(np.float32)  # heavy ties
        A = np.argmax(L, -1)
        x = A[:, :k].astype(np.int32).copy()
        x[1, 2] = (x[1, 2] + 1) % V
        x[3, 0] = (x[3, 0] + 5) % V
        Ls = W.f32_to_bf16_bits(L) if dtype == "bf16" else L
        ref = oracle.verify(Ls, None, x, None, None)
        Lt = torch.from_numpy(Ls.view(np.int16) if dtype == "bf16" else Ls).cuda()
        if dtype == "bf16":
            Lt = Lt.view(torch.bfloat16)
        out = sv.specv_verify_greedy(h, Lt, torch.from_numpy(x).cuda())
        torch.cuda.synchronize()
        for key in ("num_accepted", "out_tokens", "row_status"):
            np.testing.assert_array_equal(out[key].cpu().numpy(), ref[key])


def test_mixed_greedy_and_sampled_rows(h):
    w = W.make_random(name="mixed", B=12, k=5, V=50000, dtype="bf16", seed=12, logit_sigma=3.0,
                      draft_sigma=1.0, temperature=0.7, spike=8.0, spike_mode="position", greedy_rows=6)
    for debug in (False, True):
        got = run_gpu(h, w, debug=debug)
        _acc(compare(w, got, check_debug=debug))


def test_low_temperature(h):
    for V in (900, 40000):
        w = W.make_random(name="lowT", B=6, k=4, V=V, dtype="bf16", seed=V, logit_sigma=3.0, draft_sigma=0.3,
                          temperature=0.01)
        for debug in (False, True):
            got = run_gpu(h, w, debug=debug)
            _acc(compare(w, got, check_debug=debug))


@pytest.mark.parametrize("V", [300, 30000])
def test_status_bits(h, V):
    """Data errors set row_status bits and never fault: bad draft token,
    uniform, temperature, logits, q; an empty residual takes p (bit 16)."""
    B, k = 16, 3
    w = W.make_random(name="errors", B=B, k=k, V=V, dtype="f32", seed=77, logit_sigma=1.0, draft_sigma=0.5,
                      temperature=1.0)
    w.x[0, 0] = V
    w.x[1, 1] = -3
    w.u[2, 0, 0] = 1.0
    w.u[3, :, 1] = -0.25
    w.T[4] = -1.0
    w.T[5] = np.nan
    w.T[6] = np.inf
    w.T[7] = 1e-40
    w.logits[8, 0, 5] = np.nan
    w.logits[9, 1, 7] = np.inf
    w.logits[10, 0, :] = -np.inf
    w.q[11, 0, w.x[11, 0]] = -0.5
    w.q[12, :, 3] = np.nan
    w.u[12, :, 0] = 0.999  # reject early so the residual row is read
    # empty residual: q = 2p at every position, and a rejection at position 0
    st, M, s, e = oracle.softmax_stats(w.logits[13, 0], 1.0)
    w.q[13, 0] = (2.0 * e / s).astype(np.float32)
    w.u[13, 0, 0] = 0.9
    w.logits[14, 0, 3] = -np.inf  # a masked entry is not an error
    got = run_gpu(h, w)
    ref = oracle.verify(w.logits, w.q, w.x, w.u, w.T)
    expect = {0: 2, 1: 2, 2: 4, 4: 8, 5: 8, 6: 8, 7: 8, 8: 1, 9: 1, 10: 1, 11: 32}
    for b, bit in expect.items():
        assert ref["row_status"][b] & bit, (b, ref["row_status"][b])
    assert ref["row_status"][12] & 32 or ref["row_status"][12] == 0
    assert ref["row_status"][13] == 16
    _acc(compare(w, got, ref))


@pytest.mark.parametrize("V,dtype", [(700, "f32"), (50000, "bf16"), (50000, "f32")])
def test_masked_vocabulary(h, V, dtype):
    """Logits of -inf (masked entries) have p = 0: never sampled, and a
    draft token on a masked entry is always rejected."""
    w = W.make_random(name="masked", B=8, k=4, V=V, dtype=dtype, seed=V + 1, logit_sigma=2.0, draft_sigma=0.8,
                      temperature=0.9, spike=4.0, spike_mode="position", greedy_rows=2)
    rng = np.random.default_rng(V)
    mask = rng.random((w.B, w.k + 1, V)) < 0.4
    ninf = W.f32_to_bf16_bits(np.array([-np.inf], np.float32))[0] if dtype == "bf16" else -np.inf
    w.logits[mask] = ninf
    w.x[3, 0] = int(np.nonzero(mask[3, 0])[0][0])  # a draft on a masked entry
    for debug in (False, True):
        got = run_gpu(h, w, debug=debug)
        _acc(compare(w, got, check_debug=debug))
        assert got["num_accepted"][3] == 0


def test_deterministic(h):
    w = W.make_workload("zipf")
    a = run_gpu(h, w, debug=True)
    b = run_gpu(h, w, debug=True)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


@pytest.mark.parametrize("q_pinned", [True, False])
def test_host_buffer_entry(h, q_pinned):
    """Host buffers in: page-locked q is read in place by the kernel,
    pageable q is copied; both give the oracle's outputs."""
    import torch

    import speculative_decoding_verification_57_gb300 as sv

    w = W.make_workload("zipf")
    L = torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16).pin_memory()
    q = torch.from_numpy(w.q)
    out = sv.specv_verify_sample_host(h, L, q.pin_memory() if q_pinned else q.clone(),
                                      torch.from_numpy(w.x).pin_memory(), torch.from_numpy(w.u).pin_memory(),
                                      torch.from_numpy(w.T).pin_memory())
    _acc(compare(w, {kk: v.numpy() for kk, v in out.items()}))


@pytest.mark.parametrize("case", ["benchmark pinned q", "13 rows pageable q", "10 rows fp32 pinned q"])
def test_host_buffer_entry_large(h, case):
    """The host-buffer entry at full sizes: the benchmark workload with q read
    in place, a bf16 batch whose q is copied, and an fp32 batch at V = 151936."""
    import torch

    import speculative_decoding_verification_57_gb300 as sv

    if case == "benchmark pinned q":
        w, pinned = W.make_workload("benchmark"), True
    elif case == "13 rows pageable q":
        w = W.make_random(name="host", B=13, k=5, V=128256, dtype="bf16", seed=13, logit_sigma=3.0,
                          draft_sigma=1.0, temperature=1.0, spike=8.0, spike_mode="position", greedy_rows=2)
        pinned = False
    else:
        w = W.make_random(name="host", B=10, k=15, V=151936, dtype="f32", seed=10, logit_sigma=4.0,
                          draft_sigma=2.0, temperature=1.0)
        pinned = True
    L = torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16) if w.dtype == "bf16" else torch.from_numpy(w.logits)
    q = torch.from_numpy(w.q)
    out = sv.specv_verify_sample_host(h, L.pin_memory(), q.pin_memory() if pinned else q.clone(),
                                      torch.from_numpy(w.x).pin_memory(), torch.from_numpy(w.u).pin_memory(),
                                      torch.from_numpy(w.T).pin_memory())
    _acc(compare(w, {kk: v.numpy() for kk, v in out.items()}))


def test_empty_batch(h):
    import torch

    import speculative_decoding_verification_57_gb300 as sv

    L = torch.empty((0, 5, 1000), dtype=torch.float32, device="cuda:0")
    out = sv.specv_verify_sample(h, L, torch.empty((0, 4, 1000), device="cuda:0"),
                                 torch.empty((0, 4), dtype=torch.int32, device="cuda:0"),
                                 torch.empty((0, 5, 2), device="cuda:0"), torch.empty(0, device="cuda:0"))
    assert out["num_accepted"].numel() == 0


def test_bench_workload_many_uniforms(h):
    """The benchmarked workload (B=64, k=5, V=128256, bf16) in the bench's
    launch configuration, with 40 independent uniform sets: every row
    matches the oracle except at flagged boundaries, and disagreements stay
    below 1e-4 of all rows."""
    base = W.make_workload("benchmark")
    rng = np.random.default_rng(99)
    mism = rows = 0
    for r in range(40):
        w = W.Workload(base.name, base.dtype, base.logits, base.q, base.x,
                       rng.random(base.u.shape, dtype=np.float32), base.T)
        got = run_gpu(h, w)
        st = _acc(compare(w, got))
        mism += st["mismatched"]
        rows += st["rows"]
    print("bench workload", rows, "rows,", mism, "boundary disagreements")
    assert mism <= 1e-4 * rows + 0.5


@pytest.mark.parametrize("V,k,B,dtype", [(128256, 5, 64, "bf16"), (32000, 4, 8, "bf16"), (40003, 3, 6, "f32"),
                                        (1500, 4, 16, "f32"), (700, 6, 9, "bf16")])
def test_one_hot_drafts(h, V, k, B, dtype):
    """q = None: one-hot drafts (prompt lookup, greedy drafting).  Accept
    with p(x); a rejection samples p with x removed ("Speculative decoding."
    lesson, "One guess (lookup)", "N-gram and prompt lookup")."""
    w = W.make_random(name="onehot", B=B, k=k, V=V, dtype=dtype, seed=V + k, logit_sigma=2.5, draft_sigma=0.5,
                      temperature=0.9, spike=5.0, spike_mode="position", greedy_rows=1)
    w = W.Workload(w.name, w.dtype, w.logits, None, w.x, w.u, w.T)
    for debug in (False, True):
        got = run_gpu(h, w, debug=debug)
        st = _acc(compare(w, got, check_debug=debug))
        assert (got["row_status"] == 0).any()
        print("one-hot", V, debug, st)


def test_one_hot_many_uniforms(h):
    """The benchmark logits with one-hot drafts over 20 uniform sets."""
    base = W.make_workload("benchmark")
    rng = np.random.default_rng(5)
    for r in range(20):
        w = W.Workload(base.name, base.dtype, base.logits, None, base.x,
                       rng.random(base.u.shape, dtype=np.float32), base.T)
        _acc(compare(w, run_gpu(h, w)))


def test_zz_summary():
    """Disagreements at flagged boundaries over every parity case above."""
    print("parity totals", TOTALS)
    if TOTALS["rows"]:
        assert TOTALS["mismatched"] <= max(1, 1e-4 * TOTALS["rows"])


@pytest.mark.parametrize("kernel", ["row", "warp"])
def test_small_vocabulary_kernels(h, kernel, monkeypatch):
    """V <= 2048 has two kernels, a CTA per row (small batches) and a warp
    per row (large ones); each, forced, matches the oracle on odd sizes,
    debug outputs, one-hot drafts, masked entries and unaligned rows."""
    import torch

    import speculative_decoding_verification_57_gb300 as sv

    monkeypatch.setenv("SPECV_SMALLV", kernel)
    cases = [(1, 1, 3, "f32"), (7, 2, 3, "bf16"), (13, 16, 3, "bf16"), (1000, 4, 5, "f32"), (1001, 5, 3, "f32"),
             (2047, 3, 2, "bf16"), (2048, 31, 2, "f32"), (700, 6, 9, "bf16"), (33, 8, 40, "f32")]
    for V, k, B, dtype in cases:
        w = W.make_random(name="small", B=B, k=k, V=V, dtype=dtype, seed=V * 7 + k, logit_sigma=2.5,
                          draft_sigma=0.7, temperature=0.9, spike=4.0, spike_mode="position",
                          greedy_rows=1 if B > 2 else 0)
        for debug in (False, True):
            _acc(compare(w, run_gpu(h, w, debug=debug), check_debug=debug))
        w1 = W.Workload(w.name, w.dtype, w.logits, None, w.x, w.u, w.T)
        _acc(compare(w1, run_gpu(h, w1)))
        wm = W.make_random(name="small-masked", B=B, k=k, V=V, dtype=dtype, seed=V + 5, logit_sigma=2.0,
                           draft_sigma=0.8, temperature=1.1)
        mask = np.random.default_rng(V).random((B, k + 1, V)) < 0.3
        wm.logits[mask] = W.f32_to_bf16_bits(np.array([-np.inf], np.float32))[0] if dtype == "bf16" else -np.inf
        _acc(compare(wm, run_gpu(h, wm, debug=True), check_debug=True))
    # rows starting one element past an aligned address: unaligned heads and tails
    w = W.make_random(name="small-unaligned", B=4, k=3, V=1500, dtype="bf16", seed=8, logit_sigma=3.0,
                      draft_sigma=1.0, temperature=1.0)
    L, q, x, u, T = to_device(w, "cuda:0")
    Lb = torch.empty(L.numel() + 1, dtype=L.dtype, device="cuda:0")
    Lb[1:].copy_(L.reshape(-1))
    out = sv.specv_verify_sample(h, Lb[1:].view(L.shape), q, x, u, T)
    torch.cuda.synchronize()
    _acc(compare(w, {kk: v.cpu().numpy() for kk, v in out.items()}))
