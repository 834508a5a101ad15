"""GPU parity of greedy tree verification with the oracle (integer results:
exact).  "LLM Inference & Speculative Decoding ...", s.3 "Multi-Draft Tree
Speculation"; "Speculative Decoding: Mathematical Foundations, ...",
"SpecInfer and Tree-Based Verification"."""
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


def _run(h, logits, tok, par):
    import torch

    import speculative_decoding_verification_57_gb300 as sv

    if logits.dtype == np.uint16:
        L = torch.from_numpy(logits.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        L = torch.from_numpy(logits).cuda()
    out = sv.specv_verify_tree_greedy(h, L, torch.from_numpy(tok).cuda(), torch.from_numpy(par).cuda())
    torch.cuda.synchronize()
    return {kk: v.cpu().numpy() for kk, v in out.items()}


def _tree_workload(rng, B, M, V, dtype, agree=0.7):
    """Random trees whose draft tokens often equal the parent's argmax."""
    L = rng.normal(scale=2.0, size=(B, M + 1, V)).astype(np.float32)
    par = np.array([[int(rng.integers(-1, i)) for i in range(M)] for _ in range(B)], np.int32)
    Lq = W.f32_to_bf16_bits(L) if dtype == "bf16" else L
    A = np.argmax(W.bf16_bits_to_f32(Lq) if dtype == "bf16" else Lq, axis=-1)
    tok = rng.integers(0, V, size=(B, M)).astype(np.int32)
    hit = rng.random((B, M)) < agree
    for b in range(B):
        for i in range(M):
            if hit[b, i]:
                tok[b, i] = A[b, par[b, i] + 1]
    return Lq, tok, par


@pytest.mark.parametrize("B,M,V,dtype", [(64, 6, 128256, "bf16"), (16, 31, 32000, "bf16"), (8, 12, 70001, "f32"),
                                         (200, 16, 900, "f32"), (33, 5, 2048, "bf16"), (4, 1, 5000, "bf16")])
def test_tree_matches_oracle(h, B, M, V, dtype):
    rng = np.random.default_rng(B * 131 + M)
    L, tok, par = _tree_workload(rng, B, M, V, dtype)
    ref = oracle.tree_greedy(L, tok, par)
    got = _run(h, L, tok, par)
    for key in ("num_accepted", "out_tokens", "path", "row_status"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    assert ref["num_accepted"].max() >= min(2, M)


def test_tree_chain_equals_greedy_entry(h):
    """parent i-1 on the GPU gives what specv_verify_greedy gives."""
    import torch

    import speculative_decoding_verification_57_gb300 as sv

    rng = np.random.default_rng(3)
    B, M, V = 40, 7, 50000
    L = W.f32_to_bf16_bits(rng.normal(size=(B, M + 1, V)).astype(np.float32))
    A = np.argmax(W.bf16_bits_to_f32(L), axis=-1)
    tok = A[:, :M].astype(np.int32).copy()
    tok[rng.random(tok.shape) < 0.15] = 7
    par = np.tile(np.arange(-1, M - 1, dtype=np.int32), (B, 1))
    got = _run(h, L, tok, par)
    Lt = torch.from_numpy(L.view(np.int16)).cuda().view(torch.bfloat16)
    chain = sv.specv_verify_greedy(h, Lt, torch.from_numpy(tok).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got["num_accepted"], chain["num_accepted"].cpu().numpy())
    np.testing.assert_array_equal(got["out_tokens"], chain["out_tokens"].cpu().numpy())


def test_tree_errors_on_gpu(h):
    rng = np.random.default_rng(8)
    for V in (600, 9000):
        L, tok, par = _tree_workload(rng, 6, 5, V, "f32")
        par[0, 3] = 3          # not before the node
        tok[1, 2] = V          # out of range
        L[2, 4, 11] = np.nan   # a NaN row
        ref = oracle.tree_greedy(L, tok, par)
        got = _run(h, L, tok, par)
        assert ref["row_status"][:3].tolist() == [512, 2, 1]
        for key in ("num_accepted", "out_tokens", "path", "row_status"):
            np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
