"""Pins of the oracle's greedy tree verification ("LLM Inference &
Speculative Decoding: From Roofline Physics to Lossless Acceleration", s.3
"Multi-Draft Tree Speculation"; "Speculative Decoding: Mathematical
Foundations, ...", "SpecInfer and Tree-Based Verification")."""
import numpy as np

import oracle
from speculative_decoding_verification_57_gb300 import workloads as W

PAGE_PARENTS = [-1, 0, 0, 1, 1, 2]   # the page's tree, node depths 0,1,1,2,2,2
PAGE_DEPTHS = [0, 1, 1, 2, 2, 2]


def _logits_with_argmax(rng, amax, V):
    """Rows of random logits whose argmax is amax[r] (a clear winner)."""
    L = rng.normal(size=(len(amax), V)).astype(np.float32)
    for r, a in enumerate(amax):
        L[r, a] = L[r].max() + 1.0
    return L


def test_page_tree_path_and_depths():
    """The page's six-node tree: node depths as printed; a path through
    nodes 0 -> 2 -> 5 is kept and the bonus is the argmax after node 5."""
    rng = np.random.default_rng(1)
    V = 50
    tok = np.array([10, 11, 12, 13, 14, 15], np.int32)
    # row 0 (prefix) picks node 0's token, node 0's row picks node 2, node 2's row picks node 5, node 5's row -> 42
    amax = [10, 12, 7, 15, 8, 9, 42]
    L = _logits_with_argmax(rng, amax, V)[None]
    r = oracle.tree_greedy(L, tok[None], np.array([PAGE_PARENTS], np.int32))
    assert r["row_status"][0] == 0
    assert r["num_accepted"][0] == 3 == PAGE_DEPTHS[5] + 1
    assert r["path"][0, :3].tolist() == [0, 2, 5]
    assert r["out_tokens"][0].tolist() == [10, 12, 15, 42, -1, -1, -1]
    # depths through acceptance: accept only node k's ancestors path each time
    for node, d in enumerate(PAGE_DEPTHS):
        chain = []
        i = node
        while i >= 0:
            chain.append(i)
            i = PAGE_PARENTS[i]
        chain = chain[::-1]
        am = [0] * 7
        am[0] = int(tok[chain[0]])
        for a, c in zip(chain[:-1], chain[1:]):
            am[a + 1] = int(tok[c])
        am[node + 1] = 3
        r = oracle.tree_greedy(_logits_with_argmax(rng, am, V)[None], tok[None], np.array([PAGE_PARENTS], np.int32))
        assert r["num_accepted"][0] == d + 1, (node, r)


def test_chain_tree_is_greedy_chain():
    """parent[i] = i - 1 is the chain: the same outputs as the greedy rule."""
    w = W.make_random(name="chain", B=200, k=6, V=40, dtype="bf16", seed=4, logit_sigma=1.0, draft_sigma=0.3,
                      temperature=1.0)
    L = w.logits
    A = np.argmax(W.bf16_bits_to_f32(L), axis=-1)
    x = A[:, :6].astype(np.int32).copy()
    rng = np.random.default_rng(5)
    flip = rng.random(x.shape) < 0.2
    x[flip] = (x[flip] + 1) % 40
    chain = oracle.verify(L, None, x, None, None)
    par = np.tile(np.arange(-1, 5, dtype=np.int32), (200, 1))
    tree = oracle.tree_greedy(L, x, par)
    np.testing.assert_array_equal(tree["num_accepted"], chain["num_accepted"])
    np.testing.assert_array_equal(tree["out_tokens"], chain["out_tokens"])
    np.testing.assert_array_equal(tree["row_status"], chain["row_status"])


def _brute(L, tok, par):
    """Every node's whole path checked directly; deepest, then lowest index."""
    M = len(tok)
    A = [int(np.argmax(L[r])) for r in range(M + 1)]
    best, best_d = -1, -1
    for i in range(M):
        path = []
        n = i
        while n >= 0:
            path.append(n)
            n = par[n]
        path = path[::-1]
        ok = all(tok[c] == A[(par[c] + 1)] for c in path)
        if ok and len(path) - 1 > best_d:
            best, best_d = i, len(path) - 1
    if best < 0:
        return 0, [A[0]], []
    path = []
    n = best
    while n >= 0:
        path.append(n)
        n = par[n]
    path = path[::-1]
    return len(path), [int(tok[c]) for c in path] + [A[best + 1]], path


def test_random_trees_brute_force():
    rng = np.random.default_rng(6)
    B, M, V = 300, 12, 5  # small V: many matches and ties
    L = rng.integers(-2, 3, size=(B, M + 1, V)).astype(np.float32)
    par = np.array([[int(rng.integers(-1, i)) for i in range(M)] for _ in range(B)], np.int32)
    tok = rng.integers(0, V, size=(B, M)).astype(np.int32)
    r = oracle.tree_greedy(L, tok, par)
    for b in range(B):
        n, toks, path = _brute(L[b], tok[b], par[b])
        assert r["num_accepted"][b] == n
        assert r["out_tokens"][b, : n + 1].tolist() == toks
        assert r["path"][b, :n].tolist() == path
        assert np.all(r["out_tokens"][b, n + 1:] == -1) and np.all(r["path"][b, n:] == -1)


def test_tree_errors():
    L = np.zeros((3, 4, 6), np.float32)
    tok = np.array([[1, 2, 3], [1, 9, 3], [1, 2, 3]], np.int32)
    par = np.array([[-1, 0, 2], [-1, 0, 1], [-1, 0, 1]], np.int32)  # row 0: parent not before the node
    L[2, 3, 4] = np.nan
    r = oracle.tree_greedy(L, tok, par)
    assert r["row_status"].tolist() == [512, 2, 1]
    assert np.all(r["num_accepted"] == 0) and np.all(r["out_tokens"] == -1)
