"""The parity checker's treatment of flagged rows (CPU): a GPU token whose
CDF slot meets [u - 1e-6, u + 1e-6] is accepted, one a whole slot further
is refused."""
import numpy as np
import pytest

import oracle
from parity import compare
from speculative_decoding_verification_57_gb300 import workloads as W


def _plain(w):
    return lambda sl, u: oracle.verify(w.logits[sl], w.q[sl], w.x[sl], u, w.T[sl])


def _warped(w, top_k=20, top_p=0.9):
    tk = np.full(w.B, top_k, np.int32)
    tp = np.full(w.B, top_p, np.float32)
    return lambda sl, u: oracle.verify_warped(w.logits[sl], w.q[sl], w.x[sl], u, w.T[sl], tk[sl], tp[sl])


def _edge_row(rows_of=_plain):
    """The toy workload with row 0's draw uniform moved onto a CDF edge of
    its stop position (found by bisection on the oracle ``rows_of(w)``)."""
    w = W.make_workload("toy")
    run = rows_of(w)
    ref = run(slice(None), w.u)
    j = int(ref["num_accepted"][0])
    lo, hi = np.float32(0.0), np.float32(0.999)
    u = w.u.copy()

    def tok(v):
        u[0, j, 1] = v
        return int(run(slice(None), u)["out_tokens"][0][j])

    t_lo = tok(lo)
    for _ in range(60):  # narrow to two adjacent float32 values on either side of an edge
        mid = np.float32((np.float64(lo) + np.float64(hi)) / 2)
        if mid <= lo or mid >= hi:
            break
        if tok(mid) == t_lo:
            lo = mid
        else:
            hi = mid
    a, b = tok(lo), tok(hi)
    u[0, j, 1] = lo  # the row sits at the edge, on a's side
    return W.Workload(w.name, w.dtype, w.logits, w.q, w.x, u, w.T), j, a, b


def test_flagged_draw_across_the_edge_is_accepted():
    w, j, a, b = _edge_row()
    ref = oracle.verify(w.logits, w.q, w.x, w.u, w.T)
    assert ref["boundary"][0] != 0 and a != b
    got = {kk: np.array(v, copy=True) for kk, v in ref.items()}
    got["out_tokens"][0][j] = b  # the other side of the edge
    st = compare(w, got, ref=ref)
    assert st["mismatched"] == 1


def test_flagged_draw_far_from_the_edge_is_refused():
    w, j, a, b = _edge_row()
    ref = oracle.verify(w.logits, w.q, w.x, w.u, w.T)
    got = {kk: np.array(v, copy=True) for kk, v in ref.items()}
    got["out_tokens"][0][j] = b + 1 if b + 1 < w.V else a - 1  # a whole slot further
    with pytest.raises(AssertionError):
        compare(w, got, ref=ref)


@pytest.mark.parametrize("accept", [True, False])
def test_filtered_rule_uses_the_same_edge_rule(accept):
    """The top-k / top-p checker goes through the same rule: across the edge
    is accepted, a whole slot of the kept set further is refused."""
    w, j, a, b = _edge_row(_warped)
    run = _warped(w)
    ref = run(slice(None), w.u)
    assert ref["boundary"][0] != 0 and a != b
    got = {kk: np.array(v, copy=True) for kk, v in ref.items()}
    if accept:
        got["out_tokens"][0][j] = b
        assert compare(w, got, ref=ref, oracle_rows=run)["mismatched"] == 1
    else:
        # the next token of the kept set beyond b (the draw only lands on kept entries)
        far = [t for t in range(w.V) if t != a and t != b]
        got["out_tokens"][0][j] = far[0] if far[0] > max(a, b) or far[0] < min(a, b) else far[-1]
        with pytest.raises(AssertionError):
            compare(w, got, ref=ref, oracle_rows=run)
