"""Comparison of the CUDA path with the oracle on the same inputs.

Integer outputs (num_accepted, out_tokens, row_status) must be equal.  The
one exception is a row whose uniform lies within 1e-6 of a decision edge of
the oracle (its ``boundary`` flag): there the two precisions may land on
either side, so the GPU outcome must instead equal the oracle's outcome for
that uniform moved by at most 1e-6 (the accept test: nudged to either side
of the edge; the draw: between the oracle's tokens at u - 1e-6 and u + 1e-6,
the token being non-decreasing in the uniform).  Such disagreements are counted; intermediate values are
compared at 1e-5 relative.
"""
import numpy as np

import oracle

NUDGES = (1e-7, 3e-7, 1e-6, 3e-6)


def to_device(w, dev):
    import torch

    if w.dtype == "bf16":
        L = torch.from_numpy(w.logits.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        L = torch.from_numpy(w.logits).to(dev)
    q = None if w.q is None else torch.from_numpy(w.q).to(dev)  # None: one-hot drafts
    return (L, q, torch.from_numpy(w.x).to(dev), torch.from_numpy(w.u).to(dev), torch.from_numpy(w.T).to(dev))


def run_gpu(h, w, dev="cuda:0", debug=False):
    import torch

    import speculative_decoding_verification_57_gb300 as sv

    L, q, x, u, T = to_device(w, dev)
    out = sv.specv_verify_sample(h, L, q, x, u, T, debug=debug)
    torch.cuda.synchronize()
    return {key: v.cpu().numpy() for key, v in out.items()}


def _outcome(res, b):
    return (int(res["num_accepted"][b]), tuple(int(t) for t in res["out_tokens"][b]), int(res["row_status"][b]))


def plain_rows(w):
    """The oracle of the plain rule on rows ``sl`` of workload ``w`` with
    uniforms ``u`` for those rows."""
    def run(sl, u, debug=False):
        return oracle.verify(w.logits[sl], None if w.q is None else w.q[sl], w.x[sl], u, w.T[sl], debug=debug,
                             nthreads=8)
    return run


def compare(w, got, ref=None, *, check_debug=False, oracle_rows=None):
    """Assert parity of ``got`` (GPU outputs as numpy) with the oracle on
    workload ``w``; return counts {rows, flagged, mismatched}.
    ``oracle_rows(sl, u)`` evaluates the oracle on rows ``sl`` with uniforms
    ``u`` (default: the plain rule)."""
    if oracle_rows is None:
        oracle_rows = plain_rows(w)
        if ref is None:
            ref = oracle_rows(slice(None), w.u, debug=check_debug)
    elif ref is None:
        ref = oracle_rows(slice(None), w.u)
    B = w.B
    same = ((got["num_accepted"] == ref["num_accepted"]) & (got["row_status"] == ref["row_status"])
            & (got["out_tokens"] == ref["out_tokens"]).all(1))
    flagged = ref["boundary"] != 0
    bad = np.nonzero(~same & ~flagged)[0]
    assert len(bad) == 0, (
        f"{len(bad)} unflagged rows differ, first {bad[:5]}: gpu "
        f"{[_outcome(got, b) for b in bad[:3]]} oracle {[_outcome(ref, b) for b in bad[:3]]}")
    mism = np.nonzero(~same & flagged)[0]
    for b in mism:
        idx = int(ref["boundary"][b]) - 1
        i, slot = idx // 2, idx % 2
        top = np.nextafter(np.float32(1), np.float32(0))

        def outcome_at(u_val):
            uu = w.u[b:b + 1].copy()
            uu[0, i, slot] = np.float32(np.clip(u_val, 0.0, top))
            return _outcome(oracle_rows(slice(b, b + 1), uu), 0)

        want = _outcome(got, b)
        have = _outcome(ref, b)
        u0 = float(w.u[b, i, slot])
        j = have[0]
        same_but_draw = (want[0] == j and want[2] == have[2]
                         and all(want[1][t] == have[1][t] for t in range(len(want[1])) if t != j))
        if slot == 1 and same_but_draw:
            # the draw: the token is non-decreasing in u, so the tokens whose CDF
            # slots meet [u - 1e-6, u + 1e-6] are those between the oracle's
            # tokens at the two ends (a slot may be too narrow for any float32 u)
            tok = want[1][j]
            t_lo = outcome_at(np.float32(max(0.0, u0 - 1e-6)))[1][j]
            t_hi = outcome_at(np.float32(min(float(top), u0 + 1e-6)))[1][j]
            assert t_lo <= tok <= t_hi, (b, want, have, (t_lo, t_hi), "the GPU's token is not within 1e-6")
        else:
            # the accept test: two outcomes, either side of the edge
            alts = {outcome_at(u0 + sgn * d) for d in NUDGES for sgn in (-1.0, 1.0)}
            assert want in alts, (b, want, alts)
    if check_debug:
        ok = same & ((ref["row_status"] & oracle.ST_ERROR_MASK) == 0)
        greedy = w.T == 0
        np.testing.assert_array_equal(got["row_max"][ok], ref["row_max"][ok].astype(np.float32))
        smp = ok & ~greedy
        np.testing.assert_allclose(got["row_sumexp"][smp], ref["row_sumexp"][smp], rtol=1e-5)
        xok = (w.x >= 0) & (w.x < w.V)
        m = smp[:, None] & xok
        np.testing.assert_allclose(got["p_at_draft"][m], ref["p_at_draft"][m], rtol=1e-5, atol=1e-30)
        np.testing.assert_array_equal(got["q_at_draft"][m], ref["q_at_draft"][m].astype(np.float32))
        S = ref["residual_mass"][smp]
        G = got["residual_mass"][smp]
        off = np.abs(G - S) > 1e-5 * S + 1e-7
        assert not off.any(), ("residual_mass", np.nonzero(smp)[0][off][:8], G[off][:8], S[off][:8])
    return {"rows": B, "flagged": int(flagged.sum()), "mismatched": int(len(mism))}
