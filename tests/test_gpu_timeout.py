"""Bounded waits of the split-vocabulary kernel, exercised without a fault:
a test hook (specv_test_withhold_stage) withholds one pass-1 stage of the
grid's first CTA, so that every wait on it runs out.  The call still returns
SPECV_OK; the first row reports row_status bit 64 with num_accepted 0 and
out_tokens -1; the other rows of the same call match the oracle; and the
next call on the same handle matches the oracle in full."""
import numpy as np
import pytest

from parity import compare, run_gpu
from speculative_decoding_verification_57_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _rows(w, sl):
    return W.Workload(w.name, w.dtype, w.logits[sl], None if w.q is None else w.q[sl], w.x[sl], w.u[sl], w.T[sl])


@pytest.mark.parametrize("debug", [False, True])
@pytest.mark.parametrize("stage", [0, 3])
def test_withheld_stage_times_out_then_next_call_is_clean(stage, debug):
    import speculative_decoding_verification_57_gb300 as sv

    # 200k bf16 entries a position: even at 16 CTAs a row, every CTA holds at
    # least three 8 KB stages of position 0, so stage uses 0 and 3 are issued
    w = W.make_random(name="timeout", B=4, k=3, V=200_000, dtype="bf16", seed=11 + stage, logit_sigma=3.0,
                      draft_sigma=1.0, temperature=1.0, spike=6.0, spike_mode="position")
    h = sv.specv_create(0, max_batch=w.B, max_k=w.k, vocab=w.V)
    try:
        n0 = sv.specv_launch_count(h)
        sv.specv_test_withhold_stage(h, stage, 200_000)
        got = run_gpu(h, w, debug=debug)  # raises unless the call returns SPECV_OK
        assert sv.specv_launch_count(h) == n0 + 1
        assert got["row_status"][0] & sv.ST_TIMEOUT, got["row_status"]
        assert got["num_accepted"][0] == 0
        assert (got["out_tokens"][0] == -1).all()
        rest = slice(1, w.B)
        compare(_rows(w, rest), {key: v[rest] for key, v in got.items()})
        again = run_gpu(h, w, debug=debug)
        assert not (again["row_status"] & sv.ST_TIMEOUT).any()
        compare(w, again, check_debug=debug)
    finally:
        sv.specv_destroy(h)
