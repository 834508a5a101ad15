"""GPU parity of the paged KV-cache rollback with the oracle (integer work:
bit-exact).  "LLM Inference & Speculative Decoding: From Roofline Physics to
Lossless Acceleration", s.1, PagedKVCacheManager.rollback_to."""
import numpy as np
import pytest

import oracle
from test_oracle_rollback import _random_batch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def h():
    import speculative_decoding_verification_57_gb300 as sv

    handle = sv.specv_create(0, max_batch=4096, max_k=31, vocab=1000)
    yield handle
    sv.specv_destroy(handle)


def _gpu(h, na, k, lens, tables, nb, bs, free, fc):
    import torch

    import speculative_decoding_verification_57_gb300 as sv

    t = {name: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
         for name, a in (("na", na), ("lens", lens), ("tables", tables), ("nb", nb), ("free", free))}
    fcount = torch.tensor([fc], dtype=torch.int32, device="cuda")
    st = torch.empty(len(na), dtype=torch.int32, device="cuda")
    sv.specv_rollback(h, t["na"], k, t["lens"], t["tables"], t["nb"], bs, t["free"], fcount, row_status=st)
    torch.cuda.synchronize()
    return {"seq_lens": t["lens"].cpu().numpy(), "block_tables": t["tables"].cpu().numpy(),
            "num_blocks": t["nb"].cpu().numpy(), "free_list": t["free"].cpu().numpy(),
            "free_count": int(fcount.item()), "row_status": st.cpu().numpy()}


def _same(a, b):
    for key in ("seq_lens", "block_tables", "num_blocks", "free_list", "row_status"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    assert a["free_count"] == b["free_count"]


@pytest.mark.parametrize("B,k,bs,mb", [(1, 4, 4, 8), (37, 5, 16, 12), (1024, 8, 16, 20), (3000, 3, 1, 6),
                                       (2049, 31, 7, 40)])
def test_rollback_matches_oracle(h, B, k, bs, mb):
    rng = np.random.default_rng(B + k)
    na, lens, tables, nb = _random_batch(rng, B, k, bs, mb)
    na[::7] = k + 1  # some invalid rows
    cap = B * mb + 3
    free = np.full(cap, -5, np.int32)
    free[:3] = [100_001, 100_002, 100_003]
    ref = oracle.rollback(na, k, lens, tables, nb, bs, free, 3)
    got = _gpu(h, na, k, lens, tables, nb, bs, free, 3)
    _same(got, ref)


@pytest.mark.parametrize("B,k,bs,mb", [(4097, 6, 4, 10), (9000, 8, 2, 12)])
def test_rollback_large_batches(B, k, bs, mb):
    """Batches past 4096 rows (more than four rows a thread)."""
    import speculative_decoding_verification_57_gb300 as sv

    hl = sv.specv_create(0, max_batch=B, max_k=k, vocab=1000)
    try:
        rng = np.random.default_rng(B)
        na, lens, tables, nb = _random_batch(rng, B, k, bs, mb)
        na[::11] = -1  # some invalid rows
        cap = B * mb
        free = np.full(cap, -5, np.int32)
        ref = oracle.rollback(na, k, lens, tables, nb, bs, free, 0)
        got = _gpu(hl, na, k, lens, tables, nb, bs, free, 0)
        _same(got, ref)
    finally:
        sv.specv_destroy(hl)


def test_rollback_no_room(h):
    rng = np.random.default_rng(1)
    na, lens, tables, nb = _random_batch(rng, 64, 4, 2, 10)
    na[:] = 0
    free = np.zeros(3, np.int32)
    ref = oracle.rollback(na, 4, lens, tables, nb, 2, free, 1)
    got = _gpu(h, na, 4, lens, tables, nb, 2, free, 1)
    assert np.all(ref["row_status"] == 256)
    _same(got, ref)


def test_rollback_after_verify(h):
    """The verify call's num_accepted feeds the rollback directly on the device."""
    import torch

    import speculative_decoding_verification_57_gb300 as sv
    from speculative_decoding_verification_57_gb300 import workloads as W
    from parity import to_device

    w = W.make_workload("zipf")
    L, q, x, u, T = to_device(w, "cuda:0")
    hv = sv.specv_create(0, max_batch=w.B, max_k=w.k, vocab=w.V)
    out = sv.specv_verify_sample(hv, L, q, x, u, T)
    bs, mb = 16, 8
    lens = torch.full((w.B,), 40 + w.k, dtype=torch.int32, device="cuda")
    nb = ((lens + bs - 1) // bs).to(torch.int32)
    tables = torch.full((w.B, mb), -1, dtype=torch.int32, device="cuda")
    for b in range(w.B):
        tables[b, : int(nb[b])] = torch.arange(b * mb, b * mb + int(nb[b]), dtype=torch.int32)
    free = torch.zeros(w.B * mb, dtype=torch.int32, device="cuda")
    fc = torch.zeros(1, dtype=torch.int32, device="cuda")
    na_ref = out["num_accepted"].clone()
    sv.specv_rollback(hv, out["num_accepted"], w.k, lens, tables, nb, bs, free, fc)
    torch.cuda.synchronize()
    assert torch.equal(lens.cpu(), (40 + na_ref).cpu().to(torch.int32))
    sv.specv_destroy(hv)
