"""Argument errors of the C ABI on a live handle: every bad size, null
pointer or unknown dtype is refused with SPECV_ERR_INVALID_ARGUMENT before
anything is launched (the handle's launch count does not move), and an
empty batch is a no-op."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

OK, BAD = 0, 1


@pytest.fixture(scope="module")
def env():
    import torch

    import speculative_decoding_verification_57_gb300 as sv
    from speculative_decoding_verification_57_gb300 import _lib

    B, k, V = 4, 3, 5000
    h = sv.specv_create(0, max_batch=B, max_k=k, vocab=V)
    dev = torch.device("cuda:0")
    t = dict(
        L=torch.zeros((B, k + 1, V), dtype=torch.bfloat16, device=dev),
        q=torch.full((B, k, V), 1.0 / V, dtype=torch.float32, device=dev),
        x=torch.zeros((B, k), dtype=torch.int32, device=dev),
        u=torch.full((B, k + 1, 2), 0.5, dtype=torch.float32, device=dev),
        T=torch.ones(B, dtype=torch.float32, device=dev),
        na=torch.empty(B, dtype=torch.int32, device=dev),
        ot=torch.empty((B, k + 1), dtype=torch.int32, device=dev),
        rs=torch.empty(B, dtype=torch.int32, device=dev),
        par=torch.full((B, k), -1, dtype=torch.int32, device=dev),
        tk=torch.full((B,), 10, dtype=torch.int32, device=dev),
        tp=torch.ones(B, dtype=torch.float32, device=dev),
    )
    p = {kk: ctypes.c_void_p(v.data_ptr()) for kk, v in t.items()}
    yield sv, _lib.load(), h, B, k, V, p, t
    sv.specv_destroy(h)


def _sample(lib, h, p, *, dt=1, B=None, k=None, V=None, drop=(), base=(4, 3, 5000)):
    B = base[0] if B is None else B
    k = base[1] if k is None else k
    V = base[2] if V is None else V
    g = {kk: (None if kk in drop else v) for kk, v in p.items()}
    return lib.specv_verify_sample(h.ptr, dt, g["L"], g["q"], g["x"], g["u"], g["T"], B, k, V, g["na"], g["ot"],
                                   g["rs"], None, None)


def test_live_handle_refuses_bad_arguments_without_launching(env):
    import torch

    sv, lib, h, B, k, V, p, t = env
    assert _sample(lib, h, p) == OK  # the reference call is fine
    torch.cuda.synchronize()
    n0 = sv.specv_launch_count(h)
    cases = {
        "batch above max_batch": dict(B=B + 1),
        "negative batch": dict(B=-1),
        "k above max_k": dict(k=k + 1),
        "k zero": dict(k=0),
        "V above vocab": dict(V=V + 1),
        "V zero": dict(V=0),
        "unknown dtype": dict(dt=7),
        "null target_logits": dict(drop=("L",)),
        "null draft_tokens": dict(drop=("x",)),
        "null uniforms": dict(drop=("u",)),
        "null temperature": dict(drop=("T",)),
        "null num_accepted": dict(drop=("na",)),
        "null out_tokens": dict(drop=("ot",)),
    }
    for name, kw in cases.items():
        assert _sample(lib, h, p, **kw) == BAD, name
    # the greedy, tree and filtered entries check the same way
    assert lib.specv_verify_greedy(h.ptr, 1, None, p["x"], B, k, V, p["na"], p["ot"], p["rs"], None) == BAD
    assert lib.specv_verify_greedy(h.ptr, 1, p["L"], p["x"], B + 1, k, V, p["na"], p["ot"], p["rs"], None) == BAD
    assert lib.specv_verify_greedy(h.ptr, 3, p["L"], p["x"], B, k, V, p["na"], p["ot"], p["rs"], None) == BAD
    assert lib.specv_verify_tree_greedy(h.ptr, 1, p["L"], p["x"], None, B, k, V, p["na"], p["ot"], None, p["rs"],
                                        None) == BAD
    assert lib.specv_verify_tree_greedy(h.ptr, 1, p["L"], p["x"], p["par"], B, k + 1, V, p["na"], p["ot"], None,
                                        p["rs"], None) == BAD
    assert lib.specv_verify_sample_filtered(h.ptr, 1, p["L"], p["q"], p["x"], p["u"], p["T"], None, p["tp"], B, k, V,
                                            p["na"], p["ot"], p["rs"], None) == BAD
    assert lib.specv_verify_sample_filtered(h.ptr, 1, p["L"], p["q"], p["x"], p["u"], p["T"], p["tk"], p["tp"], B, k,
                                            V + 1, p["na"], p["ot"], p["rs"], None) == BAD
    assert lib.specv_test_withhold_stage(h.ptr, -1, 100) == BAD
    assert lib.specv_test_withhold_stage(h.ptr, 0, 0) == BAD
    torch.cuda.synchronize()
    assert sv.specv_launch_count(h) == n0


def test_empty_batch_is_a_no_op(env):
    import torch

    sv, lib, h, B, k, V, p, t = env
    t["na"].fill_(-5)
    torch.cuda.synchronize()
    n0 = sv.specv_launch_count(h)
    assert _sample(lib, h, p, B=0) == OK
    assert lib.specv_verify_greedy(h.ptr, 1, p["L"], p["x"], 0, k, V, p["na"], p["ot"], p["rs"], None) == OK
    torch.cuda.synchronize()
    assert sv.specv_launch_count(h) == n0
    assert np.all(t["na"].cpu().numpy() == -5)  # nothing written
