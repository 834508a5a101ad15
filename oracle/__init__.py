"""Python handle on the float64 CPU oracle (``specv_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg call this module; the product path never does.  It compiles the
C file with gcc on first use (or when the source is newer than the shared
object) and marshals numpy arrays to it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specv_oracle.c")
_LIB = os.path.join(_HERE, "libspecv_oracle.so")
_lock = threading.Lock()
_lib = None

ST_NONFINITE = 1
ST_TOKEN_RANGE = 2
ST_UNIFORM_RANGE = 4
ST_TEMPERATURE = 8
ST_ZERO_RESIDUAL = 16
ST_Q_INVALID = 32
ST_FILTER = 1024
ST_ERROR_MASK = ST_NONFINITE | ST_TOKEN_RANGE | ST_UNIFORM_RANGE | ST_TEMPERATURE | ST_Q_INVALID | ST_FILTER


def compile_oracle(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile an oracle source file to a shared object with gcc."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", *extra_flags, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    vp = ctypes.c_void_p
    lib.specv_oracle_verify.restype = ctypes.c_int
    lib.specv_oracle_verify.argtypes = [
        ctypes.c_int, vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
        vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_double, ctypes.c_int,
    ]
    lib.specv_oracle_softmax_stats.restype = ctypes.c_int
    lib.specv_oracle_softmax_stats.argtypes = [ctypes.c_int, vp, ctypes.c_int64, ctypes.c_double, dp, dp, vp]
    lib.specv_oracle_argmax.restype = ctypes.c_int
    lib.specv_oracle_argmax.argtypes = [ctypes.c_int, vp, ctypes.c_int64,
                                        ctypes.POINTER(ctypes.c_int64), dp]
    lib.specv_oracle_residual.restype = ctypes.c_int
    lib.specv_oracle_residual.argtypes = [vp, vp, ctypes.c_int64, vp, dp]
    lib.specv_oracle_inverse_cdf.restype = ctypes.c_int64
    lib.specv_oracle_inverse_cdf.argtypes = [vp, ctypes.c_int64, ctypes.c_double, dp, dp]
    lib.specv_oracle_tree_greedy.restype = ctypes.c_int
    lib.specv_oracle_tree_greedy.argtypes = [ctypes.c_int, vp, vp, vp, ctypes.c_int64, ctypes.c_int, ctypes.c_int64,
                                             vp, vp, vp, vp]
    lib.specv_oracle_verify_warped.restype = ctypes.c_int
    lib.specv_oracle_verify_warped.argtypes = [ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int,
                                               ctypes.c_int64, vp, vp, vp, vp, ctypes.c_double]
    lib.specv_oracle_rollback.restype = ctypes.c_int
    lib.specv_oracle_rollback.argtypes = [vp, ctypes.c_int64, ctypes.c_int, vp, vp, ctypes.c_int, vp, ctypes.c_int,
                                          vp, ctypes.c_int64, vp, vp]
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  With ``path`` given,
    load that file instead (used for deliberately broken copies in tests)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
                compile_oracle()
            _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(logits: np.ndarray) -> int:
    if logits.dtype == np.uint16:
        return 1
    if logits.dtype == np.float32:
        return 0
    raise TypeError("logits must be float32 or uint16 (bf16 bits)")


def verify(logits, q, x, u, T, *, debug=False, boundary_eps=1e-6, nthreads=1, lib=None):
    """Run the oracle over a batch.

    logits [B,k+1,V] float32 or uint16 (bf16 bits); q [B,k,V] float32 or
    None (one-hot drafts: q is the point mass at each draft token); x [B,k]
    int32; u [B,k+1,2] float32 or None; T [B] float32 or None (None: every
    row greedy).  Returns a dict of numpy arrays:
    num_accepted, out_tokens, row_status, boundary (0 or 1 + 2*i + slot of
    the uniform found within ``boundary_eps`` of a decision edge) and, with
    ``debug``, p_at_draft, q_at_draft, row_max, row_sumexp, residual_mass.
    """
    lib = lib or load()
    logits = np.ascontiguousarray(logits)
    x = np.ascontiguousarray(x, dtype=np.int32)
    B, k1, V = logits.shape
    k = k1 - 1
    assert x.shape == (B, k)
    q = None if q is None else np.ascontiguousarray(q, dtype=np.float32)
    u = None if u is None else np.ascontiguousarray(u, dtype=np.float32)
    T = None if T is None else np.ascontiguousarray(T, dtype=np.float32)
    out = {
        "num_accepted": np.empty(B, np.int32),
        "out_tokens": np.empty((B, k + 1), np.int32),
        "row_status": np.empty(B, np.int32),
        "boundary": np.empty(B, np.int32),
    }
    dbg = {}
    if debug:
        dbg = {
            "p_at_draft": np.empty((B, k), np.float64),
            "q_at_draft": np.empty((B, k), np.float64),
            "row_max": np.empty((B, k + 1), np.float64),
            "row_sumexp": np.empty((B, k + 1), np.float64),
            "residual_mass": np.empty(B, np.float64),
        }
        out.update(dbg)
    rc = lib.specv_oracle_verify(
        _dtype_code(logits), _ptr(logits), _ptr(q), _ptr(x), _ptr(u), _ptr(T), B, k, V,
        _ptr(out["num_accepted"]), _ptr(out["out_tokens"]), _ptr(out["row_status"]),
        _ptr(dbg.get("p_at_draft")), _ptr(dbg.get("q_at_draft")), _ptr(dbg.get("row_max")),
        _ptr(dbg.get("row_sumexp")), _ptr(dbg.get("residual_mass")), _ptr(out["boundary"]),
        float(boundary_eps), int(nthreads),
    )
    if rc != 0:
        raise RuntimeError(f"oracle returned {rc}")
    return out


def softmax_stats(row, T, *, lib=None):
    """(status, M, s, e) for one position's logits ``row`` [V]."""
    lib = lib or load()
    row = np.ascontiguousarray(row)
    M, s = ctypes.c_double(), ctypes.c_double()
    e = np.empty(row.shape[0], np.float64)
    st = lib.specv_oracle_softmax_stats(_dtype_code(row), _ptr(row), row.shape[0], float(T),
                                        ctypes.byref(M), ctypes.byref(s), _ptr(e))
    return st, M.value, s.value, e


def argmax(row, *, lib=None):
    """(status, index, value) of the lowest-index maximum of ``row``."""
    lib = lib or load()
    row = np.ascontiguousarray(row)
    a, m = ctypes.c_int64(), ctypes.c_double()
    st = lib.specv_oracle_argmax(_dtype_code(row), _ptr(row), row.shape[0], ctypes.byref(a), ctypes.byref(m))
    return st, a.value, m.value


def residual(p, q, *, lib=None):
    """(status, r, S): r = max(0, p - q) and S = sum r, p float64, q float32."""
    lib = lib or load()
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float32)
    r = np.empty_like(p)
    S = ctypes.c_double()
    st = lib.specv_oracle_residual(_ptr(p), _ptr(q), p.shape[0], _ptr(r), ctypes.byref(S))
    return st, r, S.value


def inverse_cdf(w, u, *, lib=None):
    """(token, lo, hi) for non-negative weights ``w`` and uniform ``u``."""
    lib = lib or load()
    w = np.ascontiguousarray(w, dtype=np.float64)
    lo, hi = ctypes.c_double(), ctypes.c_double()
    t = lib.specv_oracle_inverse_cdf(_ptr(w), w.shape[0], float(u), ctypes.byref(lo), ctypes.byref(hi))
    return t, lo.value, hi.value


def rollback(num_accepted, k, seq_lens, block_tables, num_blocks, block_size, free_list, free_count, *, lib=None):
    """Paged KV rollback after verification, on copies of the inputs.
    num_accepted [B], seq_lens [B], block_tables [B, max_blocks],
    num_blocks [B] int32; free_list [capacity] int32 and free_count (int):
    the free list and its fill.  Returns a dict: seq_lens, block_tables,
    num_blocks, free_list, free_count, row_status."""
    lib = lib or load()
    na = np.ascontiguousarray(num_accepted, dtype=np.int32)
    sl = np.array(seq_lens, dtype=np.int32, copy=True)
    bt = np.array(block_tables, dtype=np.int32, copy=True)
    nb = np.array(num_blocks, dtype=np.int32, copy=True)
    fl = np.array(free_list, dtype=np.int32, copy=True)
    fc = np.array([free_count], dtype=np.int32)
    st = np.zeros(len(na), np.int32)
    B, mb = bt.shape
    rc = lib.specv_oracle_rollback(_ptr(na), B, int(k), _ptr(sl), _ptr(bt), mb, _ptr(nb), int(block_size),
                                   _ptr(fl), len(fl), _ptr(fc), _ptr(st))
    if rc != 0:
        raise ValueError(f"specv_oracle_rollback: bad arguments ({rc})")
    return {"seq_lens": sl, "block_tables": bt, "num_blocks": nb, "free_list": fl, "free_count": int(fc[0]),
            "row_status": st}


def tree_greedy(logits, tokens, parents, *, lib=None):
    """Greedy verification of draft trees.  logits [B, M+1, V] float32 or
    uint16 (bf16 bits): row 0 after the prefix, row 1+i after node i;
    tokens, parents [B, M] int32 (parent -1: child of the prefix).  Returns
    num_accepted [B], out_tokens [B, M+1], path [B, M], row_status [B]."""
    lib = lib or load()
    logits = np.ascontiguousarray(logits)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    parents = np.ascontiguousarray(parents, dtype=np.int32)
    B, m1, V = logits.shape
    M = m1 - 1
    out = {"num_accepted": np.empty(B, np.int32), "out_tokens": np.empty((B, M + 1), np.int32),
           "path": np.empty((B, M), np.int32), "row_status": np.empty(B, np.int32)}
    rc = lib.specv_oracle_tree_greedy(_dtype_code(logits), _ptr(logits), _ptr(tokens), _ptr(parents), B, M, V,
                                      _ptr(out["num_accepted"]), _ptr(out["out_tokens"]), _ptr(out["path"]),
                                      _ptr(out["row_status"]))
    if rc != 0:
        raise ValueError(f"specv_oracle_tree_greedy: bad arguments ({rc})")
    return out


def verify_warped(logits, q, x, u, T, top_k, top_p, *, boundary_eps=1e-6, lib=None):
    """Sampled verification with top-k / top-p applied to the target p
    (top_k [B] int32 in [1, 4096], top_p [B] float32 in (0, 1]; q None:
    one-hot drafts).  Returns num_accepted, out_tokens, row_status,
    boundary."""
    lib = lib or load()
    logits = np.ascontiguousarray(logits)
    x = np.ascontiguousarray(x, dtype=np.int32)
    B, k1, V = logits.shape
    q = None if q is None else np.ascontiguousarray(q, dtype=np.float32)
    u = np.ascontiguousarray(u, dtype=np.float32)
    T = np.ascontiguousarray(T, dtype=np.float32)
    tk = np.ascontiguousarray(top_k, dtype=np.int32)
    tp = np.ascontiguousarray(top_p, dtype=np.float32)
    out = {"num_accepted": np.empty(B, np.int32), "out_tokens": np.empty((B, k1), np.int32),
           "row_status": np.empty(B, np.int32), "boundary": np.empty(B, np.int32)}
    rc = lib.specv_oracle_verify_warped(_dtype_code(logits), _ptr(logits), _ptr(q), _ptr(x), _ptr(u), _ptr(T),
                                        _ptr(tk), _ptr(tp), B, k1 - 1, V, _ptr(out["num_accepted"]),
                                        _ptr(out["out_tokens"]), _ptr(out["row_status"]), _ptr(out["boundary"]),
                                        float(boundary_eps))
    if rc != 0:
        raise ValueError(f"specv_oracle_verify_warped: bad arguments ({rc})")
    return out
