"""Batched speculative-decoding verify step on GB300 (sm_103a).

Python binding of the C ABI in ``include/specv.h``: the functions below keep
the C names and only marshal arguments (torch tensors for device memory and
the current CUDA stream); every step of the verify path runs in the
library's CUDA kernels.  There is no CPU fallback: if ``libspecv.so`` cannot
be loaded, or no sm_103 device is present, the calls raise.
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import (ST_ERROR_MASK, ST_NONFINITE, ST_Q_INVALID, ST_TEMPERATURE, ST_TIMEOUT, ST_TOKEN_RANGE,
                   ST_UNIFORM_RANGE, ST_ZERO_RESIDUAL, SPECV_BF16, SPECV_F32)

__all__ = [
    "SpecvError",
    "Handle",
    "specv_create",
    "specv_destroy",
    "specv_verify_sample",
    "specv_verify_greedy",
    "specv_verify_sample_host",
    "specv_plan_cluster",
    "specv_test_withhold_stage",
    "specv_launch_count",
    "ST_ERROR_MASK",
    "ST_NONFINITE",
    "ST_TOKEN_RANGE",
    "ST_UNIFORM_RANGE",
    "ST_TEMPERATURE",
    "ST_ZERO_RESIDUAL",
    "ST_Q_INVALID",
    "ST_TIMEOUT",
]


class SpecvError(RuntimeError):
    def __init__(self, status, what=""):
        lib = _lib.load()
        msg = lib.specv_status_string(status).decode()
        if status == _lib.SPECV_ERR_CUDA or status == _lib.SPECV_ERR_UNSUPPORTED:
            msg += ": " + lib.specv_last_cuda_error().decode()
        super().__init__(f"{what}: {msg}" if what else msg)
        self.status = status


def _check(status, what):
    if status != _lib.SPECV_OK:
        raise SpecvError(status, what)


class Handle:
    """An open ``specv_handle`` (closed by ``specv_destroy`` or on garbage
    collection)."""

    def __init__(self, ptr, device, max_batch, max_k, vocab):
        self.ptr = ptr
        self.device = device
        self.max_batch = max_batch
        self.max_k = max_k
        self.vocab = vocab

    def __del__(self):
        try:
            specv_destroy(self)
        except Exception:
            pass


def specv_create(device=0, max_batch=1 << 20, max_k=31, vocab=262144) -> Handle:
    lib = _lib.load()
    h = ctypes.c_void_p()
    _check(lib.specv_create(ctypes.byref(h), int(device), int(max_batch), int(max_k), int(vocab)), "specv_create")
    return Handle(h.value, device, max_batch, max_k, vocab)


def specv_destroy(h: Handle) -> None:
    if h is not None and h.ptr:
        _lib.load().specv_destroy(h.ptr)
        h.ptr = None


def _torch():
    import torch

    return torch


def _dev(t, dtype, name, shape=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t.data_ptr()


def _logits_dtype(logits):
    torch = _torch()
    if logits.dtype == torch.bfloat16:
        return SPECV_BF16
    if logits.dtype == torch.float32:
        return SPECV_F32
    raise TypeError("target logits must be bfloat16 or float32")


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def specv_verify_sample(h: Handle, logits, q, x, u, T, *, debug=False, out=None, stream=None):
    """Verify a batch (asynchronous on ``stream``, default: torch's current
    stream).  logits [B,k+1,V] bf16/fp32, q [B,k,V] fp32 or None (one-hot
    drafts: q is the point mass at each draft token), x [B,k] int32,
    u [B,k+1,2] fp32, T [B] fp32 (0 = greedy row), all CUDA tensors.
    Returns a dict of CUDA tensors: num_accepted [B], out_tokens [B,k+1],
    row_status [B] and, with ``debug``, p_at_draft, q_at_draft, row_max,
    row_sumexp, residual_mass.  ``out`` may supply preallocated outputs."""
    torch = _torch()
    B, k1, V = logits.shape
    k = k1 - 1
    dt = _logits_dtype(logits)
    _dev(logits, logits.dtype, "logits")
    pq = None if q is None else _dev(q, torch.float32, "q", (B, k, V))
    px = _dev(x, torch.int32, "x", (B, k))
    pu = _dev(u, torch.float32, "u", (B, k + 1, 2))
    pt = _dev(T, torch.float32, "T", (B,))
    dev = logits.device
    if out is None:
        out = {
            "num_accepted": torch.empty(B, dtype=torch.int32, device=dev),
            "out_tokens": torch.empty((B, k + 1), dtype=torch.int32, device=dev),
            "row_status": torch.empty(B, dtype=torch.int32, device=dev),
        }
    dbg_struct = None
    if debug:
        for name, shape in (("p_at_draft", (B, k)), ("q_at_draft", (B, k)), ("row_max", (B, k + 1)),
                            ("row_sumexp", (B, k + 1)), ("residual_mass", (B,))):
            if name not in out:
                out[name] = torch.empty(shape, dtype=torch.float32, device=dev)
        dbg_struct = _lib.SpecvDebug(out["p_at_draft"].data_ptr(), out["q_at_draft"].data_ptr(),
                                     out["row_max"].data_ptr(), out["row_sumexp"].data_ptr(),
                                     out["residual_mass"].data_ptr())
    lib = _lib.load()
    st = lib.specv_verify_sample(
        h.ptr, dt, ctypes.c_void_p(logits.data_ptr()), ctypes.c_void_p(pq), ctypes.c_void_p(px),
        ctypes.c_void_p(pu), ctypes.c_void_p(pt), B, k, V, ctypes.c_void_p(out["num_accepted"].data_ptr()),
        ctypes.c_void_p(out["out_tokens"].data_ptr()), ctypes.c_void_p(out["row_status"].data_ptr()),
        ctypes.byref(dbg_struct) if dbg_struct is not None else None, _stream_ptr(stream))
    _check(st, "specv_verify_sample")
    return out


def specv_verify_greedy(h: Handle, logits, x, *, out=None, stream=None):
    """Greedy verification of every row: logits [B,k+1,V], x [B,k] int32."""
    torch = _torch()
    B, k1, V = logits.shape
    k = k1 - 1
    dt = _logits_dtype(logits)
    _dev(logits, logits.dtype, "logits")
    px = _dev(x, torch.int32, "x", (B, k))
    dev = logits.device
    if out is None:
        out = {
            "num_accepted": torch.empty(B, dtype=torch.int32, device=dev),
            "out_tokens": torch.empty((B, k + 1), dtype=torch.int32, device=dev),
            "row_status": torch.empty(B, dtype=torch.int32, device=dev),
        }
    st = _lib.load().specv_verify_greedy(
        h.ptr, dt, ctypes.c_void_p(logits.data_ptr()), ctypes.c_void_p(px), B, k, V,
        ctypes.c_void_p(out["num_accepted"].data_ptr()), ctypes.c_void_p(out["out_tokens"].data_ptr()),
        ctypes.c_void_p(out["row_status"].data_ptr()), _stream_ptr(stream))
    _check(st, "specv_verify_greedy")
    return out


def specv_verify_sample_filtered(h: Handle, logits, q, x, u, T, top_k, top_p, *, out=None, stream=None):
    """Sampled verification with top-k / top-p applied to the target rows:
    as specv_verify_sample (q may be None: one-hot drafts, or a pinned CPU
    tensor, read in place), plus top_k [B] int32 in 1..4096 and top_p [B]
    fp32 in (0, 1], CUDA tensors."""
    torch = _torch()
    B, k1, V = logits.shape
    k = k1 - 1
    dt = _logits_dtype(logits)
    _dev(logits, logits.dtype, "logits")
    if q is not None and not q.is_cuda:
        if not q.is_pinned() or q.dtype != torch.float32 or not q.is_contiguous() or tuple(q.shape) != (B, k, V):
            raise ValueError("a CPU q must be a pinned, contiguous float32 tensor of shape [B, k, V]")
        pq = q.data_ptr()
    else:
        pq = None if q is None else _dev(q, torch.float32, "q", (B, k, V))
    px = _dev(x, torch.int32, "x", (B, k))
    pu = _dev(u, torch.float32, "u", (B, k + 1, 2))
    pt = _dev(T, torch.float32, "T", (B,))
    pk = _dev(top_k, torch.int32, "top_k", (B,))
    pp = _dev(top_p, torch.float32, "top_p", (B,))
    dev = logits.device
    if out is None:
        out = {
            "num_accepted": torch.empty(B, dtype=torch.int32, device=dev),
            "out_tokens": torch.empty((B, k + 1), dtype=torch.int32, device=dev),
            "row_status": torch.empty(B, dtype=torch.int32, device=dev),
        }
    st = _lib.load().specv_verify_sample_filtered(
        h.ptr, dt, ctypes.c_void_p(logits.data_ptr()), ctypes.c_void_p(pq), ctypes.c_void_p(px), ctypes.c_void_p(pu),
        ctypes.c_void_p(pt), ctypes.c_void_p(pk), ctypes.c_void_p(pp), B, k, V,
        ctypes.c_void_p(out["num_accepted"].data_ptr()), ctypes.c_void_p(out["out_tokens"].data_ptr()),
        ctypes.c_void_p(out["row_status"].data_ptr()), _stream_ptr(stream))
    _check(st, "specv_verify_sample_filtered")
    return out


def specv_verify_tree_greedy(h: Handle, logits, tokens, parents, *, out=None, stream=None):
    """Greedy verification of draft trees: logits [B, M+1, V] (row 0 after
    the prefix, row 1+i after node i), tokens and parents [B, M] int32
    (parent -1: a child of the prefix).  Returns num_accepted [B],
    out_tokens [B, M+1], path [B, M], row_status [B]."""
    torch = _torch()
    B, m1, V = logits.shape
    M = m1 - 1
    dt = _logits_dtype(logits)
    _dev(logits, logits.dtype, "logits")
    pt = _dev(tokens, torch.int32, "tokens", (B, M))
    pp = _dev(parents, torch.int32, "parents", (B, M))
    dev = logits.device
    if out is None:
        out = {
            "num_accepted": torch.empty(B, dtype=torch.int32, device=dev),
            "out_tokens": torch.empty((B, M + 1), dtype=torch.int32, device=dev),
            "path": torch.empty((B, M), dtype=torch.int32, device=dev),
            "row_status": torch.empty(B, dtype=torch.int32, device=dev),
        }
    st = _lib.load().specv_verify_tree_greedy(
        h.ptr, dt, ctypes.c_void_p(logits.data_ptr()), ctypes.c_void_p(pt), ctypes.c_void_p(pp), B, M, V,
        ctypes.c_void_p(out["num_accepted"].data_ptr()), ctypes.c_void_p(out["out_tokens"].data_ptr()),
        ctypes.c_void_p(out["path"].data_ptr()), ctypes.c_void_p(out["row_status"].data_ptr()), _stream_ptr(stream))
    _check(st, "specv_verify_tree_greedy")
    return out


def specv_verify_sample_host(h: Handle, logits, q, x, u, T, *, out=None, stream=None):
    """Host-buffer verification: CPU tensors in (pinned memory copies
    fastest), CPU tensors out; the call copies, verifies and synchronises.
    ``logits`` is a bfloat16 or float32 CPU tensor."""
    torch = _torch()
    B, k1, V = logits.shape
    k = k1 - 1
    dt = _logits_dtype(logits)
    for t, name in ((logits, "logits"), (q, "q"), (x, "x"), (u, "u"), (T, "T")):
        if t is None and name == "q":
            continue  # one-hot drafts
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    if out is None:
        pin = logits.is_pinned()
        out = {
            "num_accepted": torch.empty(B, dtype=torch.int32, pin_memory=pin),
            "out_tokens": torch.empty((B, k + 1), dtype=torch.int32, pin_memory=pin),
            "row_status": torch.empty(B, dtype=torch.int32, pin_memory=pin),
        }
    st = _lib.load().specv_verify_sample_host(
        h.ptr, dt, ctypes.c_void_p(logits.data_ptr()), ctypes.c_void_p(None if q is None else q.data_ptr()),
        ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(u.data_ptr()), ctypes.c_void_p(T.data_ptr()), B, k, V,
        ctypes.c_void_p(out["num_accepted"].data_ptr()), ctypes.c_void_p(out["out_tokens"].data_ptr()),
        ctypes.c_void_p(out["row_status"].data_ptr()), _stream_ptr(stream))
    _check(st, "specv_verify_sample_host")
    return out


def specv_rollback(h: Handle, num_accepted, k, seq_lens, block_tables, num_blocks, block_size, free_list,
                   free_count, *, row_status=None, stream=None):
    """Paged KV-cache rollback after verification, in place on CUDA int32
    tensors: num_accepted [B], seq_lens [B], block_tables [B, max_blocks],
    num_blocks [B], free_list [capacity], free_count [1]; row_status [B]
    (optional) receives 0 / 128 (invalid row) / 256 (no room)."""
    torch = _torch()
    B = num_accepted.shape[0]
    mb = block_tables.shape[1] if block_tables.dim() == 2 else 0
    ptrs = []
    for t, name, shape in ((num_accepted, "num_accepted", (B,)), (seq_lens, "seq_lens", (B,)),
                           (block_tables, "block_tables", (B, mb)), (num_blocks, "num_blocks", (B,)),
                           (free_list, "free_list", None), (free_count, "free_count", (1,))):
        ptrs.append(_dev(t, torch.int32, name, shape))
    prs = None if row_status is None else _dev(row_status, torch.int32, "row_status", (B,))
    st = _lib.load().specv_rollback(
        h.ptr, ctypes.c_void_p(ptrs[0]), B, int(k), ctypes.c_void_p(ptrs[1]), ctypes.c_void_p(ptrs[2]), mb,
        ctypes.c_void_p(ptrs[3]), int(block_size), ctypes.c_void_p(ptrs[4]), free_list.numel(),
        ctypes.c_void_p(ptrs[5]), ctypes.c_void_p(prs), _stream_ptr(stream))
    _check(st, "specv_rollback")


def specv_plan_cluster(h: Handle, logits_dtype, B, k, V) -> int:
    return int(_lib.load().specv_plan_cluster(h.ptr, logits_dtype, B, k, V))


def specv_test_withhold_stage(h: Handle, stage_use: int, polls: int) -> None:
    """Test hook: the next split-vocabulary launch on ``h`` never fills
    pass-1 stage use ``stage_use`` of CTA 0 and its waits give up after
    ``polls`` polls (see include/specv.h)."""
    _check(_lib.load().specv_test_withhold_stage(h.ptr, int(stage_use), int(polls)), "specv_test_withhold_stage")


def specv_launch_count(h: Handle) -> int:
    return int(_lib.load().specv_launch_count(h.ptr))
