"""Seeded synthetic inputs for the batched speculative-decoding verify step.

This module is the one piece shared by the oracle-side tests and the CUDA
side: it builds the arrays a verify call consumes and nothing else.  It holds
none of the verify step's arithmetic.  What it does compute stands in for the
models around the verify step:

* target logits: seeded normals (plus a spike) rounded to bf16 or fp32;
* the draft model's distribution q: a softmax of noisy logits, evaluated
  with numpy in float64 and rounded to fp32, exactly as a draft model would
  hand its probabilities over;
* draft tokens: drawn from that fp32 q (or its argmax, for a greedy draft)
  with their own uniforms, the draft model's sampling;
* the verify step's uniforms U[b, i, slot] in [0, 1) and per-row
  temperatures.

Every workload uses ``numpy.random.default_rng`` sub-streams spawned
from one ``SeedSequence``: one each for target logits, draft noise, draft
token uniforms and verify uniforms, so that changing one never shifts the
others.  Logit values are drawn in float64 and rounded to the stored type
(bf16 by round-to-nearest-even of the float32 value).

The five named workloads (``make_workload``) follow the shapes the verify
step is measured on: ``toy`` (V=1000 fp32), ``zipf`` (V=32000 bf16 with a
Zipf(1.1)-ranked boost), ``benchmark`` and ``mixed`` (the Llama-3 vocabulary,
128,256 entries, "Speculative decoding." lesson, "First: what an output
distribution is", at B=64, and at B=256 with half the rows greedy), and
``split_v`` (an fp32 V=151,936 case at small batch).
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "make_workload",
    "make_random",
    "make_from_distributions",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
]


@dataclasses.dataclass
class Workload:
    """One verify call's inputs, host-resident numpy arrays.

    logits: [B, k+1, V] float32, or uint16 holding bf16 bit patterns.
    q:      [B, k, V] float32 draft probabilities.
    x:      [B, k] int32 draft tokens.
    u:      [B, k+1, 2] float32 uniforms in [0, 1).
    T:      [B] float32 temperatures (0 = greedy row).
    """

    name: str
    dtype: str  # "bf16" or "f32"
    logits: np.ndarray
    q: np.ndarray
    x: np.ndarray
    u: np.ndarray
    T: np.ndarray

    @property
    def B(self) -> int:
        return int(self.x.shape[0])

    @property
    def k(self) -> int:
        return int(self.x.shape[1])

    @property
    def V(self) -> int:
        return int(self.logits.shape[2])

    @property
    def logit_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the
    16-bit patterns as uint16.  Inputs here are finite."""
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _store(values_f64: np.ndarray, dtype: str) -> np.ndarray:
    f32 = values_f64.astype(np.float32)
    return f32_to_bf16_bits(f32) if dtype == "bf16" else f32


def _draft_softmax_f32(draft_logits: np.ndarray) -> np.ndarray:
    """The draft model's probabilities: softmax over the last axis in
    float64, rounded to float32."""
    z = draft_logits - draft_logits.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def _draft_sample(q_f32: np.ndarray, uniforms: np.ndarray) -> np.ndarray:
    """The draft model's sampling: token = first v whose running sum of the
    fp32 q (accumulated in float64) exceeds u times the total."""
    out = np.empty(q_f32.shape[:-1], dtype=np.int32)
    flat_q = q_f32.reshape(-1, q_f32.shape[-1])
    flat_u = uniforms.reshape(-1)
    flat_o = out.reshape(-1)
    for r in range(flat_q.shape[0]):
        c = np.cumsum(flat_q[r], dtype=np.float64)
        v = int(np.searchsorted(c, flat_u[r] * c[-1], side="right"))
        flat_o[r] = min(v, flat_q.shape[1] - 1)
    return out


def make_random(
    *,
    name: str,
    B: int,
    k: int,
    V: int,
    dtype: str,
    seed: int,
    logit_sigma: float,
    draft_sigma,
    temperature,
    spike: float = 0.0,
    spike_mode: str = "none",
    zipf_s: float = 1.1,
    greedy_rows: int = 0,
) -> Workload:
    """General seeded generator.

    Target logits L ~ N(0, logit_sigma^2) per entry, plus ``spike`` added at
    one token: ``spike_mode="position"`` picks a uniform random token per
    (row, position); ``"zipf"`` picks one Zipf(zipf_s)-ranked token per row
    (rank r over 1..V, token r-1) used at every position; ``"none"`` adds
    nothing.  Draft logits are L + N(0, sigma^2) with ``draft_sigma`` a
    float or a per-row array; q = softmax(draft logits) rounded to fp32.
    Rows ``b < greedy_rows`` get T = 0 and a greedy draft (argmax of the
    draft logits); the others get ``temperature`` and tokens drawn from q.
    """
    ss = np.random.SeedSequence(seed)
    s_logit, s_noise, s_draft, s_verify = ss.spawn(4)
    rng_l = np.random.default_rng(s_logit)
    rng_n = np.random.default_rng(s_noise)
    rng_d = np.random.default_rng(s_draft)
    rng_v = np.random.default_rng(s_verify)

    store_dtype = np.uint16 if dtype == "bf16" else np.float32
    logits = np.empty((B, k + 1, V), dtype=store_dtype)
    q = np.empty((B, k, V), dtype=np.float32)
    x = np.empty((B, k), dtype=np.int32)
    sig = np.broadcast_to(np.asarray(draft_sigma, dtype=np.float64), (B,))
    draft_u = rng_d.random((B, k))

    for b in range(B):
        L = rng_l.standard_normal((k + 1, V)) * logit_sigma
        if spike_mode == "position":
            idx = rng_l.integers(0, V, size=k + 1)
            L[np.arange(k + 1), idx] += spike
        elif spike_mode == "zipf":
            while True:
                r = int(rng_l.zipf(zipf_s))
                if r <= V:
                    break
            L[:, r - 1] += spike
        D = L[:k] + rng_n.standard_normal((k, V)) * sig[b]
        logits[b] = _store(L, dtype)
        q[b] = _draft_softmax_f32(D)
        if b < greedy_rows:
            x[b] = np.argmax(D, axis=-1).astype(np.int32)
        else:
            x[b] = _draft_sample(q[b], draft_u[b])

    u = rng_v.random((B, k + 1, 2), dtype=np.float32)
    T = np.full(B, temperature, dtype=np.float32)
    T[:greedy_rows] = 0.0
    return Workload(name, dtype, logits, q, x, u, T)


def make_from_distributions(
    p: np.ndarray, q_dist: np.ndarray, *, B: int, k: int, seed: int, name: str = "fixed"
) -> Workload:
    """Identical target and draft distributions at every position: target
    logits log(p) plus a seeded N(0, 2^2) shift per (row, position) (the
    softmax ignores it; it keeps every row's max and sum distinct), stored
    as fp32 with T = 1; draft probabilities q_dist (fp32), draft tokens drawn
    from q_dist, verify uniforms seeded."""
    ss = np.random.SeedSequence(seed)
    s_draft, s_verify, s_shift = ss.spawn(3)
    V = len(p)
    logp = np.log(np.asarray(p, dtype=np.float64))
    shift = np.random.default_rng(s_shift).standard_normal((B, k + 1, 1)) * 2.0
    logits = (logp[None, None, :] + shift).astype(np.float32)
    qf = np.asarray(q_dist, dtype=np.float32)
    q = np.broadcast_to(qf, (B, k, V)).copy()
    c = np.cumsum(qf, dtype=np.float64)
    du = np.random.default_rng(s_draft).random((B, k))
    x = np.minimum(np.searchsorted(c, du * c[-1], side="right"), V - 1).astype(np.int32)
    u = np.random.default_rng(s_verify).random((B, k + 1, 2), dtype=np.float32)
    T = np.ones(B, dtype=np.float32)
    return Workload(name, "f32", logits, q, x, u, T)


def _toy(seed):
    return make_random(name="toy B=1 k=4 V=1000 fp32", B=1, k=4, V=1000, dtype="f32",
                       seed=seed, logit_sigma=2.0, draft_sigma=1.0, temperature=1.0)


def _zipf(seed):
    return make_random(name="B=8 k=4 V=32000 bf16 zipf", B=8, k=4, V=32000, dtype="bf16",
                       seed=seed, logit_sigma=3.0, draft_sigma=1.5, temperature=0.8,
                       spike=6.0, spike_mode="zipf")


def _benchmark(seed):
    return make_random(name="B=64 k=5 V=128256 bf16", B=64, k=5, V=128256, dtype="bf16",
                       seed=seed, logit_sigma=3.0, draft_sigma=1.0, temperature=1.0,
                       spike=8.0, spike_mode="position")


def _mixed(seed):
    sig = np.random.default_rng(np.random.SeedSequence([seed, 1])).uniform(0.5, 3.0, size=256)
    return make_random(name="B=256 k=8 V=128256 bf16 half greedy", B=256, k=8, V=128256,
                       dtype="bf16", seed=seed, logit_sigma=3.0, draft_sigma=sig,
                       temperature=0.7, spike=8.0, spike_mode="position", greedy_rows=128)


def _split_v(seed):
    return make_random(name="B=16 k=16 V=151936 fp32", B=16, k=16, V=151936, dtype="f32",
                       seed=seed, logit_sigma=4.0, draft_sigma=2.0, temperature=1.0)


# name -> (builder, default seed)
WORKLOADS = {
    "toy": (_toy, 57001),
    "zipf": (_zipf, 57002),
    "benchmark": (_benchmark, 57003),
    "mixed": (_mixed, 57004),
    "split_v": (_split_v, 57005),
}


def make_workload(name: str, seed: int | None = None) -> Workload:
    """The named workload (``toy``, ``zipf``, ``benchmark``, ``mixed``,
    ``split_v``), from its default seed unless one is given."""
    build, default_seed = WORKLOADS[name]
    return build(default_seed if seed is None else seed)


def make_rollback_batch(seed: int, B: int, k: int, block_size: int, max_blocks: int):
    """Paged-cache state after a verify step of B rows with k drafts each:
    num_accepted uniform on 0..k; every row holds between k and
    max_blocks * block_size positions, its blocks a slice of one random
    permutation of the pool.  Returns (num_accepted, seq_lens, block_tables,
    num_blocks), int32."""
    rng = np.random.default_rng(np.random.SeedSequence(seed))
    lens = rng.integers(k, max_blocks * block_size + 1, size=B).astype(np.int32)
    nb = ((lens + block_size - 1) // block_size).astype(np.int32)
    tables = np.full((B, max_blocks), -1, np.int32)
    perm = rng.permutation(B * max_blocks).astype(np.int32)
    for b in range(B):
        tables[b, : nb[b]] = perm[b * max_blocks: b * max_blocks + nb[b]]
    na = rng.integers(0, k + 1, size=B).astype(np.int32)
    return na, lens, tables, nb
