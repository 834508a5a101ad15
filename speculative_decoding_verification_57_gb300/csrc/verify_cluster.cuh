// verify_cluster.cuh -- split-vocabulary verify kernel: one thread-block
// cluster of C CTAs per sequence, each CTA owning a contiguous V-slice of
// all k+1 positions.
//
// Each CTA has four consumer warps and one producer warp.  The producer
// streams tiles into a ring of shared-memory stages with 1-D bulk (TMA)
// copies; "full" and "empty" mbarriers hand the stages back and forth, so no
// block-wide barrier sits in the streaming loops.
//
// Pass 1 streams the CTA's slice of every position once and keeps, per
// position, an online maximum and sum of exp((l - max) / T) (sampled rows) or
// the maximum and its lowest index (greedy rows).  The per-CTA partials meet
// over distributed shared memory after a cluster barrier; every CTA then
// evaluates the accept tests and the first rejection with one warp ballot,
// identically.  Pass 2 streams only the stop position j (target logits and,
// after a rejection, the draft row q_j), one 1024-entry tile per warp: it
// weighs every entry by max(0, p_j - q_j) (or p_k for the bonus) in
// double-float sums, evaluating the exponential exactly (a table-driven
// 2^x, or a per-row table of bf16 values) for the entries whose probability
// can move the draw, and keeps sums per tile and per 32-entry lane segment.
// After a second exchange of CTA totals the CTA whose slice holds u * W finds
// the tile, then the segment, and one warp recomputes the segment's 32
// weights exactly to pick the token.
//
// Sources (page title, section): "LLM Inference & Speculative Decoding: From
// Roofline Physics to Lossless Acceleration", s.2 (acceptance rule, residual,
// bonus token, q clamp) and s.4 (greedy rule for T = 0, FP32 or better);
// "Speculative Decoding: Mathematical Foundations, ...", "The Modified
// Rejection Sampling Algorithm"; "Speculative decoding." lesson, "First: what
// an output distribution is" (softmax with temperature, inverse CDF);
// "Speculative Decoding: Draft, Verify, Accept", demo part B (zero-mass
// residual falls back to p).
#pragma once
#include <cfloat>
#include <cstddef>
#include <cstdint>

#include <cuda_bf16.h>

#include "exp2dd.cuh"
#include "ptx.cuh"

namespace specv {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kTileBytes = 8192;
constexpr int kStages = 5;         // pass-1 ring: stages of kTileBytes
constexpr int kRingBytes = kStages * kTileBytes;
constexpr int kStages2 = 8;        // pass-2 ring: at most this many slots of one tile each
constexpr int kMaxK = 31;          // positions 0..k fit one warp
constexpr int kMaxSlice = 16384;   // elements of one position held by one CTA
constexpr int kChunk = 8;          // pass-2 entries per chunk
constexpr int kLaneEntries = 32;   // pass-2 entries per lane and tile (four chunks)
constexpr int kP2Elems = kLaneEntries * 32;  // pass-2 tile: 1024 entries, one warp
constexpr int kMaxP2Tiles = kMaxSlice / kP2Elems;
constexpr float kLargeP = 1e-5f;   // pass-2 entries with p above this take the exact e (exp2dd or the bf16 table)
constexpr uint32_t kWaitPolls = 1u << 22;
constexpr int kLookTiles = 5;      // pass 1 reads at most this many tiles past the first undecided position
constexpr uint32_t kNapNs = 1000;  // longest sleep of a producer loop that found nothing to do
constexpr float kLog2e = 1.44269504088896341f;

enum : int {
    ST_NONFINITE = 1,
    ST_TOKEN = 2,
    ST_UNIFORM = 4,
    ST_TEMP = 8,
    ST_ZERO_RESIDUAL = 16,
    ST_QBAD = 32,
    ST_TIMEOUT = 64,
    ST_PARENT = 512,   // tree verification: a parent index outside [-1, node)
    ST_FILTER = 1024,  // top-k / top-p verification: top_k outside [1, 4096] or top_p outside (0, 1]
    ST_ERRMASK = 1 | 2 | 4 | 8 | 32 | 64 | 512 | 1024,
};

// Stop-row weights: residual max(0, e - s q); bonus e; fallback e (zero
// residual mass); one-hot e except at the draft token (q = point mass there).
enum : int { MODE_RESIDUAL = 0, MODE_BONUS = 1, MODE_FALLBACK = 2, MODE_ONEHOT = 3 };

struct VerifyArgs {
    const void* logits;      // [B, k+1, V] bf16 or fp32
    const float* q;          // [B, k, V]; null: one-hot drafts (and for all-greedy calls)
    const int32_t* x;        // [B, k]
    const float* u;          // [B, k+1, 2] (nullable when every row is greedy)
    const float* temp;       // [B] (nullable: every row greedy)
    int32_t* num_accepted;   // [B]
    int32_t* out_tokens;     // [B, k+1]
    int32_t* row_status;     // [B] (nullable)
    const int32_t* parents;  // [B, k] tree verification: parent node of each draft (-1: the prefix); null: a chain
    int32_t* path;           // [B, k] tree verification: accepted node indices, root first (nullable)
    const int32_t* top_k;    // [B] top-k / top-p verification: entries kept (null: the plain rule)
    const float* top_p;      // [B] top-k / top-p verification: nucleus mass within them
    float* dbg_p;            // [B, k] (nullable)
    float* dbg_q;            // [B, k]
    float* dbg_max;          // [B, k+1]
    float* dbg_sumexp;       // [B, k+1]
    float* dbg_resid;        // [B]
    long long V;
    int B;
    int k;
    int slice;               // elements per CTA, a multiple of 64
    int pk;                  // positions per partial array in shared memory (>= k + 1)
    int q_host;              // q is page-locked host memory read in place: plain loads only, no bulk copies
    int withhold = -1;       // test only: pass-1 stage use of CTA 0 that is never filled (-1: none)
    uint32_t polls = kWaitPolls;  // poll limit of every wait
};

struct Partial {
    float m;    // running max (sampled) / best value (greedy)
    float s;    // sum of exp((l - m) / T) (sampled)
    int arg;    // lowest index of the best value (greedy)
    int flags;  // bit 0: a NaN was seen (greedy); bit 1: a wait timed out
};

// Dynamic shared memory: the ring (kRingBytes), then the per-warp partials
// [pk][kConsumerWarps], then every cluster CTA's partials [pk][C] (pushed by
// each CTA of the cluster).
inline size_t cluster_dyn_smem(int C, int pk) {
    return static_cast<size_t>(kRingBytes) + static_cast<size_t>(kConsumerWarps + C) * pk * sizeof(Partial);
}

struct alignas(16) ClusterSmem {
    int tstart[kMaxK + 2];      // first pass-1 tile of each position
    int head[kMaxK + 1];        // unaligned leading elements of each position's slice
    int nbytes[kMaxK + 1];      // bytes of the 16-byte aligned interior
    unsigned long long full[kStages];
    unsigned long long empty[kStages];
    unsigned long long full2[kStages2];
    unsigned long long empty2[kStages2];
    float tile_hi[kMaxP2Tiles];  // pass-2 weights per tile of 1024 entries (pair), and q sums
    float tile_lo[kMaxP2Tiles];
    float tile_q[kMaxP2Tiles];
    float lane_hi[kMaxP2Tiles][32];  // the same per 32-entry lane segment
    float lane_lo[kMaxP2Tiles][32];
    float lane_q[kMaxP2Tiles][32];
    alignas(16) float alltot[16][8];  // every CTA's pass-2 totals: weights (pair), sum of e (pair), q over positive residuals, flags
    float wred_hi[kConsumerWarps];
    float wred_lo[kConsumerWarps];
    float2 exp2tab[128];
    alignas(16) uint32_t lpad[4];  // one masked piece of logits (-inf)
    alignas(16) float qpad[4];     // and of q (zero)
    int xs[kMaxK + 1];          // draft tokens, for whoever writes the outputs
    unsigned long long pbar[kMaxK + 1];  // position i: complete once every cluster CTA's partial has landed here
    unsigned long long cbar[kMaxK + 1];  // position i: complete once this CTA's four consumer warps have reported it
    float posM[kMaxK + 1];      // merged per position: maximum, sum of exponentials (sampled),
    float posS[kMaxK + 1];
    int posA[kMaxK + 1];        // argmax (greedy), partial flags,
    int posF[kMaxK + 1];
    int posE[kMaxK + 1];        // error bits of its test,
    float posP[kMaxK + 1];      // p(x_i)
    int2 views[16];             // every cluster CTA's outcome (stop position, status), pushed by it
    int p1_end;                 // pass-1 stage uses issued in all, once the producer stops issuing
    int stop_pos;               // the first stopping position, once decided (-1 before)
    int j, status, mode, owner, p2fast, ntiles2, timeout, stride2, nslots2, loff2;
    float Mj, sj, thr, c_hi, c_lo, uj;
    float delta, sp_hi, sp_lo, t_hi, t_lo;
};
static_assert(sizeof(Partial) == 16, "Partial is pushed with one 16-byte store");
static_assert(kRingBytes % 16 == 0 && sizeof(Partial) % 16 == 0, "partials follow the ring 16-byte aligned");
static_assert(offsetof(ClusterSmem, alltot) % 16 == 0, "16-byte remote stores need 16-byte aligned targets");
static_assert(alignof(ClusterSmem) >= 16, "ClusterSmem must be 16-byte aligned");

__device__ __forceinline__ float load_logit(const void* base, long long idx, bool bf16) {
    if (bf16) {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(base) + idx);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    return __ldg(reinterpret_cast<const float*>(base) + idx);
}

// Combine two online-softmax partials (m, s) at the common scale.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float c) {
    const float M = fmaxf(m, m2);
    float a = (m == -INFINITY) ? 0.0f : s * ex2((m - M) * c);
    float b2 = (m2 == -INFINITY) ? 0.0f : s2 * ex2((m2 - M) * c);
    if (M == -INFINITY) {
        a = 0.0f;
        b2 = 0.0f;
    }
    // NaN sums stay NaN
    if (s != s) a = s;
    if (s2 != s2) b2 = s2;
    m = M;
    s = a + b2;
}

// One partial's sum at the common maximum M >= m, for a merge of several
// partials at once (the sums are then added): a partial whose maximum is
// -inf adds nothing, a NaN sum stays NaN.
__device__ __forceinline__ float ms_term(float m, float s, float M, float c) {
    if (m == -INFINITY) return (s != s) ? s : 0.0f;
    return s * ex2((m - M) * c);
}

// Greedy partial merge: larger value wins, equal values keep the lower index.
__device__ __forceinline__ void merge_arg(float& v, int& a, float v2, int a2) {
    if (v2 > v || (v2 == v && a2 < a)) {
        v = v2;
        a = a2;
    }
}

// One element of the online softmax (the unaligned head/tail of a slice).
__device__ __forceinline__ void online_add(float& m, float& s, float l, float c) {
    if (l > m) {
        // s is 0 while m is -inf, unless a NaN was seen: s * 0 keeps it
        s = (m == -INFINITY) ? s * 0.0f : s * ex2((m - l) * c);
        m = l;
    }
    if (m != -INFINITY || l != l) s += ex2((l - m) * c);
}

// Per-row constants of the stop-row weights.
struct RowConst {
    float M;       // row max
    float s1;      // pass-1 sum of exp((l - M) / T)
    float thr;     // entries with e above this take the double-float exponential
    float ch, cl;  // log2(e) / T as a float pair
};

// e with exp2dd, as a pair.  The difference l - M is split exactly (two-sum):
// a logit close to zero next to a large maximum does not fit one float.
template <bool BF16>
__device__ __forceinline__ df precise_e(float l, const RowConst& rc, const float2* tab) {
    float dh, dl;
    two_sum(l, -rc.M, dh, dl);
    const float xh = dh * rc.ch;
    const float xl = fmaf(dl, rc.ch, fmaf(dh, rc.cl, fmaf(dh, rc.ch, -xh)));
    const float2 e = exp2dd(xh, xl, tab);
    return df{e.x, e.y};
}

// e - s q as a pair (s q formed exactly with one fma).
__device__ __forceinline__ df minus_sq(df e, df s, float q) {
    const df p = df_mul_f(s, q);
    float rh, rl;
    two_sum(e.hi, -p.hi, rh, rl);
    return df{rh, rl + (e.lo - p.lo)};
}

// The final weight of one entry, exactly (pair): e, or max(0, e - s q) with
// the recomputed s in residual mode.
template <bool BF16>
__device__ __forceinline__ df exact_weight(float l, float qv, int md, const RowConst& rc, df s_prec,
                                           const float2* tab) {
    if (l == -INFINITY) return df_make(0.0f);
    const df e = precise_e<BF16>(l, rc, tab);
    if (md != MODE_RESIDUAL) return e;
    const df r = minus_sq(e, s_prec, qv);
    return (r.hi + r.lo > 0.0f) ? r : df_make(0.0f);
}

// precise_e for two entries at once: the same steps and roundings, lane by
// lane, with the f32x2 instructions where a step has one.  Returns the pairs
// as (EH, EL) = ((e0.hi, e1.hi), (e0.lo, e1.lo)).
__device__ __forceinline__ void precise_e_x2(f2 L, const RowConst& rc, const float2* tab, f2& EH, f2& EL) {
    // two-sum L - M
    const f2 NM = pack2(-rc.M, -rc.M);
    const f2 DH = add2(L, NM);
    const f2 BB = sub2(DH, L);
    const f2 DL = add2(sub2(L, sub2(DH, BB)), sub2(NM, BB));
    // x = (DH + DL) (ch + cl): NX = -xh exactly (round to nearest is symmetric)
    const f2 CH = pack2(rc.ch, rc.ch);
    const f2 NX = mul2(DH, pack2(-rc.ch, -rc.ch));
    const f2 XL = fma2(DL, CH, fma2(DH, pack2(rc.cl, rc.cl), fma2(DH, CH, NX)));
    // exp2dd, both lanes
    float n0, n1;
    unpack2(NX, n0, n1);
    const float xh0 = fmaxf(-n0, -125.0f), xh1 = fmaxf(-n1, -125.0f);
    const float kf0 = rintf(xh0 * 128.0f), kf1 = rintf(xh1 * 128.0f);
    const int K0 = static_cast<int>(kf0), K1 = static_cast<int>(kf1);
    const f2 F = add2(fma2(pack2(kf0, kf1), pack2(-0.0078125f, -0.0078125f), pack2(xh0, xh1)), XL);
    const f2 T = mul2(F, pack2(kLn2, kLn2));
    const f2 H = fma2(T, pack2(0.16666667f, 0.16666667f), pack2(0.5f, 0.5f));
    const f2 P = fma2(mul2(T, T), H, T);  // e^t - 1
    const float2 t0 = tab[K0 & 127], t1 = tab[K1 & 127];
    const f2 TH = pack2(t0.x, t1.x);
    const f2 LO = fma2(TH, P, pack2(t0.y, t1.y));
    const f2 SC = pack2(__int_as_float(((K0 >> 7) + 127) << 23), __int_as_float(((K1 >> 7) + 127) << 23));
    EH = mul2(TH, SC);
    EL = mul2(LO, SC);
}

// (H, L) += (XH, XL) for two pair sums advanced together, lane by lane.
__device__ __forceinline__ void df2_add_pair(f2& H, f2& L, f2 XH, f2 XL) {
    const f2 S = add2(H, XH);
    const f2 BB = sub2(S, H);
    const f2 E = add2(sub2(H, sub2(S, BB)), sub2(XH, BB));
    H = S;
    L = add2(L, add2(E, XL));
}

// ------------------------------------------------------------------ stop-row sweep
// Constants of the stop-row sweep, packed for the f32x2 instructions.
struct SweepConst {
    f2 MM;      // (M, M): the row maximum
    f2 CH;      // high part of log2(e) / T
    f2 NCH;     // its negation
    f2 CL;      // low part of log2(e) / T
    f2 LN2;     // ln 2
    f2 NS1;     // -s1, the pass-1 sum of exponentials
    float thr;  // entries whose estimate of e exceeds this are "large"
};

// SFU estimate of e = 2^((l - M) log2(e) / T) for two entries.  The exponent
// is a float pair: xh = (l - M) ch rounded, and xl = the product's rounding
// error plus (l - M) cl, folded back in to first order.  A masked entry
// (l = -inf) comes out NaN; the sweep gives it weight zero.
__device__ __forceinline__ f2 fast_e2(f2 L, const SweepConst& K) {
    const f2 D = sub2(L, K.MM);
    const f2 N = mul2(D, K.NCH);                    // -xh
    const f2 XL = fma2(D, K.CL, fma2(D, K.CH, N));  // xl
    float n0, n1;
    unpack2(N, n0, n1);
    const f2 E = pack2(ex2(-n0), ex2(-n1));
    return fma2(E, mul2(XL, K.LN2), E);
}

// (hi, lo) pairs of two sums advanced together: H + L += X, lane by lane.
__device__ __forceinline__ void df2_add(f2& H, f2& L, f2 X) {
    const f2 S = add2(H, X);
    const f2 BB = sub2(S, H);
    const f2 E = add2(sub2(H, sub2(S, BB)), sub2(X, BB));
    H = S;
    L = add2(L, E);
}

// One lane's sums over its 32 consecutive stop-row entries of a tile.
// Weights are in e-units (the row's sum of exponentials times p): residual
// mode r = max(0, e - s1 q), bonus / fallback mode e.  Small entries are
// summed in floats, sixteen at a time, and folded into the pairs; large entries
// (estimate above thr) are left out here and added exactly afterwards.
struct LaneAcc {
    f2 wh, wl;       // (weights, sum of e) as (hi, lo) pairs, packed
    float q;         // q over entries with a positive residual
    f2 qa;           // every q: a NaN or an infinity surfaces here
    uint32_t qor;    // OR of the q bit patterns: a set sign bit marks a possible negative
    uint32_t large;  // bit i: entry i of the lane's 32 is large
};

__device__ __forceinline__ void lane_init(LaneAcc& A) {
    A.wh = pack2(0.0f, 0.0f);
    A.wl = pack2(0.0f, 0.0f);
    A.q = 0.0f;
    A.qa = pack2(0.0f, 0.0f);
    A.qor = 0;
    A.large = 0;
}

// The lane's 32 entries in eight pieces of four, visited in the lane-rotated
// order (p + rot) mod 8 so that the warp's 8- and 16-byte shared loads fall
// in distinct banks.  ls / qs: this lane's logits and q in shared memory;
// pieces at or past nvl / 4 read lpad / qpad (a masked logit, q = 0).
template <bool BF16, bool RESID>
__device__ __forceinline__ void sweep_lane(LaneAcc& A, const unsigned char* ls, const float* qs, const void* lpad,
                                           const float* qpad, int rot, int nvl, const SweepConst& K) {
    f2 sw = pack2(0.0f, 0.0f), se = pack2(0.0f, 0.0f), sq = pack2(0.0f, 0.0f);
#pragma unroll
    for (int st = 0; st < 8; ++st) {
        const int p = (st + rot) & 7;
        const bool valid = 4 * p < nvl;
        f2 L0, L1;
        if (BF16) {
            const uint2 w = *reinterpret_cast<const uint2*>(valid ? static_cast<const void*>(ls + 8 * p) : lpad);
            L0 = pack2(bf16_lo(w.x), bf16_hi(w.x));
            L1 = pack2(bf16_lo(w.y), bf16_hi(w.y));
        } else {
            const float4 w = *reinterpret_cast<const float4*>(valid ? static_cast<const void*>(ls + 16 * p) : lpad);
            L0 = pack2(w.x, w.y);
            L1 = pack2(w.z, w.w);
        }
        float e[4];
        unpack2(fast_e2(L0, K), e[0], e[1]);
        unpack2(fast_e2(L1, K), e[2], e[3]);
        uint32_t bits = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            bits |= (e[i] > K.thr ? 1u : 0u) << i;
            e[i] = (e[i] <= K.thr) ? e[i] : 0.0f;  // large entries and NaN (masked) weigh nothing here
        }
        A.large |= bits << (4 * p);
        const f2 ES0 = pack2(e[0], e[1]), ES1 = pack2(e[2], e[3]);
        if (RESID) {
            const float4 qv = *reinterpret_cast<const float4*>(valid ? qs + 4 * p : qpad);
            const f2 Q0 = pack2(qv.x, qv.y), Q1 = pack2(qv.z, qv.w);
            float r[4];
            unpack2(fma2(K.NS1, Q0, ES0), r[0], r[1]);
            unpack2(fma2(K.NS1, Q1, ES1), r[2], r[3]);
            sw = add2(sw, pack2(fmaxf(r[0], 0.0f), fmaxf(r[1], 0.0f)));
            sw = add2(sw, pack2(fmaxf(r[2], 0.0f), fmaxf(r[3], 0.0f)));
            sq = add2(sq, pack2(r[0] > 0.0f ? qv.x : 0.0f, r[1] > 0.0f ? qv.y : 0.0f));
            sq = add2(sq, pack2(r[2] > 0.0f ? qv.z : 0.0f, r[3] > 0.0f ? qv.w : 0.0f));
            se = add2(se, add2(ES0, ES1));
            A.qa = add2(A.qa, add2(Q0, Q1));
            A.qor |= __float_as_uint(qv.x) | __float_as_uint(qv.y) | __float_as_uint(qv.z) | __float_as_uint(qv.w);
        } else {
            sw = add2(sw, add2(ES0, ES1));
        }
        if ((st & 3) == 3) {
            // fold the sixteen entries of the last four pieces into the pairs
            float a0, a1, b0, b1;
            unpack2(sw, a0, a1);
            unpack2(se, b0, b1);
            df2_add(A.wh, A.wl, pack2(a0 + a1, b0 + b1));
            sw = pack2(0.0f, 0.0f);
            se = pack2(0.0f, 0.0f);
        }
    }
    float q0, q1;
    unpack2(sq, q0, q1);
    A.q += q0 + q1;
}

// Greedy verification of a draft tree, one warp ("LLM Inference & Speculative
// Decoding ...", s.3 "Multi-Draft Tree Speculation"; "Speculative Decoding:
// Mathematical Foundations, ...", "SpecInfer and Tree-Based Verification":
// the longest accepted path is kept).  Lane i < k holds node i (token xi,
// parent pi in [-1, i)); lane r <= k holds the argmax A of logit row r (row
// 0 after the prefix, row 1 + i after node i) and its flags (bit 0 NaN, bit
// 1 timeout).  A node is kept iff its token is its parent row's argmax and
// every ancestor is kept (pointer jumping over the parent links, 5 rounds for
// up to 32 nodes); the deepest kept node wins, the lowest index among equals;
// the bonus is the argmax of its own row.  Writes the outputs if `write`.
__device__ __forceinline__ int tree_greedy_warp(const VerifyArgs& a, int b, int k, int lane, int xi, int pi, int A,
                                                int flags, bool write) {
    const unsigned full = 0xffffffffu;
    const bool node = lane < k;
    int err = 0;
    if (lane <= k && (flags & 1)) err |= ST_NONFINITE;
    if (lane <= k && (flags & 2)) err |= ST_TIMEOUT;
    if (node && (xi < 0 || xi >= a.V)) err |= ST_TOKEN;
    if (node && (pi < -1 || pi >= lane)) err |= ST_PARENT;
    err = static_cast<int>(__reduce_or_sync(full, static_cast<unsigned>(err)));
    const int pv = (node && !(err & ST_PARENT)) ? pi : -1;
    const int apar = __shfl_sync(full, A, pv + 1);
    bool m = node && xi == apar;      // kept along the path to the prefix
    int d = (node && pv >= 0) ? 1 : 0;  // depth (children of the prefix: 0)
    int p = pv;
    for (int s = 0; s < 5; ++s) {
        const int src = p >= 0 ? p : lane;
        const bool mp = __shfl_sync(full, m, src);
        const int dp = __shfl_sync(full, d, src);
        const int pp = __shfl_sync(full, p, src);
        if (p >= 0) {
            m = m && mp;
            d += dp;
            p = pp;
        }
    }
    const int key = (node && m) ? ((d << 6) | (63 - lane)) : -1;
    const int kb = __reduce_max_sync(full, key);
    const int best = kb < 0 ? -1 : 63 - (kb & 63);
    const int n = best < 0 ? 0 : (kb >> 6) + 1;
    const int bonus = __shfl_sync(full, A, best + 1);
    if (write) {
        int tokv = -1, pathv = -1;
        int cur = best;
        for (int s = 0; s < 32 && cur >= 0; ++s) {  // cur is the same in every lane
            const int dc = __shfl_sync(full, d, cur);
            const int tc = __shfl_sync(full, xi, cur);
            const int pc = __shfl_sync(full, pv, cur);
            if (lane == dc) {
                tokv = tc;
                pathv = cur;
            }
            cur = pc;
        }
        if (lane == n) tokv = bonus;
        if (err) {
            tokv = -1;
            pathv = -1;
        }
        if (lane <= k) a.out_tokens[static_cast<long long>(b) * (k + 1) + lane] = tokv;
        if (lane < k && a.path) a.path[static_cast<long long>(b) * k + lane] = pathv;
        if (lane == 0) {
            a.num_accepted[b] = err ? 0 : n;
            if (a.row_status) a.row_status[b] = err;
        }
    }
    return err;
}

// Write a sampled row's outputs: the kept drafts, the drawn token, -1 after.
__device__ __forceinline__ void write_sampled(const VerifyArgs& a, int b, int k, int j, int token, int st,
                                              const int* xs) {
    for (int i = 0; i <= k; ++i) {
        int tok = -1;
        if (i < j)
            tok = xs[i];
        else if (i == j)
            tok = token;
        a.out_tokens[static_cast<long long>(b) * (k + 1) + i] = tok;
    }
    a.num_accepted[b] = j;
    if (a.row_status) a.row_status[b] = st;
}

// Fold one pass-1 tile into a consumer thread's online state.  The tile is
// NT * 64 bytes of one position's logits; thread tid (0 .. NT-1) holds its
// four 16-byte chunks r = 0 .. 3 in w[r], chunk r covering the tile's
// elements (tid + r * NT) * (16 / esz) onward; tile_e0 is the index, within
// the row, of the tile's first element.  Sampled rows keep (m, s): the
// running maximum and the sum of exp((l - m) / T) (c = log2(e) / T); greedy
// rows keep the maximum m, its lowest index arg and whether a NaN was seen.
// Elements past the end of a short tile must hold -inf.
template <bool BF16, int NT = kConsumers>
__device__ __forceinline__ void p1_fold_tile(const uint4 (&w)[4], bool greedy, float c, long long tile_e0, int tid,
                                             float& m, float& s, int& arg, bool& nan_seen) {
    constexpr int kPer = 4;
    constexpr int kConsumers = NT;  // the chunk stride of this tile layout
    float lmax;
    if (BF16) {
        if (greedy) {
            // one NaN-propagating maximum: a NaN only flags the row (its
            // argmax is undefined), so it may hide the tile's other values
            uint32_t mx = 0xff80ff80u;
#pragma unroll
            for (int r = 0; r < kPer; ++r)
                mx = max_nan_bf16x2(max_nan_bf16x2(mx, w[r].x),
                                    max_nan_bf16x2(w[r].y, max_nan_bf16x2(w[r].z, w[r].w)));
            lmax = max_nan_f32(bf16_lo(mx), bf16_hi(mx));
            if (lmax != lmax) nan_seen = true;
        } else {
            uint32_t mr[kPer];  // a tree: each chunk's maximum, then theirs
#pragma unroll
            for (int r = 0; r < kPer; ++r) mr[r] = max_bf16x2(max_bf16x2(w[r].x, w[r].y), max_bf16x2(w[r].z, w[r].w));
            // (with -inf: a tile of NaN alone yields -inf, and the NaN search below)
            const uint32_t mx = max_bf16x2(max_bf16x2(max_bf16x2(mr[0], mr[1]), max_bf16x2(mr[2], mr[3])), 0xff80ff80u);
            lmax = fmaxf(bf16_lo(mx), bf16_hi(mx));
        }
    } else {
        float mx = -INFINITY, mn = -INFINITY;
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
            const float f0 = __uint_as_float(w[r].x), f1 = __uint_as_float(w[r].y);
            const float f2v = __uint_as_float(w[r].z), f3 = __uint_as_float(w[r].w);
            mx = fmaxf(fmaxf(mx, f0), fmaxf(f1, fmaxf(f2v, f3)));
            if (greedy) mn = max_nan_f32(max_nan_f32(mn, f0), max_nan_f32(f1, max_nan_f32(f2v, f3)));
        }
        lmax = mx;
        if (greedy && mn != mn) nan_seen = true;
    }
    if (greedy) {
        if (BF16 && lmax > m) {
            // lowest tile-local index holding the new maximum: the first
            // chunk whose maximum equals it (chunk r covers elements
            // ch*8 .. ch*8+7, ch = tid + r*128), then the first such
            // element in it; the packed compare takes -0 == +0
            const uint32_t h16 = __float_as_uint(lmax) >> 16;
            const uint32_t lmw = h16 | (h16 << 16);
            const __nv_bfloat162 lm2 = *reinterpret_cast<const __nv_bfloat162*>(&lmw);
            int rs = kPer - 1;
#pragma unroll
            for (int r = kPer - 2; r >= 0; --r) {
                const uint32_t cmr = max_bf16x2(max_bf16x2(w[r].x, w[r].y), max_bf16x2(w[r].z, w[r].w));
                if (__heq2_mask(*reinterpret_cast<const __nv_bfloat162*>(&cmr), lm2)) rs = r;
            }
            uint4 wc = w[kPer - 1];
#pragma unroll
            for (int r = kPer - 2; r >= 0; --r)
                if (r == rs) wc = w[r];
            const uint32_t ws[4] = {wc.x, wc.y, wc.z, wc.w};
            int q8 = 7;
#pragma unroll
            for (int q4 = 3; q4 >= 0; --q4) {
                const uint32_t eqm = __heq2_mask(*reinterpret_cast<const __nv_bfloat162*>(&ws[q4]), lm2);
                if (eqm) q8 = q4 * 2 + ((eqm & 0xffffu) ? 0 : 1);
            }
            arg = static_cast<int>(tile_e0 + (tid + rs * kConsumers) * 8 + q8);
            m = lmax;
        } else if (!BF16 && lmax > m) {
            // lowest tile-local index holding the new maximum: the
            // candidates reduced by min in a tree (chunk r of this
            // thread covers elements ch*4+..., ch = tid + r*128)
            constexpr int kPerWord = BF16 ? 2 : 1;
            constexpr int kCand = kPer * 4 * kPerWord;
            int cand[kCand];
#pragma unroll
            for (int r = 0; r < kPer; ++r) {
                const int ch = tid + r * kConsumers;
                const uint32_t ws[4] = {w[r].x, w[r].y, w[r].z, w[r].w};
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    if (BF16) {
                        cand[(r * 4 + q4) * 2] = bf16_lo(ws[q4]) == lmax ? ch * 8 + q4 * 2 : 0x7fffffff;
                        cand[(r * 4 + q4) * 2 + 1] =
                            bf16_hi(ws[q4]) == lmax ? ch * 8 + q4 * 2 + 1 : 0x7fffffff;
                    } else {
                        cand[r * 4 + q4] = __uint_as_float(ws[q4]) == lmax ? ch * 4 + q4 : 0x7fffffff;
                    }
                }
            }
#pragma unroll
            for (int half = kCand / 2; half > 0; half >>= 1)
#pragma unroll
                for (int i2 = 0; i2 < half; ++i2) cand[i2] = min(cand[i2], cand[i2 + half]);
            arg = static_cast<int>(tile_e0 + cand[0]);
            m = lmax;
        }
    } else if (lmax == -INFINITY) {
        // the max ignores NaN: look for one among -inf entries
        bool has_nan = false;
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
            const uint32_t ws[4] = {w[r].x, w[r].y, w[r].z, w[r].w};
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                if (BF16)
                    has_nan |= ((ws[q4] & 0x7fffu) > 0x7f80u) || ((ws[q4] & 0x7fff0000u) > 0x7f800000u);
                else
                    has_nan |= (ws[q4] & 0x7fffffffu) > 0x7f800000u;
            }
        }
        if (has_nan) s = __uint_as_float(0x7fc00000u);
    } else {
        if (lmax > m) {
            s = (m == -INFINITY) ? s * 0.0f : s * ex2((m - lmax) * c);
            m = lmax;
        }
        // exponents as one fma a pair: l c - r with r = m c rounded; the
        // rounding error of r (err = m c - r, exact through an fma) scales
        // every term of the tile alike and is taken out once, to first
        // order (|err| <= ulp(m c) / 2, so the neglected term is ~1e-12)
        const float rr = m * c;
        const float err = fmaf(m, c, -rr);
        const f2 cc = pack2(c, c), nr = pack2(-rr, -rr);
        f2 acc[kPer];  // one sum per chunk: four short chains instead of one long one
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
            const uint32_t ws[4] = {w[r].x, w[r].y, w[r].z, w[r].w};
            acc[r] = pack2(0.0f, 0.0f);
            if (BF16) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const f2 d = fma2(pack2(bf16_lo(ws[q4]), bf16_hi(ws[q4])), cc, nr);
                    float d0, d1;
                    unpack2(d, d0, d1);
                    acc[r] = add2(acc[r], pack2(ex2(d0), ex2(d1)));
                }
            } else {
#pragma unroll
                for (int q4 = 0; q4 < 4; q4 += 2) {
                    const f2 d = fma2(pack2(__uint_as_float(ws[q4]), __uint_as_float(ws[q4 + 1])), cc, nr);
                    float d0, d1;
                    unpack2(d, d0, d1);
                    acc[r] = add2(acc[r], pack2(ex2(d0), ex2(d1)));
                }
            }
        }
        float a0, a1;
        unpack2(add2(add2(acc[0], acc[1]), add2(acc[2], acc[3])), a0, a1);
        s += (a0 + a1) * fmaf(-err, kLn2, 1.0f);  // back to the scale of m
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 4) verify_cluster_kernel(const VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ __align__(16) ClusterSmem sh;
    constexpr int esz = BF16 ? 2 : 4;
    const unsigned full = 0xffffffffu;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const bool producer = (warp == kConsumerWarps);
    const uint32_t rank = cluster_rank();
    const uint32_t C = cluster_size();
    const int b = blockIdx.x / C;
    const int k = a.k;
    const long long V = a.V;
    const long long v0 = static_cast<long long>(rank) * a.slice;
    const int n = static_cast<int>(max(0LL, min(static_cast<long long>(a.slice), V - v0)));
    const unsigned char* lg = reinterpret_cast<const unsigned char*>(a.logits);
    unsigned char* ring = dyn_smem;
    const uint32_t polls = a.polls;
    Partial* wpart = reinterpret_cast<Partial*>(dyn_smem + kRingBytes);  // [pk][kConsumerWarps]
    Partial* allpart = wpart + kConsumerWarps * a.pk;                     // [pk][C]: every CTA's, pushed by it
    // Positions after the first stop are never read: the rule does not look
    // at them.  Draft trees (every node counts) and calls that ask for every
    // position's debug values read them all.
    const bool early = !a.parents && !(a.dbg_p || a.dbg_q || a.dbg_max || a.dbg_sumexp);

    // ---------------------------------------------------------------- row setup
    const float T = a.temp ? __ldg(a.temp + b) : 0.0f;
    const bool greedy = (T == 0.0f);
    const bool t_ok = greedy || (T >= FLT_MIN && T <= FLT_MAX);
    const float c = greedy || !t_ok ? 0.0f : kLog2e / T;

    if (tid < 128) sh.exp2tab[tid] = g_exp2_table[tid];
    if (tid < 4) {
        sh.lpad[tid] = BF16 ? 0xff80ff80u : 0xff800000u;
        sh.qpad[tid] = 0.0f;
    }
    if (tid == 32 && !greedy && t_ok) {  // log2(e) / T as a pair, for the exact exponentials
        const df c2 = log2e_over(T);
        sh.c_hi = c2.hi;
        sh.c_lo = c2.lo;
    }
    // One pass-1 tile: tile tt of the CTA's slices, position by position.
    auto issue_p1 = [&](int tt, int it) {
        int i = 0;
        while (sh.tstart[i + 1] <= tt) ++i;
        const int off = (tt - sh.tstart[i]) * kTileBytes;
        const int bytes = min(kTileBytes, sh.nbytes[i] - off);
        const long long e0 = (static_cast<long long>(b) * (k + 1) + i) * V + v0 + sh.head[i];
        const int slot = it % kStages;
        const uint32_t bar = smem_u32(&sh.full[slot]);
        if (blockIdx.x == 0 && it == a.withhold) return;  // test hook: this stage is never filled
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(bytes));
        bulk_g2s(smem_u32(ring + slot * kTileBytes), lg + e0 * esz + off, static_cast<uint32_t>(bytes), bar);
    };
    int it_prod = 0;
    int c_slot = 0, c_phase = 0;  // the consumers' stage and its phase
    if (producer && lane == 0) {
        // the producer sets up the ring, the position barriers and the slice
        // geometry
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), kConsumerWarps);
        }
        for (int s = 0; s < kStages2; ++s) {
            mbar_init(smem_u32(&sh.full2[s]), 1);
            mbar_init(smem_u32(&sh.empty2[s]), 1);
        }
        for (int i = 0; i <= k; ++i) {
            mbar_init(smem_u32(&sh.pbar[i]), 1);
            mbar_init(smem_u32(&sh.cbar[i]), kConsumerWarps);
        }
        sh.timeout = 0;
        sh.p1_end = 0x7fffffff;
        sh.stop_pos = -1;
        fence_mbar_init();
        fence_proxy_async_smem();
        // position i is complete once every CTA of the cluster has stored its
        // 16-byte partial here
        for (int i = 0; i <= k; ++i) mbar_arrive_expect_tx(smem_u32(&sh.pbar[i]), C * sizeof(Partial));
        int acc = 0;
        for (int i = 0; i <= k; ++i) {
            const long long e0 = (static_cast<long long>(b) * (k + 1) + i) * V + v0;
            const uintptr_t addr = reinterpret_cast<uintptr_t>(lg + e0 * esz);
            int h = static_cast<int>(((16 - (addr & 15)) & 15) / esz);
            if (h > n) h = n;
            const int nb = ((n - h) * esz) & ~15;
            sh.head[i] = h;
            sh.nbytes[i] = nb;
            sh.tstart[i] = acc;
            acc += (nb + kTileBytes - 1) / kTileBytes;
        }
        sh.tstart[k + 1] = acc;
    }
    if (producer) {
        // the first copies, one a lane, before the block's first barrier
        __syncwarp();
        // the tiles the rule may need: position 0's and kLookTiles more
        const int lim = t_ok ? (early ? min(sh.tstart[k + 1], sh.tstart[1] + kLookTiles) : sh.tstart[k + 1]) : 0;
        it_prod = min(kStages, lim);
        if (lane < it_prod) issue_p1(lane, lane);
    }
    __syncthreads();
    // Every CTA's position barriers are initialised before any CTA arrives on
    // them: each thread waits on this cluster barrier before its first remote
    // arrival (and before the next cluster barrier).
    cluster_arrive();
    const int total1 = t_ok ? sh.tstart[k + 1] : 0;

    // the consumers' next stage: c_slot = it % kStages, c_phase = (it / kStages) & 1
    auto next_stage = [&]() {
        if (++c_slot == kStages) {
            c_slot = 0;
            c_phase ^= 1;
        }
    };

    // per-position scalars, lane i of the producer warp holds position i
    int xi = -1, pi = lane - 1;
    float u0 = 0.0f, u1 = 0.0f, Lx = 0.0f, qx = 0.0f;
    int stop = -1;  // the first position that stops the chain (producer warp)

    // ---------------------------------------------------------------- pass 1 and the decisions
    if (producer) {
        if (lane <= k && t_ok) {
            if (lane < k) xi = __ldg(a.x + static_cast<long long>(b) * k + lane);
            if (lane < k && a.parents) pi = __ldg(a.parents + static_cast<long long>(b) * k + lane);
            if (!greedy) {
                const long long ub = (static_cast<long long>(b) * (k + 1) + lane) * 2;
                u0 = __ldg(a.u + ub);
                u1 = __ldg(a.u + ub + 1);
                if (lane < k && xi >= 0 && xi < V) {  // the accept test's scalars
                    const long long row = static_cast<long long>(b) * (k + 1) + lane;
                    Lx = load_logit(a.logits, row * V + xi, BF16);
                    qx = a.q ? __ldg(a.q + (static_cast<long long>(b) * k + lane) * V + xi) : 1.0f;
                }
            }
        }
        const int ndec = t_ok ? k + 1 : 0;
        int dpos = 0;  // positions decided so far
        int ppos = 0;  // positions of this CTA pushed to the cluster
        cluster_wait();  // the peers' position barriers are set up: pushes may start
        uint32_t idle = 0;
        unsigned long long t0 = 0;
        bool gave_up = false;
        // One loop issues the tiles (lanes 0..4) and takes the decisions (the
        // whole warp), in position order, as the CTAs' partials come in.  A
        // tile is issued only while it lies at most kLookTiles past the last
        // tile of the first undecided position, so that little is read past
        // the stop (about one position of the benchmark's slices; several
        // when a position's slice is a single tile).
        while (dpos < ndec && (stop < 0 || !early)) {
            bool progress = false;
            const int lim_t = early ? min(total1, sh.tstart[dpos + 1] + kLookTiles) : total1;
            if (it_prod < lim_t && !*reinterpret_cast<volatile int*>(&sh.timeout)) {
                // lane l looks at tile it_prod + l; the leading run of tiles that
                // may be read and whose slots are free is issued at once
                const int tt = it_prod + lane;
                bool ok = lane < kStages && tt < lim_t;
                if (ok && tt >= kStages) ok = mbar_test_wait(smem_u32(&sh.empty[tt % kStages]), ((tt / kStages) & 1) ^ 1);
                const int nn = __ffs(~__ballot_sync(full, ok)) - 1;
                if (lane < nn) issue_p1(tt, tt);
                if (nn > 0) {
                    it_prod += nn;
                    progress = true;
                }
            }
            if (ppos < ndec && __all_sync(full, mbar_test_wait(smem_u32(&sh.cbar[ppos]), 0))) {
                // the CTA's four consumer warps have folded position ppos:
                // merge their partials and push the CTA's into every CTA
                const volatile Partial* wp = wpart + ppos * kConsumerWarps;
                Partial q{-INFINITY, 0.0f, 0x7fffffff, 0};
                if (lane < kConsumerWarps) {
                    q.m = wp[lane].m;
                    q.s = wp[lane].s;
                    q.arg = wp[lane].arg;
                    q.flags = wp[lane].flags;
                }
                const int F = static_cast<int>(__reduce_or_sync(full, static_cast<unsigned>(q.flags)));
                float M, S = 0.0f;
                int A = 0x7fffffff;
                if (greedy) {
                    float mv = q.m;
                    int ar = q.arg;
                    for (int off = 2; off > 0; off >>= 1) {
                        const float m2 = __shfl_xor_sync(full, mv, off);
                        const int a2 = __shfl_xor_sync(full, ar, off);
                        merge_arg(mv, ar, m2, a2);
                    }
                    M = __shfl_sync(full, mv, 0);
                    A = __shfl_sync(full, ar, 0);
                } else {
                    M = warp_max_f32(q.m);
                    float tt = ms_term(q.m, q.s, M, c);
                    for (int off = 2; off > 0; off >>= 1) tt += __shfl_xor_sync(full, tt, off);
                    S = __shfl_sync(full, tt, 0);  // lanes 0..3 hold the sum
                }
                if (lane < static_cast<int>(C))
                    st_async_v4(map_rank(smem_u32(&allpart[ppos * C + rank]), lane), __float_as_uint(M),
                                __float_as_uint(S), static_cast<uint32_t>(A), static_cast<uint32_t>(F),
                                map_rank(smem_u32(&sh.pbar[ppos]), lane));
                ++ppos;
                progress = true;
            }
            // (a plain test first: the cluster-scope acquire is taken only once
            // the phase is seen complete)
            if (__all_sync(full, mbar_test_wait(smem_u32(&sh.pbar[dpos]), 0)) &&
                __all_sync(full, mbar_test_wait_cluster(smem_u32(&sh.pbar[dpos]), 0))) {
                // position i: merge the C partials (lane r holds CTA r's), then its test
                const int i = dpos;
                const Partial pr = lane < static_cast<int>(C) ? allpart[i * C + lane]
                                                             : Partial{-INFINITY, 0.0f, 0x7fffffff, 0};
                const int F = static_cast<int>(__reduce_or_sync(full, static_cast<unsigned>(pr.flags)));
                float M, S = 0.0f;
                int A = 0x7fffffff;
                if (greedy) {
                    float mv = pr.m;
                    int ar = pr.arg;
                    for (int off = 16; off > 0; off >>= 1) {
                        const float m2 = __shfl_xor_sync(full, mv, off);
                        const int a2 = __shfl_xor_sync(full, ar, off);
                        merge_arg(mv, ar, m2, a2);
                    }
                    M = __shfl_sync(full, mv, 0);
                    A = __shfl_sync(full, ar, 0);
                    if (A == 0x7fffffff) A = 0;  // every value is -inf: index 0
                } else {
                    M = warp_max_f32(pr.m);
                    float tt = ms_term(pr.m, pr.s, M, c);
                    for (int off = 16; off > 0; off >>= 1) tt += __shfl_xor_sync(full, tt, off);
                    S = tt;
                }
                const int x = __shfl_sync(full, xi, i);
                const float uu = __shfl_sync(full, u0, i), lx = __shfl_sync(full, Lx, i), qq = __shfl_sync(full, qx, i);
                int err = 0;
                bool stp = true;
                float p = 0.0f;
                if (F & 2) err |= ST_TIMEOUT;
                if (a.parents) {
                    stp = false;  // a tree: every node is decided at the end
                } else if (greedy) {
                    if (F & 1) err |= ST_NONFINITE;
                    if (i < k && (x < 0 || x >= V)) err |= ST_TOKEN;
                    stp = (err != 0) || i == k || x != A;
                } else {
                    if (!(isfinite(M) && isfinite(S))) err |= ST_NONFINITE;
                    if (i < k) {
                        if (x < 0 || x >= V) err |= ST_TOKEN;
                        if (!(uu >= 0.0f && uu < 1.0f)) err |= ST_UNIFORM;
                        if (x >= 0 && x < V && !(qq >= 0.0f && qq <= FLT_MAX)) err |= ST_QBAD;
                        if (!err) {
                            // p_i(x_i) with the double-float exponential (a masked
                            // entry, logit -inf, has p = 0)
                            RowConst rc;
                            rc.M = M;
                            rc.s1 = S;
                            rc.thr = 0.0f;
                            rc.ch = sh.c_hi;
                            rc.cl = sh.c_lo;
                            p = df_val(exact_weight<BF16>(lx, 0.0f, MODE_BONUS, rc, df_make(0.0f), sh.exp2tab)) / S;
                            const float rho = fminf(1.0f, p / fmaxf(qq, 1e-12f));
                            stp = !(uu < rho);
                        }
                    }
                }
                if (lane == 0) {
                    sh.posM[i] = M;
                    sh.posS[i] = S;
                    sh.posA[i] = A;
                    sh.posF[i] = F;
                    sh.posE[i] = err;
                    sh.posP[i] = p;
                }
                if (stp && stop < 0) stop = i;
                ++dpos;
                progress = true;
            }
            if (progress) {
                idle = 0;
                t0 = 0;
                continue;
            }
            bool give = ++idle >= polls;
            if ((idle & 255) == 255) {
                const unsigned long long tn = gtimer();
                if (t0 == 0)
                    t0 = tn;
                else if (tn - t0 > kWaitNs)
                    give = true;
            }
            if (__any_sync(full, give)) {
                gave_up = true;
                break;
            }
        }
        if (gave_up) {
            // a CTA's partials never came: the undecided positions end the row
            if (lane == 0) atomicOr(&sh.timeout, 1);
            if (lane >= dpos && lane <= k) {
                sh.posM[lane] = -INFINITY;
                sh.posS[lane] = 0.0f;
                sh.posA[lane] = 0;
                sh.posF[lane] = 2;
                sh.posE[lane] = ST_TIMEOUT;
                sh.posP[lane] = 0.0f;
            }
            if (stop < 0) stop = dpos;
        }
        if (lane == 0) {
            *reinterpret_cast<volatile int*>(&sh.p1_end) = it_prod;  // no pass-1 copy is issued after this
            __threadfence_block();
            *reinterpret_cast<volatile int*>(&sh.stop_pos) = stop >= 0 ? stop : k;
            if (!gave_up && it_prod < total1) {
                // The consumers go on to stage use it_prod, which is never filled:
                // complete its phase without data (once its slot's previous use
                // is released, so that the phase is that use's), which wakes
                // them at once; they see it_prod >= p1_end and stop.
                const int slot = it_prod % kStages;
                if (it_prod < kStages ||
                    mbar_wait_bounded(smem_u32(&sh.empty[slot]), ((it_prod / kStages) & 1) ^ 1, polls))
                    mbar_arrive(smem_u32(&sh.full[slot]));
            }
        }
        __syncwarp();
        cluster_wait();
    } else {
        int t = 0;
        bool bail = false;    // a wait gave up
        int reported = 0;     // positions this warp has reported
        // Report this warp's partial of position i to the producer warp, which
        // merges the CTA's four and pushes the result to the cluster.
        auto report = [&](int i, Partial P) {
            if (lane == 0) {
                wpart[i * kConsumerWarps + warp] = P;
                mbar_arrive(smem_u32(&sh.cbar[i]));  // release: the store above is seen with the phase
            }
            __syncwarp();
        };
        // the first stopping position, once the producer has decided it (-1
        // before); the same value in every lane
        auto stop_now = [&]() { return __shfl_sync(full, *reinterpret_cast<volatile int*>(&sh.stop_pos), 0); };
        for (int i = 0; i <= k && t_ok; ++i) {
            const int sp = stop_now();
            bool skip = early && sp >= 0 && i > sp;  // past the stop: copies landed are let go unread
            float m = -INFINITY, s = 0.0f;  // sampled state
            int arg = 0x7fffffff;           // greedy state (m holds the best value)
            bool nan_seen = false;
            const long long row_e0 = (static_cast<long long>(b) * (k + 1) + i) * V + v0;
            const int h = sh.head[i];
            const int ntiles = sh.tstart[i + 1] - sh.tstart[i];
            const int interior = sh.nbytes[i] / esz;

            auto scalar_elem = [&](int rel) {
                const float l = load_logit(a.logits, row_e0 + rel, BF16);
                if (greedy) {
                    if (l != l) nan_seen = true;
                    if (l > m) {
                        m = l;
                        arg = static_cast<int>(v0 + rel);
                    }
                } else {
                    online_add(m, s, l, c);
                }
            };
            if (tid == 0 && !skip)
                for (int e = 0; e < h; ++e) scalar_elem(e);
            __syncwarp();  // reconverge before the tile loop's warp-wide steps

            bool ended = false;
            for (int lt = 0; lt < ntiles; ++lt, ++t, next_stage()) {
                // 0: the stage is full; 1: pass 1 ended before issuing it; 2: a wait gave up
                int r = 2;
                {
                    unsigned long long w0 = 0;
                    for (uint32_t it = 0; it < polls; ++it) {
                        if (mbar_try_wait(smem_u32(&sh.full[c_slot]), c_phase)) {
                            // a phase completed without data marks the end of pass 1
                            r = t >= *reinterpret_cast<volatile int*>(&sh.p1_end) ? 1 : 0;
                            break;
                        }
                        if (t >= *reinterpret_cast<volatile int*>(&sh.p1_end)) {
                            r = 1;
                            break;
                        }
                        if (*reinterpret_cast<volatile int*>(&sh.timeout)) break;
                        if ((it & 255) == 255) {
                            const unsigned long long tn = gtimer();
                            if (w0 == 0)
                                w0 = tn;
                            else if (tn - w0 > kWaitNs)
                                break;
                        }
                    }
                }
                // the warp agrees on the outcome: lanes that went different ways
                // here would meet the full-mask shuffles below apart
                r = __reduce_max_sync(full, r);
                if (r == 1) {
                    ended = true;
                    break;
                }
                if (r == 2) {
                    if (lane == 0) atomicOr(&sh.timeout, 1);
                    bail = true;
                    break;
                }
                const int bytes = min(kTileBytes, sh.nbytes[i] - lt * kTileBytes);
                const int nch = bytes >> 4;
                const uint32_t tile = smem_u32(ring + c_slot * kTileBytes);
                if (early && !skip) {
                    const int sp2 = stop_now();
                    skip = sp2 >= 0 && i > sp2;
                }
                if (skip) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sh.empty[c_slot]));
                    continue;
                }
                constexpr int kPer = kTileBytes / 16 / kConsumers;  // 16-byte chunks per thread
                uint4 w[kPer];
                if (nch == kTileBytes / 16) {  // a full tile (all but a position's last)
#pragma unroll
                    for (int r2 = 0; r2 < kPer; ++r2) w[r2] = ld_shared_v4(tile + (tid + r2 * kConsumers) * 16);
                } else {
#pragma unroll
                    for (int r2 = 0; r2 < kPer; ++r2) {
                        const int ch = tid + r2 * kConsumers;
                        if (ch < nch) {
                            w[r2] = ld_shared_v4(tile + ch * 16);
                        } else if (BF16) {
                            w[r2] = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
                        } else {
                            const uint32_t ni = __float_as_uint(-INFINITY);
                            w[r2] = make_uint4(ni, ni, ni, ni);
                        }
                    }
                }
                __syncwarp();  // the data is in registers: release the stage
                if (lane == 0) mbar_arrive(smem_u32(&sh.empty[c_slot]));
                const long long tile_e0 = v0 + h + static_cast<long long>(lt) * (kTileBytes / esz);
                p1_fold_tile<BF16>(w, greedy, c, tile_e0, tid, m, s, arg, nan_seen);
            }
            if (ended || bail) break;
            if (skip) continue;
            if (tid == 0)
                for (int e = h + interior; e < n; ++e) scalar_elem(e);
            __syncwarp();  // a diverged warp makes every shuffle below slow

            // warp reduction of this position's partial
            if (greedy) {
                for (int off = 16; off > 0; off >>= 1) {
                    const float m2 = __shfl_xor_sync(full, m, off);
                    const int a2 = __shfl_xor_sync(full, arg, off);
                    merge_arg(m, arg, m2, a2);
                }
                nan_seen = __any_sync(full, nan_seen);
            } else {
                // the warp's maximum, every lane's sum brought to it, then the total
                const float Mw = warp_max_f32(m);
                float sw = ms_term(m, s, Mw, c);
                for (int off = 16; off > 0; off >>= 1) sw += __shfl_xor_sync(full, sw, off);
                m = Mw;
                s = sw;
            }
            report(i, Partial{m, s, arg, nan_seen ? 1 : 0});
            reported = i + 1;
        }
        // a wait that gave up: the positions this warp has not reported are
        // reported as timed out, so that no CTA of the cluster waits for them
        if (bail)
            for (int i = reported; i <= k; ++i) report(i, Partial{-INFINITY, 0.0f, 0x7fffffff, 2});
        cluster_wait();
    }
    __syncthreads();  // pass 1 is over: no stage is read any more
    if (sh.timeout != 0 && producer && lane == 0) {
        // no bulk copy may outlive the wait that gave up on it: wait (bounded)
        // for the last use of every stage that was issued
        for (int it = max(0, it_prod - kStages); it < it_prod; ++it)
            mbar_wait_bounded(smem_u32(&sh.full[it % kStages]), (it / kStages) & 1, polls);
    }

    // ---------------------------------------------------------------- the row's outcome
    // Every CTA decided from the same partials, so all reach the same
    // outcome unless a wait gave up somewhere; each pushes its own to every
    // CTA, and a disagreement ends the row with a timeout.  After the cluster
    // barrier below no CTA touches another's shared memory on this path.
    int oj = 0, ost = ST_TEMP;  // this CTA's outcome: stop position and status
    if (producer) {
        if (a.parents) {
            ost = 0;
            if (lane <= k && (sh.posF[lane] & 2)) ost = ST_TIMEOUT;
            ost = static_cast<int>(__reduce_or_sync(full, static_cast<unsigned>(ost)));
        } else if (t_ok) {
            oj = stop;
            ost = sh.posE[oj];
            if (!greedy && !(ost & ST_ERRMASK)) {
                const float uj = __shfl_sync(full, u1, oj);
                if (!(uj >= 0.0f && uj < 1.0f)) ost |= ST_UNIFORM;
            }
        }
        if (lane < static_cast<int>(C))
            st_cluster_v2(map_rank(smem_u32(&sh.views[rank]), lane), static_cast<uint32_t>(oj), static_cast<uint32_t>(ost));
    }
    cluster_sync();  // #1: every CTA's outcome is visible
    if (producer) {
        const bool same = lane >= static_cast<int>(C) || (sh.views[lane].x == oj && sh.views[lane].y == ost);
        const bool agreed = __all_sync(full, same);
        const bool have = lane <= k && t_ok;
        const float M = have ? sh.posM[lane] : 0.0f;
        const float S = have ? sh.posS[lane] : 0.0f;
        const int A = have ? sh.posA[lane] : 0;
        if (a.parents) {
            // a draft tree (all rows greedy): rank 0 writes the outputs
            const int F = (have ? sh.posF[lane] : 0) | (agreed ? 0 : 2);
            const int terr = tree_greedy_warp(a, b, k, lane, xi, pi, A, F, rank == 0);
            if (lane == 0) {
                sh.status = terr;
                sh.j = 0;
            }
            if (rank == 0 && lane <= k && a.dbg_max) a.dbg_max[static_cast<long long>(b) * (k + 1) + lane] = M;
        } else {
            const int j = agreed ? oj : 0;
            const int st = agreed ? ost : ST_TIMEOUT;
            const float Mj = __shfl_sync(full, M, j);
            const float Sj = __shfl_sync(full, S, j);
            const int Aj = __shfl_sync(full, A, j);
            const float ujj = __shfl_sync(full, u1, j);
            if (lane == 0) {
                sh.uj = ujj;
                sh.j = j;
                sh.status = st;
                sh.Mj = Mj;
                sh.sj = Sj;
                sh.mode = (j < k) ? (a.q ? MODE_RESIDUAL : MODE_ONEHOT) : MODE_BONUS;
                if (t_ok && !greedy && !(st & ST_ERRMASK)) {
                    // the stop row's pass-2 geometry, set here so that one block
                    // barrier publishes it with the decision
                    const bool resid = j < k && a.q;
                    const long long lrow_j = (static_cast<long long>(b) * (k + 1) + j) * V;
                    const float* qrow_j = a.q ? a.q + (static_cast<long long>(b) * k + (j < k ? j : 0)) * V : nullptr;
                    sh.thr = kLargeP * Sj;
                    // bulk copies need 16-byte aligned starts and sizes: both rows
                    // aligned at the slice start, and whole groups of 8 entries
                    const bool la = (reinterpret_cast<uintptr_t>(lg + (lrow_j + v0) * esz) & 15) == 0;
                    const bool qa = qrow_j && (reinterpret_cast<uintptr_t>(qrow_j + v0) & 15) == 0;
                    sh.p2fast = la && (!resid || (qa && !a.q_host)) && (n % kChunk) == 0;
                    sh.ntiles2 = (n + kP2Elems - 1) / kP2Elems;
                    // pass-2 slots: [q (residual rows)][logits], one tile each
                    sh.loff2 = resid ? kP2Elems * 4 : 0;
                    sh.stride2 = sh.loff2 + kP2Elems * esz;
                    sh.nslots2 = min(kStages2, kRingBytes / sh.stride2);  // at least 5: the consumers step 4 tiles at a time
                }
            }
            if (lane <= k) sh.xs[lane] = xi;
            // rank 0 writes debug values and, for greedy or failed rows, the outputs
            if (rank == 0) {
                if (have) {
                    if (a.dbg_max) a.dbg_max[static_cast<long long>(b) * (k + 1) + lane] = M;
                    if (a.dbg_sumexp) a.dbg_sumexp[static_cast<long long>(b) * (k + 1) + lane] = greedy ? 0.0f : S;
                    if (lane < k) {
                        const bool xok = xi >= 0 && xi < V;
                        if (a.dbg_p) a.dbg_p[static_cast<long long>(b) * k + lane] = (greedy || !xok) ? 0.0f : sh.posP[lane];
                        if (a.dbg_q) a.dbg_q[static_cast<long long>(b) * k + lane] = (greedy || !xok) ? 0.0f : qx;
                    }
                }
                if (lane == 0 && a.dbg_resid) a.dbg_resid[b] = 0.0f;
                if (greedy || !t_ok || (st & ST_ERRMASK)) {
                    const bool bad = (st & ST_ERRMASK) != 0;
                    if (lane <= k) {
                        int tok = -1;
                        if (!bad) tok = lane < j ? xi : (lane == j ? Aj : -1);
                        a.out_tokens[static_cast<long long>(b) * (k + 1) + lane] = tok;
                    }
                    if (lane == 0) {
                        a.num_accepted[b] = bad ? 0 : j;
                        if (a.row_status) a.row_status[b] = st;
                    }
                }
            }
        }
    }
    __syncthreads();
    const bool sample = t_ok && !greedy && !(sh.status & ST_ERRMASK);
    if (!sample) return;

    // ---------------------------------------------------------------- pass 2
    const int j = sh.j;
    const long long lrow = (static_cast<long long>(b) * (k + 1) + j) * V;
    const float* qrow = a.q ? a.q + (static_cast<long long>(b) * k + (j < k ? j : 0)) * V : nullptr;
    RowConst rc;
    rc.M = sh.Mj;
    rc.s1 = sh.sj;
    rc.thr = sh.thr;
    rc.ch = sh.c_hi;
    rc.cl = sh.c_lo;
    const bool p2fast = sh.p2fast != 0;
    const int ntiles2 = sh.ntiles2;
    const int loff2 = sh.loff2, stride2 = sh.stride2, S2 = sh.nslots2;
    int g2 = 0;  // pass-2 tiles issued / consumed so far (both sweeps): tile g uses slot g % S2
    int mode = sh.mode;

    // one stop-row entry by tile-local index, from global memory (the search)
    auto fetch1 = [&](int e0, int idx, float& l, float& q) {
        l = load_logit(a.logits, lrow + v0 + e0 + idx, BF16);
        if (mode == MODE_ONEHOT && v0 + e0 + idx == sh.xs[j]) l = -INFINITY;  // the draft token: q = 1
        q = mode == MODE_RESIDUAL ? __ldg(qrow + v0 + e0 + idx) : 0.0f;
    };
    SweepConst K;
    K.MM = pack2(rc.M, rc.M);
    K.CH = pack2(rc.ch, rc.ch);
    K.NCH = pack2(-rc.ch, -rc.ch);
    K.CL = pack2(rc.cl, rc.cl);
    K.LN2 = pack2(kLn2, kLn2);
    K.NS1 = pack2(-rc.s1, -rc.s1);
    K.thr = rc.thr;

    // Bf16 rows: the exact e of every bf16 value that can be a large entry,
    // tabulated once in the ring's unused tail, so that large entries look
    // it up instead of evaluating exp2dd.  Positive logits only (their bf16
    // bit patterns order like the values); lmin sits below every logit whose
    // estimate can exceed thr (a margin of 1/16 in the exponent).
    int tab_base = 0, tab_n = 0;
    const float2* etab = reinterpret_cast<const float2*>(ring + S2 * stride2);
    if (BF16 && !producer) {
        const int cap = (kRingBytes - S2 * stride2) / static_cast<int>(sizeof(float2));
        const float lmin = rc.M + (__log2f(rc.thr) - 0.0625f) / rc.ch;
        if (rc.M > 0.0f && lmin > 0.0f) {
            const int hb = static_cast<int>(__float_as_uint(rc.M) >> 16);
            const int lb = static_cast<int>(__float_as_uint(lmin) >> 16);
            if (hb >= lb && hb - lb + 1 <= cap) {
                tab_base = lb;
                tab_n = hb - lb + 1;
            }
        }
        float2* wtab = reinterpret_cast<float2*>(ring + S2 * stride2);
        for (int i = tid; i < tab_n; i += kConsumers) {
            const df e = precise_e<BF16>(__uint_as_float(static_cast<uint32_t>(tab_base + i) << 16), rc, sh.exp2tab);
            wtab[i] = make_float2(e.hi, e.lo);
        }
        consumers_sync();
    }

    for (;;) {
        df te = df_make(0.0f);  // this thread's sum of e (residual mode)
        bool qbad = false;
        if (producer) {
            if (p2fast) {
                // the ring's last generic-proxy reads (pass 1) are ordered
                // before these async-proxy writes by the block barrier above
                fence_proxy_async_smem();
                // Lane l looks at tile t2 + l (tile g = g2 + t2 + l: slot g % S2,
                // phase (g / S2) & 1); the leading run of tiles whose slots are
                // free is issued at once, one tile a lane: a lane waits about as
                // long to issue one bulk copy as to issue several in one step.
                uint32_t idle2 = 0;
                unsigned long long w0 = 0;
                for (int t2 = 0; t2 < ntiles2;) {
                    if (*reinterpret_cast<volatile int*>(&sh.timeout)) break;
                    const int tt = t2 + lane;
                    const int g = g2 + tt;
                    const bool ok = lane < S2 && tt < ntiles2 &&
                                    (g < S2 || mbar_test_wait(smem_u32(&sh.empty2[g % S2]), ((g / S2) & 1) ^ 1));
                    const int nn = __ffs(~__ballot_sync(full, ok)) - 1;
                    if (lane < nn) {
                        const int slot = g % S2;
                        const int e0 = tt * kP2Elems;
                        const int cnt = min(kP2Elems, n - e0);
                        const uint32_t bar = smem_u32(&sh.full2[slot]);
                        const uint32_t dst = smem_u32(ring + slot * stride2);
                        const uint32_t lbytes = static_cast<uint32_t>(cnt * esz);
                        const uint32_t qbytes = mode == MODE_RESIDUAL ? static_cast<uint32_t>(cnt * 4) : 0u;
                        mbar_arrive_expect_tx(bar, lbytes + qbytes);
                        bulk_g2s(dst + loff2, lg + (lrow + v0 + e0) * esz, lbytes, bar);
                        if (qbytes) bulk_g2s(dst, qrow + v0 + e0, qbytes, bar);
                    }
                    t2 += nn;
                    if (nn > 0) {
                        idle2 = 0;
                        w0 = 0;
                        continue;
                    }
                    if (lane == 0) {  // sleep until the next tile's slot is free (briefly)
                        const int g = g2 + t2;
                        mbar_try_wait_hint(smem_u32(&sh.empty2[g % S2]), ((g / S2) & 1) ^ 1, kNapNs);
                    }
                    __syncwarp();
                    bool give = ++idle2 >= kWaitPolls;
                    if ((idle2 & 255) == 255) {
                        const unsigned long long tn = gtimer();
                        if (w0 == 0)
                            w0 = tn;
                        else if (tn - w0 > kWaitNs)
                            give = true;
                    }
                    if (__any_sync(full, give)) {
                        if (lane == 0) atomicOr(&sh.timeout, 1);
                        break;
                    }
                }
            }
            __syncwarp();
        } else {
            // one warp per tile of 1024 entries; lane l owns entries [32l, 32l+32)
            const int rot = (lane + (lane >> 3)) & 7;
            int slot = (g2 + warp) % S2, phase = ((g2 + warp) / S2) & 1;  // advanced by 4 tiles a step (S2 > 4)
            for (int t2 = warp; t2 < ntiles2; t2 += kConsumerWarps) {
                const int e0 = t2 * kP2Elems;
                const int cnt = min(kP2Elems, n - e0);
                const int my0 = lane * kLaneEntries;
                unsigned char* stage = ring + (p2fast ? slot : warp) * stride2;
                const int my_slot = slot;
                slot += kConsumerWarps;
                const int my_phase = phase;
                if (slot >= S2) {
                    slot -= S2;
                    phase ^= 1;
                }
                bool ok = true;
                if (p2fast) {
                    ok = __all_sync(0xffffffffu, !sh.timeout &&
                                                     mbar_wait_bounded(smem_u32(&sh.full2[my_slot]), my_phase, kWaitPolls));
                    if (!ok && lane == 0) atomicOr(&sh.timeout, 1);
                } else {
                    // unaligned rows: the warp stages its own tiles in slot
                    // `warp` with plain loads; entries past the slice are masked
                    for (int idx = lane; idx < kP2Elems; idx += 32) {
                        const bool in = idx < cnt;
                        const long long gi = lrow + v0 + e0 + idx;
                        if (BF16)
                            reinterpret_cast<uint16_t*>(stage + loff2)[idx] =
                                in ? __ldg(reinterpret_cast<const unsigned short*>(a.logits) + gi) : uint16_t(0xff80u);
                        else
                            reinterpret_cast<float*>(stage + loff2)[idx] =
                                in ? __ldg(reinterpret_cast<const float*>(a.logits) + gi) : -INFINITY;
                        if (mode == MODE_RESIDUAL)
                            reinterpret_cast<float*>(stage)[idx] = in ? __ldg(qrow + v0 + e0 + idx) : 0.0f;
                    }
                }
                if (mode == MODE_ONEHOT && ok && lane == 0) {
                    // one-hot drafts: the draft token's entry weighs nothing (q = 1 there)
                    const long long rel = static_cast<long long>(sh.xs[j]) - v0 - e0;  // j < k here
                    if (rel >= 0 && rel < cnt) {
                        if (BF16)
                            reinterpret_cast<uint16_t*>(stage + loff2)[rel] = uint16_t(0xff80u);
                        else
                            reinterpret_cast<float*>(stage + loff2)[rel] = -INFINITY;
                        fence_proxy_async_smem();  // before the slot's next bulk copy
                    }
                }
                __syncwarp();
                LaneAcc A;
                lane_init(A);
                df bw = df_make(0.0f), be = df_make(0.0f);  // large entries: weights, e
                if (ok) {
                    const unsigned char* ls = stage + loff2 + my0 * esz;
                    const float* qs = reinterpret_cast<const float*>(stage) + my0;
                    const int nvl = p2fast ? max(0, min(kLaneEntries, cnt - my0)) : kLaneEntries;
                    if (mode == MODE_RESIDUAL)
                        sweep_lane<BF16, true>(A, ls, qs, sh.lpad, sh.qpad, rot, nvl, K);
                    else
                        sweep_lane<BF16, false>(A, ls, qs, sh.lpad, sh.qpad, rot, nvl, K);
                    // large entries, each lane its own, two at a time in packed
                    // arithmetic (the warp runs as many rounds as its busiest
                    // lane needs); two interleaved pair sums, joined at the end
                    f2 BWH = pack2(0.0f, 0.0f), BWL = BWH, BEH = BWH, BEL = BWH;
                    for (uint32_t m = A.large; m;) {
                        const int bit0 = __ffs(m) - 1;
                        m &= m - 1;
                        const bool two = m != 0;
                        const int bit1 = two ? __ffs(m) - 1 : bit0;
                        m &= m - 1;
                        f2 EH, EL;
                        bool tabbed = false;
                        if (BF16) {
                            const uint16_t* l16 = reinterpret_cast<const uint16_t*>(ls);
                            const uint32_t w0 = l16[bit0], w1 = l16[bit1];
                            const uint32_t i0 = w0 - static_cast<uint32_t>(tab_base);
                            const uint32_t i1 = w1 - static_cast<uint32_t>(tab_base);
                            tabbed = i0 < static_cast<uint32_t>(tab_n) && i1 < static_cast<uint32_t>(tab_n);
                            if (tabbed) {
                                const float2 t0 = etab[i0], t1 = etab[i1];
                                EH = pack2(t0.x, t1.x);
                                EL = pack2(t0.y, t1.y);
                            } else {
                                precise_e_x2(pack2(bf16_lo(w0), bf16_lo(w1)), rc, sh.exp2tab, EH, EL);
                            }
                        } else {
                            const float* l32 = reinterpret_cast<const float*>(ls);
                            precise_e_x2(pack2(l32[bit0], l32[bit1]), rc, sh.exp2tab, EH, EL);
                        }
                        if (!two) {  // a lone last entry: the second lane weighs nothing
                            float h0, h1, l0, l1;
                            unpack2(EH, h0, h1);
                            unpack2(EL, l0, l1);
                            EH = pack2(h0, 0.0f);
                            EL = pack2(l0, 0.0f);
                        }
                        if (mode == MODE_RESIDUAL) {
                            // e - s1 q: the product exact through one fma, then a two-sum
                            const float q0 = qs[bit0], q1 = two ? qs[bit1] : 0.0f;
                            const f2 Q = pack2(q0, q1);
                            const f2 NP = mul2(pack2(-rc.s1, -rc.s1), Q);
                            const f2 PL = fma2(pack2(rc.s1, rc.s1), Q, NP);
                            const f2 RH = add2(EH, NP);
                            const f2 BB = sub2(RH, EH);
                            const f2 RL = add2(add2(sub2(EH, sub2(RH, BB)), sub2(NP, BB)), sub2(EL, PL));
                            float rh0, rh1, rl0, rl1;
                            unpack2(RH, rh0, rh1);
                            unpack2(RL, rl0, rl1);
                            const bool pos0 = rh0 + rl0 > 0.0f, pos1 = rh1 + rl1 > 0.0f;
                            df2_add_pair(BWH, BWL, pack2(pos0 ? rh0 : 0.0f, pos1 ? rh1 : 0.0f),
                                         pack2(pos0 ? rl0 : 0.0f, pos1 ? rl1 : 0.0f));
                            A.q += (pos0 ? q0 : 0.0f) + (pos1 ? q1 : 0.0f);
                            df2_add_pair(BEH, BEL, EH, EL);
                        } else {
                            df2_add_pair(BWH, BWL, EH, EL);
                        }
                    }
                    {
                        float h0, h1, l0, l1;
                        unpack2(BWH, h0, h1);
                        unpack2(BWL, l0, l1);
                        bw = df_sum(df{h0, l0}, df{h1, l1});
                        unpack2(BEH, h0, h1);
                        unpack2(BEL, l0, l1);
                        be = df_sum(df{h0, l0}, df{h1, l1});
                    }
                    __syncwarp();
                    if (mode == MODE_RESIDUAL) {
                        // a NaN or infinite sum, or a set sign bit (-0 is a
                        // valid q), sends the lane through an exact check
                        float qa0, qa1;
                        unpack2(A.qa, qa0, qa1);
                        if ((A.qor & 0x80000000u) || !(fabsf(qa0 + qa1) <= FLT_MAX)) {
                            for (int i = 0; i < nvl; ++i) {
                                const float q = qs[i];
                                qbad |= !(q >= 0.0f && q <= FLT_MAX);
                            }
                        }
                        __syncwarp();
                    }
                    if (p2fast && lane == 0) mbar_arrive(smem_u32(&sh.empty2[my_slot]));
                }
                float wh, eh, wlo, elo;
                unpack2(A.wh, wh, eh);
                unpack2(A.wl, wlo, elo);
                const df lw = df_sum(df{wh, wlo}, bw);
                sh.lane_hi[t2][lane] = lw.hi;
                sh.lane_lo[t2][lane] = lw.lo;
                sh.lane_q[t2][lane] = A.q;
                te = df_sum(te, df_sum(df{eh, elo}, be));
            }
            // totals of this warp's tiles, four tiles at a time: lane 8 i + g
            // adds lane sums 4 g .. 4 g + 3 of the group's tile i (in a
            // lane-rotated order: conflict-free banks), then the tile's eight
            // lanes combine over three shuffles
            __syncwarp();
            for (int tb = warp; tb < ntiles2; tb += 4 * kConsumerWarps) {
                const int tt = tb + (lane >> 3) * kConsumerWarps;
                const int g = lane & 7;
                df v = df_make(0.0f);
                float vq = 0.0f;
                if (tt < ntiles2) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int e = 4 * g + ((i + (lane >> 3)) & 3);
                        v = df_sum(v, df{sh.lane_hi[tt][e], sh.lane_lo[tt][e]});
                        vq += sh.lane_q[tt][e];
                    }
                }
#pragma unroll
                for (int off = 1; off < 8; off <<= 1) {
                    v = df_sum(v, df{__shfl_xor_sync(0xffffffffu, v.hi, off), __shfl_xor_sync(0xffffffffu, v.lo, off)});
                    vq += __shfl_xor_sync(0xffffffffu, vq, off);
                }
                if (g == 0 && tt < ntiles2) {
                    sh.tile_hi[tt] = v.hi;
                    sh.tile_lo[tt] = v.lo;
                    sh.tile_q[tt] = vq;
                }
            }
            __syncwarp();
        }
        // CTA totals: weights, e (residual mode), q over positive residuals
        const df tw = df_warp_total(te);
        const int any_qbad = __syncthreads_or(qbad ? 1 : 0);
        if (lane == 0 && !producer) {
            sh.wred_hi[warp] = tw.hi;
            sh.wred_lo[warp] = tw.lo;
        }
        __syncthreads();
        if (warp == 0) {
            const bool in = lane < ntiles2;
            const df Wc = df_warp_total(in ? df{sh.tile_hi[lane], sh.tile_lo[lane]} : df_make(0.0f));
            float vq = in ? sh.tile_q[lane] : 0.0f;
            for (int off = 16; off > 0; off >>= 1) vq += __shfl_down_sync(0xffffffffu, vq, off);
            const df Ec = df_warp_total(lane < kConsumerWarps ? df{sh.wred_hi[lane], sh.wred_lo[lane]} : df_make(0.0f));
            // push this CTA's totals into every CTA of the cluster (lane r -> rank r)
            const uint32_t flags2 = static_cast<uint32_t>((any_qbad ? 1 : 0) | (sh.timeout ? 2 : 0));
            const df Wb = df_shfl(Wc, 0), Eb = df_shfl(Ec, 0);
            const float qb = __shfl_sync(0xffffffffu, vq, 0);
            if (lane < static_cast<int>(C)) {
                const uint32_t ra = map_rank(smem_u32(&sh.alltot[rank][0]), lane);
                st_cluster_v4(ra, __float_as_uint(Wb.hi), __float_as_uint(Wb.lo), __float_as_uint(Eb.hi),
                              __float_as_uint(Eb.lo));
                st_cluster_v2(ra + 16, __float_as_uint(qb), flags2);
            }
        }
        cluster_sync();  // #2: CTA totals visible
        if (warp == 0) {
            // lane r holds rank r's totals
            const bool has = lane < static_cast<int>(C);
            df wr = df_make(0.0f), er = df_make(0.0f);
            float qr = 0.0f;
            int fl = 0;
            if (has) {
                wr = df{sh.alltot[lane][0], sh.alltot[lane][1]};
                er = df{sh.alltot[lane][2], sh.alltot[lane][3]};
                qr = sh.alltot[lane][4];
                fl = static_cast<int>(__float_as_uint(sh.alltot[lane][5]));
            }
            __syncwarp();  // a diverged warp makes every shuffle below slow
            const df s_prec = df_shfl(df_warp_total(er), 0);
            const bool any_q = __any_sync(0xffffffffu, (fl & 1) != 0);
            const bool any_to = __any_sync(0xffffffffu, (fl & 2) != 0);
            const float delta = mode == MODE_RESIDUAL ? df_val(df_sum(s_prec, df_make(-rc.s1))) : 0.0f;
            wr = df_sum(wr, df_make(-delta * qr));
            const df Wt = df_shfl(df_warp_total(wr), 0);
            int bad = 0;
            if (any_to)
                bad = ST_TIMEOUT;
            else if (mode == MODE_RESIDUAL && any_q)
                bad = ST_QBAD;  // a draft probability of the residual row is NaN, negative or infinite
            if (bad) {
                if (lane == 0) sh.owner = -2;
                if (rank == 0 && lane <= k) a.out_tokens[static_cast<long long>(b) * (k + 1) + lane] = -1;
                if (rank == 0 && lane == 0) {
                    a.num_accepted[b] = 0;
                    if (a.row_status) a.row_status[b] = sh.status | bad;
                }
            } else if ((mode == MODE_RESIDUAL || mode == MODE_ONEHOT) && !(Wt.hi + Wt.lo > 0.0f)) {
                if (lane == 0) {
                    sh.mode = MODE_FALLBACK;
                    sh.owner = -1;
                }
            } else {
                const df target = df_mul_f(Wt, sh.uj);
                const df incl = df_warp_incl_scan(wr, lane);
                const df excl = df_sum(incl, df_neg(wr));
                const bool positive = has && (wr.hi + wr.lo > 0.0f);
                const unsigned hit =
                    __ballot_sync(0xffffffffu, positive && !df_less(target, excl) && df_less(target, incl));
                const unsigned pos = __ballot_sync(0xffffffffu, positive);
                const int owner = hit ? (__ffs(hit) - 1) : (pos ? 31 - __clz(pos) : 0);
                const df t_loc = df_sum(target, df_neg(df_shfl(excl, owner)));
                if (lane == 0) {
                    sh.owner = owner;
                    sh.t_hi = hit ? t_loc.hi : INFINITY;
                    sh.t_lo = hit ? t_loc.lo : 0.0f;
                    sh.delta = delta;
                    sh.sp_hi = s_prec.hi;
                    sh.sp_lo = s_prec.lo;
                    if (rank == 0 && a.dbg_resid && mode == MODE_RESIDUAL) a.dbg_resid[b] = df_val(Wt) / df_val(s_prec);
                    if (rank == 0 && a.dbg_resid && mode == MODE_ONEHOT) a.dbg_resid[b] = df_val(Wt) / rc.s1;
                }
            }
        }
        __syncthreads();
        if (sh.mode == MODE_FALLBACK && mode == MODE_RESIDUAL) {
            mode = MODE_FALLBACK;
            g2 += ntiles2;
            cluster_sync();  // peers are done reading this CTA's totals
            continue;
        }
        break;
    }

    // ---------------------------------------------------------------- search
    if (static_cast<int>(rank) == sh.owner && warp == 0) {
        const float delta = sh.delta;
        const df s_prec = df{sh.sp_hi, sh.sp_lo};
        df t = df{sh.t_hi, sh.t_lo};
        int st = sh.status;
        if (mode == MODE_FALLBACK) st |= ST_ZERO_RESIDUAL;
        // level 1: the tile (lane t holds tile t)
        const df vt = lane < ntiles2 ? df_sum(df{sh.tile_hi[lane], sh.tile_lo[lane]}, df_make(-delta * sh.tile_q[lane]))
                                     : df_make(0.0f);
        df ti = df_warp_incl_scan(vt, lane);
        df te2 = df_sum(ti, df_neg(vt));
        bool pz = vt.hi + vt.lo > 0.0f;
        unsigned hit = __ballot_sync(0xffffffffu, pz && !df_less(t, te2) && df_less(t, ti));
        int tile;
        if (hit) {
            tile = __ffs(hit) - 1;
        } else {
            const unsigned pos = __ballot_sync(0xffffffffu, pz);
            tile = pos ? 31 - __clz(pos) : 0;  // only through rounding at the top edge
            t = df_make(INFINITY);
        }
        const df base1 = df_shfl(te2, tile);
        // level 2: the lane's 32 entries within the tile
        const df vl = df_sum(df{sh.lane_hi[tile][lane], sh.lane_lo[tile][lane]}, df_make(-delta * sh.lane_q[tile][lane]));
        const df li = df_sum(base1, df_warp_incl_scan(vl, lane));
        const df le = df_sum(li, df_neg(vl));
        pz = vl.hi + vl.lo > 0.0f;
        hit = __ballot_sync(0xffffffffu, pz && !df_less(t, le) && df_less(t, li));
        int who;
        if (hit) {
            who = __ffs(hit) - 1;
        } else {
            const unsigned pos = __ballot_sync(0xffffffffu, pz);
            who = pos ? 31 - __clz(pos) : 0;
            t = df_make(INFINITY);
        }
        {
            // the segment's 32 entries, one per lane, with their exact weights
            const int e0 = tile * kP2Elems;
            const int cnt = min(kP2Elems, n - e0);
            const int idx = who * kLaneEntries + lane;
            float l = -INFINITY, q = 0.0f;
            if (idx < cnt) fetch1(e0, idx, l, q);
            const df we = exact_weight<BF16>(l, q, mode, rc, s_prec, sh.exp2tab);
            __syncwarp();
            const bool p = we.hi + we.lo > 0.0f;
            const df ci = df_sum(df_shfl(le, who), df_warp_incl_scan(we, lane));
            const unsigned ehit = __ballot_sync(0xffffffffu, p && df_less(t, ci));
            const unsigned epos = __ballot_sync(0xffffffffu, p);
            const int wl = ehit ? (__ffs(ehit) - 1) : (epos ? 31 - __clz(epos) : 0);
            if (lane == 0) write_sampled(a, b, k, j, static_cast<int>(v0 + e0 + who * kLaneEntries + wl), st, sh.xs);
        }
    }
    cluster_sync();  // #3: no CTA leaves while a peer may still read its totals
}

}  // namespace specv
