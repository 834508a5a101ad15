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
// after a rejection, the draft row q_j): it weighs every entry by
// max(0, p_j - q_j) (or p_k for the bonus), keeps sums per 256-entry block,
// and after a second exchange of CTA totals the CTA whose slice holds u * W
// rescans one block with one warp to find the token.
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

#include "exp2dd.cuh"
#include "ptx.cuh"

namespace specv {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kTileBytes = 8192;
constexpr int kStages = 4;
constexpr int kMaxK = 31;          // positions 0..k fit one warp
constexpr int kMaxSlice = 16384;   // elements of one position held by one CTA
constexpr int kChunk = 8;          // pass-2 entries per chunk
constexpr int kLaneEntries = 32;   // pass-2 entries per lane and tile (four chunks)
constexpr int kP2Elems = kLaneEntries * 32;  // pass-2 tile: 1024 entries, one warp
constexpr int kMaxP2Tiles = kMaxSlice / kP2Elems;
constexpr float kLargeP = 1e-5f;   // pass-2 entries with p above this use exp2dd
constexpr uint32_t kWaitPolls = 1u << 22;
constexpr float kLog2e = 1.44269504088896341f;

enum : int {
    ST_NONFINITE = 1,
    ST_TOKEN = 2,
    ST_UNIFORM = 4,
    ST_TEMP = 8,
    ST_ZERO_RESIDUAL = 16,
    ST_QBAD = 32,
    ST_TIMEOUT = 64,
    ST_ERRMASK = 1 | 2 | 4 | 8 | 32 | 64,
};

enum : int { MODE_RESIDUAL = 0, MODE_BONUS = 1, MODE_FALLBACK = 2 };

struct VerifyArgs {
    const void* logits;      // [B, k+1, V] bf16 or fp32
    const float* q;          // [B, k, V] (nullable when every row is greedy)
    const int32_t* x;        // [B, k]
    const float* u;          // [B, k+1, 2] (nullable when every row is greedy)
    const float* temp;       // [B] (nullable: every row greedy)
    int32_t* num_accepted;   // [B]
    int32_t* out_tokens;     // [B, k+1]
    int32_t* row_status;     // [B] (nullable)
    float* dbg_p;            // [B, k] (nullable)
    float* dbg_q;            // [B, k]
    float* dbg_max;          // [B, k+1]
    float* dbg_sumexp;       // [B, k+1]
    float* dbg_resid;        // [B]
    long long V;
    int B;
    int k;
    int slice;               // elements per CTA, a multiple of 64
};

struct Partial {
    float m;    // running max (sampled) / best value (greedy)
    float s;    // sum of exp((l - m) / T) (sampled)
    int arg;    // lowest index of the best value (greedy)
    int flags;  // bit 0: a NaN was seen (greedy); bit 1: a wait timed out
};

struct alignas(16) ClusterSmem {
    Partial wpart[kConsumerWarps][kMaxK + 1];
    alignas(16) Partial allpart[16][kMaxK + 1];  // every CTA's partials, pushed by each CTA of the cluster
    int tstart[kMaxK + 2];      // first pass-1 tile of each position
    int head[kMaxK + 1];        // unaligned leading elements of each position's slice
    int nbytes[kMaxK + 1];      // bytes of the 16-byte aligned interior
    unsigned long long full[kStages];
    unsigned long long empty[kStages];
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
    int xs[kMaxK + 1];          // draft tokens, for whoever writes the outputs
    int j, status, mode, owner, p2fast, ntiles2, timeout;
    float Mj, sj, thr, c_hi, c_lo, uj;
    float delta, sp_hi, sp_lo, t_hi, t_lo;
};
static_assert(sizeof(Partial) == 16, "Partial is pushed with one 16-byte store");
static_assert(offsetof(ClusterSmem, allpart) % 16 == 0, "16-byte remote stores need 16-byte aligned targets");
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

// SFU estimate of e = 2^((l - M) log2(e) / T), the exponent carried as a
// float pair (xh, xl) and folded back in to first order.
__device__ __forceinline__ float fast_e(float l, const RowConst& rc) {
    const float dh = l - rc.M;
    const float xh = dh * rc.ch;
    const float xl = fmaf(dh, rc.cl, fmaf(dh, rc.ch, -xh));
    const float ef = ex2(xh);
    return fmaf(ef, xl * kLn2, ef);
}

// e with exp2dd, as a pair (the exact difference l - M for fp32 logits).
template <bool BF16>
__device__ __forceinline__ df precise_e(float l, const RowConst& rc, const float2* tab) {
    float dh = l - rc.M, dl = 0.0f;
    if (!BF16) two_sum(l, -rc.M, dh, dl);
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

// Weight of one large entry with exp2dd: (w, q over a positive residual, e).
template <bool BF16>
__device__ __forceinline__ void large_weight(float l, float q, int md, const RowConst& rc, const float2* tab, df& w,
                                             float& wq, df& e) {
    e = precise_e<BF16>(l, rc, tab);
    if (md == MODE_RESIDUAL) {
        const df r = minus_sq(e, df_make(rc.s1), q);
        const bool pos = r.hi + r.lo > 0.0f;
        w = pos ? r : df_make(0.0f);
        wq = pos ? q : 0.0f;
    } else {
        w = e;
        wq = 0.0f;
    }
}

// A lane's 32 consecutive stop-row entries, summed per 8-entry chunk so that
// the sums can be walked in vocabulary order.  Weights are in e-units (the
// row's sum of exponentials times p): residual mode r = max(0, e - s1 q),
// bonus / fallback mode e.  Entries whose SFU estimate exceeds rc.thr are
// "large": their weight is recomputed with exp2dd.
struct Lane32 {
    float s[4];      // weights of the small entries, per chunk (entry order)
    float sq[4];     // q over positive residuals among them
    df big[4];       // weights of the large entries, per chunk (entry order)
    float bq[4];     // q over positive residuals among them
    df e;            // sum of e over the lane's entries (residual mode)
    uint32_t large;  // bit 8c+i: entry i of chunk c is large
};

__device__ __forceinline__ void lane32_init(Lane32& L) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        L.s[c] = 0.0f;
        L.sq[c] = 0.0f;
        L.big[c] = df_make(0.0f);
        L.bq[c] = 0.0f;
    }
    L.e = df_make(0.0f);
    L.large = 0;
}

// Small entries of chunk c (c is a run-time value: the chunks are visited in
// a lane-rotated order to spread shared-memory banks; the sums are stored by
// chunk).  nvalid: entries of the chunk inside the slice.  Branch-free.
__device__ __forceinline__ void lane32_fast8(Lane32& L, int c, const float* lv, const float* qv, int nvalid, int md,
                                             const RowConst& rc) {
    float s = 0.0f, sq = 0.0f, es = 0.0f;
    uint32_t bits = 0;
#pragma unroll
    for (int i = 0; i < kChunk; ++i) {
        const float l = lv[i];
        const bool live = (i < nvalid) && (l != -INFINITY);  // masked entries weigh nothing
        float ef = fast_e(l, rc);
        ef = live ? ef : 0.0f;
        const bool big = ef > rc.thr;
        bits |= (big ? 1u : 0u) << i;
        if (md == MODE_RESIDUAL) {
            const float r = fmaf(-rc.s1, qv[i], ef);
            const bool take = !big && r > 0.0f;
            s += take ? r : 0.0f;
            sq += take ? qv[i] : 0.0f;
            es += big ? 0.0f : ef;
        } else {
            s += big ? 0.0f : ef;
        }
    }
#pragma unroll
    for (int k2 = 0; k2 < 4; ++k2) {
        if (k2 == c) {
            L.s[k2] = s;
            L.sq[k2] = sq;
        }
    }
    L.large |= bits << (8 * c);
    if (md == MODE_RESIDUAL) L.e = df_sum(L.e, df_make(es));
}

// Add one large entry's result to chunk c of the lane (entry order).
__device__ __forceinline__ void lane32_add_large(Lane32& L, int c, df w, float wq, df e, int md) {
#pragma unroll
    for (int k2 = 0; k2 < 4; ++k2) {
        if (k2 == c) {
            L.big[k2] = df_sum(L.big[k2], w);
            L.bq[k2] += wq;
        }
    }
    if (md == MODE_RESIDUAL) L.e = df_sum(L.e, e);
}

// Chunk c's weight (pair) and q sum.
__device__ __forceinline__ df lane32_chunk(const Lane32& L, int c, float& q) {
    df w = df_make(0.0f);
    q = 0.0f;
#pragma unroll
    for (int k2 = 0; k2 < 4; ++k2) {
        if (k2 == c) {
            w = df_sum(df_make(L.s[k2]), L.big[k2]);
            q = L.sq[k2] + L.bq[k2];
        }
    }
    return w;
}

// The lane's total weight and q sum, chunks in vocabulary order.
__device__ __forceinline__ df lane32_total(const Lane32& L, float& q) {
    df w = df_make(0.0f);
    q = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        w = df_sum(w, df_sum(df_make(L.s[c]), L.big[c]));
        q += L.sq[c] + L.bq[c];
    }
    return w;
}

// Up to 8 consecutive entries of a logits row / a q row from global memory
// (vector loads when aligned and complete).
template <bool BF16>
__device__ __forceinline__ void load8_logits(const void* logits, long long idx, int cnt, float* lv) {
    const unsigned char* lp = reinterpret_cast<const unsigned char*>(logits) + idx * (BF16 ? 2 : 4);
    if (cnt == kChunk && (reinterpret_cast<uintptr_t>(lp) & 15) == 0) {
        if (BF16) {
            const uint4 w = ld_stream_v4(lp);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                lv[2 * q4] = bf16_lo(ws[q4]);
                lv[2 * q4 + 1] = bf16_hi(ws[q4]);
            }
        } else {
            const uint4 w0 = ld_stream_v4(lp), w1 = ld_stream_v4(lp + 16);
            lv[0] = __uint_as_float(w0.x); lv[1] = __uint_as_float(w0.y);
            lv[2] = __uint_as_float(w0.z); lv[3] = __uint_as_float(w0.w);
            lv[4] = __uint_as_float(w1.x); lv[5] = __uint_as_float(w1.y);
            lv[6] = __uint_as_float(w1.z); lv[7] = __uint_as_float(w1.w);
        }
    } else {
#pragma unroll
        for (int e = 0; e < kChunk; ++e) lv[e] = e < cnt ? load_logit(logits, idx + e, BF16) : -INFINITY;
    }
}

__device__ __forceinline__ void load8_q(const float* qp, int cnt, float* qv) {
    if (cnt == kChunk && (reinterpret_cast<uintptr_t>(qp) & 15) == 0) {
        const uint4 w0 = ld_stream_v4(qp), w1 = ld_stream_v4(qp + 4);
        qv[0] = __uint_as_float(w0.x); qv[1] = __uint_as_float(w0.y);
        qv[2] = __uint_as_float(w0.z); qv[3] = __uint_as_float(w0.w);
        qv[4] = __uint_as_float(w1.x); qv[5] = __uint_as_float(w1.y);
        qv[6] = __uint_as_float(w1.z); qv[7] = __uint_as_float(w1.w);
    } else {
#pragma unroll
        for (int e = 0; e < kChunk; ++e) qv[e] = e < cnt ? __ldg(qp + e) : 0.0f;
    }
}

__device__ __forceinline__ bool q_invalid(const float* qv, int cnt) {
    bool bad = false;
#pragma unroll
    for (int e = 0; e < kChunk; ++e) bad |= e < cnt && !(qv[e] >= 0.0f && qv[e] <= FLT_MAX);
    return bad;
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

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 4) verify_cluster_kernel(const VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ __align__(16) ClusterSmem sh;
    constexpr int esz = BF16 ? 2 : 4;

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

    // ---------------------------------------------------------------- row setup
    const float T = a.temp ? __ldg(a.temp + b) : 0.0f;
    const bool greedy = (T == 0.0f);
    const bool t_ok = greedy || (T >= FLT_MIN && T <= FLT_MAX);
    const float c = greedy || !t_ok ? 0.0f : kLog2e / T;

    // per-position scalars, lane i of warp 0 holds position i
    int xi = -1;
    float u0 = 0.0f, u1 = 0.0f, Lx = 0.0f, qx = 0.0f;
    if (warp == 0 && lane <= k && t_ok) {
        if (lane < k) xi = __ldg(a.x + static_cast<long long>(b) * k + lane);
        if (!greedy) {
            const long long ub = (static_cast<long long>(b) * (k + 1) + lane) * 2;
            u0 = __ldg(a.u + ub);
            u1 = __ldg(a.u + ub + 1);
        }
    }
    if (tid <= k) {
        // geometry of this CTA's slice of position tid
        const long long e0 = (static_cast<long long>(b) * (k + 1) + tid) * V + v0;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(lg + e0 * esz);
        int h = static_cast<int>(((16 - (addr & 15)) & 15) / esz);
        if (h > n) h = n;
        sh.head[tid] = h;
        sh.nbytes[tid] = ((n - h) * esz) & ~15;
    }
    if (tid < 128) sh.exp2tab[tid] = g_exp2_table[tid];
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), kConsumerWarps);
        }
        sh.timeout = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (tid == 0) {
        int acc = 0;
        for (int i = 0; i <= k; ++i) {
            sh.tstart[i] = acc;
            acc += (sh.nbytes[i] + kTileBytes - 1) / kTileBytes;
        }
        sh.tstart[k + 1] = acc;
    }
    __syncthreads();
    const int total1 = t_ok ? sh.tstart[k + 1] : 0;

    // Ring protocol.  Stage use number `it` (counted identically by producer
    // and consumers across both passes) occupies slot it % kStages; its full
    // barrier completes phase (it / kStages) & 1 when the copies land, its
    // empty barrier when the four consumer warps have released it.
    auto prod_acquire = [&](int it) -> bool {
        if (it < kStages) return true;
        const int slot = it % kStages;
        return mbar_wait_bounded(smem_u32(&sh.empty[slot]), ((it / kStages) & 1) ^ 1, kWaitPolls);
    };
    auto cons_wait = [&](int it) -> bool {
        const int slot = it % kStages;
        return mbar_wait_bounded(smem_u32(&sh.full[slot]), (it / kStages) & 1, kWaitPolls);
    };
    auto cons_release = [&](int it) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.empty[it % kStages]));
    };
    int it_prod = 0, it_cons = 0;

    // ---------------------------------------------------------------- pass 1
    if (producer) {
        if (lane == 0) {
            for (int tt = 0; tt < total1; ++tt, ++it_prod) {
                if (sh.timeout || !prod_acquire(it_prod)) {
                    atomicOr(&sh.timeout, 1);
                    break;
                }
                int i = 0;
                while (sh.tstart[i + 1] <= tt) ++i;
                const int off = (tt - sh.tstart[i]) * kTileBytes;
                const int bytes = min(kTileBytes, sh.nbytes[i] - off);
                const long long e0 = (static_cast<long long>(b) * (k + 1) + i) * V + v0 + sh.head[i];
                const int slot = it_prod % kStages;
                const uint32_t bar = smem_u32(&sh.full[slot]);
                mbar_arrive_expect_tx(bar, static_cast<uint32_t>(bytes));
                bulk_g2s(smem_u32(ring + slot * kTileBytes), lg + e0 * esz + off, static_cast<uint32_t>(bytes), bar);
            }
        }
        it_prod = __shfl_sync(0xffffffffu, it_prod, 0);
    } else {
        int t = 0;
        for (int i = 0; i <= k && t_ok; ++i) {
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
            if (tid == 0)
                for (int e = 0; e < h; ++e) scalar_elem(e);

            for (int lt = 0; lt < ntiles; ++lt, ++t, ++it_cons) {
                if (t == 2 && warp == 0 && lane < k && !greedy && xi >= 0 && xi < V) {
                    // the accept test's scalars; x_i has long arrived
                    const long long row = static_cast<long long>(b) * (k + 1) + lane;
                    Lx = load_logit(a.logits, row * V + xi, BF16);
                    qx = __ldg(a.q + (static_cast<long long>(b) * k + lane) * V + xi);
                }
                const bool ok = !sh.timeout && cons_wait(it_cons);
                const int bytes = min(kTileBytes, sh.nbytes[i] - lt * kTileBytes);
                const int nch = bytes >> 4;
                const uint32_t tile = smem_u32(ring + (it_cons % kStages) * kTileBytes);
                if (!ok) {
                    atomicOr(&sh.timeout, 1);
                    continue;
                }
                constexpr int kPer = kTileBytes / 16 / kConsumers;  // 16-byte chunks per thread
                uint4 w[kPer];
#pragma unroll
                for (int r = 0; r < kPer; ++r) {
                    const int ch = tid + r * kConsumers;
                    if (ch < nch) {
                        w[r] = ld_shared_v4(tile + ch * 16);
                    } else if (BF16) {
                        w[r] = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
                    } else {
                        const uint32_t ni = __float_as_uint(-INFINITY);
                        w[r] = make_uint4(ni, ni, ni, ni);
                    }
                }
                cons_release(it_cons);  // the data is in registers
                float lmax;
                if (BF16) {
                    uint32_t mx = 0xff80ff80u, mn = 0xff80ff80u;
#pragma unroll
                    for (int r = 0; r < kPer; ++r) {
                        mx = max_bf16x2(max_bf16x2(mx, w[r].x), max_bf16x2(w[r].y, max_bf16x2(w[r].z, w[r].w)));
                        if (greedy)
                            mn = max_nan_bf16x2(max_nan_bf16x2(mn, w[r].x),
                                                max_nan_bf16x2(w[r].y, max_nan_bf16x2(w[r].z, w[r].w)));
                    }
                    lmax = fmaxf(bf16_lo(mx), bf16_hi(mx));
                    if (greedy && (bf16_lo(mn) != bf16_lo(mn) || bf16_hi(mn) != bf16_hi(mn))) nan_seen = true;
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
                    if (lmax > m) {
                        // first element equal to the new maximum, in index order
                        const long long tile_e0 = v0 + h + static_cast<long long>(lt) * (kTileBytes / esz);
                        bool found = false;
#pragma unroll
                        for (int r = 0; r < kPer; ++r) {
                            const int ch = tid + r * kConsumers;
                            const uint32_t ws[4] = {w[r].x, w[r].y, w[r].z, w[r].w};
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                if (BF16) {
                                    if (!found && bf16_lo(ws[q4]) == lmax) {
                                        found = true;
                                        arg = static_cast<int>(tile_e0 + ch * 8 + q4 * 2);
                                    }
                                    if (!found && bf16_hi(ws[q4]) == lmax) {
                                        found = true;
                                        arg = static_cast<int>(tile_e0 + ch * 8 + q4 * 2 + 1);
                                    }
                                } else {
                                    if (!found && __uint_as_float(ws[q4]) == lmax) {
                                        found = true;
                                        arg = static_cast<int>(tile_e0 + ch * 4 + q4);
                                    }
                                }
                            }
                        }
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
                    const f2 mm = pack2(m, m), cc = pack2(c, c);
                    f2 acc = pack2(0.0f, 0.0f);
#pragma unroll
                    for (int r = 0; r < kPer; ++r) {
                        const uint32_t ws[4] = {w[r].x, w[r].y, w[r].z, w[r].w};
                        if (BF16) {
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                const f2 d = mul2(sub2(pack2(bf16_lo(ws[q4]), bf16_hi(ws[q4])), mm), cc);
                                float d0, d1;
                                unpack2(d, d0, d1);
                                acc = add2(acc, pack2(ex2(d0), ex2(d1)));
                            }
                        } else {
#pragma unroll
                            for (int q4 = 0; q4 < 4; q4 += 2) {
                                const f2 d =
                                    mul2(sub2(pack2(__uint_as_float(ws[q4]), __uint_as_float(ws[q4 + 1])), mm), cc);
                                float d0, d1;
                                unpack2(d, d0, d1);
                                acc = add2(acc, pack2(ex2(d0), ex2(d1)));
                            }
                        }
                    }
                    float a0, a1;
                    unpack2(acc, a0, a1);
                    s += a0 + a1;
                }
            }
            if (tid == 0)
                for (int e = h + interior; e < n; ++e) scalar_elem(e);

            // warp reduction of this position's partial
            if (greedy) {
                for (int off = 16; off > 0; off >>= 1) {
                    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
                    const int a2 = __shfl_xor_sync(0xffffffffu, arg, off);
                    merge_arg(m, arg, m2, a2);
                }
                nan_seen = __any_sync(0xffffffffu, nan_seen);
            } else {
                for (int off = 16; off > 0; off >>= 1) {
                    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
                    const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
                    merge_ms(m, s, m2, s2, c);
                }
            }
            if (lane == 0) sh.wpart[warp][i] = Partial{m, s, arg, nan_seen ? 1 : 0};
        }
        // rows too short to reach the third tile load the scalars here
        if (t_ok && total1 <= 2 && warp == 0 && lane < k && !greedy && xi >= 0 && xi < V) {
            const long long row = static_cast<long long>(b) * (k + 1) + lane;
            Lx = load_logit(a.logits, row * V + xi, BF16);
            qx = __ldg(a.q + (static_cast<long long>(b) * k + lane) * V + xi);
        }
    }
    __syncthreads();
    const bool timed_out = sh.timeout != 0;
    if (tid <= k && t_ok) {
        Partial p = sh.wpart[0][tid];
        for (int w = 1; w < kConsumerWarps; ++w) {
            const Partial o = sh.wpart[w][tid];
            if (greedy) {
                merge_arg(p.m, p.arg, o.m, o.arg);
                p.flags |= o.flags;
            } else {
                merge_ms(p.m, p.s, o.m, o.s, c);
            }
        }
        if (timed_out) p.flags |= 2;
        // push this CTA's partial of position tid into every CTA of the cluster
        const uint32_t local = smem_u32(&sh.allpart[rank][tid]);
        for (uint32_t r = 0; r < C; ++r)
            st_cluster_v4(map_rank(local, r), __float_as_uint(p.m), __float_as_uint(p.s), static_cast<uint32_t>(p.arg),
                          static_cast<uint32_t>(p.flags));
    }
    cluster_sync();  // #1: every CTA's partials are visible

    // ---------------------------------------------------------------- decisions
    if (warp == 0) {
        float M = -INFINITY, S = 0.0f;
        int A = 0x7fffffff, flags = 0;
        if (lane <= k && t_ok) {
            for (uint32_t r = 0; r < C; ++r) {
                const Partial pr = sh.allpart[r][lane];
                flags |= pr.flags;
                if (greedy)
                    merge_arg(M, A, pr.m, pr.arg);
                else
                    merge_ms(M, S, pr.m, pr.s, c);
            }
            if (greedy && A == 0x7fffffff) A = 0;  // every value is -inf: index 0
        }
        int err = 0;
        bool stop = false;
        float p = 0.0f;
        if (lane <= k && t_ok) {
            if (flags & 2) err |= ST_TIMEOUT;
            if (greedy) {
                if (flags & 1) err |= ST_NONFINITE;
                if (lane < k && (xi < 0 || xi >= V)) err |= ST_TOKEN;
                stop = (err != 0) || lane == k || xi != A;
            } else {
                if (!(isfinite(M) && isfinite(S))) err |= ST_NONFINITE;
                if (lane < k) {
                    if (xi < 0 || xi >= V) err |= ST_TOKEN;
                    if (!(u0 >= 0.0f && u0 < 1.0f)) err |= ST_UNIFORM;
                    if (xi >= 0 && xi < V && !(qx >= 0.0f && qx <= FLT_MAX)) err |= ST_QBAD;
                    if (!err) {
                        // p_i(x_i) with the double-float exponential (a masked
                        // entry, logit -inf, has p = 0)
                        const df c2 = log2e_over(T);
                        RowConst rc;
                        rc.M = M;
                        rc.s1 = S;
                        rc.thr = 0.0f;
                        rc.ch = c2.hi;
                        rc.cl = c2.lo;
                        p = df_val(exact_weight<BF16>(Lx, 0.0f, MODE_BONUS, rc, df_make(0.0f), sh.exp2tab)) / S;
                        const float rho = fminf(1.0f, p / fmaxf(qx, 1e-12f));
                        stop = !(u0 < rho);
                    } else {
                        stop = true;
                    }
                } else {
                    stop = true;
                }
            }
        }
        const unsigned mask = __ballot_sync(0xffffffffu, lane <= k && stop);
        const int j = t_ok ? (__ffs(mask) - 1) : 0;
        int st = t_ok ? __shfl_sync(0xffffffffu, err, j) : ST_TEMP;
        if (t_ok && !greedy && !(st & ST_ERRMASK)) {
            const float uj = __shfl_sync(0xffffffffu, u1, j);
            if (!(uj >= 0.0f && uj < 1.0f)) st |= ST_UNIFORM;
        }
        const float Mj = __shfl_sync(0xffffffffu, M, j);
        const float Sj = __shfl_sync(0xffffffffu, S, j);
        const int Aj = __shfl_sync(0xffffffffu, A, j);
        const float ujj = __shfl_sync(0xffffffffu, u1, j);
        if (lane == 0) {
            sh.uj = ujj;
            sh.j = j;
            sh.status = st;
            sh.Mj = Mj;
            sh.sj = Sj;
            sh.mode = (j < k) ? MODE_RESIDUAL : MODE_BONUS;
        }
        if (lane <= k) sh.xs[lane] = xi;
        // rank 0 writes debug values and, for greedy or failed rows, the outputs
        if (rank == 0) {
            if (lane <= k && t_ok) {
                if (a.dbg_max) a.dbg_max[static_cast<long long>(b) * (k + 1) + lane] = M;
                if (a.dbg_sumexp) a.dbg_sumexp[static_cast<long long>(b) * (k + 1) + lane] = greedy ? 0.0f : S;
                if (lane < k) {
                    const bool xok = xi >= 0 && xi < V;
                    if (a.dbg_p) a.dbg_p[static_cast<long long>(b) * k + lane] = (greedy || !xok) ? 0.0f : p;
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
    __syncthreads();
    const bool sample = t_ok && !greedy && !(sh.status & ST_ERRMASK);
    if (!sample) {
        cluster_sync();  // no CTA leaves while a peer may still read its partials
        return;
    }

    // ---------------------------------------------------------------- pass 2
    const int j = sh.j;
    const long long lrow = (static_cast<long long>(b) * (k + 1) + j) * V;
    const float* qrow = a.q + (static_cast<long long>(b) * k + (j < k ? j : 0)) * V;
    if (tid == 0) {
        const df c2 = log2e_over(T);
        sh.c_hi = c2.hi;
        sh.c_lo = c2.lo;
        sh.thr = kLargeP * sh.sj;
        // bulk copies need 16-byte aligned starts and sizes: both rows
        // aligned at the slice start, and whole groups of 8 entries
        const bool la = (reinterpret_cast<uintptr_t>(lg + (lrow + v0) * esz) & 15) == 0;
        const bool qa = (reinterpret_cast<uintptr_t>(qrow + v0) & 15) == 0;
        sh.p2fast = la && (j == k || qa) && (n % kChunk) == 0;
        sh.ntiles2 = (n + kP2Elems - 1) / kP2Elems;
    }
    __syncthreads();
    RowConst rc;
    rc.M = sh.Mj;
    rc.s1 = sh.sj;
    rc.thr = sh.thr;
    rc.ch = sh.c_hi;
    rc.cl = sh.c_lo;
    const bool p2fast = sh.p2fast != 0;
    const int ntiles2 = sh.ntiles2;
    int mode = sh.mode;

    // one stop-row entry by tile-local index, from the staged tile or from global memory
    auto fetch1 = [&](bool staged, uint32_t base, int e0, int idx, float& l, float& q) {
        if (staged) {
            l = BF16 ? __uint_as_float(static_cast<uint32_t>(ld_shared_u16(base + kP2Elems * 4 + idx * 2)) << 16)
                     : ld_shared_f32(base + kP2Elems * 4 + idx * 4);
            q = mode == MODE_RESIDUAL ? ld_shared_f32(base + idx * 4) : 0.0f;
        } else {
            l = load_logit(a.logits, lrow + v0 + e0 + idx, BF16);
            q = mode == MODE_RESIDUAL ? __ldg(qrow + v0 + e0 + idx) : 0.0f;
        }
    };

    for (;;) {
        df te = df_make(0.0f);  // this thread's sum of e (residual mode)
        bool qbad = false;
        if (producer) {
            if (p2fast && lane == 0) {
                for (int t2 = 0; t2 < ntiles2; ++t2, ++it_prod) {
                    if (sh.timeout || !prod_acquire(it_prod)) {
                        atomicOr(&sh.timeout, 1);
                        break;
                    }
                    const int e0 = t2 * kP2Elems;
                    const int cnt = min(kP2Elems, n - e0);
                    const int slot = it_prod % kStages;
                    const uint32_t bar = smem_u32(&sh.full[slot]);
                    const uint32_t dst = smem_u32(ring + slot * kTileBytes);
                    const uint32_t lbytes = static_cast<uint32_t>(cnt * esz);
                    const uint32_t qbytes = mode == MODE_RESIDUAL ? static_cast<uint32_t>(cnt * 4) : 0u;
                    mbar_arrive_expect_tx(bar, lbytes + qbytes);
                    bulk_g2s(dst + kP2Elems * 4, lg + (lrow + v0 + e0) * esz, lbytes, bar);
                    if (qbytes) bulk_g2s(dst, qrow + v0 + e0, qbytes, bar);
                }
            }
            it_prod = __shfl_sync(0xffffffffu, it_prod, 0);
        } else {
            // one warp per tile of 1024 entries; lane l owns entries [32l, 32l+32)
            const int it0 = it_cons;
            for (int t2 = warp; t2 < ntiles2; t2 += kConsumerWarps) {
                const int it = it0 + t2;
                const int e0 = t2 * kP2Elems;
                const int cnt = min(kP2Elems, n - e0);
                const int my0 = lane * kLaneEntries;
                bool ok = true;
                uint32_t base = 0;
                if (p2fast) {
                    ok = __all_sync(0xffffffffu, !sh.timeout && cons_wait(it));
                    base = smem_u32(ring + (it % kStages) * kTileBytes);
                    if (!ok) atomicOr(&sh.timeout, 1);
                }
                Lane32 L;
                lane32_init(L);
                if (ok) {
#pragma unroll 2
                    for (int i = 0; i < 4; ++i) {
                        const int c = (i + lane) & 3;  // rotated: spreads the lanes over the banks
                        const int off = my0 + c * kChunk;
                        const int nv = max(0, min(kChunk, cnt - off));
                        float lv[kChunk], qv[kChunk];
#pragma unroll
                        for (int e = 0; e < kChunk; ++e) {
                            lv[e] = -INFINITY;
                            qv[e] = 0.0f;
                        }
                        if (nv > 0) {
                            if (p2fast) {
                                if (BF16) {
                                    const uint4 w = ld_shared_v4(base + kP2Elems * 4 + off * 2);
                                    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                                    for (int q4 = 0; q4 < 4; ++q4) {
                                        lv[2 * q4] = bf16_lo(ws[q4]);
                                        lv[2 * q4 + 1] = bf16_hi(ws[q4]);
                                    }
                                } else {
                                    const uint4 w0 = ld_shared_v4(base + kP2Elems * 4 + off * 4);
                                    const uint4 w1 = ld_shared_v4(base + kP2Elems * 4 + off * 4 + 16);
                                    lv[0] = __uint_as_float(w0.x); lv[1] = __uint_as_float(w0.y);
                                    lv[2] = __uint_as_float(w0.z); lv[3] = __uint_as_float(w0.w);
                                    lv[4] = __uint_as_float(w1.x); lv[5] = __uint_as_float(w1.y);
                                    lv[6] = __uint_as_float(w1.z); lv[7] = __uint_as_float(w1.w);
                                }
                                if (mode == MODE_RESIDUAL) {
                                    const uint4 w0 = ld_shared_v4(base + off * 4);
                                    const uint4 w1 = ld_shared_v4(base + off * 4 + 16);
                                    qv[0] = __uint_as_float(w0.x); qv[1] = __uint_as_float(w0.y);
                                    qv[2] = __uint_as_float(w0.z); qv[3] = __uint_as_float(w0.w);
                                    qv[4] = __uint_as_float(w1.x); qv[5] = __uint_as_float(w1.y);
                                    qv[6] = __uint_as_float(w1.z); qv[7] = __uint_as_float(w1.w);
                                }
                            } else {
                                // unaligned rows: the same tiles, read straight from global memory
                                load8_logits<BF16>(a.logits, lrow + v0 + e0 + off, nv, lv);
                                if (mode == MODE_RESIDUAL) load8_q(qrow + v0 + e0 + off, nv, qv);
                            }
                        }
                        if (mode == MODE_RESIDUAL) qbad |= q_invalid(qv, nv);
                        lane32_fast8(L, c, lv, qv, nv, mode, rc);
                    }
                    // large entries, each lane its own in entry order (the warp
                    // runs as many rounds as its busiest lane has entries)
                    for (uint32_t m = L.large; m; m &= m - 1) {
                        const int bit = __ffs(m) - 1;
                        float l, q;
                        fetch1(p2fast, base, e0, my0 + bit, l, q);
                        df w, e;
                        float wq;
                        large_weight<BF16>(l, q, mode, rc, sh.exp2tab, w, wq, e);
                        lane32_add_large(L, bit >> 3, w, wq, e, mode);
                    }
                    if (p2fast) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cnt(smem_u32(&sh.empty[it % kStages]), kConsumerWarps);
                    }
                }
                float lq;
                const df lw = lane32_total(L, lq);
                sh.lane_hi[t2][lane] = lw.hi;
                sh.lane_lo[t2][lane] = lw.lo;
                sh.lane_q[t2][lane] = lq;
                te = df_sum(te, L.e);
                const df tw = df_warp_total(lw);
                float tq = lq;
                for (int off = 16; off > 0; off >>= 1) tq += __shfl_down_sync(0xffffffffu, tq, off);
                if (lane == 0) {
                    sh.tile_hi[t2] = tw.hi;
                    sh.tile_lo[t2] = tw.lo;
                    sh.tile_q[t2] = tq;
                }
            }
            it_cons = it0 + ntiles2;
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
            } else if (mode == MODE_RESIDUAL && !(Wt.hi + Wt.lo > 0.0f)) {
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
                }
            }
        }
        __syncthreads();
        if (sh.mode == MODE_FALLBACK && mode == MODE_RESIDUAL) {
            mode = MODE_FALLBACK;
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
            if (idx < cnt) fetch1(false, 0, e0, idx, l, q);
            const df we = exact_weight<BF16>(l, q, mode, rc, s_prec, sh.exp2tab);
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
