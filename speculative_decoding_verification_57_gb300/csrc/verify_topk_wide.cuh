// verify_topk_wide.cuh -- top-k / top-p verification for top_k above 64
// (up to 4096), the rows the register top-64 of verify_topk.cuh cannot hold
// ("Speculative decoding." lesson, "Why the output is exactly p": temperature,
// top-k and top-p have to be applied to p before the rule).
//
// Readings (the same as verify_topk.cuh): top-k keeps the min(K, V) largest
// logits, the lower index first among equal logits; top-p keeps the shortest
// prefix of those, in the same order, whose mass renormalised over the K
// reaches top_p.  p' = exp((l - M) / T) on the kept set P, renormalised; the
// residual max(0, p' - q) and the bonus live on P and are drawn in
// vocabulary order.
//
// One thread-block cluster of C = min(k + 1, 16) CTAs of 512 threads per
// sequence; CTA c owns positions c and c + C.  A position's kept set is found
// exactly, with no sort of the vocabulary:
//   1. a radix select on the logits' order-preserving keys (bf16: 12 + 4
//      bits, fp32: 12 + 12 + 8 bits), one pass over the row a digit, finds
//      the key of the K-th largest entry, key*, and how many entries lie
//      above it; the last digit's counts are kept per warp, each warp owning
//      a contiguous stretch of the row, so that the ties at key* that fit
//      (the lowest indices) are known per warp;
//   2. one more pass marks the kept entries in a bitmap of the vocabulary,
//      which a block scan turns into the kept list in vocabulary order
//      (index and logit, at most 4096 entries, in shared memory);
//   3. on the list: the maximum M, every weight e = exp((l - M) / T) with
//      the double-float exponential, their sum, and (top_p < 1) the top-p
//      cut by bisection on the key: the largest key whose entries and those
//      above reach top_p of the sum, and how many of its ties are needed;
//   4. p'(x_i) goes to the leader CTA over distributed shared memory.
// After a cluster barrier the leader's warp 0 walks the positions, and the
// CTA that owns the stop position draws from its kept list: weights in
// double-float, a block scan in vocabulary order, the first entry whose
// prefix exceeds u * W.
#pragma once
#include <cfloat>
#include <climits>
#include <cstdint>

#include "exp2dd.cuh"
#include "ptx.cuh"
#include "verify_cluster.cuh"
#include "verify_topk.cuh"

namespace specv {

constexpr int kWideThreads = 512;
constexpr int kWideWarps = kWideThreads / 32;
constexpr int kWideEpt = kWideKMax / kWideThreads;  // kept-list entries per thread
constexpr int kWideClusterMax = 16;                // CTAs per sequence
constexpr int kWideWorkBytes = 32768;              // histograms, then the bitmap (V <= 262144), then the weights
constexpr int kWideSlotBytes = kWideKMax * 8;      // one position's kept list: index and logit
constexpr int kWideSlots = (kMaxK + kWideClusterMax) / kWideClusterMax;  // positions a CTA owns at most
static_assert(kWideEpt * kWideThreads == kWideKMax, "the kept list is split evenly over the threads");
static_assert(kWideKMax * 8 <= kWideWorkBytes, "the weights of a kept list fit the work area");
static_assert(262144 / 8 <= kWideWorkBytes, "the bitmap of the largest vocabulary fits the work area");

inline int wide_cluster(int k) { return k + 1 < kWideClusterMax ? k + 1 : kWideClusterMax; }

// Dynamic shared memory: the work area, then one kept list per owned position.
inline size_t wide_dyn_smem(int k) {
    const int C = wide_cluster(k);
    const int P = (k + C) / C;  // ceil((k + 1) / C)
    return static_cast<size_t>(kWideWorkBytes) + static_cast<size_t>(P) * kWideSlotBytes;
}

// Order-preserving keys (a larger logit has a larger key; -0 is +0).  bf16:
// 16 bits from the bf16 pattern; fp32: 32 bits.  -inf maps above 0, so key
// 0 belongs to no logit.
__device__ __forceinline__ uint32_t key16(uint32_t b) {
    if (b == 0x8000u) b = 0u;
    return (b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u);
}

__device__ __forceinline__ uint32_t key32(uint32_t f) {
    if (f == 0x80000000u) f = 0u;
    return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}

template <bool BF16>
__device__ __forceinline__ uint32_t val_key(float v) {
    return BF16 ? key16(__float_as_uint(v) >> 16) : key32(__float_as_uint(v));
}

template <bool BF16>
__device__ __forceinline__ float ld_val(const unsigned char* rowp, int e) {
    if (BF16) return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(rowp) + e)) << 16);
    return __ldg(reinterpret_cast<const float*>(rowp) + e);
}

// One logit's bit pattern: its key, whether it takes part (not NaN), and
// whether it makes the row non-finite (NaN or +inf).
template <bool BF16>
__device__ __forceinline__ bool take_bits(uint32_t bits, uint32_t& key, bool& bad) {
    if (BF16) {
        const bool nan = (bits & 0x7fffu) > 0x7f80u;
        bad |= nan || bits == 0x7f80u;
        key = key16(bits);
        return !nan;
    }
    const bool nan = (bits & 0x7fffffffu) > 0x7f800000u;
    bad |= nan || bits == 0x7f800000u;
    key = key32(bits);
    return !nan;
}

// Walks one warp's stretch of a row in vocabulary order: the scalar head
// (entries before the first 16-byte boundary) belongs to warp 0, before its
// groups; the scalar tail to the last warp, after its groups; the 16-byte
// groups between are split evenly over the warps.  Every lane calls
// f(e0, keys, vmask) once a round, the same number of times: keys[q] is
// entry e0 + q's key, bit q of vmask says it exists (and is not NaN).
// Within a round the lanes' entries follow lane order.
template <bool BF16, typename F>
__device__ __forceinline__ void wide_walk(const unsigned char* rowp, int n, int h, int ng, int warp, int lane,
                                          bool& bad, F&& f) {
    constexpr int G = BF16 ? 8 : 4;
    constexpr int esz = BF16 ? 2 : 4;
    uint32_t keys[G];
    auto scalar_round = [&](int e) {
        uint32_t vm = 0;
        if (e >= 0) {
            const uint32_t bits = BF16 ? static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(rowp) + e))
                                       : __float_as_uint(__ldg(reinterpret_cast<const float*>(rowp) + e));
            vm = take_bits<BF16>(bits, keys[0], bad) ? 1u : 0u;
        }
        f(e < 0 ? 0 : e, keys, vm);
    };
    if (warp == 0 && h > 0) scalar_round(lane < h ? lane : -1);
    const int g0 = static_cast<int>(static_cast<long long>(ng) * warp / kWideWarps);
    const int g1 = static_cast<int>(static_cast<long long>(ng) * (warp + 1) / kWideWarps);
    for (int base = g0; base < g1; base += 128) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = base + 32 * u + lane;
            w[u] = g < g1 ? __ldg(reinterpret_cast<const uint4*>(rowp + (static_cast<long long>(h) + static_cast<long long>(g) * G) * esz))
                          : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = base + 32 * u + lane;
            uint32_t vm = 0;
            if (g < g1) {
                const uint32_t wd[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
                if (BF16) {
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        vm |= (take_bits<true>(wd[m] & 0xffffu, keys[2 * m], bad) ? 1u : 0u) << (2 * m);
                        vm |= (take_bits<true>(wd[m] >> 16, keys[2 * m + 1], bad) ? 1u : 0u) << (2 * m + 1);
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < 4; ++m) vm |= (take_bits<false>(wd[m], keys[m], bad) ? 1u : 0u) << m;
                }
            }
            f(h + g * G, keys, vm);
        }
    }
    const int t0 = h + ng * G;
    if (warp == kWideWarps - 1 && t0 < n) scalar_round(lane < n - t0 ? t0 + lane : -1);
}

struct WideSlot {
    df S;           // mass of the kept set P, in e-units
    float M;        // the row maximum
    uint32_t cut;   // P: list entries with a key above cut, and the first
    int m_cut;      // m_cut (vocabulary order) whose key equals it (cut 0: every entry)
    int n;          // kept-list entries: min(top_k, V)
    int bad;        // a NaN or +inf logit, or every logit -inf
};

struct alignas(16) WideSmem {
    float2 exp2tab[128];
    WideSlot slot[kWideSlots];
    df red_df[kWideWarps];
    uint32_t red_u[kWideWarps];
    float red_f[kWideWarps];
    uint32_t quota[kWideWarps];  // ties at key* each warp keeps
    int xs[kMaxK + 1];
    float lpx[kMaxK + 1];        // this CTA's p'(x_i) and flags, pushed to the leader at the end
    int lbad[kMaxK + 1];
    float px[kMaxK + 1];         // the leader's copy of every position's
    int pbad[kMaxK + 1];
    df e_cut;
    int dstar;
    uint32_t dabove;
    int xr;
    int m_cut;
    df S;
    int dj, dst;                 // the decision (written by the leader into every CTA)
    float du1;
};

// Block-wide helpers over the 512 threads; each ends with a barrier, so the
// scratch may be reused at once.
__device__ __forceinline__ uint32_t wide_sum_u32(uint32_t v, uint32_t* red) {
    v = __reduce_add_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t t = 0;
    for (int i = 0; i < kWideWarps; ++i) t += red[i];
    __syncthreads();
    return t;
}

__device__ __forceinline__ uint32_t wide_min_u32(uint32_t v, uint32_t* red) {
    v = __reduce_min_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t t = 0xffffffffu;
    for (int i = 0; i < kWideWarps; ++i) t = min(t, red[i]);
    __syncthreads();
    return t;
}

__device__ __forceinline__ uint32_t wide_max_u32(uint32_t v, uint32_t* red) {
    v = __reduce_max_sync(0xffffffffu, v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t t = 0;
    for (int i = 0; i < kWideWarps; ++i) t = max(t, red[i]);
    __syncthreads();
    return t;
}

__device__ __forceinline__ float wide_max_f(float v, float* red) {
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = -INFINITY;
    for (int i = 0; i < kWideWarps; ++i) t = fmaxf(t, red[i]);
    __syncthreads();
    return t;
}

// Exclusive prefix in thread order, and the total.
__device__ __forceinline__ uint32_t wide_excl_scan_u32(uint32_t v, uint32_t* red, uint32_t& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t incl = v;
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) red[w] = incl;
    __syncthreads();
    uint32_t base = 0, tot = 0;
    for (int i = 0; i < kWideWarps; ++i) {
        const uint32_t r = red[i];
        if (i < w) base += r;
        tot += r;
    }
    __syncthreads();
    total = tot;
    return base + incl - v;
}

// Sum of pairs (fixed order: warp trees, then the warps in order).
__device__ __forceinline__ df wide_sum_df(df v, df* red) {
    v = df_warp_total(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    df t = df_make(0.0f);
    for (int i = 0; i < kWideWarps; ++i) t = df_sum(t, red[i]);
    __syncthreads();
    return t;
}

// Exclusive prefix of pairs in thread order.
__device__ __forceinline__ df wide_excl_scan_df(df v, df* red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const df incl = df_warp_incl_scan(v, lane);
    if (lane == 31) red[w] = incl;
    __syncthreads();
    df base = df_make(0.0f);
    for (int i = 0; i < w; ++i) base = df_sum(base, red[i]);
    __syncthreads();
    const df up = df_shfl_up(incl, 1);  // every lane takes part; lane 0 then drops it
    return lane == 0 ? base : df_sum(base, up);
}

// The digit d of hist[0, nb) with above(d) < need <= above(d) + hist[d],
// above(d) being the count in the digits over d: sh.dstar (-1 if the bins
// hold fewer than need entries) and sh.dabove = above(d).
__device__ __forceinline__ void wide_find_digit(const uint32_t* hist, int nb, uint32_t need, WideSmem& sh) {
    const int tid = threadIdx.x;
    const int bpt = (nb + kWideThreads - 1) / kWideThreads;
    const int d0 = min(nb, tid * bpt), d1 = min(nb, d0 + bpt);
    uint32_t local = 0;
    for (int d = d0; d < d1; ++d) local += hist[d];
    if (tid == 0) sh.dstar = -1;
    uint32_t total;
    const uint32_t excl = wide_excl_scan_u32(local, sh.red_u, total);
    const uint32_t above = total - excl - local;
    if (local > 0 && above < need && need <= above + local) {
        uint32_t acc = above;
        for (int d = d1 - 1; d >= d0; --d) {
            const uint32_t hv = hist[d];
            if (acc + hv >= need) {
                sh.dstar = d;
                sh.dabove = acc;
                break;
            }
            acc += hv;
        }
    }
    __syncthreads();
}

template <bool BF16>
__global__ void __launch_bounds__(kWideThreads, 2) verify_topk_wide_kernel(const VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ WideSmem sh;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int G = 16 / esz;
    constexpr int KB = BF16 ? 16 : 32;  // key bits
    const unsigned full = 0xffffffffu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = static_cast<int>(cluster_size());
    const int crank = static_cast<int>(cluster_rank());
    const int b = static_cast<int>(blockIdx.x) / C;
    const int k = a.k;
    const int n = static_cast<int>(a.V);

    const float T = __ldg(a.temp + b);
    const int K = __ldg(a.top_k + b);
    const float top_p = __ldg(a.top_p + b);
    if (!wide_row(T, K, top_p)) return;  // the whole cluster leaves: verify_topk_kernel has the row
    cluster_arrive();                      // paired with the wait before the first remote store

    uint32_t* work = reinterpret_cast<uint32_t*>(dyn_smem);
    df* ework = reinterpret_cast<df*>(dyn_smem);
    if (tid < 128) sh.exp2tab[tid] = g_exp2_table[tid];
    if (tid <= k) sh.xs[tid] = tid < k ? __ldg(a.x + static_cast<long long>(b) * k + tid) : -1;
    RowConst rc;
    rc.s1 = 0.0f;
    rc.thr = 0.0f;
    {
        const df c2 = log2e_over(T);
        rc.ch = c2.hi;
        rc.cl = c2.lo;
    }
    const int Kp = K < n ? K : n;
    const int P = (k - crank) / C + 1;  // owned positions crank + C p, p < P

    for (int p = 0; p < P; ++p) {
        const int i = crank + C * p;
        int* lidx = reinterpret_cast<int*>(dyn_smem + kWideWorkBytes + p * kWideSlotBytes);
        float* lval = reinterpret_cast<float*>(dyn_smem + kWideWorkBytes + p * kWideSlotBytes + kWideKMax * 4);
        const unsigned char* rowp = reinterpret_cast<const unsigned char*>(a.logits) +
                                    (static_cast<long long>(b) * (k + 1) + i) * static_cast<long long>(n) * esz;
        int h = static_cast<int>(((16 - (reinterpret_cast<uintptr_t>(rowp) & 15)) & 15) / esz);
        if (h > n) h = n;
        const int ng = (n - h) / G;

        // ------------------------------------------------ 1. radix select of key*
        bool badl = false;
        bool bad = false;
        uint32_t prefix = 0, c_above = 0;
        const int nlev = BF16 ? 2 : 3;
        int nb_last = 0;
        for (int lev = 0; lev < nlev; ++lev) {
            const int width = BF16 ? (lev == 0 ? 12 : 4) : (lev == 2 ? 8 : 12);
            const int shift = BF16 ? (lev == 0 ? 4 : 0) : (lev == 0 ? 20 : (lev == 1 ? 8 : 0));
            const int nb = 1 << width;
            const bool last = lev == nlev - 1;
            const int hs = shift + width;  // the bits above this digit must equal prefix
            for (int d = tid; d < (last ? kWideWarps * nb : nb); d += kWideThreads) work[d] = 0u;
            __syncthreads();
            uint32_t* hist = last ? work + warp * nb : work;
            wide_walk<BF16>(rowp, n, h, ng, warp, lane, badl, [&](int, const uint32_t* keys, uint32_t vm) {
#pragma unroll
                for (int q = 0; q < G; ++q)
                    if ((vm >> q) & 1u) {
                        const uint32_t key = keys[q];
                        if (lev == 0 || (key >> hs) == prefix) atomicAdd(&hist[(key >> shift) & (nb - 1)], 1u);
                    }
            });
            if (lev == 0) {
                bad = __syncthreads_or(badl ? 1 : 0) != 0;
                if (bad) break;  // the row is non-finite: nothing more is needed of it
            } else {
                __syncthreads();
            }
            const uint32_t need = static_cast<uint32_t>(Kp) - c_above;
            if (last) {
                for (int d = tid; d < nb; d += kWideThreads) {
                    uint32_t s = 0;
                    for (int w = 0; w < kWideWarps; ++w) s += work[w * nb + d];
                    work[kWideWarps * nb + d] = s;
                }
                __syncthreads();
                wide_find_digit(work + kWideWarps * nb, nb, need, sh);
            } else {
                wide_find_digit(work, nb, need, sh);
            }
            if (sh.dstar < 0) {  // fewer entries than top_k take part: only NaNs do that
                bad = true;
                break;
            }
            c_above += sh.dabove;
            prefix = (prefix << width) | static_cast<uint32_t>(sh.dstar);
            nb_last = nb;
        }
        int nl = 0;
        float M = -INFINITY;
        uint32_t cut = 0;
        int m_cut = 0;
        df S = df_make(0.0f);
        if (!bad) {
            const uint32_t kstar = prefix;
            const int dl = static_cast<int>(prefix & static_cast<uint32_t>(nb_last - 1));
            const uint32_t t = static_cast<uint32_t>(Kp) - c_above;  // ties at key* that are kept (>= 1)
            if (warp == 0) {
                const uint32_t tie = lane < kWideWarps ? work[lane * nb_last + dl] : 0u;
                uint32_t incl = tie;
                for (int off = 1; off < 32; off <<= 1) {
                    const uint32_t o = __shfl_up_sync(full, incl, off);
                    if (lane >= off) incl += o;
                }
                const uint32_t excl = incl - tie;
                if (lane < kWideWarps) sh.quota[lane] = t > excl ? min(tie, t - excl) : 0u;
            }
            __syncthreads();

            // -------------------------------------------- 2. the kept entries: bitmap, then the list
            const int nwords = (n + 31) >> 5;
            for (int d = tid; d < nwords; d += kWideThreads) work[d] = 0u;
            __syncthreads();
            const uint32_t quota = sh.quota[warp];
            uint32_t seen = 0;  // ties at key* this warp has passed (the same in every lane)
            wide_walk<BF16>(rowp, n, h, ng, warp, lane, badl, [&](int e0, const uint32_t* keys, uint32_t vm) {
                uint32_t sel = 0, tm = 0;
#pragma unroll
                for (int q = 0; q < G; ++q)
                    if ((vm >> q) & 1u) {
                        if (keys[q] > kstar) sel |= 1u << q;
                        else if (keys[q] == kstar) tm |= 1u << q;
                    }
                const uint32_t tc = __popc(tm);
                if (__any_sync(full, tc != 0)) {
                    // ranks of the ties in vocabulary order: lanes first, then a lane's entries
                    uint32_t incl = tc;
                    for (int off = 1; off < 32; off <<= 1) {
                        const uint32_t o = __shfl_up_sync(full, incl, off);
                        if (lane >= off) incl += o;
                    }
                    uint32_t r = seen + incl - tc;
                    for (uint32_t m = tm; m;) {
                        const int q = __ffs(m) - 1;
                        m &= m - 1;
                        if (r < quota) sel |= 1u << q;
                        ++r;
                    }
                    seen += __shfl_sync(full, incl, 31);
                }
                for (uint32_t m = sel; m;) {
                    const int q = __ffs(m) - 1;
                    m &= m - 1;
                    const int e = e0 + q;
                    atomicOr(&work[e >> 5], 1u << (e & 31));
                }
            });
            __syncthreads();
            {
                const int wpt = (nwords + kWideThreads - 1) / kWideThreads;
                const int w0 = min(nwords, tid * wpt), w1 = min(nwords, w0 + wpt);
                uint32_t c = 0;
                for (int w = w0; w < w1; ++w) c += __popc(work[w]);
                uint32_t total;
                uint32_t pos = wide_excl_scan_u32(c, sh.red_u, total);
                for (int w = w0; w < w1; ++w)
                    for (uint32_t m = work[w]; m;) {
                        const int bit = __ffs(m) - 1;
                        m &= m - 1;
                        if (pos < static_cast<uint32_t>(kWideKMax)) lidx[pos] = w * 32 + bit;
                        ++pos;
                    }
                nl = static_cast<int>(min(total, static_cast<uint32_t>(kWideKMax)));
                bad = total != static_cast<uint32_t>(Kp);  // cannot happen on a finite row
            }
            __syncthreads();
            for (int r = tid; r < nl; r += kWideThreads) lval[r] = ld_val<BF16>(rowp, lidx[r]);
            __syncthreads();

            // -------------------------------------------- 3. weights, their sum, the top-p cut
            const int r0 = tid * kWideEpt;
            float mx = -INFINITY;
            for (int q = 0; q < kWideEpt; ++q)
                if (r0 + q < nl) mx = fmaxf(mx, lval[r0 + q]);
            M = wide_max_f(mx, sh.red_f);
            if (!(M > -INFINITY)) bad = true;
            if (!bad) {
                rc.M = M;
                df part = df_make(0.0f);
                for (int q = 0; q < kWideEpt; ++q) {
                    const int r = r0 + q;
                    if (r < nl) {
                        const float l = lval[r];
                        const df e = l == -INFINITY ? df_make(0.0f) : precise_e<BF16>(l, rc, sh.exp2tab);
                        ework[r] = e;
                        part = df_sum(part, e);
                    }
                }
                const df SK = wide_sum_df(part, sh.red_df);
                S = SK;
                if (top_p < 1.0f) {
                    const df target = df_mul_f(SK, top_p);
                    // the largest key whose entries and those above weigh at least target
                    unsigned long long lo = 0, hi = 1ull << KB;
                    while (hi - lo > 1) {
                        const unsigned long long mid = (lo + hi) >> 1;
                        df s = df_make(0.0f);
                        for (int q = 0; q < kWideEpt; ++q) {
                            const int r = r0 + q;
                            if (r < nl && val_key<BF16>(lval[r]) >= mid) s = df_sum(s, ework[r]);
                        }
                        const df tot = wide_sum_df(s, sh.red_df);
                        if (!df_less(tot, target))
                            lo = mid;
                        else
                            hi = mid;
                    }
                    cut = static_cast<uint32_t>(lo);
                    df above = df_make(0.0f);
                    uint32_t ceq = 0;
                    for (int q = 0; q < kWideEpt; ++q) {
                        const int r = r0 + q;
                        if (r < nl) {
                            const uint32_t key = val_key<BF16>(lval[r]);
                            if (key > cut) {
                                above = df_sum(above, ework[r]);
                            } else if (key == cut) {
                                ++ceq;
                                sh.e_cut = ework[r];  // every tie has the same weight
                            }
                        }
                    }
                    const df mass_gt = wide_sum_df(above, sh.red_df);
                    const int cnt_eq = static_cast<int>(wide_sum_u32(ceq, sh.red_u));
                    if (tid == 0) {
                        // the fewest ties at the cut that bring the mass to target
                        const df ec = sh.e_cut;
                        const df delta = df_sum(target, df_neg(mass_gt));
                        int m = 1;
                        if (ec.hi > 0.0f) {
                            const float f = ceilf(df_val(delta) / df_val(ec));
                            m = f < 1.0f ? 1 : (f > static_cast<float>(cnt_eq) ? cnt_eq : static_cast<int>(f));
                        }
                        if (m < 1) m = 1;
                        while (m > 1 && !df_less(df_sum(mass_gt, df_mul_f(ec, static_cast<float>(m - 1))), target)) --m;
                        while (m < cnt_eq && df_less(df_sum(mass_gt, df_mul_f(ec, static_cast<float>(m))), target)) ++m;
                        sh.m_cut = m;
                        sh.S = df_sum(mass_gt, df_mul_f(ec, static_cast<float>(m)));
                    }
                    __syncthreads();
                    m_cut = sh.m_cut;
                    S = sh.S;
                }
            }
        }

        // ------------------------------------------------ 4. p'(x_i)
        float px = 0.0f;
        if (!bad && i < k) {
            const int x = sh.xs[i];
            if (tid == 0) sh.xr = -1;
            __syncthreads();
            const int r0 = tid * kWideEpt;
            for (int q = 0; q < kWideEpt; ++q)
                if (r0 + q < nl && lidx[r0 + q] == x) sh.xr = r0 + q;
            __syncthreads();
            const int xr = sh.xr;
            if (xr >= 0) {
                const uint32_t xkey = val_key<BF16>(lval[xr]);
                uint32_t before = 0;  // ties at the cut ahead of x in vocabulary order
                if (cut != 0 && xkey == cut)
                    for (int q = 0; q < kWideEpt; ++q) {
                        const int r = r0 + q;
                        if (r < xr && val_key<BF16>(lval[r]) == cut) ++before;
                    }
                const uint32_t rank = wide_sum_u32(before, sh.red_u);  // uniform branch: xkey is the same everywhere
                const bool kept = xkey > cut || (xkey == cut && static_cast<int>(rank) < m_cut);
                if (kept) px = df_val(ework[xr]) / df_val(S);
            }
        }
        if (tid == 0) {
            sh.lpx[i] = px;
            sh.lbad[i] = bad ? 1 : 0;
            WideSlot& s = sh.slot[p];
            s.S = S;
            s.M = M;
            s.cut = cut;
            s.m_cut = m_cut;
            s.n = nl;
            s.bad = bad ? 1 : 0;
        }
        __syncthreads();
    }

    // the leader's walk inputs (lane i: position i), loaded before the barrier
    float pu0 = 0.0f, pu1 = 0.0f, pqx = 0.0f;
    if (crank == 0 && warp == 0 && lane <= k) {
        const long long ub = (static_cast<long long>(b) * (k + 1) + lane) * 2;
        pu0 = __ldg(a.u + ub);
        pu1 = __ldg(a.u + ub + 1);
        const int x = lane < k ? sh.xs[lane] : -1;
        if (x >= 0 && x < n) pqx = a.q ? __ldg(a.q + (static_cast<long long>(b) * k + lane) * a.V + x) : 1.0f;
    }
    cluster_wait();  // every CTA of the cluster runs: its shared memory may be written
    if (tid == 0)
        for (int p = 0; p < P; ++p) {
            const int i = crank + C * p;
            st_cluster_u32(map_rank(smem_u32(&sh.px[i]), 0), __float_as_uint(sh.lpx[i]));
            st_cluster_u32(map_rank(smem_u32(&sh.pbad[i]), 0), static_cast<uint32_t>(sh.lbad[i]));
        }
    cluster_sync();  // #1: every position's p'(x_i) is in the leader

    // ---------------------------------------------------- the walk (leader, warp 0)
    if (crank == 0 && warp == 0) {
        int st = 0, j = 0;
        for (int i = 0; i <= k; ++i) {
            int pst = sh.pbad[i] ? ST_NONFINITE : 0;
            const int x = i < k ? sh.xs[i] : -1;
            float u0 = 0.0f, qx = 0.0f;
            if (i < k) {
                u0 = __shfl_sync(full, pu0, i);
                qx = __shfl_sync(full, pqx, i);
                if (x < 0 || x >= n) pst |= ST_TOKEN;
                if (!(u0 >= 0.0f && u0 < 1.0f)) pst |= ST_UNIFORM;
                if (x >= 0 && x < n && !(qx >= 0.0f && qx <= FLT_MAX)) pst |= ST_QBAD;
            }
            if (pst) {
                st |= pst;
                break;
            }
            if (i == k) {
                j = k;
                break;
            }
            const float rho = fminf(1.0f, sh.px[i] / fmaxf(qx, 1e-12f));
            if (!(u0 < rho)) {
                j = i;
                break;
            }
        }
        const float u1 = __shfl_sync(full, pu1, j);
        if (!st && !(u1 >= 0.0f && u1 < 1.0f)) st |= ST_UNIFORM;
        if (st & ST_ERRMASK) {
            if (lane <= k) a.out_tokens[static_cast<long long>(b) * (k + 1) + lane] = -1;
            if (lane == 0) {
                a.num_accepted[b] = 0;
                if (a.row_status) a.row_status[b] = st;
            }
        }
        if (lane < C) {
            st_cluster_u32(map_rank(smem_u32(&sh.dj), lane), static_cast<uint32_t>(j));
            st_cluster_u32(map_rank(smem_u32(&sh.dst), lane), static_cast<uint32_t>(st));
            st_cluster_u32(map_rank(smem_u32(&sh.du1), lane), __float_as_uint(u1));
        }
    }
    cluster_sync();  // #2: the decision is in every CTA; no shared memory is touched across CTAs after it
    const int j = sh.dj;
    int st = sh.dst;
    if ((st & ST_ERRMASK) || j % C != crank) return;

    // ---------------------------------------------------- the draw (the stop position's owner)
    const int p = j / C;
    const WideSlot sl = sh.slot[p];
    const int* lidx = reinterpret_cast<const int*>(dyn_smem + kWideWorkBytes + p * kWideSlotBytes);
    const float* lval = reinterpret_cast<const float*>(dyn_smem + kWideWorkBytes + p * kWideSlotBytes + kWideKMax * 4);
    const int nl = sl.n;
    const int r0 = tid * kWideEpt;
    const int mode = j < k ? (a.q ? MODE_RESIDUAL : MODE_ONEHOT) : MODE_BONUS;
    const int xj = j < k ? sh.xs[j] : -1;
    const float* qrow = a.q && j < k ? a.q + (static_cast<long long>(b) * k + j) * a.V : nullptr;
    rc.M = sl.M;
    uint32_t tc = 0;
    if (sl.cut != 0)
        for (int q = 0; q < kWideEpt; ++q)
            if (r0 + q < nl && val_key<BF16>(lval[r0 + q]) == sl.cut) ++tc;
    uint32_t ttot;
    uint32_t trank = wide_excl_scan_u32(tc, sh.red_u, ttot);
    df e[kWideEpt], w[kWideEpt];
    uint32_t inmask = 0;
    bool qbad = false;
    df local = df_make(0.0f);
#pragma unroll
    for (int q = 0; q < kWideEpt; ++q) {
        const int r = r0 + q;
        e[q] = df_make(0.0f);
        w[q] = df_make(0.0f);
        if (r < nl) {
            const float l = lval[r];
            const uint32_t key = val_key<BF16>(l);
            bool in = key > sl.cut;
            if (sl.cut != 0 && key == sl.cut) {
                in = static_cast<int>(trank) < sl.m_cut;
                ++trank;
            }
            if (in) {
                inmask |= 1u << q;
                e[q] = l == -INFINITY ? df_make(0.0f) : precise_e<BF16>(l, rc, sh.exp2tab);
                if (mode == MODE_BONUS) {
                    w[q] = e[q];
                } else {
                    const int v = lidx[r];
                    const float qv = qrow ? __ldg(qrow + v) : (v == xj ? 1.0f : 0.0f);
                    qbad |= !(qv >= 0.0f && qv <= FLT_MAX);
                    const df rr = minus_sq(e[q], sl.S, qv);
                    w[q] = rr.hi + rr.lo > 0.0f ? rr : df_make(0.0f);
                }
                local = df_sum(local, w[q]);
            }
        }
    }
    if (__syncthreads_or(qbad ? 1 : 0)) st |= ST_QBAD;
    if (!(st & ST_ERRMASK)) {
        df W = wide_sum_df(local, sh.red_df);
        if (mode != MODE_BONUS && !(W.hi + W.lo > 0.0f)) {  // zero residual mass: draw from p'
            st |= ST_ZERO_RESIDUAL;
            local = df_make(0.0f);
#pragma unroll
            for (int q = 0; q < kWideEpt; ++q) {
                w[q] = ((inmask >> q) & 1u) ? e[q] : df_make(0.0f);
                local = df_sum(local, w[q]);
            }
            W = wide_sum_df(local, sh.red_df);
        }
        const df target = df_mul_f(W, sh.du1);
        df pre = wide_excl_scan_df(local, sh.red_df);
        uint32_t cand = 0xffffffffu, lastpos = 0;  // lastpos: 1 + the last positive entry
#pragma unroll
        for (int q = 0; q < kWideEpt; ++q) {
            const int r = r0 + q;
            if (r < nl) {
                pre = df_sum(pre, w[q]);
                if (w[q].hi + w[q].lo > 0.0f) {
                    lastpos = static_cast<uint32_t>(r + 1);
                    if (cand == 0xffffffffu && df_less(target, pre)) cand = static_cast<uint32_t>(r);
                }
            }
        }
        cand = wide_min_u32(cand, sh.red_u);
        lastpos = wide_max_u32(lastpos, sh.red_u);
        // only through rounding at the top edge: the last entry with positive weight
        const int rs = cand != 0xffffffffu ? static_cast<int>(cand) : static_cast<int>(lastpos) - 1;
        const int token = rs >= 0 ? lidx[rs] : -1;
        if (tid <= k) a.out_tokens[static_cast<long long>(b) * (k + 1) + tid] = tid < j ? sh.xs[tid] : (tid == j ? token : -1);
        if (tid == 0) {
            a.num_accepted[b] = j;
            if (a.row_status) a.row_status[b] = st;
        }
    } else {
        if (tid <= k) a.out_tokens[static_cast<long long>(b) * (k + 1) + tid] = -1;
        if (tid == 0) {
            a.num_accepted[b] = 0;
            if (a.row_status) a.row_status[b] = st;
        }
    }
}

}  // namespace specv
