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
// One thread-block cluster of C = min(k + 1, 16) CTAs of 256 threads per
// sequence; CTA c owns positions c and c + C.  A position's kept set is found
// exactly, with no sort of the vocabulary:
//   1. a radix select on the logits' order-preserving keys finds key*, the key
//      of the K-th largest entry, and how many entries lie above it.  The
//      first pass counts every entry by its key's top 12 bits (two keys a
//      32-bit word for bf16).  bf16 rows then take one more pass that marks
//      the entries of the higher bins in one bitmap of the vocabulary and
//      those of key*'s bin in a second, and counts that bin's last 4 bits
//      (key*); the bin's entries are read again and sorted into the two
//      bitmaps (above key*, equal to it).  fp32 rows take two more digit
//      passes (12 and 8 bits) and a marking pass.  The later passes skip, by
//      packed compares, the entries below the range that matters;
//   2. a block scan over the two bitmaps in vocabulary order keeps the ties
//      that fit (the lowest indices first) and writes the kept list, index
//      and logit, at most 4096 entries, into shared memory;
//   3. on the list: the maximum M and, for top_p < 1, the first rank (key
//      descending, index ascending) where the prefix of the weights
//      e = exp((l - M) / T) (double-float exponential and sums) reaches top_p
//      of the total: that entry's (key, index) is the cut.  The prefix comes
//      per key from a count histogram of the list when its keys span at most
//      4096 values (bf16: a key's entries share one weight), else from a
//      bitonic sort of the list;
//   4. p'(x_i) goes to the leader CTA over distributed shared memory.
// After a cluster barrier the leader's warp 0 walks the positions, and the
// CTA that owns the stop position draws from its kept list: weights in
// double-float, a block scan in vocabulary order, the first entry whose
// prefix exceeds u * W.  Threads walk 16 consecutive list entries; the lists
// hold a pad word after every 16 so that a warp's accesses spread over the
// banks.
#pragma once
#include <cfloat>
#include <climits>
#include <cstdint>

#include <cuda_bf16.h>

#include "exp2dd.cuh"
#include "ptx.cuh"
#include "verify_cluster.cuh"
#include "verify_topk.cuh"

namespace specv {

constexpr int kWideThreads = 256;
constexpr int kWideWarps = kWideThreads / 32;
constexpr int kWideEpt = kWideKMax / kWideThreads;  // kept-list entries per thread
constexpr int kWideClusterMax = 16;                // CTAs per sequence
constexpr int kWideListPad = kWideKMax + kWideKMax / 16;  // a kept list with a pad word after every 16 entries
constexpr int kWideSlotBytes = kWideListPad * 8;   // one position's kept list: index and logit
constexpr int kWideSlots = (kMaxK + kWideClusterMax) / kWideClusterMax;  // positions a CTA owns at most
constexpr int kWideHistBins = 4096;                // 12-bit digits
static_assert(kWideEpt * kWideThreads == kWideKMax, "the kept list is split evenly over the threads");

// Place of kept-list entry r: one pad word after every 16 entries, so that
// threads walking 16 consecutive entries each touch 32 different banks.
__device__ __forceinline__ int lp(int r) { return r + (r >> 4); }

inline int wide_cluster(int k) { return k + 1 < kWideClusterMax ? k + 1 : kWideClusterMax; }

// Work area: the digit histogram, then the two bitmaps, then the top-p cut's
// histogram or sort keys, then the draw's weights.
__host__ __device__ inline int wide_work_bytes(long long V) {
    const long long bitmaps = 2 * ((V + 31) / 32) * 4;
    const long long least = kWideListPad * 8;  // the draw's weights (and the sort keys, and 4096 bins)
    return static_cast<int>(bitmaps > least ? bitmaps : least);
}

// Dynamic shared memory: the work area, then one kept list per owned position.
inline size_t wide_dyn_smem(int k, long long V) {
    const int C = wide_cluster(k);
    const int P = (k + C) / C;  // ceil((k + 1) / C)
    return static_cast<size_t>(wide_work_bytes(V)) + static_cast<size_t>(P) * kWideSlotBytes;
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

// key16 of both halves of a word at once: a set sign bit flips all 16 bits,
// a clear one the sign bit only; -0 (which comes out 0x7fff) is moved to +0.
__device__ __forceinline__ uint32_t key16x2(uint32_t w) {
    const uint32_t k = w ^ 0x80008000u ^ (((w >> 15) & 0x00010001u) * 0x7fffu);
    return k + (__vcmpeq2(k, 0x7fff7fffu) & 0x00010001u);
}

template <bool BF16>
__device__ __forceinline__ uint32_t val_key(float v) {
    return BF16 ? key16(__float_as_uint(v) >> 16) : key32(__float_as_uint(v));
}

// The value of a key (NaN for the keys no logit has).
template <bool BF16>
__device__ __forceinline__ float key_val(uint32_t key) {
    if (BF16) {
        const uint32_t b = (key & 0x8000u) ? (key ^ 0x8000u) : (~key & 0xffffu);
        return __uint_as_float(b << 16);
    }
    return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

template <bool BF16>
__device__ __forceinline__ float ld_val(const unsigned char* rowp, int e) {
    if (BF16) return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(rowp) + e)) << 16);
    return __ldg(reinterpret_cast<const float*>(rowp) + e);
}

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) {
    __nv_bfloat162 r;
    memcpy(&r, &w, 4);
    return r;
}

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) {
    uint32_t r;
    memcpy(&r, &v, 4);
    return r;
}

// Level 0: every entry of the row counted by its key's top 12 bits; returns
// whether this thread met a NaN or +inf (the row is then refused, and what
// the counts hold does not matter).  Threads take 16-byte groups in turn.
template <bool BF16>
__device__ __forceinline__ bool wide_hist0(const unsigned char* rowp, int n, int h, int ng, uint32_t* hist) {
    constexpr int G = BF16 ? 8 : 4;
    constexpr int esz = BF16 ? 2 : 4;
    const int tid = threadIdx.x;
    bool bad = false;
    auto scalar = [&](int e) {
        uint32_t key;
        if (BF16) {
            const uint32_t b = __ldg(reinterpret_cast<const unsigned short*>(rowp) + e);
            bad |= (b & 0x7fffu) > 0x7f80u || b == 0x7f80u;
            key = key16(b);
            atomicAdd(&hist[key >> 4], 1u);
        } else {
            const uint32_t f = __float_as_uint(__ldg(reinterpret_cast<const float*>(rowp) + e));
            bad |= (f & 0x7fffffffu) > 0x7f800000u || f == 0x7f800000u;
            key = key32(f);
            atomicAdd(&hist[key >> 20], 1u);
        }
    };
    if (tid < h) scalar(tid);
    const int t0 = h + ng * G;
    if (tid < n - t0) scalar(t0 + tid);
    uint32_t mxb = BF16 ? 0xff80ff80u : __float_as_uint(-INFINITY);  // running maximum, NaN kept
    for (int base = 0; base < ng; base += 4 * kWideThreads) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = base + u * kWideThreads + tid;
            w[u] = g < ng ? __ldg(reinterpret_cast<const uint4*>(rowp + (static_cast<long long>(h) + static_cast<long long>(g) * G) * esz))
                          : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = base + u * kWideThreads + tid;
            if (g < ng) {
                const uint32_t wd[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    if (BF16) {
                        mxb = bf2_bits(__hmax2_nan(as_bf2(mxb), as_bf2(wd[m])));
                        const uint32_t k = key16x2(wd[m]);
                        atomicAdd(&hist[(k >> 4) & 0xfffu], 1u);
                        atomicAdd(&hist[k >> 20], 1u);
                    } else {
                        mxb = __float_as_uint(max_nan_f32(__uint_as_float(mxb), __uint_as_float(wd[m])));
                        uint32_t k = wd[m] ^ (static_cast<uint32_t>(static_cast<int>(wd[m]) >> 31) | 0x80000000u);
                        k += k == 0x7fffffffu ? 1u : 0u;
                        atomicAdd(&hist[k >> 20], 1u);
                    }
                }
            }
        }
    }
    if (BF16) {
        const uint32_t lo = mxb & 0xffffu, hi = mxb >> 16;
        bad |= (lo & 0x7fffu) > 0x7f80u || lo == 0x7f80u || (hi & 0x7fffu) > 0x7f80u || hi == 0x7f80u;
    } else {
        bad |= (mxb & 0x7fffffffu) > 0x7f800000u || mxb == 0x7f800000u;
    }
    return bad;
}

// The later passes: f(e, key) for every entry of a 16-byte group whose
// largest value is at least vmin (and for the scalar head and tail), so that
// the groups entirely below the range of interest cost one packed maximum.
// The row is finite here (level 0 refused it otherwise).
template <bool BF16, typename F>
__device__ __forceinline__ void wide_scan(const unsigned char* rowp, int n, int h, int ng, float vmin, F&& f) {
    constexpr int G = BF16 ? 8 : 4;
    constexpr int esz = BF16 ? 2 : 4;
    const int tid = threadIdx.x;
    if (tid < h) {
        const float v = ld_val<BF16>(rowp, tid);
        f(tid, val_key<BF16>(v));
    }
    const int t0 = h + ng * G;
    if (tid < n - t0) {
        const float v = ld_val<BF16>(rowp, t0 + tid);
        f(t0 + tid, val_key<BF16>(v));
    }
    for (int base = 0; base < ng; base += 4 * kWideThreads) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = base + u * kWideThreads + tid;
            w[u] = g < ng ? __ldg(reinterpret_cast<const uint4*>(rowp + (static_cast<long long>(h) + static_cast<long long>(g) * G) * esz))
                          : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = base + u * kWideThreads + tid;
            if (g >= ng) continue;
            const uint32_t wd[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
            float gm;
            if (BF16) {
                const __nv_bfloat162 a = __hmax2(__hmax2(as_bf2(wd[0]), as_bf2(wd[1])), __hmax2(as_bf2(wd[2]), as_bf2(wd[3])));
                gm = fmaxf(__low2float(a), __high2float(a));
            } else {
                gm = fmaxf(fmaxf(__uint_as_float(wd[0]), __uint_as_float(wd[1])),
                           fmaxf(__uint_as_float(wd[2]), __uint_as_float(wd[3])));
            }
            if (!(gm >= vmin)) continue;
            const int e0 = h + g * G;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (BF16) {
                    const uint32_t k = key16x2(wd[m]);
                    f(e0 + 2 * m, k & 0xffffu);
                    f(e0 + 2 * m + 1, k >> 16);
                } else {
                    f(e0 + m, key32(wd[m]));
                }
            }
        }
    }
}

// The second pass of bf16 rows: every entry whose first digit is above d1
// is marked in A, every entry of bin d1 in B, and the bin's last digits are
// counted.  One packed compare a word finds a group's entries at or above
// the bin (a few percent of the row); the warp then runs the marking as many
// times as its busiest lane has such entries, instead of issuing a
// predicated step for every entry.
__device__ __forceinline__ void wide_pass2_bf16(const unsigned char* rowp, int n, int h, int ng, uint32_t d1, float vmin,
                                                uint32_t* A, uint32_t* Bm, uint32_t* hist1) {
    const int tid = threadIdx.x;
    const unsigned full = 0xffffffffu;
    auto mark = [&](int e, uint32_t key) {
        const uint32_t dg = key >> 4;
        if (dg > d1) {
            atomicOr(&A[e >> 5], 1u << (e & 31));
        } else if (dg == d1) {
            atomicOr(&Bm[e >> 5], 1u << (e & 31));
            atomicAdd(&hist1[key & 15u], 1u);
        }
    };
    const unsigned short* row16 = reinterpret_cast<const unsigned short*>(rowp);
    if (tid < h) mark(tid, key16(__ldg(row16 + tid)));
    const int t0 = h + ng * 8;
    if (tid < n - t0) mark(t0 + tid, key16(__ldg(row16 + t0 + tid)));
    const __nv_bfloat162 vmin2 = __float2bfloat162_rn(vmin);  // exact: a bf16 value or -inf
    for (int base = 0; base < ng; base += 4 * kWideThreads) {
        uint4 w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = base + u * kWideThreads + tid;
            w[u] = g < ng ? __ldg(reinterpret_cast<const uint4*>(rowp + (static_cast<long long>(h) + static_cast<long long>(g) * 8) * 2))
                          : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int g = base + u * kWideThreads + tid;
            uint32_t rel = 0;  // bit q: entry q of the group is at or above vmin
            if (g < ng) {
                const uint32_t m0 = __hge2_mask(as_bf2(w[u].x), vmin2), m1 = __hge2_mask(as_bf2(w[u].y), vmin2);
                const uint32_t m2 = __hge2_mask(as_bf2(w[u].z), vmin2), m3 = __hge2_mask(as_bf2(w[u].w), vmin2);
                rel = (m0 & 1u) | ((m0 >> 15) & 2u) | ((m1 & 1u) << 2) | ((m1 >> 13) & 8u) | ((m2 & 1u) << 4) |
                      ((m2 >> 11) & 32u) | ((m3 & 1u) << 6) | ((m3 >> 9) & 128u);
            }
            const int rounds = __reduce_max_sync(full, static_cast<unsigned>(__popc(rel)));
            const int e0 = h + g * 8;
            for (int it = 0; it < rounds; ++it) {
                if (rel) {
                    const int q = __ffs(rel) - 1;
                    rel &= rel - 1;
                    const int wi = q >> 1;  // (selects, not an indexed array: no local memory)
                    const uint32_t wd = wi < 2 ? (wi == 0 ? w[u].x : w[u].y) : (wi == 2 ? w[u].z : w[u].w);
                    mark(e0 + q, key16((q & 1) ? (wd >> 16) : (wd & 0xffffu)));
                }
            }
        }
    }
}

struct WideSlot {
    df S;             // mass of the kept set P, in e-units
    float M;          // the row maximum
    uint32_t cut;     // P: list entries with a key above cut, or equal to it
    int cutidx;       // with an index up to cutidx (cut 0: every entry)
    int n;            // kept-list entries: min(top_k, V)
    int bad;          // a NaN or +inf logit, or every logit -inf
};

struct alignas(16) WideSmem {
    float2 exp2tab[128];
    WideSlot slot[kWideSlots];
    df red_df[kWideWarps];
    uint32_t red_u[kWideWarps];
    float red_f[kWideWarps];
    int xs[kMaxK + 1];
    float lpx[kMaxK + 1];        // this CTA's p'(x_i) and flags, pushed to the leader at the end
    int lbad[kMaxK + 1];
    float px[kMaxK + 1];         // the leader's copy of every position's
    int pbad[kMaxK + 1];
    int dstar;
    uint32_t dabove;
    df S;
    uint32_t hist1[16];          // bf16 rows: the last digit of the entries in key*'s first-digit bin
    int mties;                   // ties at the top-p cut that are kept
    int cutidx;
    float xpx;
    int dj, dst;                 // the decision (written by the leader into every CTA)
    float du1;
};

// Block-wide helpers over the CTA's threads; each ends with a barrier, so the
// scratch may be reused at once.
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

// Exclusive prefix of pairs in thread order, and the total.
__device__ __forceinline__ df wide_excl_scan_df(df v, df* red, df& total) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const df incl = df_warp_incl_scan(v, lane);
    if (lane == 31) red[w] = incl;
    __syncthreads();
    df base = df_make(0.0f), tot = df_make(0.0f);
    for (int i = 0; i < kWideWarps; ++i) {
        if (i == w) base = tot;
        tot = df_sum(tot, red[i]);
    }
    __syncthreads();
    total = tot;
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

// Bitonic sort of n2 (a power of two, at most kWideKMax) 64-bit keys in
// shared memory into descending order.
__device__ __forceinline__ void wide_sort_desc(unsigned long long* s, int n2) {
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < (n2 >> 1); i += kWideThreads) {
                const int a = ((i & ~(stride - 1)) << 1) | (i & (stride - 1));
                const int c = a + stride;
                const unsigned long long x = s[a], y = s[c];
                const bool desc = (a & size) == 0;
                if ((x < y) == desc) {
                    s[a] = y;
                    s[c] = x;
                }
            }
            __syncthreads();
        }
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kWideThreads, 3) verify_topk_wide_kernel(const VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ WideSmem sh;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int G = 16 / esz;
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

    const int work_bytes = wide_work_bytes(a.V);
    uint32_t* work = reinterpret_cast<uint32_t*>(dyn_smem);
    const int nwords = (n + 31) >> 5;
    uint32_t* strict_bm = work;         // entries above key*
    uint32_t* tie_bm = work + nwords;   // entries equal to key*
    unsigned long long* skeys = reinterpret_cast<unsigned long long*>(dyn_smem);
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
    const int r0 = tid * kWideEpt;      // this thread's kept-list entries

    for (int p = 0; p < P; ++p) {
        const int i = crank + C * p;
        int* lidx = reinterpret_cast<int*>(dyn_smem + work_bytes + p * kWideSlotBytes);
        float* lval = reinterpret_cast<float*>(dyn_smem + work_bytes + p * kWideSlotBytes + kWideListPad * 4);
        const unsigned char* rowp = reinterpret_cast<const unsigned char*>(a.logits) +
                                    (static_cast<long long>(b) * (k + 1) + i) * static_cast<long long>(n) * esz;
        int h = static_cast<int>(((16 - (reinterpret_cast<uintptr_t>(rowp) & 15)) & 15) / esz);
        if (h > n) h = n;
        const int ng = (n - h) / G;

        // ------------------------------------------------ 1. radix select of key*
        for (int d = tid; d < kWideHistBins; d += kWideThreads) work[d] = 0u;
        __syncthreads();
        bool bad = __syncthreads_or(wide_hist0<BF16>(rowp, n, h, ng, work) ? 1 : 0) != 0;
        uint32_t prefix = 0, c_above = 0;
        int pbits = BF16 ? 4 : 20;  // key bits below the digits found so far
        if (!bad) {
            wide_find_digit(work, kWideHistBins, static_cast<uint32_t>(Kp), sh);
            if (sh.dstar < 0) bad = true;  // cannot happen on a finite row
            else {
                c_above = sh.dabove;
                prefix = static_cast<uint32_t>(sh.dstar);
            }
        }
        // bf16 rows: one more pass marks the entries of the higher first-digit
        // bins in the first bitmap and those of key*'s bin in the second, and
        // counts the bin's last digits, which give key*; the bin's entries are
        // then sorted into the two bitmaps by their logits, read again (a few
        // thousand at most on ordinary rows).  No store in the pass waits for
        // a reply.
        const bool fast = BF16 && !bad;
        if (fast) {
            const uint32_t d1 = prefix;
            __syncthreads();  // the histogram is read no more
            for (int d = tid; d < 2 * nwords; d += kWideThreads) work[d] = 0u;
            if (tid < 16) sh.hist1[tid] = 0u;
            __syncthreads();
            float vmin = key_val<BF16>(d1 << 4);
            if (vmin != vmin) vmin = -INFINITY;
            wide_pass2_bf16(rowp, n, h, ng, d1, vmin, strict_bm, tie_bm, sh.hist1);
            __syncthreads();
            wide_find_digit(sh.hist1, 16, static_cast<uint32_t>(Kp) - c_above, sh);
            if (sh.dstar < 0) {
                bad = true;
            } else {
                c_above += sh.dabove;
                prefix = (prefix << 4) | static_cast<uint32_t>(sh.dstar);
                pbits = 0;
                // this thread's words: the bin's entries above key* move to the
                // first bitmap, those below leave the second (ties stay)
                const int wpt = (nwords + kWideThreads - 1) / kWideThreads;
                const int w0 = min(nwords, tid * wpt), w1 = min(nwords, w0 + wpt);
                constexpr int kBatch = 16;
                int eb[kBatch];
                int nbat = 0;
                auto classify = [&]() {
                    float vb[kBatch];
#pragma unroll
                    for (int q = 0; q < kBatch; ++q) vb[q] = q < nbat ? ld_val<BF16>(rowp, eb[q]) : 0.0f;
#pragma unroll
                    for (int q = 0; q < kBatch; ++q)
                        if (q < nbat) {
                            const uint32_t key = val_key<BF16>(vb[q]);
                            const int e = eb[q];
                            const uint32_t bit = 1u << (e & 31);
                            if (key > prefix) strict_bm[e >> 5] |= bit;
                            if (key != prefix) tie_bm[e >> 5] &= ~bit;
                        }
                    nbat = 0;
                };
                for (int w = w0; w < w1; ++w)
                    for (uint32_t m = tie_bm[w]; m;) {
                        const int bit = __ffs(m) - 1;
                        m &= m - 1;
                        eb[nbat++] = w * 32 + bit;
                        if (nbat == kBatch) classify();
                    }
                classify();
                __syncthreads();
            }
        }
        const int nlev = fast ? 0 : (BF16 ? 1 : 2);  // digits after the first, on the general path
        for (int lev = 0; lev < nlev && !bad; ++lev) {
            const int width = BF16 ? 4 : (lev == 0 ? 12 : 8);
            const int shift = pbits - width;
            const int nb = 1 << width;
            for (int d = tid; d < nb; d += kWideThreads) work[d] = 0u;
            __syncthreads();
            float vmin = key_val<BF16>(prefix << pbits);
            if (vmin != vmin) vmin = -INFINITY;
            wide_scan<BF16>(rowp, n, h, ng, vmin, [&](int, uint32_t key) {
                if ((key >> pbits) == prefix) atomicAdd(&work[(key >> shift) & (nb - 1)], 1u);
            });
            __syncthreads();
            wide_find_digit(work, nb, static_cast<uint32_t>(Kp) - c_above, sh);
            if (sh.dstar < 0) {
                bad = true;
            } else {
                c_above += sh.dabove;
                prefix = (prefix << width) | static_cast<uint32_t>(sh.dstar);
                pbits = shift;
            }
        }

        int nl = 0;
        float M = -INFINITY;
        uint32_t cut = 0;
        int cutidx = 0;
        df S = df_make(0.0f);
        if (!bad) {
            // -------------------------------------------- 2. the kept list
            const uint32_t kstar = prefix;
            const uint32_t t = static_cast<uint32_t>(Kp) - c_above;  // ties at key* kept (>= 1)
            if (!fast) {
                for (int d = tid; d < 2 * nwords; d += kWideThreads) work[d] = 0u;
                __syncthreads();
                wide_scan<BF16>(rowp, n, h, ng, key_val<BF16>(kstar), [&](int e, uint32_t key) {
                    if (key > kstar)
                        atomicOr(&strict_bm[e >> 5], 1u << (e & 31));
                    else if (key == kstar)
                        atomicOr(&tie_bm[e >> 5], 1u << (e & 31));
                });
                __syncthreads();
            }
            {
                const int wpt = (nwords + kWideThreads - 1) / kWideThreads;
                const int w0 = min(nwords, tid * wpt), w1 = min(nwords, w0 + wpt);
                uint32_t ct = 0;
                for (int w = w0; w < w1; ++w) ct += __popc(tie_bm[w]);
                uint32_t ttot;
                uint32_t tseen = wide_excl_scan_u32(ct, sh.red_u, ttot);  // ties in lower words
                // the ties this thread keeps (the first t of the row in vocabulary
                // order) join its words of the first bitmap, which then holds the list
                uint32_t cs = 0;
                for (int w = w0; w < w1; ++w) {
                    uint32_t tm = tie_bm[w], kt = 0;
                    while (tm && tseen < t) {
                        const uint32_t low = tm & (0u - tm);
                        kt |= low;
                        tm ^= low;
                        ++tseen;
                    }
                    const uint32_t kw = strict_bm[w] | kt;
                    strict_bm[w] = kw;
                    cs += __popc(kw);
                }
                uint32_t total;
                uint32_t pos = wide_excl_scan_u32(cs, sh.red_u, total);
                for (int w = w0; w < w1; ++w)
                    for (uint32_t m = strict_bm[w]; m;) {
                        const int bit = __ffs(m) - 1;
                        m &= m - 1;
                        if (pos < static_cast<uint32_t>(kWideKMax)) lidx[lp(pos)] = w * 32 + bit;
                        ++pos;
                    }
                nl = static_cast<int>(min(total, static_cast<uint32_t>(kWideKMax)));
                bad = total != static_cast<uint32_t>(Kp);  // cannot happen on a finite row
            }
            __syncthreads();
            {
                float lv[kWideEpt];  // the loads issued together, then stored
#pragma unroll
                for (int q = 0; q < kWideEpt; ++q) {
                    const int r = tid + q * kWideThreads;
                    lv[q] = r < nl ? ld_val<BF16>(rowp, lidx[lp(r)]) : 0.0f;
                }
#pragma unroll
                for (int q = 0; q < kWideEpt; ++q) {
                    const int r = tid + q * kWideThreads;
                    if (r < nl) lval[lp(r)] = lv[q];
                }
            }
            __syncthreads();

            // -------------------------------------------- 3. the maximum, the weights' sum, the top-p cut
            float mx = -INFINITY;
            for (int q = 0; q < kWideEpt; ++q)
                if (r0 + q < nl) mx = fmaxf(mx, lval[lp(r0 + q)]);
            M = wide_max_f(mx, sh.red_f);
            if (!(M > -INFINITY)) bad = true;
            if (!bad) {
                rc.M = M;
                if (top_p < 1.0f) {
                    uint32_t kmn = 0xffffffffu;
                    for (int q = 0; q < kWideEpt; ++q)
                        if (r0 + q < nl) kmn = min(kmn, val_key<BF16>(lval[lp(r0 + q)]));
                    kmn = wide_min_u32(kmn, sh.red_u);
                    const uint32_t kmx = val_key<BF16>(M);
                    if (BF16 && kmx - kmn < static_cast<uint32_t>(kWideHistBins)) {
                        // every entry with one key has one weight: bin b counts the
                        // entries with key kmx - b (rank order), its mass is count * e
                        const int R = static_cast<int>(kmx - kmn) + 1;
                        uint32_t* cnt = work;
                        for (int d = tid; d < R; d += kWideThreads) cnt[d] = 0u;
                        __syncthreads();
                        for (int q = 0; q < kWideEpt; ++q)
                            if (r0 + q < nl) atomicAdd(&cnt[kmx - val_key<BF16>(lval[lp(r0 + q)])], 1u);
                        __syncthreads();
                        const int bpt = (R + kWideThreads - 1) / kWideThreads;
                        const int b0 = min(R, tid * bpt), b1 = min(R, b0 + bpt);
                        auto bin_e = [&](int bn) {
                            const float l = key_val<BF16>(kmx - static_cast<uint32_t>(bn));
                            return l == -INFINITY ? df_make(0.0f) : precise_e<BF16>(l, rc, sh.exp2tab);
                        };
                        df part = df_make(0.0f);
                        for (int bn = b0; bn < b1; ++bn) {
                            const uint32_t cn = cnt[bn];
                            if (cn) part = df_sum(part, df_mul_f(bin_e(bn), static_cast<float>(cn)));
                        }
                        df SK;
                        df c = wide_excl_scan_df(part, sh.red_df, SK);
                        const df target = df_mul_f(SK, top_p);
                        uint32_t cand = 0xffffffffu, ccount = 0;
                        df above = df_make(0.0f), ecut = df_make(0.0f);
                        for (int bn = b0; bn < b1; ++bn) {
                            const uint32_t cn = cnt[bn];
                            if (!cn) continue;
                            const df eb = bin_e(bn);
                            const df before = c;
                            c = df_sum(c, df_mul_f(eb, static_cast<float>(cn)));
                            if (cand == 0xffffffffu && !df_less(c, target)) {
                                cand = static_cast<uint32_t>(bn);
                                above = before;
                                ecut = eb;
                                ccount = cn;
                            }
                        }
                        const uint32_t first = wide_min_u32(cand, sh.red_u);
                        if (first != 0xffffffffu && cand == first) {
                            // the fewest ties at this key that bring the mass to target
                            const int ce = static_cast<int>(ccount);
                            int m = 1;
                            if (ecut.hi > 0.0f) {
                                const float f = ceilf(df_val(df_sum(target, df_neg(above))) / df_val(ecut));
                                m = f < 1.0f ? 1 : (f > static_cast<float>(ce) ? ce : static_cast<int>(f));
                            }
                            while (m > 1 && !df_less(df_sum(above, df_mul_f(ecut, static_cast<float>(m - 1))), target)) --m;
                            while (m < ce && df_less(df_sum(above, df_mul_f(ecut, static_cast<float>(m))), target)) ++m;
                            sh.mties = m;
                            sh.S = df_sum(above, df_mul_f(ecut, static_cast<float>(m)));
                        }
                        __syncthreads();
                        if (first == 0xffffffffu) {  // through rounding only: every entry
                            S = SK;
                        } else {
                            // the cut: the m-th entry (vocabulary order) with the cut key
                            cut = kmx - first;
                            const uint32_t m = static_cast<uint32_t>(sh.mties);
                            S = sh.S;
                            uint32_t mine = 0;
                            for (int q = 0; q < kWideEpt; ++q)
                                if (r0 + q < nl && val_key<BF16>(lval[lp(r0 + q)]) == cut) ++mine;
                            uint32_t tot;
                            uint32_t seen = wide_excl_scan_u32(mine, sh.red_u, tot);
                            if (seen < m && m <= seen + mine)
                                for (int q = 0; q < kWideEpt; ++q)
                                    if (r0 + q < nl && val_key<BF16>(lval[lp(r0 + q)]) == cut && ++seen == m) sh.cutidx = lidx[lp(r0 + q)];
                            __syncthreads();
                            cutidx = sh.cutidx;
                        }
                    } else {
                        // rank order: key descending, then index ascending (one 64-bit key)
                        int n2 = 2;
                        while (n2 < nl) n2 <<= 1;
                        for (int r = tid; r < n2; r += kWideThreads)
                            skeys[r] = r < nl ? (static_cast<unsigned long long>(val_key<BF16>(lval[lp(r)])) << 32) |
                                                    (0xffffffffu - static_cast<uint32_t>(lidx[lp(r)]))
                                              : 0ull;
                        __syncthreads();
                        wide_sort_desc(skeys, n2);
                        auto rank_e = [&](int r) {  // the weight at rank r (the same value on every call)
                            if (r >= nl) return df_make(0.0f);
                            const float l = key_val<BF16>(static_cast<uint32_t>(skeys[r] >> 32));
                            return l == -INFINITY ? df_make(0.0f) : precise_e<BF16>(l, rc, sh.exp2tab);
                        };
                        df part = df_make(0.0f);
                        for (int q = 0; q < kWideEpt; ++q) part = df_sum(part, rank_e(r0 + q));
                        df SK;
                        df c = wide_excl_scan_df(part, sh.red_df, SK);
                        const df target = df_mul_f(SK, top_p);
                        // the first rank whose prefix reaches target, and the prefix there
                        uint32_t cand = 0xffffffffu;
                        df cS = df_make(0.0f);
                        for (int q = 0; q < kWideEpt; ++q) {
                            const int r = r0 + q;
                            c = df_sum(c, rank_e(r));
                            if (r < nl && cand == 0xffffffffu && !df_less(c, target)) {
                                cand = static_cast<uint32_t>(r);
                                cS = c;
                            }
                        }
                        const uint32_t first = wide_min_u32(cand, sh.red_u);
                        if (first != 0xffffffffu && cand == first) sh.S = cS;
                        __syncthreads();
                        if (first == 0xffffffffu) {  // through rounding only: every entry
                            S = SK;
                        } else {
                            const unsigned long long ck = skeys[first];
                            cut = static_cast<uint32_t>(ck >> 32);
                            cutidx = static_cast<int>(0xffffffffu - static_cast<uint32_t>(ck));
                            S = sh.S;
                        }
                        __syncthreads();  // the sort keys are not read again
                    }
                } else {
                    df part = df_make(0.0f);
                    for (int q = 0; q < kWideEpt; ++q) {
                        const int r = r0 + q;
                        if (r < nl && lval[lp(r)] != -INFINITY) part = df_sum(part, precise_e<BF16>(lval[lp(r)], rc, sh.exp2tab));
                    }
                    S = wide_sum_df(part, sh.red_df);
                }
            }
        }

        // ------------------------------------------------ 4. p'(x_i)
        float px = 0.0f;
        if (!bad && i < k) {
            const int x = sh.xs[i];
            if (tid == 0) sh.xpx = 0.0f;
            __syncthreads();
            for (int q = 0; q < kWideEpt; ++q) {
                const int r = r0 + q;
                if (r < nl && lidx[lp(r)] == x) {
                    const float l = lval[lp(r)];
                    const uint32_t key = val_key<BF16>(l);
                    if (l != -INFINITY && (key > cut || (key == cut && x <= cutidx)))
                        sh.xpx = df_val(precise_e<BF16>(l, rc, sh.exp2tab)) / df_val(S);
                }
            }
            __syncthreads();
            px = sh.xpx;
        }
        if (tid == 0) {
            sh.lpx[i] = px;
            sh.lbad[i] = bad ? 1 : 0;
            WideSlot& s = sh.slot[p];
            s.S = S;
            s.M = M;
            s.cut = cut;
            s.cutidx = cutidx;
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
    const int* lidx = reinterpret_cast<const int*>(dyn_smem + work_bytes + p * kWideSlotBytes);
    const float* lval = reinterpret_cast<const float*>(dyn_smem + work_bytes + p * kWideSlotBytes + kWideListPad * 4);
    const int nl = sl.n;
    const int mode = j < k ? (a.q ? MODE_RESIDUAL : MODE_ONEHOT) : MODE_BONUS;
    const int xj = j < k ? sh.xs[j] : -1;
    const float* qrow = a.q && j < k ? a.q + (static_cast<long long>(b) * k + j) * a.V : nullptr;
    rc.M = sl.M;
    // weights of the kept entries: e on P for the bonus, max(0, e - S q) on P
    // at a rejection (e once the residual mass is zero), 0 off P; kept in
    // the work area for the scan
    df* wbuf = reinterpret_cast<df*>(dyn_smem);
    float qv[kWideEpt];
#pragma unroll
    for (int q = 0; q < kWideEpt; ++q) {  // the draft probabilities at this thread's entries, loaded together
        const int r = r0 + q;
        qv[q] = 0.0f;
        if (r < nl && mode != MODE_BONUS) {
            const int v = lidx[lp(r)];
            qv[q] = qrow ? __ldg(qrow + v) : (v == xj ? 1.0f : 0.0f);
        }
    }
    bool qbad = false;
    uint32_t inmask = 0;
    df local = df_make(0.0f);
#pragma unroll
    for (int q = 0; q < kWideEpt; ++q) {
        const int r = r0 + q;
        df wr = df_make(0.0f);
        if (r < nl) {
            const float l = lval[lp(r)];
            const uint32_t key = val_key<BF16>(l);
            if (key > sl.cut || (key == sl.cut && lidx[lp(r)] <= sl.cutidx)) {
                inmask |= 1u << q;
                const df e = l == -INFINITY ? df_make(0.0f) : precise_e<BF16>(l, rc, sh.exp2tab);
                if (mode == MODE_BONUS) {
                    wr = e;
                } else {
                    qbad |= !(qv[q] >= 0.0f && qv[q] <= FLT_MAX);
                    const df rr = minus_sq(e, sl.S, qv[q]);
                    wr = rr.hi + rr.lo > 0.0f ? rr : df_make(0.0f);
                }
            }
            wbuf[lp(r)] = wr;
        }
        local = df_sum(local, wr);
    }
    if (__syncthreads_or(qbad ? 1 : 0)) st |= ST_QBAD;
    if (!(st & ST_ERRMASK)) {
        df W = wide_sum_df(local, sh.red_df);
        if (mode != MODE_BONUS && !(W.hi + W.lo > 0.0f)) {  // zero residual mass: draw from p'
            st |= ST_ZERO_RESIDUAL;
            local = df_make(0.0f);
            for (int q = 0; q < kWideEpt; ++q) {
                const int r = r0 + q;
                if (r < nl) {
                    const float l = lval[lp(r)];
                    const df wr = ((inmask >> q) & 1u) && l != -INFINITY ? precise_e<BF16>(l, rc, sh.exp2tab) : df_make(0.0f);
                    wbuf[lp(r)] = wr;
                    local = df_sum(local, wr);
                }
            }
            W = wide_sum_df(local, sh.red_df);
        }
        const df target = df_mul_f(W, sh.du1);
        df tot;
        df pre = wide_excl_scan_df(local, sh.red_df, tot);
        uint32_t cand = 0xffffffffu, lastpos = 0;  // lastpos: 1 + the last positive entry
        for (int q = 0; q < kWideEpt; ++q) {
            const int r = r0 + q;
            if (r < nl) {
                const df wr = wbuf[lp(r)];
                pre = df_sum(pre, wr);
                if (wr.hi + wr.lo > 0.0f) {
                    lastpos = static_cast<uint32_t>(r + 1);
                    if (cand == 0xffffffffu && df_less(target, pre)) cand = static_cast<uint32_t>(r);
                }
            }
        }
        cand = wide_min_u32(cand, sh.red_u);
        lastpos = wide_max_u32(lastpos, sh.red_u);
        // only through rounding at the top edge: the last entry with positive weight
        const int rs = cand != 0xffffffffu ? static_cast<int>(cand) : static_cast<int>(lastpos) - 1;
        const int token = rs >= 0 ? lidx[lp(rs)] : -1;
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
