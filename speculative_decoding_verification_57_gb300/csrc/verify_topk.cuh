// verify_topk.cuh -- verification with top-k / top-p applied to the target
// distribution before the rule ("Speculative decoding." lesson, "Why the
// output is exactly p": temperature, top-k and top-p have to be applied to p
// before the rule; "Speculative Decoding: Draft, Verify, Accept", "The
// rejection-sampling correctness argument": the rule reproduces whatever p
// it is given).
//
// Readings (the pages name the filters only): top-k keeps the K (<= 64)
// largest logits, the lower index first among equal logits; top-p keeps the
// shortest prefix of those, in the same order, whose mass renormalised over
// the K reaches top_p.  p' is exp((l - M) / T) on the kept set P,
// renormalised.  The residual max(0, p' - q) and the bonus live on P, so the
// vocabulary is streamed once, to select, and no softmax over V is needed:
// the stop position's draft probabilities are gathered at the kept entries.
//
// One thread-block cluster of C = min(k + 1, 8) CTAs per sequence; CTA c
// owns positions c, c + C, ...  In each CTA a producer warp streams the
// owned rows through a ring of shared-memory stages (1-D bulk copies); the
// four consumer warps take the tiles in turn, whole, and each keeps the best
// 64 entries of its tiles in registers, as 64-bit keys (two a lane, in rank
// order).  A block of a tile is tested against the CTA's entry bound first:
// one packed bf16x2 maximum per two logits and one compare, so most blocks
// are done there.  Entries that pass collect in a per-warp buffer (a warp
// scan places a whole tile's at once); a full buffer is sorted with a
// register bitonic network and merged into the warp's 64 (half cleaner +
// bitonic merge).  At the end of a position the four warp lists
// merge in a tree and the result goes into the leader CTA's shared memory
// over DSMEM; after a cluster barrier the leader's warp 0 walks the
// positions with double-float weights.
#pragma once
#include <cfloat>
#include <cstdint>

#include <cuda_bf16.h>

#include "exp2dd.cuh"
#include "ptx.cuh"
#include "verify_cluster.cuh"

namespace specv {

constexpr int kTopKMax = 64;       // largest top_k this path takes
constexpr int kWideKMax = 4096;    // largest top_k at all: rows above kTopKMax are verify_topk_wide_kernel's

// Rows verify_topk_wide_kernel verifies (sampled, valid filters, top_k above
// this path's 64); this kernel leaves them untouched.
__device__ __forceinline__ bool wide_row(float T, int K, float top_p) {
    return T >= FLT_MIN && T <= FLT_MAX && K > kTopKMax && K <= kWideKMax && top_p > 0.0f && top_p <= 1.0f;
}
constexpr int kTopkClusterMax = 8;  // CTAs per sequence
constexpr int kTopkLocalMax = (kMaxK + 1 + kTopkClusterMax - 1) / kTopkClusterMax;  // positions per CTA
constexpr int kTopkStages = 8;     // ring stages of kTileBytes: the four warps drift apart by a few tiles
constexpr int kTopkRingBytes = kTopkStages * kTileBytes;

struct Cand {
    float v;  // logit
    int i;    // vocabulary index
};

// Rank key: a larger key comes first.  The high word orders the logit (the
// float bits made monotone), the low word is ~index, so among equal logits
// the lower index comes first.  Key 0 is the padding entry: no logit (NaN
// aside, which never enters) maps to it.
using key_t = unsigned long long;

// Float bits made monotone as unsigned (-0 ranks as +0); 0 stands for "none".
__device__ __forceinline__ uint32_t ord_f32(float v) {
    const uint32_t f = v == 0.0f ? 0u : __float_as_uint(v);
    return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}

__device__ __forceinline__ float unord_f32(uint32_t m) {
    if (m == 0) return -INFINITY;
    return __uint_as_float((m & 0x80000000u) ? (m & 0x7fffffffu) : ~m);
}

__device__ __forceinline__ key_t make_key(float v, int i) {
    return (static_cast<key_t>(ord_f32(v)) << 32) | static_cast<uint32_t>(~i);
}

__device__ __forceinline__ float key_value(key_t k) { return unord_f32(static_cast<uint32_t>(k >> 32)); }

__device__ __forceinline__ Cand key_cand(key_t k) {
    if (k == 0) return Cand{-INFINITY, 0x7fffffff};
    return Cand{key_value(k), static_cast<int>(~static_cast<uint32_t>(k))};
}

__device__ __forceinline__ key_t shfl_xor_key(key_t k, int m) {
    const uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(k), m);
    const uint32_t hi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(k >> 32), m);
    return (static_cast<key_t>(hi) << 32) | lo;
}

__device__ __forceinline__ key_t shfl_key(key_t k, int src) {
    const uint32_t lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(k), src);
    const uint32_t hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(k >> 32), src);
    return (static_cast<key_t>(hi) << 32) | lo;
}

// One compare-exchange stage across lanes (lane ^ stride): the lane keeps
// the larger key when it wants the first of the pair, else the smaller.
__device__ __forceinline__ key_t cx_lanes(key_t a, int stride, bool want_first) {
    const key_t o = shfl_xor_key(a, stride);
    return ((o > a) == want_first) ? o : a;
}

// Bitonic sort of 64 keys held two a lane (element lane and lane + 32) into
// descending order.
__device__ __forceinline__ void sort64(key_t& a0, key_t& a1, int lane) {
#pragma unroll
    for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride == 32) {
                if (a1 > a0) {
                    const key_t t = a0;
                    a0 = a1;
                    a1 = t;
                }
            } else {
                const bool lower = (lane & stride) == 0;
                a0 = cx_lanes(a0, stride, lower == ((lane & size) == 0));
                a1 = cx_lanes(a1, stride, lower == (((lane + 32) & size) == 0));
            }
        }
    }
}

// a = the 64 largest of a and b, both descending, in descending order: the
// half cleaner of a ++ reverse(b), then a bitonic merge.
__device__ __forceinline__ void merge64(key_t& a0, key_t& a1, key_t b0, key_t b1, int lane) {
    const key_t r0 = shfl_xor_key(b1, 31);  // b[63 - lane]
    const key_t r1 = shfl_xor_key(b0, 31);  // b[31 - lane]
    a0 = a0 > r0 ? a0 : r0;
    a1 = a1 > r1 ? a1 : r1;
    if (a1 > a0) {
        const key_t t = a0;
        a0 = a1;
        a1 = t;
    }
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) {
        const bool lower = (lane & stride) == 0;
        a0 = cx_lanes(a0, stride, lower);
        a1 = cx_lanes(a1, stride, lower);
    }
}

struct alignas(16) TopkSmem {
    unsigned long long full[kTopkStages];
    unsigned long long empty[kTopkStages];
    key_t wb[kConsumerWarps][kTopKMax];  // per-warp candidate buffers; the walk's scratch
    key_t ms[3][kTopKMax];               // lists on their way through the end-of-position merge
    int tstart[kTopkLocalMax + 1];       // first tile of each owned position
    int head[kTopkLocalMax];             // unaligned leading elements of each owned row
    int nbytes[kTopkLocalMax];           // bytes of the 16-byte aligned interior
    // Entry bound of each owned position (ord_f32; only rises): a logit below it
    // cannot be among the position's best 64.  It is the larger of any warp's
    // 64th-best value and the smallest of the four warps' 16th-best values
    // (b16): either way at least 64 distinct entries reach it.
    uint32_t tau[kTopkLocalMax];
    float b16[kTopkLocalMax][kConsumerWarps];
    int lbad[kTopkLocalMax];             // bit 0: a NaN in this CTA's share of an owned position
    int ltimeout;
    int bad[kMaxK + 1];                  // leader: bit 0 NaN, bit 1 the owner timed out
    int xs[kMaxK + 1];
    float2 exp2tab[128];
};

// Dynamic shared memory: the ring, then the leader's lists [k+1][64].
inline size_t topk_dyn_smem(int k) {
    return static_cast<size_t>(kTopkRingBytes) + static_cast<size_t>(k + 1) * kTopKMax * sizeof(key_t);
}

inline int topk_cluster(int k) { return k + 1 < kTopkClusterMax ? k + 1 : kTopkClusterMax; }

__device__ __forceinline__ uint32_t geu_bf16x2(uint32_t w, __nv_bfloat162 t) {
    return __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w), t);
}

// A consumer warp's selection state for one position.
struct WarpTop {
    key_t c0, c1;  // the best 64 so far, ranks lane and lane + 32 (0: none)
    key_t t63;     // rank 63: an entry must beat it to enter
    int cnt;       // entries waiting in the warp's buffer
    int nf;        // flushes so far
};

__device__ __forceinline__ void warp_flush(WarpTop& w, key_t* wb, int lane) {
    __syncwarp();
    key_t s0 = lane < w.cnt ? wb[lane] : 0;
    key_t s1 = lane + 32 < w.cnt ? wb[lane + 32] : 0;
    __syncwarp();
    sort64(s0, s1, lane);
    merge64(w.c0, w.c1, s0, s1, lane);
    w.t63 = shfl_key(w.c1, 31);
    w.cnt = 0;
    ++w.nf;
}

// Append each lane's pending elements (bit e of pend[s]; get(s, e, v, idx)
// reads that element) to the warp's buffer.  The offsets come from one
// ballot per bit of the counts; each lane then writes its elements, two at a
// time, and a full buffer is flushed into the 64.  A NaN never enters (it
// leaves a padding entry) and sets nan.
template <int NW, typename Get>
__device__ __forceinline__ void warp_take(WarpTop& w, key_t* wb, uint32_t (&pend)[NW], Get get, int lane, int& nan) {
    static_assert(NW >= 1 && NW <= 4, "at most 128 pending bits a lane");
    const unsigned full = 0xffffffffu;
    unsigned long long pl = pend[0], ph = 0;
    if constexpr (NW > 1) pl |= static_cast<unsigned long long>(pend[1]) << 32;
    if constexpr (NW > 2) ph = pend[2];
    if constexpr (NW > 3) ph |= static_cast<unsigned long long>(pend[3]) << 32;
    const uint32_t lt = lanemask_lt();
    auto next = [&]() {  // the lowest pending bit (0..127), cleared
        int g;
        if (pl) {
            g = __ffsll(pl) - 1;
            pl &= pl - 1;
        } else {
            g = 64 + __ffsll(ph) - 1;
            ph &= ph - 1;
        }
        return g;
    };
    auto key_of = [&](int g) {
        float v;
        int idx;
        get(g >> 5, g & 31, v, idx);
        if (v != v) {
            nan = 1;
            return key_t(0);
        }
        return make_key(v, idx);
    };
    for (;;) {
        const int c = __popcll(pl) + __popcll(ph);  // <= 128
        int before = 0, tot = 0;
#pragma unroll
        for (int bit = 0; bit < 8; ++bit) {
            const unsigned bb = __ballot_sync(full, (c >> bit) & 1);
            before += __popc(bb & lt) << bit;
            tot += __popc(bb) << bit;
        }
        if (tot == 0) return;
        int o = w.cnt + before;
        while ((pl | ph) != 0 && o < kTopKMax) {
            const int g0 = next();
            const bool two = (pl | ph) != 0 && o + 1 < kTopKMax;
            const int g1 = two ? next() : g0;
            const key_t k0 = key_of(g0);
            const key_t k1 = key_of(g1);
            wb[o] = k0;
            if (two) wb[o + 1] = k1;
            o += two ? 2 : 1;
        }
        __syncwarp();
        const int room = kTopKMax - w.cnt;
        if (tot < room) {
            w.cnt += tot;
            return;
        }
        w.cnt = kTopKMax;
        warp_flush(w, wb, lane);  // what did not fit is still pending
        if (tot == room) return;
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 3) verify_topk_kernel(const VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ __align__(16) TopkSmem sh;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int kEpc = 16 / esz;                       // elements per chunk
    const unsigned full = 0xffffffffu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool producer = warp == kConsumerWarps;
    const int C = static_cast<int>(cluster_size());
    const int crank = static_cast<int>(cluster_rank());
    const int b = static_cast<int>(blockIdx.x) / C;
    const int k = a.k;
    const long long V = a.V;
    const int n = static_cast<int>(V);
    const int P = (k - crank) / C + 1;  // owned positions crank + C p, p < P
    const unsigned char* lg = reinterpret_cast<const unsigned char*>(a.logits);
    unsigned char* ring = dyn_smem;
    key_t* lists = reinterpret_cast<key_t*>(dyn_smem + kTopkRingBytes);  // [k+1][64]; the leader's are read

    const float T = a.temp ? __ldg(a.temp + b) : 0.0f;
    const bool greedy = T == 0.0f;
    const bool t_ok = greedy || (T >= FLT_MIN && T <= FLT_MAX);
    const int K = a.top_k ? __ldg(a.top_k + b) : kTopKMax;
    const float top_p = a.top_p ? __ldg(a.top_p + b) : 1.0f;
    if (wide_row(T, K, top_p)) return;  // the whole cluster leaves: the wide kernel has the row
    const bool f_ok = greedy || (K >= 1 && K <= kWideKMax && top_p > 0.0f && top_p <= 1.0f);
    const bool run = t_ok && f_ok;

    // ---------------------------------------------------------------- setup
    if (tid < 128) sh.exp2tab[tid] = g_exp2_table[tid];
    if (tid <= k) sh.xs[tid] = tid < k ? __ldg(a.x + static_cast<long long>(b) * k + tid) : -1;
    if (tid < kTopkLocalMax * kConsumerWarps) sh.b16[tid / kConsumerWarps][tid % kConsumerWarps] = -INFINITY;
    if (tid < kTopkLocalMax) {
        sh.lbad[tid] = 0;
        sh.tau[tid] = 0u;
    }
    auto issue = [&](int tt) {
        int p = 0;
        while (sh.tstart[p + 1] <= tt) ++p;
        const int i = crank + C * p;
        const int off = (tt - sh.tstart[p]) * kTileBytes;
        const int bytes = min(kTileBytes, sh.nbytes[p] - off);
        const long long e0 = (static_cast<long long>(b) * (k + 1) + i) * V + sh.head[p];
        const int slot = tt % kTopkStages;
        const uint32_t bar = smem_u32(&sh.full[slot]);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(bytes));
        bulk_g2s(smem_u32(ring + slot * kTileBytes), lg + e0 * esz + off, static_cast<uint32_t>(bytes), bar);
    };
    int issued = 0;
    if (producer && lane == 0) {
        for (int s = 0; s < kTopkStages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), 1);  // the one warp that took the tile
        }
        sh.ltimeout = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        int acc = 0;
        for (int p = 0; p < P; ++p) {
            const int i = crank + C * p;
            const uintptr_t addr =
                reinterpret_cast<uintptr_t>(lg + (static_cast<long long>(b) * (k + 1) + i) * V * esz);
            int h = static_cast<int>(((16 - (addr & 15)) & 15) / esz);
            if (h > n) h = n;
            const int nb = ((n - h) * esz) & ~15;
            sh.head[p] = h;
            sh.nbytes[p] = nb;
            sh.tstart[p] = acc;
            if (run) acc += (nb + kTileBytes - 1) / kTileBytes;
        }
        sh.tstart[P] = acc;
        for (; issued < min(kTopkStages, acc); ++issued) issue(issued);
    }
    __syncthreads();
    cluster_arrive();  // the matching wait comes before the first store into the leader
    const int total = sh.tstart[P];

    // ---------------------------------------------------------------- stream
    if (producer) {
        if (lane == 0) {
            for (; issued < total; ++issued) {
                const int slot = issued % kTopkStages;
                if (sh.ltimeout || !mbar_wait_bounded(smem_u32(&sh.empty[slot]), ((issued / kTopkStages) & 1) ^ 1,
                                                      kWaitPolls)) {
                    atomicOr(&sh.ltimeout, 1);
                    break;
                }
                issue(issued);
            }
            if (sh.ltimeout) {
                // no copy may still be writing this CTA's shared memory when it exits
                for (int s = 0; s < kTopkStages && s < issued; ++s) {
                    const int last = s + kTopkStages * ((issued - 1 - s) / kTopkStages);
                    mbar_wait_bounded(smem_u32(&sh.full[s]), (last / kTopkStages) & 1, kWaitPolls);
                }
            }
        }
        __syncwarp();
        cluster_wait();
    } else {
        key_t* wb = sh.wb[warp];
        for (int p = 0; p < P; ++p) {
            const int i = crank + C * p;
            WarpTop w;
            w.c0 = w.c1 = w.t63 = 0;
            w.cnt = 0;
            w.nf = 0;
            int nan = 0;
            const long long row_e0 = (static_cast<long long>(b) * (k + 1) + i) * V;
            const int h = sh.head[p];
            const int interior = sh.nbytes[p] / esz;
            const int t0 = sh.tstart[p];
            const int ntiles = sh.tstart[p + 1] - t0;
            // unaligned head and tail: warp 0 reads them with plain loads, a lane an element
            auto scalar_part = [&](int lo, int hi) {
                uint32_t pe[1] = {lane < hi - lo ? 1u : 0u};
                warp_take(w, wb, pe, [&](int, int, float& v, int& idx) {
                    idx = lo + lane;
                    v = load_logit(a.logits, row_e0 + idx, BF16);
                }, lane, nan);
            };
            if (run && warp == 0 && h > 0) scalar_part(0, h);
            // publish the warp's bounds after its 64 changed
            auto publish = [&]() {
                const key_t r15 = shfl_key(w.c0, 15);
                if (lane == 0) {
                    if (w.t63) atomicMax(&sh.tau[p], static_cast<uint32_t>(w.t63 >> 32));
                    if (r15) {
                        sh.b16[p][warp] = fmaxf(sh.b16[p][warp], key_value(r15));
                        const float m = fminf(fminf(sh.b16[p][0], sh.b16[p][1]), fminf(sh.b16[p][2], sh.b16[p][3]));
                        if (m > -INFINITY) atomicMax(&sh.tau[p], ord_f32(m));
                    }
                }
                __syncwarp();
            };
            // Warp w takes tiles w, w + 4, ... of the position whole: lane l reads chunks
            // l + 32 j (j < 16) in four blocks of four.  The first pass runs in every warp,
            // with or without a tile, for the barrier that shares the first bounds.
            for (int lt = warp; ntiles > 0; lt += kConsumerWarps) {
                const bool first = lt == warp;
                if (!first && lt >= ntiles) break;
                const bool has = lt < ntiles;
                const int it = t0 + lt;
                const int slot = it % kTopkStages;
                const bool ok = has && __all_sync(full, !sh.ltimeout &&
                                                            mbar_wait_bounded(smem_u32(&sh.full[slot]),
                                                                              (it / kTopkStages) & 1, kWaitPolls));
                if (has && !ok && lane == 0) atomicOr(&sh.ltimeout, 1);
                const int nch = ok ? min(kTileBytes, sh.nbytes[p] - lt * kTileBytes) >> 4 : 0;
                const uint32_t tile = smem_u32(ring + slot * kTileBytes);
                const int tile_e = h + lt * (kTileBytes / esz);  // row index of the tile's first element
                float tau_first = -INFINITY;
                if (first) {
                    // bounds from the lanes' largest two values of the first block (a NaN
                    // counts as -inf here)
                    float mx = -INFINITY, mx2 = -INFINITY;
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int ch = lane + 32 * r;
                        if (ch < nch) {
                            const uint4 dd = ld_shared_v4(tile + ch * 16);
                            const uint32_t wd[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
                            for (int q = 0; q < kEpc; ++q) {
                                float l;
                                if constexpr (BF16)
                                    l = (q & 1) ? bf16_hi(wd[q >> 1]) : bf16_lo(wd[q >> 1]);
                                else
                                    l = __uint_as_float(wd[q & 3]);
                                l = l == l ? l : -INFINITY;
                                mx2 = fmaxf(mx2, fminf(mx, l));
                                mx = fmaxf(mx, l);
                            }
                        }
                    }
                    // 64 entries reach the smallest second-largest of the 32 lanes
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) mx2 = fminf(mx2, __shfl_xor_sync(full, mx2, off));
                    // 16 entries reach the 16th largest lane maximum: sort the maxima, descending
#pragma unroll
                    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
                        for (int stride = size >> 1; stride > 0; stride >>= 1) {
                            const float o = __shfl_xor_sync(full, mx, stride);
                            const bool first_of_pair = ((lane & stride) == 0) == ((lane & size) == 0);
                            mx = first_of_pair ? fmaxf(mx, o) : fminf(mx, o);
                        }
                    }
                    const float m16 = __shfl_sync(full, mx, 15);
                    if (lane == 0) {
                        sh.b16[p][warp] = m16;
                        if (mx2 > -INFINITY) atomicMax(&sh.tau[p], ord_f32(mx2));
                    }
                    consumers_sync();
                    tau_first = fmaxf(mx2, fminf(fminf(sh.b16[p][0], sh.b16[p][1]), fminf(sh.b16[p][2], sh.b16[p][3])));
                    if (lane == 0 && tau_first > -INFINITY) atomicMax(&sh.tau[p], ord_f32(tau_first));
                }
                if (!ok) continue;  // no tile here, or the stream gave up: the barrier sequence is kept
                const float tau = fmaxf(tau_first, unord_f32(sh.tau[p]));
                // elements that may enter (NaN included: it is caught and flagged in warp_take)
                uint32_t pend[4];
#pragma unroll
                for (int sb = 0; sb < 4; ++sb) {
                    uint4 d[4];
#pragma unroll
                    for (int r = 0; r < 4; ++r) {
                        const int ch = lane + 32 * (sb * 4 + r);
                        d[r] = ch < nch ? ld_shared_v4(tile + ch * 16) : make_uint4(0u, 0u, 0u, 0u);
                    }
                    uint32_t pm = 0;
                    if constexpr (BF16) {
                        // bit r*4+q: the low element of word q of chunk r; bit 16+r*4+q: the high one
                        const __nv_bfloat162 t2 = __float2bfloat162_rn(tau);
                        uint32_t cm[4];  // each chunk's maximum (NaN kept)
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            cm[r] = lane + 32 * (sb * 4 + r) < nch
                                        ? max_nan_bf16x2(max_nan_bf16x2(d[r].x, d[r].y), max_nan_bf16x2(d[r].z, d[r].w))
                                        : 0xff80ff80u;  // (-inf, -inf)
                        const uint32_t mw = max_nan_bf16x2(max_nan_bf16x2(cm[0], cm[1]), max_nan_bf16x2(cm[2], cm[3]));
                        if (geu_bf16x2(mw, t2)) {
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                if (lane + 32 * (sb * 4 + r) < nch && geu_bf16x2(cm[r], t2)) {
                                    const uint32_t wd[4] = {d[r].x, d[r].y, d[r].z, d[r].w};
#pragma unroll
                                    for (int q = 0; q < 4; ++q)
                                        pm |= (geu_bf16x2(wd[q], t2) & 0x00010001u) << (r * 4 + q);
                                }
                            }
                        }
                    } else {
                        // bit r*4+q: element q of chunk r
#pragma unroll
                        for (int r = 0; r < 4; ++r) {
                            if (lane + 32 * (sb * 4 + r) < nch) {
                                const uint32_t wd[4] = {d[r].x, d[r].y, d[r].z, d[r].w};
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    pm |= (__uint_as_float(wd[q]) < tau ? 0u : 1u) << (r * 4 + q);
                            }
                        }
                    }
                    pend[sb] = pm;
                }
                if (__any_sync(full, (pend[0] | pend[1] | pend[2] | pend[3]) != 0)) {
                    const int nf0 = w.nf;
                    warp_take(w, wb, pend, [&](int sb, int e, float& v, int& idx) {
                        if constexpr (BF16) {
                            const int r = (e & 15) >> 2, q = 2 * (e & 3) + (e >> 4);
                            const int ch = lane + 32 * (sb * 4 + r);
                            v = __uint_as_float(static_cast<uint32_t>(ld_shared_u16(tile + ch * 16 + q * 2)) << 16);
                            idx = tile_e + ch * kEpc + q;
                        } else {
                            const int r = e >> 2, q = e & 3, ch = lane + 32 * (sb * 4 + r);
                            v = ld_shared_f32(tile + ch * 16 + q * 4);
                            idx = tile_e + ch * kEpc + q;
                        }
                    }, lane, nan);
                    if (w.nf != nf0) publish();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.empty[slot]));
            }
            if (run && warp == 0 && h + interior < n) scalar_part(h + interior, n);
            if (w.cnt > 0) warp_flush(w, wb, lane);
            if (__any_sync(full, nan) && lane == 0) atomicOr(&sh.lbad[p], 1);
            // the four warp lists merge in a tree: (1 -> 0, 3 -> 2), then 2 -> 0
            if (warp == 1 || warp == 3) {
                sh.ms[warp >> 1][lane] = w.c0;
                sh.ms[warp >> 1][lane + 32] = w.c1;
            }
            consumers_sync();
            if (warp == 0 || warp == 2) merge64(w.c0, w.c1, sh.ms[warp >> 1][lane], sh.ms[warp >> 1][lane + 32], lane);
            if (warp == 2) {
                sh.ms[2][lane] = w.c0;
                sh.ms[2][lane + 32] = w.c1;
            }
            consumers_sync();
            if (warp == 0) {
                merge64(w.c0, w.c1, sh.ms[2][lane], sh.ms[2][lane + 32], lane);
                if (p == 0) cluster_wait();  // the leader has started: its shared memory may be written
                const uint32_t dst = map_rank(smem_u32(lists + static_cast<size_t>(i) * kTopKMax), 0);
                st_cluster_v2(dst + lane * 8, static_cast<uint32_t>(w.c0), static_cast<uint32_t>(w.c0 >> 32));
                st_cluster_v2(dst + (lane + 32) * 8, static_cast<uint32_t>(w.c1), static_cast<uint32_t>(w.c1 >> 32));
                if (lane == 0)
                    st_cluster_u32(map_rank(smem_u32(&sh.bad[i]), 0),
                                   static_cast<uint32_t>(sh.lbad[p] | (sh.ltimeout ? 2 : 0)));
            }
        }
        if (warp != 0) cluster_wait();
    }
    // the walk's per-position inputs (lane i: position i), loaded while the cluster barrier completes
    float pu0 = 0.0f, pu1 = 0.0f, pqx = 0.0f;
    if (crank == 0 && warp == 0 && lane <= k) {
        const long long ub = (static_cast<long long>(b) * (k + 1) + lane) * 2;
        pu0 = __ldg(a.u + ub);
        pu1 = __ldg(a.u + ub + 1);
        const int x = lane < k ? sh.xs[lane] : -1;
        if (x >= 0 && x < V) pqx = a.q ? __ldg(a.q + (static_cast<long long>(b) * k + lane) * V + x) : 1.0f;
    }
    cluster_sync();  // every list and flag is in the leader
    if (crank != 0 || warp != 0) return;

    // ---------------------------------------------------------------- walk
    const bool timed_out = __any_sync(full, lane <= k && (sh.bad[lane] & 2));
    int st = !t_ok ? ST_TEMP : (!f_ok ? ST_FILTER : (timed_out ? ST_TIMEOUT : 0));
    int j = 0, token = -1;
    if (!st && greedy) {
        for (int i = 0; i <= k; ++i) {
            const int A = key_cand(lists[static_cast<size_t>(i) * kTopKMax]).i;
            const int x = i < k ? sh.xs[i] : -1;
            int pst = (sh.bad[i] & 1) ? ST_NONFINITE : 0;  // a NaN: the argmax is undefined
            if (i < k && (x < 0 || x >= V)) pst |= ST_TOKEN;
            if (pst) {
                st |= pst;
                break;
            }
            if (i == k || x != A) {
                j = i;
                token = A;
                break;
            }
        }
    } else if (!st) {
        RowConst rc;
        rc.s1 = 0.0f;
        rc.thr = 0.0f;
        const df c2 = log2e_over(T);
        rc.ch = c2.hi;
        rc.cl = c2.lo;
        // lane r holds ranks r and r + 32 of the current position
        Cand c0 = key_cand(0), c1 = key_cand(0);
        df e0 = df_make(0.0f), e1 = df_make(0.0f), SP = df_make(0.0f);
        int np = 0;
        for (int i = 0; i <= k; ++i) {
            const key_t* m = lists + static_cast<size_t>(i) * kTopKMax;
            c0 = key_cand(m[lane]);
            c1 = key_cand(m[lane + 32]);
            rc.M = key_value(m[0]);
            // this position's errors, in the walk's order of checks (+inf: the maximum is infinite)
            int pst = ((sh.bad[i] & 1) || !(rc.M > -INFINITY && rc.M < INFINITY)) ? ST_NONFINITE : 0;
            const int x = i < k ? sh.xs[i] : -1;
            float u0 = 0.0f, qx = 0.0f;
            if (i < k) {
                u0 = __shfl_sync(full, pu0, i);
                qx = __shfl_sync(full, pqx, i);
                if (x < 0 || x >= V) pst |= ST_TOKEN;
                if (!(u0 >= 0.0f && u0 < 1.0f)) pst |= ST_UNIFORM;
                if (x >= 0 && x < V && !(qx >= 0.0f && qx <= FLT_MAX)) pst |= ST_QBAD;
            }
            if (pst) {
                st |= pst;
                break;
            }
            const bool k0 = lane < K && c0.v != -INFINITY, k1 = lane + 32 < K && c1.v != -INFINITY;
            e0 = k0 ? precise_e<BF16>(c0.v, rc, sh.exp2tab) : df_make(0.0f);
            e1 = k1 ? precise_e<BF16>(c1.v, rc, sh.exp2tab) : df_make(0.0f);
            __syncwarp();
            // cumulative mass in rank order, and the top-p cut
            const df s0 = df_warp_incl_scan(e0, lane);
            const df t0 = df_shfl(s0, 31);
            const df s1 = df_sum(t0, df_warp_incl_scan(e1, lane));
            const df SK = df_shfl(s1, 31);
            np = K;
            if (top_p < 1.0f) {
                const df target = df_mul_f(SK, top_p);
                const unsigned h0 = __ballot_sync(full, lane < K && !df_less(s0, target));
                const unsigned h1 = __ballot_sync(full, lane + 32 < K && !df_less(s1, target));
                np = h0 ? __ffs(h0) : (h1 ? 32 + __ffs(h1) : K);
            }
            SP = np <= 32 ? df_shfl(s0, np - 1) : df_shfl(s1, np - 33);
            if (i == k) {
                j = k;
                break;
            }
            // p'(x): x among the kept ranks
            const bool h0 = lane < np && c0.i == x, h1 = lane + 32 < np && c1.i == x;
            const unsigned b0 = __ballot_sync(full, h0), b1 = __ballot_sync(full, h1);
            float px = 0.0f;
            if (b0 || b1) {
                const df ex = b0 ? df_shfl(e0, __ffs(b0) - 1) : df_shfl(e1, __ffs(b1) - 1);
                px = df_val(ex) / df_val(SP);
            }
            const float rho = fminf(1.0f, px / fmaxf(qx, 1e-12f));
            if (!(u0 < rho)) {
                j = i;
                break;
            }
        }
        float u1 = 0.0f;
        if (!st) {
            u1 = __shfl_sync(full, pu1, j);
            if (!(u1 >= 0.0f && u1 < 1.0f)) st |= ST_UNIFORM;
        }
        if (!st) {
            // weights on the kept set: max(0, e - S_P q) at a rejection, e for the bonus
            // kept: ranks below np that hold an entry (with V < 64 the list ends in padding)
            const bool v0 = lane < np && c0.i != 0x7fffffff, v1 = lane + 32 < np && c1.i != 0x7fffffff;
            df w0 = v0 ? e0 : df_make(0.0f), w1 = v1 ? e1 : df_make(0.0f);
            if (j < k) {
                const int xj = sh.xs[j];
                const float* qrow = a.q ? a.q + (static_cast<long long>(b) * k + j) * V : nullptr;
                const float q0 = v0 ? (qrow ? __ldg(qrow + c0.i) : (c0.i == xj ? 1.0f : 0.0f)) : 0.0f;
                const float q1 = v1 ? (qrow ? __ldg(qrow + c1.i) : (c1.i == xj ? 1.0f : 0.0f)) : 0.0f;
                const bool qb = !(q0 >= 0.0f && q0 <= FLT_MAX) || !(q1 >= 0.0f && q1 <= FLT_MAX);
                if (__any_sync(full, qb)) st |= ST_QBAD;
                const df r0 = minus_sq(e0, SP, q0), r1 = minus_sq(e1, SP, q1);
                w0 = (v0 && r0.hi + r0.lo > 0.0f) ? r0 : df_make(0.0f);
                w1 = (v1 && r1.hi + r1.lo > 0.0f) ? r1 : df_make(0.0f);
                const df W = df_shfl(df_warp_total(df_sum(w0, w1)), 0);
                if (!(W.hi + W.lo > 0.0f)) {  // zero residual mass: sample p'
                    st |= ST_ZERO_RESIDUAL;
                    w0 = v0 ? e0 : df_make(0.0f);
                    w1 = v1 ? e1 : df_make(0.0f);
                }
            }
            if (!(st & ST_ERRMASK)) {
                // the kept entries in vocabulary order: sort (index, rank) keys, the lowest index first
                key_t o0 = v0 ? (static_cast<key_t>(~static_cast<uint32_t>(c0.i)) << 32) | static_cast<uint32_t>(lane) : 0;
                key_t o1 = v1 ? (static_cast<key_t>(~static_cast<uint32_t>(c1.i)) << 32) | static_cast<uint32_t>(lane + 32)
                              : 0;
                sort64(o0, o1, lane);
                // the weight of the entry at each sorted place
                auto weight_at = [&](key_t o) {
                    const int r = static_cast<int>(o & 63u);
                    const float hA = __shfl_sync(full, w0.hi, r & 31), lA = __shfl_sync(full, w0.lo, r & 31);
                    const float hB = __shfl_sync(full, w1.hi, r & 31), lB = __shfl_sync(full, w1.lo, r & 31);
                    return o == 0 ? df_make(0.0f) : (r < 32 ? df{hA, lA} : df{hB, lB});
                };
                const df a0 = weight_at(o0), a1 = weight_at(o1);
                const df p0 = df_warp_incl_scan(a0, lane);
                const df p1 = df_sum(df_shfl(p0, 31), df_warp_incl_scan(a1, lane));
                const df W = df_shfl(p1, 31);
                const df target = df_mul_f(W, u1);
                const bool pos0 = a0.hi + a0.lo > 0.0f, pos1 = a1.hi + a1.lo > 0.0f;
                const unsigned g0 = __ballot_sync(full, pos0 && df_less(target, p0));
                const unsigned g1 = __ballot_sync(full, pos1 && df_less(target, p1));
                int slot = -1;
                if (g0)
                    slot = __ffs(g0) - 1;
                else if (g1)
                    slot = 32 + __ffs(g1) - 1;
                else {  // only through rounding at the top edge: the last positive entry
                    const unsigned q0b = __ballot_sync(full, pos0), q1b = __ballot_sync(full, pos1);
                    slot = q1b ? 32 + 31 - __clz(q1b) : (q0b ? 31 - __clz(q0b) : 0);
                }
                const key_t kA = shfl_key(o0, slot & 31), kB = shfl_key(o1, slot & 31);
                token = static_cast<int>(~static_cast<uint32_t>((slot < 32 ? kA : kB) >> 32));
            }
        }
    }
    const bool bad = (st & ST_ERRMASK) != 0;
    if (lane <= k) {
        int tok = -1;
        if (!bad) tok = lane < j ? sh.xs[lane] : (lane == j ? token : -1);
        a.out_tokens[static_cast<long long>(b) * (k + 1) + lane] = tok;
    }
    if (lane == 0) {
        a.num_accepted[b] = bad ? 0 : j;
        if (a.row_status) a.row_status[b] = st;
    }
}

}  // namespace specv
