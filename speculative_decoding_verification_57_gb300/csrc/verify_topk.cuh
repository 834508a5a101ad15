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
// owned rows through a ring of shared-memory stages (1-D bulk copies); each
// of the four consumer warps keeps the best 64 entries of its share in
// registers, as 64-bit keys (two a lane, in rank order).  An entry is
// tested against a threshold first: a packed bf16x2 (or fp32) compare with
// the largest 64th-best value any warp of the CTA has published, so after
// the first tiles almost every tile passes with one compare per two logits.
// Entries that pass collect in a per-warp buffer; a full buffer is sorted
// with a register bitonic network and merged into the warp's 64 (half
// cleaner + bitonic merge).  At the end of a position the four warp lists
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
constexpr int kTopkClusterMax = 8;  // CTAs per sequence
constexpr int kTopkLocalMax = (kMaxK + 1 + kTopkClusterMax - 1) / kTopkClusterMax;  // positions per CTA

struct Cand {
    float v;  // logit
    int i;    // vocabulary index
};

// Rank key: a larger key comes first.  The high word orders the logit (the
// float bits made monotone), the low word is ~index, so among equal logits
// the lower index comes first.  Key 0 is the padding entry: no logit (NaN
// aside, which never enters) maps to it.
using key_t = unsigned long long;

__device__ __forceinline__ key_t make_key(float v, int i) {
    const uint32_t f = v == 0.0f ? 0u : __float_as_uint(v);  // -0 ranks as +0
    const uint32_t m = (f & 0x80000000u) ? ~f : (f | 0x80000000u);
    return (static_cast<key_t>(m) << 32) | static_cast<uint32_t>(~i);
}

__device__ __forceinline__ float key_value(key_t k) {
    if (k == 0) return -INFINITY;
    const uint32_t m = static_cast<uint32_t>(k >> 32);
    return __uint_as_float((m & 0x80000000u) ? (m & 0x7fffffffu) : ~m);
}

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
    unsigned long long full[kStages];
    unsigned long long empty[kStages];
    key_t wb[kConsumerWarps][kTopKMax];  // per-warp candidate buffers; the walk's scratch
    key_t ms[3][kTopKMax];               // lists on their way through the end-of-position merge
    int tstart[kTopkLocalMax + 1];       // first tile of each owned position
    int head[kTopkLocalMax];             // unaligned leading elements of each owned row
    int nbytes[kTopkLocalMax];           // bytes of the 16-byte aligned interior
    float wthr[kTopkLocalMax][kConsumerWarps];  // published 64th-best values (inclusive bounds)
    int lbad[kTopkLocalMax];             // bit 0: a NaN in this CTA's share of an owned position
    int ltimeout;
    int bad[kMaxK + 1];                  // leader: bit 0 NaN, bit 1 the owner timed out
    int xs[kMaxK + 1];
    float2 exp2tab[128];
};

// Dynamic shared memory: the ring, then the leader's lists [k+1][64].
inline size_t topk_dyn_smem(int k) {
    return static_cast<size_t>(kRingBytes) + static_cast<size_t>(k + 1) * kTopKMax * sizeof(key_t);
}

inline int topk_cluster(int k) { return k + 1 < kTopkClusterMax ? k + 1 : kTopkClusterMax; }

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t geu_bf16x2(uint32_t w, __nv_bfloat162 t) {
    return __hgeu2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w), t);
}

// A consumer warp's selection state for one position.
struct WarpTop {
    key_t c0, c1;  // the best 64 so far, ranks lane and lane + 32 (0: none)
    key_t t63;     // rank 63: an entry must beat it to enter
    int cnt;       // entries waiting in the warp's buffer
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
}

// Offer each lane's pending elements (bit e of pend; get(e, v, idx) reads
// element e) to the warp's 64, one element a lane per round.  A NaN never
// enters; it sets nan.
template <typename Get>
__device__ __forceinline__ void warp_take(WarpTop& w, key_t* wb, uint32_t pend, Get get, int lane, int& nan) {
    const unsigned full = 0xffffffffu;
    for (;;) {
        const bool has = pend != 0;
        if (!__any_sync(full, has)) break;
        key_t key = 0;
        bool take = false;
        if (has) {
            const int e = __ffs(pend) - 1;
            pend &= pend - 1;
            float v;
            int idx;
            get(e, v, idx);
            if (v != v) {
                nan = 1;
            } else {
                key = make_key(v, idx);
                take = key > w.t63;
            }
        }
        __syncwarp();
        unsigned bal = __ballot_sync(full, take);
        if (w.cnt + __popc(bal) > kTopKMax) {
            warp_flush(w, wb, lane);
            take = take && key > w.t63;
            bal = __ballot_sync(full, take);
        }
        if (take) wb[w.cnt + __popc(bal & lanemask_lt())] = key;
        w.cnt += __popc(bal);
        __syncwarp();
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 3) verify_topk_kernel(const VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ __align__(16) TopkSmem sh;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int kPer = kTileBytes / 16 / kConsumers;  // 16-byte chunks per consumer thread and tile
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
    key_t* lists = reinterpret_cast<key_t*>(dyn_smem + kRingBytes);  // [k+1][64]; the leader's are read

    const float T = a.temp ? __ldg(a.temp + b) : 0.0f;
    const bool greedy = T == 0.0f;
    const bool t_ok = greedy || (T >= FLT_MIN && T <= FLT_MAX);
    const int K = a.top_k ? __ldg(a.top_k + b) : kTopKMax;
    const float top_p = a.top_p ? __ldg(a.top_p + b) : 1.0f;
    const bool f_ok = greedy || (K >= 1 && K <= kTopKMax && top_p > 0.0f && top_p <= 1.0f);
    const bool run = t_ok && f_ok;

    // ---------------------------------------------------------------- setup
    if (tid < 128) sh.exp2tab[tid] = g_exp2_table[tid];
    if (tid <= k) sh.xs[tid] = tid < k ? __ldg(a.x + static_cast<long long>(b) * k + tid) : -1;
    if (tid < kTopkLocalMax * kConsumerWarps) sh.wthr[tid / kConsumerWarps][tid % kConsumerWarps] = -INFINITY;
    if (tid < kTopkLocalMax) sh.lbad[tid] = 0;
    auto issue = [&](int tt) {
        int p = 0;
        while (sh.tstart[p + 1] <= tt) ++p;
        const int i = crank + C * p;
        const int off = (tt - sh.tstart[p]) * kTileBytes;
        const int bytes = min(kTileBytes, sh.nbytes[p] - off);
        const long long e0 = (static_cast<long long>(b) * (k + 1) + i) * V + sh.head[p];
        const int slot = tt % kStages;
        const uint32_t bar = smem_u32(&sh.full[slot]);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(bytes));
        bulk_g2s(smem_u32(ring + slot * kTileBytes), lg + e0 * esz + off, static_cast<uint32_t>(bytes), bar);
    };
    int issued = 0;
    if (producer && lane == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), kConsumerWarps);
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
        for (; issued < min(kStages, acc); ++issued) issue(issued);
    }
    __syncthreads();
    cluster_arrive();  // the matching wait comes before the first store into the leader
    const int total = sh.tstart[P];

    // ---------------------------------------------------------------- stream
    if (producer) {
        if (lane == 0) {
            for (; issued < total; ++issued) {
                const int slot = issued % kStages;
                if (sh.ltimeout || !mbar_wait_bounded(smem_u32(&sh.empty[slot]), ((issued / kStages) & 1) ^ 1,
                                                      kWaitPolls)) {
                    atomicOr(&sh.ltimeout, 1);
                    break;
                }
                issue(issued);
            }
            if (sh.ltimeout) {
                // no copy may still be writing this CTA's shared memory when it exits
                for (int s = 0; s < kStages && s < issued; ++s) {
                    const int last = s + kStages * ((issued - 1 - s) / kStages);
                    mbar_wait_bounded(smem_u32(&sh.full[s]), (last / kStages) & 1, kWaitPolls);
                }
            }
        }
        __syncwarp();
        cluster_wait();
    } else {
        int it = 0;
        key_t* wb = sh.wb[warp];
        for (int p = 0; p < P; ++p) {
            const int i = crank + C * p;
            WarpTop w;
            w.c0 = w.c1 = w.t63 = 0;
            w.cnt = 0;
            int nan = 0;
            bool fresh = true;
            const long long row_e0 = (static_cast<long long>(b) * (k + 1) + i) * V;
            const int h = sh.head[p];
            const int interior = sh.nbytes[p] / esz;
            const int ntiles = sh.tstart[p + 1] - sh.tstart[p];
            // unaligned head and tail: warp 0 reads them with plain loads, a lane an element
            auto scalar_part = [&](int lo, int hi) {
                warp_take(w, wb, lane < hi - lo ? 1u : 0u, [&](int, float& v, int& idx) {
                    idx = lo + lane;
                    v = load_logit(a.logits, row_e0 + idx, BF16);
                }, lane, nan);
            };
            if (run && warp == 0 && h > 0) scalar_part(0, h);
            for (int lt = 0; lt < ntiles; ++lt, ++it) {
                const int slot = it % kStages;
                const bool ok = __all_sync(full, !sh.ltimeout && mbar_wait_bounded(smem_u32(&sh.full[slot]),
                                                                                   (it / kStages) & 1, kWaitPolls));
                if (!ok) {
                    if (lane == 0) atomicOr(&sh.ltimeout, 1);
                    continue;  // the rest of the stream is skipped, the barrier sequence kept
                }
                const int bytes = min(kTileBytes, sh.nbytes[p] - lt * kTileBytes);
                const int nch = bytes >> 4;
                const uint32_t tile = smem_u32(ring + slot * kTileBytes);
                const int tile_e = h + lt * (kTileBytes / esz);  // row index of the tile's first element
                uint4 d[kPer];
#pragma unroll
                for (int r = 0; r < kPer; ++r) {
                    const int ch = tid + r * kConsumers;
                    d[r] = ch < nch ? ld_shared_v4(tile + ch * 16) : make_uint4(0u, 0u, 0u, 0u);
                }
                // the entry bound: the best 64th value any warp has published
                float tau = fmaxf(key_value(w.t63), fmaxf(fmaxf(sh.wthr[p][0], sh.wthr[p][1]),
                                                          fmaxf(sh.wthr[p][2], sh.wthr[p][3])));
                if (fresh) {
                    // a position's first tile: at least 64 of the warp's elements reach the
                    // smallest second-largest of the 32 lanes (a NaN counts as -inf here)
                    float mx = -INFINITY, mx2 = -INFINITY;
#pragma unroll
                    for (int r = 0; r < kPer; ++r) {
                        if (tid + r * kConsumers < nch) {
                            const uint32_t wd[4] = {d[r].x, d[r].y, d[r].z, d[r].w};
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
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) mx2 = fminf(mx2, __shfl_xor_sync(full, mx2, off));
                    tau = fmaxf(tau, mx2);
                    if (lane == 0) sh.wthr[p][warp] = fmaxf(sh.wthr[p][warp], mx2);
                    fresh = false;
                }
                // elements that may enter (NaN included: it is caught and flagged in warp_take)
                uint32_t pend = 0;
                if constexpr (BF16) {
                    const __nv_bfloat162 t2 = __float2bfloat162_rn(tau);
                    uint32_t m[kPer][4];
                    uint32_t any = 0;
#pragma unroll
                    for (int r = 0; r < kPer; ++r) {
                        const bool v = tid + r * kConsumers < nch;
                        m[r][0] = v ? geu_bf16x2(d[r].x, t2) : 0u;
                        m[r][1] = v ? geu_bf16x2(d[r].y, t2) : 0u;
                        m[r][2] = v ? geu_bf16x2(d[r].z, t2) : 0u;
                        m[r][3] = v ? geu_bf16x2(d[r].w, t2) : 0u;
                        any |= m[r][0] | m[r][1] | m[r][2] | m[r][3];
                    }
                    if (any) {
#pragma unroll
                        for (int r = 0; r < kPer; ++r)
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                pend |= ((m[r][q] & 1u) | ((m[r][q] >> 15) & 2u)) << (r * 8 + q * 2);
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < kPer; ++r) {
                        if (tid + r * kConsumers < nch) {
                            const uint32_t wd[4] = {d[r].x, d[r].y, d[r].z, d[r].w};
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                pend |= (__uint_as_float(wd[q]) < tau ? 0u : 1u) << (r * 4 + q);
                        }
                    }
                }
                if (__any_sync(full, pend != 0)) {
                    warp_take(w, wb, pend, [&](int e, float& v, int& idx) {
                        const int r = e / kEpc, q = e % kEpc, ch = tid + r * kConsumers;
                        v = BF16 ? __uint_as_float(static_cast<uint32_t>(ld_shared_u16(tile + ch * 16 + q * 2)) << 16)
                                 : ld_shared_f32(tile + ch * 16 + q * 4);
                        idx = tile_e + ch * kEpc + q;
                    }, lane, nan);
                    if (lane == 0 && w.t63 != 0) sh.wthr[p][warp] = fmaxf(sh.wthr[p][warp], key_value(w.t63));
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
                u0 = __ldg(a.u + (static_cast<long long>(b) * (k + 1) + i) * 2);
                if (x < 0 || x >= V) pst |= ST_TOKEN;
                if (!(u0 >= 0.0f && u0 < 1.0f)) pst |= ST_UNIFORM;
                if (x >= 0 && x < V) {
                    qx = a.q ? __ldg(a.q + (static_cast<long long>(b) * k + i) * V + x) : 1.0f;
                    if (!(qx >= 0.0f && qx <= FLT_MAX)) pst |= ST_QBAD;
                }
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
            u1 = __ldg(a.u + (static_cast<long long>(b) * (k + 1) + j) * 2 + 1);
            if (!(u1 >= 0.0f && u1 < 1.0f)) st |= ST_UNIFORM;
        }
        if (!st) {
            // weights on the kept set: max(0, e - S_P q) at a rejection, e for the bonus
            const bool v0 = lane < np, v1 = lane + 32 < np;
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
                // the kept entries in vocabulary order (rank of each index among them)
                int o0 = 0, o1 = 0;
                for (int s2 = 0; s2 < np; ++s2) {
                    const int is = s2 < 32 ? __shfl_sync(full, c0.i, s2) : __shfl_sync(full, c1.i, s2 - 32);
                    o0 += is < c0.i ? 1 : 0;
                    o1 += is < c1.i ? 1 : 0;
                }
                // scratch (the candidate buffers, free now): (weight hi, index) then (weight lo, index)
                Cand* ohi = reinterpret_cast<Cand*>(sh.wb[0]);
                Cand* olo = reinterpret_cast<Cand*>(sh.wb[1]);
                for (int t = lane; t < kTopKMax; t += 32) {
                    ohi[t] = Cand{0.0f, 0x7fffffff};
                    olo[t] = Cand{0.0f, 0x7fffffff};
                }
                __syncwarp();
                if (v0) {
                    ohi[o0] = Cand{w0.hi, c0.i};
                    olo[o0] = Cand{w0.lo, c0.i};
                }
                if (v1) {
                    ohi[o1] = Cand{w1.hi, c1.i};
                    olo[o1] = Cand{w1.lo, c1.i};
                }
                __syncwarp();
                const df a0 = df{ohi[lane].v, olo[lane].v}, a1 = df{ohi[lane + 32].v, olo[lane + 32].v};
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
                token = ohi[slot].i;
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
