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
// renormalised.  The residual max(0, p' - q) and the bonus live on P, so no
// second sweep of the vocabulary is needed: the stop position's draft
// probabilities are gathered at the kept entries.
//
// One CTA per sequence: a producer warp streams every position's logits
// through a ring of shared-memory stages; each of the four consumer warps
// keeps the best candidates of its share in a 128-entry buffer (an element
// enters when it reaches the warp's threshold, the 64th best so far; a full
// buffer is sorted and cut back to 64); at the end of a position each warp
// leaves its best 64 in a per-position merge area.  After the stream the
// warps merge positions in parallel (256 -> 64) and warp 0 walks the
// positions with double-float weights.
#pragma once
#include <cfloat>
#include <cstdint>

#include "exp2dd.cuh"
#include "ptx.cuh"
#include "verify_cluster.cuh"

namespace specv {

constexpr int kTopKMax = 64;                     // largest top_k this path takes
constexpr int kCandCap = 128;                    // per-warp candidate buffer
constexpr int kMergeLen = kConsumerWarps * kTopKMax;  // one position's warp lists

struct Cand {
    float v;  // logit
    int i;    // vocabulary index
};

// Rank order: larger logit first, lower index first among equal logits.
__device__ __forceinline__ bool cand_before(Cand a, Cand b) { return a.v > b.v || (a.v == b.v && a.i < b.i); }

__device__ __forceinline__ Cand cand_pad() { return Cand{-INFINITY, 0x7fffffff}; }

// Bitonic sort of n (a power of two) candidates in shared memory into rank
// order, by one warp.
__device__ __forceinline__ void warp_sort_cands(Cand* buf, int n, int lane) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = lane; t < n / 2; t += 32) {
                const int i = 2 * stride * (t / stride) + (t % stride);
                const int j = i + stride;
                const bool up = (i & size) == 0;  // this block ends in rank order
                const Cand a = buf[i], b = buf[j];
                if (up ? cand_before(b, a) : cand_before(a, b)) {
                    buf[i] = b;
                    buf[j] = a;
                }
            }
            __syncwarp();
        }
    }
}

// Sort the warp's buffer, keep the best 64 and raise the threshold to the
// 64th (while fewer than 64 are known every element qualifies).
__device__ __forceinline__ void warp_compact(Cand* wb, int& cnt, float& thr, int lane) {
    for (int t = cnt + lane; t < kCandCap; t += 32) wb[t] = cand_pad();
    __syncwarp();
    warp_sort_cands(wb, kCandCap, lane);
    if (cnt >= kTopKMax) {
        cnt = kTopKMax;
        thr = wb[kTopKMax - 1].v;
    }
}

// Add each lane's pending elements (bit e of pend: element e, get(e) gives
// it) that reach the threshold to the warp's buffer, one per lane a round.
template <typename Get>
__device__ __forceinline__ void warp_insert(Cand* wb, int& cnt, float& thr, uint32_t pend, Get get, int lane) {
    const unsigned full = 0xffffffffu;
    for (;;) {
        const bool has = pend != 0;
        if (!__any_sync(full, has)) break;
        const int e = has ? __ffs(pend) - 1 : 0;
        const Cand c = has ? get(e) : cand_pad();
        if (has) pend &= pend - 1;
        bool take = has && !(c.v < thr);  // ties enter; the sort orders them
        unsigned bal = __ballot_sync(full, take);
        if (cnt + __popc(bal) > kCandCap) {
            warp_compact(wb, cnt, thr, lane);
            take = take && !(c.v < thr);
            bal = __ballot_sync(full, take);
        }
        if (take) wb[cnt + __popc(bal & lanemask_lt())] = c;
        cnt += __popc(bal);
        __syncwarp();
    }
}

struct alignas(16) TopkSmem {
    unsigned long long full[kStages];
    unsigned long long empty[kStages];
    int tstart[kMaxK + 2];  // first tile of each position
    int head[kMaxK + 1];    // unaligned leading elements of each row
    int nbytes[kMaxK + 1];  // bytes of the 16-byte aligned interior
    int bad[kMaxK + 1];     // bit 0: a NaN was seen at this position; bit 1: a +inf
    int timeout;
    float2 exp2tab[128];
    int xs[kMaxK + 1];
};

// Dynamic shared memory of the top-k kernel: the ring, the per-position merge
// areas [k+1][kMergeLen], the per-warp candidate buffers [4][kCandCap].
inline size_t topk_dyn_smem(int k) {
    return static_cast<size_t>(kRingBytes) + static_cast<size_t>(k + 1) * kMergeLen * sizeof(Cand) +
           static_cast<size_t>(kConsumerWarps) * kCandCap * sizeof(Cand);
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1) verify_topk_kernel(const VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ __align__(16) TopkSmem sh;
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int kPer = kTileBytes / 16 / kConsumers;  // 16-byte chunks per consumer thread and tile
    constexpr int kEpc = 16 / esz;                       // elements per chunk
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool producer = warp == kConsumerWarps;
    const int b = blockIdx.x;
    const int k = a.k;
    const long long V = a.V;
    const int n = static_cast<int>(V);
    const unsigned char* lg = reinterpret_cast<const unsigned char*>(a.logits);
    unsigned char* ring = dyn_smem;
    Cand* merge = reinterpret_cast<Cand*>(dyn_smem + kRingBytes);             // [k+1][kMergeLen]
    Cand* wbuf = merge + static_cast<size_t>(k + 1) * kMergeLen + warp * kCandCap;  // this warp's buffer

    const float T = a.temp ? __ldg(a.temp + b) : 0.0f;
    const bool greedy = T == 0.0f;
    const bool t_ok = greedy || (T >= FLT_MIN && T <= FLT_MAX);
    const int K = a.top_k ? __ldg(a.top_k + b) : kTopKMax;
    const float top_p = a.top_p ? __ldg(a.top_p + b) : 1.0f;
    const bool f_ok = greedy || (K >= 1 && K <= kTopKMax && top_p > 0.0f && top_p <= 1.0f);

    // ---------------------------------------------------------------- setup
    if (tid < 128) sh.exp2tab[tid] = g_exp2_table[tid];
    if (tid <= k) {
        sh.bad[tid] = 0;
        sh.xs[tid] = tid < k ? __ldg(a.x + static_cast<long long>(b) * k + tid) : -1;
    }
    auto issue = [&](int tt, int it) {
        int i = 0;
        while (sh.tstart[i + 1] <= tt) ++i;
        const int off = (tt - sh.tstart[i]) * kTileBytes;
        const int bytes = min(kTileBytes, sh.nbytes[i] - off);
        const long long e0 = (static_cast<long long>(b) * (k + 1) + i) * V + sh.head[i];
        const int slot = it % kStages;
        const uint32_t bar = smem_u32(&sh.full[slot]);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(bytes));
        bulk_g2s(smem_u32(ring + slot * kTileBytes), lg + e0 * esz + off, static_cast<uint32_t>(bytes), bar);
    };
    int it_prod = 0;
    if (producer && lane == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&sh.full[s]), 1);
            mbar_init(smem_u32(&sh.empty[s]), kConsumerWarps);
        }
        sh.timeout = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
        int acc = 0;
        for (int i = 0; i <= k; ++i) {
            const uintptr_t addr = reinterpret_cast<uintptr_t>(lg + (static_cast<long long>(b) * (k + 1) + i) * V * esz);
            int h = static_cast<int>(((16 - (addr & 15)) & 15) / esz);
            if (h > n) h = n;
            const int nb = ((n - h) * esz) & ~15;
            sh.head[i] = h;
            sh.nbytes[i] = nb;
            sh.tstart[i] = acc;
            acc += (nb + kTileBytes - 1) / kTileBytes;
        }
        sh.tstart[k + 1] = acc;
        if (t_ok && f_ok)
            for (; it_prod < min(kStages, acc); ++it_prod) issue(it_prod, it_prod);
    }
    __syncthreads();
    const int total = (t_ok && f_ok) ? sh.tstart[k + 1] : 0;

    // ---------------------------------------------------------------- stream
    if (producer) {
        if (lane == 0) {
            for (int tt = it_prod; tt < total; ++tt) {
                const int slot = tt % kStages;
                if (sh.timeout || (tt >= kStages && !mbar_wait_bounded(smem_u32(&sh.empty[slot]),
                                                                        ((tt / kStages) & 1) ^ 1, kWaitPolls))) {
                    atomicOr(&sh.timeout, 1);
                    break;
                }
                issue(tt, tt);
            }
        }
        __syncwarp();
    } else {
        int it = 0;
        for (int i = 0; i <= k && t_ok && f_ok; ++i) {
            int cnt = 0;
            float thr = -INFINITY;
            const long long row_e0 = (static_cast<long long>(b) * (k + 1) + i) * V;
            const int h = sh.head[i];
            const int interior = sh.nbytes[i] / esz;
            const int ntiles = sh.tstart[i + 1] - sh.tstart[i];
            // unaligned head and tail: thread 0 reads them with plain loads
            auto scalar_part = [&](int lo, int hi) {
                uint32_t pend = 0;
                int bad = 0;
                if (tid == 0)
                    for (int e = lo; e < hi; ++e) {
                        const float l = load_logit(a.logits, row_e0 + e, BF16);
                        bad |= (l != l ? 1 : 0) | (l == INFINITY ? 2 : 0);
                        pend |= 1u << (e - lo);
                    }
                if (bad) atomicOr(&sh.bad[i], bad);
                __syncwarp();
                if (warp == 0)
                    warp_insert(wbuf, cnt, thr, pend,
                                [&](int e) { return Cand{load_logit(a.logits, row_e0 + lo + e, BF16), lo + e}; }, lane);
            };
            if (warp == 0 && h > 0) scalar_part(0, h);
            for (int lt = 0; lt < ntiles; ++lt, ++it) {
                const int slot = it % kStages;
                const bool ok = __all_sync(0xffffffffu, !sh.timeout && mbar_wait_bounded(smem_u32(&sh.full[slot]),
                                                                                          (it / kStages) & 1,
                                                                                          kWaitPolls));
                if (!ok) {
                    if (lane == 0) atomicOr(&sh.timeout, 1);
                    break;
                }
                const int bytes = min(kTileBytes, sh.nbytes[i] - lt * kTileBytes);
                const int nch = bytes >> 4;
                const unsigned char* tile = ring + slot * kTileBytes;
                const int tile_e = h + lt * (kTileBytes / esz);  // row index of the tile's first element
                // this lane's elements: chunk r = tid + 128 r, element q of the chunk -> bit r * kEpc + q
                float mx = -INFINITY, mx2 = -INFINITY;
                int bad = 0;
                uint32_t ge = 0;
#pragma unroll
                for (int r = 0; r < kPer; ++r) {
                    const int ch = tid + r * kConsumers;
                    if (ch < nch) {
#pragma unroll
                        for (int q = 0; q < kEpc; ++q) {
                            const float l = BF16 ? bf16_lo(reinterpret_cast<const uint16_t*>(tile + ch * 16)[q])
                                                 : reinterpret_cast<const float*>(tile + ch * 16)[q];
                            bad |= (l != l ? 1 : 0) | (l == INFINITY ? 2 : 0);
                            if (l > mx) {
                                mx2 = mx;
                                mx = l;
                            } else if (l > mx2) {
                                mx2 = l;
                            }
                            ge |= (l >= thr ? 1u : 0u) << (r * kEpc + q);
                        }
                    }
                }
                bad = static_cast<int>(__reduce_or_sync(0xffffffffu, static_cast<unsigned>(bad)));
                if (bad && lane == 0) atomicOr(&sh.bad[i], bad);
                if (thr == -INFINITY) {
                    // a position's first tile: at least 64 of its elements reach
                    // the smallest second-largest of the 32 lanes
                    float t0 = mx2;
                    for (int off = 16; off > 0; off >>= 1) t0 = fminf(t0, __shfl_xor_sync(0xffffffffu, t0, off));
                    thr = t0;
                }
                // elements below the (possibly raised) threshold drop out in warp_insert
                warp_insert(wbuf, cnt, thr, ge, [&](int e) {
                    const int r = e / kEpc, q = e % kEpc, ch = tid + r * kConsumers;
                    const float l = BF16 ? bf16_lo(reinterpret_cast<const uint16_t*>(tile + ch * 16)[q])
                                         : reinterpret_cast<const float*>(tile + ch * 16)[q];
                    return Cand{l, tile_e + ch * kEpc + q};
                }, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.empty[slot]));
            }
            if (warp == 0 && h + interior < n) scalar_part(h + interior, n);
            // the warp's best 64 of this position go to the merge area
            warp_compact(wbuf, cnt, thr, lane);
            Cand* dst = merge + static_cast<size_t>(i) * kMergeLen + warp * kTopKMax;
            for (int t = lane; t < kTopKMax; t += 32) dst[t] = t < cnt ? wbuf[t] : cand_pad();
            __syncwarp();
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- merge
    // each position's four warp lists (256) sorted: its best 64 come first
    if (!producer && t_ok && f_ok && !sh.timeout)
        for (int i = warp; i <= k; i += kConsumerWarps) warp_sort_cands(merge + static_cast<size_t>(i) * kMergeLen,
                                                                          kMergeLen, lane);
    __syncthreads();

    // ---------------------------------------------------------------- walk
    if (warp != 0) return;
    int st = !t_ok ? ST_TEMP : (!f_ok ? ST_FILTER : (sh.timeout ? ST_TIMEOUT : 0));
    int j = 0, token = -1;
    if (!st && greedy) {
        for (int i = 0; i <= k; ++i) {
            const int A = merge[static_cast<size_t>(i) * kMergeLen].i;
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
        Cand c0 = cand_pad(), c1 = cand_pad();
        df e0 = df_make(0.0f), e1 = df_make(0.0f), SP = df_make(0.0f);
        int np = 0;
        for (int i = 0; i <= k; ++i) {
            const Cand* m = merge + static_cast<size_t>(i) * kMergeLen;
            c0 = m[lane];
            c1 = m[lane + 32];
            rc.M = m[0].v;
            // this position's errors, in the walk's order of checks
            int pst = (sh.bad[i] || rc.M == -INFINITY) ? ST_NONFINITE : 0;  // NaN, +inf, or all -inf
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
                const unsigned h0 = __ballot_sync(0xffffffffu, lane < K && !df_less(s0, target));
                const unsigned h1 = __ballot_sync(0xffffffffu, lane + 32 < K && !df_less(s1, target));
                np = h0 ? __ffs(h0) : (h1 ? 32 + __ffs(h1) : K);
            }
            SP = np <= 32 ? df_shfl(s0, np - 1) : df_shfl(s1, np - 33);
            if (i == k) {
                j = k;
                break;
            }
            // p'(x): x among the kept ranks
            const bool h0 = lane < np && c0.i == x, h1 = lane + 32 < np && c1.i == x;
            const unsigned b0 = __ballot_sync(0xffffffffu, h0), b1 = __ballot_sync(0xffffffffu, h1);
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
                if (__any_sync(0xffffffffu, qb)) st |= ST_QBAD;
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
                    const int is = s2 < 32 ? __shfl_sync(0xffffffffu, c0.i, s2) : __shfl_sync(0xffffffffu, c1.i, s2 - 32);
                    o0 += is < c0.i ? 1 : 0;
                    o1 += is < c1.i ? 1 : 0;
                }
                // scratch: this warp's candidate buffer holds (weight hi, index) then (weight lo, index)
                Cand* ohi = wbuf;
                Cand* olo = wbuf + kTopKMax;
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
                const unsigned g0 = __ballot_sync(0xffffffffu, pos0 && df_less(target, p0));
                const unsigned g1 = __ballot_sync(0xffffffffu, pos1 && df_less(target, p1));
                int slot = -1;
                if (g0)
                    slot = __ffs(g0) - 1;
                else if (g1)
                    slot = 32 + __ffs(g1) - 1;
                else {  // only through rounding at the top edge: the last positive entry
                    const unsigned q0b = __ballot_sync(0xffffffffu, pos0), q1b = __ballot_sync(0xffffffffu, pos1);
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
