// verify_warp.cuh -- verify kernel for small vocabularies: one warp per
// sequence.  Same rule, same status bits and same inverse-CDF convention as
// the split-vocabulary kernel.
//
// Pass 1 reads each position's logits with 16-byte loads (lane l takes
// chunks l, l + 32, ...; an unaligned head and tail take scalar loads) and
// folds each chunk into an online (max, sum of exponentials), or (max,
// lowest argmax) for greedy rows.  Pass 2 evaluates the exact e of every
// entry of the stop row once (the double-float exponential, cheap at small
// V) into shared memory, recomputes the normaliser from them, turns them into
// weights, and draws the token with a warp scan: each lane sums a contiguous
// chunk of entries, an inclusive scan over the lanes finds the chunk holding
// u * W, and that lane walks its chunk.
#pragma once
#include <cfloat>
#include <cstdint>

#include "exp2dd.cuh"
#include "ptx.cuh"
#include "verify_cluster.cuh"

namespace specv {

constexpr int kWarpKernelMaxV = 2048;
constexpr int kWarpsPerBlock = 2;  // each warp keeps its stop row's weights (16 KB at most) in shared memory

// Fold one value into the online (max, sum) or (max, argmax) state.
__device__ __forceinline__ void warp_fold1(bool greedy, float l, int v, float c, float& m, float& s, int& arg,
                                           bool& nan_seen) {
    if (greedy) {
        if (l != l) nan_seen = true;
        if (l > m) {
            m = l;
            arg = v;
        }
    } else {
        online_add(m, s, l, c);
    }
}

// One row of V logits starting at element row_e0: this lane's share of its
// (max, sum of exp((l - max) c)) or (max, lowest argmax), before the warp
// reduction.  The values of a 16-byte chunk are folded together: the chunk's
// maximum first, then every value's exponential at the (possibly raised)
// running maximum -- the same arithmetic as one value at a time, in another
// order, and the same outcome for NaN and infinite logits.
template <bool BF16>
__device__ __forceinline__ void warp_row_fold(const void* logits, long long row_e0, int V, bool greedy, float c,
                                              int lane, float& m, float& s, int& arg, bool& nan_seen) {
    constexpr int esz = BF16 ? 2 : 4;
    constexpr int vw = 16 / esz;  // values per 16-byte chunk
    const unsigned char* p = reinterpret_cast<const unsigned char*>(logits) + row_e0 * esz;
    const int h = min(V, static_cast<int>(((16 - (reinterpret_cast<uintptr_t>(p) & 15)) & 15) / esz));
    const int nch = (V - h) / vw;
    const int tail0 = h + nch * vw;
    if (lane < h) warp_fold1(greedy, load_logit(logits, row_e0 + lane, BF16), lane, c, m, s, arg, nan_seen);
    const uint4* cp = reinterpret_cast<const uint4*>(p + h * esz);
    // eight chunks a lane are loaded before any is folded: eight loads in flight
    constexpr int kU = 8;
    for (int ch0 = lane; ch0 < nch; ch0 += 32 * kU) {
        uint4 wq[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int ch = ch0 + 32 * u;
            const uint32_t ninf = BF16 ? 0xff80ff80u : 0xff800000u;
            wq[u] = ch < nch ? __ldg(cp + ch) : make_uint4(ninf, ninf, ninf, ninf);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
        const int ch = ch0 + 32 * u;
        if (ch >= nch) break;
        const uint4 w = wq[u];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        float f[vw];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            if (BF16) {
                f[2 * t] = bf16_lo(ws[t]);
                f[2 * t + 1] = bf16_hi(ws[t]);
            } else {
                f[t] = __uint_as_float(ws[t]);
            }
        }
        const int v0 = h + ch * vw;
        if (greedy) {
#pragma unroll
            for (int t = 0; t < vw; ++t) warp_fold1(true, f[t], v0 + t, c, m, s, arg, nan_seen);
        } else {
            float cm = f[0];
#pragma unroll
            for (int t = 1; t < vw; ++t) cm = fmaxf(cm, f[t]);
            if (cm > m) {
                s = (m == -INFINITY) ? s * 0.0f : s * ex2((m - cm) * c);
                m = cm;
            }
#pragma unroll
            for (int t = 0; t < vw; ++t)
                if (m != -INFINITY || f[t] != f[t]) s += ex2((f[t] - m) * c);
        }
        }
    }
    if (lane < V - tail0)
        warp_fold1(greedy, load_logit(logits, row_e0 + tail0 + lane, BF16), tail0 + lane, c, m, s, arg, nan_seen);
}

template <bool BF16>
__global__ void __launch_bounds__(32 * kWarpsPerBlock) verify_warp_kernel(const VerifyArgs a) {
    __shared__ float2 tab[128];
    // the stop row's e, then its weights (pairs); entry v at v + v / 32, so
    // that lanes walking contiguous chunks fall in different banks
    __shared__ float2 wbuf[kWarpsPerBlock][kWarpKernelMaxV + kWarpKernelMaxV / 32];
    for (int i = threadIdx.x; i < 128; i += blockDim.x) tab[i] = g_exp2_table[i];
    __syncthreads();
    const unsigned full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int b = blockIdx.x * kWarpsPerBlock + wib;
    if (b >= a.B) return;
    float2* wbase = wbuf[wib];
    auto wv = [&](int v) -> float2& { return wbase[v + (v >> 5)]; };
    const int k = a.k;
    const int V = static_cast<int>(a.V);
    const float T = a.temp ? __ldg(a.temp + b) : 0.0f;
    const bool greedy = (T == 0.0f);
    const bool t_ok = greedy || (T >= FLT_MIN && T <= FLT_MAX);
    const float c = (greedy || !t_ok) ? 0.0f : kLog2e / T;
    const df c2 = (greedy || !t_ok) ? df_make(0.0f) : log2e_over(T);
    const long long base = static_cast<long long>(b) * (k + 1) * V;

    int xi = -1, pi = lane - 1;
    float u0 = 0.0f, u1 = 0.0f, Mi = -INFINITY, Si = 0.0f, p = 0.0f, qx = 0.0f;
    int Ai = 0x7fffffff, nanf = 0;
    if (lane <= k && t_ok) {
        if (lane < k) xi = __ldg(a.x + static_cast<long long>(b) * k + lane);
        if (lane < k && a.parents) pi = __ldg(a.parents + static_cast<long long>(b) * k + lane);
        if (!greedy) {
            u0 = __ldg(a.u + (static_cast<long long>(b) * (k + 1) + lane) * 2);
            u1 = __ldg(a.u + (static_cast<long long>(b) * (k + 1) + lane) * 2 + 1);
        }
    }
    // pass 1: per position, lanes over 16-byte chunks, then the warp reduction
    for (int i = 0; i <= k && t_ok; ++i) {
        float m = -INFINITY, s = 0.0f;
        int arg = 0x7fffffff;
        bool nan_seen = false;
        warp_row_fold<BF16>(a.logits, base + static_cast<long long>(i) * V, V, greedy, c, lane, m, s, arg, nan_seen);
        __syncwarp();
        if (greedy) {
            for (int off = 16; off > 0; off >>= 1) {
                const float m2 = __shfl_xor_sync(full, m, off);
                const int a2 = __shfl_xor_sync(full, arg, off);
                merge_arg(m, arg, m2, a2);
            }
            nan_seen = __any_sync(full, nan_seen);
            if (arg == 0x7fffffff) arg = 0;
        } else {
            for (int off = 16; off > 0; off >>= 1) {
                const float m2 = __shfl_xor_sync(full, m, off);
                const float s2 = __shfl_xor_sync(full, s, off);
                merge_ms(m, s, m2, s2, c);
            }
        }
        if (lane == i) {
            Mi = m;
            Si = s;
            Ai = arg;
            nanf = nan_seen ? 1 : 0;
        }
    }
    __syncwarp();
    if (a.parents) {
        // a draft tree (all rows greedy)
        tree_greedy_warp(a, b, k, lane, xi, pi, Ai == 0x7fffffff ? 0 : Ai, nanf, true);
        if (lane <= k && a.dbg_max) a.dbg_max[static_cast<long long>(b) * (k + 1) + lane] = Mi;
        return;
    }
    // accept tests, one lane per position
    int err = 0;
    bool stop = false;
    if (lane <= k && t_ok) {
        if (greedy) {
            if (nanf) err |= ST_NONFINITE;
            if (lane < k && (xi < 0 || xi >= V)) err |= ST_TOKEN;
            stop = err != 0 || lane == k || xi != Ai;
        } else {
            if (!(isfinite(Mi) && isfinite(Si))) err |= ST_NONFINITE;
            if (lane < k) {
                if (xi < 0 || xi >= V) err |= ST_TOKEN;
                if (!(u0 >= 0.0f && u0 < 1.0f)) err |= ST_UNIFORM;
                if (xi >= 0 && xi < V) {
                    qx = a.q ? __ldg(a.q + (static_cast<long long>(b) * k + lane) * V + xi) : 1.0f;
                    if (!(qx >= 0.0f && qx <= FLT_MAX)) err |= ST_QBAD;
                }
                if (!err) {
                    const float Lx = load_logit(a.logits, base + static_cast<long long>(lane) * V + xi, BF16);
                    RowConst rc;
                    rc.M = Mi;
                    rc.s1 = Si;
                    rc.thr = 0.0f;
                    rc.ch = c2.hi;
                    rc.cl = c2.lo;
                    p = df_val(exact_weight<BF16>(Lx, 0.0f, MODE_BONUS, rc, df_make(0.0f), tab)) / Si;
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
    __syncwarp();
    const unsigned mask = __ballot_sync(full, lane <= k && stop);
    const int j = t_ok ? __ffs(mask) - 1 : 0;
    int st = t_ok ? __shfl_sync(full, err, j) : ST_TEMP;
    const float uj = __shfl_sync(full, u1, j);
    if (t_ok && !greedy && !(st & ST_ERRMASK) && !(uj >= 0.0f && uj < 1.0f)) st |= ST_UNIFORM;
    const float Mj = __shfl_sync(full, Mi, j);
    const int Aj = __shfl_sync(full, Ai, j);

    if (lane <= k && t_ok) {
        if (a.dbg_max) a.dbg_max[static_cast<long long>(b) * (k + 1) + lane] = Mi;
        if (a.dbg_sumexp) a.dbg_sumexp[static_cast<long long>(b) * (k + 1) + lane] = greedy ? 0.0f : Si;
        if (lane < k) {
            const bool xok = xi >= 0 && xi < V;
            if (a.dbg_p) a.dbg_p[static_cast<long long>(b) * k + lane] = (greedy || !xok) ? 0.0f : p;
            if (a.dbg_q) a.dbg_q[static_cast<long long>(b) * k + lane] = (greedy || !xok) ? 0.0f : qx;
        }
    }
    if (lane == 0 && a.dbg_resid) a.dbg_resid[b] = 0.0f;

    int token = -1;
    const bool bad = (st & ST_ERRMASK) != 0;
    if (!bad && greedy) token = Aj;
    if (!bad && !greedy) {
        // pass 2 on row j: the exact e of every entry, once (the draft token's
        // entry of a one-hot row weighs nothing); s recomputed from them
        const long long row = base + static_cast<long long>(j) * V;
        const float* qrow = a.q ? a.q + (static_cast<long long>(b) * k + (j < k ? j : 0)) * V : nullptr;
        int mode = (j < k) ? (a.q ? MODE_RESIDUAL : MODE_ONEHOT) : MODE_BONUS;
        const int xj = __shfl_sync(full, xi, j < k ? j : 0);
        RowConst rc;
        rc.M = Mj;
        rc.s1 = 0.0f;
        rc.thr = 0.0f;
        rc.ch = c2.hi;
        rc.cl = c2.lo;
        auto exact_e = [&](int v, bool drop_draft) -> df {
            const float l = (drop_draft && v == xj) ? -INFINITY : load_logit(a.logits, row + v, BF16);
            return l == -INFINITY ? df_make(0.0f) : precise_e<BF16>(l, rc, tab);
        };
        // entries v = lane + 32 t, eight at a time: their loads are issued
        // together, before any of them is used
        constexpr int kB = 8;
        df se = df_make(0.0f);
        for (int v0 = lane; v0 < V; v0 += 32 * kB) {
            float lb[kB];
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int v = v0 + 32 * u;
                lb[u] = v < V ? load_logit(a.logits, row + v, BF16) : -INFINITY;
            }
#pragma unroll
            for (int u = 0; u < kB; ++u) {
                const int v = v0 + 32 * u;
                if (v >= V) break;
                const float l = (mode == MODE_ONEHOT && v == xj) ? -INFINITY : lb[u];
                const df e = l == -INFINITY ? df_make(0.0f) : precise_e<BF16>(l, rc, tab);
                wv(v) = make_float2(e.hi, e.lo);
                se = df_sum(se, e);
            }
        }
        const df s_prec = df_shfl(df_warp_total(se), 0);
        df W = s_prec;  // bonus and one-hot rows: the weights are the e
        if (mode == MODE_RESIDUAL) {
            // w = max(0, e - s q), the product exact through one fma
            bool qbad = false;
            df Wl = df_make(0.0f);
            for (int v0 = lane; v0 < V; v0 += 32 * kB) {
                float qb[kB];
#pragma unroll
                for (int u = 0; u < kB; ++u) {
                    const int v = v0 + 32 * u;
                    qb[u] = v < V ? __ldg(qrow + v) : 0.0f;
                }
#pragma unroll
                for (int u = 0; u < kB; ++u) {
                    const int v = v0 + 32 * u;
                    if (v >= V) break;
                    const float qq = qb[u];
                    qbad |= !(qq >= 0.0f && qq <= FLT_MAX);
                    const float2 e2 = wv(v);
                    df r = minus_sq(df{e2.x, e2.y}, s_prec, qq);
                    if (!(r.hi + r.lo > 0.0f)) r = df_make(0.0f);
                    wv(v) = make_float2(r.hi, r.lo);
                    Wl = df_sum(Wl, r);
                }
            }
            W = df_shfl(df_warp_total(Wl), 0);
            if (__any_sync(full, qbad)) st |= ST_QBAD;
        }
        if ((mode == MODE_RESIDUAL || mode == MODE_ONEHOT) && !(st & ST_ERRMASK)) {
            const float Sj = __shfl_sync(full, Si, j);
            if (lane == 0 && a.dbg_resid)
                a.dbg_resid[b] = df_val(W) / (mode == MODE_RESIDUAL ? df_val(s_prec) : Sj);
            if (!(W.hi + W.lo > 0.0f)) {
                // empty residual: sample p itself, every entry
                mode = MODE_FALLBACK;
                st |= ST_ZERO_RESIDUAL;
                df se2 = df_make(0.0f);
                for (int v = lane; v < V; v += 32) {
                    const df e = exact_e(v, false);
                    wv(v) = make_float2(e.hi, e.lo);
                    se2 = df_sum(se2, e);
                }
                W = df_shfl(df_warp_total(se2), 0);
            }
        }
        __syncwarp();  // every lane's weights are in shared memory
        if (!(st & ST_ERRMASK)) {
            // inverse CDF: lane l sums entries [l cs, (l + 1) cs) in order; the
            // first lane with a positive sum whose inclusive prefix exceeds
            // u W holds the token, which it finds by walking its entries
            const df target = df_mul_f(W, uj);
            const int cs = (V + 31) / 32;
            const int c0 = min(V, lane * cs), c1 = min(V, c0 + cs);
            df lsum = df_make(0.0f);
            int lastpos = -1;
            for (int v = c0; v < c1; ++v) {
                const float2 w2 = wv(v);
                if (w2.x + w2.y > 0.0f) {
                    lsum = df_sum(lsum, df{w2.x, w2.y});
                    lastpos = v;
                }
            }
            const df incl = df_warp_incl_scan(lsum, lane);
            const df excl = df_shfl_up(incl, 1);
            const bool lpos = lastpos >= 0;
            const unsigned hit = __ballot_sync(full, lpos && df_less(target, incl));
            if (hit) {
                const int L = __ffs(hit) - 1;
                if (lane == L) {
                    df acc = lane == 0 ? df_make(0.0f) : excl;
                    for (int v = c0; v < c1 && token < 0; ++v) {
                        const float2 w2 = wv(v);
                        if (w2.x + w2.y > 0.0f) {
                            acc = df_sum(acc, df{w2.x, w2.y});
                            if (df_less(target, acc)) token = v;
                        }
                    }
                    if (token < 0) token = lastpos;  // only through rounding at the chunk's end
                }
                token = __shfl_sync(full, token, L);
            } else {
                // only through rounding at the top edge: the last positive entry
                token = __reduce_max_sync(full, static_cast<unsigned>(lastpos + 1)) - 1;
            }
        }
    }
    const bool bad2 = (st & ST_ERRMASK) != 0;
    if (lane <= k) {
        int tok = -1;
        if (!bad2) tok = lane < j ? xi : (lane == j ? token : -1);
        a.out_tokens[static_cast<long long>(b) * (k + 1) + lane] = tok;
    }
    if (lane == 0) {
        a.num_accepted[b] = bad2 ? 0 : j;
        if (a.row_status) a.row_status[b] = st;
    }
}

// ------------------------------------------------------------------ one CTA per row
// The same rule for small batches: one CTA of kRowWarps warps per row, so that
// a row's positions are folded in parallel (warp w takes positions w, w +
// kRowWarps, ...) and its stop row is weighed by every thread.  Warp 0 takes
// the accept tests (lane i, position i); the draw is a block-wide scan: each
// thread sums a contiguous chunk of the weights, the chunk sums are scanned
// (lanes, then warps), and the thread whose chunk holds u * W walks it.
constexpr int kRowWarps = 8;
constexpr int kRowThreads = kRowWarps * 32;

// Pair total over the block, in every thread (red: kRowWarps pairs of shared
// memory; the warps' totals are added in warp order).
__device__ __forceinline__ df row_block_total(df v, float2* red, int warp, int lane) {
    v = df_warp_total(v);
    if (lane == 0) red[warp] = make_float2(v.hi, v.lo);
    __syncthreads();
    df t = df_make(0.0f);
    for (int w = 0; w < kRowWarps; ++w) t = df_sum(t, df{red[w].x, red[w].y});
    __syncthreads();  // red may be reused
    return t;
}

template <bool BF16>
__global__ void __launch_bounds__(kRowThreads) verify_row_kernel(const VerifyArgs a) {
    __shared__ float2 tab[128];
    __shared__ float2 wbuf[kWarpKernelMaxV + kWarpKernelMaxV / 32];  // entry v at v + v / 32
    __shared__ float posM[kMaxK + 1], posS[kMaxK + 1];
    __shared__ int posA[kMaxK + 1], posF[kMaxK + 1];
    __shared__ float2 red[kRowWarps];
    __shared__ int s_j, s_st, s_token, s_hit[kRowWarps];
    __shared__ float s_uj, s_Mj, s_Sj;
    const unsigned full = 0xffffffffu;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < 128; i += kRowThreads) tab[i] = g_exp2_table[i];
    auto wv = [&](int v) -> float2& { return wbuf[v + (v >> 5)]; };
    const int b = blockIdx.x;
    const int k = a.k;
    const int V = static_cast<int>(a.V);
    const float T = a.temp ? __ldg(a.temp + b) : 0.0f;
    const bool greedy = (T == 0.0f);
    const bool t_ok = greedy || (T >= FLT_MIN && T <= FLT_MAX);
    const float c = (greedy || !t_ok) ? 0.0f : kLog2e / T;
    const df c2 = (greedy || !t_ok) ? df_make(0.0f) : log2e_over(T);
    const long long base = static_cast<long long>(b) * (k + 1) * V;

    // pass 1: warp w folds positions w, w + kRowWarps, ...
    for (int i = warp; i <= k && t_ok; i += kRowWarps) {
        float m = -INFINITY, s = 0.0f;
        int arg = 0x7fffffff;
        bool nan_seen = false;
        warp_row_fold<BF16>(a.logits, base + static_cast<long long>(i) * V, V, greedy, c, lane, m, s, arg, nan_seen);
        __syncwarp();
        if (greedy) {
            for (int off = 16; off > 0; off >>= 1) {
                const float m2 = __shfl_xor_sync(full, m, off);
                const int a2 = __shfl_xor_sync(full, arg, off);
                merge_arg(m, arg, m2, a2);
            }
            nan_seen = __any_sync(full, nan_seen);
            if (arg == 0x7fffffff) arg = 0;
        } else {
            for (int off = 16; off > 0; off >>= 1) {
                const float m2 = __shfl_xor_sync(full, m, off);
                const float s2 = __shfl_xor_sync(full, s, off);
                merge_ms(m, s, m2, s2, c);
            }
        }
        if (lane == 0) {
            posM[i] = m;
            posS[i] = s;
            posA[i] = arg;
            posF[i] = nan_seen ? 1 : 0;
        }
    }
    __syncthreads();

    // decisions: warp 0, lane i = position i
    if (warp == 0) {
        int xi = -1, pi = lane - 1;
        float u0 = 0.0f, u1 = 0.0f, p = 0.0f, qx = 0.0f;
        const bool have = lane <= k && t_ok;
        const float Mi = have ? posM[lane] : -INFINITY, Si = have ? posS[lane] : 0.0f;
        const int Ai = have ? posA[lane] : 0, nanf = have ? posF[lane] : 0;
        if (have) {
            if (lane < k) xi = __ldg(a.x + static_cast<long long>(b) * k + lane);
            if (lane < k && a.parents) pi = __ldg(a.parents + static_cast<long long>(b) * k + lane);
            if (!greedy) {
                u0 = __ldg(a.u + (static_cast<long long>(b) * (k + 1) + lane) * 2);
                u1 = __ldg(a.u + (static_cast<long long>(b) * (k + 1) + lane) * 2 + 1);
            }
        }
        if (a.parents) {
            // a draft tree (all rows greedy)
            tree_greedy_warp(a, b, k, lane, xi, pi, Ai, nanf, true);
            if (lane <= k && a.dbg_max) a.dbg_max[static_cast<long long>(b) * (k + 1) + lane] = Mi;
            if (lane == 0) s_st = ST_TEMP;  // nothing more to do
        } else {
            int err = 0;
            bool stop = false;
            if (have) {
                if (greedy) {
                    if (nanf) err |= ST_NONFINITE;
                    if (lane < k && (xi < 0 || xi >= V)) err |= ST_TOKEN;
                    stop = err != 0 || lane == k || xi != Ai;
                } else {
                    if (!(isfinite(Mi) && isfinite(Si))) err |= ST_NONFINITE;
                    if (lane < k) {
                        if (xi < 0 || xi >= V) err |= ST_TOKEN;
                        if (!(u0 >= 0.0f && u0 < 1.0f)) err |= ST_UNIFORM;
                        if (xi >= 0 && xi < V) {
                            qx = a.q ? __ldg(a.q + (static_cast<long long>(b) * k + lane) * V + xi) : 1.0f;
                            if (!(qx >= 0.0f && qx <= FLT_MAX)) err |= ST_QBAD;
                        }
                        if (!err) {
                            const float Lx = load_logit(a.logits, base + static_cast<long long>(lane) * V + xi, BF16);
                            RowConst rc;
                            rc.M = Mi;
                            rc.s1 = Si;
                            rc.thr = 0.0f;
                            rc.ch = c2.hi;
                            rc.cl = c2.lo;
                            p = df_val(exact_weight<BF16>(Lx, 0.0f, MODE_BONUS, rc, df_make(0.0f), tab)) / Si;
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
            __syncwarp();
            const unsigned mask = __ballot_sync(full, lane <= k && stop);
            const int j = t_ok ? __ffs(mask) - 1 : 0;
            int st = t_ok ? __shfl_sync(full, err, j) : ST_TEMP;
            const float uj = __shfl_sync(full, u1, j);
            if (t_ok && !greedy && !(st & ST_ERRMASK) && !(uj >= 0.0f && uj < 1.0f)) st |= ST_UNIFORM;
            if (have) {
                if (a.dbg_max) a.dbg_max[static_cast<long long>(b) * (k + 1) + lane] = Mi;
                if (a.dbg_sumexp) a.dbg_sumexp[static_cast<long long>(b) * (k + 1) + lane] = greedy ? 0.0f : Si;
                if (lane < k) {
                    const bool xok = xi >= 0 && xi < V;
                    if (a.dbg_p) a.dbg_p[static_cast<long long>(b) * k + lane] = (greedy || !xok) ? 0.0f : p;
                    if (a.dbg_q) a.dbg_q[static_cast<long long>(b) * k + lane] = (greedy || !xok) ? 0.0f : qx;
                }
            }
            const int Aj = __shfl_sync(full, Ai, j);
            const int xj = __shfl_sync(full, xi, j < k ? j : 0);
            const float Mj = __shfl_sync(full, Mi, j), Sj = __shfl_sync(full, Si, j);
            if (lane == 0) {
                if (a.dbg_resid) a.dbg_resid[b] = 0.0f;
                s_j = j;
                s_st = st;
                s_uj = uj;
                s_Mj = Mj;
                s_Sj = Sj;
                s_token = greedy ? Aj : -1;
                s_hit[0] = xj;  // the draft token at j (one-hot rows leave it out of the residual)
            }
            // the kept drafts and the -1 after j (the token at j is written after the draw)
            const bool bad = (st & ST_ERRMASK) != 0;
            if (lane <= k && lane != j)
                a.out_tokens[static_cast<long long>(b) * (k + 1) + lane] = (!bad && lane < j) ? xi : -1;
        }
    }
    __syncthreads();
    if (a.parents) return;
    const int j = s_j;
    int st = s_st;
    const int xj = s_hit[0];
    __syncthreads();  // s_hit is reused by the draw
    int token = s_token;
    if (!(st & ST_ERRMASK) && !greedy) {
        const long long row = base + static_cast<long long>(j) * V;
        const float* qrow = a.q ? a.q + (static_cast<long long>(b) * k + (j < k ? j : 0)) * V : nullptr;
        int mode = (j < k) ? (a.q ? MODE_RESIDUAL : MODE_ONEHOT) : MODE_BONUS;
        RowConst rc;
        rc.M = s_Mj;
        rc.s1 = 0.0f;
        rc.thr = 0.0f;
        rc.ch = c2.hi;
        rc.cl = c2.lo;
        auto exact_e = [&](int v, bool drop_draft) -> df {
            const float l = (drop_draft && v == xj) ? -INFINITY : load_logit(a.logits, row + v, BF16);
            return l == -INFINITY ? df_make(0.0f) : precise_e<BF16>(l, rc, tab);
        };
        df se = df_make(0.0f);
        for (int v = tid; v < V; v += kRowThreads) {
            const df e = exact_e(v, mode == MODE_ONEHOT);
            wv(v) = make_float2(e.hi, e.lo);
            se = df_sum(se, e);
        }
        const df s_prec = row_block_total(se, red, warp, lane);
        df W = s_prec;
        if (mode == MODE_RESIDUAL) {
            bool qbad = false;
            df Wl = df_make(0.0f);
            for (int v = tid; v < V; v += kRowThreads) {
                const float qq = __ldg(qrow + v);
                qbad |= !(qq >= 0.0f && qq <= FLT_MAX);
                const float2 e2 = wv(v);
                df r = minus_sq(df{e2.x, e2.y}, s_prec, qq);
                if (!(r.hi + r.lo > 0.0f)) r = df_make(0.0f);
                wv(v) = make_float2(r.hi, r.lo);
                Wl = df_sum(Wl, r);
            }
            if (__syncthreads_or(qbad ? 1 : 0)) st |= ST_QBAD;
            W = row_block_total(Wl, red, warp, lane);
        }
        if ((mode == MODE_RESIDUAL || mode == MODE_ONEHOT) && !(st & ST_ERRMASK)) {
            if (tid == 0 && a.dbg_resid) a.dbg_resid[b] = df_val(W) / (mode == MODE_RESIDUAL ? df_val(s_prec) : s_Sj);
            if (!(W.hi + W.lo > 0.0f)) {
                // empty residual: sample p itself, every entry
                mode = MODE_FALLBACK;
                st |= ST_ZERO_RESIDUAL;
                df se2 = df_make(0.0f);
                for (int v = tid; v < V; v += kRowThreads) {
                    const df e = exact_e(v, false);
                    wv(v) = make_float2(e.hi, e.lo);
                    se2 = df_sum(se2, e);
                }
                W = row_block_total(se2, red, warp, lane);
            }
        }
        __syncthreads();  // every thread's weights are in shared memory
        if (!(st & ST_ERRMASK)) {
            // inverse CDF: thread t sums entries [t cs, (t + 1) cs) in order; the
            // first thread with a positive sum whose inclusive prefix exceeds
            // u W holds the token and walks its entries
            const df target = df_mul_f(W, s_uj);
            const int cs = (V + kRowThreads - 1) / kRowThreads;
            const int c0 = min(V, tid * cs), c1 = min(V, c0 + cs);
            df lsum = df_make(0.0f);
            int lastpos = -1;
            for (int v = c0; v < c1; ++v) {
                const float2 w2 = wv(v);
                if (w2.x + w2.y > 0.0f) {
                    lsum = df_sum(lsum, df{w2.x, w2.y});
                    lastpos = v;
                }
            }
            const df incl_w = df_warp_incl_scan(lsum, lane);
            if (lane == 31) red[warp] = make_float2(incl_w.hi, incl_w.lo);
            __syncthreads();
            df basew = df_make(0.0f);
            for (int w = 0; w < warp; ++w) basew = df_sum(basew, df{red[w].x, red[w].y});
            const df incl = df_sum(basew, incl_w);
            // (every lane takes part in the shuffle; lane 0 then drops its value)
            const df up = df_shfl_up(incl_w, 1);
            const df excl = df_sum(basew, lane == 0 ? df_make(0.0f) : up);
            const unsigned hit = __ballot_sync(full, lastpos >= 0 && df_less(target, incl));
            if (lane == 0) s_hit[warp] = hit ? warp * 32 + __ffs(hit) - 1 : 0x7fffffff;
            const int lastall = static_cast<int>(__reduce_max_sync(full, static_cast<unsigned>(lastpos + 1))) - 1;
            __syncthreads();
            int owner = 0x7fffffff;
            for (int w = 0; w < kRowWarps; ++w) owner = min(owner, s_hit[w]);
            if (lane == 0) red[warp] = make_float2(__int_as_float(lastall), 0.0f);
            __syncthreads();
            if (owner == 0x7fffffff) {
                // only through rounding at the top edge: the last positive entry
                if (tid == 0) {
                    int lp = -1;
                    for (int w = 0; w < kRowWarps; ++w) lp = max(lp, __float_as_int(red[w].x));
                    s_token = lp;
                }
            } else if (tid == owner) {
                df acc = excl;
                int tk = -1;
                for (int v = c0; v < c1 && tk < 0; ++v) {
                    const float2 w2 = wv(v);
                    if (w2.x + w2.y > 0.0f) {
                        acc = df_sum(acc, df{w2.x, w2.y});
                        if (df_less(target, acc)) tk = v;
                    }
                }
                s_token = tk >= 0 ? tk : lastpos;  // (lastpos: only through rounding at the chunk's end)
            }
        }
        __syncthreads();
        token = s_token;
    }
    if (tid == 0) {
        const bool bad = (st & ST_ERRMASK) != 0;
        a.out_tokens[static_cast<long long>(b) * (k + 1) + j] = bad ? -1 : token;
        a.num_accepted[b] = bad ? 0 : j;
        if (a.row_status) a.row_status[b] = st;
    }
}

}  // namespace specv
