// verify_warp.cuh -- verify kernel for small vocabularies: one warp per
// sequence, lanes striding over V.  Same rule, same status bits and same
// inverse-CDF convention as the split-vocabulary kernel; here the whole stop
// row is weighted with the double-float exponential and summed as float pairs,
// which costs little at small V.
#pragma once
#include <cfloat>
#include <cstdint>

#include "exp2dd.cuh"
#include "ptx.cuh"
#include "verify_cluster.cuh"

namespace specv {

constexpr int kWarpKernelMaxV = 2048;
constexpr int kWarpsPerBlock = 4;

template <bool BF16>
__global__ void __launch_bounds__(32 * kWarpsPerBlock) verify_warp_kernel(const VerifyArgs a) {
    __shared__ float2 tab[128];
    for (int i = threadIdx.x; i < 128; i += blockDim.x) tab[i] = g_exp2_table[i];
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (b >= a.B) return;
    const int k = a.k;
    const long long V = a.V;
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
    // pass 1: per position, lanes stride over the vocabulary
    for (int i = 0; i <= k && t_ok; ++i) {
        float m = -INFINITY, s = 0.0f;
        int arg = 0x7fffffff;
        bool nan_seen = false;
        for (long long v = lane; v < V; v += 32) {
            const float l = load_logit(a.logits, base + i * V + v, BF16);
            if (greedy) {
                if (l != l) nan_seen = true;
                if (l > m) {
                    m = l;
                    arg = static_cast<int>(v);
                }
            } else {
                online_add(m, s, l, c);
            }
        }
        if (greedy) {
            for (int off = 16; off > 0; off >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
                const int a2 = __shfl_xor_sync(0xffffffffu, arg, off);
                merge_arg(m, arg, m2, a2);
            }
            nan_seen = __any_sync(0xffffffffu, nan_seen);
            if (arg == 0x7fffffff) arg = 0;
        } else {
            for (int off = 16; off > 0; off >>= 1) {
                const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
                const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
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
                    const float Lx = load_logit(a.logits, base + lane * V + xi, BF16);
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
    const unsigned mask = __ballot_sync(0xffffffffu, lane <= k && stop);
    const int j = t_ok ? __ffs(mask) - 1 : 0;
    int st = t_ok ? __shfl_sync(0xffffffffu, err, j) : ST_TEMP;
    const float uj = __shfl_sync(0xffffffffu, u1, j);
    if (t_ok && !greedy && !(st & ST_ERRMASK) && !(uj >= 0.0f && uj < 1.0f)) st |= ST_UNIFORM;
    const float Mj = __shfl_sync(0xffffffffu, Mi, j);
    const int Aj = __shfl_sync(0xffffffffu, Ai, j);

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
        // pass 2 on row j: every entry with exp2dd, sums as float pairs;
        // weights r = max(0, e - s q) (residual, s recomputed exactly), or e
        // (bonus, or empty residual)
        const long long row = base + j * V;
        const float* qrow = a.q ? a.q + (static_cast<long long>(b) * k + (j < k ? j : 0)) * V : nullptr;
        int mode = (j < k) ? (a.q ? MODE_RESIDUAL : MODE_ONEHOT) : MODE_BONUS;
        const int xj = __shfl_sync(0xffffffffu, xi, j < k ? j : 0);  // one-hot drafts: left out of the residual
        RowConst rc;
        rc.M = Mj;
        rc.s1 = 0.0f;
        rc.thr = 0.0f;
        rc.ch = c2.hi;
        rc.cl = c2.lo;
        df s_prec = df_make(0.0f);
        if (mode == MODE_RESIDUAL) {
            for (long long v = lane; v < V; v += 32)
                s_prec = df_sum(s_prec, exact_weight<BF16>(load_logit(a.logits, row + v, BF16), 0.0f, MODE_BONUS, rc,
                                                           df_make(0.0f), tab));
            s_prec = df_shfl(df_warp_total(s_prec), 0);
        }
        auto weight = [&](long long v) -> df {
            const float qq = mode == MODE_RESIDUAL ? __ldg(qrow + v) : 0.0f;
            const float l = (mode == MODE_ONEHOT && v == xj) ? -INFINITY : load_logit(a.logits, row + v, BF16);
            return exact_weight<BF16>(l, qq, mode, rc, s_prec, tab);
        };
        bool qbad = false;
        df W = df_make(0.0f);
        for (long long v = lane; v < V; v += 32) {
            W = df_sum(W, weight(v));
            if (mode == MODE_RESIDUAL) {
                const float qq = __ldg(qrow + v);
                qbad |= !(qq >= 0.0f && qq <= FLT_MAX);
            }
        }
        W = df_shfl(df_warp_total(W), 0);
        if (__any_sync(0xffffffffu, qbad)) st |= ST_QBAD;
        if ((mode == MODE_RESIDUAL || mode == MODE_ONEHOT) && !(st & ST_ERRMASK)) {
            const float Sj = __shfl_sync(0xffffffffu, Si, j);
            if (lane == 0 && a.dbg_resid)
                a.dbg_resid[b] = df_val(W) / (mode == MODE_RESIDUAL ? df_val(s_prec) : Sj);
            if (!(W.hi + W.lo > 0.0f)) {
                mode = MODE_FALLBACK;
                st |= ST_ZERO_RESIDUAL;
                W = df_make(0.0f);
                for (long long v = lane; v < V; v += 32) W = df_sum(W, weight(v));
                W = df_shfl(df_warp_total(W), 0);
            }
        }
        if (!(st & ST_ERRMASK)) {
            const df target = df_mul_f(W, uj);
            df acc = df_make(0.0f);
            int lastpos = -1;
            for (long long v0 = 0; v0 < V && token < 0; v0 += 32) {
                const long long v = v0 + lane;
                const df w = v < V ? weight(v) : df_make(0.0f);
                const bool pos = w.hi + w.lo > 0.0f;
                const df incl = df_sum(acc, df_warp_incl_scan(w, lane));
                const unsigned posm = __ballot_sync(0xffffffffu, pos);
                if (posm) lastpos = static_cast<int>(v0 + 31 - __clz(posm));
                const unsigned hit = __ballot_sync(0xffffffffu, pos && df_less(target, incl));
                if (hit) token = static_cast<int>(v0 + __ffs(hit) - 1);
                acc = df_shfl(incl, 31);
            }
            if (token < 0) token = lastpos;
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

}  // namespace specv
