// verify_warp.cuh -- verify kernel for small vocabularies: one warp per
// sequence, lanes striding over V.  Same rule, same status bits and same
// inverse-CDF convention as the split-vocabulary kernel; here the whole stop
// row is weighted with the double-float exponential and summed in float64,
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

__device__ __forceinline__ float2 row_exp2dd(float l, float M, float ch, float cl, bool bf16, const float2* tab) {
    if (l == -INFINITY) return make_float2(0.0f, 0.0f);  // a masked entry
    float dh = l - M, dl = 0.0f;
    if (!bf16) two_sum(l, -M, dh, dl);
    const float xh = dh * ch;
    const float xl = fmaf(dl, ch, fmaf(dh, cl, fmaf(dh, ch, -xh)));
    return exp2dd(xh, xl, tab);
}

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
    const double cd = (greedy || !t_ok) ? 0.0 : 1.4426950408889634 / static_cast<double>(T);
    const float ch = static_cast<float>(cd), cl = static_cast<float>(cd - static_cast<double>(ch));
    const long long base = static_cast<long long>(b) * (k + 1) * V;

    int xi = -1;
    float u0 = 0.0f, u1 = 0.0f, Mi = -INFINITY, Si = 0.0f, p = 0.0f, qx = 0.0f;
    int Ai = 0x7fffffff, nanf = 0;
    if (lane <= k && t_ok) {
        if (lane < k) xi = __ldg(a.x + static_cast<long long>(b) * k + lane);
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
                    qx = __ldg(a.q + (static_cast<long long>(b) * k + lane) * V + xi);
                    if (!(qx >= 0.0f && qx <= FLT_MAX)) err |= ST_QBAD;
                }
                if (!err) {
                    const float Lx = load_logit(a.logits, base + lane * V + xi, BF16);
                    const float2 e = row_exp2dd(Lx, Mi, ch, cl, BF16, tab);
                    p = (e.x + e.y) / Si;
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
        // pass 2 on row j in float64: weights r = max(0, e - s q) (residual,
        // s recomputed exactly), or e (bonus, or empty residual)
        const long long row = base + j * V;
        const float* qrow = a.q + (static_cast<long long>(b) * k + (j < k ? j : 0)) * V;
        int mode = (j < k) ? MODE_RESIDUAL : MODE_BONUS;
        double s_prec = 0.0;
        if (mode == MODE_RESIDUAL) {
            for (long long v = lane; v < V; v += 32) {
                const float2 e = row_exp2dd(load_logit(a.logits, row + v, BF16), Mj, ch, cl, BF16, tab);
                s_prec += static_cast<double>(e.x) + static_cast<double>(e.y);
            }
            for (int off = 16; off > 0; off >>= 1) s_prec += __shfl_xor_sync(0xffffffffu, s_prec, off);
        }
        auto weight = [&](long long v) -> double {
            const float2 e = row_exp2dd(load_logit(a.logits, row + v, BF16), Mj, ch, cl, BF16, tab);
            double w = static_cast<double>(e.x) + static_cast<double>(e.y);
            if (mode == MODE_RESIDUAL) {
                w -= s_prec * static_cast<double>(__ldg(qrow + v));
                if (w < 0.0) w = 0.0;
            }
            return w;
        };
        bool qbad = false;
        double W = 0.0;
        for (long long v = lane; v < V; v += 32) {
            W += weight(v);
            if (mode == MODE_RESIDUAL) {
                const float qq = __ldg(qrow + v);
                qbad |= !(qq >= 0.0f && qq <= FLT_MAX);
            }
        }
        for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
        if (__any_sync(0xffffffffu, qbad)) st |= ST_QBAD;
        if (mode == MODE_RESIDUAL && !(st & ST_ERRMASK)) {
            if (lane == 0 && a.dbg_resid) a.dbg_resid[b] = static_cast<float>(W / s_prec);
            if (!(W > 0.0)) {
                mode = MODE_FALLBACK;
                st |= ST_ZERO_RESIDUAL;
                W = 0.0;
                for (long long v = lane; v < V; v += 32) W += weight(v);
                for (int off = 16; off > 0; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
            }
        }
        if (!(st & ST_ERRMASK)) {
            const double target = static_cast<double>(uj) * W;
            double acc = 0.0;
            int lastpos = -1;
            for (long long v0 = 0; v0 < V && token < 0; v0 += 32) {
                const long long v = v0 + lane;
                const double w = v < V ? weight(v) : 0.0;
                double incl = w;
                for (int off = 1; off < 32; off <<= 1) {
                    const double o = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += o;
                }
                const unsigned pos = __ballot_sync(0xffffffffu, w > 0.0);
                if (pos) lastpos = static_cast<int>(v0 + 31 - __clz(pos));
                const unsigned hit = __ballot_sync(0xffffffffu, w > 0.0 && target < acc + incl);
                if (hit) token = static_cast<int>(v0 + __ffs(hit) - 1);
                acc += __shfl_sync(0xffffffffu, incl, 31);
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
