// verify_cluster.cuh -- split-vocabulary verify kernel: one thread-block
// cluster of C CTAs per sequence, each CTA owning a contiguous V-slice of
// all k+1 positions.
//
// Pass 1 streams the CTA's slice of every position once through a ring of
// shared-memory tiles filled by 1-D bulk (TMA) copies and keeps, per
// position, an online maximum and sum of exp((l - max) / T) (sampled rows) or
// the maximum and its lowest index (greedy rows).  The per-CTA partials meet
// over distributed shared memory after a cluster barrier; every CTA then
// evaluates the accept tests and the first rejection with one warp ballot,
// identically.  Pass 2 revisits only the stop position j: it builds residual
// weights max(0, p_j - q_j) (or the bonus weights p_k) chunk by chunk, the
// CTA totals meet again over distributed shared memory, and the CTA whose
// slice holds u * W finds the token with a block-wide prefix scan.
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
#include <cstdint>

#include "exp2dd.cuh"
#include "ptx.cuh"

namespace specv {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kTileBytes = 8192;
constexpr int kStages = 4;
constexpr int kMaxK = 31;          // positions 0..k fit one warp
constexpr int kMaxSlice = 16384;   // elements of one position held by one CTA
constexpr int kChunk = 8;          // pass-2 elements per chunk
constexpr int kMaxChunks = kMaxSlice / kChunk;
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

struct ClusterSmem {
    Partial wpart[kWarps][kMaxK + 1];
    Partial part[kMaxK + 1];
    int tstart[kMaxK + 2];      // first tile of each position
    int head[kMaxK + 1];        // unaligned leading elements of each position's slice
    int nbytes[kMaxK + 1];      // bytes of the 16-byte aligned interior
    unsigned long long mbar[kStages];
    double tot[4];              // pass-2 CTA totals: weights, sum of e, q over positive residuals, bad-q flag
    double thr_w[kThreads];     // per-thread pass-2 sums (contiguous chunk blocks)
    double thr_q[kThreads];
    float2 exp2tab[128];
    // row decisions, broadcast to the block
    int j, status, mode, owner, last_pos;
    float Mj, sj, thr;
    float c_hi, c_lo;
    double s_prec, delta, t_local;
};

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
    // NaN sums stay NaN through the products above
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

// One element of the online softmax (used for the unaligned head/tail).
__device__ __forceinline__ void online_add(float& m, float& s, float l, float c) {
    if (l > m) {
        s = (m == -INFINITY) ? 0.0f : s * ex2((m - l) * c);
        m = l;
    }
    if (m != -INFINITY || l != l) s += ex2((l - m) * c);
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads) verify_cluster_kernel(const VerifyArgs a) {
    extern __shared__ __align__(128) unsigned char dyn_smem[];
    __shared__ ClusterSmem sh;
    constexpr int esz = BF16 ? 2 : 4;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
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
        const int nb = ((n - h) * esz) & ~15;
        sh.head[tid] = h;
        sh.nbytes[tid] = nb;
    }
    if (tid < 128) sh.exp2tab[tid] = g_exp2_table[tid];
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sh.mbar[s]), 1);
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
    const int total_tiles = t_ok ? sh.tstart[k + 1] : 0;

    auto issue = [&](int tt) {
        int i = 0;
        while (sh.tstart[i + 1] <= tt) ++i;
        const int off = (tt - sh.tstart[i]) * kTileBytes;
        const int bytes = min(kTileBytes, sh.nbytes[i] - off);
        const long long e0 = (static_cast<long long>(b) * (k + 1) + i) * V + v0 + sh.head[i];
        const int slot = tt % kStages;
        const uint32_t bar = smem_u32(&sh.mbar[slot]);
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(bytes));
        bulk_g2s(smem_u32(ring + slot * kTileBytes), lg + e0 * esz + off, static_cast<uint32_t>(bytes), bar);
    };

    int issued = 0;
    if (tid == 0) {
        for (; issued < min(kStages, total_tiles); ++issued) issue(issued);
    }
    // dependent scalar loads of the accept test (x_i has landed by now)
    if (warp == 0 && lane < k && t_ok && !greedy && xi >= 0 && xi < V) {
        const long long row = static_cast<long long>(b) * (k + 1) + lane;
        Lx = load_logit(a.logits, row * V + xi, BF16);
        qx = __ldg(a.q + (static_cast<long long>(b) * k + lane) * V + xi);
    }

    // ---------------------------------------------------------------- pass 1
    bool timed_out = false;
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

        for (int lt = 0; lt < ntiles; ++lt, ++t) {
            const int slot = t % kStages;
            const uint32_t phase = (t / kStages) & 1;
            const bool ok = timed_out ? false : mbar_wait_bounded(smem_u32(&sh.mbar[slot]), phase, kWaitPolls);
            const int bytes = min(kTileBytes, sh.nbytes[i] - lt * kTileBytes);
            const int nch = bytes >> 4;
            const uint32_t tile = smem_u32(ring + slot * kTileBytes);
            if (ok) {
                constexpr int kPer = kTileBytes / 16 / kThreads;  // 16-byte chunks per thread
                uint4 w[kPer];
#pragma unroll
                for (int r = 0; r < kPer; ++r) {
                    const int ch = tid + r * kThreads;
                    if (ch < nch) {
                        w[r] = ld_shared_v4(tile + ch * 16);
                    } else if (BF16) {
                        w[r] = make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
                    } else {
                        const uint32_t ni = __float_as_uint(-INFINITY);
                        w[r] = make_uint4(ni, ni, ni, ni);
                    }
                }
                // tile maximum of this thread's elements
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
                            const int ch = tid + r * kThreads;
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
                        s = (m == -INFINITY) ? 0.0f : s * ex2((m - lmax) * c);
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
                                const f2 d = mul2(sub2(pack2(__uint_as_float(ws[q4]), __uint_as_float(ws[q4 + 1])), mm), cc);
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
            // the slot is free once every thread is past it; a timeout
            // anywhere in the block stops the stream for the whole block
            if (__syncthreads_or(!ok)) timed_out = true;
            if (tid == 0 && !timed_out && issued < total_tiles) issue(issued++);
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
    if (timed_out && tid == 0) {
        // let the copies still in flight (at most one per stage) land before
        // the buffers are reused or the block exits
        for (int tt = max(0, issued - kStages); tt < issued; ++tt)
            mbar_wait_bounded(smem_u32(&sh.mbar[tt % kStages]), (tt / kStages) & 1, kWaitPolls);
    }
    __syncthreads();
    if (tid <= k && t_ok) {
        Partial p = sh.wpart[0][tid];
        for (int w = 1; w < kWarps; ++w) {
            const Partial o = sh.wpart[w][tid];
            if (greedy) {
                merge_arg(p.m, p.arg, o.m, o.arg);
                p.flags |= o.flags;
            } else {
                merge_ms(p.m, p.s, o.m, o.s, c);
            }
        }
        if (timed_out) p.flags |= 2;
        sh.part[tid] = p;
    }
    cluster_sync();  // #1: every CTA's partials are visible

    // ---------------------------------------------------------------- decisions
    if (warp == 0) {
        float M = -INFINITY, S = 0.0f;
        int A = 0x7fffffff, flags = 0;
        if (lane <= k && t_ok) {
            const uint32_t local = smem_u32(&sh.part[lane]);
            for (uint32_t r = 0; r < C; ++r) {
                const uint32_t ra = map_rank(local, r);
                const float m2 = ld_cluster_f32(ra);
                const float s2 = ld_cluster_f32(ra + 4);
                const int a2 = ld_cluster_s32(ra + 8);
                flags |= ld_cluster_s32(ra + 12);
                if (greedy)
                    merge_arg(M, A, m2, a2);
                else
                    merge_ms(M, S, m2, s2, c);
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
                        const double cd = 1.4426950408889634 / static_cast<double>(T);
                        const float ch = static_cast<float>(cd);
                        const float cl = static_cast<float>(cd - static_cast<double>(ch));
                        if (Lx != -INFINITY) {
                            float dh = Lx - M, dl = 0.0f;
                            if (!BF16) two_sum(Lx, -M, dh, dl);  // fp32 logits: keep the rounding error
                            const float xh = dh * ch;
                            const float xl = fmaf(dh, cl, fmaf(dh, ch, -xh)) + dl * ch;
                            const float2 e = exp2dd(xh, xl, sh.exp2tab);
                            p = (e.x + e.y) / S;
                        }
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
        if (lane == 0) {
            sh.j = j;
            sh.status = st;
            sh.Mj = Mj;
            sh.sj = Sj;
            sh.mode = (j < k) ? MODE_RESIDUAL : MODE_BONUS;
        }
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
        if (lane <= k) {
            // keep the draft tokens for whoever writes the sampled outputs
            sh.wpart[0][lane].arg = xi;
        }
    }
    __syncthreads();
    const bool sample = t_ok && !greedy && !(sh.status & ST_ERRMASK);
    if (!sample) {
        cluster_sync();  // no CTA leaves while a peer may still read its partials
        return;
    }

    // ---------------------------------------------------------------- pass 2
    if (tid == 0) {
        const double cd = 1.4426950408889634 / static_cast<double>(T);
        sh.c_hi = static_cast<float>(cd);
        sh.c_lo = static_cast<float>(cd - static_cast<double>(sh.c_hi));
        sh.thr = kLargeP * sh.sj;
        sh.last_pos = -1;
    }
    __syncthreads();
    const int j = sh.j;
    const float Mj = sh.Mj, sj = sh.sj, thr = sh.thr, ch = sh.c_hi, cl = sh.c_lo;
    const long long lrow = (static_cast<long long>(b) * (k + 1) + j) * V;
    const float* qrow = a.q + (static_cast<long long>(b) * k + (j < k ? j : 0)) * V;
    const int nch = (n + kChunk - 1) / kChunk;
    float* ch_hi = reinterpret_cast<float*>(ring);
    float* ch_lo = ch_hi + kMaxChunks;
    float* ch_q = ch_lo + kMaxChunks;
    int mode = sh.mode;

    // weights of one chunk: returns its (hi, lo) and its q sum over positive
    // residuals; adds e to the thread's (eh, el) sum (residual mode)
    auto chunk_weights = [&](int cidx, int md, float& whi, float& wlo, float& wq, float& teh, float& tel,
                             bool& qbad) {
        const long long e0 = v0 + static_cast<long long>(cidx) * kChunk;
        const int cnt = min(kChunk, n - cidx * kChunk);
        float lv[kChunk], qv[kChunk];
        const unsigned char* lp = lg + (lrow + e0) * esz;
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
            for (int e = 0; e < kChunk; ++e) lv[e] = e < cnt ? load_logit(a.logits, lrow + e0 + e, BF16) : -INFINITY;
        }
        if (md == MODE_RESIDUAL) {
            const float* qp = qrow + e0;
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
#pragma unroll
            for (int e = 0; e < kChunk; ++e) qbad |= !(qv[e] >= 0.0f && qv[e] <= FLT_MAX);
        }
        float rs = 0.0f, qs = 0.0f, es = 0.0f;
        float lh = 0.0f, ll = 0.0f;
#pragma unroll
        for (int e = 0; e < kChunk; ++e) {
            const float l = lv[e];
            if (e >= cnt || l == -INFINITY) continue;  // masked entries weigh nothing
            const float dh = l - Mj;
            const float xh = dh * ch;
            float xl = fmaf(dh, cl, fmaf(dh, ch, -xh));
            float ef = ex2(xh);
            ef = fmaf(ef, xl * kLn2, ef);
            if (ef > thr) {
                if (!BF16) {
                    float d2, dl;
                    two_sum(l, -Mj, d2, dl);
                    xl = fmaf(dl, ch, xl);
                }
                const float2 ed = exp2dd(xh, xl, sh.exp2tab);
                if (md == MODE_RESIDUAL) {
                    const float qq = qv[e];
                    const float ph = sj * qq;
                    const float pl = fmaf(sj, qq, -ph);
                    float rh, rl;
                    two_sum(ed.x, -ph, rh, rl);
                    rl = rl + (ed.y - pl);
                    if (rh + rl > 0.0f) {
                        df_add(lh, ll, rh, rl);
                        qs += qq;
                    }
                    df_add(teh, tel, ed.x, ed.y);
                } else {
                    df_add(lh, ll, ed.x, ed.y);
                }
            } else {
                if (md == MODE_RESIDUAL) {
                    const float r = fmaf(-sj, qv[e], ef);
                    if (r > 0.0f) {
                        rs += r;
                        qs += qv[e];
                    }
                    es += ef;
                } else {
                    rs += ef;
                }
            }
        }
        float hi, lo;
        two_sum(rs, lh, hi, lo);
        whi = hi;
        wlo = lo + ll;
        wq = qs;
        if (md == MODE_RESIDUAL) df_add(teh, tel, es, 0.0f);
    };

    for (;;) {
        // sweep: chunk weights of this CTA's slice of row j
        float teh = 0.0f, tel = 0.0f;
        bool qbad = false;
        for (int cidx = tid; cidx < nch; cidx += kThreads) {
            float whi, wlo, wq;
            chunk_weights(cidx, mode, whi, wlo, wq, teh, tel, qbad);
            ch_hi[cidx] = whi;
            ch_lo[cidx] = wlo;
            ch_q[cidx] = wq;
        }
        __syncthreads();
        // per-thread sums over contiguous chunk blocks (vocabulary order)
        const int cpt = (nch + kThreads - 1) / kThreads;
        const int c_begin = min(nch, tid * cpt), c_end = min(nch, c_begin + cpt);
        float sh_hi = 0.0f, sh_lo = 0.0f, sq = 0.0f;
        for (int cc = c_begin; cc < c_end; ++cc) {
            df_add(sh_hi, sh_lo, ch_hi[cc], ch_lo[cc]);
            sq += ch_q[cc];
        }
        double w_d = static_cast<double>(sh_hi) + static_cast<double>(sh_lo);
        double q_d = static_cast<double>(sq);
        double e_d = static_cast<double>(teh) + static_cast<double>(tel);
        sh.thr_w[tid] = w_d;
        sh.thr_q[tid] = q_d;
        for (int off = 16; off > 0; off >>= 1) {
            w_d += __shfl_xor_sync(0xffffffffu, w_d, off);
            q_d += __shfl_xor_sync(0xffffffffu, q_d, off);
            e_d += __shfl_xor_sync(0xffffffffu, e_d, off);
        }
        __shared__ double wsum[kWarps][3];
        const int any_qbad = __syncthreads_or(qbad ? 1 : 0);
        if (lane == 0) {
            wsum[warp][0] = w_d;
            wsum[warp][1] = e_d;
            wsum[warp][2] = q_d;
        }
        __syncthreads();
        if (tid == 0) {
            double t0 = 0.0, t1 = 0.0, t2 = 0.0;
            for (int w = 0; w < kWarps; ++w) {
                t0 += wsum[w][0];
                t1 += wsum[w][1];
                t2 += wsum[w][2];
            }
            sh.tot[0] = t0;
            sh.tot[1] = t1;
            sh.tot[2] = t2;
            sh.tot[3] = any_qbad ? 1.0 : 0.0;
        }
        cluster_sync();  // #2: CTA totals visible
        if (tid == 0) {
            const uint32_t local = smem_u32(&sh.tot[0]);
            double wr[16], qr[16];
            double s_prec = 0.0, qflag = 0.0;
            for (uint32_t r = 0; r < C; ++r) {
                const uint32_t ra = map_rank(local, r);
                wr[r] = ld_cluster_f64(ra);
                s_prec += ld_cluster_f64(ra + 8);
                qr[r] = ld_cluster_f64(ra + 16);
                qflag += ld_cluster_f64(ra + 24);
            }
            double delta = 0.0;
            if (mode == MODE_RESIDUAL) delta = s_prec - static_cast<double>(sj);
            double W = 0.0;
            for (uint32_t r = 0; r < C; ++r) {
                wr[r] -= delta * qr[r];
                W += wr[r];
            }
            sh.delta = delta;
            sh.s_prec = (mode == MODE_RESIDUAL) ? s_prec : 0.0;
            if (mode == MODE_RESIDUAL && qflag > 0.0) {
                // a draft probability of the residual row is NaN, negative or infinite
                sh.owner = -2;
                if (rank == 0) {
                    for (int i = 0; i <= k; ++i) a.out_tokens[static_cast<long long>(b) * (k + 1) + i] = -1;
                    a.num_accepted[b] = 0;
                    if (a.row_status) a.row_status[b] = sh.status | ST_QBAD;
                }
            } else if (mode == MODE_RESIDUAL && !(W > 0.0)) {
                sh.mode = MODE_FALLBACK;
                sh.owner = -1;
            } else {
                const float uj = a.u[(static_cast<long long>(b) * (k + 1) + j) * 2 + 1];
                const double target = static_cast<double>(uj) * W;
                double pre = 0.0;
                int owner = -1, last = -1;
                for (uint32_t r = 0; r < C; ++r) {
                    if (wr[r] > 0.0) last = static_cast<int>(r);
                    if (owner < 0 && target < pre + wr[r]) {
                        owner = static_cast<int>(r);
                        sh.t_local = target - pre;
                    }
                    if (owner < 0) pre += wr[r];
                }
                if (owner < 0) {
                    owner = last;
                    sh.t_local = INFINITY;
                }
                sh.owner = owner;
                if (rank == 0 && a.dbg_resid && mode == MODE_RESIDUAL) a.dbg_resid[b] = static_cast<float>(W / s_prec);
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
    if (static_cast<int>(rank) == sh.owner) {
        const double delta = sh.delta;
        const double tl = sh.t_local;
        // inclusive scan of the corrected per-thread sums (fixed order)
        double wt = sh.thr_w[tid] - delta * sh.thr_q[tid];
        double incl = wt;
        for (int off = 1; off < 32; off <<= 1) {
            const double o = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += o;
        }
        __shared__ double wtot[kWarps];
        if (lane == 31) wtot[warp] = incl;
        __syncthreads();
        double before_warp = 0.0;
        for (int w = 0; w < warp; ++w) before_warp += wtot[w];
        incl += before_warp;
        const double excl = incl - wt;
        if (wt > 0.0) atomicMax(&sh.last_pos, tid);
        __syncthreads();
        bool mine = (wt > 0.0) && (tl >= excl) && (tl < incl);
        // no thread holds the target only through rounding at the top edge:
        // the last thread with positive weight takes it
        const int owner_found = __syncthreads_or(mine ? 1 : 0);
        if (!owner_found && tid == sh.last_pos) mine = true;
        if (mine) {
            const int cpt = (nch + kThreads - 1) / kThreads;
            const int c_begin = min(nch, tid * cpt), c_end = min(nch, c_begin + cpt);
            double acc = excl;
            int cstar = -1, clast = -1;
            for (int cc = c_begin; cc < c_end; ++cc) {
                const double w = static_cast<double>(ch_hi[cc]) + static_cast<double>(ch_lo[cc]) -
                                 delta * static_cast<double>(ch_q[cc]);
                if (w > 0.0) clast = cc;
                if (tl < acc + w) {
                    cstar = cc;
                    break;
                }
                acc += w;
            }
            if (cstar < 0) {
                cstar = clast >= 0 ? clast : c_begin;
                acc = -INFINITY;  // take the chunk's last positive element
            }
            // exact walk through the chunk's entries
            const long long e0 = v0 + static_cast<long long>(cstar) * kChunk;
            const int cnt = min(kChunk, n - cstar * kChunk);
            int token = -1, lastpos = -1;
            for (int e = 0; e < cnt; ++e) {
                const float l = load_logit(a.logits, lrow + e0 + e, BF16);
                if (l == -INFINITY) continue;
                float dh = l - Mj, dl = 0.0f;
                if (!BF16) two_sum(l, -Mj, dh, dl);
                const float xh = dh * ch;
                const float xl = fmaf(dl, ch, fmaf(dh, cl, fmaf(dh, ch, -xh)));
                const float2 ed = exp2dd(xh, xl, sh.exp2tab);
                double w = static_cast<double>(ed.x) + static_cast<double>(ed.y);
                if (mode == MODE_RESIDUAL) {
                    w -= sh.s_prec * static_cast<double>(__ldg(qrow + e0 + e));
                    if (w < 0.0) w = 0.0;
                }
                if (w > 0.0) lastpos = static_cast<int>(e0 + e);
                acc += w;
                if (token < 0 && w > 0.0 && tl < acc) token = static_cast<int>(e0 + e);
            }
            if (token < 0) token = lastpos;
            int st = sh.status;
            if (mode == MODE_FALLBACK) st |= ST_ZERO_RESIDUAL;
            for (int i = 0; i <= k; ++i) {
                int tok = -1;
                if (i < j)
                    tok = sh.wpart[0][i].arg;
                else if (i == j)
                    tok = token;
                a.out_tokens[static_cast<long long>(b) * (k + 1) + i] = tok;
            }
            a.num_accepted[b] = j;
            if (a.row_status) a.row_status[b] = st;
        }
    }
    cluster_sync();  // #3: no CTA leaves while a peer may still read its totals
}

}  // namespace specv
