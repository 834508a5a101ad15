// specv.cu -- C ABI of the verify step: argument checks, launch planning
// (small-vocabulary warp kernel or split-vocabulary cluster kernel) and the
// host-buffer convenience call.  The kernels live in verify_cluster.cuh and
// verify_warp.cuh.
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "../../include/specv.h"
#include "verify_cluster.cuh"
#include "verify_warp.cuh"
#include "rollback.cuh"
#include "verify_topk.cuh"
#include "verify_topk_wide.cuh"

using namespace specv;

struct specv_ctx {
    int device = 0;
    int sm_count = 0;
    int max_batch = 0;
    int max_k = 0;
    int64_t vocab = 0;
    std::atomic<int64_t> launches{0};
    // most clusters of each size (1..16) that can be resident at once, per
    // logits type (index 0: fp32, 1: bf16); 0 if that size cannot launch
    int max_clusters[2][17] = {};
    // device staging for specv_verify_sample_host
    void* stage = nullptr;
    size_t stage_bytes = 0;
    // one-shot test hook: the next cluster-kernel launch withholds one
    // pass-1 stage of CTA 0 and waits at most `test_polls` polls
    int test_withhold = -1;
    uint32_t test_polls = 0;
};

static thread_local char g_last_error[256] = "";

static specv_status cuda_fail(cudaError_t e, const char* what) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", what, cudaGetErrorString(e));
    return SPECV_ERR_CUDA;
}

#define SPECV_CUDA(call)                                         \
    do {                                                         \
        cudaError_t e_ = (call);                                 \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call);      \
    } while (0)

namespace {

struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) == cudaSuccess) ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};


struct Plan {
    bool warp = false;  // V <= kWarpKernelMaxV: one warp per row, or (row) one CTA per row
    bool row = false;
    int cluster = 1;
    int slice = 0;
};

Plan make_plan(const specv_ctx* h, specv_dtype dt, int batch, int64_t V) {
    Plan p;
    if (V <= kWarpKernelMaxV) {
        // a CTA per row while the batch leaves SMs idle (its positions and
        // its stop row are then worked on in parallel), else a warp per row
        p.warp = true;
        p.row = batch <= 2 * h->sm_count;
        if (const char* env = getenv("SPECV_SMALLV")) {
            if (!strcmp(env, "row")) p.row = true;
            if (!strcmp(env, "warp")) p.row = false;
        }
        return p;
    }
    const int cmin = static_cast<int>((V + kMaxSlice - 1) / kMaxSlice);
    // the widest split whose clusters are all resident at once; if the batch
    // does not fit in one wave at any size, the narrowest split
    int C = cmin;
    const int* mc = h->max_clusters[dt == SPECV_BF16 ? 1 : 0];
    for (int c = 16; c >= cmin; --c) {
        if (mc[c] >= batch) {
            C = c;
            break;
        }
    }
    if (const char* env = getenv("SPECV_CLUSTER")) {
        const int forced = atoi(env);
        if (forced >= cmin && forced <= 16) C = forced;
    }
    int64_t slice = (V + C - 1) / C;
    slice = (slice + 63) / 64 * 64;
    if (slice > kMaxSlice) slice = kMaxSlice;
    p.cluster = static_cast<int>((V + slice - 1) / slice);
    p.slice = static_cast<int>(slice);
    return p;
}

template <bool BF16>
cudaError_t launch_cluster(const VerifyArgs& a, const Plan& p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.B) * p.cluster, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = cluster_dyn_smem(p.cluster, a.pk);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, verify_cluster_kernel<BF16>, a);
}

template <bool BF16>
cudaError_t launch_warp(const VerifyArgs& a, bool row, cudaStream_t stream) {
    if (row) {
        verify_row_kernel<BF16><<<static_cast<unsigned>(a.B), kRowThreads, 0, stream>>>(a);
    } else {
        const unsigned blocks = static_cast<unsigned>((a.B + kWarpsPerBlock - 1) / kWarpsPerBlock);
        verify_warp_kernel<BF16><<<blocks, 32 * kWarpsPerBlock, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

template <bool BF16>
void query_clusters(int* out, int pk) {
    for (int c = 1; c <= 16; ++c) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(c) * 256, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = cluster_dyn_smem(c, pk);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = c;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, verify_cluster_kernel<BF16>, &cfg) != cudaSuccess) {
            n = 0;
            cudaGetLastError();
        }
        out[c] = n;
    }
}

template <bool BF16>
cudaError_t set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(verify_cluster_kernel<BF16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(verify_topk_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(topk_dyn_smem(kMaxK)));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(verify_topk_wide_kernel<BF16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(verify_topk_wide_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(wide_dyn_smem(kMaxK, 262144)));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(verify_cluster_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(cluster_dyn_smem(16, kMaxK + 1)));
}

specv_status check_sizes(const specv_ctx* h, specv_dtype dt, int batch, int k, int64_t V) {
    if (!h) return SPECV_ERR_INVALID_ARGUMENT;
    if (dt != SPECV_F32 && dt != SPECV_BF16) return SPECV_ERR_INVALID_ARGUMENT;
    if (batch < 0 || batch > h->max_batch) return SPECV_ERR_INVALID_ARGUMENT;
    if (k < 1 || k > h->max_k) return SPECV_ERR_INVALID_ARGUMENT;
    if (V < 1 || V > h->vocab) return SPECV_ERR_INVALID_ARGUMENT;
    return SPECV_OK;
}

specv_status run(specv_ctx* h, specv_dtype dt, const VerifyArgs& a, void* stream) {
    if (a.B == 0) return SPECV_OK;
    DeviceGuard g(h->device);
    if (!g.ok) return cuda_fail(cudaErrorInvalidDevice, "cudaSetDevice");
    const Plan p = make_plan(h, dt, a.B, a.V);
    VerifyArgs args = a;
    args.slice = p.slice;
    args.pk = h->max_k + 1;
    if (!p.warp && h->test_withhold >= 0) {  // the test hook arms one launch
        args.withhold = h->test_withhold;
        args.polls = h->test_polls;
        h->test_withhold = -1;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (p.warp)
        e = dt == SPECV_BF16 ? launch_warp<true>(args, p.row, s) : launch_warp<false>(args, p.row, s);
    else
        e = dt == SPECV_BF16 ? launch_cluster<true>(args, p, s) : launch_cluster<false>(args, p, s);
    if (e != cudaSuccess) return cuda_fail(e, "verify kernel launch");
    h->launches.fetch_add(1, std::memory_order_relaxed);
    return SPECV_OK;
}

}  // namespace

extern "C" {

specv_status specv_create(specv_handle* out, int device, int max_batch, int max_k, int64_t vocab) {
    if (!out) return SPECV_ERR_INVALID_ARGUMENT;
    *out = nullptr;
    if (max_batch < 0 || max_k < 1 || max_k > kMaxK || vocab < 1 || vocab > (int64_t)kMaxSlice * 16)
        return SPECV_ERR_INVALID_ARGUMENT;
    int ndev = 0;
    SPECV_CUDA(cudaGetDeviceCount(&ndev));
    if (device < 0 || device >= ndev) return SPECV_ERR_INVALID_ARGUMENT;
    cudaDeviceProp prop;
    SPECV_CUDA(cudaGetDeviceProperties(&prop, device));
    if (prop.major != 10 || prop.minor != 3) {
        snprintf(g_last_error, sizeof g_last_error, "device %d is sm_%d%d, this library is built for sm_103a",
                 device, prop.major, prop.minor);
        return SPECV_ERR_UNSUPPORTED;
    }
    DeviceGuard g(device);
    if (!g.ok) return cuda_fail(cudaErrorInvalidDevice, "cudaSetDevice");
    float2 tab[128];
    for (int j = 0; j < 128; ++j) {
        const double v = std::exp2(j / 128.0);
        tab[j].x = static_cast<float>(v);
        tab[j].y = static_cast<float>(v - static_cast<double>(tab[j].x));
    }
    SPECV_CUDA(cudaMemcpyToSymbol(g_exp2_table, tab, sizeof tab));
    {
        cudaError_t e = set_attributes<true>();
        if (e == cudaSuccess) e = set_attributes<false>();
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    }
    specv_ctx* h = new (std::nothrow) specv_ctx();
    if (!h) return SPECV_ERR_CUDA;
    h->device = device;
    h->sm_count = prop.multiProcessorCount;
    h->max_batch = max_batch;
    h->max_k = max_k;
    h->vocab = vocab;
    query_clusters<false>(h->max_clusters[0], max_k + 1);
    query_clusters<true>(h->max_clusters[1], max_k + 1);
    *out = h;
    return SPECV_OK;
}

static specv_status verify_sample(specv_handle h, specv_dtype logits_dtype, const void* target_logits,
                                  const float* draft_probs, const int32_t* draft_tokens, const float* uniforms,
                                  const float* temperature, int batch, int k, int64_t V, int32_t* num_accepted,
                                  int32_t* out_tokens, int32_t* row_status, const specv_debug* dbg, void* stream,
                                  bool q_host) {
    specv_status st = check_sizes(h, logits_dtype, batch, k, V);
    if (st != SPECV_OK) return st;
    if (batch > 0 && (!target_logits || !draft_tokens || !uniforms || !temperature ||
                      !num_accepted || !out_tokens))
        return SPECV_ERR_INVALID_ARGUMENT;
    VerifyArgs a = {};
    a.logits = target_logits;
    a.q = draft_probs;
    a.x = draft_tokens;
    a.u = uniforms;
    a.temp = temperature;
    a.num_accepted = num_accepted;
    a.out_tokens = out_tokens;
    a.row_status = row_status;
    if (dbg) {
        a.dbg_p = dbg->p_at_draft;
        a.dbg_q = dbg->q_at_draft;
        a.dbg_max = dbg->row_max;
        a.dbg_sumexp = dbg->row_sumexp;
        a.dbg_resid = dbg->residual_mass;
    }
    a.V = V;
    a.B = batch;
    a.k = k;
    a.q_host = q_host ? 1 : 0;
    return run(h, logits_dtype, a, stream);
}

specv_status specv_verify_sample(specv_handle h, specv_dtype logits_dtype, const void* target_logits,
                                 const float* draft_probs, const int32_t* draft_tokens, const float* uniforms,
                                 const float* temperature, int batch, int k, int64_t V, int32_t* num_accepted,
                                 int32_t* out_tokens, int32_t* row_status, const specv_debug* dbg, void* stream) {
    return verify_sample(h, logits_dtype, target_logits, draft_probs, draft_tokens, uniforms, temperature, batch, k,
                         V, num_accepted, out_tokens, row_status, dbg, stream, false);
}

specv_status specv_verify_greedy(specv_handle h, specv_dtype logits_dtype, const void* target_logits,
                                 const int32_t* draft_tokens, int batch, int k, int64_t V, int32_t* num_accepted,
                                 int32_t* out_tokens, int32_t* row_status, void* stream) {
    specv_status st = check_sizes(h, logits_dtype, batch, k, V);
    if (st != SPECV_OK) return st;
    if (batch > 0 && (!target_logits || !draft_tokens || !num_accepted || !out_tokens))
        return SPECV_ERR_INVALID_ARGUMENT;
    VerifyArgs a = {};
    a.logits = target_logits;
    a.x = draft_tokens;
    a.num_accepted = num_accepted;
    a.out_tokens = out_tokens;
    a.row_status = row_status;
    a.V = V;
    a.B = batch;
    a.k = k;
    return run(h, logits_dtype, a, stream);
}

specv_status specv_verify_sample_filtered(specv_handle h, specv_dtype logits_dtype, const void* target_logits,
                                          const float* draft_probs, const int32_t* draft_tokens, const float* uniforms,
                                          const float* temperature, const int32_t* top_k, const float* top_p,
                                          int batch, int k, int64_t V, int32_t* num_accepted, int32_t* out_tokens,
                                          int32_t* row_status, void* stream) {
    specv_status st = check_sizes(h, logits_dtype, batch, k, V);
    if (st != SPECV_OK) return st;
    if (batch > 0 && (!target_logits || !draft_tokens || !uniforms || !temperature || !top_k || !top_p ||
                      !num_accepted || !out_tokens))
        return SPECV_ERR_INVALID_ARGUMENT;
    if (batch == 0) return SPECV_OK;
    DeviceGuard g(h->device);
    if (!g.ok) return cuda_fail(cudaErrorInvalidDevice, "cudaSetDevice");
    // draft_probs may be page-locked host memory: the kernel reads the few
    // entries it needs in place (plain loads); pageable host memory is refused
    const float* q = draft_probs;
    if (q) {
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, q) != cudaSuccess) {
            cudaGetLastError();
            return SPECV_ERR_INVALID_ARGUMENT;
        }
        if (pa.type == cudaMemoryTypeUnregistered) return SPECV_ERR_INVALID_ARGUMENT;
        if (pa.type == cudaMemoryTypeHost) {
            if (!pa.devicePointer) return SPECV_ERR_INVALID_ARGUMENT;
            q = static_cast<const float*>(pa.devicePointer);
        }
    }
    VerifyArgs a = {};
    a.logits = target_logits;
    a.q = q;
    a.x = draft_tokens;
    a.u = uniforms;
    a.temp = temperature;
    a.top_k = top_k;
    a.top_p = top_p;
    a.num_accepted = num_accepted;
    a.out_tokens = out_tokens;
    a.row_status = row_status;
    a.V = V;
    a.B = batch;
    a.k = k;
    const int C = topk_cluster(k);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(batch) * C, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = topk_dyn_smem(k);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = logits_dtype == SPECV_BF16 ? cudaLaunchKernelEx(&cfg, verify_topk_kernel<true>, a)
                                               : cudaLaunchKernelEx(&cfg, verify_topk_kernel<false>, a);
    if (e != cudaSuccess) return cuda_fail(e, "verify_topk launch");
    h->launches.fetch_add(1, std::memory_order_relaxed);
    // Rows with top_k above 64 go to the wide kernel, rows up to 64 (and
    // greedy or refused rows) to the one above: each kernel leaves the
    // other's rows untouched, so the two launches share nothing but the
    // stream.  top_k is on the device, so both are always launched.
    const int Cw = wide_cluster(k);
    cfg.gridDim = dim3(static_cast<unsigned>(batch) * Cw, 1, 1);
    cfg.blockDim = dim3(kWideThreads, 1, 1);
    cfg.dynamicSmemBytes = wide_dyn_smem(k, V);
    attr[0].val.clusterDim.x = static_cast<unsigned>(Cw);
    e = logits_dtype == SPECV_BF16 ? cudaLaunchKernelEx(&cfg, verify_topk_wide_kernel<true>, a)
                                   : cudaLaunchKernelEx(&cfg, verify_topk_wide_kernel<false>, a);
    if (e != cudaSuccess) return cuda_fail(e, "verify_topk_wide launch");
    h->launches.fetch_add(1, std::memory_order_relaxed);
    return SPECV_OK;
}

specv_status specv_verify_tree_greedy(specv_handle h, specv_dtype logits_dtype, const void* target_logits,
                                      const int32_t* tokens, const int32_t* parents, int batch, int M, int64_t V,
                                      int32_t* num_accepted, int32_t* out_tokens, int32_t* path,
                                      int32_t* row_status, void* stream) {
    specv_status st = check_sizes(h, logits_dtype, batch, M, V);
    if (st != SPECV_OK) return st;
    if (batch > 0 && (!target_logits || !tokens || !parents || !num_accepted || !out_tokens))
        return SPECV_ERR_INVALID_ARGUMENT;
    VerifyArgs a = {};
    a.logits = target_logits;
    a.x = tokens;
    a.parents = parents;
    a.path = path;
    a.num_accepted = num_accepted;
    a.out_tokens = out_tokens;
    a.row_status = row_status;
    a.V = V;
    a.B = batch;
    a.k = M;
    return run(h, logits_dtype, a, stream);
}

specv_status specv_verify_sample_host(specv_handle h, specv_dtype logits_dtype, const void* target_logits,
                                      const float* draft_probs, const int32_t* draft_tokens,
                                      const float* uniforms, const float* temperature, int batch, int k,
                                      int64_t V, int32_t* num_accepted, int32_t* out_tokens,
                                      int32_t* row_status, void* stream) {
    specv_status st = check_sizes(h, logits_dtype, batch, k, V);
    if (st != SPECV_OK) return st;
    if (batch == 0) return SPECV_OK;
    if (!target_logits || !draft_tokens || !uniforms || !temperature || !num_accepted || !out_tokens)
        return SPECV_ERR_INVALID_ARGUMENT;
    const size_t esz = logits_dtype == SPECV_BF16 ? 2 : 4;
    const size_t B = static_cast<size_t>(batch), K = static_cast<size_t>(k), VV = static_cast<size_t>(V);
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t nL = B * (K + 1) * VV * esz, nQ = B * K * VV * 4, nX = B * K * 4, nU = B * (K + 1) * 2 * 4,
                 nT = B * 4, nA = B * 4, nO = B * (K + 1) * 4, nS = B * 4;
    // page-locked q is read in place by the kernel: only the entries the rule
    // needs (the draft tokens' and the stop rows') cross the link
    const float* q_mapped = nullptr;
    if (draft_probs) {
        cudaPointerAttributes pa;
        if (cudaPointerGetAttributes(&pa, draft_probs) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
            pa.devicePointer)
            q_mapped = static_cast<const float*>(pa.devicePointer);
        else
            cudaGetLastError();
    }
    const size_t nQc = (draft_probs && !q_mapped) ? nQ : 0;  // one-hot drafts or in-place q: no q to copy
    const size_t need = al(nL) + al(nQc) + al(nX) + al(nU) + al(nT) + al(nA) + al(nO) + al(nS);
    DeviceGuard g(h->device);
    if (!g.ok) return cuda_fail(cudaErrorInvalidDevice, "cudaSetDevice");
    if (h->stage_bytes < need) {
        if (h->stage) cudaFree(h->stage);
        h->stage = nullptr;
        h->stage_bytes = 0;
        SPECV_CUDA(cudaMalloc(&h->stage, need));
        h->stage_bytes = need;
    }
    unsigned char* p = static_cast<unsigned char*>(h->stage);
    unsigned char* dL = p;
    unsigned char* dQ = dL + al(nL);
    unsigned char* dX = dQ + al(nQc);
    unsigned char* dU = dX + al(nX);
    unsigned char* dT = dU + al(nU);
    unsigned char* dA = dT + al(nT);
    unsigned char* dO = dA + al(nA);
    unsigned char* dS = dO + al(nO);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    SPECV_CUDA(cudaMemcpyAsync(dL, target_logits, nL, cudaMemcpyHostToDevice, s));
    if (nQc) SPECV_CUDA(cudaMemcpyAsync(dQ, draft_probs, nQc, cudaMemcpyHostToDevice, s));
    SPECV_CUDA(cudaMemcpyAsync(dX, draft_tokens, nX, cudaMemcpyHostToDevice, s));
    SPECV_CUDA(cudaMemcpyAsync(dU, uniforms, nU, cudaMemcpyHostToDevice, s));
    SPECV_CUDA(cudaMemcpyAsync(dT, temperature, nT, cudaMemcpyHostToDevice, s));
    const float* q_arg = q_mapped ? q_mapped : (draft_probs ? reinterpret_cast<const float*>(dQ) : nullptr);
    st = verify_sample(h, logits_dtype, dL, q_arg, reinterpret_cast<const int32_t*>(dX),
                       reinterpret_cast<const float*>(dU), reinterpret_cast<const float*>(dT), batch, k, V,
                       reinterpret_cast<int32_t*>(dA), reinterpret_cast<int32_t*>(dO), reinterpret_cast<int32_t*>(dS),
                       nullptr, stream, q_mapped != nullptr);
    if (st != SPECV_OK) return st;
    SPECV_CUDA(cudaMemcpyAsync(num_accepted, dA, nA, cudaMemcpyDeviceToHost, s));
    SPECV_CUDA(cudaMemcpyAsync(out_tokens, dO, nO, cudaMemcpyDeviceToHost, s));
    if (row_status) SPECV_CUDA(cudaMemcpyAsync(row_status, dS, nS, cudaMemcpyDeviceToHost, s));
    SPECV_CUDA(cudaStreamSynchronize(s));
    return SPECV_OK;
}

int specv_plan_cluster(specv_handle h, specv_dtype logits_dtype, int batch, int k, int64_t V) {
    if (check_sizes(h, logits_dtype, batch, k, V) != SPECV_OK) return 0;
    const Plan p = make_plan(h, logits_dtype, batch, V);
    return p.warp ? 1 : p.cluster;
}

int64_t specv_launch_count(specv_handle h) { return h ? h->launches.load() : 0; }

void specv_destroy(specv_handle h) {
    if (!h) return;
    if (h->stage) {
        DeviceGuard g(h->device);
        cudaFree(h->stage);
    }
    delete h;
}

specv_status specv_test_withhold_stage(specv_handle h, int stage_use, int polls) {
    if (!h || stage_use < 0 || polls < 1) return SPECV_ERR_INVALID_ARGUMENT;
    h->test_withhold = stage_use;
    h->test_polls = static_cast<uint32_t>(polls);
    return SPECV_OK;
}

const char* specv_status_string(specv_status s) {
    switch (s) {
        case SPECV_OK: return "ok";
        case SPECV_ERR_INVALID_ARGUMENT: return "invalid argument";
        case SPECV_ERR_UNSUPPORTED: return "unsupported device";
        case SPECV_ERR_CUDA: return "CUDA error";
        case SPECV_ERR_TIMEOUT: return "wait timed out";
    }
    return "unknown status";
}

const char* specv_last_cuda_error(void) { return g_last_error; }

specv_status specv_rollback(specv_handle h, const int32_t* num_accepted, int batch, int k, int32_t* seq_lens,
                            int32_t* block_tables, int max_blocks, int32_t* num_blocks, int block_size,
                            int32_t* free_list, int64_t free_capacity, int32_t* free_count, int32_t* row_status,
                            void* stream) {
    // free_count is an int32: a list longer than INT32_MAX entries could not be counted
    if (!h || batch < 0 || k < 0 || k > h->max_k || max_blocks < 0 || block_size < 1 || free_capacity < 0 ||
        free_capacity > INT32_MAX)
        return SPECV_ERR_INVALID_ARGUMENT;
    if (!free_count || (free_capacity > 0 && !free_list)) return SPECV_ERR_INVALID_ARGUMENT;
    if (batch > 0 && (!num_accepted || !seq_lens || !num_blocks || (max_blocks > 0 && !block_tables)))
        return SPECV_ERR_INVALID_ARGUMENT;
    DeviceGuard g(h->device);
    if (!g.ok) return cuda_fail(cudaErrorInvalidDevice, "cudaSetDevice");
    RollbackArgs r;
    r.num_accepted = num_accepted;
    r.seq_lens = seq_lens;
    r.block_tables = block_tables;
    r.num_blocks = num_blocks;
    r.free_list = free_list;
    r.free_count = free_count;
    r.row_status = row_status;
    r.capacity = free_capacity;
    r.B = batch;
    r.k = k;
    r.max_blocks = max_blocks;
    r.block_size = block_size;
    rollback_kernel<<<1, kRollbackThreads, 0, static_cast<cudaStream_t>(stream)>>>(r);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "rollback launch");
    h->launches.fetch_add(1);
    return SPECV_OK;
}

}  // extern "C"

