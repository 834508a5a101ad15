// rollback.cuh -- paged KV-cache bookkeeping after verification, on the
// device: for every row, drop the cache positions of the rejected drafts,
// pop the blocks the shorter sequence no longer needs and append them to the
// free list ("LLM Inference & Speculative Decoding: From Roofline Physics to
// Lossless Acceleration", s.1, PagedKVCacheManager.rollback_to).
//
// The result equals rolling the rows back one at a time in batch order: row
// b's popped blocks land in the free list after those of rows 0..b-1, each
// row's blocks last-first, as popping them one at a time would.  One CTA of
// 1024 threads; thread t owns a contiguous run of rows, so one block-wide
// exclusive scan of the per-thread counts places every row's blocks.
#pragma once
#include <cstdint>

namespace specv {

constexpr int kRollbackThreads = 1024;

enum : int { RB_INVALID = 128, RB_NO_ROOM = 256 };

struct RollbackArgs {
    const int32_t* num_accepted;  // [B]
    int32_t* seq_lens;            // [B] in/out: positions held, the last k the drafts
    int32_t* block_tables;        // [B, max_blocks] in/out: popped entries become -1
    int32_t* num_blocks;          // [B] in/out
    int32_t* free_list;           // [capacity]
    int32_t* free_count;          // [1] in/out: fill of free_list
    int32_t* row_status;          // [B] (nullable): 0, RB_INVALID or RB_NO_ROOM
    long long capacity;
    int B, k, max_blocks, block_size;
};

// Blocks row b gives back, or -1 if its inputs are invalid.
__device__ __forceinline__ int rollback_count(const RollbackArgs& r, int b, int& target, int& needed) {
    const int n = r.num_accepted[b], len = r.seq_lens[b], nb = r.num_blocks[b];
    if (n < 0 || n > r.k || len - (r.k - n) < 0 || nb < 0 || nb > r.max_blocks) return -1;
    target = len - (r.k - n);
    needed = target > 0 ? (target + r.block_size - 1) / r.block_size : 0;
    return nb > needed ? nb - needed : 0;
}

// Exclusive prefix sum over the CTA (1024 threads); *total gets the sum.
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* warp_sums, long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long incl = v;
    for (int off = 1; off < 32; off <<= 1) {
        const long long o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        long long w = warp_sums[lane];
        for (int off = 1; off < 32; off <<= 1) {
            const long long o = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += o;
        }
        warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const long long before = warp == 0 ? 0 : warp_sums[warp - 1];
    *total = warp_sums[31];
    __syncthreads();  // warp_sums is reused by the next call
    return before + incl - v;
}

// Batches of up to kRollbackThreads * kRollbackCached rows: each thread keeps
// its rows in registers, loads them all before the scan and every table
// entry it pops (the first two a row) before its first store, so the
// loads of a run overlap instead of queueing behind one another.
constexpr int kRollbackCached = 4;

__device__ __forceinline__ void rollback_cached(const RollbackArgs& r, int lo, int hi, long long* warp_sums) {
    int cnt[kRollbackCached], tgt[kRollbackCached], nbv[kRollbackCached];
    long long mine = 0;
#pragma unroll
    for (int t = 0; t < kRollbackCached; ++t) {
        const int b = lo + t;
        cnt[t] = 0;
        tgt[t] = 0;
        nbv[t] = 0;
        if (b < hi) {
            int needed = 0;
            cnt[t] = rollback_count(r, b, tgt[t], needed);
            nbv[t] = r.num_blocks[b];
            mine += cnt[t] > 0 ? cnt[t] : 0;
        }
    }
    long long total = 0;
    const long long before = block_exclusive_scan(mine, warp_sums, &total);
    const long long base0 = *r.free_count;
    __syncthreads();  // every thread has read free_count before thread 0 writes it
    if (base0 + total > r.capacity) {
        if (r.row_status)
            for (int b = lo; b < hi; ++b) r.row_status[b] = RB_NO_ROOM;
        return;
    }
    int v0[kRollbackCached], v1[kRollbackCached];  // the first two blocks each row pops
#pragma unroll
    for (int t = 0; t < kRollbackCached; ++t) {
        const int32_t* table = r.block_tables + static_cast<long long>(lo + t) * r.max_blocks;
        v0[t] = cnt[t] >= 1 ? table[nbv[t] - 1] : -1;
        v1[t] = cnt[t] >= 2 ? table[nbv[t] - 2] : -1;
    }
    long long off = base0 + before;
#pragma unroll
    for (int t = 0; t < kRollbackCached; ++t) {
        const int b = lo + t;
        if (b >= hi) continue;
        if (cnt[t] < 0) {
            if (r.row_status) r.row_status[b] = RB_INVALID;
            continue;
        }
        int32_t* table = r.block_tables + static_cast<long long>(b) * r.max_blocks;
        if (cnt[t] >= 1) r.free_list[off] = v0[t];
        if (cnt[t] >= 2) r.free_list[off + 1] = v1[t];
        for (int i = 2; i < cnt[t]; ++i) r.free_list[off + i] = table[nbv[t] - 1 - i];
        for (int i = 0; i < cnt[t]; ++i) table[nbv[t] - 1 - i] = -1;
        off += cnt[t];
        r.num_blocks[b] = nbv[t] - cnt[t];
        r.seq_lens[b] = tgt[t];
        if (r.row_status) r.row_status[b] = 0;
    }
    if (threadIdx.x == 0) *r.free_count = static_cast<int32_t>(base0 + total);
}

__global__ void __launch_bounds__(kRollbackThreads, 1) rollback_kernel(const RollbackArgs r) {
    __shared__ long long warp_sums[32];
    // thread t owns rows [lo, hi): contiguous runs in thread order keep batch order
    const long long per = (static_cast<long long>(r.B) + kRollbackThreads - 1) / kRollbackThreads;
    const long long lo0 = static_cast<long long>(threadIdx.x) * per;
    const int lo = static_cast<int>(lo0 < r.B ? lo0 : r.B);
    const int hi = static_cast<int>(lo0 + per < r.B ? lo0 + per : r.B);
    if (per <= kRollbackCached) {  // uniform over the block
        rollback_cached(r, lo, hi, warp_sums);
        return;
    }
    // 1. the run's count, its place in the free list, and the total
    long long mine = 0;
    for (int b = lo; b < hi; ++b) {
        int target = 0, needed = 0;
        const int cnt = rollback_count(r, b, target, needed);
        mine += cnt > 0 ? cnt : 0;
    }
    long long total = 0;
    const long long before = block_exclusive_scan(mine, warp_sums, &total);
    const long long base0 = *r.free_count;
    __syncthreads();  // every thread has read free_count before thread 0 writes it
    if (base0 + total > r.capacity) {
        if (r.row_status)
            for (int b = lo; b < hi; ++b) r.row_status[b] = RB_NO_ROOM;
        return;
    }
    // 2. pop, last block first, into the run's place
    long long off = base0 + before;
    for (int b = lo; b < hi; ++b) {
        int target = 0, needed = 0;
        const int cnt = rollback_count(r, b, target, needed);
        if (cnt < 0) {
            if (r.row_status) r.row_status[b] = RB_INVALID;
            continue;
        }
        int32_t* table = r.block_tables + static_cast<long long>(b) * r.max_blocks;
        const int nb = r.num_blocks[b];
        for (int i = 0; i < cnt; ++i) {
            r.free_list[off + i] = table[nb - 1 - i];
            table[nb - 1 - i] = -1;
        }
        off += cnt;
        r.num_blocks[b] = nb - cnt;
        r.seq_lens[b] = target;
        if (r.row_status) r.row_status[b] = 0;
    }
    if (threadIdx.x == 0) *r.free_count = static_cast<int32_t>(base0 + total);
}

}  // namespace specv
