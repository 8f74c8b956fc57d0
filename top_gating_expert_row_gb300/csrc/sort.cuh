// CTA-level building blocks of the MoE sorting step (FlyDSL PR 582,
// moe_sorting: bucket every (token, slot) pair by expert into block_m-padded
// blocks; the padded layout is the one FlyDSL PR 947's grouped GEMMs consume,
// where id = token*topk + slot and a sentinel past the last row contributes 0).
//
//   histogram  warp-aggregated shared-memory counts: lanes holding the same
//              expert id find each other with __match_any_sync and one leader
//              adds the group's size
//   scan       padded counts -> exclusive offsets (block scan over E_tot)
//   scatter    stable: each warp owns a contiguous run of flat ids; per-warp
//              per-expert counts give each warp its start inside the expert's
//              range, and within a 32-entry step a pair's rank is the number of
//              lower lanes holding the same expert
//   pads       every padded position past an expert's pairs gets the sentinel,
//              every block of an expert's range its id (a thread per expert)
#pragma once

#include "common.cuh"

namespace mr {

constexpr int kInvalidExpert = -1;

// Warp-aggregated increment of hist[e] for each lane's expert e (lanes with
// e < 0 skip). All 32 lanes must call.
__device__ __forceinline__ void warp_hist_add(uint32_t* hist, int e, int lane)
{
    const unsigned peers = __match_any_sync(kFull, e);
    const int leader = __ffs(peers) - 1;
    if (e >= 0 && lane == leader) atomicAdd(hist + e, static_cast<uint32_t>(__popc(peers)));
}

// Exclusive scan of a[0..n) in place by the whole CTA; returns the total to
// every thread. tmp: 33 words of shared scratch. At most 32 warps.
__device__ inline uint32_t cta_exclusive_scan(uint32_t* a, int n, uint32_t* tmp)
{
    const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + nt - 1) / nt;
    const int b = tid * per;
    uint32_t local = 0u;
    for (int i = 0; i < per; ++i)
        if (b + i < n) local += a[b + i];
    const uint32_t wex = warp_exclusive_scan(local, lane);
    if (lane == 31) tmp[warp] = wex + local;
    __syncthreads();
    if (warp == 0) {
        const int nw = nt >> 5;
        const uint32_t v = lane < nw ? tmp[lane] : 0u;
        const uint32_t ex = warp_exclusive_scan(v, lane);
        __syncwarp();
        if (lane < nw) tmp[lane] = ex;
        if (lane == 31) tmp[32] = ex + v;  // grand total
    }
    __syncthreads();
    uint32_t run = tmp[warp] + wex;
    for (int i = 0; i < per; ++i)
        if (b + i < n) {
            const uint32_t x = a[b + i];
            a[b + i] = run;
            run += x;
        }
    const uint32_t total = tmp[32];
    __syncthreads();
    return total;
}

// Stable scatter of flat ids [f0, f1), f1 - f0 <= kSortChunk, by a CTA of at
// least kSortThreads threads (the sort's CTAs have 512, the fused decode's 512
// or 1024): then no warp owns more than kMaxSteps steps of 32 ids, the number
// each warp keeps in registers. base[e] is the absolute position of the first
// pair of expert e handled by this CTA. wh: nwarps*E_tot 16-bit counters
// (shared). Pairs with ids outside [0, E_tot) are skipped.
__device__ inline void cta_scatter(const int32_t* idx, const float* w, int f0, int f1, int E_tot,
                            const uint32_t* base, uint16_t* wh, int32_t* out_ids, float* out_w)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int n = f1 - f0;
    const int sub = ((n + nw - 1) / nw + 31) & ~31;
    const int r0 = f0 + warp * sub;
    const int r1 = min(r0 + sub, f1);
    uint16_t* mine = wh + warp * E_tot;
    for (int i = tid; i < nw * E_tot; i += blockDim.x) wh[i] = 0;
    // the warp's ids, loaded once (all steps in flight) and kept for both passes;
    // a warp owns ceil(n / warps) ids rounded up to 32, at most kMaxSteps steps
    // of 32 for n <= kSortChunk and at least kSortThreads / 32 warps
    constexpr int kMaxSteps = (kSortChunk + kSortThreads - 1) / kSortThreads;
    int ev[kMaxSteps];
    float wv[kMaxSteps];  // and their weights
#pragma unroll
    for (int u = 0; u < kMaxSteps; ++u) {
        const int i = r0 + u * 32 + lane;
        int e = (i < r1) ? idx[i] : kInvalidExpert;
        ev[u] = (e >= E_tot) ? kInvalidExpert : e;
        wv[u] = (w && i < r1) ? w[i] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kMaxSteps; ++u) {
        if (r0 + u * 32 >= r1) break;
        const int e = ev[u];
        const unsigned peers = __match_any_sync(kFull, e);
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] = static_cast<uint16_t>(mine[e] + __popc(peers));
        __syncwarp();
    }
    __syncthreads();
    for (int e = tid; e < E_tot; e += blockDim.x) {
        uint32_t run = 0u;
        for (int q = 0; q < nw; ++q) {
            const uint32_t c = wh[q * E_tot + e];
            wh[q * E_tot + e] = static_cast<uint16_t>(run);
            run += c;
        }
    }
    __syncthreads();
    const unsigned lt = lanemask_lt();
#pragma unroll
    for (int u = 0; u < kMaxSteps; ++u) {
        if (r0 + u * 32 >= r1) break;
        const int i = r0 + u * 32 + lane;
        const int e = ev[u];
        const unsigned peers = __match_any_sync(kFull, e);
        if (e >= 0) {
            const uint32_t pos = base[e] + mine[e] + __popc(peers & lt);
            out_ids[pos] = i;
            if (out_w) out_w[pos] = wv[u];
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] = static_cast<uint16_t>(mine[e] + __popc(peers));
        __syncwarp();
    }
}

// Sentinels and expert ids of experts [e0, e1), one thread per expert: the
// padded tail of the expert's range, [off[e] + cnt[e], off[e+1]), gets the
// sentinel (weight 0) and each block of the range gets the expert's id. off:
// E_tot+1 exclusive offsets (multiples of bm), cnt: pairs per expert.
__device__ inline void cta_fill_pads(const uint32_t* off, const uint32_t* cnt, int e0, int e1, int bm,
                                     int32_t sentinel, int32_t* out_ids, float* out_w, int32_t* expert_ids)
{
    for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += blockDim.x) {
        const uint32_t a = off[e], b = off[e + 1];
        for (uint32_t p = a + cnt[e]; p < b; ++p) {
            out_ids[p] = sentinel;
            if (out_w) out_w[p] = 0.0f;
        }
        for (uint32_t blk = a / bm; blk < b / bm; ++blk) expert_ids[blk] = e;
    }
}

}  // namespace mr
