// CTA- and cluster-level building blocks of the MoE sorting step (FlyDSL PR
// 582, moe_sorting: bucket every (token, slot) pair by expert into
// block_m-padded blocks; the padded layout is the one FlyDSL PR 947's grouped
// GEMMs consume, where id = token*topk + slot and a sentinel past the last row
// contributes 0).
//
//   histogram  warp-aggregated shared-memory counts: lanes holding the same
//              expert id find each other with __match_any_sync and one leader
//              adds the group's size
//   cluster    the counts of 8 consecutive chunks (one thread-block cluster)
//   prefix     become within-cluster exclusive prefixes and a cluster total,
//              the CTAs splitting the experts and reading each other's counts
//              through distributed shared memory
//   scan       padded counts -> exclusive offsets (block scan over experts)
//   scatter    stable: each warp owns a contiguous run of flat ids; per-warp
//              per-expert counts give each warp its start inside the expert's
//              range, and within a 32-entry step a pair's rank is the number of
//              lower lanes holding the same expert
//   pads       a warp per block of block_m positions: the block's expert by a
//              binary search over the offsets, the sentinel at every position
//              past the expert's pairs, and the block's expert id
#pragma once

#include "common.cuh"

namespace mr {

constexpr int kSortThreads = 512;
constexpr int kSortChunk = 4096;  // flat (token, slot) pairs per sort CTA, at most
// the one-cluster sort: CTAs of 1024 threads, up to 2 pairs per thread (each
// warp walks its pairs in serial steps of 32; with more steps the chunked
// sort's many more warps win)
constexpr int kClusterSortThreads = 1024;
constexpr int kClusterSortUseSteps = 2;
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

// Stable placement of flat ids [f0, f1) by a CTA, in two halves so that the
// positions can be settled in between (by the CTA alone or by its cluster):
//   warp_runs_count  each warp owns a contiguous run of ceil(n / warps) ids
//                    rounded up to 32 (at most STEPS steps of 32, kept in
//                    registers with their weights) and counts its run's pairs
//                    per expert into wh[warp][e] (16-bit, shared)
//   warp_runs_place  writes each pair at base[e] + wh[warp][e] (the warps
//                    before it, after the caller's exclusive scan over warps)
//                    + its rank among the warp's earlier pairs of e (per step,
//                    the lower lanes holding the same expert)
// Pairs with ids outside [0, E_tot) are skipped.
template <int STEPS>
struct WarpRuns {
    int ev[STEPS];
    float wv[STEPS];
    int r0, r1;
};

// The warp's run of flat pairs [f0, f1) into R (pair i is idx[i - base],
// w[i - base]; global or shared memory). Returns whether any of the thread's
// ids lay outside [0, E_tot).
template <int STEPS>
__device__ __forceinline__ bool warp_runs_load(const int32_t* idx, const float* w, int base, int f0, int f1, int E_tot,
                                               WarpRuns<STEPS>& R)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int n = f1 - f0;
    const int sub = ((n + nw - 1) / nw + 31) & ~31;
    R.r0 = min(f1, f0 + warp * sub);
    R.r1 = min(R.r0 + sub, f1);
    // the warp's ids and weights, loaded once (all steps in flight)
    bool bad = false;
#pragma unroll
    for (int u = 0; u < STEPS; ++u) {
        const int i = R.r0 + u * 32 + lane;
        const int e = (i < R.r1) ? idx[i - base] : kInvalidExpert;
        bad |= i < R.r1 && (e < 0 || e >= E_tot);
        R.ev[u] = (e < 0 || e >= E_tot) ? kInvalidExpert : e;
        R.wv[u] = (w && i < R.r1) ? w[i - base] : 0.0f;
    }
    return bad;
}

// The per-warp counts of the loaded runs into wh[warp][e].
template <int STEPS>
__device__ __forceinline__ void warp_runs_tally(int E_tot, uint16_t* wh, const WarpRuns<STEPS>& R)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    uint16_t* mine = wh + warp * E_tot;
    for (int i = tid; i < nw * E_tot; i += blockDim.x) wh[i] = 0;
    __syncthreads();
#pragma unroll
    for (int u = 0; u < STEPS; ++u) {
        if (R.r0 + u * 32 >= R.r1) break;
        const int e = R.ev[u];
        const unsigned peers = __match_any_sync(kFull, e);
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] = static_cast<uint16_t>(mine[e] + __popc(peers));
        __syncwarp();
    }
}

// warp_runs_load (from pair 0 of idx / w) and warp_runs_tally.
template <int STEPS>
__device__ __forceinline__ bool warp_runs_count(const int32_t* idx, const float* w, int f0, int f1, int E_tot,
                                                uint16_t* wh, WarpRuns<STEPS>& R)
{
    const bool bad = warp_runs_load<STEPS>(idx, w, 0, f0, f1, E_tot, R);
    warp_runs_tally<STEPS>(E_tot, wh, R);
    return bad;
}

template <int STEPS>
__device__ __forceinline__ void warp_runs_place(const WarpRuns<STEPS>& R, int E_tot, const uint32_t* base,
                                                uint16_t* wh, int32_t* out_ids, float* out_w)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint16_t* mine = wh + warp * E_tot;
    const unsigned lt = lanemask_lt();
#pragma unroll
    for (int u = 0; u < STEPS; ++u) {
        if (R.r0 + u * 32 >= R.r1) break;
        const int i = R.r0 + u * 32 + lane;
        const int e = R.ev[u];
        const unsigned peers = __match_any_sync(kFull, e);
        if (e >= 0) {
            const uint32_t pos = base[e] + mine[e] + __popc(peers & lt);
            out_ids[pos] = i;
            if (out_w) out_w[pos] = R.wv[u];
        }
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) mine[e] = static_cast<uint16_t>(mine[e] + __popc(peers));
        __syncwarp();
    }
}

// Stable scatter of flat ids [f0, f1), f1 - f0 <= kSortChunk, by a CTA of at
// least kSortThreads threads (then no warp owns more than kSortChunk /
// kSortThreads steps of 32). base[e] is the absolute position of the first
// pair of expert e handled by this CTA. wh: nwarps*E_tot 16-bit counters
// (shared).
__device__ inline void cta_scatter(const int32_t* idx, const float* w, int f0, int f1, int E_tot,
                                   const uint32_t* base, uint16_t* wh, int32_t* out_ids, float* out_w)
{
    constexpr int kSteps = (kSortChunk + kSortThreads - 1) / kSortThreads;
    const int nw = blockDim.x >> 5;
    WarpRuns<kSteps> R;
    warp_runs_count<kSteps>(idx, w, f0, f1, E_tot, wh, R);
    __syncthreads();
    for (int e = threadIdx.x; e < E_tot; e += blockDim.x) {
        uint32_t run = 0u;
        for (int q = 0; q < nw; ++q) {
            const uint32_t c = wh[q * E_tot + e];
            wh[q * E_tot + e] = static_cast<uint16_t>(run);
            run += c;
        }
    }
    __syncthreads();
    warp_runs_place<kSteps>(R, E_tot, base, wh, out_ids, out_w);
}

// Sentinels and expert ids by expert, a warp per expert (the lanes cover the
// expert's padded positions and blocks): for sorts with few pairs per expert,
// where a search per block costs more than a look at every expert.
__device__ inline void cta_fill_pads_by_expert(const uint32_t* off, const uint32_t* cnt, int E_tot, int bm,
                                               int32_t sentinel, int32_t* out_ids, float* out_w, int32_t* expert_ids)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int e = warp; e < E_tot; e += nw) {
        const uint32_t a = off[e], b = off[e + 1];
        if (a == b) continue;
        for (uint32_t p = a + cnt[e] + lane; p < b; p += 32) {
            out_ids[p] = sentinel;
            if (out_w) out_w[p] = 0.0f;
        }
        for (uint32_t blk = a / bm + lane; blk < b / bm; blk += 32) expert_ids[blk] = e;
    }
}

// Chunks of flat pairs per thread-block cluster of the sort (and of the route
// kernel that feeds it).
constexpr int kClusterChunks = 8;

// Called by every thread of every CTA of a cluster of kClusterChunks CTAs
// (blockIdx.x / kClusterChunks = cluster g, rank q = chunk g*8 + q), each with
// its chunk's per-expert counts in hist[0..E_tot) (shared). Writes
//   pre[(g*8 + q)*E_tot + e] = sum of the counts of chunks g*8 .. g*8+q-1
//   ctot[g*E_tot + e]        = sum of the counts of the cluster's 8 chunks
// The experts are split over the cluster's CTAs; the other CTAs' counts are
// read through distributed shared memory. Starts and ends with a cluster
// barrier, so no CTA leaves while its counts may still be read.
__device__ inline void cluster_prefix_counts(const uint32_t* hist, int E_tot, uint32_t* pre, uint32_t* ctot)
{
    cluster_sync();
    const uint32_t r = cluster_ctarank();
    const size_t g = blockIdx.x / kClusterChunks;
    const int S = (E_tot + kClusterChunks - 1) / kClusterChunks;
    const int e0 = static_cast<int>(r) * S, e1 = min(E_tot, e0 + S);
    const uint32_t* remote[kClusterChunks];
#pragma unroll
    for (int q = 0; q < kClusterChunks; ++q) remote[q] = cluster_peer(hist, static_cast<uint32_t>(q));
    for (int e = e0 + static_cast<int>(threadIdx.x); e < e1; e += blockDim.x) {
        uint32_t v[kClusterChunks];
#pragma unroll
        for (int q = 0; q < kClusterChunks; ++q) v[q] = remote[q][e];
        uint32_t run = 0u;
#pragma unroll
        for (int q = 0; q < kClusterChunks; ++q) {
            pre[(g * kClusterChunks + q) * E_tot + e] = run;
            run += v[q];
        }
        ctot[g * E_tot + e] = run;
    }
    cluster_sync();
}

// Sentinels and expert ids of blocks [b0, b1) of the padded layout, a warp
// per block. off: E_tot+1 exclusive offsets (multiples of bm, off[E_tot] the
// padded total), cnt: pairs per expert (both shared). A block's expert is the
// last e with off[e] <= its first position (an empty expert's range is empty,
// so the search skips it); the block's positions past the expert's pairs get
// the sentinel (weight 0).
__device__ inline void cta_fill_pad_blocks(const uint32_t* off, const uint32_t* cnt, int E_tot, int b0, int b1,
                                           int bm, int32_t sentinel, int32_t* out_ids, float* out_w,
                                           int32_t* expert_ids)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    for (int b = b0 + warp; b < b1; b += nw) {
        const uint32_t p0 = static_cast<uint32_t>(b) * static_cast<uint32_t>(bm);
        int lo = 0, hi = E_tot;  // off[lo] <= p0 < off[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (off[mid] <= p0) lo = mid;
            else hi = mid;
        }
        const uint32_t filled = cnt[lo] > p0 - off[lo] ? cnt[lo] - (p0 - off[lo]) : 0u;  // real pairs in the block
        for (int r = lane; r < bm; r += 32) {
            if (static_cast<uint32_t>(r) >= filled) {
                out_ids[p0 + r] = sentinel;
                if (out_w) out_w[p0 + r] = 0.0f;
            }
        }
        if (lane == 0) expert_ids[b] = lo;
    }
}

// Shared memory of the one-cluster sort: per-warp counts and the CTA's
// per-expert arrays.
struct ClusterSortLayout {
    int wh, hist, before, base, off, cnt, tmp, bytes;
};

__host__ __device__ inline ClusterSortLayout cluster_sort_layout(int E_tot)
{
    ClusterSortLayout L;
    int o = 0;
    L.wh = o; o += align16((kClusterSortThreads / 32) * E_tot * 2);
    L.hist = o; o += align16(E_tot * 4);
    L.before = o; o += align16(E_tot * 4);
    L.base = o; o += align16(E_tot * 4);
    L.off = o; o += align16((E_tot + 1) * 4);
    L.cnt = o; o += align16(E_tot * 4);
    L.tmp = o; o += align16(33 * 4);
    L.bytes = o;
    return L;
}

// The sort of one thread-block cluster (cs CTAs, each with the runs of its
// pairs already loaded into R): per-warp counts and each CTA's count per
// expert; after one cluster barrier every CTA reads all CTAs' counts through
// distributed shared memory (its exclusive prefix over the CTAs before it and
// the totals), scans the padded totals itself, and places its pairs and its
// share of the padded blocks. The CTA arrives at a second barrier once its
// remote reads are done and waits on it only before it exits. `smem` is the
// CTA's region of cluster_sort_layout(E_tot).bytes. Called by every thread of
// every CTA of the cluster.
template <int STEPS>
__device__ __forceinline__ void cluster_sort_runs(WarpRuns<STEPS>& R, bool bad, int N, int E_tot, int bm,
                                                  unsigned char* smem, int32_t* ids, float* sw, int32_t* eids,
                                                  int32_t* npp, int32_t* status)
{
    const uint32_t cs = cluster_nctarank(), r = cluster_ctarank();
    const ClusterSortLayout L = cluster_sort_layout(E_tot);
    uint16_t* wh = reinterpret_cast<uint16_t*>(smem + L.wh);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + L.hist);
    uint32_t* before = reinterpret_cast<uint32_t*>(smem + L.before);
    uint32_t* base = reinterpret_cast<uint32_t*>(smem + L.base);
    uint32_t* off = reinterpret_cast<uint32_t*>(smem + L.off);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + L.cnt);
    uint32_t* tmp = reinterpret_cast<uint32_t*>(smem + L.tmp);
    const int tid = threadIdx.x, lane = tid & 31, nw = blockDim.x >> 5;

    // 1. the CTA's pairs (in registers), counted per warp
    warp_runs_tally<STEPS>(E_tot, wh, R);
    if (__any_sync(kFull, bad) && lane == 0) report_status(status, kStatusRange);
    __syncthreads();
    // 2. the CTA's count per expert; the warps' counts become exclusive prefixes
    for (int e = tid; e < E_tot; e += blockDim.x) {
        uint32_t run = 0u;
        for (int q = 0; q < nw; ++q) {
            const uint32_t c = wh[q * E_tot + e];
            wh[q * E_tot + e] = static_cast<uint16_t>(run);
            run += c;
        }
        hist[e] = run;
    }
    cluster_sync();
    // 3. every CTA's count of every expert: the CTAs before this one, and all
    for (int e = tid; e < E_tot; e += blockDim.x) {
        uint32_t b = 0u, t = 0u;
#pragma unroll 4
        for (uint32_t q = 0; q < cs; ++q) {
            const uint32_t v = cluster_peer(hist, q)[e];
            b += q < r ? v : 0u;
            t += v;
        }
        before[e] = b;
        cnt[e] = t;
        off[e] = (t + bm - 1) / bm * bm;
    }
    cluster_arrive();  // this CTA reads no other CTA's shared memory after this
    __syncthreads();
    // 4. padded offsets, this CTA's base per expert
    const uint32_t all = cta_exclusive_scan(off, E_tot, tmp);
    if (tid == 0) off[E_tot] = all;
    for (int e = tid; e < E_tot; e += blockDim.x) base[e] = off[e] + before[e];
    __syncthreads();
    if (r == 0 && tid == 0) *npp = static_cast<int32_t>(all);
    // 5. the pairs, and the CTA's share of the padded blocks
    warp_runs_place<STEPS>(R, E_tot, base, wh, ids, sw);
    const long long nb = all / static_cast<uint32_t>(bm);
    const int b0 = static_cast<int>(nb * r / cs), b1 = static_cast<int>(nb * (r + 1) / cs);
    cta_fill_pad_blocks(off, cnt, E_tot, b0, b1, bm, N, ids, sw, eids);
    cluster_wait();  // no CTA leaves while another may still read its counts
}

}  // namespace mr
