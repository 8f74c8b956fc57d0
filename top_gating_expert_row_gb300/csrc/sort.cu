// MoE sorting (FlyDSL PR 582, moe_sorting; layout as FlyDSL PR 947's grouped
// GEMMs consume it). No grid-wide waiting anywhere: kernel boundaries and
// thread-block cluster barriers are the only cross-CTA ordering.
//
//   k_sort_small    at most kSortChunk pairs: ONE CTA counts, scans, scatters
//                   and pads (one launch)
//   k_sort_cluster  up to cs*1024*2 pairs (cs = 16 CTAs where the GPU allows
//                   clusters that large, else 8): ONE launch of one
//                   thread-block cluster; each CTA keeps its share of the ids
//                   in registers, counts them per warp, and the cluster's CTAs
//                   prefix the counts across CTAs, scan the padded counts and
//                   exchange the offsets through distributed shared memory
//                   before every CTA places its pairs and pads its share of the
//                   blocks (no workspace)
//   k_sort_hist     CTA c counts the experts of flat pairs [c*PC, (c+1)*PC);
//                   clusters of 8 consecutive chunks turn their counts into
//                   within-cluster prefixes pre[c][e] and cluster totals
//                   ctot[g][e] (distributed shared memory); ids outside
//                   [0, E_tot) are dropped and reported in *status
//   k_sort_scatter  clusters of 8 again, one CTA per chunk: the cluster's CTAs
//                   split the experts, sum the totals of the clusters before
//                   theirs and of all clusters, scan the padded counts (slice
//                   totals exchanged through distributed shared memory) and
//                   gather every expert's offset; then each CTA scatters its
//                   chunk's pairs stably and writes its share of the padded
//                   blocks' sentinels and expert ids
//
// Every CTA reads the cluster totals (chunks / 8 rows), never the whole
// per-chunk table, so the cost grows about linearly with the pairs.
#include "internal.h"
#include "sort.cuh"

namespace mr {

// Counts the experts of flat pairs [f0, f1) (f1 - f0 <= kSortChunk, at most
// kSortChunk / kSortThreads per thread) into hist (shared, zeroed); ids outside
// [0, E_tot) are skipped and reported in *status.
__device__ __forceinline__ void cta_count(const int32_t* idx, int f0, int f1, int E_tot,
                                          uint32_t* hist, int32_t* status)
{
    const int tid = threadIdx.x, lane = tid & 31;
    bool bad = false;
    // every id of this thread loaded first (one memory latency, not one per step)
    constexpr int kSteps = kSortChunk / kSortThreads;
    int ev[kSteps];
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
        const int i = f0 + u * kSortThreads + tid;
        ev[u] = (i < f1) ? __ldcg(idx + i) : kInvalidExpert;
    }
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
        if (f0 + u * kSortThreads + (tid & ~31) >= f1) break;  // the warp's ids all past the chunk
        int e = ev[u];
        if (f0 + u * kSortThreads + tid < f1 && (e < 0 || e >= E_tot)) {
            bad = true;
            e = kInvalidExpert;
        }
        warp_hist_add(hist, e, lane);
    }
    if (__any_sync(kFull, bad) && lane == 0) report_status(status, kStatusRange);
}

__global__ void __launch_bounds__(kSortThreads) k_sort_small(const int32_t* idx,
                                                             const float* w, int N, int E_tot, int bm,
                                                             int32_t* ids, float* sw,
                                                             int32_t* eids, int32_t* npp,
                                                             int32_t* status)
{
    pdl_trigger_small();
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* p = smem;
    uint32_t* cnt = reinterpret_cast<uint32_t*>(p); p += align16(E_tot * 4);
    uint32_t* off = reinterpret_cast<uint32_t*>(p); p += align16((E_tot + 1) * 4);
    uint32_t* base = reinterpret_cast<uint32_t*>(p); p += align16(E_tot * 4);
    uint32_t* tmp = reinterpret_cast<uint32_t*>(p); p += align16(33 * 4);
    uint16_t* wh = reinterpret_cast<uint16_t*>(p);
    const int tid = threadIdx.x;
    for (int e = tid; e < E_tot; e += blockDim.x) cnt[e] = 0u;
    __syncthreads();
    pdl_wait();
    cta_count(idx, 0, N, E_tot, cnt, status);
    __syncthreads();
    for (int e = tid; e < E_tot; e += blockDim.x) off[e] = (cnt[e] + bm - 1) / bm * bm;
    __syncthreads();
    const uint32_t P = cta_exclusive_scan(off, E_tot, tmp);
    if (tid == 0) {
        off[E_tot] = P;
        *npp = static_cast<int32_t>(P);
    }
    for (int e = tid; e < E_tot; e += blockDim.x) base[e] = off[e];
    __syncthreads();
    if (N > 0) cta_scatter(idx, w, 0, N, E_tot, base, wh, ids, sw);
    cta_fill_pad_blocks(off, cnt, E_tot, 0, static_cast<int>(P) / bm, bm, N, ids, sw, eids);
}

__global__ void __cluster_dims__(kClusterChunks, 1, 1) __launch_bounds__(kSortThreads)
    k_sort_hist(const int32_t* idx, int N, int PC, int E_tot, uint32_t* pre,
                uint32_t* ctot, int32_t* status)
{
    pdl_trigger_small();
    extern __shared__ __align__(16) uint32_t hist[];
    const int tid = threadIdx.x;
    for (int e = tid; e < E_tot; e += blockDim.x) hist[e] = 0u;
    __syncthreads();
    pdl_wait();
    const long long f0l = static_cast<long long>(blockIdx.x) * PC;
    const int f0 = static_cast<int>(f0l < N ? f0l : N);
    const int f1 = min(f0 + PC, N);
    if (f0 < f1) cta_count(idx, f0, f1, E_tot, hist, status);
    __syncthreads();
    cluster_prefix_counts(hist, E_tot, pre, ctot);
}

// Shared memory of k_sort_scatter: the CTA's expert slice (S = ceil(E_tot/8)
// entries each) and the gathered per-expert arrays.
struct ScatterLayout {
    int s_bsum, s_tot, s_off, s_slice, tmp, base, off, cnt, wh, bytes;
};

__host__ __device__ inline ScatterLayout scatter_layout(int E_tot, int threads)
{
    const int S = (E_tot + kClusterChunks - 1) / kClusterChunks;
    ScatterLayout L;
    int o = 0;
    L.s_bsum = o; o += align16(S * 4);
    L.s_tot = o; o += align16(S * 4);
    L.s_off = o; o += align16(S * 4);
    L.s_slice = o; o += 16;
    L.tmp = o; o += align16(33 * 4);
    L.base = o; o += align16(E_tot * 4);
    L.off = o; o += align16((E_tot + 1) * 4);
    L.cnt = o; o += align16(E_tot * 4);
    L.wh = o; o += align16((threads / 32) * E_tot * 2);
    L.bytes = o;
    return L;
}

__global__ void __cluster_dims__(kClusterChunks, 1, 1) __launch_bounds__(kSortThreads)
    k_sort_scatter(const int32_t* idx, const float* w, int N, int PC, int E_tot, int bm,
                   int ncl, const uint32_t* pre, const uint32_t* ctot,
                   int32_t* ids, float* sw, int32_t* eids,
                   int32_t* npp)
{
    pdl_trigger_small();
    extern __shared__ __align__(16) unsigned char smem[];
    const ScatterLayout L = scatter_layout(E_tot, blockDim.x);
    uint32_t* s_bsum = reinterpret_cast<uint32_t*>(smem + L.s_bsum);
    uint32_t* s_tot = reinterpret_cast<uint32_t*>(smem + L.s_tot);
    uint32_t* s_off = reinterpret_cast<uint32_t*>(smem + L.s_off);
    uint32_t* s_slice = reinterpret_cast<uint32_t*>(smem + L.s_slice);
    uint32_t* tmp = reinterpret_cast<uint32_t*>(smem + L.tmp);
    uint32_t* base = reinterpret_cast<uint32_t*>(smem + L.base);
    uint32_t* off = reinterpret_cast<uint32_t*>(smem + L.off);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(smem + L.cnt);
    uint16_t* wh = reinterpret_cast<uint16_t*>(smem + L.wh);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int c = blockIdx.x;
    const int g = c / kClusterChunks;
    const uint32_t r = cluster_ctarank();
    const int S = (E_tot + kClusterChunks - 1) / kClusterChunks;
    const int e0 = min(E_tot, static_cast<int>(r) * S), len = min(E_tot, e0 + S) - e0;

    // 1. for the CTA's expert slice: pairs in the clusters before this one and
    //    in all clusters. Lanes take 32 consecutive experts (coalesced rows of
    //    ctot), the warps split the clusters between them.
    for (int i = tid; i < len; i += blockDim.x) {
        s_bsum[i] = 0u;
        s_tot[i] = 0u;
    }
    __syncthreads();
    pdl_wait();
    {
        const int nblk = (len + 31) / 32;
        const int parts = max(1, nw / max(1, nblk));
        const int per = (ncl + parts - 1) / parts;
        for (int task = warp; task < nblk * parts; task += nw) {
            const int eb = task % nblk, part = task / nblk;
            const int i = eb * 32 + lane;
            const int q0 = part * per, q1 = min(ncl, q0 + per);
            uint32_t before = 0u, total = 0u;
            if (i < len) {
#pragma unroll 4
                for (int q = q0; q < q1; ++q) {
                    const uint32_t v = __ldcg(ctot + static_cast<size_t>(q) * E_tot + e0 + i);
                    before += q < g ? v : 0u;
                    total += v;
                }
                if (total) {
                    atomicAdd(s_bsum + i, before);
                    atomicAdd(s_tot + i, total);
                }
            }
        }
    }
    __syncthreads();
    // 2. padded counts of the slice, scanned within the slice
    for (int i = tid; i < len; i += blockDim.x) s_off[i] = (s_tot[i] + bm - 1) / bm * bm;
    __syncthreads();
    const uint32_t P = cta_exclusive_scan(s_off, len, tmp);
    if (tid == 0) s_slice[0] = P;
    cluster_sync();
    // 3. the slice's start from the other slices' totals; this cluster's base
    //    for each expert of the slice
    uint32_t soff = 0u, all = 0u;
#pragma unroll
    for (int q = 0; q < kClusterChunks; ++q) {
        const uint32_t t = *cluster_peer(s_slice, static_cast<uint32_t>(q));
        soff += static_cast<uint32_t>(q) < r ? t : 0u;
        all += t;
    }
    for (int i = tid; i < len; i += blockDim.x) {
        s_off[i] += soff;
        s_bsum[i] += s_off[i];
    }
    cluster_sync();
    // 4. every expert's offset, count and base from its slice's CTA, plus this
    //    chunk's prefix inside the cluster
    {
        const uint32_t* prow = pre + static_cast<size_t>(c) * E_tot;
        for (int e = tid; e < E_tot; e += blockDim.x) {
            const uint32_t q = static_cast<uint32_t>(e / S);
            const int i = e - static_cast<int>(q) * S;
            base[e] = cluster_peer(s_bsum, q)[i] + __ldcg(prow + e);
            off[e] = cluster_peer(s_off, q)[i];
            cnt[e] = cluster_peer(s_tot, q)[i];
        }
        if (tid == 0) off[E_tot] = all;
    }
    cluster_sync();  // no CTA reads another CTA's shared memory after this point
    if (c == 0 && tid == 0) *npp = static_cast<int32_t>(all);
    // 5. this chunk's pairs
    const long long f0l = static_cast<long long>(c) * PC;
    const int f0 = static_cast<int>(f0l < N ? f0l : N);
    const int f1 = min(f0 + PC, N);
    if (f0 < f1) cta_scatter(idx, w, f0, f1, E_tot, base, wh, ids, sw);
    // 6. the CTA's share of the padded blocks
    const long long nb = all / static_cast<uint32_t>(bm);
    const int G = gridDim.x;
    const int b0 = static_cast<int>(nb * c / G), b1 = static_cast<int>(nb * (c + 1) / G);
    cta_fill_pad_blocks(off, cnt, E_tot, b0, b1, bm, N, ids, sw, eids);
}

// CTA r of the cluster handles flat pairs [r*P, (r+1)*P), P <= 1024 * 2.
__global__ void __launch_bounds__(kClusterSortThreads, 1)
    k_sort_cluster(const int32_t* idx, const float* w, int N, int P, int E_tot, int bm, int32_t* ids, float* sw,
                   int32_t* eids, int32_t* npp, int32_t* status)
{
    pdl_trigger_small();
    pdl_wait();
    extern __shared__ __align__(16) unsigned char smem[];
    const uint32_t r = cluster_ctarank();
    const long long f0l = static_cast<long long>(r) * P;
    const int f0 = static_cast<int>(f0l < N ? f0l : N), f1 = min(N, f0 + P);
    WarpRuns<kClusterSortUseSteps> R;
    const bool bad = warp_runs_load<kClusterSortUseSteps>(idx, w, 0, f0, f1, E_tot, R);
    cluster_sort_runs<kClusterSortUseSteps>(R, bad, N, E_tot, bm, smem, ids, sw, eids, npp, status);
}

size_t scatter_smem_bytes(int E_tot) { return static_cast<size_t>(scatter_layout(E_tot, kSortThreads).bytes); }

size_t small_sort_smem_bytes(int E_tot)
{
    return static_cast<size_t>(align16(E_tot * 4)) * 2 + align16((E_tot + 1) * 4) + align16(33 * 4) +
           align16((kSortThreads / 32) * E_tot * 2);
}

int launch_sort_scatter(const int32_t* idx, const float* w, int N, int PC, int nchunk_pad, int E_tot, int block_m,
                        const uint32_t* pre, const uint32_t* ctot, int32_t* ids, float* sw, int32_t* eids,
                        int32_t* npp, cudaStream_t st)
{
    const size_t smem = scatter_smem_bytes(E_tot);
    int err = ensure_smem(reinterpret_cast<const void*>(k_sort_scatter), smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(k_sort_scatter, dim3(nchunk_pad), dim3(kSortThreads), smem, st, 0, idx, w, N, PC, E_tot,
                         block_m, nchunk_pad / kClusterChunks, pre, ctot, ids, sw, eids, npp);
}

namespace {
// The largest cluster k_sort_cluster can use with E_tot experts on the current
// device: 16 where the device schedules non-portable clusters of 16, else 8;
// 0 if neither fits (the shared memory for E_tot does not).
int cluster_sort_size(int E_tot)
{
    const void* f = reinterpret_cast<const void*>(k_sort_cluster);
    for (int cs : {16, 8})
        if (cluster_fits(f, kClusterSortThreads, static_cast<size_t>(cluster_sort_layout(E_tot).bytes), cs))
            return cs;
    return 0;
}
}  // namespace

int launch_sort(const int32_t* idx, const float* w, int N, int E_tot, int block_m, int32_t* ids, float* sw,
                int32_t* eids, int32_t* npp, uint32_t* ws, int32_t* status, cudaStream_t st)
{
    if (N > kSortChunk) {
        const int cs = cluster_sort_size(E_tot);
        const long long per_cta = static_cast<long long>(kClusterSortThreads) * kClusterSortUseSteps;
        if (cs > 0 && N <= cs * per_cta) {
            // pairs per CTA: whole steps of the CTA's threads
            const long long P = ((N + cs - 1) / cs + kClusterSortThreads - 1) / kClusterSortThreads * kClusterSortThreads;
            const size_t smem = static_cast<size_t>(cluster_sort_layout(E_tot).bytes);
            const int err = ensure_smem(reinterpret_cast<const void*>(k_sort_cluster), smem);
            if (err != cudaSuccess) return err;
            return launch_kernel(k_sort_cluster, dim3(cs), dim3(kClusterSortThreads), smem, st, cs, idx, w, N,
                                 static_cast<int>(P), E_tot, block_m, ids, sw, eids, npp, status);
        }
    }
    if (N <= kSortChunk) {
        const size_t smem = small_sort_smem_bytes(E_tot);
        int err = ensure_smem(reinterpret_cast<const void*>(k_sort_small), smem);
        if (err != cudaSuccess) return err;
        return launch_kernel(k_sort_small, dim3(1), dim3(kSortThreads), smem, st, 0, idx, w, N, E_tot, block_m, ids, sw,
                             eids, npp, status);
    }
    const SortPlan plan = sort_plan(N, E_tot);
    uint32_t* pre = ws;
    uint32_t* ctot = ws + static_cast<size_t>(plan.nchunk_pad) * E_tot;
    const size_t smem_h = static_cast<size_t>(E_tot) * 4;
    int err = ensure_smem(reinterpret_cast<const void*>(k_sort_hist), smem_h);
    if (err != cudaSuccess) return err;
    err = launch_kernel(k_sort_hist, dim3(plan.nchunk_pad), dim3(kSortThreads), smem_h, st, 0, idx, N, plan.pc, E_tot,
                        pre, ctot, status);
    if (err != cudaSuccess) return err;
    return launch_sort_scatter(idx, w, N, plan.pc, plan.nchunk_pad, E_tot, block_m, pre, ctot, ids, sw, eids, npp,
                               st);
}

}  // namespace mr
