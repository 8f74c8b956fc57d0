// Multi-CTA MoE sorting (FlyDSL PR 582, moe_sorting; layout as FlyDSL PR 947's
// grouped GEMMs consume it). Two launches, no grid-wide waiting:
//
//   k_sort_hist     CTA c counts the experts of flat pairs [c*4096, (c+1)*4096)
//                   into ws[c][E_tot] (warp-aggregated shared atomics); ids
//                   outside [0, E_tot) are dropped and flagged in *status
//   k_sort_scatter  every CTA reads the whole (chunks x E_tot) count table,
//                   derives the padded per-expert offsets (block scan) and its
//                   own start inside each expert's range (counts of the chunks
//                   before it), scatters its pairs stably, and writes the
//                   sentinels / expert ids of its share of the experts
//
// The kernel boundary is the only grid-wide ordering, so nothing spins.
#include "internal.h"
#include "sort.cuh"

namespace mr {

__global__ void __launch_bounds__(kSortThreads) k_sort_hist(const int32_t* __restrict__ idx, int N,
                                                            int E_tot, uint32_t* __restrict__ ws,
                                                            int32_t* status)
{
    extern __shared__ __align__(16) uint32_t hist[];
    const int tid = threadIdx.x, lane = tid & 31;
    for (int e = tid; e < E_tot; e += blockDim.x) hist[e] = 0u;
    __syncthreads();
    const int f0 = blockIdx.x * kSortChunk;
    const int f1 = min(f0 + kSortChunk, N);
    bool bad = false;
    // every id of this thread loaded first (one memory latency, not one per step)
    constexpr int kSteps = kSortChunk / kSortThreads;
    int ev[kSteps];
#pragma unroll
    for (int u = 0; u < kSteps; ++u) {
        const int i = f0 + u * kSortThreads + tid;
        ev[u] = (i < f1) ? __ldg(idx + i) : kInvalidExpert;
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
    __syncthreads();
    uint32_t* out = ws + static_cast<size_t>(blockIdx.x) * E_tot;
    for (int e = tid; e < E_tot; e += blockDim.x) out[e] = hist[e];
}

__global__ void __launch_bounds__(kSortThreads) k_sort_scatter(
    const int32_t* __restrict__ idx, const float* __restrict__ w, int N, int E_tot, int bm, int nchunk,
    const uint32_t* __restrict__ ws, int32_t* __restrict__ ids, float* __restrict__ sw,
    int32_t* __restrict__ eids, int32_t* __restrict__ npp)
{
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned char* p = smem;
    uint32_t* cnt = reinterpret_cast<uint32_t*>(p); p += align16(E_tot * 4);
    uint32_t* off = reinterpret_cast<uint32_t*>(p); p += align16((E_tot + 1) * 4);
    uint32_t* base = reinterpret_cast<uint32_t*>(p); p += align16(E_tot * 4);
    uint32_t* tmp = reinterpret_cast<uint32_t*>(p); p += align16(33 * 4);
    uint16_t* wh = reinterpret_cast<uint16_t*>(p);
    const int tid = threadIdx.x, c = blockIdx.x;

    for (int e = tid; e < E_tot; e += blockDim.x) {
        uint32_t before = 0u, total = 0u;
#pragma unroll 8
        for (int q = 0; q < nchunk; ++q) {
            const uint32_t v = __ldg(ws + static_cast<size_t>(q) * E_tot + e);
            before += (q < c) ? v : 0u;
            total += v;
        }
        cnt[e] = total;
        base[e] = before;
        off[e] = (total + bm - 1) / bm * bm;
    }
    __syncthreads();
    const uint32_t P = cta_exclusive_scan(off, E_tot, tmp);
    if (tid == 0) off[E_tot] = P;
    for (int e = tid; e < E_tot; e += blockDim.x) base[e] += off[e];
    if (c == 0 && tid == 0) *npp = static_cast<int32_t>(P);
    __syncthreads();
    const int f0 = c * kSortChunk;
    const int f1 = min(f0 + kSortChunk, N);
    cta_scatter(idx, w, f0, f1, E_tot, base, wh, ids, sw);
    // this CTA's share of the experts' padding and block ids
    const int share = (E_tot + nchunk - 1) / nchunk;
    const int e0 = min(E_tot, c * share);
    const int e1 = min(E_tot, e0 + share);
    cta_fill_pads(off, cnt, e0, e1, bm, N, ids, sw, eids);
}

int launch_sort(const int32_t* idx, const float* w, int N, int E_tot, int block_m, int32_t* ids, float* sw,
                int32_t* eids, int32_t* npp, uint32_t* ws, int32_t* status, cudaStream_t st)
{
    const int nchunk = sort_chunks(N);
    const size_t smem_h = static_cast<size_t>(E_tot) * 4;
    int err = ensure_smem(reinterpret_cast<const void*>(k_sort_hist), smem_h);
    if (err != cudaSuccess) return err;
    k_sort_hist<<<nchunk, kSortThreads, smem_h, st>>>(idx, N, E_tot, ws, status);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const size_t smem_s = static_cast<size_t>(align16(E_tot * 4)) * 2 + align16((E_tot + 1) * 4) +
                          align16(33 * 4) + align16((kSortThreads / 32) * E_tot * 2);
    err = ensure_smem(reinterpret_cast<const void*>(k_sort_scatter), smem_s);
    if (err != cudaSuccess) return err;
    k_sort_scatter<<<nchunk, kSortThreads, smem_s, st>>>(idx, w, N, E_tot, block_m, nchunk, ws, ids, sw,
                                                         eids, npp);
    return cudaGetLastError();
}

}  // namespace mr
