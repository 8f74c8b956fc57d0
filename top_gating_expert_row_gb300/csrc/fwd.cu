// Router forward and fused decode route+sort kernels for one (score function,
// logits dtype) pair. Compiled once per pair with -DMR_SCORE_FN=0|1 and
// -DMR_IN_BF16=0|1 so the four instantiation sets build in parallel.
//
//   k_router_fwd     persistent grid, 8 warps per CTA, one token row per warp
//                    at a time (TransformerEngine PR 3012, fused_topk_with_
//                    score_function; also serves fused_score_for_moe_aux_loss)
//   k_fused_decode   ONE CTA for T <= 16 tokens: warp t routes token t, then
//                    the whole CTA histograms, scans and scatters the T*topk
//                    pairs in shared memory (FlyDSL PR 582, fused top-k gating
//                    + MoE sorting at decode sizes)
#include "internal.h"
#include "sort.cuh"

#ifndef MR_SCORE_FN
#error "MR_SCORE_FN must be defined (0 softmax, 1 sigmoid)"
#endif
#ifndef MR_IN_BF16
#error "MR_IN_BF16 must be defined (0 fp32, 1 bf16)"
#endif

#define MR_CAT2(a, b) a##b
#define MR_CAT(a, b) MR_CAT2(a, b)
#define MR_SUFFIX MR_CAT(MR_CAT(_s, MR_SCORE_FN), MR_CAT(_d, MR_IN_BF16))

namespace mr {

#if MR_IN_BF16
using InT = __nv_bfloat16;
#else
using InT = float;
#endif
constexpr int kScore = MR_SCORE_FN;

template <int NV, bool SELECT>
__global__ void __launch_bounds__(kFwdThreads) k_router_fwd(RouteArgs a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, SELECT, a.n_group > 0);
    unsigned char* wsm = smem + static_cast<size_t>(warp) * L.bytes;
    for (int t = blockIdx.x * nw + warp; t < a.T; t += gridDim.x * nw) {
        const float scale = route_row<kScore, InT, NV, SELECT>(a, t, wsm, L, lane);
        if (a.topk_idx || a.topk_w) {
            const size_t o = static_cast<size_t>(t) * a.topk;
            emit_compact(a, wsm, L, scale, lane, a.topk_idx ? a.topk_idx + o : nullptr,
                         a.topk_w ? a.topk_w + o : nullptr);
        }
        __syncwarp();
    }
}

template <int NV, bool SELECT>
__global__ void __launch_bounds__(kFusedThreads) k_fused_decode(RouteArgs a, SortArgs s)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, SELECT, a.n_group > 0);
    const int N = a.T * a.topk;
    unsigned char* p = smem + static_cast<size_t>(nw) * L.bytes;
    int32_t* s_idx = reinterpret_cast<int32_t*>(p); p += align16(N * 4);
    float* s_w = reinterpret_cast<float*>(p); p += align16(N * 4);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(p); p += align16(s.E_tot * 4);
    uint32_t* off = reinterpret_cast<uint32_t*>(p); p += align16((s.E_tot + 1) * 4);
    uint32_t* tmp = reinterpret_cast<uint32_t*>(p); p += align16(33 * 4);
    uint16_t* wh = reinterpret_cast<uint16_t*>(p);

    for (int e = tid; e < s.E_tot; e += blockDim.x) cnt[e] = 0u;
    if (warp < a.T) {
        unsigned char* wsm = smem + static_cast<size_t>(warp) * L.bytes;
        const float scale = route_row<kScore, InT, NV, SELECT>(a, warp, wsm, L, lane);
        const size_t o = static_cast<size_t>(warp) * a.topk;
        emit_compact(a, wsm, L, scale, lane, s_idx + o, s_w + o);
        if (a.topk_idx || a.topk_w)
            emit_compact(a, wsm, L, scale, lane, a.topk_idx ? a.topk_idx + o : nullptr,
                         a.topk_w ? a.topk_w + o : nullptr);
    }
    __syncthreads();
    // histogram of the T*topk pairs (ids are in range for finite logits; the
    // check keeps a NaN row from indexing outside the counters)
    for (int i0 = warp * 32; i0 < N; i0 += blockDim.x) {
        const int i = i0 + lane;
        const int e = i < N ? s_idx[i] : kInvalidExpert;
        warp_hist_add(cnt, (e >= 0 && e < s.E_tot) ? e : kInvalidExpert, lane);
    }
    __syncthreads();
    for (int e = tid; e < s.E_tot; e += blockDim.x) {
        const uint32_t c = cnt[e];
        off[e] = (c + s.block_m - 1) / s.block_m * s.block_m;
    }
    __syncthreads();
    const uint32_t total = cta_exclusive_scan(off, s.E_tot, tmp);
    if (tid == 0) {
        off[s.E_tot] = total;
        *s.num_post_pad = static_cast<int32_t>(total);
    }
    __syncthreads();
    cta_scatter(s_idx, s_w, 0, N, s.E_tot, off, wh, s.ids, s.w);
    cta_fill_pads(off, cnt, s.E_tot, s.block_m, 0, static_cast<int>(total), N, s.ids, s.w,
                  s.expert_ids);
}

namespace {

using FwdFn = void (*)(RouteArgs);
using FusedFn = void (*)(RouteArgs, SortArgs);

template <bool SELECT>
FwdFn fwd_kernel(int nv_idx)
{
    switch (kNvBuckets[nv_idx]) {
        case 1: return k_router_fwd<1, SELECT>;
        case 2: return k_router_fwd<2, SELECT>;
        case 3: return k_router_fwd<3, SELECT>;
        case 4: return k_router_fwd<4, SELECT>;
        case 6: return k_router_fwd<6, SELECT>;
        case 8: return k_router_fwd<8, SELECT>;
        case 12: return k_router_fwd<12, SELECT>;
        case 18: return k_router_fwd<18, SELECT>;
    }
    return nullptr;
}

template <bool SELECT>
FusedFn fused_kernel(int nv_idx)
{
    switch (kNvBuckets[nv_idx]) {
        case 1: return k_fused_decode<1, SELECT>;
        case 2: return k_fused_decode<2, SELECT>;
        case 3: return k_fused_decode<3, SELECT>;
        case 4: return k_fused_decode<4, SELECT>;
        case 6: return k_fused_decode<6, SELECT>;
        case 8: return k_fused_decode<8, SELECT>;
    }
    return nullptr;
}

}  // namespace

int MR_CAT(launch_fwd, MR_SUFFIX)(const RouteArgs& a, int nv_idx, bool select, cudaStream_t st)
{
    const FwdFn f = select ? fwd_kernel<true>(nv_idx) : fwd_kernel<false>(nv_idx);
    if (!f) return cudaErrorInvalidValue;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, select, a.n_group > 0);
    const size_t smem = static_cast<size_t>(L.bytes) * (kFwdThreads / 32);
    int err = ensure_smem(reinterpret_cast<const void*>(f), smem);
    if (err != cudaSuccess) return err;
    const long long ctas_needed = (static_cast<long long>(a.T) + kFwdThreads / 32 - 1) / (kFwdThreads / 32);
    const int grid = persistent_grid(reinterpret_cast<const void*>(f), kFwdThreads, smem, ctas_needed);
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    f<<<grid, kFwdThreads, smem, st>>>(a);
    return cudaGetLastError();
}

int MR_CAT(launch_fused, MR_SUFFIX)(const RouteArgs& a, const SortArgs& s, int nv_idx, bool select,
                                    cudaStream_t st)
{
    const FusedFn f = select ? fused_kernel<true>(nv_idx) : fused_kernel<false>(nv_idx);
    if (!f) return cudaErrorInvalidValue;
    const int nw = kFusedThreads / 32;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, select, a.n_group > 0);
    const size_t smem = static_cast<size_t>(L.bytes) * nw + fused_sort_smem(a.T * a.topk, s.E_tot, nw);
    int err = ensure_smem(reinterpret_cast<const void*>(f), smem);
    if (err != cudaSuccess) return err;
    f<<<1, kFusedThreads, smem, st>>>(a, s);
    return cudaGetLastError();
}

}  // namespace mr
