// Router backward and aux-score backward (TransformerEngine PR 3012, "Two-pass
// fused design": pass 1 reduces the row sums in registers with warp
// all-reduces, pass 2 forms each element's gradient; no shared-memory buffer).
//
// One warp per token row, the row held in registers (g, s, routing map):
//   ds_i = c * m_i * g_i                         (no renorm)
//   ds_i = (c * m_i / A) * (g_i - B / A)          (renorm; A = sum m s, B = sum m s g)
//   softmax: dx_i = s_i * (ds_i - sum_j s_j ds_j);  sigmoid: dx_i = ds_i * s_i * (1 - s_i)
// The aux-score backward is the same with m = 1, c = 1 and no renorm.
#include "internal.h"

namespace mr {

template <int SCORE, int NV, bool HAS_MAP>
__global__ void __launch_bounds__(kBwdThreads) k_router_bwd(const float* __restrict__ grad,
                                                            const float* __restrict__ inter,
                                                            const uint8_t* __restrict__ map,
                                                            float* __restrict__ dx, int T, int E,
                                                            int renorm, float c, int vec)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int t = blockIdx.x * nw + warp; t < T; t += gridDim.x * nw) {
        const size_t ro = static_cast<size_t>(t) * E;
        float g[NV][4], s[NV][4];
        uint32_t m[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e0 = (v * 32 + lane) * 4;
            if (vec && e0 + 4 <= E) {
                const float4 a = __ldcs(reinterpret_cast<const float4*>(grad + ro + e0));
                const float4 b = __ldcs(reinterpret_cast<const float4*>(inter + ro + e0));
                g[v][0] = a.x; g[v][1] = a.y; g[v][2] = a.z; g[v][3] = a.w;
                s[v][0] = b.x; s[v][1] = b.y; s[v][2] = b.z; s[v][3] = b.w;
                m[v] = HAS_MAP ? __ldcs(reinterpret_cast<const unsigned int*>(map + ro + e0)) : 0x01010101u;
            } else {
                m[v] = 0u;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const bool in = e0 + q < E;
                    g[v][q] = in ? __ldcs(grad + ro + e0 + q) : 0.0f;
                    s[v][q] = in ? __ldcs(inter + ro + e0 + q) : 0.0f;
                    const uint32_t mb = in ? (HAS_MAP ? static_cast<uint32_t>(map[ro + e0 + q] != 0) : 1u) : 0u;
                    m[v] |= mb << (8 * q);
                }
            }
        }
        // pass 1: row sums
        float A = 0.0f, B = 0.0f;
        if (HAS_MAP && renorm) {
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if ((m[v] >> (8 * q)) & 0xffu) {
                        A += s[v][q];
                        B += s[v][q] * g[v][q];
                    }
            A = warp_sum(A);
            B = warp_sum(B);
        }
        const bool rn = HAS_MAP && renorm;
        const float cA = (rn && A != 0.0f) ? c / A : 0.0f;
        const float BA = (rn && A != 0.0f) ? B / A : 0.0f;
        // pass 2: ds, then the score-function Jacobian
        float D = 0.0f;
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool mk = (m[v] >> (8 * q)) & 0xffu;
                const float ds = mk ? (rn ? cA * (g[v][q] - BA) : c * g[v][q]) : 0.0f;
                g[v][q] = ds;
                if (SCORE == kSoftmax) D += s[v][q] * ds;
            }
        if (SCORE == kSoftmax) D = warp_sum(D);
        float* out = dx + ro;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e0 = (v * 32 + lane) * 4;
            if (e0 >= E) continue;
            float r[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                r[q] = (SCORE == kSoftmax) ? s[v][q] * (g[v][q] - D) : g[v][q] * s[v][q] * (1.0f - s[v][q]);
            if (vec && e0 + 4 <= E) {
                __stcs(reinterpret_cast<float4*>(out + e0), make_float4(r[0], r[1], r[2], r[3]));
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (e0 + q < E) out[e0 + q] = r[q];
            }
        }
    }
}

namespace {
using BwdFn = void (*)(const float*, const float*, const uint8_t*, float*, int, int, int, float, int);

template <int SCORE, bool HAS_MAP>
BwdFn bwd_kernel(int nv_idx)
{
    switch (kNvBuckets[nv_idx]) {
        case 1: return k_router_bwd<SCORE, 1, HAS_MAP>;
        case 2: return k_router_bwd<SCORE, 2, HAS_MAP>;
        case 3: return k_router_bwd<SCORE, 3, HAS_MAP>;
        case 4: return k_router_bwd<SCORE, 4, HAS_MAP>;
        case 6: return k_router_bwd<SCORE, 6, HAS_MAP>;
        case 8: return k_router_bwd<SCORE, 8, HAS_MAP>;
        case 12: return k_router_bwd<SCORE, 12, HAS_MAP>;
        case 18: return k_router_bwd<SCORE, 18, HAS_MAP>;
    }
    return nullptr;
}
}  // namespace

int launch_bwd(int score_fn, int nv_idx, const float* g, const float* s, const uint8_t* m, float* dx, int T,
               int E, int renorm, float scaling, bool vec, cudaStream_t st)
{
    BwdFn f;
    if (score_fn == kSoftmax) f = m ? bwd_kernel<kSoftmax, true>(nv_idx) : bwd_kernel<kSoftmax, false>(nv_idx);
    else f = m ? bwd_kernel<kSigmoid, true>(nv_idx) : bwd_kernel<kSigmoid, false>(nv_idx);
    if (!f) return cudaErrorInvalidValue;
    const long long ctas_needed = (static_cast<long long>(T) + kBwdThreads / 32 - 1) / (kBwdThreads / 32);
    const int grid = persistent_grid(reinterpret_cast<const void*>(f), kBwdThreads, 0, ctas_needed);
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    f<<<grid, kBwdThreads, 0, st>>>(g, s, m, dx, T, E, renorm, scaling, vec ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace mr
