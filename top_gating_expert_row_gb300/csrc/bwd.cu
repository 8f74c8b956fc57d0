// Router backward and aux-score backward (TransformerEngine PR 3012, "Two-pass
// fused design": pass 1 reduces the row sums in registers with warp
// all-reduces, pass 2 forms each element's gradient; no shared-memory buffer).
//
// One warp per token row, the row held in registers (g, s, routing map):
//   ds_i = c * m_i * g_i                         (no renorm)
//   ds_i = (c * m_i / A) * (g_i - B / A)          (renorm; A = sum m s, B = sum m s g)
//   softmax: dx_i = s_i * (ds_i - sum_j s_j ds_j);  sigmoid: dx_i = ds_i * s_i * (1 - s_i)
// The aux-score backward is the same with m = 1, c = 1 and no renorm.
#include <type_traits>

#include "internal.h"

namespace mr {

// 4 warps, one token row per warp at a time. Rows live in registers, so
// registers bound the warps per SM; small CTAs let the occupancy reach that
// bound (bf16 grads at 166 registers: 3 CTAs = 12 warps, where one 8-warp CTA
// would leave the rest of the register file idle).
constexpr int kBwdThreads = 128;

// GradT: the dtype of grad and dx (fp32, or bf16 for bf16 logits: the
// gradient is computed in fp32 and rounded once when stored).
template <int SCORE, int NV, bool HAS_MAP, typename GradT>
__global__ void __launch_bounds__(kBwdThreads) k_router_bwd(const GradT* grad,
                                                            const float* inter,
                                                            const uint8_t* map,
                                                            GradT* dx, int T, int E,
                                                            int renorm, float c, int vec)
{
    pdl_trigger_small();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    constexpr bool kPacked = !std::is_same<GradT, float>::value;
    for (int t = blockIdx.x * nw + warp; t < T; t += gridDim.x * nw) {
        const size_t ro = static_cast<size_t>(t) * E;
        // fp32 grads go straight into d; bf16 grads stay packed (two per word)
        // until used, so every row load can be in flight at once within the
        // register budget. d then holds ds.
        float d[NV][4], s[NV][4];
        uint2 gp[NV];
        uint32_t m[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e0 = (v * 32 + lane) * 4;
            if (vec && e0 + 4 <= E) {
                if constexpr (kPacked) {
                    gp[v] = __ldcs(reinterpret_cast<const uint2*>(grad + ro + e0));
                } else {
                    const float4 a = __ldcs(reinterpret_cast<const float4*>(grad + ro + e0));
                    d[v][0] = a.x; d[v][1] = a.y; d[v][2] = a.z; d[v][3] = a.w;
                }
                const float4 b = __ldcs(reinterpret_cast<const float4*>(inter + ro + e0));
                s[v][0] = b.x; s[v][1] = b.y; s[v][2] = b.z; s[v][3] = b.w;
                m[v] = HAS_MAP ? __ldcs(reinterpret_cast<const unsigned int*>(map + ro + e0)) : 0x01010101u;
            } else {
                m[v] = 0u;
                if constexpr (kPacked) gp[v] = make_uint2(0u, 0u);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const bool in = e0 + q < E;
                    if constexpr (kPacked) {
                        const uint32_t bits = in ? __ldcs(reinterpret_cast<const unsigned short*>(grad + ro + e0 + q)) : 0u;
                        if (q < 2) gp[v].x |= bits << (16 * q);
                        else gp[v].y |= bits << (16 * (q - 2));
                    } else {
                        d[v][q] = in ? load_scalar<GradT>(grad + ro + e0 + q) : 0.0f;
                    }
                    s[v][q] = in ? __ldcs(inter + ro + e0 + q) : 0.0f;
                    const uint32_t mb = in ? (HAS_MAP ? static_cast<uint32_t>(map[ro + e0 + q] != 0) : 1u) : 0u;
                    m[v] |= mb << (8 * q);
                }
            }
        }
        // element q of chunk v of the grad row, as fp32
        auto gval = [&](int v, int q) -> float {
            if constexpr (!kPacked) {
                return d[v][q];
            } else {
                const uint32_t w = q < 2 ? gp[v].x : gp[v].y;
                return bf16_bits_to_f32((q & 1) ? (w >> 16) : (w & 0xffffu));
            }
        };
        // pass 1: row sums
        float A = 0.0f, B = 0.0f;
        if (HAS_MAP && renorm) {
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if ((m[v] >> (8 * q)) & 0xffu) {
                        A += s[v][q];
                        B += s[v][q] * gval(v, q);
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
                const float gq = gval(v, q);
                const float ds = mk ? (rn ? cA * (gq - BA) : c * gq) : 0.0f;
                d[v][q] = ds;
                if (SCORE == kSoftmax) D += s[v][q] * ds;
            }
        if (SCORE == kSoftmax) D = warp_sum(D);
        GradT* out = dx + ro;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e0 = (v * 32 + lane) * 4;
            if (e0 >= E) continue;
            float r[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                r[q] = (SCORE == kSoftmax) ? s[v][q] * (d[v][q] - D) : d[v][q] * s[v][q] * (1.0f - s[v][q]);
            if (vec && e0 + 4 <= E) {
                store4_stream<GradT>(out + e0, r);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (e0 + q < E) store_scalar<GradT>(out + e0 + q, r[q]);
            }
        }
    }
}

// Rows too wide to hold in registers (E > 2304): one warp per row, two passes
// over the row in global memory (the second mostly from L2). Pass 1 sums
// A = sum m s and B = sum m s g; the softmax correction sum_j s_j ds_j then has
// the closed form c*B without renorm and 0 with it (the renormalised weights'
// gradient sums to zero against s), and pass 2 forms each element's gradient.
template <int SCORE, bool HAS_MAP, typename GradT>
__global__ void __launch_bounds__(kBwdThreads) k_router_bwd_wide(const GradT* grad, const float* inter,
                                                                 const uint8_t* map, GradT* dx, int T, int E,
                                                                 int renorm, float c, int vec)
{
    pdl_trigger_small();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const bool rn = HAS_MAP && renorm;
    // four consecutive elements starting at e0 (g, s, m), any alignment
    auto load = [&](size_t ro, int e0, float (&g)[4], float (&sv)[4], uint32_t& m, bool first) {
        if (vec && e0 + 4 <= E) {
            if constexpr (std::is_same<GradT, float>::value) {
                const float4 a = first ? __ldcg(reinterpret_cast<const float4*>(grad + ro + e0))
                                       : __ldcs(reinterpret_cast<const float4*>(grad + ro + e0));
                g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
            } else {
                const uint2 q = first ? __ldcg(reinterpret_cast<const uint2*>(grad + ro + e0))
                                      : __ldcs(reinterpret_cast<const uint2*>(grad + ro + e0));
                g[0] = bf16_bits_to_f32(q.x & 0xffffu); g[1] = bf16_bits_to_f32(q.x >> 16);
                g[2] = bf16_bits_to_f32(q.y & 0xffffu); g[3] = bf16_bits_to_f32(q.y >> 16);
            }
            const float4 b = first ? __ldcg(reinterpret_cast<const float4*>(inter + ro + e0))
                                   : __ldcs(reinterpret_cast<const float4*>(inter + ro + e0));
            sv[0] = b.x; sv[1] = b.y; sv[2] = b.z; sv[3] = b.w;
            m = HAS_MAP ? (first ? __ldcg(reinterpret_cast<const unsigned int*>(map + ro + e0))
                                 : __ldcs(reinterpret_cast<const unsigned int*>(map + ro + e0)))
                        : 0x01010101u;
        } else {
            m = 0u;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool in = e0 + q < E;
                g[q] = in ? load_scalar<GradT>(grad + ro + e0 + q) : 0.0f;
                sv[q] = in ? inter[ro + e0 + q] : 0.0f;
                const uint32_t mb = in ? (HAS_MAP ? static_cast<uint32_t>(map[ro + e0 + q] != 0) : 1u) : 0u;
                m |= mb << (8 * q);
            }
        }
    };
    for (int t = blockIdx.x * nw + warp; t < T; t += gridDim.x * nw) {
        const size_t ro = static_cast<size_t>(t) * E;
        float A = 0.0f, B = 0.0f;
        if (rn || SCORE == kSoftmax) {
            for (int e0 = lane * 4; e0 < E; e0 += 128) {
                float g[4], sv[4];
                uint32_t m;
                load(ro, e0, g, sv, m, true);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if ((m >> (8 * q)) & 0xffu) {
                        A += sv[q];
                        B += sv[q] * g[q];
                    }
            }
            A = warp_sum(A);
            B = warp_sum(B);
        }
        const float cA = (rn && A != 0.0f) ? c / A : 0.0f;
        const float BA = (rn && A != 0.0f) ? B / A : 0.0f;
        const float D = (SCORE == kSoftmax && !rn) ? c * B : 0.0f;
        GradT* out = dx + ro;
        for (int e0 = lane * 4; e0 < E; e0 += 128) {
            float g[4], sv[4], r[4];
            uint32_t m;
            load(ro, e0, g, sv, m, false);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool mk = (m >> (8 * q)) & 0xffu;
                const float ds = mk ? (rn ? cA * (g[q] - BA) : c * g[q]) : 0.0f;
                r[q] = (SCORE == kSoftmax) ? sv[q] * (ds - D) : ds * sv[q] * (1.0f - sv[q]);
            }
            if (vec && e0 + 4 <= E) {
                store4_stream<GradT>(out + e0, r);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (e0 + q < E) store_scalar<GradT>(out + e0 + q, r[q]);
            }
        }
    }
}

namespace {
template <typename GradT>
using BwdFn = void (*)(const GradT*, const float*, const uint8_t*, GradT*, int, int, int, float, int);

// nv_idx < 0: rows wider than the register-resident buckets
template <int SCORE, bool HAS_MAP, typename GradT>
BwdFn<GradT> bwd_kernel(int nv_idx)
{
    if (nv_idx < 0) return k_router_bwd_wide<SCORE, HAS_MAP, GradT>;
    switch (kNvBuckets[nv_idx]) {
        case 1: return k_router_bwd<SCORE, 1, HAS_MAP, GradT>;
        case 2: return k_router_bwd<SCORE, 2, HAS_MAP, GradT>;
        case 3: return k_router_bwd<SCORE, 3, HAS_MAP, GradT>;
        case 4: return k_router_bwd<SCORE, 4, HAS_MAP, GradT>;
        case 6: return k_router_bwd<SCORE, 6, HAS_MAP, GradT>;
        case 8: return k_router_bwd<SCORE, 8, HAS_MAP, GradT>;
        case 12: return k_router_bwd<SCORE, 12, HAS_MAP, GradT>;
        case 18: return k_router_bwd<SCORE, 18, HAS_MAP, GradT>;
    }
    return nullptr;
}

template <typename GradT>
int launch(BwdFn<GradT> f, const GradT* g, const float* s, const uint8_t* m, GradT* dx, int T, int E, int renorm,
           float scaling, bool vec, cudaStream_t st)
{
    if (!f) return cudaErrorInvalidValue;
    const long long ctas_needed = (static_cast<long long>(T) + kBwdThreads / 32 - 1) / (kBwdThreads / 32);
    const int grid = persistent_grid(reinterpret_cast<const void*>(f), kBwdThreads, 0, ctas_needed, true);
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    return launch_kernel(f, dim3(grid), dim3(kBwdThreads), 0, st, 0, g, s, m, dx, T, E, renorm, scaling, vec ? 1 : 0);
}
}  // namespace

int launch_bwd(int score_fn, int nv_idx, const float* g, const float* s, const uint8_t* m, float* dx, int T,
               int E, int renorm, float scaling, bool vec, cudaStream_t st)
{
    BwdFn<float> f;
    if (score_fn == kSoftmax) f = m ? bwd_kernel<kSoftmax, true, float>(nv_idx) : bwd_kernel<kSoftmax, false, float>(nv_idx);
    else f = m ? bwd_kernel<kSigmoid, true, float>(nv_idx) : bwd_kernel<kSigmoid, false, float>(nv_idx);
    return launch<float>(f, g, s, m, dx, T, E, renorm, scaling, vec, st);
}

int launch_bwd_bf16(int score_fn, int nv_idx, const __nv_bfloat16* g, const float* s, const uint8_t* m,
                    __nv_bfloat16* dx, int T, int E, int renorm, float scaling, bool vec, cudaStream_t st)
{
    const BwdFn<__nv_bfloat16> f = score_fn == kSoftmax ? bwd_kernel<kSoftmax, true, __nv_bfloat16>(nv_idx)
                                                         : bwd_kernel<kSigmoid, true, __nv_bfloat16>(nv_idx);
    return launch<__nv_bfloat16>(f, g, s, m, dx, T, E, renorm, scaling, vec, st);
}

}  // namespace mr
