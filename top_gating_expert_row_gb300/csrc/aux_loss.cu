// The aux-loss scalar and its helpers (TransformerEngine PR 3012 names the
// fused_moe_aux_loss kernel, which consumes the scores and routing map of
// fused_score_for_moe_aux_loss; the pages print no formula, and the loss is
// read as the switch-style load-balancing loss):
//
//   loss = C * sum_e tokens_per_expert[e] * sum_t probs[t][e],
//   C    = coeff * E / (topk * N^2),  N = total_num_tokens
//   d loss / d probs[t][e] = C * tokens_per_expert[e] * grad_loss
//
//   k_aux_colsum        per-column sums of probs over a chunk of rows, one
//                       128-column slab per CTA (8 warps over the rows, lane l
//                       on columns 4l..4l+3), written to the caller's workspace
//   k_aux_loss_final    one CTA: sums the chunks of every column in a fixed
//                       order, forms the dot product with the counts in fp64
//   k_aux_loss_bwd      the broadcast gradient, one store stream
//   k_tokens_per_expert per-column counts of a routing map
//
// Column sums are Kahan-compensated fp32 in a fixed order, so the loss is
// deterministic and within a few ulp of the exact sum.
#include <algorithm>

#include "internal.h"

namespace mr {

namespace {

constexpr int kAuxWarps = kAuxThreads / 32;

struct Kahan {
    float s = 0.0f, c = 0.0f;
    __device__ __forceinline__ void add(float x)
    {
        const float y = __fsub_rn(x, c);
        const float t = __fadd_rn(s, y);
        c = __fsub_rn(__fsub_rn(t, s), y);
        s = t;
    }
};

__global__ void __launch_bounds__(kAuxThreads) k_aux_colsum(const float* __restrict__ probs, int T, int E,
                                                            int rows_per_chunk, int vec, float* __restrict__ partial)
{
    __shared__ float red[kAuxWarps][128];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col0 = blockIdx.x * 128 + lane * 4;
    const int t0 = blockIdx.y * rows_per_chunk;
    const int t1 = min(T, t0 + rows_per_chunk);
    const bool whole = vec && col0 + 4 <= E;
    Kahan acc[4];
    auto load = [&](int t, float (&x)[4]) {
        const float* p = probs + static_cast<size_t>(t) * E + col0;
        if (whole) {
            const float4 q = __ldcs(reinterpret_cast<const float4*>(p));
            x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) x[c] = col0 + c < E ? __ldcs(p + c) : 0.0f;
        }
    };
    // rows t0 + warp, + 8, ...; four rows in flight per warp
    int t = t0 + warp;
    for (; t + 3 * kAuxWarps < t1; t += 4 * kAuxWarps) {
        float x[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) load(t + u * kAuxWarps, x[u]);
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[c].add(x[u][c]);
    }
    for (; t < t1; t += kAuxWarps) {
        float x[4];
        load(t, x);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[c].add(x[c]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) red[warp][lane * 4 + c] = acc[c].s;
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (col0 + c >= E) break;
            Kahan k;
            for (int w = 0; w < kAuxWarps; ++w) k.add(red[w][lane * 4 + c]);
            partial[static_cast<size_t>(blockIdx.y) * E + col0 + c] = k.s;
        }
    }
}

__global__ void __launch_bounds__(1024) k_aux_loss_final(const float* __restrict__ partial, int R, int E,
                                                         const int32_t* __restrict__ tokens_per_expert, double C,
                                                         float* loss)
{
    __shared__ double red[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    double acc = 0.0;
    for (int col = threadIdx.x; col < E; col += blockDim.x) {
        Kahan k;
        for (int r = 0; r < R; ++r) k.add(partial[static_cast<size_t>(r) * E + col]);
        acc += static_cast<double>(k.s) * static_cast<double>(tokens_per_expert[col]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(kFull, acc, o);
    if (lane == 0) red[warp] = acc;
    __syncthreads();
    if (warp == 0) {
        double v = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
        if (lane == 0) loss[0] = static_cast<float>(v * C);
    }
}

__global__ void __launch_bounds__(kAuxThreads) k_aux_loss_bwd(const int32_t* __restrict__ tokens_per_expert,
                                                              const float* __restrict__ grad_loss, double C, int T,
                                                              int E, int rows_per_chunk, int vec,
                                                              float* __restrict__ grad_probs)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col0 = blockIdx.x * 128 + lane * 4;
    const int t0 = blockIdx.y * rows_per_chunk;
    const int t1 = min(T, t0 + rows_per_chunk);
    const double g = static_cast<double>(grad_loss[0]);
    float f[4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
        f[c] = col0 + c < E ? static_cast<float>(C * static_cast<double>(tokens_per_expert[col0 + c]) * g) : 0.0f;
    const bool whole = vec && col0 + 4 <= E;
    for (int t = t0 + warp; t < t1; t += kAuxWarps) {
        float* p = grad_probs + static_cast<size_t>(t) * E + col0;
        if (whole) {
            *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (col0 + c < E) p[c] = f[c];
        }
    }
}

__global__ void __launch_bounds__(kAuxThreads) k_tokens_per_expert(const uint8_t* __restrict__ map, int T, int E,
                                                                   int rows_per_chunk, int vec, int32_t* out)
{
    __shared__ uint32_t red[kAuxWarps][128];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col0 = blockIdx.x * 128 + lane * 4;
    const int t0 = blockIdx.y * rows_per_chunk;
    const int t1 = min(T, t0 + rows_per_chunk);
    const bool whole = vec && col0 + 4 <= E;
    uint32_t cnt[4] = {0u, 0u, 0u, 0u};
    for (int t = t0 + warp; t < t1; t += kAuxWarps) {
        const uint8_t* p = map + static_cast<size_t>(t) * E + col0;
        if (whole) {
            const uint32_t w = __ldcs(reinterpret_cast<const unsigned int*>(p));
#pragma unroll
            for (int c = 0; c < 4; ++c) cnt[c] += ((w >> (8 * c)) & 0xffu) != 0u;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) cnt[c] += (col0 + c < E && p[c] != 0) ? 1u : 0u;
        }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) red[warp][lane * 4 + c] = cnt[c];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (col0 + c >= E) break;
            uint32_t s = 0u;
            for (int w = 0; w < kAuxWarps; ++w) s += red[w][lane * 4 + c];
            if (s) atomicAdd(reinterpret_cast<unsigned int*>(out + col0 + c), s);
        }
    }
}

}  // namespace

int aux_chunks(long long T) { return static_cast<int>(T <= 0 ? 0 : std::min<long long>((T + kAuxRowsPerChunk - 1) / kAuxRowsPerChunk, kAuxMaxChunks)); }

int launch_aux_loss_fwd(const float* probs, const int32_t* tokens_per_expert, int T, int E, double C, float* loss,
                        float* partial, cudaStream_t st)
{
    const int R = aux_chunks(T);
    const int S = (E + 127) / 128;
    if (R > 0) {
        const int rows = (T + R - 1) / R;
        const int vec = (E % 4 == 0) && (reinterpret_cast<uintptr_t>(probs) % 16 == 0);
        k_aux_colsum<<<dim3(S, R), kAuxThreads, 0, st>>>(probs, T, E, rows, vec, partial);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    k_aux_loss_final<<<1, 1024, 0, st>>>(partial, R, E, tokens_per_expert, C, loss);
    return cudaGetLastError();
}

int launch_aux_loss_bwd(const int32_t* tokens_per_expert, const float* grad_loss, int T, int E, double C,
                        float* grad_probs, cudaStream_t st)
{
    if (T <= 0) return cudaSuccess;
    const int R = std::min((T + kAuxRowsPerChunk - 1) / kAuxRowsPerChunk, 4096);
    const int rows = (T + R - 1) / R;
    const int S = (E + 127) / 128;
    const int vec = (E % 4 == 0) && (reinterpret_cast<uintptr_t>(grad_probs) % 16 == 0);
    k_aux_loss_bwd<<<dim3(S, R), kAuxThreads, 0, st>>>(tokens_per_expert, grad_loss, C, T, E, rows, vec, grad_probs);
    return cudaGetLastError();
}

int launch_tokens_per_expert(const uint8_t* map, int T, int E, int32_t* out, cudaStream_t st)
{
    cudaError_t e = cudaMemsetAsync(out, 0, static_cast<size_t>(E) * sizeof(int32_t), st);
    if (e != cudaSuccess || T <= 0) return e;
    const int R = std::min((T + kAuxRowsPerChunk - 1) / kAuxRowsPerChunk, 4096);
    const int rows = (T + R - 1) / R;
    const int S = (E + 127) / 128;
    const int vec = (E % 4 == 0) && (reinterpret_cast<uintptr_t>(map) % 4 == 0);
    k_tokens_per_expert<<<dim3(S, R), kAuxThreads, 0, st>>>(map, T, E, rows, vec, out);
    return cudaGetLastError();
}

}  // namespace mr
