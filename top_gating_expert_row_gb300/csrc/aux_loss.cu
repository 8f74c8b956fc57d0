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

__global__ void __launch_bounds__(kAuxThreads) k_aux_colsum(const float* probs, int T, int E,
                                                            int rows_per_chunk, int vec, float* partial,
                                                            unsigned int* done)
{
    pdl_trigger_small();
    pdl_wait();
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
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *done = 0u;  // for k_aux_loss_final
    // rows t0 + warp, + 8, ...; eight rows in flight per warp
    int t = t0 + warp;
    for (; t + 7 * kAuxWarps < t1; t += 8 * kAuxWarps) {
        float x[8][4];
#pragma unroll
        for (int u = 0; u < 8; ++u) load(t + u * kAuxWarps, x[u]);
#pragma unroll
        for (int u = 0; u < 8; ++u)
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

// One CTA per 128-column slab: the slab's column sums (chunks in a fixed
// order), their dot product with the counts in fp64, written to `dots`; the
// CTA that finishes last (a counter, no waiting) adds the slab results in slab
// order and writes the loss.
__global__ void __launch_bounds__(kAuxThreads) k_aux_loss_final(const float* partial, int R, int E,
                                                                const int32_t* tokens_per_expert,
                                                                double C, double* dots, unsigned int* done,
                                                                float* loss)
{
    pdl_trigger_small();
    pdl_wait();
    __shared__ float red[kAuxWarps][128];
    __shared__ bool last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col0 = blockIdx.x * 128 + lane * 4;
    Kahan acc[4];
    // four chunks per warp at a time, all loads issued before the adds
    for (int r0 = warp; r0 < R; r0 += 4 * kAuxWarps) {
        float x[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int r = r0 + u * kAuxWarps;
            const float* p = partial + static_cast<size_t>(r) * E + col0;
#pragma unroll
            for (int c = 0; c < 4; ++c) x[u][c] = (r < R && col0 + c < E) ? __ldcg(p + c) : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (r0 + u * kAuxWarps < R)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[c].add(x[u][c]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) red[warp][lane * 4 + c] = acc[c].s;
    __syncthreads();
    if (warp == 0) {
        double d = 0.0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if (col0 + c >= E) break;
            Kahan k;
            for (int w = 0; w < kAuxWarps; ++w) k.add(red[w][lane * 4 + c]);
            d += static_cast<double>(k.s) * static_cast<double>(tokens_per_expert[col0 + c]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(kFull, d, o);
        if (lane == 0) {
            dots[blockIdx.x] = d;
            __threadfence();
            last = atomicAdd(done, 1u) == gridDim.x - 1;
        }
    }
    __syncthreads();
    if (last && threadIdx.x == 0) {
        __threadfence();
        double v = 0.0;
        for (unsigned int b = 0; b < gridDim.x; ++b) v += __ldcg(dots + b);
        loss[0] = static_cast<float>(v * C);
    }
}

__global__ void __launch_bounds__(kAuxThreads) k_aux_loss_bwd(const int32_t* tokens_per_expert,
                                                              const float* grad_loss, double C, int T,
                                                              int E, int rows_per_chunk, int vec,
                                                              float* grad_probs)
{
    pdl_trigger_small();
    pdl_wait();
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
    const float4 f4 = make_float4(f[0], f[1], f[2], f[3]);
    int t = t0 + warp;
    if (whole) {
        for (; t + 3 * kAuxWarps < t1; t += 4 * kAuxWarps) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                *reinterpret_cast<float4*>(grad_probs + static_cast<size_t>(t + u * kAuxWarps) * E + col0) = f4;
        }
    }
    for (; t < t1; t += kAuxWarps) {
        float* p = grad_probs + static_cast<size_t>(t) * E + col0;
        if (whole) {
            *reinterpret_cast<float4*>(p) = f4;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (col0 + c < E) p[c] = f[c];
        }
    }
}

// Counts: a CTA covers a 512-column slab (lane l on columns 16l..16l+15, one
// 16-byte load per row) of a chunk of rows, eight rows in flight per warp; the
// warps' counts are added in shared memory and then once per column into `out`.
__global__ void __launch_bounds__(kAuxThreads) k_tokens_per_expert(const uint8_t* map, int T, int E,
                                                                   int rows_per_chunk, int vec, int32_t* out)
{
    pdl_trigger_small();
    pdl_wait();
    __shared__ uint32_t red[kAuxWarps][512];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col0 = blockIdx.x * 512 + lane * 16;
    const int t0 = blockIdx.y * rows_per_chunk;
    const int t1 = min(T, t0 + rows_per_chunk);
    const bool whole = vec && col0 + 16 <= E;
    uint32_t cnt[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) cnt[c] = 0u;
    // Counting in SIMD-within-a-register form: each byte is folded to 0/1 and
    // four bytes are added at once into byte-wide counters (packed[i]), which
    // are moved into cnt before any of them can reach 256.
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
    int held = 0;  // rows added into packed since the last flush
    auto flush = [&]() {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int b = 0; b < 4; ++b) cnt[4 * i + b] += (packed[i] >> (8 * b)) & 0xffu;
            packed[i] = 0u;
        }
        held = 0;
    };
    auto add = [&](const uint4& q) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t f = w[i] | (w[i] >> 4);
            f |= f >> 2;
            f |= f >> 1;
            packed[i] += f & 0x01010101u;
        }
    };
    int t = t0 + warp;
    if (whole) {
        for (; t + 7 * kAuxWarps < t1; t += 8 * kAuxWarps) {
            uint4 q[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                q[u] = __ldcs(reinterpret_cast<const uint4*>(map + static_cast<size_t>(t + u * kAuxWarps) * E + col0));
#pragma unroll
            for (int u = 0; u < 8; ++u) add(q[u]);
            held += 8;
            if (held > 240) flush();
        }
    }
    for (; t < t1; t += kAuxWarps) {
        const uint8_t* p = map + static_cast<size_t>(t) * E + col0;
        if (whole) {
            add(__ldcs(reinterpret_cast<const uint4*>(p)));
            if (++held > 240) flush();
        } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) cnt[c] += (col0 + c < E && p[c] != 0) ? 1u : 0u;
        }
    }
    flush();
#pragma unroll
    for (int c = 0; c < 16; ++c) red[warp][lane * 16 + c] = cnt[c];
    __syncthreads();
    for (int i = threadIdx.x; i < 512; i += kAuxThreads) {
        const int col = blockIdx.x * 512 + i;
        if (col >= E) break;
        uint32_t sum = 0u;
#pragma unroll
        for (int w = 0; w < kAuxWarps; ++w) sum += red[w][i];
        if (sum) atomicAdd(reinterpret_cast<unsigned int*>(out + col), sum);
    }
}

// Counts of rows with 16-byte aligned map rows: a CTA covers a 64-column slab of
// a chunk of rows; lane (r, c) of a warp (r = lane / 4, c = lane % 4) loads the
// 16 bytes of columns 16c .. 16c+15 of row 8i + r, so one warp load covers 8
// rows and every row's slab is one 64-byte segment. The lanes' byte-wise counts
// are added across the 8 row lanes by shuffles (two counts per 32-bit word),
// across the warps in shared memory, and once per column into `out`: a chunk of
// 512 rows or more per CTA, so a column takes few atomics.
__global__ void __launch_bounds__(kAuxThreads) k_tokens_per_expert_slab(const uint8_t* map, int T, int E,
                                                                        int rows_per_chunk, int32_t* out)
{
    pdl_trigger_small();
    pdl_wait();
    __shared__ uint32_t red[kAuxWarps][64];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = lane >> 2, c = lane & 3;
    const int col0 = blockIdx.x * 64 + c * 16;
    const bool live = col0 < E;  // E is a multiple of 16: a lane's 16 columns are all in or all out
    const int t0 = blockIdx.y * rows_per_chunk;
    const int t1 = min(T, t0 + rows_per_chunk);
    uint32_t cnt[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) cnt[i] = 0u;
    uint32_t packed[4] = {0u, 0u, 0u, 0u};  // byte-wide counters, flushed before any reaches 256
    int held = 0;
    auto flush = [&]() {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int b = 0; b < 4; ++b) cnt[4 * i + b] += (packed[i] >> (8 * b)) & 0xffu;
            packed[i] = 0u;
        }
        held = 0;
    };
    auto add = [&](const uint4& q) {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t f = w[i] | (w[i] >> 4);
            f |= f >> 2;
            f |= f >> 1;
            packed[i] += f & 0x01010101u;
        }
    };
    const uint8_t* base = map + col0;
    // rows t0 + 8 (warp + 8 j) + r: eight loads in flight per lane
    constexpr int kStep = 8 * kAuxWarps;  // rows per CTA-wide load
    int t = t0 + 8 * warp + r;
    if (live) {
        for (; t + 7 * kStep < t1; t += 8 * kStep) {
            uint4 q[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                q[u] = __ldcs(reinterpret_cast<const uint4*>(base + static_cast<size_t>(t + u * kStep) * E));
#pragma unroll
            for (int u = 0; u < 8; ++u) add(q[u]);
            held += 8;
            if (held > 248) flush();
        }
        for (; t < t1; t += kStep) {
            add(__ldcs(reinterpret_cast<const uint4*>(base + static_cast<size_t>(t) * E)));
            if (++held > 248) flush();
        }
    }
    flush();
    // the 8 row lanes of each column group: counts of one chunk stay below 2^16,
    // so two travel in one word
    uint32_t two[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) two[i] = cnt[2 * i] | (cnt[2 * i + 1] << 16);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i) two[i] += __shfl_xor_sync(kFull, two[i], o);
    if (r == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            red[warp][c * 16 + 2 * i] = two[i] & 0xffffu;
            red[warp][c * 16 + 2 * i + 1] = two[i] >> 16;
        }
    }
    __syncthreads();
    if (threadIdx.x < 64) {
        const int col = blockIdx.x * 64 + threadIdx.x;
        uint32_t sum = 0u;
#pragma unroll
        for (int w = 0; w < kAuxWarps; ++w) sum += red[w][threadIdx.x];
        if (col < E && sum) atomicAdd(reinterpret_cast<unsigned int*>(out + col), sum);
    }
}

}  // namespace

int aux_chunks(long long T)
{
    return static_cast<int>(T <= 0 ? 0
                                   : std::min<long long>((T + kAuxRowsPerChunk - 1) / kAuxRowsPerChunk, kAuxMaxChunks));
}

size_t aux_workspace_bytes(long long T, int E)
{
    if (T <= 0) return 0;
    const size_t slabs = static_cast<size_t>((E + 127) / 128);
    const size_t part = (static_cast<size_t>(aux_chunks(T)) * E * sizeof(float) + 15) / 16 * 16;
    return part + slabs * sizeof(double) + 16;
}

int launch_aux_loss_fwd(const float* probs, const int32_t* tokens_per_expert, int T, int E, double C, float* loss,
                        void* workspace, cudaStream_t st)
{
    if (T <= 0) return cudaMemsetAsync(loss, 0, sizeof(float), st);
    const int R = aux_chunks(T);
    const int S = (E + 127) / 128;
    float* partial = static_cast<float*>(workspace);
    const size_t part = (static_cast<size_t>(R) * E * sizeof(float) + 15) / 16 * 16;
    double* dots = reinterpret_cast<double*>(static_cast<unsigned char*>(workspace) + part);
    unsigned int* done = reinterpret_cast<unsigned int*>(dots + S);
    const int rows = (T + R - 1) / R;
    const int vec = (E % 4 == 0) && (reinterpret_cast<uintptr_t>(probs) % 16 == 0);
    const int e = launch_kernel(k_aux_colsum, dim3(S, R), dim3(kAuxThreads), 0, st, 0, probs, T, E, rows, vec, partial,
                                done);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_aux_loss_final, dim3(S), dim3(kAuxThreads), 0, st, 0, partial, R, E, tokens_per_expert, C,
                         dots, done, loss);
}

int launch_aux_loss_bwd(const int32_t* tokens_per_expert, const float* grad_loss, int T, int E, double C,
                        float* grad_probs, cudaStream_t st)
{
    if (T <= 0) return cudaSuccess;
    const int R = std::min((T + kAuxRowsPerChunk - 1) / kAuxRowsPerChunk, 4096);
    const int rows = (T + R - 1) / R;
    const int S = (E + 127) / 128;
    const int vec = (E % 4 == 0) && (reinterpret_cast<uintptr_t>(grad_probs) % 16 == 0);
    return launch_kernel(k_aux_loss_bwd, dim3(S, R), dim3(kAuxThreads), 0, st, 0, tokens_per_expert, grad_loss, C, T, E,
                         rows, vec, grad_probs);
}

int launch_tokens_per_expert(const uint8_t* map, int T, int E, int32_t* out, cudaStream_t st)
{
    cudaError_t e = cudaMemsetAsync(out, 0, static_cast<size_t>(E) * sizeof(int32_t), st);
    if (e != cudaSuccess || T <= 0) return e;
    const int vec = (E % 16 == 0) && (reinterpret_cast<uintptr_t>(map) % 16 == 0);
    if (vec) {
        // 64-column slabs, chunks of at least 512 rows and at most 65535 (a
        // chunk's counts stay below 2^16), about four CTAs per SM in all
        const int S = (E + 63) / 64;
        int dev = 0, sms = 152;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const long long want = std::max<long long>(1, (4LL * sms + S - 1) / S);
        const long long by_rows = std::max<long long>(1, (static_cast<long long>(T) + 511) / 512);
        const long long need = (static_cast<long long>(T) + 65534) / 65535;
        const int R = static_cast<int>(std::max(need, std::min(want, by_rows)));
        const int rows = static_cast<int>((static_cast<long long>(T) + R - 1) / R);
        return launch_kernel(k_tokens_per_expert_slab, dim3(S, R), dim3(kAuxThreads), 0, st, 0, map, T, E, rows,
                             out);
    }
    constexpr int kRows = 128;
    const int R = std::min((T + kRows - 1) / kRows, 8192);
    const int rows = (T + R - 1) / R;
    const int S = (E + 511) / 512;
    return launch_kernel(k_tokens_per_expert, dim3(S, R), dim3(kAuxThreads), 0, st, 0, map, T, E, rows, vec, out);
}

}  // namespace mr
