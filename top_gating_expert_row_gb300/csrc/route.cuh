// One token row of the router forward, computed by one warp.
//
// Follows fused_topk_with_score_function as TransformerEngine PR 3012 describes
// it (flowchart: convert to the compute type, apply the score function,
// top-k-and-mask, write probs + routing_map), rebuilt for one warp per row:
//
//   1. load     the row: lane l holds elements v*128 + 4l .. +3 for v < NV, so
//               every v is one coalesced 512 B (fp32) access; only the u32
//               selection keys stay in registers, the scores go to a per-warp
//               shared-memory row buffer
//   2. groups   (optional) group scores = sum of each group's top-m keys; the
//               topk_group best groups are kept, the others' keys set to 0
//   3. select   k_r winners by (key desc, index asc):
//               ARGMAX  - k_r rounds of warp arg-max (REDUX max/min), for small k
//               SELECT  - bisection on the key for a threshold that leaves at most
//                         `stop` candidates, compaction to shared memory, then an
//                         exact all-pairs rank of the candidates; ties at the
//                         threshold are taken in index order
//   4. weights  renormalise over the winners and scale
//   5. emit     dense probs / routing_map / intermediate (compact topk_idx/w:
//               emit_compact)
//
// Both selection paths produce the identical winner list. SET (threshold select
// only; for calls without compact outputs) finds the winners as a set: the
// bisection runs to the exact threshold and the winners are patched straight
// from the registers, with no candidate list and no ranking.
#pragma once

#include <type_traits>

#include "common.cuh"

namespace mr {

struct RouteArgs {
    const void* logits;
    const float* bias;
    void* probs;
    uint8_t* map;
    float* inter;
    int32_t* topk_idx;
    float* topk_w;
    int T, E, k_r, topk, n_shared;
    int renorm, n_group, topk_group;
    float scaling, shared_weight;
    int vec;       // rows and all arrays allow 16-byte (fp32) / 8-byte (bf16) vector access
    int prefetch;  // rows are 16-byte aligned and a multiple of 16 bytes: L2 bulk prefetch allowed
    int stop;      // SELECT: candidate capacity (>= k_r); bisection stops at or below it
    int32_t* status;      // device status word, raised to kStatusTimeout when a bounded wait gives up
    uint32_t wait_tries;  // attempts (about 1 us each) before a bounded wait gives up
    int drop_copies;      // test mode: arm the staging barriers but issue no copies
    int warm_code;        // fused decode under the launch overlap: warm-up pass before the wait
    int rung;             // SELECT: rung of the lane-maxima ladder tried as a pivot (1..32, 0: none)
};

// Byte offsets of one warp's shared-memory region (same formula on host and device).
//   vbuf     E fp32: the row's scores (softmax: exp(x - max), unnormalised; sigmoid: s)
//   win_*    k_r winners in selection order
//   cand     SELECT candidates, (key << 32 | ~index)
//   keys     E u32, group-limited selection only
//   scal     last winner's key and index, partial-tie flag
struct WarpLayout {
    int vbuf, win_idx, win_val, cand, keys, scal, bytes;
};

__host__ __device__ inline int align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline WarpLayout warp_layout(int k_r, int stop, int E, bool select, bool groups)
{
    WarpLayout L;
    int o = 0;
    L.vbuf = o; o += align16(E * 4);
    L.win_idx = o; o += align16(k_r * 4);
    L.win_val = o; o += align16(k_r * 4);
    L.cand = o; o += select ? align16(stop * 8) : 0;
    L.keys = o; o += groups ? align16(E * 4) : 0;
    L.scal = o; o += 16;
    L.bytes = o;
    return L;
}

// ---------------------------------------------------------------------------
// Group limit over keys staged in shared memory: sets to 0 the keys of every
// group that is not among the topk_group best. A group's score is the fp32 sum
// of its m largest keys, largest first. MAXM >= m bounds the per-lane list.
// ---------------------------------------------------------------------------
// group_kept: the same selection, returned as a mask of the kept groups (bit g
// set: group g is kept) without touching the keys.
// Insert k into the descending list top[0..MAXM).
template <int MAXM>
__device__ __forceinline__ void top_insert(uint32_t (&top)[MAXM], uint32_t k)
{
#pragma unroll
    for (int q = 0; q < MAXM; ++q) {
        const uint32_t hi = max(k, top[q]);
        k = min(k, top[q]);
        top[q] = hi;
    }
}

// The group selection from each lane's partial list (lanes g*lpg .. g*lpg+lpg-1
// hold group g's): merge the lists across the group's lanes, score the group
// (fp32 sum of its m largest keys, largest first), rank the G scores (ties to
// the lower group index) and return the mask of the gk best.
template <int MAXM>
__device__ __forceinline__ uint32_t group_finish(uint32_t (&top)[MAXM], int G, int lpg, int gk, int m, int lane)
{
    for (int o = 1; o < lpg; o <<= 1) {
        uint32_t other[MAXM];
#pragma unroll
        for (int i = 0; i < MAXM; ++i) other[i] = __shfl_xor_sync(kFull, top[i], o);
#pragma unroll
        for (int i = 0; i < MAXM; ++i) top_insert(top, other[i]);
    }
    float acc = float_of(top[0]);
#pragma unroll
    for (int i = 1; i < MAXM; ++i)
        if (i < m) acc = __fadd_rn(acc, float_of(top[i]));
    const uint32_t sk = key_of(acc);
    const uint32_t mine = __shfl_sync(kFull, sk, (lane < G ? lane : 0) * lpg);
    uint32_t rank = 0;
    for (int q = 0; q < G; ++q) {
        const uint32_t o = __shfl_sync(kFull, sk, q * lpg);
        rank += (o > mine) || (o == mine && q < lane);
    }
    return __ballot_sync(kFull, lane < G && rank < (uint32_t)gk);
}

// lanes per group: 32 / G rounded down to a power of 2
__device__ __forceinline__ int group_lanes(int G)
{
    const int lpg = 32 / G;
    return 1 << (31 - __clz(lpg));
}

template <int MAXM>
__device__ uint32_t group_kept(const uint32_t* skeys, int E, int G, int gk, int m, int lane)
{
    const int gs = E / G;
    const int lpg = group_lanes(G);
    const int g = lane / lpg, j = lane % lpg;
    uint32_t top[MAXM];
#pragma unroll
    for (int i = 0; i < MAXM; ++i) top[i] = 0u;
    if (g < G) {
#pragma unroll 4
        for (int i = j; i < gs; i += lpg) top_insert(top, skeys[g * gs + i]);
    }
    return group_finish(top, G, lpg, gk, m, lane);
}

// group_kept over per-chunk lists: for rows whose groups are whole chunks of 4
// keys (gs % 4 == 0), entry n = the MAXM largest of keys 4n .. 4n+3, sorted;
// group g is entries [g * gs/4, (g+1) * gs/4).
template <int MAXM>
__device__ uint32_t group_kept_entries(const uint32_t* ent, int G, int epg, int gk, int m, int lane)
{
    const int lpg = group_lanes(G);
    const int g = lane / lpg, j = lane % lpg;
    uint32_t top[MAXM];
#pragma unroll
    for (int i = 0; i < MAXM; ++i) top[i] = 0u;
    if (g < G) {
        for (int i = j; i < epg; i += lpg)
#pragma unroll
            for (int q = 0; q < MAXM; ++q) top_insert(top, ent[(g * epg + i) * MAXM + q]);
    }
    return group_finish(top, G, lpg, gk, m, lane);
}

template <int MAXM>
__device__ void group_limit(uint32_t* skeys, int E, int G, int gk, int m, int lane)
{
    const int gs = E / G;
    const uint32_t kept = group_kept<MAXM>(skeys, E, G, gk, m, lane);
    for (int q = 0; q < G; ++q)
        if (!((kept >> q) & 1u))
            for (int i = lane; i < gs; i += 32) skeys[q * gs + i] = 0u;
}

// The j-th largest (1 <= j <= 32) of the 32 lanes' values, returned to every
// lane: a bitonic sort of the warp's values (ascending by lane), then a
// broadcast from lane 32 - j.
//
// Used as a bisection pivot, the j-th largest of the lanes' row maxima bounds
// the count from below: at least j keys (each of those lanes' maxima) are >= it.
// On rows of similar entries, with m keys per lane, about
// E * (1 - ((33 - j) / 33)^(1/m)) keys are; the host picks j for the count it
// wants (route_rung), so a row with no usable previous threshold still starts
// with one pivot that usually leaves between k_r and `stop` candidates.
__device__ __forceinline__ uint32_t warp_kth_largest(uint32_t v, int j, int lane)
{
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1)
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint32_t o = __shfl_xor_sync(kFull, v, stride);
            const bool ascending = (lane & size) == 0;
            const bool lower = (lane & stride) == 0;
            v = (lower == ascending) ? min(v, o) : max(v, o);
        }
    return __shfl_sync(kFull, v, 32 - j);
}

// ---------------------------------------------------------------------------
// route_row: the whole forward for token t. Winners are left in the warp's
// shared region (win_idx / win_val = their score s, k_r entries in selection
// order); returns the factor that turns a score into its weight (dense probs
// and compact weights are both s * factor, so they agree bit for bit).
// ---------------------------------------------------------------------------
// FULL: E == 128 * NV and a.vec, so every chunk is whole and vector-aligned and
// the per-element edge tests compile away.
// Exact rank of the n candidates in selection order. Each candidate is a
// 64-bit word (key << 32 | ~index), so all are distinct and a larger word
// comes first; a candidate's rank is the number of larger words, counted
// over all pairs. Two candidates per lane per pass over the list; with
// MAXW = 3, three when more than 64 remain, so up to 96 take one pass (worth
// it only where n can exceed 64: in a fully unrolled kernel the extra code
// costs more than it saves at smaller n). Ranks below k_r go to win_idx /
// win_val (score(idx, key) gives the value); the key at rank warm_rank goes
// to *warm_key.
template <int MAXW, typename ScoreFn>
__device__ __forceinline__ void rank_candidates(const unsigned long long* cand, uint32_t n, int k_r,
                                                uint32_t warm_rank, int lane, uint32_t* win_idx, float* win_val,
                                                uint32_t* warm_key, ScoreFn score)
{
    auto pass = [&](uint32_t b, auto wc) {
        constexpr int W = decltype(wc)::value;
        unsigned long long c[W];
        uint32_t r[W];
#pragma unroll
        for (int h = 0; h < W; ++h) {
            const uint32_t i = b + 32u * h + lane;
            c[h] = (i < n) ? cand[i] : 0ull;
            r[h] = 0u;
        }
#pragma unroll 8
        for (uint32_t q = 0; q < n; ++q) {
            const unsigned long long cq = cand[q];
#pragma unroll
            for (int h = 0; h < W; ++h) r[h] += (cq > c[h]);
        }
#pragma unroll
        for (int h = 0; h < W; ++h) {
            const uint32_t i = b + 32u * h + lane;
            if (i < n) {
                const uint32_t idx = ~static_cast<uint32_t>(c[h]);
                const uint32_t kk = static_cast<uint32_t>(c[h] >> 32);
                if (r[h] < static_cast<uint32_t>(k_r)) {
                    win_idx[r[h]] = idx;
                    win_val[r[h]] = score(idx, kk);
                }
                if (r[h] == warm_rank) *warm_key = kk;
            }
        }
    };
    static_assert(MAXW == 2 || MAXW == 3, "two or three candidates per lane");
    if constexpr (MAXW == 3) {
        uint32_t b = 0;
        for (; b < n && n - b > 64u; b += 96u) pass(b, std::integral_constant<int, 3>{});
        if (b < n) pass(b, std::integral_constant<int, 2>{});
    } else {
        for (uint32_t b = 0; b < n; b += 64u) pass(b, std::integral_constant<int, 2>{});
    }
}

template <int SCORE, typename InT, int NV, bool SELECT, bool FULL = false, int RANKW = 2, bool SET = false>
__device__ __forceinline__ float route_row(const RouteArgs& a, int t, unsigned char* wsm,
                                           const WarpLayout& L, int lane, uint32_t& warm)
{
    static_assert(!SET || SELECT, "the set-only selection is a form of the threshold select");
    float* vbuf = reinterpret_cast<float*>(wsm + L.vbuf);
    uint32_t* win_idx = reinterpret_cast<uint32_t*>(wsm + L.win_idx);
    float* win_val = reinterpret_cast<float*>(wsm + L.win_val);
    uint32_t* scal = reinterpret_cast<uint32_t*>(wsm + L.scal);
    const int E = a.E;
    const int k_r = a.k_r;
    const InT* row = static_cast<const InT*>(a.logits) + static_cast<size_t>(t) * E;
    const int lane4 = lane * 4;
    // a chunk (4 consecutive elements) is either whole or partly past E
    auto whole = [&](int v) { return FULL || v * 128 + lane4 + 4 <= E; };
    auto inside = [&](int v, int c) { return FULL || v * 128 + lane4 + c < E; };
    const bool vec = FULL || a.vec;

    uint32_t key[NV][4];
    float vmul = 1.0f;  // vbuf * vmul = s
    uint32_t kmax;
    uint32_t lane_max;  // the largest of this lane's keys

    // 1. load, selection keys, scores into vbuf; padding keys are 0
    {
        float x[NV][4];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e0 = v * 128 + lane4;
            if (vec && whole(v)) {
                load4<InT>(row + e0, x[v]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) x[v][c] = inside(v, c) ? load_scalar<InT>(row + e0 + c) : 0.0f;
            }
        }
        if (SCORE == kSoftmax) {
            // keys (4 independent max chains), raw logits to vbuf
            uint32_t lm[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int v = 0; v < NV; ++v) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    key[v][c] = inside(v, c) ? key_of(x[v][c]) : 0u;
                    lm[c] = max(lm[c], key[v][c]);
                }
                const int e0 = v * 128 + lane4;
                if (whole(v)) {
                    *reinterpret_cast<float4*>(vbuf + e0) = make_float4(x[v][0], x[v][1], x[v][2], x[v][3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (inside(v, c)) vbuf[e0 + c] = x[v][c];
                }
            }
            lane_max = max(max(lm[0], lm[1]), max(lm[2], lm[3]));
            kmax = __reduce_max_sync(kFull, lane_max);
            const float m = float_of(kmax);
            // exp(x - max) in place over the row buffer (exp_value: only the value
            // matters here); a rolled loop keeps the code short (the row's chunks
            // all run through the same instructions)
            float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 2
            for (int v = 0; v < NV; ++v) {
                const int e0 = v * 128 + lane4;
                if (whole(v)) {
                    // packed fp32x2 (bit-identical to exp_value / __fadd_rn per value);
                    // x - m as x + (-m), the same IEEE result
                    const float4 q = *reinterpret_cast<const float4*>(vbuf + e0);
                    const float2 negm = make_float2(-m, -m);
                    const float2 e01 = exp_value2(__fadd2_rn(make_float2(q.x, q.y), negm));
                    const float2 e23 = exp_value2(__fadd2_rn(make_float2(q.z, q.w), negm));
                    const float2 s01 = __fadd2_rn(make_float2(sum[0], sum[1]), e01);
                    const float2 s23 = __fadd2_rn(make_float2(sum[2], sum[3]), e23);
                    sum[0] = s01.x; sum[1] = s01.y; sum[2] = s23.x; sum[3] = s23.y;
                    *reinterpret_cast<float4*>(vbuf + e0) = make_float4(e01.x, e01.y, e23.x, e23.y);
                } else {
                    for (int c = 0; c < 4; ++c)
                        if (inside(v, c)) {
                            const float ev = exp_value(__fsub_rn(vbuf[e0 + c], m));
                            vbuf[e0 + c] = ev;
                            sum[c] = __fadd_rn(sum[c], ev);
                        }
                }
            }
            vmul = __frcp_rn(warp_sum(__fadd_rn(__fadd_rn(sum[0], sum[1]), __fadd_rn(sum[2], sum[3]))));
        } else {
            uint32_t lm[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int e0 = v * 128 + lane4;
                float b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (a.bias) {
                    if (vec && whole(v)) {
                        const float4 q = __ldcg(reinterpret_cast<const float4*>(a.bias + e0));
                        b[0] = q.x; b[1] = q.y; b[2] = q.z; b[3] = q.w;
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) b[c] = inside(v, c) ? __ldcg(a.bias + e0 + c) : 0.0f;
                    }
                }
                const float2 s01 = sigmoid_f32x2(make_float2(x[v][0], x[v][1]));
                const float2 s23 = sigmoid_f32x2(make_float2(x[v][2], x[v][3]));
                float sv[4] = {s01.x, s01.y, s23.x, s23.y};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    key[v][c] = inside(v, c) ? key_of(a.bias ? __fadd_rn(sv[c], b[c]) : sv[c]) : 0u;
                    lm[c] = max(lm[c], key[v][c]);
                }
                if (whole(v)) {
                    *reinterpret_cast<float4*>(vbuf + e0) = make_float4(sv[0], sv[1], sv[2], sv[3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (inside(v, c)) vbuf[e0 + c] = sv[c];
                }
            }
            lane_max = max(max(lm[0], lm[1]), max(lm[2], lm[3]));
            kmax = __reduce_max_sync(kFull, lane_max);
        }
    }

    // 2. group limit (keys staged through shared memory)
    if (a.n_group > 0) {
        uint32_t* sk = reinterpret_cast<uint32_t*>(wsm + L.keys);
        const int m = k_r / a.topk_group;
        const uint32_t gs = static_cast<uint32_t>(E / a.n_group);
        uint32_t kept;
        // An index's group n / d is taken as umulhi(n, ceil(2^32 / d)), exact for
        // n and d below 2^12 (d = 1: the group is n itself).
        auto group_of = [](uint32_t n, uint32_t d, uint32_t inv) { return d > 1u ? __umulhi(n, inv) : n; };
        if (FULL && (gs & 3u) == 0u && m <= 4) {
            // groups of whole chunks: each lane's chunk v lies in one group, so
            // the lane stages the m largest of its 4 keys (entry 32 v + lane) and
            // the group pass merges gs / 4 short lists instead of gs keys
            auto stage = [&](auto mc) {
                constexpr int M = decltype(mc)::value;
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    uint32_t top[M];
#pragma unroll
                    for (int i = 0; i < M; ++i) top[i] = 0u;
#pragma unroll
                    for (int c = 0; c < 4; ++c) top_insert(top, key[v][c]);
#pragma unroll
                    for (int i = 0; i < M; ++i) sk[(v * 32 + lane) * M + i] = top[i];
                }
                __syncwarp();
                return group_kept_entries<M>(sk, a.n_group, static_cast<int>(gs >> 2), a.topk_group, m, lane);
            };
            if (m <= 1) kept = stage(std::integral_constant<int, 1>{});
            else if (m <= 2) kept = stage(std::integral_constant<int, 2>{});
            else kept = stage(std::integral_constant<int, 4>{});
        } else {
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int e0 = v * 128 + lane4;
                if (whole(v)) {
                    *reinterpret_cast<uint4*>(sk + e0) = make_uint4(key[v][0], key[v][1], key[v][2], key[v][3]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (inside(v, c)) sk[e0 + c] = key[v][c];
                }
            }
            __syncwarp();
            if (m <= 1) kept = group_kept<1>(sk, E, a.n_group, a.topk_group, m, lane);
            else if (m <= 2) kept = group_kept<2>(sk, E, a.n_group, a.topk_group, m, lane);
            else if (m <= 4) kept = group_kept<4>(sk, E, a.n_group, a.topk_group, m, lane);
            else kept = group_kept<8>(sk, E, a.n_group, a.topk_group, m, lane);
        }
        // the keys are still in registers: drop those of the groups not kept
        uint32_t lmax = 0u;
        if (FULL && (gs & 3u) == 0u) {
            // a chunk's 4 keys share one group: one division per chunk
            const uint32_t epg = gs >> 2;
            const uint32_t inv = epg > 1u ? 0xffffffffu / epg + 1u : 0u;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const bool keep = (kept >> group_of(static_cast<uint32_t>(v * 32 + lane), epg, inv)) & 1u;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    key[v][c] = keep ? key[v][c] : 0u;
                    lmax = max(lmax, key[v][c]);
                }
            }
        } else {
            const uint32_t inv_gs = gs > 1u ? 0xffffffffu / gs + 1u : 0u;
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t e = static_cast<uint32_t>(v * 128 + lane4 + c);
                    const bool keep = e < static_cast<uint32_t>(E) && ((kept >> group_of(e, gs, inv_gs)) & 1u);
                    key[v][c] = keep ? key[v][c] : 0u;
                    lmax = max(lmax, key[v][c]);
                }
        }
        lane_max = lmax;
        kmax = __reduce_max_sync(kFull, lmax);
        __syncwarp();  // the staged keys are read no more; the region may be reused
    }

    // dense rows of step 5: intermediate = s; probs and routing_map as zero
    // vectors (the winners are patched in afterwards, after a __syncwarp)
    InT* prow = a.probs ? static_cast<InT*>(a.probs) + static_cast<size_t>(t) * E : nullptr;
    uint8_t* mrow = a.map ? a.map + static_cast<size_t>(t) * E : nullptr;
    float* irow = a.inter ? a.inter + static_cast<size_t>(t) * E : nullptr;
    auto dense_rows = [&]() {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e0 = v * 128 + lane4;
            if (!FULL && e0 >= E) continue;
            if (vec && whole(v)) {
                if (irow) {
                    const float4 q = *reinterpret_cast<const float4*>(vbuf + e0);
                    const float2 xy = __fmul2_rn(make_float2(q.x, q.y), make_float2(vmul, vmul));
                    const float2 zw = __fmul2_rn(make_float2(q.z, q.w), make_float2(vmul, vmul));
                    *reinterpret_cast<float4*>(irow + e0) = make_float4(xy.x, xy.y, zw.x, zw.y);
                }
                if (prow) {
                    const float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    store4<InT>(prow + e0, z);
                }
                if (mrow) *reinterpret_cast<uint32_t*>(mrow + e0) = 0u;
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (!inside(v, c)) break;
                    if (irow) irow[e0 + c] = __fmul_rn(vbuf[e0 + c], vmul);
                    if (prow) store_scalar<InT>(prow + e0 + c, 0.0f);
                    if (mrow) mrow[e0 + c] = 0;
                }
            }
        }
    };

    // 3. selection
    // bf16 softmax rows select on bf16 logits, whose keys carry a constant low
    // half (0 or 0xffff, by sign): key & 0xffff0000 | ~index & 0xffff then
    // orders exactly like (key, then lower index), so an arg-max round is one
    // warp reduction that yields the winner and its index at once
    constexpr bool kPacked = SCORE == kSoftmax && sizeof(InT) == 2;
    if (!SELECT && kPacked) {
        uint32_t b1 = 0u, b2 = 0u;    // the lane's best two composites after lc
        uint32_t lc = 0xffffffffu;    // the lane's last winner (none yet)
        auto rescan = [&]() {
            b1 = 0u;
            b2 = 0u;
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t q = (key[v][c] & 0xffff0000u) |
                                       (~static_cast<uint32_t>(v * 128 + lane4 + c) & 0xffffu);
                    const bool after = q < lc;
                    const bool gt1 = after && q > b1;
                    const bool gt2 = after && !gt1 && q > b2;
                    b2 = gt1 ? b1 : (gt2 ? q : b2);
                    b1 = gt1 ? q : b1;
                }
        };
        rescan();
        bool has2 = true;
        for (int j = 0; j < k_r; ++j) {
            const uint32_t w = __reduce_max_sync(kFull, b1);
            const uint32_t widx = ~w & 0xffffu;
            if (lane == 0) {
                win_idx[j] = widx;
                win_val[j] = __fmul_rn(vbuf[min(widx, static_cast<uint32_t>(E - 1))], vmul);
            }
            if (b1 == w) {  // this lane supplied the winner (composites are distinct)
                lc = b1;
                if (has2) {
                    b1 = b2;
                    has2 = false;
                } else if (j + 1 < k_r) {
                    rescan();
                    has2 = true;
                }
            }
        }
    } else if (!SELECT) {
        // k_r rounds of arg-max over the lanes' best keys. Each lane keeps its two
        // best (key, index) pairs in selection order (larger key, then lower
        // index; the lane's elements are scanned in index order with strict
        // compares); a round takes the warp's best and only the winning lane
        // moves on. A lane gives its elements away in selection order, so what it
        // has left is exactly what comes after its last winner (lk, li); it
        // rescans for its next two only when both have been taken.
        uint32_t b1 = 0u, i1 = 0xffffffffu, b2 = 0u, i2 = 0xffffffffu;
        uint32_t lk = 0xffffffffu, li = 0xffffffffu;  // nothing taken yet: every key is after it
        auto rescan = [&]() {
            b1 = 0u; i1 = 0xffffffffu; b2 = 0u; i2 = 0xffffffffu;
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t k = key[v][c];
                    const uint32_t idx = static_cast<uint32_t>(v * 128 + lane4 + c);
                    const bool after = k < lk || (k == lk && idx > li);
                    const bool gt1 = after && k > b1;
                    const bool gt2 = after && !gt1 && k > b2;
                    b2 = gt1 ? b1 : (gt2 ? k : b2);
                    i2 = gt1 ? i1 : (gt2 ? idx : i2);
                    b1 = gt1 ? k : b1;
                    i1 = gt1 ? idx : i1;
                }
        };
        rescan();
        bool has2 = true;  // (b2, i2) is the lane's next after (b1, i1)
        for (int j = 0; j < k_r; ++j) {
            const uint32_t wmax = __reduce_max_sync(kFull, b1);
            const uint32_t widx = __reduce_min_sync(kFull, b1 == wmax ? i1 : 0xffffffffu);
            if (lane == 0) {
                win_idx[j] = widx;
                win_val[j] = __fmul_rn(vbuf[min(widx, static_cast<uint32_t>(E - 1))], vmul);
            }
            bool more = false;
            if (i1 == widx && b1 == wmax) {  // this lane supplied the winner
                lk = b1;
                li = i1;
                if (has2) {
                    b1 = b2;
                    i1 = i2;
                    has2 = false;
                } else {
                    more = true;
                }
            }
            if (j + 1 < k_r && __any_sync(kFull, more) && more) {
                rescan();
                has2 = true;
            }
        }
    } else {
        unsigned long long* cand = reinterpret_cast<unsigned long long*>(wsm + L.cand);
        // SET: the bisection runs until exactly k_r keys are >= lo (or the k_r-th
        // key is tied at lo); otherwise it stops at `stop` candidates for the rank
        const uint32_t cap = static_cast<uint32_t>(SET ? k_r : a.stop);
        const uint32_t n_valid = static_cast<uint32_t>(a.n_group > 0 ? a.topk_group * (E / a.n_group) : E);
        // Invariant: count(key >= lo) = cnt_lo >= k_r > count(key >= hi) = cnt_hi.
        // lo starts at 1, below every real key (count = n_valid); the row minimum
        // is only computed when the bisection needs a real lower end.
        uint32_t lo = 1u, hi = kmax + 1u;
        uint32_t cnt_lo = n_valid, cnt_hi = 0u;
        int lane_lo = -1, lane_hi = 0;  // per-lane counts at lo / hi (-1: not yet counted)
        auto count_ge = [&](uint32_t piv) {
            uint32_t cq[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int q = 0; q < 4; ++q) cq[q] += (key[v][q] >= piv);
            return (cq[0] + cq[1]) + (cq[2] + cq[3]);
        };
        auto split = [&](uint32_t piv) {
            const uint32_t c = count_ge(piv);
            const uint32_t tot = __reduce_add_sync(kFull, c);
            if (tot >= static_cast<uint32_t>(k_r)) {
                lo = piv; cnt_lo = tot; lane_lo = static_cast<int>(c);
            } else {
                hi = piv; cnt_hi = tot; lane_hi = static_cast<int>(c);
            }
        };
        // warm start: the previous row's threshold (rows of one batch are alike,
        // so it usually leaves between k_r and `stop` candidates in one pass)
        if (cnt_lo > cap && warm > lo && warm < hi) split(warm);
        // no previous threshold, or it left too few or too many candidates: a
        // rung of the lanes' maxima; when that leaves too few, the lowest rung
        // (at least 32 keys reach it) before the row minimum is needed
        if (cnt_lo > cap && a.rung > 0) {
            const uint32_t r = warp_kth_largest(lane_max, a.rung, lane);
            if (r > lo && r < hi) split(r);
            if (cnt_lo > cap && lo == 1u) {
                const uint32_t r32 = __reduce_min_sync(kFull, lane_max);
                if (r32 > lo && r32 < hi) split(r32);
            }
        }
        if (cnt_lo > cap && lo == 1u) {
            uint32_t ln[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 4; ++c) ln[c] = min(ln[c], key[v][c] - 1u);  // 0 wraps to the top
            lo = __reduce_min_sync(kFull, min(min(ln[0], ln[1]), min(ln[2], ln[3]))) + 1u;
        }
        for (int it = 0; it < 64 && cnt_lo > cap && hi - lo > 1u; ++it) {
            const uint32_t umid = lo + ((hi - lo) >> 1);
            uint32_t mid = umid;
            if (it < 8) {  // value-space midpoint first: fast on smooth key distributions
                const float fm = __fadd_rn(__fmul_rn(float_of(lo), 0.5f), __fmul_rn(float_of(hi - 1u), 0.5f));
                const uint32_t km = key_of(fm);
                if (km > lo && km < hi) mid = km;
            }
            split(mid);
        }
        if constexpr (SET) {
            // The winners as a set (bit v*4 + c of the lane's elements): with
            // exactly k_r keys >= lo, those; else hi == lo + 1, and the keys >= hi
            // are followed by the keys equal to lo in index order.
            static_assert(NV <= 8, "one bit per element of the lane");
            uint32_t winmask = 0u;
            if (cnt_lo <= cap) {
#pragma unroll
                for (int v = 0; v < NV; ++v)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (key[v][c] >= lo) winmask |= 1u << (v * 4 + c);
            } else {
                uint32_t base = cnt_hi;
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    uint32_t m4 = 0u;
#pragma unroll
                    for (int c = 0; c < 4; ++c) m4 += (key[v][c] == lo);
                    const uint32_t off = warp_exclusive_scan(m4, lane);
                    const uint32_t tot = __shfl_sync(kFull, off + m4, 31);
                    uint32_t p = base + off;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (key[v][c] >= hi) {
                            winmask |= 1u << (v * 4 + c);
                        } else if (key[v][c] == lo) {
                            if (p < static_cast<uint32_t>(k_r)) winmask |= 1u << (v * 4 + c);
                            ++p;
                        }
                    }
                    base += tot;
                }
            }
            warm = lo;  // the next row's first pivot: this row's threshold
            float scale = a.scaling;
            if (a.renorm) {
                float ws = 0.0f;
#pragma unroll
                for (int v = 0; v < NV; ++v)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (winmask & (1u << (v * 4 + c)))
                            ws = __fadd_rn(ws, __fmul_rn(vbuf[v * 128 + lane4 + c], vmul));
                const float wsum = warp_sum(ws);
                scale = wsum > 0.0f ? __fdiv_rn(a.scaling, wsum) : 0.0f;
            }
            dense_rows();
            __syncwarp();  // the winners' writes below land after every lane's zeros
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (winmask & (1u << (v * 4 + c))) {
                        const int e = v * 128 + lane4 + c;
                        if (prow) store_scalar<InT>(prow + e, __fmul_rn(__fmul_rn(vbuf[e], vmul), scale));
                        if (mrow) mrow[e] = 1;
                    }
            return scale;
        }
        auto comp = [&](uint32_t k, int v, int c) {
            return (static_cast<unsigned long long>(k) << 32) |
                   static_cast<uint32_t>(~static_cast<uint32_t>(v * 128 + lane4 + c));
        };
        uint32_t n;
        if (cnt_lo <= cap) {
            // candidates: every key >= lo
            if (lane_lo < 0) {
                uint32_t c = 0u;
#pragma unroll
                for (int v = 0; v < NV; ++v)
#pragma unroll
                    for (int q = 0; q < 4; ++q) c += (key[v][q] >= lo);
                lane_lo = static_cast<int>(c);
            }
            uint32_t pos = warp_exclusive_scan(static_cast<uint32_t>(lane_lo), lane);
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (key[v][c] >= lo) {  // exact counts keep pos below cnt_lo <= cap
                        cand[pos] = comp(key[v][c], v, c);
                        ++pos;
                    }
            n = cnt_lo;
        } else {
            // hi == lo + 1: the k_r-th key is exactly lo. Take every key >= hi
            // (fewer than k_r), then keys equal to lo in index order.
            const uint32_t lim = static_cast<uint32_t>(k_r);
            uint32_t pos = warp_exclusive_scan(static_cast<uint32_t>(lane_hi), lane);
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (key[v][c] >= hi) {
                        if (pos < lim) cand[pos] = comp(key[v][c], v, c);
                        ++pos;
                    }
            uint32_t base = cnt_hi;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                uint32_t m4 = 0u;
#pragma unroll
                for (int c = 0; c < 4; ++c) m4 += (key[v][c] == lo);
                const uint32_t off = warp_exclusive_scan(m4, lane);
                const uint32_t tot = __shfl_sync(kFull, off + m4, 31);
                uint32_t p = base + off;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (key[v][c] == lo) {
                        if (p < lim) cand[p] = comp(lo, v, c);
                        ++p;
                    }
                base += tot;
            }
            n = min(base, lim);
        }
        n = min(n, cap);
        const uint32_t warm_rank = min(n - 1u, static_cast<uint32_t>(k_r + k_r / 4));
        if (lane == 0) scal[3] = lo;
        __syncwarp();
        rank_candidates<RANKW>(cand, n, k_r, warm_rank, lane, win_idx, win_val, scal + 3, [&](uint32_t idx, uint32_t) {
            return __fmul_rn(vbuf[min(idx, static_cast<uint32_t>(E - 1))], vmul);
        });
        __syncwarp();
        warm = scal[3];
    }
    __syncwarp();

    // 4. weights (the sum of the winners' scores only matters with renorm)
    float scale = a.scaling;
    if (a.renorm) {
        float wsum = 0.0f;
        for (int j = lane; j < k_r; j += 32) wsum = __fadd_rn(wsum, win_val[j]);
        wsum = warp_sum(wsum);
        scale = wsum > 0.0f ? __fdiv_rn(a.scaling, wsum) : 0.0f;
    }

    // 5. dense rows: intermediate = s; probs and routing_map are written as zero
    //    vectors and the k_r winners are patched in afterwards (compact outputs:
    //    emit_compact)
    if (a.probs || a.map || a.inter) {
        dense_rows();
        __syncwarp();  // the winners' writes below land after the zeros above
        if (prow || mrow) {
            for (int j = lane; j < k_r; j += 32) {
                const uint32_t idx = min(win_idx[j], static_cast<uint32_t>(E - 1));
                if (prow) store_scalar<InT>(prow + idx, __fmul_rn(win_val[j], scale));
                if (mrow) mrow[idx] = 1;
            }
        }
    }
    return scale;
}

// Compact outputs of one row from the winner list: routed slots in selection
// order, then the shared experts E..E+n_shared-1 with shared_weight. `scale`
// is route_row's return value (score -> weight).
__device__ __forceinline__ void emit_compact(const RouteArgs& a, const unsigned char* wsm,
                                             const WarpLayout& L, float scale, int lane,
                                             int32_t* idx_row, float* w_row)
{
    const uint32_t* win_idx = reinterpret_cast<const uint32_t*>(wsm + L.win_idx);
    const float* win_val = reinterpret_cast<const float*>(wsm + L.win_val);
    for (int j = lane; j < a.topk; j += 32) {
        const bool routed = j < a.k_r;
        if (idx_row) idx_row[j] = routed ? static_cast<int32_t>(win_idx[j]) : a.E + (j - a.k_r);
        if (w_row) w_row[j] = routed ? __fmul_rn(win_val[j], scale) : a.shared_weight;
    }
}

}  // namespace mr
