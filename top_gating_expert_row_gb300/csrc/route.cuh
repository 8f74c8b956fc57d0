// One token row of the router forward, computed by one warp.
//
// Follows fused_topk_with_score_function as TransformerEngine PR 3012 describes
// it (flowchart: convert to the compute type, apply the score function,
// top-k-and-mask, write probs + routing_map), rebuilt for one warp per row:
//
//   1. load     the row into registers: lane l holds elements (v*32+l)*4 .. +3
//               for v < NV, so every v is one coalesced 512 B (fp32) access
//   2. score    softmax (warp max, written exp, warp sum) or sigmoid; the
//               selection key (logit, or sigmoid + bias) as an order-preserving u32
//   3. groups   (optional) group scores = sum of each group's top-m keys; the
//               topk_group best groups are kept, the others' keys set to 0
//   4. select   k_r winners by (key desc, index asc):
//               ARGMAX  - k_r rounds of warp arg-max (REDUX max/min), for small k
//               SELECT  - bisection on the key for a threshold that leaves at most
//                         `stop` candidates, compaction to shared memory, then an
//                         exact all-pairs rank of the candidates; ties at the
//                         threshold are taken in index order
//   5. weights  renormalise over the winners and scale
//   6. emit     dense probs / routing_map / intermediate and compact topk_idx/w
//
// Both selection paths produce the identical winner list.
#pragma once

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
    int vec;   // rows and all arrays allow 16-byte (fp32) / 8-byte (bf16) vector access
    int stop;  // SELECT: candidate capacity (>= k_r); bisection stops at or below it
};

// Byte offsets of one warp's shared-memory region (same formula on host and device).
struct WarpLayout {
    int win_idx, win_val, cand_comp, cand_val, keys, scal, bytes;
};

__host__ __device__ inline int align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline WarpLayout warp_layout(int k_r, int stop, int E, bool select, bool groups)
{
    WarpLayout L;
    int o = 0;
    L.win_idx = o; o += align16(k_r * 4);
    L.win_val = o; o += align16(k_r * 4);
    L.cand_comp = o; o += select ? align16(stop * 8) : 0;
    L.cand_val = o; o += select ? align16(stop * 4) : 0;
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
template <int MAXM>
__device__ void group_limit(uint32_t* skeys, int E, int G, int gk, int m, int lane)
{
    const int gs = E / G;
    int lpg = 32 / G;                      // lanes per group, rounded down to a power of 2
    lpg = 1 << (31 - __clz(lpg));
    const int g = lane / lpg, j = lane % lpg;
    uint32_t top[MAXM];
#pragma unroll
    for (int i = 0; i < MAXM; ++i) top[i] = 0u;
    if (g < G) {
        for (int i = j; i < gs; i += lpg) {
            uint32_t k = skeys[g * gs + i];
#pragma unroll
            for (int q = 0; q < MAXM; ++q) {
                const uint32_t hi = max(k, top[q]);
                k = min(k, top[q]);
                top[q] = hi;
            }
        }
    }
    for (int o = 1; o < lpg; o <<= 1) {
        uint32_t other[MAXM];
#pragma unroll
        for (int i = 0; i < MAXM; ++i) other[i] = __shfl_xor_sync(kFull, top[i], o);
#pragma unroll
        for (int i = 0; i < MAXM; ++i) {
            uint32_t k = other[i];
#pragma unroll
            for (int q = 0; q < MAXM; ++q) {
                const uint32_t hi = max(k, top[q]);
                k = min(k, top[q]);
                top[q] = hi;
            }
        }
    }
    float acc = float_of(top[0]);
#pragma unroll
    for (int i = 1; i < MAXM; ++i)
        if (i < m) acc = __fadd_rn(acc, float_of(top[i]));
    const uint32_t sk = key_of(acc);
    // rank the G group scores: ties go to the lower group index
    const uint32_t mine = __shfl_sync(kFull, sk, (lane < G ? lane : 0) * lpg);
    uint32_t rank = 0;
    for (int q = 0; q < G; ++q) {
        const uint32_t o = __shfl_sync(kFull, sk, q * lpg);
        rank += (o > mine) || (o == mine && q < lane);
    }
    const uint32_t kept = __ballot_sync(kFull, lane < G && rank < (uint32_t)gk);
    for (int q = 0; q < G; ++q)
        if (!((kept >> q) & 1u))
            for (int i = lane; i < gs; i += 32) skeys[q * gs + i] = 0u;
}

// ---------------------------------------------------------------------------
// route_row: the whole forward for token t. Winners are left in the warp's
// shared region (win_idx / win_val, k_r entries in selection order); returns
// the factor that turns a winner's score into its weight.
// ---------------------------------------------------------------------------
template <int SCORE, typename InT, int NV, bool SELECT>
__device__ __forceinline__ float route_row(const RouteArgs& a, int t, unsigned char* wsm,
                                           const WarpLayout& L, int lane)
{
    uint32_t* win_idx = reinterpret_cast<uint32_t*>(wsm + L.win_idx);
    float* win_val = reinterpret_cast<float*>(wsm + L.win_val);
    uint32_t* scal = reinterpret_cast<uint32_t*>(wsm + L.scal);
    const int E = a.E;
    const int k_r = a.k_r;
    const InT* row = static_cast<const InT*>(a.logits) + static_cast<size_t>(t) * E;

    float val[NV][4];
    uint32_t key[NV][4];

    // 1. load
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        const int e0 = (v * 32 + lane) * 4;
        if (a.vec && e0 + 4 <= E) {
            load4<InT>(row + e0, val[v]);
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) val[v][c] = (e0 + c < E) ? load_scalar<InT>(row + e0 + c) : 0.0f;
        }
    }

    // 2. scores and selection keys; padding lanes get key 0 and score 0
    if (SCORE == kSoftmax) {
        float m = -__int_as_float(0x7f800000);
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if ((v * 32 + lane) * 4 + c < E) m = fmaxf(m, val[v][c]);
        m = warp_max(m);
        float sum = 0.0f;
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if ((v * 32 + lane) * 4 + c < E) {
                    key[v][c] = key_of(val[v][c]);
                    const float e = exp_f32(__fsub_rn(val[v][c], m));
                    val[v][c] = e;
                    sum = __fadd_rn(sum, e);
                } else {
                    key[v][c] = 0u;
                    val[v][c] = 0.0f;
                }
            }
        sum = warp_sum(sum);
        const float inv = __fdiv_rn(1.0f, sum);
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int c = 0; c < 4; ++c) val[v][c] = __fmul_rn(val[v][c], inv);
    } else {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e0 = (v * 32 + lane) * 4;
            float b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (a.bias) {
                if (a.vec && e0 + 4 <= E) {
                    const float4 q = __ldg(reinterpret_cast<const float4*>(a.bias + e0));
                    b[0] = q.x; b[1] = q.y; b[2] = q.z; b[3] = q.w;
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) b[c] = (e0 + c < E) ? __ldg(a.bias + e0 + c) : 0.0f;
                }
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (e0 + c < E) {
                    const float s = sigmoid_f32(val[v][c]);
                    key[v][c] = key_of(a.bias ? __fadd_rn(s, b[c]) : s);
                    val[v][c] = s;
                } else {
                    key[v][c] = 0u;
                    val[v][c] = 0.0f;
                }
            }
        }
    }

    // 3. group limit (keys staged through shared memory)
    if (a.n_group > 0) {
        uint32_t* sk = reinterpret_cast<uint32_t*>(wsm + L.keys);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e0 = (v * 32 + lane) * 4;
            if (e0 + 4 <= E) {
                *reinterpret_cast<uint4*>(sk + e0) = make_uint4(key[v][0], key[v][1], key[v][2], key[v][3]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (e0 + c < E) sk[e0 + c] = key[v][c];
            }
        }
        __syncwarp();
        const int m = k_r / a.topk_group;
        if (m <= 1) group_limit<1>(sk, E, a.n_group, a.topk_group, m, lane);
        else if (m <= 2) group_limit<2>(sk, E, a.n_group, a.topk_group, m, lane);
        else if (m <= 4) group_limit<4>(sk, E, a.n_group, a.topk_group, m, lane);
        else group_limit<8>(sk, E, a.n_group, a.topk_group, m, lane);
        __syncwarp();
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e0 = (v * 32 + lane) * 4;
            if (e0 + 4 <= E) {
                const uint4 q = *reinterpret_cast<const uint4*>(sk + e0);
                key[v][0] = q.x; key[v][1] = q.y; key[v][2] = q.z; key[v][3] = q.w;
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (e0 + c < E) key[v][c] = sk[e0 + c];
            }
        }
        __syncwarp();
    }

    // 4. selection
    uint32_t K = 0u, I = 0u;  // last winner (SELECT path membership test)
    if (!SELECT) {
        // k_r rounds of arg-max; a winner's key becomes 1 (below every real key,
        // above the 0 of padding / dropped groups), which also marks it as chosen.
        for (int j = 0; j < k_r; ++j) {
            uint32_t best = 0u, bidx = 0xffffffffu;
            float bv = 0.0f;
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const bool gt = key[v][c] > best;
                    best = gt ? key[v][c] : best;
                    bidx = gt ? static_cast<uint32_t>((v * 32 + lane) * 4 + c) : bidx;
                    bv = gt ? val[v][c] : bv;
                }
            const uint32_t wmax = __reduce_max_sync(kFull, best);
            const uint32_t widx = __reduce_min_sync(kFull, best == wmax ? bidx : 0xffffffffu);
            const float wv = __shfl_sync(kFull, bv, (widx >> 2) & 31u);
            if (lane == 0) {
                win_idx[j] = widx;
                win_val[j] = wv;
            }
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (static_cast<uint32_t>((v * 32 + lane) * 4 + c) == widx) key[v][c] = 1u;
        }
    } else {
        unsigned long long* cand = reinterpret_cast<unsigned long long*>(wsm + L.cand_comp);
        float* cval = reinterpret_cast<float*>(wsm + L.cand_val);
        const uint32_t cap = static_cast<uint32_t>(a.stop);
        uint32_t lmax = 0u, lmin = 0xffffffffu, lcnt = 0u;
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t k = key[v][c];
                lmax = max(lmax, k);
                lmin = (k != 0u) ? min(lmin, k) : lmin;
                lcnt += (k != 0u);
            }
        const uint32_t kmax = __reduce_max_sync(kFull, lmax);
        uint32_t lo = __reduce_min_sync(kFull, lmin);
        uint32_t hi = kmax + 1u;               // count(key >= hi) == 0
        uint32_t cnt_lo = __reduce_add_sync(kFull, lcnt), lane_lo = lcnt;
        uint32_t cnt_hi = 0u, lane_hi = 0u;
        // Invariant: count(key >= lo) = cnt_lo >= k_r > count(key >= hi) = cnt_hi.
        for (int it = 0; it < 64 && cnt_lo > cap && hi - lo > 1u; ++it) {
            const uint32_t umid = lo + ((hi - lo) >> 1);
            uint32_t mid = umid;
            if (it < 8) {  // value-space midpoint first: fast on smooth key distributions
                const float fm = __fadd_rn(__fmul_rn(float_of(lo), 0.5f), __fmul_rn(float_of(hi - 1u), 0.5f));
                const uint32_t km = key_of(fm);
                if (km > lo && km < hi) mid = km;
            }
            uint32_t c = 0u;
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int q = 0; q < 4; ++q) c += (key[v][q] >= mid);
            const uint32_t tot = __reduce_add_sync(kFull, c);
            if (tot >= static_cast<uint32_t>(k_r)) {
                lo = mid; cnt_lo = tot; lane_lo = c;
            } else {
                hi = mid; cnt_hi = tot; lane_hi = c;
            }
        }
        uint32_t n;
        if (cnt_lo <= cap) {
            // candidates: every key >= lo
            uint32_t pos = warp_exclusive_scan(lane_lo, lane);
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (key[v][c] >= lo) {
                        if (pos < cap) {
                            cand[pos] = (static_cast<unsigned long long>(key[v][c]) << 32) |
                                        static_cast<uint32_t>(~static_cast<uint32_t>((v * 32 + lane) * 4 + c));
                            cval[pos] = val[v][c];
                        }
                        ++pos;
                    }
            n = cnt_lo;
        } else {
            // hi == lo + 1: the k_r-th key is exactly lo. Take every key >= hi
            // (fewer than k_r), then keys equal to lo in index order.
            const uint32_t lim = static_cast<uint32_t>(k_r);
            uint32_t pos = warp_exclusive_scan(lane_hi, lane);
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (key[v][c] >= hi) {
                        if (pos < lim) {
                            cand[pos] = (static_cast<unsigned long long>(key[v][c]) << 32) |
                                        static_cast<uint32_t>(~static_cast<uint32_t>((v * 32 + lane) * 4 + c));
                            cval[pos] = val[v][c];
                        }
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
                        if (p < lim) {
                            cand[p] = (static_cast<unsigned long long>(lo) << 32) |
                                      static_cast<uint32_t>(~static_cast<uint32_t>((v * 32 + lane) * 4 + c));
                            cval[p] = val[v][c];
                        }
                        ++p;
                    }
                base += tot;
            }
            n = min(base, lim);
        }
        n = min(n, cap);
        __syncwarp();
        // exact rank of each candidate in selection order
        for (uint32_t b = 0; b < n; b += 64) {
            const uint32_t i0 = b + lane, i1 = b + 32 + lane;
            const unsigned long long c0 = (i0 < n) ? cand[i0] : 0ull;
            const unsigned long long c1 = (i1 < n) ? cand[i1] : 0ull;
            uint32_t r0 = 0u, r1 = 0u;
            for (uint32_t q = 0; q < n; ++q) {
                const unsigned long long cq = cand[q];
                r0 += (cq > c0);
                r1 += (cq > c1);
            }
            if (i0 < n && r0 < static_cast<uint32_t>(k_r)) {
                win_idx[r0] = ~static_cast<uint32_t>(c0);
                win_val[r0] = cval[i0];
                if (r0 == static_cast<uint32_t>(k_r - 1)) {
                    scal[0] = static_cast<uint32_t>(c0 >> 32);
                    scal[1] = ~static_cast<uint32_t>(c0);
                }
            }
            if (i1 < n && r1 < static_cast<uint32_t>(k_r)) {
                win_idx[r1] = ~static_cast<uint32_t>(c1);
                win_val[r1] = cval[i1];
                if (r1 == static_cast<uint32_t>(k_r - 1)) {
                    scal[0] = static_cast<uint32_t>(c1 >> 32);
                    scal[1] = ~static_cast<uint32_t>(c1);
                }
            }
        }
        __syncwarp();
        K = scal[0];
        I = scal[1];
    }
    __syncwarp();

    // 5. weights
    float wsum = 0.0f;
    for (int j = lane; j < k_r; j += 32) wsum = __fadd_rn(wsum, win_val[j]);
    wsum = warp_sum(wsum);
    const float scale = a.renorm ? (wsum > 0.0f ? __fdiv_rn(a.scaling, wsum) : 0.0f) : a.scaling;

    // 6. emit the dense rows (compact outputs: emit_compact)
    if (a.probs || a.map || a.inter) {
        InT* prow = a.probs ? static_cast<InT*>(a.probs) + static_cast<size_t>(t) * E : nullptr;
        uint8_t* mrow = a.map ? a.map + static_cast<size_t>(t) * E : nullptr;
        float* irow = a.inter ? a.inter + static_cast<size_t>(t) * E : nullptr;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int e0 = (v * 32 + lane) * 4;
            if (e0 >= E) continue;
            float p4[4];
            uint32_t m4 = 0u;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t idx = static_cast<uint32_t>(e0 + c);
                const uint32_t k = key[v][c];
                const bool member = SELECT ? (k > K || (k == K && idx <= I)) : (k == 1u);
                p4[c] = member ? __fmul_rn(val[v][c], scale) : 0.0f;
                m4 |= (member ? 1u : 0u) << (8 * c);
            }
            if (a.vec && e0 + 4 <= E) {
                if (prow) store4<InT>(prow + e0, p4);
                if (mrow) *reinterpret_cast<uint32_t*>(mrow + e0) = m4;
                if (irow) *reinterpret_cast<float4*>(irow + e0) = make_float4(val[v][0], val[v][1], val[v][2], val[v][3]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (e0 + c >= E) break;
                    if (prow) store_scalar<InT>(prow + e0 + c, p4[c]);
                    if (mrow) mrow[e0 + c] = static_cast<uint8_t>((m4 >> (8 * c)) & 1u);
                    if (irow) irow[e0 + c] = val[v][c];
                }
            }
        }
    }
    return scale;
}

// Compact outputs of one row from the winner list: routed slots in selection
// order, then the shared experts E..E+n_shared-1 with shared_weight.
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
