// One token row of the router forward for wide rows (E > 1024), computed by
// one warp with the row held in shared memory.
//
// Same steps and results as route_row (route.cuh), laid out for a short
// instruction stream: the selection keys (and, for sigmoid, the scores) live in
// a per-warp shared-memory row padded to whole 128-element chunks, and every
// per-element pass is one small loop over the lane's chunks. With the row in
// registers the fully unrolled passes over E=2304 keys made the code larger
// than the instruction caches, so warps stalled on instruction fetch; here the
// whole routine is a few hundred instructions.
//
// Scores never take shared memory, so each warp needs only its 9 KB of keys
// (E = 2304), which keeps twice as many warps resident as a second shared row
// would. Softmax makes two exp passes over the keys (the key map is
// invertible): the first sums the numerators exp(x - max) (and, once the
// threshold is known, writes out the candidates), the second writes the final
// scores into the intermediate row; a winner's score is recomputed from its
// key. Sigmoid writes its scores into the intermediate row as it makes the
// keys (or, without that output, keeps them in a shared row) and reads the
// winners' back.
#pragma once

#include "route.cuh"

namespace mr {

// Per-warp shared memory of the wide routine.
//   kbuf   keys, nv*128 u32 (positions >= E hold 0, "not a candidate"); with
//          staging it first receives the raw row (fp32 at its start, bf16 in
//          its upper half) and the load pass turns it into keys in place
//   vbuf   sigmoid scores when there is no intermediate output, nv*128 fp32
//   win_*, cand, scal as in WarpLayout
//   bar    mbarrier on which the staging copy completes
struct WideLayout {
    int kbuf, vbuf, win_idx, win_val, cand, scal, bar, bytes;
};

// Staging of the next row: while a warp finishes row t (the threshold select's
// ranking of its candidates, the weights and the dense outputs, none of which
// read kbuf) the bulk-copy engine brings row `next` into kbuf, so the next
// row's load pass reads shared memory.
struct Stage {
    uint64_t* bar;
    const void* next;  // nullptr: no next row for this warp
    uint32_t bytes;    // row bytes (E * element size)
    uint32_t off;      // byte offset of the raw row inside kbuf
    int drop;          // test mode: arm the barrier, issue no copy
};

__host__ __device__ inline WideLayout wide_layout(int k_r, int stop, int E, bool select, bool keep_scores)
{
    WideLayout L;
    const int padded = (E + 127) / 128 * 128;
    int o = 0;
    L.kbuf = o; o += padded * 4;
    L.vbuf = o; o += keep_scores ? padded * 4 : 0;
    L.win_idx = o; o += align16(k_r * 4);
    L.win_val = o; o += align16(k_r * 4);
    L.cand = o; o += select ? align16(stop * 8) : 0;
    L.scal = o; o += 16;
    L.bar = o; o += 16;
    L.bytes = o;
    return L;
}

// FULL: every chunk is whole and vector-aligned (a.vec and E % 128 == 0), so the
// per-chunk edge handling compiles away; rows are then staged in shared memory
// by the bulk-copy engine (the caller has waited for this row's copy).
template <int SCORE, typename InT, bool SELECT, bool FULL>
__device__ __forceinline__ float route_row_wide(const RouteArgs& a, int t, unsigned char* wsm,
                                                const WideLayout& L, int lane, uint32_t& warm, const Stage& st)
{
    uint32_t* kbuf = reinterpret_cast<uint32_t*>(wsm + L.kbuf);
    float* vbuf = reinterpret_cast<float*>(wsm + L.vbuf);
    uint32_t* win_idx = reinterpret_cast<uint32_t*>(wsm + L.win_idx);
    float* win_val = reinterpret_cast<float*>(wsm + L.win_val);
    uint32_t* scal = reinterpret_cast<uint32_t*>(wsm + L.scal);
    const int E = a.E;
    const int k_r = a.k_r;
    const int nv = (E + 127) >> 7;
    const int lane4 = lane * 4;
    const InT* row = static_cast<const InT*>(a.logits) + static_cast<size_t>(t) * E;
    auto whole = [&](int v) { return FULL || v * 128 + lane4 + 4 <= E; };
    const bool vec = FULL || a.vec;
    // every pass below touches only the lane's own chunks (v*128 + 4*lane .. +3)
    auto k4 = [&](int v) -> uint4& { return *reinterpret_cast<uint4*>(kbuf + v * 128 + lane4); };

    float* irow0 = a.inter ? a.inter + static_cast<size_t>(t) * E : nullptr;  // intermediate output row
    // The previous row's threshold key, when there is one, is tested while the
    // keys are made: cw = this lane's count of keys >= warm (0 is never a key
    // of a real element, so warm = 0 means none).
    const bool has_warm = SELECT && a.n_group == 0 && warm >= 2u;
    const uint32_t wpiv = has_warm ? warm : 0xffffffffu;
    uint32_t cw = 0u;
    // 1. load (8 chunks in flight), selection keys, sigmoid scores
    uint32_t lm = 0u;
    float m = 0.0f;    // softmax: the row max
    float vmul = 1.0f; // score = stored/recomputed value * vmul
    for (int v0 = 0; v0 < nv; v0 += 8) {
        float x[8][4];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int v = v0 + u;
            const int e0 = v * 128 + lane4;
            if (v < nv) {
                if (FULL) {
                    load4_shared<InT>(wsm + L.kbuf + st.off, e0, x[u]);
                } else if (vec && whole(v)) {
                    load4<InT>(row + e0, x[u]);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) x[u][c] = (e0 + c < E) ? load_scalar<InT>(row + e0 + c) : 0.0f;
                }
            }
        }
        // bf16 staging: keys of a batch overwrite raw elements that other lanes
        // read in this same batch (never in a later one)
        if (FULL && sizeof(InT) == 2) __syncwarp();
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int v = v0 + u;
            const int e0 = v * 128 + lane4;
            if (v >= nv) continue;
            uint32_t kk[4];
            if (SCORE == kSoftmax) {
#pragma unroll
                for (int c = 0; c < 4; ++c) kk[c] = (FULL || e0 + c < E) ? key_of(x[u][c]) : 0u;
            } else {
                float b[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (a.bias) {
                    if (vec && whole(v)) {
                        const float4 q = __ldcg(reinterpret_cast<const float4*>(a.bias + e0));
                        b[0] = q.x; b[1] = q.y; b[2] = q.z; b[3] = q.w;
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) b[c] = (e0 + c < E) ? __ldcg(a.bias + e0 + c) : 0.0f;
                    }
                }
                const float2 s01 = sigmoid_f32x2(make_float2(x[u][0], x[u][1]));
                const float2 s23 = sigmoid_f32x2(make_float2(x[u][2], x[u][3]));
                float sv[4] = {s01.x, s01.y, s23.x, s23.y};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    sv[c] = (FULL || e0 + c < E) ? sv[c] : 0.0f;
                    kk[c] = (FULL || e0 + c < E) ? key_of(a.bias ? __fadd_rn(sv[c], b[c]) : sv[c]) : 0u;
                }
                if (irow0) {
                    if (vec && whole(v)) {
                        *reinterpret_cast<float4*>(irow0 + e0) = make_float4(sv[0], sv[1], sv[2], sv[3]);
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            if (e0 + c < E) irow0[e0 + c] = sv[c];
                    }
                } else {
                    *reinterpret_cast<float4*>(vbuf + e0) = make_float4(sv[0], sv[1], sv[2], sv[3]);
                }
            }
            lm = max(lm, max(max(kk[0], kk[1]), max(kk[2], kk[3])));
            if (SELECT) cw += (kk[0] >= wpiv) + (kk[1] >= wpiv) + (kk[2] >= wpiv) + (kk[3] >= wpiv);
            k4(v) = make_uint4(kk[0], kk[1], kk[2], kk[3]);
        }
    }
    uint32_t kmax = __reduce_max_sync(kFull, lm);
    // warm tested: its count decides whether it already bounds the candidates
    const bool warm_tested = has_warm && wpiv <= kmax;
    const uint32_t cnt_w = warm_tested ? __reduce_add_sync(kFull, cw) : 0u;
    const uint32_t cap = static_cast<uint32_t>(a.stop);
    unsigned long long* cand = reinterpret_cast<unsigned long long*>(wsm + L.cand);
    auto comp = [&](uint32_t k, uint32_t idx) {
        return (static_cast<unsigned long long>(k) << 32) | static_cast<uint32_t>(~idx);
    };

    // Threshold select state. Invariant: count(key >= lo) = cnt_lo >= k_r >
    // count(key >= hi) = cnt_hi; lane_lo / lane_hi are this lane's counts (-1:
    // not yet counted). lo starts at 1, below every real key.
    const uint32_t n_valid = static_cast<uint32_t>(a.n_group > 0 ? a.topk_group * (E / a.n_group) : E);
    uint32_t lo = 1u, hi = 0u;
    uint32_t cnt_lo = n_valid, cnt_hi = 0u;
    int lane_lo = -1, lane_hi = 0;
    auto count_ge = [&](uint32_t piv) {
        uint32_t c0 = 0u, c1 = 0u;
#pragma unroll 4
        for (int v = 0; v < nv; ++v) {
            const uint4 q = k4(v);
            c0 += (q.x >= piv) + (q.y >= piv);
            c1 += (q.z >= piv) + (q.w >= piv);
        }
        return c0 + c1;
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
    // Bisection until at most cap keys are >= lo, or the k_r-th key is tied at
    // lo (hi == lo + 1). Pivots: the previous row's threshold (counted with the
    // keys), a rung of the lanes' maxima (then the lowest rung, at least 32
    // keys reach it, when that left too few), then value-space midpoints, then
    // key-space midpoints (at most 64 rounds in all).
    auto bisect = [&]() {
        hi = kmax + 1u;
        if (warm_tested) {
            if (cnt_w >= static_cast<uint32_t>(k_r)) {
                lo = wpiv; cnt_lo = cnt_w; lane_lo = static_cast<int>(cw);
            } else {
                hi = wpiv; cnt_hi = cnt_w; lane_hi = static_cast<int>(cw);
            }
        }
        if (cnt_lo > cap && a.rung > 0) {
            const uint32_t r = warp_kth_largest(lm, a.rung, lane);
            if (r > lo && r < hi) split(r);
            if (cnt_lo > cap && lo == 1u) {
                const uint32_t r32 = __reduce_min_sync(kFull, lm);
                if (r32 > lo && r32 < hi) split(r32);
            }
        }
        for (int it = 0; it < 64 && cnt_lo > cap && hi - lo > 1u; ++it) {
            if (lo == 1u) {  // a real lower end: the row's smallest key
                uint32_t ln = 0xffffffffu;
                for (int v = 0; v < nv; ++v) {
                    const uint4 q = k4(v);
                    ln = min(ln, min(min(q.x - 1u, q.y - 1u), min(q.z - 1u, q.w - 1u)));  // 0 wraps to the top
                }
                lo = __reduce_min_sync(kFull, ln) + 1u;
                if (!(cnt_lo > cap && hi - lo > 1u)) break;
            }
            uint32_t piv = lo + ((hi - lo) >> 1);
            if (it < 8) {
                const float fm = __fadd_rn(__fmul_rn(float_of(lo), 0.5f), __fmul_rn(float_of(hi - 1u), 0.5f));
                const uint32_t km = key_of(fm);
                if (km > lo && km < hi) piv = km;
            }
            split(piv);
        }
    };
    // Softmax rows without groups select before the exp pass: once at most cap
    // keys are >= lo, the exp pass writes those candidates out as it reads the
    // keys (no pass of its own). With groups the exp pass must see every key
    // before the group limit drops some, so the selection comes after it.
    const bool early = SELECT && SCORE == kSoftmax && a.n_group == 0;
    if (early) bisect();
    const bool fused_pick = early && cnt_lo <= cap;
    if (fused_pick && lane_lo < 0) lane_lo = static_cast<int>(count_ge(lo));
    if (SCORE == kSoftmax) {
        m = float_of(kmax);
        uint32_t cpos = fused_pick ? warp_exclusive_scan(static_cast<uint32_t>(lane_lo), lane) : 0u;
        const uint32_t ppiv = lo;  // fused_pick: candidates are the keys >= lo
        unsigned long long cm = 0ull;  // fused_pick: bit v set when chunk v holds a candidate
        float2 sum01 = make_float2(0.0f, 0.0f), sum23 = make_float2(0.0f, 0.0f);
        const float2 negm = make_float2(-m, -m);
        // exp(x - m) of a chunk's keys, x - m computed as x + (-m) (the same
        // IEEE result); padding keys (0) give 0
        auto chunk_exp = [&](const uint4& q) {
            const float2 e01 = exp_value2(__fadd2_rn(make_float2(float_of(q.x), float_of(q.y)), negm));
            const float2 e23 = exp_value2(__fadd2_rn(make_float2(float_of(q.z), float_of(q.w)), negm));
            return FULL ? make_float4(e01.x, e01.y, e23.x, e23.y)
                        : make_float4(q.x ? e01.x : 0.0f, q.y ? e01.y : 0.0f, q.z ? e23.x : 0.0f, q.w ? e23.y : 0.0f);
        };
        // first pass: the sum (batches of kExpBatch chunks, keys loaded first)
        constexpr int kExpBatch = 2;
        for (int v0 = 0; v0 < nv; v0 += kExpBatch) {
            uint4 qb[kExpBatch];
#pragma unroll
            for (int u = 0; u < kExpBatch; ++u)
                qb[u] = (v0 + u < nv) ? k4(v0 + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < kExpBatch; ++u) {
                const int v = v0 + u;
                if (v >= nv) break;
                const uint4 q = qb[u];
                const float4 e = chunk_exp(q);
                sum01 = __fadd2_rn(sum01, make_float2(e.x, e.y));
                sum23 = __fadd2_rn(sum23, make_float2(e.z, e.w));
                if (SELECT && fused_pick)
                    cm |= static_cast<unsigned long long>(max(max(q.x, q.y), max(q.z, q.w)) >= ppiv) << v;
            }
        }
        // the candidates, from the marked chunks only (a few per lane)
        if (SELECT && fused_pick) {
            while (cm) {
                const int v = __ffsll(static_cast<long long>(cm)) - 1;
                cm &= cm - 1ull;
                const uint4 q = k4(v);
                const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
                const uint32_t e0i = static_cast<uint32_t>(v * 128 + lane4);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // positions come from exact counts of these same keys, so
                    // cpos stays below cnt_lo <= cap
                    const bool in = kq[c] >= ppiv;
                    if (in) cand[cpos] = comp(kq[c], e0i + c);
                    cpos += in ? 1u : 0u;
                }
            }
        }
        vmul = __frcp_rn(warp_sum(__fadd_rn(__fadd_rn(sum01.x, sum01.y), __fadd_rn(sum23.x, sum23.y))));
        // second pass: the final scores s = exp(x - m) * (1 / sum), the values a
        // winner's score_of gives too
        if (irow0) {
            const float2 vm = make_float2(vmul, vmul);
            for (int v0 = 0; v0 < nv; v0 += kExpBatch) {
                uint4 qb[kExpBatch];
#pragma unroll
                for (int u = 0; u < kExpBatch; ++u)
                    qb[u] = (v0 + u < nv) ? k4(v0 + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < kExpBatch; ++u) {
                    const int v = v0 + u;
                    if (v >= nv) break;
                    const float4 e = chunk_exp(qb[u]);
                    const float2 s01 = __fmul2_rn(make_float2(e.x, e.y), vm);
                    const float2 s23 = __fmul2_rn(make_float2(e.z, e.w), vm);
                    const int o = v * 128 + lane4;
                    if (vec && whole(v)) {
                        *reinterpret_cast<float4*>(irow0 + o) = make_float4(s01.x, s01.y, s23.x, s23.y);
                    } else {
                        const float sv[4] = {s01.x, s01.y, s23.x, s23.y};
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            if (o + c < E) irow0[o + c] = sv[c];
                    }
                }
            }
        }
    }
    __syncwarp();  // scores written by one lane are read by another below
    // a winner's score: softmax recomputes it from the key; sigmoid reads it back
    auto score_of = [&](uint32_t idx, uint32_t key) {
        if (SCORE == kSoftmax) return __fmul_rn(exp_value(__fsub_rn(float_of(key), m)), vmul);
        const uint32_t i = min(idx, static_cast<uint32_t>(E - 1));
        return irow0 ? __ldcg(irow0 + i) : vbuf[i];
    };

    // 2. group limit, directly on the shared keys
    if (a.n_group > 0) {
        __syncwarp();
        const int mg = k_r / a.topk_group;
        if (mg <= 1) group_limit<1>(kbuf, E, a.n_group, a.topk_group, mg, lane);
        else if (mg <= 2) group_limit<2>(kbuf, E, a.n_group, a.topk_group, mg, lane);
        else if (mg <= 4) group_limit<4>(kbuf, E, a.n_group, a.topk_group, mg, lane);
        else group_limit<8>(kbuf, E, a.n_group, a.topk_group, mg, lane);
        __syncwarp();
        lm = 0u;
        for (int v = 0; v < nv; ++v) {
            const uint4 q = k4(v);
            lm = max(lm, max(max(q.x, q.y), max(q.z, q.w)));
        }
        kmax = __reduce_max_sync(kFull, lm);
    }

    // 3. selection
    if (!SELECT) {
        // k_r rounds of arg-max; round j only considers keys that come after the
        // previous winner in selection order (keys stay intact: softmax scores
        // are recomputed from them)
        uint32_t Kp = 0xffffffffu, Ip = 0xffffffffu;
        for (int j = 0; j < k_r; ++j) {
            uint32_t best = 0u, bidx = 0xffffffffu;
            for (int v = 0; v < nv; ++v) {
                const uint4 q = k4(v);
                const uint32_t e0 = static_cast<uint32_t>(v * 128 + lane4);
                const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const bool after = kq[c] < Kp || (kq[c] == Kp && e0 + c > Ip);
                    if (after && kq[c] > best) {
                        best = kq[c];
                        bidx = e0 + c;
                    }
                }
            }
            const uint32_t wmax = __reduce_max_sync(kFull, best);
            const uint32_t widx = __reduce_min_sync(kFull, best == wmax ? bidx : 0xffffffffu);
            if (lane == 0 && widx < static_cast<uint32_t>(E)) {
                win_idx[j] = widx;
                win_val[j] = score_of(widx, wmax);
            }
            Kp = wmax;
            Ip = widx;
        }
    } else {
        if (!early) bisect();
        uint32_t n;
        if (fused_pick) {
            n = cnt_lo;  // written by the exp pass
        } else if (cnt_lo <= cap) {
            if (lane_lo < 0) lane_lo = static_cast<int>(count_ge(lo));
            uint32_t pos = warp_exclusive_scan(static_cast<uint32_t>(lane_lo), lane);
            for (int v0 = 0; v0 < nv; v0 += 4) {
                uint4 qb[4];  // keys first (see the exp pass)
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    qb[u] = (v0 + u < nv) ? k4(v0 + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t e0 = static_cast<uint32_t>((v0 + u) * 128 + lane4);
                    const uint32_t kq[4] = {qb[u].x, qb[u].y, qb[u].z, qb[u].w};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        // positions come from exact counts of these same keys, so
                        // pos stays below cnt_lo <= cap (padding keys 0 never pass)
                        const bool in = kq[c] >= lo;
                        if (in) cand[pos] = comp(kq[c], e0 + c);
                        pos += in ? 1u : 0u;
                    }
                }
            }
            n = cnt_lo;
        } else {
            // hi == lo + 1: the k_r-th key is lo; take keys >= hi, then keys == lo
            // in index order
            const uint32_t lim = static_cast<uint32_t>(k_r);
            uint32_t pos = warp_exclusive_scan(static_cast<uint32_t>(lane_hi), lane);
            uint32_t base = cnt_hi;
            for (int v = 0; v < nv; ++v) {
                const uint4 q = k4(v);
                const uint32_t e0 = static_cast<uint32_t>(v * 128 + lane4);
                const uint32_t kq[4] = {q.x, q.y, q.z, q.w};
                uint32_t m4 = 0u;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (kq[c] >= hi) {
                        if (pos < lim) cand[pos] = comp(kq[c], e0 + c);
                        ++pos;
                    }
                    m4 += (kq[c] == lo);
                }
                const uint32_t off = warp_exclusive_scan(m4, lane);
                const uint32_t tot = __shfl_sync(kFull, off + m4, 31);
                uint32_t p = base + off;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    if (kq[c] == lo) {
                        if (p < lim) cand[p] = comp(lo, e0 + c);
                        ++p;
                    }
                base += tot;
            }
            n = min(base, lim);
        }
        n = min(n, cap);
        const uint32_t warm_rank = min(n - 1u, static_cast<uint32_t>(k_r + k_r / 4));
        if (lane == 0) scal[3] = lo;
        // the ranking reads only cand: kbuf is free from here on, so the next
        // row's copy starts now and lands while this row is ranked and written.
        // The proxy fence orders this lane's generic accesses to kbuf before
        // the copy's writes.
        if (FULL && st.next) fence_proxy_async_smem();
        __syncwarp();
        if (FULL && st.next && lane == 0) bulk_load_row(wsm + L.kbuf + st.off, st.next, st.bytes, st.bar, st.drop);
        rank_candidates<3>(cand, n, k_r, warm_rank, lane, win_idx, win_val, scal + 3, score_of);
        __syncwarp();
        warm = scal[3];
    }
    // arg-max rounds read kbuf to the end: stage the next row only now (the
    // threshold select staged it before its ranking)
    if (!SELECT && FULL && st.next) fence_proxy_async_smem();
    __syncwarp();
    if (!SELECT && FULL && st.next && lane == 0) bulk_load_row(wsm + L.kbuf + st.off, st.next, st.bytes, st.bar, st.drop);

    // 4. weights (the sum of the winners' scores only matters with renorm)
    float scale = a.scaling;
    if (a.renorm) {
        float wsum = 0.0f;
        for (int j = lane; j < k_r; j += 32) wsum = __fadd_rn(wsum, win_val[j]);
        wsum = warp_sum(wsum);
        scale = wsum > 0.0f ? __fdiv_rn(a.scaling, wsum) : 0.0f;
    }

    // 5. dense rows (the intermediate row holds its final scores already):
    //    probs and routing_map are written as zero vectors and the k_r winners
    //    are patched in afterwards, so no per-element membership test is needed
    if (a.probs || a.map) {
        InT* prow = a.probs ? static_cast<InT*>(a.probs) + static_cast<size_t>(t) * E : nullptr;
        uint8_t* mrow = a.map ? a.map + static_cast<size_t>(t) * E : nullptr;
        for (int v = 0; v < nv; ++v) {
            const int e0 = v * 128 + lane4;
            if (!FULL && e0 >= E) continue;
            if (vec && whole(v)) {
                if (prow) {
                    const float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    store4<InT>(prow + e0, z);
                }
                if (mrow) *reinterpret_cast<uint32_t*>(mrow + e0) = 0u;
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (e0 + c >= E) break;
                    if (prow) store_scalar<InT>(prow + e0 + c, 0.0f);
                    if (mrow) mrow[e0 + c] = 0;
                }
            }
        }
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

}  // namespace mr
