// Router forward and fused decode route+sort kernels for one (score function,
// logits dtype) pair. Compiled once per pair with -DMR_SCORE_FN=0|1 and
// -DMR_IN_BF16=0|1 so the four instantiation sets build in parallel.
//
//   k_router_fwd     persistent grid, 8 warps per CTA, one token row per warp
//                    at a time (TransformerEngine PR 3012, fused_topk_with_
//                    score_function; also serves fused_score_for_moe_aux_loss)
//   k_fused_tiny     T*topk <= 32 pairs: a warp per token, then one warp sorts
//                    the pairs (a pair per lane) with no pass over all experts
//   k_fused_small    T*topk <= 128 pairs, T <= 16: a warp per token, warp 0
//                    ranks the pairs and scans the padded counts, the CTA
//                    writes the sentinels
//   k_fused_decode   ONE CTA for T <= 16 tokens (T <= 64 for E <= 256, with 32
//                    warps): warp t routes token t (and t + 32), then
//                    the whole CTA histograms, scans and scatters the T*topk
//                    pairs in shared memory (FlyDSL PR 582, fused top-k gating
//                    + MoE sorting at decode sizes)
//   k_fused_cluster  ONE thread-block cluster for up to 32 tokens per CTA:
//                    each warp routes a token, the CTAs keep their pairs in
//                    shared memory and the cluster sorts them together
//                    (cluster_sort_runs), so larger batches stay one launch
#include <type_traits>

#include "internal.h"
#include "route_wide.cuh"
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

// RANKW: candidates per lane in a pass of the candidate rank (3 only where the
// candidate cap exceeds 64, see rank_candidates). SET: no compact outputs, the
// winners are selected as a set (route_row).
template <int NV, bool SELECT, bool FULL, int RANKW = 2, bool SET = false>
__global__ void __launch_bounds__(kFwdThreads, fwd_min_blocks(NV)) k_router_fwd(RouteArgs a)
{
    pdl_trigger_small();
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, SELECT, a.n_group > 0);
    unsigned char* wsm = smem + static_cast<size_t>(warp) * L.bytes;
    const int stride = gridDim.x * nw;
    const uint32_t row_bytes = static_cast<uint32_t>(a.E) * sizeof(InT);
    uint32_t warm = 0u;  // threshold carried from this warp's previous row
    pdl_wait();
    for (int t = blockIdx.x * nw + warp; t < a.T; t += stride) {
        // the warp's next row streams into L2 while this one is computed
        if (a.prefetch && lane == 0 && t + stride < a.T)
            prefetch_l2(static_cast<const InT*>(a.logits) + static_cast<size_t>(t + stride) * a.E, row_bytes);
        const float scale = route_row<kScore, InT, NV, SELECT, FULL, RANKW, SET>(a, t, wsm, L, lane, warm);
        if (!SET && (a.topk_idx || a.topk_w)) {
            const size_t o = static_cast<size_t>(t) * a.topk;
            emit_compact(a, wsm, L, scale, lane, a.topk_idx ? a.topk_idx + o : nullptr,
                         a.topk_w ? a.topk_w + o : nullptr);
        }
        __syncwarp();
    }
}

// Wide rows (E > 1024): the row lives in shared memory, one warp per row.
template <bool SELECT, bool FULL>
__global__ void __launch_bounds__(kWideThreads, kWideMinBlocks) k_router_fwd_wide(RouteArgs a)
{
    pdl_trigger_small();
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const WideLayout L = wide_layout(a.k_r, a.stop, a.E, SELECT, kScore == kSigmoid && !a.inter);
    unsigned char* wsm = smem + static_cast<size_t>(warp) * L.bytes;
    const int stride = gridDim.x * nw;
    const uint32_t row_bytes = static_cast<uint32_t>(a.E) * sizeof(InT);
    uint32_t warm = 0u;
    // FULL rows are staged in shared memory by bulk copies: the first one here,
    // each next one while the previous row writes its outputs
    Stage st;
    st.bar = reinterpret_cast<uint64_t*>(wsm + L.bar);
    st.bytes = row_bytes;
    st.off = sizeof(InT) == 4 ? 0u : static_cast<uint32_t>(a.E) * 2u;
    st.next = nullptr;
    st.drop = a.drop_copies;
    uint32_t phase = 0u;
    int t = blockIdx.x * nw + warp;
    if (FULL) {
        if (lane == 0) mbar_init(st.bar, 1);
        __syncwarp();
    }
    pdl_wait();
    const InT* rows = static_cast<const InT*>(a.logits);
    if (FULL) {
        if (lane == 0 && t < a.T) bulk_load_row(wsm + L.kbuf + st.off, rows + static_cast<size_t>(t) * a.E, row_bytes,
                                                st.bar, st.drop);
    }
    for (; t < a.T; t += stride) {
        // rows that are not staged stream into L2 one row ahead (staged rows do
        // not gain from it: their bulk copy is issued about half a row ahead)
        if (!FULL && a.prefetch && lane == 0 && t + stride < a.T)
            prefetch_l2(rows + static_cast<size_t>(t + stride) * a.E, row_bytes);
        if (FULL) {
            const bool ok = __all_sync(kFull, mbar_wait(st.bar, phase, a.wait_tries));
            if (!ok) {
                // the copy did not land within the wait limit: report it, give
                // the copy one more bounded wait (so that, short of a failed
                // memory system, it has landed before the warp leaves), and stop
                // (no further rows)
                if (lane == 0) report_status(a.status, kStatusTimeout);
                mbar_wait(st.bar, phase, a.wait_tries);
                return;
            }
            phase ^= 1u;
            st.next = t + stride < a.T ? rows + static_cast<size_t>(t + stride) * a.E : nullptr;
        }
        const float scale = route_row_wide<kScore, InT, SELECT, FULL>(a, t, wsm, L, lane, warm, st);
        if (a.topk_idx || a.topk_w) {
            const size_t o = static_cast<size_t>(t) * a.topk;
            const uint32_t* win_idx = reinterpret_cast<const uint32_t*>(wsm + L.win_idx);
            const float* win_val = reinterpret_cast<const float*>(wsm + L.win_val);
            for (int j = lane; j < a.topk; j += 32) {
                const bool routed = j < a.k_r;
                if (a.topk_idx) a.topk_idx[o + j] = routed ? static_cast<int32_t>(win_idx[j]) : a.E + (j - a.k_r);
                if (a.topk_w) a.topk_w[o + j] = routed ? __fmul_rn(win_val[j], scale) : a.shared_weight;
            }
        }
        __syncwarp();
    }
}

// A row of zeros for the fused decode kernel's warm-up pass (E <= 1024 logits).
static __device__ __align__(16) float g_zero_row[kFusedMaxNv * 128];

template <int NV, bool SELECT, bool FULL, int THREADS>
__global__ void __launch_bounds__(THREADS, 1) k_fused_decode(RouteArgs a, SortArgs s)
{
    // A decode call is one short launch on one SM whose instruction cache is
    // usually cold, so this kernel keeps its executed code short: per-expert
    // token bitmasks give every pair its stable rank directly (a token's topk
    // experts are distinct, so the rank of (t, j) inside expert e is the number
    // of earlier tokens that chose e), one warp scans the padded counts, and
    // three block barriers separate the phases. The 32-warp form routes up to
    // 64 tokens (warp w: tokens w and w + 32) with 64-bit masks.
    using Mask = typename std::conditional<(THREADS > kFusedThreads), unsigned long long, uint32_t>::type;
    pdl_trigger_small();
    extern __shared__ __align__(16) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5, nt = blockDim.x;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, SELECT, a.n_group > 0);
    const int N = a.T * a.topk;
    const int E_tot = s.E_tot, bm = s.block_m;
    const FusedSortLayout F = fused_sort_layout(N, E_tot, bm, sizeof(Mask));
    unsigned char* base = smem + static_cast<size_t>(nw) * L.bytes;
    int32_t* s_idx = reinterpret_cast<int32_t*>(base + F.idx);
    float* s_w = reinterpret_cast<float*>(base + F.w);
    Mask* mask = reinterpret_cast<Mask*>(base + F.mask);
    uint32_t* off = reinterpret_cast<uint32_t*>(base + F.off);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(base + F.cnt);
    int32_t* blk = reinterpret_cast<int32_t*>(base + F.blk);
    auto popc = [](Mask m) { return static_cast<uint32_t>(sizeof(Mask) == 8 ? __popcll(m) : __popc(static_cast<uint32_t>(m))); };

    for (int e = tid; e < E_tot; e += nt) mask[e] = 0u;
    {
        unsigned char* wsm = smem + static_cast<size_t>(warp) * L.bytes;
        // With the launch overlap the kernel may start while its predecessor
        // still runs; the routing warps then first run their row routine on a
        // row of zeros (outputs off), through the same single call site, so its
        // code is in this SM's instruction caches when the real rows are routed
        // after the wait. Pass 1 is the real one.
#pragma unroll 1
        for (int pass = a.warm_code ? 0 : 1; pass < 2; ++pass) {
            if (pass == 1) pdl_wait();
            RouteArgs ar = a;
            if (pass == 0) {
                ar.logits = g_zero_row;
                ar.bias = nullptr;
                ar.probs = nullptr;
                ar.map = nullptr;
                ar.inter = nullptr;
            }
            uint32_t warm = 0u;
            for (int tok = warp; tok < a.T; tok += nw) {
            const float scale = route_row<kScore, InT, NV, SELECT, FULL>(ar, pass ? tok : 0, wsm, L, lane, warm);
            if (pass == 0) {
                __syncwarp();
                continue;
            }
            const size_t o = static_cast<size_t>(tok) * a.topk;
            const uint32_t* win_idx = reinterpret_cast<const uint32_t*>(wsm + L.win_idx);
            const float* win_val = reinterpret_cast<const float*>(wsm + L.win_val);
            for (int j = lane; j < a.topk; j += 32) {  // compact outputs, to shared and global
                const bool routed = j < a.k_r;
                const int32_t id = routed ? static_cast<int32_t>(win_idx[j]) : a.E + (j - a.k_r);
                const float wv = routed ? __fmul_rn(win_val[j], scale) : a.shared_weight;
                s_idx[o + j] = id;
                s_w[o + j] = wv;
                if (a.topk_idx) a.topk_idx[o + j] = id;
                if (a.topk_w) a.topk_w[o + j] = wv;
            }
            __syncwarp();  // the winner lists are rewritten by the warp's next token
            }
        }
    }
    __syncthreads();
    for (int tok = warp; tok < a.T; tok += nw) {
        for (int j = lane; j < a.topk; j += 32) {
            const int e = s_idx[tok * a.topk + j];
            if (e >= 0 && e < E_tot) atomicOr(mask + e, Mask(1) << tok);  // range check: NaN rows only
        }
    }
    __syncthreads();
    // one warp: counts and padded counts -> exclusive offsets (lane l takes
    // experts l*per .. l*per+per-1; a power-of-two block_m, the usual case, pads
    // with a shift, not a division)
    if (warp == 0) {
        const int per = (E_tot + 31) / 32;
        const int e0 = lane * per, e1 = min(E_tot, e0 + per);
        const uint32_t add = static_cast<uint32_t>(bm - 1);
        uint32_t local = 0u;
        if (s.bm_shift >= 0) {
            for (int e = e0; e < e1; ++e) local += (popc(mask[e]) + add) >> s.bm_shift;
        } else {
            for (int e = e0; e < e1; ++e) local += (popc(mask[e]) + add) / static_cast<uint32_t>(bm);
        }
        uint32_t run = warp_exclusive_scan(local, lane) * static_cast<uint32_t>(bm);  // in positions
        if (s.bm_shift >= 0) {
            for (int e = e0; e < e1; ++e) {
                const uint32_t c = popc(mask[e]);
                cnt[e] = c;
                off[e] = run;
                run += ((c + add) >> s.bm_shift) << s.bm_shift;
            }
        } else {
            for (int e = e0; e < e1; ++e) {
                const uint32_t c = popc(mask[e]);
                cnt[e] = c;
                off[e] = run;
                run += (c + add) / static_cast<uint32_t>(bm) * static_cast<uint32_t>(bm);
            }
        }
        if (lane == 31) {
            off[E_tot] = run;
            *s.num_post_pad = static_cast<int32_t>(run);
        }
    }
    __syncthreads();
    // the block -> expert map, a thread per expert (an expert's blocks are
    // few at these sizes)
    if (s.bm_shift >= 0) {
        for (int e = tid; e < E_tot; e += nt)
            for (uint32_t q = off[e]; q < off[e + 1]; q += bm) blk[q >> s.bm_shift] = e;
    } else {
        for (int e = tid; e < E_tot; e += nt)
            for (uint32_t q = off[e]; q < off[e + 1]; q += bm) blk[q / static_cast<uint32_t>(bm)] = e;
    }
    // real pairs: a token's warp writes its slots
    for (int tok = warp; tok < a.T; tok += nw) {
        const Mask before = (Mask(1) << tok) - 1u;
        for (int j = lane; j < a.topk; j += 32) {
            const int f = tok * a.topk + j;
            const int e = s_idx[f];
            if (e < 0 || e >= E_tot) continue;
            const uint32_t pos = off[e] + popc(mask[e] & before);
            s.ids[pos] = f;
            if (s.w) s.w[pos] = s_w[f];
        }
    }
    __syncthreads();
    // sentinels and expert ids, one block of block_m positions per warp step
    const int nblk = static_cast<int>(off[E_tot]) / bm;
    for (int b = warp; b < nblk; b += nw) {
        const int e = blk[b];
        const uint32_t r_first = static_cast<uint32_t>(b * bm) - off[e];
        const uint32_t c = cnt[e];
        for (int r = lane; r < bm; r += 32) {
            if (r_first + r >= c) {
                s.ids[b * bm + r] = N;
                if (s.w) s.w[b * bm + r] = 0.0f;
            }
        }
        if (lane == 0) s.expert_ids[b] = e;
    }
}

// Fused route + sort for at most 32 pairs (T * topk <= 32): T warps, a warp per
// token, then warp 0 sorts with a pair per lane. A match on the expert ids gives
// each pair its stable rank within its expert (lanes in pair order) and its
// expert's count; an expert's offset is the sum of the padded counts of the
// smaller expert ids present, read from the other lanes by shuffles. No pass
// over all E_tot experts and at most one block barrier (none for one token):
// a decode call waits on this chain alone.
template <int NV, bool SELECT, bool FULL>
__global__ void __launch_bounds__(kFusedThreads, 1) k_fused_tiny(RouteArgs a, SortArgs s)
{
    pdl_trigger_small();
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, SELECT, a.n_group > 0);
    int32_t* s_idx = reinterpret_cast<int32_t*>(smem + static_cast<size_t>(a.T) * L.bytes);
    float* s_w = reinterpret_cast<float*>(s_idx + kFusedTinyPairs);
    const int N = a.T * a.topk;
    pdl_wait();
    {
        unsigned char* wsm = smem + static_cast<size_t>(warp) * L.bytes;
        uint32_t warm = 0u;
        const int tok = warp;
        const float scale = route_row<kScore, InT, NV, SELECT, FULL>(a, tok, wsm, L, lane, warm);
        const size_t o = static_cast<size_t>(tok) * a.topk;
        const uint32_t* win_idx = reinterpret_cast<const uint32_t*>(wsm + L.win_idx);
        const float* win_val = reinterpret_cast<const float*>(wsm + L.win_val);
        if (lane < a.topk) {  // compact outputs, to shared and global
            const bool routed = lane < a.k_r;
            const int32_t id = routed ? static_cast<int32_t>(win_idx[lane]) : a.E + (lane - a.k_r);
            const float wv = routed ? __fmul_rn(win_val[lane], scale) : a.shared_weight;
            s_idx[o + lane] = id;
            s_w[o + lane] = wv;
            if (a.topk_idx) a.topk_idx[o + lane] = id;
            if (a.topk_w) a.topk_w[o + lane] = wv;
        }
    }
    if (a.T > 1) {
        __syncthreads();
    } else {
        __syncwarp();
    }
    if (warp != 0) return;
    // lane p: pair p (token p / topk, slot p % topk); ids outside [0, E_tot)
    // (NaN rows) are left out
    const int e = lane < N ? s_idx[lane] : -1;
    const bool valid = e >= 0 && e < s.E_tot;
    const uint32_t key = valid ? static_cast<uint32_t>(e) : 0xffffffffu;
    const uint32_t same = __match_any_sync(kFull, key);
    const uint32_t rank = static_cast<uint32_t>(__popc(same & ((1u << lane) - 1u)));
    const uint32_t c = static_cast<uint32_t>(__popc(same));
    const uint32_t bm = static_cast<uint32_t>(s.block_m);
    const uint32_t pad = s.bm_shift >= 0 ? ((c + bm - 1u) >> s.bm_shift) << s.bm_shift : (c + bm - 1u) / bm * bm;
    const uint32_t lead = (valid && rank == 0u) ? pad : 0u;  // each expert's padded count, once
    uint32_t off = 0u;
#pragma unroll 8
    for (int q = 0; q < N; ++q) {  // lanes N.. hold no pair
        const uint32_t kq = __shfl_sync(kFull, key, q);
        const uint32_t pq = __shfl_sync(kFull, lead, q);
        off += kq < key ? pq : 0u;
    }
    const uint32_t npp = __reduce_add_sync(kFull, lead);
    // every position a sentinel first, then the pairs over them (__syncwarp
    // orders the two sets of stores)
    for (uint32_t q = lane; q < npp; q += 32) {
        s.ids[q] = N;
        if (s.w) s.w[q] = 0.0f;
    }
    __syncwarp();
    if (valid) {
        s.ids[off + rank] = lane;
        if (s.w) s.w[off + rank] = s_w[lane];
        if (rank == 0u)
            for (uint32_t q = off; q < off + pad; q += bm)
                s.expert_ids[s.bm_shift >= 0 ? q >> s.bm_shift : q / bm] = e;
    }
    if (lane == 0) *s.num_post_pad = static_cast<int32_t>(npp);
}

// Fused route + sort for 32 < T * topk <= 128 pairs, T <= 16: T warps route a
// token each; warp 0 takes the pairs in four slots of 32 (pair 32 s + lane),
// gives each its stable rank from a match on the expert ids within the slot
// plus the count of its expert in the earlier slots (shared per-expert
// counters the slot's leaders advance), and scans the experts' padded counts;
// the CTA writes the sentinels, then warp 0 the pairs over them. Three block
// barriers.
template <int NV, bool SELECT, bool FULL>
__global__ void __launch_bounds__(kFusedThreads, 1) k_fused_small(RouteArgs a, SortArgs s)
{
    pdl_trigger_small();
    extern __shared__ __align__(16) unsigned char smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nt = blockDim.x;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, SELECT, a.n_group > 0);
    const int E_tot = s.E_tot;
    const SmallSortLayout F = small_sort_layout(E_tot);
    unsigned char* base = smem + static_cast<size_t>(a.T) * L.bytes;
    int32_t* s_idx = reinterpret_cast<int32_t*>(base + F.idx);
    float* s_w = reinterpret_cast<float*>(base + F.w);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(base + F.cnt);
    uint32_t* off = reinterpret_cast<uint32_t*>(base + F.off);
    uint32_t* s_npp = reinterpret_cast<uint32_t*>(base + F.npp);
    const int N = a.T * a.topk;
    const uint32_t bm = static_cast<uint32_t>(s.block_m);
    auto padded = [&](uint32_t c) {
        return s.bm_shift >= 0 ? ((c + bm - 1u) >> s.bm_shift) << s.bm_shift : (c + bm - 1u) / bm * bm;
    };
    for (int e = tid; e < E_tot; e += nt) cnt[e] = 0u;
    pdl_wait();
    {
        unsigned char* wsm = smem + static_cast<size_t>(warp) * L.bytes;
        uint32_t warm = 0u;
        const int tok = warp;
        const float scale = route_row<kScore, InT, NV, SELECT, FULL>(a, tok, wsm, L, lane, warm);
        const size_t o = static_cast<size_t>(tok) * a.topk;
        const uint32_t* win_idx = reinterpret_cast<const uint32_t*>(wsm + L.win_idx);
        const float* win_val = reinterpret_cast<const float*>(wsm + L.win_val);
        for (int j = lane; j < a.topk; j += 32) {  // compact outputs, to shared and global
            const bool routed = j < a.k_r;
            const int32_t id = routed ? static_cast<int32_t>(win_idx[j]) : a.E + (j - a.k_r);
            const float wv = routed ? __fmul_rn(win_val[j], scale) : a.shared_weight;
            s_idx[o + j] = id;
            s_w[o + j] = wv;
            if (a.topk_idx) a.topk_idx[o + j] = id;
            if (a.topk_w) a.topk_w[o + j] = wv;
        }
    }
    __syncthreads();  // pairs in shared memory, counters zeroed
    constexpr int kSlots = kFusedSmallPairs / 32;
    int e_s[kSlots];
    uint32_t rank_s[kSlots];
    if (warp == 0) {
        const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
        for (int sl = 0; sl < kSlots; ++sl) {
            const int p = sl * 32 + lane;
            const int e = p < N ? s_idx[p] : -1;
            // ids outside [0, E_tot) (NaN rows) are left out
            const bool valid = e >= 0 && e < E_tot;
            const uint32_t key = valid ? static_cast<uint32_t>(e) : 0xffffffffu;
            const uint32_t same = __match_any_sync(kFull, key);
            const int leader = __ffs(same) - 1;
            uint32_t b = 0u;
            if (valid && lane == leader) {  // the expert's count in the earlier slots, advanced by this one's
                b = cnt[e];
                cnt[e] = b + static_cast<uint32_t>(__popc(same));
            }
            b = __shfl_sync(kFull, b, leader);
            e_s[sl] = valid ? e : -1;
            rank_s[sl] = b + static_cast<uint32_t>(__popc(same & lt));
            __syncwarp();  // this slot's counts before the next slot reads them
        }
        // exclusive scan of the padded counts: lane l takes experts l*per ..
        const int per = (E_tot + 31) >> 5;
        const int e0 = lane * per, e1 = min(E_tot, e0 + per);
        uint32_t local = 0u;
        for (int e = e0; e < e1; ++e) local += padded(cnt[e]);
        uint32_t run = warp_exclusive_scan(local, lane);
        for (int e = e0; e < e1; ++e) {
            off[e] = run;
            run += padded(cnt[e]);
        }
        if (lane == 31) *s_npp = run;
    }
    __syncthreads();  // offsets and the padded total
    const uint32_t npp = *s_npp;
    for (uint32_t q = static_cast<uint32_t>(tid); q < npp; q += static_cast<uint32_t>(nt)) {
        s.ids[q] = N;
        if (s.w) s.w[q] = 0.0f;
    }
    __syncthreads();  // the sentinels before the pairs over them
    if (warp == 0) {
#pragma unroll
        for (int sl = 0; sl < kSlots; ++sl) {
            const int e = e_s[sl];
            if (e < 0) continue;
            const int p = sl * 32 + lane;
            const uint32_t oe = off[e];
            s.ids[oe + rank_s[sl]] = p;
            if (s.w) s.w[oe + rank_s[sl]] = s_w[p];
            if (rank_s[sl] == 0u)  // the expert's first pair writes its block ids
                for (uint32_t q = oe; q < oe + padded(cnt[e]); q += bm)
                    s.expert_ids[s.bm_shift >= 0 ? q >> s.bm_shift : q / bm] = e;
        }
        if (lane == 0) *s.num_post_pad = static_cast<int32_t>(npp);
    }
}

// Fused route + sort in one launch of one thread-block cluster (cs CTAs of 32
// warps): CTA r routes tokens [r*TP, min(T, (r+1)*TP)), a warp per token,
// writes the compact outputs and keeps the pairs in shared memory, then the
// cluster sorts all T*topk pairs (each CTA places its own pairs).
template <int NV, bool SELECT, bool FULL>
__global__ void __launch_bounds__(kClusterSortThreads, 1) k_fused_cluster(RouteArgs a, SortArgs s, int TP)
{
    pdl_trigger_small();
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, SELECT, a.n_group > 0);
    const int pairs = align16(TP * a.topk * 4);
    int32_t* s_idx = reinterpret_cast<int32_t*>(smem + static_cast<size_t>(nw) * L.bytes);
    float* s_w = reinterpret_cast<float*>(smem + static_cast<size_t>(nw) * L.bytes + pairs);
    unsigned char* sort_smem = smem + static_cast<size_t>(nw) * L.bytes + 2 * pairs;
    const int r = static_cast<int>(cluster_ctarank());
    const int t0 = min(a.T, r * TP), t1 = min(a.T, t0 + TP);
    pdl_wait();
    {
        unsigned char* wsm = smem + static_cast<size_t>(warp) * L.bytes;
        uint32_t warm = 0u;
        for (int tok = t0 + warp; tok < t1; tok += nw) {
            const float scale = route_row<kScore, InT, NV, SELECT, FULL>(a, tok, wsm, L, lane, warm);
            const size_t o = static_cast<size_t>(tok) * a.topk;
            const int lo = (tok - t0) * a.topk;
            const uint32_t* win_idx = reinterpret_cast<const uint32_t*>(wsm + L.win_idx);
            const float* win_val = reinterpret_cast<const float*>(wsm + L.win_val);
            for (int j = lane; j < a.topk; j += 32) {  // compact outputs, to shared and global
                const bool routed = j < a.k_r;
                const int32_t id = routed ? static_cast<int32_t>(win_idx[j]) : a.E + (j - a.k_r);
                const float wv = routed ? __fmul_rn(win_val[j], scale) : a.shared_weight;
                s_idx[lo + j] = id;
                s_w[lo + j] = wv;
                if (a.topk_idx) a.topk_idx[o + j] = id;
                if (a.topk_w) a.topk_w[o + j] = wv;
            }
            __syncwarp();
        }
    }
    __syncthreads();
    const int f0 = t0 * a.topk, f1 = t1 * a.topk;
    WarpRuns<kClusterSortUseSteps> R;
    const bool bad = warp_runs_load<kClusterSortUseSteps>(s_idx, s_w, f0, f0, f1, s.E_tot, R);
    cluster_sort_runs<kClusterSortUseSteps>(R, bad, a.T * a.topk, s.E_tot, s.block_m, sort_smem, s.ids, s.w,
                                            s.expert_ids, s.num_post_pad, a.status);
}

namespace {

using FwdFn = void (*)(RouteArgs);
using FusedFn = void (*)(RouteArgs, SortArgs);

template <bool SELECT, bool FULL, int RANKW = 2, bool SET = false>
FwdFn fwd_kernel(int nv_idx)
{
    switch (kNvBuckets[nv_idx]) {
        case 1: return k_router_fwd<1, SELECT, FULL, RANKW, SET>;
        case 2: return k_router_fwd<2, SELECT, FULL, RANKW, SET>;
        case 3: return k_router_fwd<3, SELECT, FULL, RANKW, SET>;
        case 4: return k_router_fwd<4, SELECT, FULL, RANKW, SET>;
        case 6: return k_router_fwd<6, SELECT, FULL, RANKW, SET>;
        case 8: return k_router_fwd<8, SELECT, FULL, RANKW, SET>;
    }
    return nullptr;
}

using ClusterFn = void (*)(RouteArgs, SortArgs, int);

template <bool SELECT, bool FULL>
ClusterFn cluster_kernel(int nv_idx)
{
    switch (kNvBuckets[nv_idx]) {
        case 1: return k_fused_cluster<1, SELECT, FULL>;
        case 2: return k_fused_cluster<2, SELECT, FULL>;
        case 3: return k_fused_cluster<3, SELECT, FULL>;
        case 4: return k_fused_cluster<4, SELECT, FULL>;
        case 6: return k_fused_cluster<6, SELECT, FULL>;
        case 8: return k_fused_cluster<8, SELECT, FULL>;
    }
    return nullptr;
}

template <bool SELECT, bool FULL>
FusedFn small_kernel(int nv_idx)
{
    switch (kNvBuckets[nv_idx]) {
        case 1: return k_fused_small<1, SELECT, FULL>;
        case 2: return k_fused_small<2, SELECT, FULL>;
        case 3: return k_fused_small<3, SELECT, FULL>;
        case 4: return k_fused_small<4, SELECT, FULL>;
        case 6: return k_fused_small<6, SELECT, FULL>;
        case 8: return k_fused_small<8, SELECT, FULL>;
    }
    return nullptr;
}

template <bool SELECT, bool FULL>
FusedFn tiny_kernel(int nv_idx)
{
    switch (kNvBuckets[nv_idx]) {
        case 1: return k_fused_tiny<1, SELECT, FULL>;
        case 2: return k_fused_tiny<2, SELECT, FULL>;
        case 3: return k_fused_tiny<3, SELECT, FULL>;
        case 4: return k_fused_tiny<4, SELECT, FULL>;
        case 6: return k_fused_tiny<6, SELECT, FULL>;
        case 8: return k_fused_tiny<8, SELECT, FULL>;
    }
    return nullptr;
}

template <bool SELECT, bool FULL>
FusedFn fused_kernel(int nv_idx, bool wide)
{
    if (wide) {
        switch (kNvBuckets[nv_idx]) {
            case 1: return k_fused_decode<1, SELECT, FULL, kFusedWideThreads>;
            case 2: return k_fused_decode<2, SELECT, FULL, kFusedWideThreads>;
        }
        return nullptr;
    }
    switch (kNvBuckets[nv_idx]) {
        case 1: return k_fused_decode<1, SELECT, FULL, kFusedThreads>;
        case 2: return k_fused_decode<2, SELECT, FULL, kFusedThreads>;
        case 3: return k_fused_decode<3, SELECT, FULL, kFusedThreads>;
        case 4: return k_fused_decode<4, SELECT, FULL, kFusedThreads>;
        case 6: return k_fused_decode<6, SELECT, FULL, kFusedThreads>;
        case 8: return k_fused_decode<8, SELECT, FULL, kFusedThreads>;
    }
    return nullptr;
}

}  // namespace

int MR_CAT(launch_fwd, MR_SUFFIX)(const RouteArgs& a, int nv_idx, bool select, cudaStream_t st)
{
    if (kNvBuckets[nv_idx] > kRegisterMaxNv) {
        // whole chunks and 16-byte aligned rows: the rows can be staged by bulk copies
        const bool full = a.vec && a.prefetch && a.E % 128 == 0;
        const FwdFn f = select ? (full ? k_router_fwd_wide<true, true> : k_router_fwd_wide<true, false>)
                               : (full ? k_router_fwd_wide<false, true> : k_router_fwd_wide<false, false>);
        const WideLayout L = wide_layout(a.k_r, a.stop, a.E, select, kScore == kSigmoid && !a.inter);
        const size_t smem = static_cast<size_t>(L.bytes) * (kWideThreads / 32);
        int err = ensure_smem(reinterpret_cast<const void*>(f), smem);
        if (err != cudaSuccess) return err;
        const long long ctas_needed = (static_cast<long long>(a.T) + kWideThreads / 32 - 1) / (kWideThreads / 32);
        const int grid = persistent_grid(reinterpret_cast<const void*>(f), kWideThreads, smem, ctas_needed);
        if (grid <= 0) return cudaErrorInvalidConfiguration;
        return launch_kernel(f, dim3(grid), dim3(kWideThreads), smem, st, 0, a);
    }
    // every chunk whole and vector-aligned: the specialisation without edge tests
    const bool full = a.vec && a.E == 128 * kNvBuckets[nv_idx];
    // more than 64 candidates possible (k_r > 32): rank three per lane per pass
    const bool rank3 = full && a.stop > 64;
    // no compact outputs and more than 64 candidates possible (k_r > 32): the
    // winners are selected as a set, without the candidate rank (at smaller k_r
    // the rank costs less than the bisection rounds to the exact threshold)
    const bool set_only = rank3 && !a.topk_idx && !a.topk_w;
    const FwdFn f = select ? (set_only ? fwd_kernel<true, true, 2, true>(nv_idx)
                              : rank3 ? fwd_kernel<true, true, 3>(nv_idx)
                                      : (full ? fwd_kernel<true, true>(nv_idx) : fwd_kernel<true, false>(nv_idx)))
                           : (full ? fwd_kernel<false, true>(nv_idx) : fwd_kernel<false, false>(nv_idx));
    if (!f) return cudaErrorInvalidValue;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, select, a.n_group > 0);
    const size_t smem = static_cast<size_t>(L.bytes) * (kFwdThreads / 32);
    int err = ensure_smem(reinterpret_cast<const void*>(f), smem);
    if (err != cudaSuccess) return err;
    const long long ctas_needed = (static_cast<long long>(a.T) + kFwdThreads / 32 - 1) / (kFwdThreads / 32);
    const int grid = persistent_grid(reinterpret_cast<const void*>(f), kFwdThreads, smem, ctas_needed);
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    return launch_kernel(f, dim3(grid), dim3(kFwdThreads), smem, st, 0, a);
}

// The cluster-fused call: returns cudaErrorNotSupported (nothing launched)
// when no cluster of this kernel fits the device for these sizes (the caller
// then runs the separate launches).
int MR_CAT(launch_fused_cluster, MR_SUFFIX)(const RouteArgs& a, const SortArgs& s, int nv_idx, bool select,
                                            cudaStream_t st)
{
    if (kNvBuckets[nv_idx] > kRegisterMaxNv) return cudaErrorNotSupported;
    const bool full = a.vec && a.E == 128 * kNvBuckets[nv_idx];
    const ClusterFn f = select ? (full ? cluster_kernel<true, true>(nv_idx) : cluster_kernel<true, false>(nv_idx))
                               : (full ? cluster_kernel<false, true>(nv_idx) : cluster_kernel<false, false>(nv_idx));
    if (!f) return cudaErrorNotSupported;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, select, a.n_group > 0);
    for (int cs : {16, 8}) {
        const int TP = (a.T + cs - 1) / cs;
        if (TP > kClusterSortThreads / 32 || TP * a.topk > kClusterSortThreads * kClusterSortUseSteps) continue;
        const size_t smem = static_cast<size_t>(L.bytes) * (kClusterSortThreads / 32) +
                            2 * static_cast<size_t>(align16(TP * a.topk * 4)) +
                            static_cast<size_t>(cluster_sort_layout(s.E_tot).bytes);
        if (!cluster_fits(reinterpret_cast<const void*>(f), kClusterSortThreads, smem, cs)) continue;
        return launch_kernel(f, dim3(cs), dim3(kClusterSortThreads), smem, st, cs, a, s, TP);
    }
    return cudaErrorNotSupported;
}

int MR_CAT(launch_fused, MR_SUFFIX)(const RouteArgs& a, const SortArgs& s, int nv_idx, bool select,
                                    cudaStream_t st)
{
    // every chunk whole and vector-aligned: the specialisation without edge tests
    // (a shorter instruction stream, which is what a decode call waits on)
    const bool full = a.vec && a.E == 128 * kNvBuckets[nv_idx];
    const bool wide = a.T > 16;  // one warp per token: 32 warps
    const FusedFn f = select ? (full ? fused_kernel<true, true>(nv_idx, wide) : fused_kernel<true, false>(nv_idx, wide))
                             : (full ? fused_kernel<false, true>(nv_idx, wide)
                                     : fused_kernel<false, false>(nv_idx, wide));
    if (!f) return cudaErrorInvalidValue;
    const int threads = wide ? kFusedWideThreads : kFusedThreads;
    const int nw = threads / 32;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, select, a.n_group > 0);
    const size_t smem = static_cast<size_t>(L.bytes) * nw +
                        fused_sort_layout(a.T * a.topk, s.E_tot, s.block_m, wide ? 8 : 4).bytes;
    int err = ensure_smem(reinterpret_cast<const void*>(f), smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(f, dim3(1), dim3(threads), smem, st, 0, a, s);
}

int MR_CAT(launch_fused_tiny, MR_SUFFIX)(const RouteArgs& a, const SortArgs& s, int nv_idx, bool select,
                                         cudaStream_t st)
{
    const bool full = a.vec && a.E == 128 * kNvBuckets[nv_idx];
    const FusedFn f = select ? (full ? tiny_kernel<true, true>(nv_idx) : tiny_kernel<true, false>(nv_idx))
                             : (full ? tiny_kernel<false, true>(nv_idx) : tiny_kernel<false, false>(nv_idx));
    if (!f) return cudaErrorInvalidValue;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, select, a.n_group > 0);
    const size_t smem = static_cast<size_t>(L.bytes) * a.T + 2 * kFusedTinyPairs * 4;
    int err = ensure_smem(reinterpret_cast<const void*>(f), smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(f, dim3(1), dim3(32 * a.T), smem, st, 0, a, s);
}

int MR_CAT(launch_fused_small, MR_SUFFIX)(const RouteArgs& a, const SortArgs& s, int nv_idx, bool select,
                                          cudaStream_t st)
{
    const bool full = a.vec && a.E == 128 * kNvBuckets[nv_idx];
    const FusedFn f = select ? (full ? small_kernel<true, true>(nv_idx) : small_kernel<true, false>(nv_idx))
                             : (full ? small_kernel<false, true>(nv_idx) : small_kernel<false, false>(nv_idx));
    if (!f) return cudaErrorInvalidValue;
    const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, select, a.n_group > 0);
    const size_t smem = static_cast<size_t>(L.bytes) * a.T + small_sort_layout(s.E_tot).bytes;
    int err = ensure_smem(reinterpret_cast<const void*>(f), smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(f, dim3(1), dim3(32 * a.T), smem, st, 0, a, s);
}

}  // namespace mr
