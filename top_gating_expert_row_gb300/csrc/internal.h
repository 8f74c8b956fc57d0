// Host-side interface between the C ABI (api.cu) and the kernel translation
// units. Not installed; not part of the public header.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "route.cuh"
#include "sort.cuh"

namespace mr {

constexpr int kFwdThreads = 256;     // 8 warps, one token row per warp at a time
constexpr int kFusedThreads = 512;   // 16 warps: one per decode token, then the whole CTA sorts

// Register-resident row widths: NV chunks of 128 elements per row (E <= 2304).
constexpr int kNvBuckets[] = {1, 2, 3, 4, 6, 8, 12, 18};
constexpr int kNumNv = sizeof(kNvBuckets) / sizeof(kNvBuckets[0]);

// Index into kNvBuckets of the smallest width that holds E experts, or -1.
inline int nv_index(int E)
{
    const int need = (E + 127) / 128;
    for (int i = 0; i < kNumNv; ++i)
        if (kNvBuckets[i] >= need) return i;
    return -1;
}

// The forward's row bucket for E: the register-resident buckets up to 2304,
// the last (shared-memory rows, any width up to MR_MAX_EXPERTS) beyond; -1 past
// MR_MAX_EXPERTS (passed in as max_e).
inline int fwd_nv_index(int E, int max_e)
{
    const int i = nv_index(E);
    if (i >= 0) return i;
    return E <= max_e ? kNumNv - 1 : -1;
}

// The one-CTA fused decode kernel keeps rows up to this many chunks (E <= 1024).
constexpr int kFusedMaxNv = 8;
// 16 < T <= 64 (E <= 256): the same one-CTA kernel with 32 warps, each routing
// up to two tokens, and 64-bit token masks
constexpr int kFusedWideThreads = 1024;
constexpr int kFusedWideMaxNv = 2;
constexpr int kFusedWideMaxTokens = 64;
// T * topk <= 32 pairs (rows of E <= 1024): T warps route, one warp sorts
constexpr int kFusedTinyPairs = 32;
// T * topk <= 128 pairs, T <= 16: T warps route, one warp ranks the pairs (up
// to four per lane) and scans the experts' padded counts, the CTA writes the
// sentinels
constexpr int kFusedSmallPairs = 128;
// shared memory of that kernel after the warp regions: pairs (ids, weights),
// per-expert counts and offsets, the padded total
struct SmallSortLayout {
    int idx, w, cnt, off, npp, bytes;
};
__host__ __device__ inline SmallSortLayout small_sort_layout(int E_tot)
{
    SmallSortLayout F;
    int o = 0;
    F.idx = o; o += kFusedSmallPairs * 4;
    F.w = o; o += kFusedSmallPairs * 4;
    F.cnt = o; o += (E_tot * 4 + 15) / 16 * 16;
    F.off = o; o += (E_tot * 4 + 15) / 16 * 16;
    F.npp = o; o += 16;
    F.bytes = o;
    return F;
}
// whether moe_router_fused_fwd_sort runs as one launch for T tokens of row bucket nv
inline bool fused_one_launch(int T, int nv_bucket)
{
    return (T <= 16 && nv_bucket <= kFusedMaxNv) || (T <= kFusedWideMaxTokens && nv_bucket <= kFusedWideMaxNv);
}
// The forward keeps rows of up to this many chunks in registers (E <= 1024);
// wider rows take the shared-memory routine, two warps per CTA.
constexpr int kRegisterMaxNv = 8;
// Resident CTAs per SM the forward's register budget is sized for (the row's
// keys take 4*NV registers per lane). At NV = 4 (E = 512) five CTAs (48
// registers, a few bytes of spills) measured faster than four; at NV = 3 the
// spills cost more than the extra CTA gains.
constexpr int fwd_min_blocks(int nv) { return nv >= 12 ? 2 : (nv >= 6 ? 3 : (nv == 4 ? 5 : 4)); }
constexpr int kWideThreads = 64;
// Registers are capped so that shared memory, not registers, bounds residency
// (a 9 KB key row per warp at E = 2304 allows about 22 warps per SM).
constexpr int kWideMinBlocks = 10;
constexpr int kAuxThreads = 256;        // aux-loss kernels: 8 warps over the rows of one 128-column slab
constexpr int kAuxRowsPerChunk = 256;   // rows per aux-loss CTA (before the cap on chunks)
constexpr int kAuxMaxChunks = 256;      // row chunks of the aux-loss forward (workspace = chunks * E floats)

struct SortArgs {
    int32_t* ids;
    float* w;
    int32_t* expert_ids;
    int32_t* num_post_pad;
    int E_tot;
    int block_m;
    int bm_shift;  // log2(block_m) when block_m is a power of two, else -1
};

inline int log2_if_pow2(int x)
{
    if (x <= 0 || (x & (x - 1))) return -1;
    int s = 0;
    while ((1 << s) < x) ++s;
    return s;
}

// Shared memory of the fused decode kernel after the warp regions: the T*topk
// pairs, one token bitmask per expert, the padded offsets, the counts and the
// block -> expert map.
struct FusedSortLayout {
    int idx, w, mask, off, cnt, blk, bytes;
};

// mask_bytes: bytes of one expert's token mask (4 for T <= 32, 8 for T <= 64)
__host__ __device__ inline FusedSortLayout fused_sort_layout(int N, int E_tot, int bm, int mask_bytes)
{
    FusedSortLayout F;
    const int nonempty = N < E_tot ? N : E_tot;
    const int nblk = (N + nonempty * (bm - 1) + bm - 1) / bm;
    int o = 0;
    F.idx = o; o += align16(N * 4);
    F.w = o; o += align16(N * 4);
    F.mask = o; o += align16(E_tot * mask_bytes);
    F.off = o; o += align16((E_tot + 1) * 4);
    F.cnt = o; o += align16(E_tot * 4);
    F.blk = o; o += align16((nblk > 0 ? nblk : 1) * 4);
    F.bytes = o;
    return F;
}

// Launch helpers; each returns a cudaError_t value (cudaSuccess on success).
int launch_fwd(int score_fn, int in_dtype, const RouteArgs& a, int nv_idx, bool select,
               cudaStream_t st);
int launch_fused_decode(int score_fn, int in_dtype, const RouteArgs& a, const SortArgs& s,
                        int nv_idx, bool select, cudaStream_t st);
int launch_fused_tiny(int score_fn, int in_dtype, const RouteArgs& a, const SortArgs& s, int nv_idx,
                      bool select, cudaStream_t st);
int launch_fused_small(int score_fn, int in_dtype, const RouteArgs& a, const SortArgs& s, int nv_idx,
                       bool select, cudaStream_t st);
// The fused call as one launch of one thread-block cluster (a warp per token);
// cudaErrorNotSupported, with nothing launched, when no cluster fits.
int launch_fused_cluster(int score_fn, int in_dtype, const RouteArgs& a, const SortArgs& s, int nv_idx,
                         bool select, cudaStream_t st);
// Tokens the cluster-fused call takes at most (32 per CTA, 16 CTAs).
constexpr int kFusedClusterMaxTokens = 512;
int launch_bwd(int score_fn, int nv_idx, const float* g, const float* s, const uint8_t* m,
               float* dx, int T, int E, int renorm, float scaling, bool vec, cudaStream_t st);
int launch_bwd_bf16(int score_fn, int nv_idx, const __nv_bfloat16* g, const float* s, const uint8_t* m,
                    __nv_bfloat16* dx, int T, int E, int renorm, float scaling, bool vec, cudaStream_t st);
int launch_sort(const int32_t* idx, const float* w, int N, int E_tot, int block_m, int32_t* ids,
                float* sw, int32_t* eids, int32_t* npp, uint32_t* ws, int32_t* status,
                cudaStream_t st);
// The multi-CTA sort's second launch on chunks of PC pairs (nchunk_pad CTAs, a
// multiple of kClusterChunks) whose within-cluster prefixes and cluster totals
// are in pre / ctot.
int launch_sort_scatter(const int32_t* idx, const float* w, int N, int PC, int nchunk_pad, int E_tot, int block_m,
                        const uint32_t* pre, const uint32_t* ctot, int32_t* ids, float* sw, int32_t* eids,
                        int32_t* npp, cudaStream_t st);
int launch_expf(const float* x, float* y, int n, cudaStream_t st);
int aux_chunks(long long T);
size_t aux_workspace_bytes(long long T, int E);
int launch_aux_loss_fwd(const float* probs, const int32_t* tokens_per_expert, int T, int E, double C, float* loss,
                        void* workspace, cudaStream_t st);
int launch_aux_loss_bwd(const int32_t* tokens_per_expert, const float* grad_loss, int T, int E, double C,
                        float* grad_probs, cudaStream_t st);
int launch_tokens_per_expert(const uint8_t* map, int T, int E, int32_t* out, cudaStream_t st);
int launch_noop(cudaStream_t st);

// Chunking of the multi-CTA sort: PC pairs per CTA, nchunk CTAs padded to whole
// clusters. At most kSortChunk pairs take the one-CTA sort. Larger sorts use
// chunks of about N/256 pairs (1024..4096, multiples of 512) so that the grid
// spreads over the GPU; with more than 1024 experts the per-CTA cost of the
// expert-wide steps dominates, so chunks stay at 4096.
struct SortPlan {
    int pc, nchunk, nchunk_pad;
};

inline SortPlan sort_plan(long long N, int E_tot)
{
    long long pc = kSortChunk;
    if (N > kSortChunk && E_tot <= 1024) {
        pc = ((N + 255) / 256 + 511) / 512 * 512;
        pc = pc < 1024 ? 1024 : (pc > kSortChunk ? kSortChunk : pc);
    }
    SortPlan p;
    p.pc = static_cast<int>(pc);
    p.nchunk = N <= 0 ? 1 : static_cast<int>((N + pc - 1) / pc);
    p.nchunk_pad = (p.nchunk + kClusterChunks - 1) / kClusterChunks * kClusterChunks;
    return p;
}

// Workspace of the sort: the per-chunk prefixes and the cluster totals (none for
// the one-CTA sort).
inline size_t sort_table_bytes(int nchunk_pad, int E_tot)
{
    return (static_cast<size_t>(nchunk_pad) + nchunk_pad / kClusterChunks) * static_cast<size_t>(E_tot) * 4;
}

inline size_t sort_ws_bytes(long long N, int E_tot)
{
    if (N <= kSortChunk) return 0;
    return sort_table_bytes(sort_plan(N, E_tot).nchunk_pad, E_tot);
}

// Whether launches let the next kernel of the stream start while this one
// finishes (programmatic dependent launch; moe_router_set_launch_overlap).
bool launch_overlap();

// Launches kernel(args...) on st with `cluster` CTAs per cluster (0: none, or
// the kernel's compile-time size) and, when launch_overlap(), the
// programmatic-serialization attribute (the kernel may start before the
// previous one in the stream completes; it waits for it in pdl_wait). Returns
// a cudaError_t value.
template <typename... KArgs, typename... Args>
int launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, int cluster,
                  Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (launch_overlap()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Persistent-grid size: min(units, SMs x resident CTAs) for a kernel; with
// balance, reduced to the fewest CTAs that take the same number of rounds.
int persistent_grid(const void* func, int threads, size_t smem, long long units, bool balance = false);
// Raise a kernel's dynamic shared-memory limit when needed.
int ensure_smem(const void* func, size_t smem);
// Whether a cluster of cs CTAs of this kernel (threads each, smem bytes of
// dynamic shared memory) fits on the current device; sets the kernel's
// shared-memory limit and, for cs > 8, allows non-portable cluster sizes.
// Cached.
bool cluster_fits(const void* func, int threads, size_t smem, int cs);

}  // namespace mr
