// C ABI of the MoE routing library: argument validation (before anything is
// enqueued), path and grid selection, and the launches. Host checks follow
// TransformerEngine PR 3012 "Hardening" (T*E <= INT_MAX, topk in [1, E],
// topk % group_topk == 0) plus this library's own limits.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "moe_router.h"
#include "internal.h"

namespace mr {

// ---- launch configuration helpers -------------------------------------------------------------

namespace {
struct OccEntry {
    const void* func;
    size_t smem;
    int device;
    int blocks;
};
std::mutex g_occ_mu;
OccEntry g_occ[128];
int g_occ_n = 0;

struct SmemEntry {
    const void* func;
    int device;
    size_t bytes;
};
SmemEntry g_smem[128];
int g_smem_n = 0;

int g_sm_count[64] = {0};
}  // namespace

int persistent_grid(const void* func, int threads, size_t smem, long long units, bool balance)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    std::lock_guard<std::mutex> lk(g_occ_mu);
    if (dev < 0 || dev >= 64) return -1;
    if (g_sm_count[dev] == 0) {
        if (cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return -1;
    }
    int blocks = -1;
    for (int i = 0; i < g_occ_n; ++i)
        if (g_occ[i].func == func && g_occ[i].smem == smem && g_occ[i].device == dev) blocks = g_occ[i].blocks;
    if (blocks < 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, func, threads, smem) != cudaSuccess) return -1;
        if (g_occ_n < 128) g_occ[g_occ_n++] = OccEntry{func, smem, dev, blocks};
    }
    if (blocks < 1) return -1;
    const long long cap = static_cast<long long>(blocks) * g_sm_count[dev];
    long long g = units < cap ? units : cap;
    if (g < 1) return 1;
    if (balance) {
        // as many CTAs as give every CTA the same number of rounds: with the
        // full capacity the last round runs on only part of the GPU, while the
        // same rounds on fewer CTAs keep every SM busy to the end (the backward,
        // bound by memory, gains; the forwards lose more latency hiding than the
        // idle tail costs them)
        const long long rounds = (units + g - 1) / g;
        g = (units + rounds - 1) / rounds;
    }
    return static_cast<int>(g);
}

// The limit is only ever raised: one entry per (kernel, device) remembers the
// largest size set, so a later launch with less shared memory never lowers the
// limit another size relies on.
int ensure_smem(const void* func, size_t bytes)
{
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_occ_mu);
    SmemEntry* ent = nullptr;
    for (int i = 0; i < g_smem_n; ++i)
        if (g_smem[i].func == func && g_smem[i].device == dev) ent = &g_smem[i];
    if (ent && ent->bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    if (ent) ent->bytes = bytes;
    else if (g_smem_n < 128) g_smem[g_smem_n++] = SmemEntry{func, dev, bytes};
    return cudaSuccess;
}

bool cluster_fits(const void* func, int threads, size_t smem, int cs)
{
    struct Entry {
        const void* func;
        size_t smem;
        int dev, cs;
        bool fits;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int n = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < n; ++i)
            if (cache[i].func == func && cache[i].smem == smem && cache[i].dev == dev && cache[i].cs == cs)
                return cache[i].fits;
    }
    bool fits = false;
    int maxsm = 0;
    if (cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess &&
        smem <= static_cast<size_t>(maxsm) && ensure_smem(func, smem) == cudaSuccess &&
        (cs <= 8 || cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs, 1, 1);
        cfg.blockDim = dim3(threads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = cs;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int clusters = 0;
        fits = cudaOccupancyMaxActiveClusters(&clusters, func, &cfg) == cudaSuccess && clusters >= 1;
    }
    cudaGetLastError();  // a refused size is not an error of the call
    std::lock_guard<std::mutex> lk(mu);
    if (n < 64) cache[n++] = Entry{func, smem, dev, cs, fits};
    return fits;
}

// ---- per-(score, dtype) launchers defined in fwd.cu compilations --------------------------------

int launch_fused_cluster_s0_d0(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_cluster_s0_d1(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_cluster_s1_d0(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_cluster_s1_d1(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fwd_s0_d0(const RouteArgs&, int, bool, cudaStream_t);
int launch_fwd_s0_d1(const RouteArgs&, int, bool, cudaStream_t);
int launch_fwd_s1_d0(const RouteArgs&, int, bool, cudaStream_t);
int launch_fwd_s1_d1(const RouteArgs&, int, bool, cudaStream_t);
int launch_fused_s0_d0(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_s0_d1(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_s1_d0(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_s1_d1(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_tiny_s0_d0(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_tiny_s0_d1(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_tiny_s1_d0(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_tiny_s1_d1(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_small_s0_d0(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_small_s0_d1(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_small_s1_d0(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);
int launch_fused_small_s1_d1(const RouteArgs&, const SortArgs&, int, bool, cudaStream_t);

int launch_fwd(int score_fn, int in_dtype, const RouteArgs& a, int nv_idx, bool select, cudaStream_t st)
{
    if (score_fn == kSoftmax)
        return in_dtype ? launch_fwd_s0_d1(a, nv_idx, select, st) : launch_fwd_s0_d0(a, nv_idx, select, st);
    return in_dtype ? launch_fwd_s1_d1(a, nv_idx, select, st) : launch_fwd_s1_d0(a, nv_idx, select, st);
}

int launch_fused_cluster(int score_fn, int in_dtype, const RouteArgs& a, const SortArgs& s, int nv_idx, bool select,
                         cudaStream_t st)
{
    auto f = score_fn == kSoftmax ? (in_dtype ? launch_fused_cluster_s0_d1 : launch_fused_cluster_s0_d0)
                                  : (in_dtype ? launch_fused_cluster_s1_d1 : launch_fused_cluster_s1_d0);
    return f(a, s, nv_idx, select, st);
}

int launch_fused_decode(int score_fn, int in_dtype, const RouteArgs& a, const SortArgs& s, int nv_idx,
                        bool select, cudaStream_t st)
{
    if (score_fn == kSoftmax)
        return in_dtype ? launch_fused_s0_d1(a, s, nv_idx, select, st) : launch_fused_s0_d0(a, s, nv_idx, select, st);
    return in_dtype ? launch_fused_s1_d1(a, s, nv_idx, select, st) : launch_fused_s1_d0(a, s, nv_idx, select, st);
}

int launch_fused_tiny(int score_fn, int in_dtype, const RouteArgs& a, const SortArgs& s, int nv_idx, bool select,
                      cudaStream_t st)
{
    if (score_fn == kSoftmax)
        return in_dtype ? launch_fused_tiny_s0_d1(a, s, nv_idx, select, st)
                        : launch_fused_tiny_s0_d0(a, s, nv_idx, select, st);
    return in_dtype ? launch_fused_tiny_s1_d1(a, s, nv_idx, select, st) : launch_fused_tiny_s1_d0(a, s, nv_idx, select, st);
}

int launch_fused_small(int score_fn, int in_dtype, const RouteArgs& a, const SortArgs& s, int nv_idx, bool select,
                       cudaStream_t st)
{
    if (score_fn == kSoftmax)
        return in_dtype ? launch_fused_small_s0_d1(a, s, nv_idx, select, st)
                        : launch_fused_small_s0_d0(a, s, nv_idx, select, st);
    return in_dtype ? launch_fused_small_s1_d1(a, s, nv_idx, select, st)
                    : launch_fused_small_s1_d0(a, s, nv_idx, select, st);
}

// ---- launch overlap ---------------------------------------------------------------------------

namespace {
std::atomic<int>& overlap_flag();
}

bool launch_overlap() { return overlap_flag().load(std::memory_order_relaxed) != 0; }

// ---- diagnostics ------------------------------------------------------------------------------

// Evaluates the specification through both device forms the kernels use, the
// scalar exp_f32 and the packed exp_spec2 (on the pair (x[i], -x[i])), and
// writes the scalar result; a NaN with payload 0x0badba is written instead
// wherever the two forms disagree for a non-NaN input, and likewise where the
// softmax-value exponential's packed form exp_value2 disagrees with its
// scalar form exp_value on (-|x[i]|, -|x[i]|/2).
__global__ void k_expf(const float* x, float* y, int n)
{
    pdl_trigger_small();
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const float v = x[i];
        const float s = exp_f32(v);
        const float2 p = exp_spec2(make_float2(v, -v));
        const float a = -fabsf(v), b = __fmul_rn(a, 0.5f);
        const float2 q = exp_value2(make_float2(a, b));
        const bool same = (v != v) || (__float_as_uint(p.x) == __float_as_uint(s) &&
                                       __float_as_uint(p.y) == __float_as_uint(exp_f32(-v)) &&
                                       __float_as_uint(q.x) == __float_as_uint(exp_value(a)) &&
                                       __float_as_uint(q.y) == __float_as_uint(exp_value(b)));
        y[i] = same ? s : __uint_as_float(0x7f8badbau);
    }
}

// The softmax-value exponential on each input (the forward's numerators).
__global__ void k_exp_value(const float* x, float* y, int n)
{
    pdl_trigger_small();
    pdl_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) y[i] = exp_value(x[i]);
}

// The decode launch floor: an empty kernel launched the way the routing
// kernels are (it takes part in the launch overlap like them).
__global__ void k_noop()
{
    pdl_trigger_small();
    pdl_wait();
}

int launch_expf(const float* x, float* y, int n, cudaStream_t st)
{
    const long long blocks = (static_cast<long long>(n) + 255) / 256;
    const int grid = static_cast<int>(blocks < 4096 ? blocks : 4096);
    return launch_kernel(k_expf, dim3(grid), dim3(256), 0, st, 0, x, y, n);
}

int launch_noop(cudaStream_t st)
{
    return launch_kernel(k_noop, dim3(1), dim3(32), 0, st, 0);
}

// ---- device status word ------------------------------------------------------------------------

static_assert(MR_MAX_FUSED_TOKENS == 16 && MR_MAX_FUSED_TOKENS_SMALL_E == kFusedWideMaxTokens &&
                  MR_MAX_FUSED_EXPERTS_SMALL == 128 * kFusedWideMaxNv,
              "the header's fused-launch limits and the kernels' must agree");
static_assert(kStatusTimeout == MR_ETIMEOUT && kStatusRange == MR_ERANGE,
              "the device status codes and the C ABI's must agree");

// The library's status word on each device: kernels whose waits are bounded
// raise it to MR_ETIMEOUT when one gives up and the call had no status word.
static __device__ int32_t g_device_status;

__global__ void k_take_status(int32_t* word, int32_t* out, int clear)
{
    pdl_trigger_small();
    pdl_wait();
    out[0] = *word;
    if (clear) *word = 0;
}

namespace {
std::mutex g_status_mu;
void* g_status_ptr[64] = {nullptr};

// Device address of g_device_status on the current device, looked up once per
// device and cached (nullptr on failure).
int32_t* device_status_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = ptr;
    }
    return static_cast<int32_t*>(g_status_ptr[dev]);
}
}  // namespace

// ---- top-k path configuration -----------------------------------------------------------------

namespace {
// Read by every launch and set by moe_router_set_topk_path, possibly from
// other host threads: atomics (relaxed: each value stands alone).
struct PathConfig {
    std::atomic<int> threshold{8};
    std::atomic<int> force{0};  // 0 by threshold, 1 arg-max, 2 threshold-select
    PathConfig()
    {
        if (const char* t = std::getenv("MR_TOPK_SELECT_THRESHOLD")) {
            const int v = std::atoi(t);
            if (v >= 0) threshold.store(v, std::memory_order_relaxed);
        }
        if (const char* f = std::getenv("MR_FORCE_PATH")) {
            if (!std::strcmp(f, "argmax")) force.store(1, std::memory_order_relaxed);
            else if (!std::strcmp(f, "select")) force.store(2, std::memory_order_relaxed);
        }
    }
    int forced() const { return force.load(std::memory_order_relaxed); }
};
PathConfig g_path;

// Programmatic dependent launch of every kernel (moe_router_set_launch_overlap;
// on unless the environment sets MR_LAUNCH_OVERLAP=0).
std::atomic<int>& overlap_flag()
{
    static std::atomic<int> flag{[] {
        const char* v = std::getenv("MR_LAUNCH_OVERLAP");
        return (v && v[0] == '0') ? 0 : 1;
    }()};
    return flag;
}

// Test hook for the bounded waits (moe_router_set_wait_test).
struct WaitTest {
    std::atomic<unsigned> tries{0};  // 0: kWaitLimit
    std::atomic<int> drop{0};
};
WaitTest g_wait_test;

bool use_select(int k_r)
{
    const int f = g_path.forced();
    return f == 2 || (f == 0 && k_r >= g_path.threshold.load(std::memory_order_relaxed));
}

int select_stop(int k_r)
{
    int s = 2 * k_r > 64 ? 2 * k_r : 64;
    return (s + 31) & ~31;
}

// Rung of the lanes'-maxima ladder (warp_kth_largest) tried as a pivot when a
// row has no usable previous threshold: the first j whose expected count of
// keys at or above it reaches max(k_r + 4, 1.4 k_r) (capped at stop), for rows
// of n similar entries over the lanes that hold any (a lane holds 4 of every
// 128 experts: all 32 lanes from n = 128 on). The j-th largest of L lane
// maxima sits near the (L + 1 - j) / (L + 1) quantile of a lane's maximum,
// i.e. that quantile's m-th root (m = n / L keys per lane) for one key. With
// k_r <= L the rung is at least k_r, so its count never falls short of k_r.
int route_rung(int n, int k_r, int stop)
{
    if (k_r < 1 || n < 1) return 0;
    const int lanes = n >= 128 ? 32 : (n + 3) / 4;
    const double m = static_cast<double>(n) / lanes;
    const double target = std::min<double>(stop, std::max(k_r + 4.0, 1.4 * k_r));
    int j = lanes;
    for (int r = 1; r <= lanes; ++r)
        if (n * (1.0 - std::pow((lanes + 1.0 - r) / (lanes + 1.0), 1.0 / m)) >= target) {
            j = r;
            break;
        }
    return k_r <= lanes && j < k_r ? k_r : j;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int from_cuda(int e) { return e == cudaSuccess ? MR_OK : MR_ECUDA; }

// Validation shared by the forward calls. Returns MR_OK or an error code.
int check_router(const mr_router_params* p)
{
    if (!p) return MR_EINVAL;
    if (p->T < 0 || p->E < 1 || p->topk < 1 || p->n_shared < 0) return MR_EINVAL;
    if (p->score_fn != MR_SOFTMAX && p->score_fn != MR_SIGMOID) return MR_EINVAL;
    if (p->in_dtype != MR_F32 && p->in_dtype != MR_BF16) return MR_EINVAL;
    const int k_r = p->topk - p->n_shared;
    if (k_r < 1 || k_r > p->E) return MR_EINVAL;
    if (static_cast<long long>(p->T) * p->E > INT_MAX) return MR_EINVAL;
    if (static_cast<long long>(p->T) * p->topk >= INT_MAX) return MR_EINVAL;
    if (p->n_group < 0) return MR_EINVAL;
    if (p->n_group > 0) {
        if (p->E % p->n_group != 0) return MR_EINVAL;
        if (p->topk_group < 1 || p->topk_group > p->n_group) return MR_EINVAL;
        if (k_r % p->topk_group != 0) return MR_EINVAL;
        if (k_r / p->topk_group > p->E / p->n_group) return MR_EINVAL;
    }
    if (p->E > MR_MAX_EXPERTS || k_r > MR_MAX_TOPK) return MR_EUNSUPPORTED;
    if (p->n_group > MR_MAX_GROUPS) return MR_EUNSUPPORTED;
    if (p->n_group > 0 && k_r / p->topk_group > MR_MAX_GROUP_TOPK) return MR_EUNSUPPORTED;
    if (p->score_fn == MR_SOFTMAX && (p->bias || p->n_group > 0)) return MR_EUNSUPPORTED;
    return MR_OK;
}

RouteArgs route_args(const mr_router_params* p, const void* logits, void* probs, uint8_t* map, float* inter,
                     int32_t* idx, float* w, int32_t* status)
{
    RouteArgs a;
    a.logits = logits;
    a.bias = p->bias;
    a.probs = probs;
    a.map = map;
    a.inter = inter;
    a.topk_idx = idx;
    a.topk_w = w;
    a.T = p->T;
    a.E = p->E;
    a.topk = p->topk;
    a.n_shared = p->n_shared;
    a.k_r = p->topk - p->n_shared;
    a.renorm = p->renorm ? 1 : 0;
    a.n_group = p->n_group;
    a.topk_group = p->n_group > 0 ? p->topk_group : 0;
    a.scaling = p->scaling;
    a.shared_weight = p->shared_weight;
    a.stop = select_stop(a.k_r);
    a.rung = route_rung(a.n_group > 0 ? a.topk_group * (a.E / a.n_group) : a.E, a.k_r, a.stop);
    a.status = status ? status : device_status_address();
    const unsigned tries = g_wait_test.tries.load(std::memory_order_relaxed);
    a.wait_tries = tries ? tries : kWaitLimit;
    a.drop_copies = g_wait_test.drop.load(std::memory_order_relaxed);
    a.warm_code = 0;
    const uintptr_t in_al = p->in_dtype == MR_BF16 ? 8 : 16;
    a.vec = (p->E % 4 == 0) && aligned(logits, in_al) && aligned(probs, in_al) && aligned(inter, 16) &&
            aligned(map, 4) && aligned(p->bias, 16);
    const size_t row_bytes = static_cast<size_t>(p->E) * (p->in_dtype == MR_BF16 ? 2 : 4);
    a.prefetch = a.vec && row_bytes % 16 == 0 && aligned(logits, 16);
    return a;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int check_sort(int T, int topk, int E_tot, int block_m)
{
    if (T < 0 || topk < 1 || E_tot < 1 || block_m < 1) return MR_EINVAL;
    const long long N = static_cast<long long>(T) * topk;
    if (N >= INT_MAX) return MR_EINVAL;
    const long long nonempty = N < E_tot ? N : E_tot;
    if (N + nonempty * (block_m - 1) >= INT_MAX) return MR_EINVAL;
    if (E_tot > MR_MAX_SORT_EXPERTS) return MR_EUNSUPPORTED;
    return MR_OK;
}
}  // namespace

// ---- allocation-free sort: scratch in a file-scope device array ----------------------------------

// Scratch of moe_sort_noalloc: the per-chunk expert-count table that moe_sort
// keeps in its caller's workspace. Every GPU that loads the library holds this
// array until the process exits; all calls on a device share it.
static __device__ __align__(256) uint32_t g_sort_scratch[MR_SORT_NOALLOC_SCRATCH_BYTES / 4];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {nullptr};

// Device address of g_sort_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device with that device current and cached. Returns nullptr on failure.
void* sort_scratch_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_sort_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}
}  // namespace

}  // namespace mr

using namespace mr;

extern "C" {

const char* moe_router_strerror(int code)
{
    switch (code) {
        case MR_OK: return "MR_OK: success";
        case MR_EINVAL: return "MR_EINVAL: invalid argument";
        case MR_EUNSUPPORTED: return "MR_EUNSUPPORTED: outside the library's supported limits";
        case MR_ECUDA: return "MR_ECUDA: CUDA launch or query failed";
        case MR_ERANGE: return "MR_ERANGE: expert id out of range (dropped)";
        case MR_ETIMEOUT: return "MR_ETIMEOUT: a bounded in-kernel wait gave up (outputs not valid)";
    }
    return "unknown moe_router status";
}

int moe_router_set_launch_overlap(int enable)
{
    if (enable != 0 && enable != 1) return MR_EINVAL;
    overlap_flag().store(enable, std::memory_order_relaxed);
    return MR_OK;
}

int moe_router_set_wait_test(unsigned int tries, int drop_copies)
{
    if (drop_copies != 0 && drop_copies != 1) return MR_EINVAL;
    g_wait_test.tries.store(tries, std::memory_order_relaxed);
    g_wait_test.drop.store(drop_copies, std::memory_order_relaxed);
    return MR_OK;
}

int moe_router_set_topk_path(int select_threshold, int force_path)
{
    if (select_threshold < 0 || force_path < 0 || force_path > 2) return MR_EINVAL;
    g_path.threshold.store(select_threshold, std::memory_order_relaxed);
    g_path.force.store(force_path, std::memory_order_relaxed);
    return MR_OK;
}

int moe_router_fwd(const mr_router_params* p, const void* logits, void* probs, uint8_t* routing_map,
                   float* intermediate, int32_t* topk_idx, float* topk_w, int32_t* status, mr_stream_t stream)
{
    int rc = check_router(p);
    if (rc != MR_OK) return rc;
    if (!logits) return MR_EINVAL;
    if (!probs && !routing_map && !intermediate && !topk_idx && !topk_w) return MR_EINVAL;
    if (p->T == 0) return MR_OK;
    const RouteArgs a = route_args(p, logits, probs, routing_map, intermediate, topk_idx, topk_w, status);
    const int nv = fwd_nv_index(p->E, MR_MAX_EXPERTS);
    if (nv < 0) return MR_EUNSUPPORTED;
    return from_cuda(launch_fwd(p->score_fn, p->in_dtype, a, nv, use_select(a.k_r),
                                reinterpret_cast<cudaStream_t>(stream)));
}

int moe_aux_scores_fwd(int T, int E, int topk, int score_fn, int in_dtype, const void* logits, float* scores,
                       uint8_t* routing_map, mr_stream_t stream)
{
    mr_router_params p;
    std::memset(&p, 0, sizeof p);
    p.T = T;
    p.E = E;
    p.topk = topk;
    p.score_fn = score_fn;
    p.in_dtype = in_dtype;
    p.scaling = 1.0f;
    int rc = check_router(&p);
    if (rc != MR_OK) return rc;
    if (!logits || (!scores && !routing_map)) return MR_EINVAL;
    if (T == 0) return MR_OK;
    const RouteArgs a = route_args(&p, logits, nullptr, routing_map, scores, nullptr, nullptr, nullptr);
    const int nv = fwd_nv_index(E, MR_MAX_EXPERTS);
    if (nv < 0) return MR_EUNSUPPORTED;
    return from_cuda(launch_fwd(score_fn, in_dtype, a, nv, use_select(a.k_r), reinterpret_cast<cudaStream_t>(stream)));
}

int moe_router_bwd(const mr_router_params* p, const float* grad_probs, const float* intermediate,
                   const uint8_t* routing_map, float* grad_logits, mr_stream_t stream)
{
    if (!p || !grad_probs || !intermediate || !routing_map || !grad_logits) return MR_EINVAL;
    if (p->T < 0 || p->E < 1) return MR_EINVAL;
    if (p->score_fn != MR_SOFTMAX && p->score_fn != MR_SIGMOID) return MR_EINVAL;
    if (static_cast<long long>(p->T) * p->E > INT_MAX) return MR_EINVAL;
    if (p->E > MR_MAX_EXPERTS) return MR_EUNSUPPORTED;
    if (p->T == 0) return MR_OK;
    const int nv = nv_index(p->E);
    const bool vec = p->E % 4 == 0 && aligned(grad_probs, 16) && aligned(intermediate, 16) &&
                     aligned(grad_logits, 16) && aligned(routing_map, 4);
    return from_cuda(launch_bwd(p->score_fn, nv, grad_probs, intermediate, routing_map, grad_logits, p->T, p->E,
                                p->renorm ? 1 : 0, p->scaling, vec, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_router_bwd_dtype(const mr_router_params* p, int grad_dtype, const void* grad_probs,
                         const float* intermediate, const uint8_t* routing_map, void* grad_logits, mr_stream_t stream)
{
    if (grad_dtype == MR_F32)
        return moe_router_bwd(p, static_cast<const float*>(grad_probs), intermediate, routing_map,
                              static_cast<float*>(grad_logits), stream);
    if (grad_dtype != MR_BF16) return MR_EINVAL;
    if (!p || !grad_probs || !intermediate || !routing_map || !grad_logits) return MR_EINVAL;
    if (p->T < 0 || p->E < 1) return MR_EINVAL;
    if (p->score_fn != MR_SOFTMAX && p->score_fn != MR_SIGMOID) return MR_EINVAL;
    if (static_cast<long long>(p->T) * p->E > INT_MAX) return MR_EINVAL;
    if (p->E > MR_MAX_EXPERTS) return MR_EUNSUPPORTED;
    if (p->T == 0) return MR_OK;
    const int nv = nv_index(p->E);
    const bool vec = p->E % 4 == 0 && aligned(grad_probs, 8) && aligned(intermediate, 16) &&
                     aligned(grad_logits, 8) && aligned(routing_map, 4);
    return from_cuda(launch_bwd_bf16(p->score_fn, nv, static_cast<const __nv_bfloat16*>(grad_probs), intermediate,
                                     routing_map, static_cast<__nv_bfloat16*>(grad_logits), p->T, p->E,
                                     p->renorm ? 1 : 0, p->scaling, vec, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_aux_scores_bwd(int T, int E, int score_fn, const float* grad_scores, const float* scores,
                       float* grad_logits, mr_stream_t stream)
{
    if (!grad_scores || !scores || !grad_logits) return MR_EINVAL;
    if (T < 0 || E < 1) return MR_EINVAL;
    if (score_fn != MR_SOFTMAX && score_fn != MR_SIGMOID) return MR_EINVAL;
    if (static_cast<long long>(T) * E > INT_MAX) return MR_EINVAL;
    if (E > MR_MAX_EXPERTS) return MR_EUNSUPPORTED;
    if (T == 0) return MR_OK;
    const int nv = nv_index(E);
    const bool vec = E % 4 == 0 && aligned(grad_scores, 16) && aligned(scores, 16) && aligned(grad_logits, 16);
    return from_cuda(launch_bwd(score_fn, nv, grad_scores, scores, nullptr, grad_logits, T, E, 0, 1.0f, vec,
                                reinterpret_cast<cudaStream_t>(stream)));
}

static int check_aux_loss(int T, int E, int topk, long long total_num_tokens)
{
    if (T < 0 || E < 1 || topk < 1 || total_num_tokens < 1) return MR_EINVAL;
    if (static_cast<long long>(T) * E > INT_MAX) return MR_EINVAL;
    return MR_OK;
}

static double aux_loss_factor(int E, int topk, float coeff, long long total_num_tokens)
{
    const double N = static_cast<double>(total_num_tokens);
    return static_cast<double>(coeff) * static_cast<double>(E) / (static_cast<double>(topk) * N * N);
}

int moe_tokens_per_expert(int T, int E, const uint8_t* routing_map, int32_t* tokens_per_expert,
                          mr_stream_t stream)
{
    if (T < 0 || E < 1 || !tokens_per_expert || (T > 0 && !routing_map)) return MR_EINVAL;
    if (static_cast<long long>(T) * E > INT_MAX) return MR_EINVAL;
    return from_cuda(launch_tokens_per_expert(routing_map, T, E, tokens_per_expert,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_aux_loss_workspace_bytes(int T, int E)
{
    if (T < 0 || E < 1 || static_cast<long long>(T) * E > INT_MAX) return 0;
    return aux_workspace_bytes(T, E);
}

int moe_aux_loss_fwd(int T, int E, int topk, float coeff, long long total_num_tokens, const float* probs,
                     const int32_t* tokens_per_expert, float* loss, void* workspace, size_t ws_bytes,
                     mr_stream_t stream)
{
    const int c = check_aux_loss(T, E, topk, total_num_tokens);
    if (c != MR_OK) return c;
    if (!tokens_per_expert || !loss || (T > 0 && (!probs || !workspace))) return MR_EINVAL;
    if (ws_bytes < moe_aux_loss_workspace_bytes(T, E)) return MR_EINVAL;
    if (T > 0 && !aligned(workspace, 16)) return MR_EINVAL;
    return from_cuda(launch_aux_loss_fwd(probs, tokens_per_expert, T, E,
                                         aux_loss_factor(E, topk, coeff, total_num_tokens), loss, workspace,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

int moe_aux_loss_bwd(int T, int E, int topk, float coeff, long long total_num_tokens,
                     const int32_t* tokens_per_expert, const float* grad_loss, float* grad_probs,
                     mr_stream_t stream)
{
    const int c = check_aux_loss(T, E, topk, total_num_tokens);
    if (c != MR_OK) return c;
    if (!tokens_per_expert || !grad_loss || (T > 0 && !grad_probs)) return MR_EINVAL;
    return from_cuda(launch_aux_loss_bwd(tokens_per_expert, grad_loss, T, E,
                                         aux_loss_factor(E, topk, coeff, total_num_tokens), grad_probs,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_sort_capacity(int T, int topk, int E_tot, int block_m)
{
    if (T < 0 || topk < 1 || E_tot < 1 || block_m < 1) return 0;
    const size_t N = static_cast<size_t>(T) * static_cast<size_t>(topk);
    const size_t nonempty = N < static_cast<size_t>(E_tot) ? N : static_cast<size_t>(E_tot);
    return N + nonempty * static_cast<size_t>(block_m - 1);
}

size_t moe_sort_workspace_bytes(int T, int topk, int E_tot, int block_m)
{
    if (check_sort(T, topk, E_tot, block_m) != MR_OK) return 0;
    return sort_ws_bytes(static_cast<long long>(T) * topk, E_tot);
}

int moe_sort(const int32_t* topk_idx, const float* topk_w, int T, int topk, int E_tot, int block_m,
             int32_t* sorted_token_ids, float* sorted_weights, int32_t* expert_ids, int32_t* num_tokens_post_pad,
             void* workspace, size_t ws_bytes, int32_t* status, mr_stream_t stream)
{
    int rc = check_sort(T, topk, E_tot, block_m);
    if (rc != MR_OK) return rc;
    if (!sorted_token_ids || !expert_ids || !num_tokens_post_pad) return MR_EINVAL;
    if (T > 0 && !topk_idx) return MR_EINVAL;
    const long long N = static_cast<long long>(T) * topk;
    const size_t need = sort_ws_bytes(N, E_tot);
    if (need > 0 && (!workspace || ws_bytes < need || !aligned(workspace, 4))) return MR_EINVAL;
    return from_cuda(launch_sort(topk_idx, topk_w, static_cast<int>(N), E_tot, block_m, sorted_token_ids,
                                 sorted_weights, expert_ids, num_tokens_post_pad, static_cast<uint32_t*>(workspace),
                                 status, reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_sort_noalloc_scratch_bytes(void) { return sizeof(g_sort_scratch); }

int moe_sort_noalloc(const int32_t* topk_idx, const float* topk_w, int T, int topk, int E_tot, int block_m,
                     int32_t* sorted_token_ids, float* sorted_weights, int32_t* expert_ids,
                     int32_t* num_tokens_post_pad, int32_t* status, mr_stream_t stream)
{
    int rc = check_sort(T, topk, E_tot, block_m);
    if (rc != MR_OK) return rc;
    if (!sorted_token_ids || !expert_ids || !num_tokens_post_pad) return MR_EINVAL;
    if (T > 0 && !topk_idx) return MR_EINVAL;
    const long long N = static_cast<long long>(T) * topk;
    if (sort_ws_bytes(N, E_tot) > MR_SORT_NOALLOC_SCRATCH_BYTES) return MR_EUNSUPPORTED;
    // The count table is fully rewritten by every call, so nothing in the
    // scratch has to start at zero.
    void* scratch = sort_scratch_address();
    if (!scratch) return MR_ECUDA;
    return from_cuda(launch_sort(topk_idx, topk_w, static_cast<int>(N), E_tot, block_m, sorted_token_ids,
                                 sorted_weights, expert_ids, num_tokens_post_pad, static_cast<uint32_t*>(scratch),
                                 status, reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_router_fused_workspace_bytes(const mr_router_params* p, int block_m)
{
    if (check_router(p) != MR_OK || block_m < 1) return 0;
    if (check_sort(p->T, p->topk, p->E + p->n_shared, block_m) != MR_OK) return 0;
    const int nv = fwd_nv_index(p->E, MR_MAX_EXPERTS);
    if (nv < 0) return 0;
    if (fused_one_launch(p->T, kNvBuckets[nv])) return 0;
    const size_t N = static_cast<size_t>(p->T) * p->topk;
    return align_up(N * 4, 256) * 2 + sort_ws_bytes(static_cast<long long>(N), p->E + p->n_shared);
}

int moe_router_fused_fwd_sort(const mr_router_params* p, const void* logits, int block_m, int32_t* topk_idx,
                              float* topk_w, int32_t* sorted_token_ids, float* sorted_weights, int32_t* expert_ids,
                              int32_t* num_tokens_post_pad, void* workspace, size_t ws_bytes, int32_t* status,
                              mr_stream_t stream)
{
    int rc = check_router(p);
    if (rc != MR_OK) return rc;
    const int E_tot = p->E + p->n_shared;
    rc = check_sort(p->T, p->topk, E_tot, block_m);
    if (rc != MR_OK) return rc;
    if (!logits || !sorted_token_ids || !expert_ids || !num_tokens_post_pad) return MR_EINVAL;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int nv = fwd_nv_index(p->E, MR_MAX_EXPERTS);
    if (nv < 0) return MR_EUNSUPPORTED;
    const int k_r = p->topk - p->n_shared;
    // above 16 tokens, rows held in registers: one launch of one thread-block
    // cluster when one fits (else the one-CTA kernel up to 64 tokens, or the
    // separate launches)
    // a warp routes one token in either one-launch form, so the arg-max path
    // (the shorter chain of dependent steps for one row) is the default up to
    // k_r = 32
    const int force = g_path.forced();
    const bool decode_select = force == 2 || (force == 0 && k_r > 32);
    // at most 32 pairs: a warp per token, one warp sorts (16 warps at most)
    if (p->T >= 1 && p->T <= 16 && p->T * p->topk <= kFusedTinyPairs && kNvBuckets[nv] <= kRegisterMaxNv) {
        RouteArgs a = route_args(p, logits, nullptr, nullptr, nullptr, topk_idx, topk_w, status);
        SortArgs s{sorted_token_ids, sorted_weights, expert_ids, num_tokens_post_pad, E_tot, block_m,
                   log2_if_pow2(block_m)};
        return from_cuda(launch_fused_tiny(p->score_fn, p->in_dtype, a, s, nv, decode_select, st));
    }
    // at most 128 pairs and 16 tokens: a warp per token, one warp ranks and scans
    if (p->T >= 1 && p->T <= 16 && p->T * p->topk <= kFusedSmallPairs && kNvBuckets[nv] <= kRegisterMaxNv) {
        RouteArgs a = route_args(p, logits, nullptr, nullptr, nullptr, topk_idx, topk_w, status);
        SortArgs s{sorted_token_ids, sorted_weights, expert_ids, num_tokens_post_pad, E_tot, block_m,
                   log2_if_pow2(block_m)};
        const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, decode_select, a.n_group > 0);
        const size_t smem = static_cast<size_t>(L.bytes) * p->T + small_sort_layout(E_tot).bytes;
        int dev = 0, maxsm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return MR_ECUDA;
        if (smem <= static_cast<size_t>(maxsm))
            return from_cuda(launch_fused_small(p->score_fn, p->in_dtype, a, s, nv, decode_select, st));
    }
    if (p->T > 16 && p->T <= kFusedClusterMaxTokens && kNvBuckets[nv] <= kRegisterMaxNv) {
        RouteArgs a = route_args(p, logits, nullptr, nullptr, nullptr, topk_idx, topk_w, status);
        SortArgs s{sorted_token_ids, sorted_weights, expert_ids, num_tokens_post_pad, E_tot, block_m,
                   log2_if_pow2(block_m)};
        const int e = launch_fused_cluster(p->score_fn, p->in_dtype, a, s, nv, decode_select, st);
        if (e != cudaErrorNotSupported) return from_cuda(e);
        cudaGetLastError();
    }
    if (fused_one_launch(p->T, kNvBuckets[nv])) {
        RouteArgs a = route_args(p, logits, nullptr, nullptr, nullptr, topk_idx, topk_w, status);
        SortArgs s{sorted_token_ids, sorted_weights, expert_ids, num_tokens_post_pad, E_tot, block_m,
                   log2_if_pow2(block_m)};
        const bool sel = decode_select;
        a.warm_code = launch_overlap() ? 1 : 0;
        const int nw = (p->T > 16 ? kFusedWideThreads : kFusedThreads) / 32;
        const WarpLayout L = warp_layout(a.k_r, a.stop, a.E, sel, a.n_group > 0);
        const size_t smem = static_cast<size_t>(L.bytes) * nw +
                            fused_sort_layout(p->T * p->topk, E_tot, block_m, p->T > 16 ? 8 : 4).bytes;
        int dev = 0, maxsm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return MR_ECUDA;
        if (smem > static_cast<size_t>(maxsm)) return MR_EUNSUPPORTED;
        return from_cuda(launch_fused_decode(p->score_fn, p->in_dtype, a, s, nv, sel, st));
    }
    const size_t N = static_cast<size_t>(p->T) * p->topk;
    if (!workspace || ws_bytes < moe_router_fused_workspace_bytes(p, block_m)) return MR_EINVAL;
    unsigned char* w = static_cast<unsigned char*>(workspace);
    if (!aligned(w, 4)) return MR_EINVAL;
    int32_t* idx = topk_idx ? topk_idx : reinterpret_cast<int32_t*>(w);
    float* wt = topk_w ? topk_w : reinterpret_cast<float*>(w + align_up(N * 4, 256));
    uint32_t* sws = reinterpret_cast<uint32_t*>(w + align_up(N * 4, 256) * 2);
    const RouteArgs a = route_args(p, logits, nullptr, nullptr, nullptr, idx, wt, status);
    int e = launch_fwd(p->score_fn, p->in_dtype, a, nv, use_select(k_r), st);
    if (e != cudaSuccess) return MR_ECUDA;
    return from_cuda(launch_sort(idx, wt, static_cast<int>(N), E_tot, block_m, sorted_token_ids, sorted_weights,
                                 expert_ids, num_tokens_post_pad, sws, status, st));
}

int moe_router_expf(const float* x, float* y, int n, mr_stream_t stream)
{
    if (n < 0 || (n > 0 && (!x || !y))) return MR_EINVAL;
    if (n == 0) return MR_OK;
    return from_cuda(launch_expf(x, y, n, reinterpret_cast<cudaStream_t>(stream)));
}

int moe_router_exp_value(const float* x, float* y, int n, mr_stream_t stream)
{
    if (n < 0 || (n > 0 && (!x || !y))) return MR_EINVAL;
    if (n == 0) return MR_OK;
    const long long blocks = (static_cast<long long>(n) + 255) / 256;
    const int grid = static_cast<int>(blocks < 4096 ? blocks : 4096);
    return from_cuda(launch_kernel(k_exp_value, dim3(grid), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream), 0,
                                   x, y, n));
}

int moe_router_noop(mr_stream_t stream) { return from_cuda(launch_noop(reinterpret_cast<cudaStream_t>(stream))); }

int moe_router_device_status(int32_t* out, int clear, mr_stream_t stream)
{
    if (!out) return MR_EINVAL;
    int32_t* word = device_status_address();
    if (!word) return MR_ECUDA;
    return from_cuda(launch_kernel(k_take_status, dim3(1), dim3(1), 0, reinterpret_cast<cudaStream_t>(stream), 0, word,
                                   out, clear));
}

}  // extern "C"
