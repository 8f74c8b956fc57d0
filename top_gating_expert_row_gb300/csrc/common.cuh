// Device helpers shared by the routing kernels: the written fp32 exponential,
// order-preserving selection keys, warp reductions and row loads/stores.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace mr {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kSoftmax = 0;
constexpr int kSigmoid = 1;

// ---------------------------------------------------------------------------
// fp32 exponential, reproducible bit for bit on any IEEE-754 machine.
//
// Cody & Waite argument reduction ("Software Manual for the Elementary
// Functions", 1980) and the degree-7 Taylor polynomial of exp about 0:
//   n = rint(x * log2 e);  r = (x - n*ln2_hi) - n*ln2_lo;  p = sum_{i<=7} r^i/i!
//   exp(x) = (p * 2^(n/2)) * 2^(n - n/2)      (n/2 truncates toward zero)
// ln2_hi is ln 2 cut to 16 fraction bits, so n*ln2_hi is exact; every step is a
// single correctly rounded fp32 operation written with an explicit _rn
// intrinsic, so the compiler cannot contract or reorder it. Error: < 1 ulp
// (the Taylor remainder r^8/8! is under 0.1 ulp for |r| <= ln2/2).
// Specification at the ends: x >= 89 -> +inf, x <= -104 -> +0, NaN -> NaN.
// Clamping x to [-104, 89] first reproduces those ends exactly (the formula
// overflows to +inf from 88.73 up and rounds to +0 at -104), so exp_spec is
// the specification for every non-NaN x without a branch.
// ---------------------------------------------------------------------------
constexpr double kLn2 = 0.693147180559945309417232121458176568;
constexpr float kLog2e = static_cast<float>(1.0 / kLn2);
constexpr float kLn2Hi = static_cast<float>(static_cast<double>(static_cast<long long>(kLn2 * 65536.0)) / 65536.0);
constexpr float kLn2Lo = static_cast<float>(kLn2 - static_cast<double>(kLn2Hi));

__device__ __forceinline__ float pow2_normal(int k)  // 2^k, -126 <= k <= 127
{
    return __int_as_float((k + 127) << 23);
}

// p(r) ~ exp(r) for |r| <= ln2/2, Horner form of the degree-7 Taylor polynomial.
__device__ __forceinline__ float exp_poly(float r)
{
    float p = static_cast<float>(1.0 / 5040.0);
    p = __fmaf_rn(p, r, static_cast<float>(1.0 / 720.0));
    p = __fmaf_rn(p, r, static_cast<float>(1.0 / 120.0));
    p = __fmaf_rn(p, r, static_cast<float>(1.0 / 24.0));
    p = __fmaf_rn(p, r, static_cast<float>(1.0 / 6.0));
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmaf_rn(p, r, 1.0f);
}

__device__ __forceinline__ float exp_spec(float x)
{
    x = fminf(fmaxf(x, -104.0f), 89.0f);
    const float nf = rintf(__fmul_rn(x, kLog2e));
    const int n = __float2int_rn(nf);
    float r = __fmaf_rn(-nf, kLn2Hi, x);
    r = __fmaf_rn(-nf, kLn2Lo, r);
    const float p = exp_poly(r);
    const int n1 = n / 2;
    const int n2 = n - n1;
    return __fmul_rn(__fmul_rn(p, pow2_normal(n1)), pow2_normal(n2));
}

// The specification including NaN (used by the diagnostic entry point).
__device__ __forceinline__ float exp_f32(float x) { return (x != x) ? x : exp_spec(x); }

// exp_spec on two values, bit-identical to two exp_spec calls: the reduction
// and the scaling per value as in exp_spec, the degree-7 polynomial (8 of the
// ~24 operations) on both values at once as packed fp32x2 fused multiply-adds,
// each lane rounding as __fmaf_rn. (An all-packed form, with the rounding of
// x*log2 e and the exponent split in packed and integer operations, was
// computed wrong in one lane by this toolchain; the device exp diagnostic
// checks this form against exp_spec on every input it evaluates.)
__device__ __forceinline__ float2 exp_spec2(float2 x)
{
    const float ax = fminf(fmaxf(x.x, -104.0f), 89.0f);
    const float ay = fminf(fmaxf(x.y, -104.0f), 89.0f);
    const float nfx = rintf(__fmul_rn(ax, kLog2e));
    const float nfy = rintf(__fmul_rn(ay, kLog2e));
    const float2 r = make_float2(__fmaf_rn(-nfx, kLn2Lo, __fmaf_rn(-nfx, kLn2Hi, ax)),
                                 __fmaf_rn(-nfy, kLn2Lo, __fmaf_rn(-nfy, kLn2Hi, ay)));
    float2 p = make_float2(static_cast<float>(1.0 / 5040.0), static_cast<float>(1.0 / 5040.0));
    p = __ffma2_rn(p, r, make_float2(static_cast<float>(1.0 / 720.0), static_cast<float>(1.0 / 720.0)));
    p = __ffma2_rn(p, r, make_float2(static_cast<float>(1.0 / 120.0), static_cast<float>(1.0 / 120.0)));
    p = __ffma2_rn(p, r, make_float2(static_cast<float>(1.0 / 24.0), static_cast<float>(1.0 / 24.0)));
    p = __ffma2_rn(p, r, make_float2(static_cast<float>(1.0 / 6.0), static_cast<float>(1.0 / 6.0)));
    p = __ffma2_rn(p, r, make_float2(0.5f, 0.5f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    p = __ffma2_rn(p, r, make_float2(1.0f, 1.0f));
    const int nx = __float2int_rn(nfx), ny = __float2int_rn(nfy);
    const int hx = nx / 2, hy = ny / 2;
    return make_float2(__fmul_rn(__fmul_rn(p.x, pow2_normal(hx)), pow2_normal(nx - hx)),
                       __fmul_rn(__fmul_rn(p.y, pow2_normal(hy)), pow2_normal(ny - hy)));
}

constexpr float kLog2eHi = kLog2e;
constexpr float kLog2eLo = static_cast<float>(1.0 / kLn2 - static_cast<double>(kLog2e));

__device__ __forceinline__ float exp2_hw(float f)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(f));
    return y;
}

// exp(x) for x <= 0 where only the value matters (softmax numerators), in
// three instructions: the hardware base-2 exponential of x log2 e, formed as
// fma(x, L2E_HI, x * L2E_LO) from a two-part log2 e with one rounding. Its
// relative error is that rounding (at most |x log2 e| * 2^-24, ln 2 times that
// in the result) plus the hardware exponential's; results below 2^-126 flush
// to zero. Not the specification exp_spec: these values decide no selection
// (softmax selects on the logits), they are compared within a tolerance.
__device__ __forceinline__ float exp_value(float x)
{
    return exp2_hw(__fmaf_rn(x, kLog2eHi, __fmul_rn(x, kLog2eLo)));
}

// exp_value on two values at once: the same operations, with the floating-point
// ones issued as packed fp32x2 instructions (each lane of a packed op rounds
// exactly as the scalar op), so each result is bit-identical to exp_value's.
__device__ __forceinline__ float2 exp_value2(float2 x)
{
    const float2 y = __ffma2_rn(x, make_float2(kLog2eHi, kLog2eHi),
                                __fmul2_rn(x, make_float2(kLog2eLo, kLog2eLo)));
    return make_float2(exp2_hw(y.x), exp2_hw(y.y));
}

// Logistic function 1 / (1 + exp(-x)), IEEE add and correctly rounded
// reciprocal (the same number as an IEEE divide of 1 by the sum).
__device__ __forceinline__ float sigmoid_f32(float x)
{
    return __frcp_rn(__fadd_rn(1.0f, exp_spec(-x)));
}

// sigmoid_f32 on two values (bit-identical), through exp_spec2.
__device__ __forceinline__ float2 sigmoid_f32x2(float2 x)
{
    const float2 e = __fadd2_rn(make_float2(1.0f, 1.0f), exp_spec2(make_float2(-x.x, -x.y)));
    return make_float2(__frcp_rn(e.x), __frcp_rn(e.y));
}

// ---------------------------------------------------------------------------
// Selection keys: a strictly increasing map from fp32 to uint32, so that
// "larger key" is an unsigned compare. Adding +0 folds -0 onto +0 (they compare
// equal as floats). Every non-NaN float maps to a key >= 0x007fffff; key 0 is
// reserved for "not a candidate" (padding, experts of dropped groups). NaN
// inputs give unspecified keys.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t key_of(float f)
{
    const uint32_t u = __float_as_uint(__fadd_rn(f, 0.0f));
    return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
}

__device__ __forceinline__ float float_of(uint32_t k)
{
    // top bit set (non-negative float): flip the top bit; else flip all bits
    const uint32_t s = static_cast<uint32_t>(static_cast<int32_t>(k) >> 31);
    return __uint_as_float(k ^ (~s | 0x80000000u));
}

// ---------------------------------------------------------------------------
// Warp reductions (all 32 lanes participate).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// Exclusive prefix sum over lanes.
__device__ __forceinline__ uint32_t warp_exclusive_scan(uint32_t v, int lane)
{
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    return incl - v;
}

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Bulk prefetch of [p, p + bytes) into L2 (one instruction; p 16-byte aligned,
// bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// Bulk global -> shared copies completing on an mbarrier (the TMA engine, 1-D
// form). Addresses 16-byte aligned, sizes a multiple of 16 bytes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic-proxy shared accesses before later
// async-proxy (bulk copy) writes to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arms the barrier for `bytes` and issues the copy. drop != 0 (a test mode)
// arms the barrier without issuing the copy, so its wait runs out while no
// copy is in flight.
__device__ __forceinline__ void bulk_load_row(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              int drop = 0)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
    if (drop) return;
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(dst)),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// One wait attempt of at most about 1 us (the suspend-time hint, in ns).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "r"(1000u)
        : "memory");
    return ok != 0;
}

// Codes a kernel reports in a device status word (the C ABI's MR_ERANGE and
// MR_ETIMEOUT). A word is raised to a code with an atomic maximum, so it holds
// the most severe code reported since it was zeroed.
constexpr int32_t kStatusRange = 4;
constexpr int32_t kStatusTimeout = 5;

__device__ __forceinline__ void report_status(int32_t* word, int32_t code)
{
    if (word) atomicMax(word, code);
}

// Bounded wait for phase `parity` of the barrier: at most `tries` attempts of
// about a microsecond each (the default, 2^20, is about a second); false if it
// gave up.
constexpr uint32_t kWaitLimit = 1u << 20;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t tries = kWaitLimit)
{
    for (uint32_t i = 0; i < tries; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. Every kernel of the library may call
// pdl_trigger on entry (the next kernel in the stream may be launched now and
// run its own entry while this one works) and calls pdl_wait before its first
// access to global memory (it returns once the previous kernel in the stream
// has completed and its writes are visible; at once for a kernel launched
// without the overlap). Since every kernel waits for its predecessor, each also
// completes after all the kernels before it.
// ---------------------------------------------------------------------------
// Under the overlap a kernel runs while its predecessor is still writing, so
// nothing that kernel produced may be read through the non-coherent read-only
// path (ld.global.nc: __ldg, or plain loads through const __restrict__
// pointers, which the compiler may turn into it): that path assumes the data
// stays unchanged for the whole life of the reading kernel, and an SM may keep
// serving stale lines from it after the wait. The kernels therefore take no
// __restrict__ pointers and load with coherent cache operators (__ldcs,
// __ldcg, plain loads), which the wait's memory clobber keeps after it.
//
// Only small grids trigger on entry (pdl_trigger_small): a large grid's
// dependents would be placed wherever its CTAs free slots first, unevenly, so
// a large grid lets its dependents launch when it completes, as in plain
// stream order.
constexpr unsigned kPdlSmallGrid = 32;
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger_small()
{
    if (gridDim.x * gridDim.y * gridDim.z <= kPdlSmallGrid) pdl_trigger();
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Thread-block clusters: rank, barrier and distributed shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank()
{
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}

// Barrier over every thread of the cluster (all threads of all its CTAs must
// reach it, from converged warps); orders the shared-memory accesses made
// before it, including those to other CTAs' shared memory, before those after.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The two halves of cluster_sync: arrive (does not block) and wait (blocks
// until every thread of the cluster has arrived). A CTA that reads another
// CTA's shared memory arrives once its last such read is done and waits before
// it exits, so no CTA leaves while its shared memory may still be read.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Generic pointer to the same variable in the shared memory of the cluster's
// CTA `rank`: plain loads through it reach that CTA's shared memory, and the
// compiler is free to keep several in flight (the cluster barriers, whose asm
// clobbers memory, still order them).
template <typename T>
__device__ __forceinline__ const T* cluster_peer(const T* p, uint32_t rank)
{
    uint64_t r;
    asm("mapa.u64 %0, %1, %2;" : "=l"(r) : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
    return reinterpret_cast<const T*>(r);
}

// ---------------------------------------------------------------------------
// Element access for logits (fp32 or bf16 storage, fp32 compute).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

template <typename InT>
__device__ __forceinline__ float load_scalar(const InT* p);
template <>
__device__ __forceinline__ float load_scalar<float>(const float* p) { return __ldcs(p); }
template <>
__device__ __forceinline__ float load_scalar<__nv_bfloat16>(const __nv_bfloat16* p)
{
    return bf16_bits_to_f32(__ldcs(reinterpret_cast<const unsigned short*>(p)));
}

// Four consecutive elements starting at a 4-element-aligned position.
template <typename InT>
__device__ __forceinline__ void load4(const InT* p, float (&x)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&x)[4])
{
    const float4 q = __ldcs(reinterpret_cast<const float4*>(p));
    x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&x)[4])
{
    const uint2 q = __ldcs(reinterpret_cast<const uint2*>(p));
    x[0] = bf16_bits_to_f32(q.x & 0xffffu); x[1] = bf16_bits_to_f32(q.x >> 16);
    x[2] = bf16_bits_to_f32(q.y & 0xffffu); x[3] = bf16_bits_to_f32(q.y >> 16);
}

// Four consecutive elements, starting at element e0 (a multiple of 4), of a row
// held raw in shared memory at `base`.
template <typename InT>
__device__ __forceinline__ void load4_shared(const unsigned char* base, int e0, float (&x)[4]);
template <>
__device__ __forceinline__ void load4_shared<float>(const unsigned char* base, int e0, float (&x)[4])
{
    const float4 q = *reinterpret_cast<const float4*>(base + static_cast<size_t>(e0) * 4);
    x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
}
template <>
__device__ __forceinline__ void load4_shared<__nv_bfloat16>(const unsigned char* base, int e0, float (&x)[4])
{
    const uint2 q = *reinterpret_cast<const uint2*>(base + static_cast<size_t>(e0) * 2);
    x[0] = bf16_bits_to_f32(q.x & 0xffffu); x[1] = bf16_bits_to_f32(q.x >> 16);
    x[2] = bf16_bits_to_f32(q.y & 0xffffu); x[3] = bf16_bits_to_f32(q.y >> 16);
}

template <typename OutT>
__device__ __forceinline__ void store_scalar(OutT* p, float v);
template <>
__device__ __forceinline__ void store_scalar<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void store_scalar<__nv_bfloat16>(__nv_bfloat16* p, float v)
{
    *p = __float2bfloat16_rn(v);
}

// Four consecutive values with the streaming (evict-first) cache hint.
template <typename OutT>
__device__ __forceinline__ void store4_stream(OutT* p, const float (&v)[4]);
template <>
__device__ __forceinline__ void store4_stream<float>(float* p, const float (&v)[4])
{
    __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
}
template <>
__device__ __forceinline__ void store4_stream<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[4])
{
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 q;
    q.x = *reinterpret_cast<const uint32_t*>(&a);
    q.y = *reinterpret_cast<const uint32_t*>(&b);
    __stcs(reinterpret_cast<uint2*>(p), q);
}

template <typename OutT>
__device__ __forceinline__ void store4(OutT* p, const float (&v)[4]);
template <>
__device__ __forceinline__ void store4<float>(float* p, const float (&v)[4])
{
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[4])
{
    const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 q;
    q.x = *reinterpret_cast<const uint32_t*>(&a);
    q.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = q;
}

}  // namespace mr
