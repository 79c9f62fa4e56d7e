// sdv_common.cuh - shared device helpers of the sm_103a verify-pass kernels.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "sdverify.h"

namespace sdv {

// An NVTX range around one library call (host side): a profiler's timeline shows each call, named as
// in the C ABI, over the kernels it enqueues.  Without a profiler attached a push / pop costs a
// test of a function pointer.
struct NvtxScope {
    explicit NvtxScope(const char *name) { nvtxRangePushA(name); }
    ~NvtxScope() { nvtxRangePop(); }
    NvtxScope(const NvtxScope &) = delete;
    NvtxScope &operator=(const NvtxScope &) = delete;
};
#define SD_NVTX(name) ::sdv::NvtxScope sd_nvtx_scope_(name)

// ---------------------------------------------------------------------------
// host-side plumbing
// ---------------------------------------------------------------------------

// Device address of this device's status word (a __device__ int in sdv_abi.cu),
// looked up once per device.  nullptr if the lookup failed.
int *status_ptr();
// SM count of the current device (cached per device).
int num_sms();
// Whether launches carry the programmatic-stream-serialisation attribute.
bool pdl_enabled();
// sd_qmatmul_multipos restricted by a previous launch on the stream: only the row tiles set in
// unit_mask (bit per 32-row tile; null: all) are computed, and nothing at all if *skip_if != 0
// (null: always).  af_pre / af_meta_pre (nullable): the activation fragments and records of q / scales
// in this format's layout, formed by an earlier launch (else the call forms them).  Outputs of a
// computed tile equal the unrestricted call's bit for bit.
sd_status qmatmul_restricted(int qtype, const void *w, int64_t n_out, int64_t k_in, const int8_t *q,
                             const float *scales, int32_t M, float *y, const float *residual, uint32_t epilogue,
                             int64_t requant_col0, int8_t *q_next, float *scales_next, void *workspace,
                             size_t ws_bytes, const uint32_t *unit_mask, const int *skip_if, const uint8_t *af_pre,
                             const float *af_meta_pre, sd_stream_t stream);
// Raise a kernel's dynamic shared-memory limit to everything the device lets one block have, once
// per (kernel, device).  The limit is a property of the function, not of a launch: set per call to
// that call's size, it would be lowered by a smaller call after a larger one had been captured into
// a graph, and any later re-launch of the larger node with the function's current limit would fail.
cudaError_t allow_max_dynamic_smem(const void *kernel);
template <typename... KArgs>
cudaError_t allow_max_dynamic_smem(void (*kernel)(KArgs...)) {
    return allow_max_dynamic_smem(reinterpret_cast<const void *>(kernel));
}

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Launch with programmatic dependent launch (when enabled): the kernel may
// begin before the previous kernel on the stream finishes; it must execute
// griddepcontrol.wait before touching anything that kernel produced.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                   Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t gtimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: gives up after `limit_ns` nanoseconds of polling, or as soon
// as *abort becomes non-zero.  Returns false when it gave up (the caller then
// records SD_ETIMEOUT and unwinds).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                                  const volatile int *abort = nullptr) {
    // the global timer is read only once a wait has lasted 64 polls (then every 64): short waits, the
    // common case, never pay for the read; the bound counts from the first read
    uint64_t t0 = 0;
    for (uint32_t k = 1;; ++k) {
        if (mbar_try_wait(bar, parity)) return true;
        if (abort && *abort) return false;
        if ((k & 63u) == 0) {
            const uint64_t now = gtimer_ns();
            if (k == 64) t0 = now;
            else if (now - t0 > limit_ns) return false;
        }
    }
}

// 1-D bulk copy global -> shared through the TMA engine, completing on `bar`.
// dst, src 16-byte aligned, bytes % 16 == 0.  L2 hint: evict-first (weights are
// read exactly once per pass).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 1-D bulk copy global -> shared without a cache hint (data many CTAs read: left in L2).
__device__ __forceinline__ void bulk_g2s_l2keep(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// Orders this thread's generic-proxy accesses against later async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Named barrier over `nthreads` threads.  The non-.aligned form: callers may reach it from
// code where a warp's lanes are not converged (after per-lane spin loops or lane-0 branches).
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    __syncwarp();
    asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads: every thread gets
// the same answer at the same point, so decisions taken on it stay uniform without a shared
// flag that one thread might rewrite before a slower one has read it.
__device__ __forceinline__ bool bar_any(int id, int nthreads, bool v) {
    __syncwarp();
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbarrier.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void set_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// Bounds checks of the debug build (compiled with SD_DEBUG_BOUNDS): a failed check records
// SD_EDEVICE with the site's number (>= 100) in the status word's second entry, and the caller skips
// the access.  The release build compiles every check to `true`, so the condition is never evaluated.
__device__ __forceinline__ bool bounds_check(bool ok, int *status, int site) {
    if (!ok && status && atomicCAS(status, 0, SD_EDEVICE) == 0) status[1] = site;
    return ok;
}
#ifdef SD_DEBUG_BOUNDS
#define SD_INB(cond, status, site) (::sdv::bounds_check((cond), (status), (site)))
#else
#define SD_INB(cond, status, site) (true)
#endif

__device__ __forceinline__ int dp4a(int a, int b, int c) { return __dp4a(a, b, c); }

// Packed fp32 pairs (two IEEE operations per instruction, each rounded as its scalar form)
__device__ __forceinline__ unsigned long long f2_bits(float2 v) { return *reinterpret_cast<unsigned long long *>(&v); }
__device__ __forceinline__ float2 bits_f2(unsigned long long v) { return *reinterpret_cast<float2 *>(&v); }
__device__ __forceinline__ float2 ffma2_rn(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
    return bits_f2(d);
}
__device__ __forceinline__ float2 fadd2_rn(float2 a, float2 b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return bits_f2(d);
}
__device__ __forceinline__ float2 fmul2_rn(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return bits_f2(d);
}

// ---------------------------------------------------------------------------
// Canonical arithmetic shared by every kernel whose float results decide an
// integer.  Compiled without FMA contraction; fused operations are explicit.
// ---------------------------------------------------------------------------

// exp(x) by Cody & Waite reduction (k = rint(x log2 e); r = x - k ln2 with ln2
// as a 16-bit head and a tail, each applied by one fused multiply-add), e^r by
// its degree-7 Taylor series in Horner form with fused multiply-adds, and 2^k
// applied as two exact powers of two so a subnormal result rounds once.
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

__device__ __forceinline__ float cexpf_canon(float x) {
    if (x != x) return x;
    if (x > 100.0f) return __int_as_float(0x7f800000);
    if (x < -104.0f) return 0.0f;
    const float log2e = 1.44269504088896340736f;
    const float ln2_hi = 0.693145751953125f;
    const float ln2_lo = 1.42860682030941723212e-6f;
    float k = rintf(__fmul_rn(x, log2e));
    float r = __fmaf_rn(-k, ln2_hi, x);
    r = __fmaf_rn(-k, ln2_lo, r);
    float p = 1.0f / 5040.0f;
    p = __fmaf_rn(p, r, 1.0f / 720.0f);
    p = __fmaf_rn(p, r, 1.0f / 120.0f);
    p = __fmaf_rn(p, r, 1.0f / 24.0f);
    p = __fmaf_rn(p, r, 1.0f / 6.0f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    int ki = static_cast<int>(k);
    int k1 = ki / 2, k2 = ki - k1;
    return __fmul_rn(__fmul_rn(p, pow2i(k1)), pow2i(k2));
}

// per-32 requantisation of one value held by each lane of a full warp:
// d = amax/127, q = round-half-away(y/d) clamped to +-127, 0 when d == 0.
__device__ __forceinline__ int requant_lane(float y, float &d_out) {
    float a = fabsf(y);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    float d = __fdiv_rn(a, 127.0f);
    d_out = d;
    int v = 0;
    if (d != 0.0f) {
        v = static_cast<int>(roundf(__fdiv_rn(y, d)));
        v = v > 127 ? 127 : (v < -127 ? -127 : v);
    }
    return v;
}

// SiLU gate of the FFN: silu(g) * u with silu(g) = g / (1 + exp(-g)).
__device__ __forceinline__ float silu_mul(float g, float u) {
    float s = __fdiv_rn(g, __fadd_rn(1.0f, cexpf_canon(-g)));
    return __fmul_rn(s, u);
}

// Pairwise tree over 1024 slots held by one warp, slot e = lane + 32*r in v[r]:
// the sum at strides 512, 256, ..., 1 (v[j] += v[j+s] for j < s).  Lane 0 returns it.
__device__ __forceinline__ float tree1024_warp(float (&v)[32]) {
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1)
#pragma unroll
        for (int r = 0; r < h; ++r) v[r] = __fadd_rn(v[r], v[r + h]);
    float x = v[0];
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        float o = __shfl_down_sync(0xffffffffu, x, s);
        if ((threadIdx.x & 31) < s) x = __fadd_rn(x, o);
    }
    return x;
}

// Philox4x32-10 (Salmon et al., SC'11): counter c, key (k0, k1).
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
        uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

}  // namespace sdv
