// sdv_norm.cu - RMSNorm fused with per-32 int8 requantisation, and the small
// test hooks (canonical exp, SiLU*mul requant, Philox, bounded-wait timeout).
#include "sdv_qmatmul.cuh"

namespace sdv {

// One CTA of 1024 threads per row.  Sum of squares: per 32-element block a
// pairwise tree over the block's squares (strides 16..1), then a pairwise tree
// over the block sums zero-padded to a power of two (at least 256 slots);
// inv = 1/sqrt(s/K + eps) correctly rounded.  Each warp requantises 32-element
// blocks of t = x*w and scales them by inv: the requantisation of y = x*inv*w.  The matmul epilogues form the same block sums
// where they finish a block of the residual stream, so the verify pass reaches
// identical bits.
constexpr int NORM_WARPS = 32;

__global__ void __launch_bounds__(NORM_WARPS * 32) rmsnorm_quant_kernel(const float *__restrict__ x, int64_t ldx,
                                                            const float *__restrict__ w, float eps, int64_t K,
                                                            int8_t *__restrict__ q, float *__restrict__ sc) {
    __shared__ float slots[NORM_MAX_KB];
    __shared__ float s_inv;
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = blockIdx.x;
    const float *xr = x + static_cast<int64_t>(m) * ldx;
    const int KB = static_cast<int>(K / 32);
    constexpr int UNR = 8;  // blocks a warp loads together: their loads are in flight at once
    float inv = 1.0f;
    if (w) {
        int P = 256;
        while (P < KB) P <<= 1;
        for (int b0 = warp; b0 < P; b0 += NORM_WARPS * UNR) {
            float v[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int b = b0 + NORM_WARPS * u;
                v[u] = b < KB ? xr[static_cast<int64_t>(b) * 32 + lane] : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                const int b = b0 + NORM_WARPS * u;
                if (b >= P) break;
                float t = 0.0f;
                if (b < KB) {
                    t = __fmul_rn(v[u], v[u]);
#pragma unroll
                    for (int s = 16; s >= 1; s >>= 1) {
                        const float o = __shfl_down_sync(0xffffffffu, t, s);
                        if (lane < s) t = __fadd_rn(t, o);
                    }
                }
                if (lane == 0) slots[b] = t;
            }
        }
        __syncthreads();
        for (int st = P / 2; st >= 1; st >>= 1) {
            for (int j = tid; j < st; j += NORM_WARPS * 32) slots[j] = __fadd_rn(slots[j], slots[j + st]);
            __syncthreads();
        }
        if (tid == 0) {
            const float mean = __fdiv_rn(slots[0], static_cast<float>(K));
            s_inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
        }
        __syncthreads();
        inv = s_inv;
    }
    // codes from t = x * w (the row factor inv cancels in t / (max|t| / 127)); scale inv * max|t| / 127
    for (int64_t b0 = warp; b0 < KB; b0 += NORM_WARPS * UNR) {
        float t[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int64_t b = b0 + NORM_WARPS * u;
            t[u] = b < KB ? xr[b * 32 + lane] : 0.0f;
            if (w && b < KB) t[u] = __fmul_rn(t[u], w[b * 32 + lane]);
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int64_t b = b0 + NORM_WARPS * u;
            if (b >= KB) break;
            float c;
            const int v = requant_lane(t[u], c);
            q[static_cast<int64_t>(m) * K + b * 32 + lane] = static_cast<int8_t>(v);
            if (lane == 0) sc[static_cast<int64_t>(m) * KB + b] = w ? __fmul_rn(inv, c) : c;
        }
    }
}

__global__ void cexp_kernel(const float *__restrict__ x, int64_t n, float *__restrict__ y) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        y[i] = cexpf_canon(x[i]);
}

__global__ void silu_requant_kernel(const float *__restrict__ g, const float *__restrict__ u, int64_t F,
                                    int8_t *__restrict__ q, float *__restrict__ sc) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int m = blockIdx.x;
    for (int64_t b = warp; b < F / 32; b += blockDim.x / 32) {
        int64_t i = static_cast<int64_t>(m) * F + b * 32 + lane;
        float h = silu_mul(g[i], u[i]);
        float d;
        int v = requant_lane(h, d);
        q[i] = static_cast<int8_t>(v);
        if (lane == 0) sc[static_cast<int64_t>(m) * (F / 32) + b] = d;
    }
}

__global__ void philox_kernel(uint64_t seed, int64_t pos, int64_t n, uint4 *out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        uint64_t p = static_cast<uint64_t>(pos + i);
        out[i] = philox4x32_10(make_uint4(static_cast<uint32_t>(p), static_cast<uint32_t>(p >> 32), 0u, 0u),
                               static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
    }
}

// Waits on an mbarrier that nothing ever completes, bounded by limit_ns.
__global__ void wait_timeout_kernel(uint64_t limit_ns, int *status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        if (!mbar_wait_bounded(&bar, 0, limit_ns)) set_status(status, SD_ETIMEOUT);
    }
}

}  // namespace sdv

using namespace sdv;

static inline cudaStream_t cs(sd_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }
static inline sd_status launched(cudaError_t e) { return e == cudaSuccess ? SD_OK : SD_ECUDA; }

extern "C" {

sd_status sd_rmsnorm_quant_acts(const float *x, int64_t ldx, const float *norm_w, float eps, int32_t M, int64_t K,
                                int8_t *q, float *scales, sd_stream_t stream) {
    SD_NVTX("sd_rmsnorm_quant_acts");
    if (!x || !q || !scales || M < 1 || M > 65535 || K <= 0 || K % 32 || ldx < K) return SD_EINVAL;
    if (norm_w && K / 32 > NORM_MAX_KB) return SD_EUNSUPPORTED;
    if (!aligned(x, 4) || !aligned(q, 16)) return SD_EINVAL;
    return launched(launch(rmsnorm_quant_kernel, dim3(M), dim3(NORM_WARPS * 32), 0, cs(stream), x, ldx, norm_w, eps, K, q,
                           scales));
}

sd_status sd_debug_cexp(const float *x, int64_t n, float *y, sd_stream_t stream) {
    if (!x || !y || n < 0) return SD_EINVAL;
    if (n == 0) return SD_OK;
    int grid = static_cast<int>(n / 256 + 1 < 4096 ? n / 256 + 1 : 4096);
    cexp_kernel<<<grid, 256, 0, cs(stream)>>>(x, n, y);
    return launched(cudaGetLastError());
}

sd_status sd_debug_silu_mul_requant(const float *g, const float *u, int32_t M, int64_t F, int8_t *q, float *scales,
                                    sd_stream_t stream) {
    if (!g || !u || !q || !scales || M < 1 || M > 65535 || F <= 0 || F % 32) return SD_EINVAL;
    silu_requant_kernel<<<M, 256, 0, cs(stream)>>>(g, u, F, q, scales);
    return launched(cudaGetLastError());
}

sd_status sd_debug_philox(uint64_t seed, int64_t pos, int64_t n, uint32_t *out, sd_stream_t stream) {
    if (!out || n < 0 || !aligned(out, 16)) return SD_EINVAL;
    if (n == 0) return SD_OK;
    int grid = static_cast<int>(n / 256 + 1 < 4096 ? n / 256 + 1 : 4096);
    philox_kernel<<<grid, 256, 0, cs(stream)>>>(seed, pos, n, reinterpret_cast<uint4 *>(out));
    return launched(cudaGetLastError());
}

sd_status sd_debug_wait_timeout(int64_t limit_ns, sd_stream_t stream) {
    if (limit_ns < 1 || limit_ns > 10000000000ll) return SD_EINVAL;
    int *st = status_ptr();
    if (!st) return SD_ECUDA;
    wait_timeout_kernel<<<1, 32, 0, cs(stream)>>>(static_cast<uint64_t>(limit_ns), st);
    return launched(cudaGetLastError());
}

}  // extern "C"
