// Consumer-loop microbenchmark (run by `python bench.py --probe consumer`): 4-bit records pre-staged
// in shared memory, 8 (or 16) consumer warps per SM, one CTA per SM; prints SM cycles per 32x32-weight
// record at M = 5 for the library's own stage_compute (v0) and for alternatives that were measured
// against it: f32x2 scaling and zero-padded activations (v5-v8), one activation fragment reused over
// R units' records (v1, v2, v4), and v0 beside other warps that copy like the producer, poll like the
// finishers, or run from a large code footprint (instruction-cache pressure).
// All shared-memory indexes are bounded by construction (checked on the host below).
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "sdv_qmatmul.cuh"

using namespace sdv;

constexpr int NBLK = 32;        // blocks per unit in the stage
constexpr int NU_MAX = 4;       // units per stage
constexpr int REC = 576;
constexpr int M_POS = 5;

struct Layout {
    static constexpr uint32_t rec_off = 0;
    static constexpr uint32_t rec_bytes = NU_MAX * NBLK * REC;                      // 73,728
    static constexpr uint32_t act_off = rec_bytes;
    static constexpr uint32_t act_bytes = NBLK * 64 * 8;                             // fragments for up to 8 positions
    static constexpr uint32_t meta_off = act_off + act_bytes;
    static constexpr uint32_t meta_bytes = NBLK * 64;
    static constexpr uint32_t total = meta_off + meta_bytes;
    static constexpr uint32_t with_ring = total + 64 + 36864;
};

__device__ __forceinline__ uint32_t hash32(uint32_t x) {
    x ^= x >> 16; x *= 0x7feb352dU; x ^= x >> 15; x *= 0x846ca68bU; x ^= x >> 16;
    return x;
}

__device__ void fill(uint8_t *smem, int M) {
    const int tid = threadIdx.x, nt = blockDim.x;
    uint32_t *w = reinterpret_cast<uint32_t *>(smem);
    // records: codes random, scales fp16 in [0.001, 0.002)
    for (int r = 0; r < NU_MAX * NBLK; ++r) {
        uint32_t *rw = w + r * (REC / 4);
        for (int i = tid; i < 128; i += nt) rw[i] = hash32(r * 1000 + i + 17 * blockIdx.x);
        __half *sc = reinterpret_cast<__half *>(reinterpret_cast<uint8_t *>(rw) + 512);
        for (int i = tid; i < 32; i += nt) sc[i] = __float2half(0.001f * (1.0f + (hash32(r * 77 + i) & 1023) / 1024.0f));
    }
    // activation fragments (NT = 1): per block M*4 uint4 entries of fp16 pairs (values -127..127, k+8 halves / 16)
    uint4 *act = reinterpret_cast<uint4 *>(smem + Layout::act_off);
    for (int i = tid; i < NBLK * 8 * 4; i += nt) {
        uint32_t h = hash32(i * 13 + 5);
        int a0 = static_cast<int>(h & 255) - 128, a1 = static_cast<int>((h >> 8) & 255) - 128;
        if (a0 < -127) a0 = -127;
        if (a1 < -127) a1 = -127;
        act[i] = make_uint4(pack_h2(a0, a1, 1.0f), pack_h2(a1, a0, 0.0625f), pack_h2(a0, -a1, 1.0f), pack_h2(-a0, a1, 0.0625f));
    }
    float2 *meta = reinterpret_cast<float2 *>(smem + Layout::meta_off);
    for (int i = tid; i < NBLK * 8; i += nt) {
        const int m = i & 7;
        meta[i] = m < M ? make_float2(-1032.0f * ((i * 7) % 50), 0.01f + 0.001f * m) : make_float2(0.0f, 0.0f);
    }
}

// --- variant 0: the product's stage_compute over a 64-record stage (units 0, 1 x 32 blocks in unit-major order)
// --- variant R (1, 2, 4): one B fragment per block reused over R units' records

__device__ __forceinline__ unsigned long long as_u64(float2 v) { return *reinterpret_cast<unsigned long long *>(&v); }
__device__ __forceinline__ float2 as_f2(unsigned long long v) { return *reinterpret_cast<float2 *>(&v); }
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(as_u64(a)), "l"(as_u64(b)), "l"(as_u64(c)));
    return as_f2(d);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(as_u64(a)), "l"(as_u64(b)));
    return as_f2(d);
}

// VAR 5..8: the product's loop shape (RPW = 4 records per warp per 32-record sub-step, unrolled) with
//  PACK: scaling in f32x2 (pairs over the two positions of a lane: (w_r, w_r) x (da0, da1))
//  PAD : activation fragments zero-padded to 8 positions (unconditional load)
template <bool PACK, bool PAD>
__device__ __forceinline__ void stage_v(const uint8_t *sbase, const uint8_t *act, const float *meta, int M, int warp,
                                        int lane, float2 (&acc)[2][2]) {
    const int lg = lane >> 2, lc = lane & 3;
    const uint4 *act4 = reinterpret_cast<const uint4 *>(act);
    const float4 *meta4 = reinterpret_cast<const float4 *>(meta);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = warp + 8 * i;
        const uint8_t *rp = sbase + r * REC;
        const int jb = r;
        uint32_t af[2][2][4];
        q4_frag(*reinterpret_cast<const uint4 *>(rp + lane * 16), af);
        const uint2 sw = *reinterpret_cast<const uint2 *>(rp + 512 + lg * 8);
        uint4 bf;
        if (PAD) bf = act4[jb * 32 + lane];
        else bf = lg < M ? act4[jb * 4 * M + lane] : make_uint4(0u, 0u, 0u, 0u);
        const float4 mt = meta4[jb * 4 + lc];
        const float2 corr = make_float2(mt.x, mt.z);
        const float2 da = make_float2(mt.y, mt.w);
        float d[2][4];
        record_dots(af, bf, corr, d);
        if (PACK) {
            const __half2 h01 = *reinterpret_cast<const __half2 *>(&sw.x), h23 = *reinterpret_cast<const __half2 *>(&sw.y);
            const float2 wr[4] = {__half22float2(__low2half2(h01)), __half22float2(__high2half2(h01)),
                                  __half22float2(__low2half2(h23)), __half22float2(__high2half2(h23))};
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    acc[t][h] = ffma2(make_float2(d[t][2 * h], d[t][2 * h + 1]), fmul2(wr[2 * t + h], da), acc[t][h]);
        } else {
            const float2 w01 = __half22float2(*reinterpret_cast<const __half2 *>(&sw.x));
            const float2 w23 = __half22float2(*reinterpret_cast<const __half2 *>(&sw.y));
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const float2 w = t ? w23 : w01;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float ww = h ? w.y : w.x;
                    acc[t][h].x = __fmaf_rn(d[t][2 * h], __fmul_rn(ww, da.x), acc[t][h].x);
                    acc[t][h].y = __fmaf_rn(d[t][2 * h + 1], __fmul_rn(ww, da.y), acc[t][h].y);
                }
            }
        }
    }
}

template <int R, int NW>
__device__ __forceinline__ void stage_reuse(const uint8_t *sbase, const uint8_t *act, const float *meta, int M,
                                            int warp, int lane, float (&acc)[R][2][4]) {
    const int lg = lane >> 2, lc = lane & 3;
    const uint4 *act4 = reinterpret_cast<const uint4 *>(act);
    const float4 *meta4 = reinterpret_cast<const float4 *>(meta);
#pragma unroll 1
    for (int i = 0; i < NBLK / NW; ++i) {
        const int jb = warp + NW * i;
        const uint4 bf = lg < M ? act4[jb * 4 * M + lane] : make_uint4(0u, 0u, 0u, 0u);
        const float4 mt = meta4[jb * 4 + lc];
        const float2 corr = make_float2(mt.x, mt.z);
        const float da0 = mt.y, da1 = mt.w;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t *rp = sbase + (r * NBLK + jb) * REC;
            uint32_t af[2][2][4];
            q4_frag(*reinterpret_cast<const uint4 *>(rp + lane * 16), af);
            const uint2 sw = *reinterpret_cast<const uint2 *>(rp + 512 + lg * 8);
            const float2 w01 = __half22float2(*reinterpret_cast<const __half2 *>(&sw.x));
            const float2 w23 = __half22float2(*reinterpret_cast<const __half2 *>(&sw.y));
            float d[2][4];
            record_dots(af, bf, corr, d);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const float2 w = t ? w23 : w01;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[r][t][e] = __fmaf_rn(d[t][e], __fmul_rn((e >> 1) ? w.y : w.x, (e & 1) ? da1 : da0), acc[r][t][e]);
            }
        }
    }
}

__device__ int g_done[1024];

// a large straight-line code region (N fused multiply-adds with distinct immediates)
template <int N>
__device__ __noinline__ float bigcode(float x) {
#pragma unroll
    for (int i = 0; i < N; ++i) x = __fmaf_rn(x, 1.0f + static_cast<float>(i) * 1e-7f, static_cast<float>(i & 7) * 1e-3f);
    return x;
}

template <int VAR, int NW>
__global__ void __launch_bounds__(NW * 32 + 128, 1) probe(float *out, long long *cyc, int iters, int M, int interfere,
                                                            const uint8_t *src, size_t src_bytes) {
    const int nwarps = NW;
    extern __shared__ __align__(1024) uint8_t smem[];
    fill(smem, M);
    if (threadIdx.x == 0) g_done[blockIdx.x] = 0;
    __syncthreads();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float s = 0.0f;
    long long t0 = clock64();
    if (warp < nwarps) {
        if constexpr (VAR >= 5) {
            constexpr bool PACK = VAR == 6 || VAR == 8, PAD = VAR == 7 || VAR == 8;
            float2 acc[2][2] = {};
            for (int it = 0; it < iters; ++it) {
#pragma unroll 1
                for (int h = 0; h < 2; ++h)
                    stage_v<PACK, PAD>(smem + h * 32 * REC, smem + Layout::act_off,
                                       reinterpret_cast<const float *>(smem + Layout::meta_off), M, warp, lane, acc);
            }
            for (int t = 0; t < 2; ++t)
                for (int e = 0; e < 2; ++e) s += acc[t][e].x + acc[t][e].y;
        } else if constexpr (VAR == 0) {
            float acc[1][2][4] = {}, accu[1][2][4] = {};
            const float2 inv[1] = {make_float2(1.0f, 1.0f)};
            for (int it = 0; it < iters; ++it) {
                // 64 records: records 0..31 (unit 0 blocks 0..31), 32..63 (unit 1)
#pragma unroll 1
                for (int h = 0; h < 2; ++h)
                    stage_compute<SD_Q4_32, 0, 1, true>(smem + h * 32 * REC, 32, 0, smem + Layout::act_off,
                                                        reinterpret_cast<const float *>(smem + Layout::meta_off), M,
                                                        warp, lane, inv, acc, accu);
            }
            for (int t = 0; t < 2; ++t)
                for (int e = 0; e < 4; ++e) s += acc[0][t][e];
        } else {
            constexpr int R = VAR;
            float acc[R][2][4] = {};
            for (int it = 0; it < iters; ++it) {
                // the same number of records per iteration: 64 (R units x 32 blocks, repeated 2/R times)
                for (int rep = 0; rep < (R == 1 ? 2 : 1); ++rep)
                    stage_reuse<R, NW>(smem, smem + Layout::act_off,
                                       reinterpret_cast<const float *>(smem + Layout::meta_off), M, warp, lane, acc);
            }
            for (int r = 0; r < R; ++r)
                for (int t = 0; t < 2; ++t)
                    for (int e = 0; e < 4; ++e) s += acc[r][t][e];
        }
    }
    long long t1 = clock64();
    if (warp < nwarps) {
        __syncwarp();
        if (lane == 0) atomicAdd(&g_done[blockIdx.x], 1);
    } else if (interfere && warp == nwarps) {
        // a producer warp: bulk copies of 36 KB from a global buffer into the spare ring, back to back,
        // until every consumer warp is done (bounded by a cycle budget)
        if (lane == 0) {
            uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Layout::total);
            uint8_t *dst = smem + Layout::total + 64;
            mbar_init(bar, 1);
            fence_barrier_init();
            uint32_t ph = 0;
            const long long tlim = clock64() + 2000000000ll;
            while (atomicAdd(&g_done[blockIdx.x], 0) < nwarps && clock64() < tlim) {
                mbar_arrive_expect_tx(bar, 36864);
                bulk_g2s_l2keep(dst, src + (static_cast<size_t>(blockIdx.x) * 36864) % src_bytes, 36864, bar);
                if (!mbar_wait_bounded(bar, ph, 1000000000ull)) break;
                ph ^= 1u;
            }
        }
    } else if (interfere == 2 && warp > nwarps) {
        // finisher-like warps polling until the consumers are done
        const long long tlim = clock64() + 2000000000ll;
        while (atomicAdd(&g_done[blockIdx.x], 0) < nwarps && clock64() < tlim) __nanosleep(100);
    } else if (interfere >= 3 && warp > nwarps) {
        // warps running through a large code region until the consumers are done (instruction cache)
        const long long tlim = clock64() + 2000000000ll;
        float x = static_cast<float>(tid);
        while (atomicAdd(&g_done[blockIdx.x], 0) < nwarps && clock64() < tlim) {
            x = interfere == 3 ? bigcode<2048>(x) : bigcode<8192>(x);
            if (interfere == 5) __nanosleep(2000);
        }
        s = x;
    }
    out[blockIdx.x * blockDim.x + tid] = s;
    __syncthreads();
    if (tid == 0) cyc[blockIdx.x] = t1 - t0;
}

// records per iteration processed by the CTA for each variant
static int recs_per_iter(int var) {
    switch (var) {
        case 0: return 64;
        case 1: return 2 * 32;  // rep = 2, R = 1
        case 2: return 1 * 64;  // rep = 1, R = 2
        case 4: return 1 * 128; // rep = 1, R = 4
        case 3: return 0;
        case 5: case 6: case 7: case 8: return 64;
    }
    return 0;
}

static uint8_t *g_src = nullptr;
static size_t g_src_bytes = 0;

template <int VAR, int NW>
static void run(const char *name, int sms, int iters, int M, float *d_out, long long *d_cyc, int interfere = 0) {
    const int nwarps = NW;
    auto k = probe<VAR, NW>;
    const size_t smem = Layout::with_ring;
    cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    for (int rep = 0; rep < 3; ++rep) k<<<sms, NW * 32 + 128, smem>>>(d_out, d_cyc, iters, M, interfere, g_src, g_src_bytes);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        printf("%s: %s\n", name, cudaGetErrorString(e));
        exit(1);
    }
    std::vector<long long> cyc(sms);
    cudaMemcpy(cyc.data(), d_cyc, sms * sizeof(long long), cudaMemcpyDeviceToHost);
    double mean = 0;
    long long mx = 0;
    for (auto c : cyc) {
        mean += c;
        mx = c > mx ? c : mx;
    }
    mean /= sms;
    const double recs = (double)iters * recs_per_iter(VAR);
    printf("%-36s warps=%2d M=%d interfere=%d  cycles/record mean %.2f  max %.2f\n", name, nwarps, M, interfere,
           mean / recs, mx / recs);
}

int main(int argc, char **argv) {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    const int iters = argc > 1 ? atoi(argv[1]) : 200;
    const char *only = argc > 2 ? argv[2] : "";
    // host check of the bounds: the largest record index is (NU_MAX * NBLK - 1), act index NBLK*4*M - 1 < NBLK*4*8
    static_assert(Layout::with_ring <= 227 * 1024, "shared memory");
    float *d_out;
    long long *d_cyc;
    cudaMalloc(&d_out, sms * 1024 * sizeof(float));
    cudaMalloc(&d_cyc, sms * sizeof(long long));
    printf("SMs %d, iters %d\n", sms, iters);
    auto want = [&](const char *n) { return only[0] == 0 || strstr(n, only) != nullptr; };
    g_src_bytes = 152ull * 36864 * 2;
    cudaMalloc(&g_src, g_src_bytes);
    cudaMemset(g_src, 1, g_src_bytes);
    if (want("v0")) run<0, 8>("v0 product stage_compute", sms, iters, M_POS, d_out, d_cyc);
    if (want("intf")) {
        run<0, 8>("v0 + producer copies", sms, iters, M_POS, d_out, d_cyc, 1);
        run<0, 8>("v0 + producer + pollers", sms, iters, M_POS, d_out, d_cyc, 2);
    }
    if (want("v5")) run<5, 8>("v5 product shape, scalar", sms, iters, M_POS, d_out, d_cyc);
    if (want("v6")) run<6, 8>("v6 f32x2 scaling", sms, iters, M_POS, d_out, d_cyc);
    if (want("v7")) run<7, 8>("v7 padded acts", sms, iters, M_POS, d_out, d_cyc);
    if (want("v8")) run<8, 8>("v8 f32x2 + padded acts", sms, iters, M_POS, d_out, d_cyc);
    if (want("v8i")) run<8, 8>("v8 + producer + pollers", sms, iters, M_POS, d_out, d_cyc, 2);
    if (want("icache")) {
        run<0, 8>("v0 + 3 warps in 32 KB of code", sms, iters, M_POS, d_out, d_cyc, 3);
        run<0, 8>("v0 + 3 warps in 128 KB of code", sms, iters, M_POS, d_out, d_cyc, 4);
        run<0, 8>("v0 + 3 warps in 128 KB, sleeping", sms, iters, M_POS, d_out, d_cyc, 5);
    }
    if (want("v1")) run<1, 8>("v1 reuse R=1", sms, iters, M_POS, d_out, d_cyc);
    if (want("v2")) run<2, 8>("v2 reuse R=2", sms, iters, M_POS, d_out, d_cyc);
    if (want("v4")) run<4, 8>("v4 reuse R=4", sms, iters, M_POS, d_out, d_cyc);
    if (want("w16")) {
        run<1, 16>("v1 reuse R=1 (16 warps)", sms, iters, M_POS, d_out, d_cyc);
        run<2, 16>("v2 reuse R=2 (16 warps)", sms, iters, M_POS, d_out, d_cyc);
        run<4, 16>("v4 reuse R=4 (16 warps)", sms, iters, M_POS, d_out, d_cyc);
    }
    cudaFree(d_out);
    cudaFree(d_cyc);
    return 0;
}
