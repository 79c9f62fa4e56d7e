// tcgen05 microbenchmark (run by `python bench.py --probe tcgen05`), for the choice between legacy
// mma.sync in the consumer warps and the 5th-generation tensor-core instructions:
// (1) one kind::f16 MMA, M=128 N=8 K=16, A (fp16 integers) in tensor memory, B in shared memory
//     (K-major, no swizzle), D fp32 in tensor memory, checked against the exact integer products;
// (2) the cost of tcgen05.st x16 + tcgen05.ld x8 (with their waits) per warp, 8 warps per SM: the
//     tensor-memory traffic of one 32x32 record (A in, D out);
// (3) the issue rate of back-to-back MMAs of that shape from one thread (a commit and a wait every 32).
// kind::i8 is not accepted by ptxas for sm_103a, so the integer form cannot be timed.
// Every wait is bounded; the tensor memory is released before the kernel ends.
#include <cstdint>
#include <cstdio>
#include <cuda_fp16.h>

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    const long long lim = clock64() + 4000000000ll;  // about 2 s
    while (!mbar_try(bar, parity))
        if (clock64() > lim) return false;
    return true;
}

__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3FFF);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version (sm_100 family)
    return d;                             // base offset 0, no swizzle
}

__device__ __forceinline__ void mma_f16_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.u32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                 ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

constexpr int R_ST = 2048, R_MMA = 2048;

__global__ void __launch_bounds__(256, 1) probe(int *err, long long *cyc_st, long long *cyc_mma, float *dsample) {
    __shared__ __align__(1024) uint8_t bbuf[16384];
    __shared__ uint64_t bar;
    __shared__ uint32_t tbase;
    __shared__ int fail;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    for (int i = tid; i < 16384 / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(bbuf)[i] = 0u;
    // B (N=8 x K=16, K-major): element (n, k) at (k / 8) * 128 + n * 16 + (k % 8) * 2
    if (tid < 128) {
        const int n = tid / 16, k = tid % 16;
        reinterpret_cast<__half *>(bbuf)[((k / 8) * 128 + n * 16 + (k % 8) * 2) / 2] =
            __int2half_rn((n + k) % 5 - 2);
    }
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fail = 0;
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&tbase)) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B writes before the tensor core reads them
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t base = tbase;
    const uint32_t quarter = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t idesc = (1u << 4) | (1u << 17) | (8u << 24);  // D f32, A/B f16, K-major, N=8, M=128
    const uint64_t bd = sdesc(smem_u32(bbuf), 128, 256);

    // (1) A rows r = 0..127 (lane r of TMEM), K = 16 fp16 in columns 0..7: a[r][k] = (r + 3k) % 7 - 3
    if (warp < 4) {
        const int r = 32 * warp + lane;
        uint32_t v[8];
        for (int j = 0; j < 8; ++j) {
            const __half2 h = __halves2half2(__int2half_rn((r + 6 * j) % 7 - 3), __int2half_rn((r + 6 * j + 3) % 7 - 3));
            v[j] = *reinterpret_cast<const uint32_t *>(&h);
        }
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(base + quarter),
                     "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]) : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (tid == 0) {
        mma_f16_ts(base + 64, base, bd, idesc, 0u);
        commit(&bar);
    }
    if (!mbar_wait(&bar, 0)) fail = 1;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp < 4 && !fail) {
        const int r = 32 * warp + lane;
        uint32_t d[8];
        asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7])
                     : "r"(base + quarter + 64) : "memory");
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        int bad = 0;
        for (int n = 0; n < 8; ++n) {
            int e = 0;
            for (int k = 0; k < 16; ++k) e += ((r + 3 * k) % 7 - 3) * ((n + k) % 5 - 2);
            if (__uint_as_float(d[n]) != static_cast<float>(e)) ++bad;
            if (blockIdx.x == 0 && r < 4) dsample[r * 8 + n] = __uint_as_float(d[n]);
        }
        if (bad) atomicAdd(err, bad);
    }
    if (fail && tid == 0) atomicAdd(err + 1, 1);

    // (2) tcgen05.st x16 + ld x8 per warp, all 8 warps (two per lane quarter, separate columns)
    {
        uint32_t v[16];
        for (int j = 0; j < 16; ++j) v[j] = static_cast<uint32_t>(tid * 16 + j);
        const uint32_t col = 128 + static_cast<uint32_t>(warp >> 2) * 64;
        uint32_t sum = 0;
        __syncthreads();
        const long long t0 = clock64();
        for (int i = 0; i < R_ST; ++i) {
            const uint32_t c = col + static_cast<uint32_t>(i & 1) * 16;
            asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                         ::"r"(base + quarter + c), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                         "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
                         "r"(v[14]), "r"(v[15]) : "memory");
            asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            uint32_t d[8];
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                         : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3]), "=r"(d[4]), "=r"(d[5]), "=r"(d[6]), "=r"(d[7])
                         : "r"(base + quarter + c) : "memory");
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            for (int j = 0; j < 8; ++j) sum += d[j];
            v[i & 15] += sum & 1u;
        }
        const long long t1 = clock64();
        if (lane == 0) cyc_st[blockIdx.x * 8 + warp] = t1 - t0;
        if (sum == 0x12345678u) atomicAdd(err + 2, 1);  // keeps the loads live
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // (3) back-to-back MMAs (D columns 256..383 in 16 groups of 8), one thread issues, a commit every 32
    if (tid == 0 && !fail) {
        const long long t0 = clock64();
        uint32_t ph = 1;  // phase 0 of the barrier completed in (1)
        for (int i = 0; i < R_MMA; ++i) {
            mma_f16_ts(base + 256 + static_cast<uint32_t>(i & 15) * 8, base, bd, idesc, 1u);
            if ((i & 31) == 31) {
                commit(&bar);
                if (!mbar_wait(&bar, ph)) {
                    fail = 1;
                    break;
                }
                ph ^= 1u;
            }
        }
        const long long t1 = clock64();
        cyc_mma[blockIdx.x] = t1 - t0;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (fail && tid == 0) atomicAdd(err + 1, 1);
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(base) : "memory");
}

int main() {
    int nsm = 0;
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, 0);
    int *err;
    long long *cs, *cm;
    float *ds;
    cudaMalloc(&err, 16);
    cudaMemset(err, 0, 16);
    cudaMalloc(&cs, sizeof(long long) * nsm * 8);
    cudaMalloc(&cm, sizeof(long long) * nsm);
    cudaMalloc(&ds, sizeof(float) * 32);
    cudaMemset(cm, 0, sizeof(long long) * nsm);
    probe<<<nsm, 256>>>(err, cs, cm, ds);
    cudaError_t e = cudaDeviceSynchronize();
    printf("launch: %s\n", cudaGetErrorString(e));
    if (e != cudaSuccess) return 1;
    int h_err[4];
    long long h_cs[152 * 8], h_cm[152];
    float h_ds[32];
    cudaMemcpy(h_err, err, 16, cudaMemcpyDeviceToHost);
    cudaMemcpy(h_cs, cs, sizeof(long long) * nsm * 8, cudaMemcpyDeviceToHost);
    cudaMemcpy(h_cm, cm, sizeof(long long) * nsm, cudaMemcpyDeviceToHost);
    cudaMemcpy(h_ds, ds, sizeof(h_ds), cudaMemcpyDeviceToHost);
    printf("mma result mismatches: %d, waits failed: %d\n", h_err[0], h_err[1]);
    printf("D rows 0..3: ");
    for (int i = 0; i < 32; ++i) printf("%g%s", h_ds[i], (i % 8 == 7) ? " | " : " ");
    printf("\nexpected rows 0..3: ");
    for (int r = 0; r < 4; ++r) {
        for (int n = 0; n < 8; ++n) {
            int ex = 0;
            for (int k = 0; k < 16; ++k) ex += ((r + 3 * k) % 7 - 3) * ((n + k) % 5 - 2);
            printf("%d ", ex);
        }
        printf("| ");
    }
    double st = 0, stmax = 0, mm = 0;
    for (int i = 0; i < nsm * 8; ++i) {
        st += h_cs[i];
        if (h_cs[i] > stmax) stmax = h_cs[i];
    }
    for (int i = 0; i < nsm; ++i) mm += h_cm[i];
    printf("\nst x16 + ld x8 (+waits) per warp iteration: %.1f cycles mean, %.1f max (8 warps per SM running together)\n",
           st / (nsm * 8) / R_ST, stmax / R_ST);
    printf("  per SM: %.2f cycles per (st+ld) pair\n", stmax / R_ST / 8);
    printf("MMA M128 N8 K16 f16 (A in TMEM), one thread issuing, commit+wait every 32: %.2f cycles per MMA\n",
           mm / nsm / R_MMA);
    return 0;
}
