// sdv_attn.cu - decode attention of the verify pass over the K+1 positions ("Inside OpenJet
// Engine", section "Cheap drafting, careful state management": split-K flash decoding of the
// full-attention layers, fp16 K/V with fp32 accumulation; "How Kinetic is fast", section "Where
// the guesses come from": each row of a draft tree sees only its own path; "Speculative Decoding
// with Open-Weights Models", section "Engineering the Architecture: KV Cache Synchronization":
// rejected entries are dropped in place).
//
// Cache: per KV head, fp16 K and V rows [S_max][D]; L committed rows, then the M new positions.
// Query row (i, h) sees every committed row and new row j iff j is on i's path; query head h
// reads KV head h / (H / H_kv); out = softmax(q k^T / sqrt(D)) v.
//
// The context is read once per KV head for all its query rows (M positions x the heads of the
// group, up to 8 per CTA): the keys are split into chunks, one CTA per (chunk, query group, KV
// head) streaming its K and V rows through shared memory (attn_tc_kernel below: fp16 tensor-core
// products with fp32 accumulation); each CTA leaves an unnormalised (max, sum, o) per row and a
// second kernel combines the chunks.  Scores are kept in log2 units (q is scaled by
// log2(e)/sqrt(D) once) and exponentials are exp2f.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "sdv_common.cuh"

namespace sdv {

constexpr int AT_TQ = 8;     // query rows per CTA
constexpr int AT_MIN_CHUNK_PAIRS = 32;
constexpr float AT_NEG = -3.402823466e38f;  // running-max start: finite, below every score

struct AttnArgs {
    const float *q;         // [M][H][D]
    const __half *kc, *vc;  // [H_kv][S_max][D]
    const int32_t *parent;  // [M] or nullptr (chain)
    float *part_ml;         // [H_kv][QG][S][AT_TQ][2]: running max (log2 units), sum of exp2
    float *part_o;          // [H_kv][QG][S][AT_TQ][D]: unnormalised output
    float *out;             // [M][H][D]
    int64_t S_max, L, NK;   // NK = L + M keys
    int64_t chunk_pairs;    // key pairs per chunk
    int32_t M, H, H_kv, g;  // g = H / H_kv
    int32_t QG, S;          // query groups per KV head, key chunks
    float qscale;           // log2(e) / sqrt(D)
    int *status;
};

// bit j set: new row L+j is visible to position i (i itself and its ancestors)
__device__ __forceinline__ uint32_t path_mask(const AttnArgs &a, int i) {
    if (!a.parent) return (2u << i) - 1u;
    uint32_t m = 0;
    int x = i;
    for (int step = 0; step <= i && x >= 0; ++step) {
        m |= 1u << x;
        const int p = a.parent[x];
        if (p >= x) {  // parents come before their children; anything else is a bad tree
            set_status(a.status, SD_EDEVICE);
            break;
        }
        x = p;
    }
    return m;
}

// ---------------------------------------------------------------------------
// Tensor-core partial attention.  One CTA per (key chunk, query group of 8 rows, KV head): a producer
// thread streams the chunk's K and V rows (fp16, as cached) into a ring of shared-memory stages of
// AT_KT keys with tensor copies (TMA; tiles of AT_KT rows x 64 halves, 128-byte swizzled so the
// fragment loads are free of bank conflicts; rows past the last key arrive as zeros); four
// consumer warps each take 16 keys of a stage:
//   S^T = K Q^T on mma m16n8k16 (keys x rows, fp32 accumulation), with q split into an fp16 high
//   part and an fp16 remainder (two mma into the same accumulator), each row pre-scaled by a power
//   of two so neither part is subnormal; scores in exp2 units;
//   online softmax per row (running max and sum in fp32, masked keys at -inf);
//   O^T += V^T P^T on the same mma, P split the same way (scaled by 2^14), its fragments moved from
//   the score layout to the operand layout by register transposes (movmatrix).
// Each warp keeps its own (max, sum, O) per row; the CTA merges its warps at the end and leaves one
// partial per row for the combine kernel.
// ---------------------------------------------------------------------------
constexpr int AT_KT = 64;          // keys per stage (16 per consumer warp)
constexpr int AT_NST = 2;          // ring stages (three CTAs per SM)
constexpr int AT_CW = 4;           // consumer warps
constexpr float AT_PS = 16384.0f;  // P scaling into the fp16 operand (a power of two: exact)

template <int D>
struct AtLayout {
    static constexpr int TILE = AT_KT * 128;              // one tensor tile: AT_KT rows x 64 halves
    static constexpr int NB = D / 64;                     // tiles across a row
    static constexpr int STAGE = 2 * NB * TILE;           // K tiles then V tiles
    static constexpr int RING = AT_NST * STAGE;
    static constexpr int BARS = RING;                     // full[AT_NST], empty[AT_NST], abort flag
    static constexpr int TOTAL = 1024 + RING + 16 * AT_NST + 16;  // + room to align the ring to 1024 B
    static_assert((AT_CW + 1) * AT_TQ * (D + 2) * 4 <= RING, "the warps' states and the chunk's partial fit in the ring");
};

// byte offset, inside a stage's K or V tiles, of the 16-byte chunk holding halves d .. d+7 of row r
// (the 128-byte swizzle: chunk j of a 128-byte row r sits at chunk j ^ (r & 7))
template <int D>
__device__ __forceinline__ uint32_t at_off(int r, int d) {
    return static_cast<uint32_t>((d >> 6) * AtLayout<D>::TILE + r * 128 + ((((d & 63) >> 3) ^ (r & 7)) << 4));
}

// one tile of a cache viewed as [H_kv][NK][D] halves (x = d, y = key, z = KV head)
__device__ __forceinline__ void tma_3d(void *dst, const CUtensorMap *tm, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// thread-block cluster: a barrier of every thread of every CTA (release / acquire), this CTA's rank,
// and an fp32 load from the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t local_addr, int rank) {
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}
__device__ __forceinline__ void hmma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// (x0, x1) as an fp16 pair plus the fp16 pair of what that leaves over
__device__ __forceinline__ void split_h2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// CL > 0: the grid's CL chunks of each (query group, KV head) form one thread-block cluster, and the
// chunks are merged through distributed shared memory at the end (no partials in global memory, no
// combine launch); CL = 0: partials for attn_combine_kernel.
template <int D, int CL>
__global__ void __launch_bounds__(32 * (AT_CW + 1)) attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                                                                   const __grid_constant__ CUtensorMap tmv) {
    using LY = AtLayout<D>;
    constexpr int KS = D / 16;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);  // the swizzle wants 1024 B
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + LY::BARS);
    uint64_t *empty = full + AT_NST;
    volatile int *abort = reinterpret_cast<volatile int *>(smem + LY::BARS + 16 * AT_NST);
    const int sc = blockIdx.x, qg = blockIdx.y, kh = blockIdx.z;
    const int warp = static_cast<int>(threadIdx.x) >> 5, lane = static_cast<int>(threadIdx.x) & 31;
    const int g = lane >> 2, c = lane & 3;
    const int rows = a.M * a.g;
    const int64_t k0 = static_cast<int64_t>(sc) * a.chunk_pairs * 2;  // the chunk's keys [k0, k1)
    const int64_t k1 = min(a.NK, k0 + a.chunk_pairs * 2);
    const int nst = k1 > k0 ? static_cast<int>((k1 - k0 + AT_KT - 1) / AT_KT) : 0;

    // every row of a tile holds finite values (cache rows below NK, zeros past it): masked keys weigh
    // their V rows by exactly 0
    if (threadIdx.x == 0) {
        for (int i = 0; i < AT_NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], AT_CW);
        }
        *abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    float m0 = AT_NEG, m1 = AT_NEG, l0 = 0.0f, l1 = 0.0f;  // rows 2c, 2c+1 of this warp
    float o[KS][4];                                         // O^T: d = 16 dt + g (+8), rows 2c, 2c+1
#pragma unroll
    for (int dt = 0; dt < KS; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dt][e] = 0.0f;

    if (warp == AT_CW) {  // producer: one thread issues the stage's tensor copies
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < nst; ++i) {
                const int slot = i % AT_NST;
                if (i >= AT_NST && !mbar_wait_bounded(&empty[slot], ((i / AT_NST) - 1) & 1u, 2000000000ull, abort)) {
                    set_status(a.status, SD_ETIMEOUT);
                    *abort = 1;
                    break;
                }
                const int y = static_cast<int>(k0) + i * AT_KT;
                mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(LY::STAGE));  // zero-filled rows count too
                uint8_t *st = smem + slot * LY::STAGE;
#pragma unroll
                for (int b = 0; b < LY::NB; ++b) {
                    tma_3d(st + b * LY::TILE, &tmk, 64 * b, y, kh, &full[slot]);
                    tma_3d(st + (LY::NB + b) * LY::TILE, &tmv, 64 * b, y, kh, &full[slot]);
                }
                ++issued;
            }
            // never leave with copies in flight
            for (int i = issued > AT_NST ? issued - AT_NST : 0; i < issued; ++i)
                mbar_wait_bounded(&full[i % AT_NST], (i / AT_NST) & 1u, 2000000000ull);
        }
        __syncwarp();
    } else {
        // B fragments of query row g (high and low fp16 parts), scaled by 2^(11-e) for max |q| in [2^(e-1), 2^e)
        uint32_t qh[KS][2], ql[KS][2];
        float rsc = 0.0f;  // the scale back, 2^(e-11), of row g
        {
            const int tg = qg * AT_TQ + g;
            const bool real = tg < rows;
            const int i = real ? tg / a.g : 0, h = real ? kh * a.g + tg % a.g : 0;
            const float *qp = a.q + (static_cast<int64_t>(i) * a.H + h) * D;
            float qv[KS][4];
            float mx = 0.0f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int d = 16 * ks + 2 * c + (e & 1) + 8 * (e >> 1);
                    qv[ks][e] = real ? __fmul_rn(qp[d], a.qscale) : 0.0f;
                    mx = fmaxf(mx, fabsf(qv[ks][e]));
                }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            int ex = 0;
            if (mx > 0.0f) (void)frexpf(mx, &ex);
            const float up = ldexpf(1.0f, 11 - ex);
            rsc = mx > 0.0f ? ldexpf(1.0f, ex - 11) : 0.0f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                split_h2(qv[ks][0] * up, qv[ks][1] * up, qh[ks][0], ql[ks][0]);
                split_h2(qv[ks][2] * up, qv[ks][3] * up, qh[ks][1], ql[ks][1]);
            }
        }
        // rows 2c and 2c+1 of the score fragments: scale back, visibility, validity
        const float rs0 = __shfl_sync(0xffffffffu, rsc, 8 * c), rs1 = __shfl_sync(0xffffffffu, rsc, 8 * c + 4);
        uint32_t vis0 = 0, vis1 = 0;
        const int t0r = qg * AT_TQ + 2 * c;
        const bool ok0 = t0r < rows, ok1 = t0r + 1 < rows;
        if (ok0) vis0 = path_mask(a, t0r / a.g);
        if (ok1) vis1 = path_mask(a, (t0r + 1) / a.g);
        const uint32_t sbase = smem_u32(smem);
        // ldmatrix row addresses of this lane: the K tiles (keys x d) and, transposed, the V tiles
        const int kr = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8, kd = (lane >> 4) * 8;
        const int vr = 16 * warp + (lane & 7) + (lane >> 4) * 8, vd = ((lane >> 3) & 1) * 8;
        constexpr uint32_t VOFF = LY::NB * LY::TILE;  // the V tiles after the K tiles
        for (int i = 0; i < nst; ++i) {
            const int slot = i % AT_NST;
            const bool ready = mbar_wait_bounded(&full[slot], (i / AT_NST) & 1u, 2000000000ull, abort);
            if (!__all_sync(0xffffffffu, ready)) {
                if (lane == 0) {
                    set_status(a.status, SD_ETIMEOUT);
                    *abort = 1;
                }
                break;
            }
            const uint32_t st = sbase + slot * LY::STAGE;
            // four independent accumulator chains (high / low part x even / odd k step), then summed
            float sa[4][4] = {};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t ka[4];
                ldsm_x4(st + at_off<D>(kr, 16 * ks + kd), ka);
                hmma(sa[ks & 1], ka, qh[ks][0], qh[ks][1]);
                hmma(sa[2 + (ks & 1)], ka, ql[ks][0], ql[ks][1]);
            }
            float s[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) s[e] = (sa[0][e] + sa[1][e]) + (sa[2][e] + sa[3][e]);
            // s0, s1: key 16w + g, rows 2c, 2c+1; s2, s3: key 16w + g + 8
            const int64_t ja = k0 + static_cast<int64_t>(i) * AT_KT + 16 * warp + g, jb = ja + 8;
            const bool va0 = ok0 && ja < k1 && (ja < a.L || ((vis0 >> static_cast<int>(ja - a.L)) & 1u));
            const bool va1 = ok1 && ja < k1 && (ja < a.L || ((vis1 >> static_cast<int>(ja - a.L)) & 1u));
            const bool vb0 = ok0 && jb < k1 && (jb < a.L || ((vis0 >> static_cast<int>(jb - a.L)) & 1u));
            const bool vb1 = ok1 && jb < k1 && (jb < a.L || ((vis1 >> static_cast<int>(jb - a.L)) & 1u));
            s[0] = va0 ? s[0] * rs0 : -INFINITY;
            s[1] = va1 ? s[1] * rs1 : -INFINITY;
            s[2] = vb0 ? s[2] * rs0 : -INFINITY;
            s[3] = vb1 ? s[3] * rs1 : -INFINITY;
            float x0 = fmaxf(s[0], s[2]), x1 = fmaxf(s[1], s[3]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, off));
                x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, off));
            }
            const float n0 = fmaxf(m0, x0), n1 = fmaxf(m1, x1);
            const float al0 = exp2f(m0 - n0), al1 = exp2f(m1 - n1);
            const float p0 = exp2f(s[0] - n0), p1 = exp2f(s[1] - n1), p2 = exp2f(s[2] - n0), p3 = exp2f(s[3] - n1);
            float r0 = p0 + p2, r1 = p1 + p3;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                r0 += __shfl_xor_sync(0xffffffffu, r0, off);
                r1 += __shfl_xor_sync(0xffffffffu, r1, off);
            }
            l0 = fmaf(l0, al0, r0);
            l1 = fmaf(l1, al1, r1);
            m0 = n0;
            m1 = n1;
#pragma unroll
            for (int dt = 0; dt < KS; ++dt) {
                o[dt][0] *= al0;
                o[dt][1] *= al1;
                o[dt][2] *= al0;
                o[dt][3] *= al1;
            }
            // P^T (keys x rows) as the B operand, high and low fp16 parts
            uint32_t ph01, pl01, ph23, pl23;
            split_h2(p0 * AT_PS, p1 * AT_PS, ph01, pl01);
            split_h2(p2 * AT_PS, p3 * AT_PS, ph23, pl23);
            const uint32_t bh0 = movm_t(ph01), bh1 = movm_t(ph23), bl0 = movm_t(pl01), bl1 = movm_t(pl23);
#pragma unroll
            for (int dt = 0; dt < KS; ++dt) {
                uint32_t va[4];
                ldsm_x4_t(st + VOFF + at_off<D>(vr, 16 * dt + vd), va);
                hmma(o[dt], va, bh0, bh1);
                hmma(o[dt], va, bl0, bl1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }
    __syncthreads();  // every consumer past its loop and every copy landed: the ring is free
    float *sm_m = reinterpret_cast<float *>(smem), *sm_l = sm_m + AT_CW * AT_TQ, *sm_o = sm_l + AT_CW * AT_TQ;
    if (warp < AT_CW) {
        if (g == 0) {
            sm_m[warp * AT_TQ + 2 * c] = m0;
            sm_m[warp * AT_TQ + 2 * c + 1] = m1;
            sm_l[warp * AT_TQ + 2 * c] = l0;
            sm_l[warp * AT_TQ + 2 * c + 1] = l1;
        }
#pragma unroll
        for (int dt = 0; dt < KS; ++dt) {
            float *ow = sm_o + static_cast<size_t>(warp) * AT_TQ * D;
            ow[(2 * c) * D + 16 * dt + g] = o[dt][0];
            ow[(2 * c + 1) * D + 16 * dt + g] = o[dt][1];
            ow[(2 * c) * D + 16 * dt + g + 8] = o[dt][2];
            ow[(2 * c + 1) * D + 16 * dt + g + 8] = o[dt][3];
        }
    }
    __syncthreads();
    const int64_t base = ((static_cast<int64_t>(kh) * a.QG + qg) * a.S + sc) * AT_TQ;
    // the chunk's partial (max, sum, output) per row: to global memory, or (clusters) to shared memory
    // after the warps' states
    float *cm = sm_o + AT_CW * AT_TQ * D, *cl = cm + AT_TQ, *co = cl + AT_TQ;
    for (int idx = threadIdx.x; idx < AT_TQ * D; idx += blockDim.x) {
        const int t = idx / D, d = idx % D;
        float mx = sm_m[t];
#pragma unroll
        for (int w = 1; w < AT_CW; ++w) mx = fmaxf(mx, sm_m[w * AT_TQ + t]);
        float ov = 0.0f, lv = 0.0f;
#pragma unroll
        for (int w = 0; w < AT_CW; ++w) {
            const float f = exp2f(sm_m[w * AT_TQ + t] - mx);
            ov = fmaf(sm_o[(static_cast<size_t>(w) * AT_TQ + t) * D + d], f, ov);
            lv = fmaf(sm_l[w * AT_TQ + t], f, lv);
        }
        if constexpr (CL > 0) {
            co[t * D + d] = ov * (1.0f / AT_PS);
            if (d == 0) {
                cm[t] = mx;
                cl[t] = lv;
            }
        } else {
            a.part_o[(base + t) * D + d] = ov * (1.0f / AT_PS);
            if (d == 0) {
                a.part_ml[(base + t) * 2] = mx;
                a.part_ml[(base + t) * 2 + 1] = lv;
            }
        }
    }
    if constexpr (CL > 0) {
        // every chunk's partial is in its CTA's shared memory; CTA r of the cluster merges columns
        // [r D / CL, (r + 1) D / CL) of every row, reading the CL partials in chunk order
        cluster_sync();
        constexpr int DC = D / CL;
        const uint32_t rank = cluster_rank();
        for (int idx = threadIdx.x; idx < AT_TQ * DC; idx += blockDim.x) {
            const int t = idx / DC, d = static_cast<int>(rank) * DC + idx % DC;
            const int tg = qg * AT_TQ + t;
            if (tg >= rows) continue;
            const uint32_t mt = smem_u32(cm + t), lt = smem_u32(cl + t), ot = smem_u32(co + t * D + d);
            float mx = AT_NEG;
#pragma unroll
            for (int r = 0; r < CL; ++r) mx = fmaxf(mx, ld_cluster_f32(mt, r));
            float lv = 0.0f, ov = 0.0f;
#pragma unroll
            for (int r = 0; r < CL; ++r) {
                const float f = exp2f(ld_cluster_f32(mt, r) - mx);
                lv = fmaf(ld_cluster_f32(lt, r), f, lv);
                ov = fmaf(ld_cluster_f32(ot, r), f, ov);
            }
            const int i = tg / a.g, h = kh * a.g + tg % a.g;
            a.out[(static_cast<int64_t>(i) * a.H + h) * D + d] = ov / lv;
        }
        cluster_sync();  // no CTA leaves while another still reads its shared memory
    }
}

// combine the chunks of one (KV head, query group): one warp per query row, lanes over d.  Each lane
// holds the weight of one chunk (32 chunks at a time) and the warp walks them with the loads of
// several chunks in flight.
template <int DV>
struct VecF;
template <>
struct VecF<2> {
    using T = float2;
    static __device__ __forceinline__ float at(const T &v, int e) { return e == 0 ? v.x : v.y; }
};
template <>
struct VecF<4> {
    using T = float4;
    static __device__ __forceinline__ float at(const T &v, int e) {
        return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    }
};

template <int D>
__global__ void __launch_bounds__(32 * AT_TQ, 1) attn_combine_kernel(const AttnArgs a) {
    constexpr int DV = D / 32;  // elements per lane
    using V = typename VecF<DV>::T;
    static_assert(D % 64 == 0, "two or four floats per lane");
    pdl_wait();
    pdl_launch_dependents();
    const int qg = blockIdx.x, kh = blockIdx.y;
    const int t = static_cast<int>(threadIdx.x) / 32, lane = static_cast<int>(threadIdx.x) & 31;
    const int tg = qg * AT_TQ + t;
    if (tg >= a.M * a.g) return;
    const int i = tg / a.g, h = kh * a.g + tg % a.g;
    const int64_t base = (static_cast<int64_t>(kh) * a.QG + qg) * a.S;
    float mx = AT_NEG;
    for (int s = lane; s < a.S; s += 32) mx = fmaxf(mx, a.part_ml[((base + s) * AT_TQ + t) * 2]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float lv = 0.0f, ov[DV];
#pragma unroll
    for (int e = 0; e < DV; ++e) ov[e] = 0.0f;
    for (int s0 = 0; s0 < a.S; s0 += 32) {
        float f = 0.0f;
        if (s0 + lane < a.S) {
            const int64_t r = (base + s0 + lane) * AT_TQ + t;
            f = exp2f(a.part_ml[r * 2] - mx);
            lv = fmaf(a.part_ml[r * 2 + 1], f, lv);
        }
        const int n = min(32, a.S - s0);
#pragma unroll 8
        for (int j = 0; j < n; ++j) {
            const float fj = __shfl_sync(0xffffffffu, f, j);
            const V v = *reinterpret_cast<const V *>(a.part_o + ((base + s0 + j) * AT_TQ + t) * D + lane * DV);
#pragma unroll
            for (int e = 0; e < DV; ++e) ov[e] = fmaf(VecF<DV>::at(v, e), fj, ov[e]);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lv += __shfl_xor_sync(0xffffffffu, lv, off);
    float *op = a.out + (static_cast<int64_t>(i) * a.H + h) * D + lane * DV;
#pragma unroll
    for (int e = 0; e < DV; ++e) op[e] = ov[e] / lv;
}

// new K/V rows: fp32 [M][H_kv][D] -> fp16 (nearest even) cache slots [L, L+M)
__global__ void kv_append_kernel(const float *k_new, const float *v_new, int32_t M, int32_t H_kv, int32_t D,
                                 __half *kc, __half *vc, int64_t S_max, int64_t L) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t n = static_cast<int64_t>(M) * H_kv * D;
    for (int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < n;
         x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t d = x % D, h = (x / D) % H_kv, i = x / (static_cast<int64_t>(D) * H_kv);
        const int64_t dst = (h * S_max + L + i) * D + d;
        kc[dst] = __float2half_rn(k_new[x]);
        vc[dst] = __float2half_rn(v_new[x]);
    }
}

constexpr int KC_MAXD = 256;

// keep the accepted path: rows L+path[t] -> L+t, t < n = *count; one CTA per KV head stages the
// rows in shared memory first, so moves whose source another move overwrites stay correct
__global__ void __launch_bounds__(128) kv_commit_kernel(__half *kc, __half *vc, int32_t D, int64_t S_max, int64_t L,
                                                        int32_t M, const int32_t *path, const int32_t *count,
                                                        int *status) {
    __shared__ __half sk[16][KC_MAXD], sv[16][KC_MAXD];
    __shared__ int ok;
    pdl_wait();
    pdl_launch_dependents();
    const int n = *count;
    if (threadIdx.x == 0) {
        int good = n >= 1 && n <= M;
        for (int t = 0; good && t < n; ++t)
            good = path[t] >= 0 && path[t] < M && (t == 0 || path[t] > path[t - 1]);
        ok = good;
        if (!good && blockIdx.x == 0) set_status(status, SD_EDEVICE);
    }
    __syncthreads();
    if (!ok) return;
    const int64_t head = static_cast<int64_t>(blockIdx.x) * S_max;
    for (int x = threadIdx.x; x < n * D; x += blockDim.x) {
        const int t = x / D, d = x % D;
        const int64_t src = (head + L + path[t]) * D + d;
        sk[t][d] = kc[src];
        sv[t][d] = vc[src];
    }
    __syncthreads();
    for (int x = threadIdx.x; x < n * D; x += blockDim.x) {
        const int t = x / D, d = x % D;
        const int64_t dst = (head + L + t) * D + d;
        kc[dst] = sk[t][d];
        vc[dst] = sv[t][d];
    }
}

constexpr int AT_CL = 8;                 // chunks per cluster when the chunks merge on chip
constexpr int64_t AT_CL_MAX_KEYS = 16384;  // ... for contexts of at most this many keys

struct AttnPlan {
    int32_t QG, S, CL;  // CL: 0, or S = CL chunks per (query group, KV head) merged in a cluster
    int64_t chunk_pairs;
    size_t off_o, total;
};

static bool attn_plan(int32_t M, int32_t H, int32_t H_kv, int32_t D, int64_t L, AttnPlan &p) {
    if (M < 1 || M > 16 || H_kv < 1 || H < H_kv || H % H_kv || (D != 64 && D != 128) || L < 0) return false;
    const int sms = num_sms();
    if (sms < 1) return false;
    const int64_t rows = static_cast<int64_t>(M) * (H / H_kv);
    p.QG = static_cast<int32_t>((rows + AT_TQ - 1) / AT_TQ);
    const int64_t NP = (L + M + 1) / 2;
    // three CTAs per SM over all (chunk, query group, KV head), in one wave; chunks of whole stages
    const int64_t per = static_cast<int64_t>(p.QG) * H_kv;
    int64_t want = 3 * static_cast<int64_t>(sms) / per;
    if (want < 1) want = 1;
    int64_t cp = (NP + want - 1) / want;
    cp = (cp + AT_KT / 2 - 1) / (AT_KT / 2) * (AT_KT / 2);
    if (cp < AT_MIN_CHUNK_PAIRS) cp = AT_MIN_CHUNK_PAIRS;
    p.chunk_pairs = cp;
    p.S = static_cast<int32_t>((NP + cp - 1) / cp);  // <= want, whatever the context
    // short contexts: AT_CL chunks of at least two stages each, merged in one cluster per (query group,
    // KV head) when those clusters fit in one wave: no partials, no combine launch
    p.CL = 0;
    const int64_t NKeys = L + M;
    if (NKeys <= AT_CL_MAX_KEYS && NKeys >= 2 * AT_KT * AT_CL && per * AT_CL <= 3 * static_cast<int64_t>(sms)) {
        p.CL = AT_CL;
        p.S = AT_CL;
        p.chunk_pairs = ((NP + AT_CL - 1) / AT_CL + AT_KT / 2 - 1) / (AT_KT / 2) * (AT_KT / 2);
    }
    // partials sized for `want` chunks, so one workspace serves every context length
    const size_t nrow = static_cast<size_t>(H_kv) * p.QG * static_cast<size_t>(want) * AT_TQ;
    p.off_o = (nrow * 2 * sizeof(float) + 255) & ~static_cast<size_t>(255);
    p.total = p.off_o + ((nrow * D * sizeof(float) + 255) & ~static_cast<size_t>(255));
    return true;
}

// The driver's tensor-map encoder, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A cache [H_kv][S_max][D] fp16 seen as [H_kv][NK][D]: tiles of AT_KT keys x 64 halves, 128-byte
// swizzle, zeros past key NK.
bool cache_map(CUtensorMap *tm, const void *base, int D, int64_t NK, int64_t S_max, int H_kv) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(NK),
                                static_cast<cuuint64_t>(H_kv)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(S_max) * D * 2};
    const cuuint32_t box[3] = {64, AT_KT, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One launch in clusters of AT_CL CTAs along x (with programmatic dependent launch when enabled).
template <typename K>
cudaError_t attn_cluster_launch(K kernel, dim3 grid, size_t smem, cudaStream_t s, const AttnArgs &a,
                                const CUtensorMap &tmk, const CUtensorMap &tmv) {
    cudaError_t e = allow_max_dynamic_smem(kernel);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(32 * (AT_CW + 1));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = AT_CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, a, tmk, tmv);
}

}  // namespace sdv

using namespace sdv;

extern "C" {

size_t sd_attn_workspace_bytes(int32_t M, int32_t H, int32_t H_kv, int32_t D, int64_t L) {
    AttnPlan p;
    return attn_plan(M, H, H_kv, D, L, p) ? p.total : 0;
}

sd_status sd_kv_append(const float *k_new, const float *v_new, int32_t M, int32_t H_kv, int32_t D, void *k_cache,
                       void *v_cache, int64_t S_max, int64_t L, sd_stream_t stream) {
    SD_NVTX("sd_kv_append");
    if (!k_new || !v_new || !k_cache || !v_cache) return SD_EINVAL;
    if (M < 1 || M > 16 || H_kv < 1 || D < 1 || L < 0 || S_max < L + M) return SD_EINVAL;
    if (!aligned(k_new, 4) || !aligned(v_new, 4) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return SD_EINVAL;
    const int64_t n = static_cast<int64_t>(M) * H_kv * D;
    const int grid = static_cast<int>((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    return launch(kv_append_kernel, dim3(grid), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream), k_new, v_new,
                  M, H_kv, D, static_cast<__half *>(k_cache), static_cast<__half *>(v_cache), S_max, L) ==
                   cudaSuccess
               ? SD_OK
               : SD_ECUDA;
}

sd_status sd_attn_decode(const float *q, const void *k_cache, const void *v_cache, int32_t M, int32_t H,
                         int32_t H_kv, int32_t D, int64_t S_max, int64_t L, const int32_t *parent, float *out,
                         void *workspace, size_t ws_bytes, sd_stream_t stream) {
    SD_NVTX("sd_attn_decode");
    if (!q || !k_cache || !v_cache || !out || !workspace) return SD_EINVAL;
    if (M < 1 || H_kv < 1 || H < H_kv || H % H_kv || L < 0 || S_max < L + M) return SD_EINVAL;
    if (M > 16 || (D != 64 && D != 128)) return SD_EUNSUPPORTED;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(workspace, 256))
        return SD_EINVAL;
    if (L + M > INT32_MAX - AT_KT) return SD_EUNSUPPORTED;  // tensor-copy coordinates are 32-bit
    AttnPlan p;
    if (!attn_plan(M, H, H_kv, D, L, p)) return SD_EINVAL;
    if (ws_bytes < p.total) return SD_EINVAL;
    CUtensorMap tmk, tmv;
    if (!cache_map(&tmk, k_cache, D, L + M, S_max, H_kv) || !cache_map(&tmv, v_cache, D, L + M, S_max, H_kv))
        return SD_ECUDA;
    int *st = status_ptr();
    if (!st) return SD_ECUDA;
    AttnArgs a = {};
    a.q = q;
    a.kc = static_cast<const __half *>(k_cache);
    a.vc = static_cast<const __half *>(v_cache);
    a.parent = parent;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.part_ml = reinterpret_cast<float *>(ws);
    a.part_o = reinterpret_cast<float *>(ws + p.off_o);
    a.out = out;
    a.S_max = S_max;
    a.L = L;
    a.NK = L + M;
    a.chunk_pairs = p.chunk_pairs;
    a.M = M;
    a.H = H;
    a.H_kv = H_kv;
    a.g = H / H_kv;
    a.QG = p.QG;
    a.S = p.S;
    a.qscale = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    a.status = st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const dim3 grid(p.S, p.QG, H_kv);
    cudaError_t e;
    if (p.CL) {
        e = D == 128 ? attn_cluster_launch(attn_tc_kernel<128, AT_CL>, grid, AtLayout<128>::TOTAL, s, a, tmk, tmv)
                     : attn_cluster_launch(attn_tc_kernel<64, AT_CL>, grid, AtLayout<64>::TOTAL, s, a, tmk, tmv);
    } else if (D == 128) {
        e = allow_max_dynamic_smem(attn_tc_kernel<128, 0>);
        if (e == cudaSuccess)
            e = launch(attn_tc_kernel<128, 0>, grid, dim3(32 * (AT_CW + 1)), AtLayout<128>::TOTAL, s, a, tmk, tmv);
        if (e == cudaSuccess) e = launch(attn_combine_kernel<128>, dim3(p.QG, H_kv), dim3(32 * AT_TQ), 0, s, a);
    } else {
        e = allow_max_dynamic_smem(attn_tc_kernel<64, 0>);
        if (e == cudaSuccess)
            e = launch(attn_tc_kernel<64, 0>, grid, dim3(32 * (AT_CW + 1)), AtLayout<64>::TOTAL, s, a, tmk, tmv);
        if (e == cudaSuccess) e = launch(attn_combine_kernel<64>, dim3(p.QG, H_kv), dim3(32 * AT_TQ), 0, s, a);
    }
    return e == cudaSuccess ? SD_OK : SD_ECUDA;
}

sd_status sd_kv_commit(void *k_cache, void *v_cache, int32_t H_kv, int32_t D, int64_t S_max, int64_t L, int32_t M,
                       const int32_t *path, const int32_t *count, sd_stream_t stream) {
    SD_NVTX("sd_kv_commit");
    if (!k_cache || !v_cache || !count) return SD_EINVAL;
    if (H_kv < 1 || D < 1 || D > KC_MAXD || M < 1 || M > 16 || L < 0 || S_max < L + M) return SD_EINVAL;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return SD_EINVAL;
    if (!path) return SD_OK;  // a chain keeps its first n rows where they are
    int *st = status_ptr();
    if (!st) return SD_ECUDA;
    return launch(kv_commit_kernel, dim3(H_kv), dim3(128), 0, reinterpret_cast<cudaStream_t>(stream),
                  static_cast<__half *>(k_cache), static_cast<__half *>(v_cache), D, S_max, L, M, path, count, st) ==
                   cudaSuccess
               ? SD_OK
               : SD_ECUDA;
}

}  // extern "C"
