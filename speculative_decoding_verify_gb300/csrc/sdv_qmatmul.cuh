// sdv_qmatmul.cuh - multi-position quantised matmul (one weight read serves
// all M verify positions), with the requantising, SiLU*mul and head epilogues.
//
// Work decomposition ("stream-K"): the weights of a matrix are 32-row tiles
// (or gate|up tile pairs) x k-blocks.  The k range is cut into KS splits of at
// most 80 blocks so the activations of one split fit in shared memory.  Steps
// (one record of 32 rows x 32 weights, or a gate|up pair of records) are
// ordered (split, unit, block) and every CTA of a grid of min(#SMs, steps)
// CTAs takes one contiguous, equal share.  A unit whose steps all fall in one
// CTA is finished directly; otherwise each CTA writes its partial sums to the
// workspace and the last one to arrive adds them in (split, piece) order.
// All of this depends on (n_out, k_in, SM count) only, never on M, which
// makes every output row bit-identical whatever the number of positions.
//
// Inside a CTA: warp 8 (one elected lane) streams records with TMA bulk copies
// into a ring of shared-memory stages guarded by mbarriers; warps 0..7 consume
// them.  Each record's exact int32 block dots come from mma.sync m16n8k16
// (f16 operands, f32 accumulate): the weight codes enter as the fp16 values
// 1024 + code (4-bit, one LOP3 per two values; codes in bits 4..7 of a byte
// enter as 1024 + 16 code against activations pre-divided by 16) or 1152 + q
// (Q8_0, one PRMT per two values), activations as exact fp16 integers, and the
// accumulator starts at minus the offsets' contribution, so it ends at the
// exact integer dot (every partial sum is an integer below 2^23).  Each lane
// then adds d_w * d_a * dot for its 8 (row, position) results.  The 8 warps'
// partials are added in warp order at the end of each piece.
#pragma once

#include "sdv_common.cuh"

namespace sdv {

constexpr int NCW = 8;                 // consumer warps
constexpr int QMM_THREADS = (NCW + 1) * 32;
constexpr int KB_SPLIT_MAX = 80;       // blocks per k-split
constexpr int MPAD = 16;               // position stride of workspace partials
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s bound on any in-kernel wait
constexpr int STAT_TILE = 1024;        // vocabulary tile of the softmax statistics

struct QmmArgs {
    const uint8_t *w;
    int64_t n_out;       // output columns (2F for a gate|up pair)
    int32_t KB;          // k blocks
    int32_t NU;          // units: 32-row tiles, or gate|up tile pairs
    int32_t KS, KBs, KBlast;
    int64_t W;           // total steps
    int32_t G;           // CTAs
    int32_t P;           // max pieces per (unit, split)
    int32_t SB;          // steps per stage
    int32_t NS;          // stages
    uint32_t step_bytes; // bytes of one step
    const int8_t *q;
    const float *sc;
    int32_t M;
    float *y;
    const float *residual;
    uint32_t epi;
    int64_t col0;
    int8_t *q_next;
    float *s_next;
    int64_t nq;          // row width of q_next
    float *part;         // workspace partials [NU][KS][P][rows][MPAD]
    uint32_t *cnt;       // workspace counters [NU]
    // head statistics
    int head;
    float T;
    int32_t *argmax;
    float *row_max;
    float *row_sumexp;
    float4 *st_part;     // [n_stiles][MPAD]
    uint32_t *st_cnt;    // [n_stiles]
    uint32_t *st_done;   // [1]
    int32_t n_stiles;
    int *status;
    uint32_t off_ring, off_act, off_meta, off_red;
};

__device__ __forceinline__ void decode_step(const QmmArgs &a, int64_t g, int &s, int &u, int &j, int &len) {
    int64_t per = static_cast<int64_t>(a.NU) * a.KBs;
    int64_t ss = g / per;
    if (ss > a.KS - 1) ss = a.KS - 1;
    s = static_cast<int>(ss);
    int64_t rem = g - per * ss;
    len = (s == a.KS - 1) ? a.KBlast : a.KBs;
    u = static_cast<int>(rem / len);
    j = static_cast<int>(rem - static_cast<int64_t>(u) * len);
}

__device__ __forceinline__ int64_t unit_start(const QmmArgs &a, int s, int u) {
    int len = (s == a.KS - 1) ? a.KBlast : a.KBs;
    return static_cast<int64_t>(a.NU) * a.KBs * s + static_cast<int64_t>(u) * len;
}

// CTA owning step x: largest c with floor(c W / G) <= x
__device__ __forceinline__ int owner_of(const QmmArgs &a, int64_t x) {
    return static_cast<int>(((x + 1) * a.G - 1) / a.W);
}

__device__ __forceinline__ int npieces(const QmmArgs &a, int s, int u) {
    int len = (s == a.KS - 1) ? a.KBlast : a.KBs;
    int64_t st = unit_start(a, s, u);
    return owner_of(a, st + len - 1) - owner_of(a, st) + 1;
}

// ---------------------------------------------------------------------------
// record layout and exact block dots on the tensor cores
//
// Lane l = 4g + c of a warp owns, for a 32-row x 32-weight record, the A
// fragments of mma m16n8k16 for row tiles t = 0, 1 (rows 16t + g, 16t + g + 8)
// and k steps s = 0, 1 (k = 16s + 2c, +1 and 16s + 2c + 8, +9).
//  4-bit: 16 code bytes per lane, word j = 2t + s; nibble i of the word holds
//    i=0,4: (row 16t+g,   k 16s+2c, +1)   i=2,6: (row 16t+g+8, k 16s+2c, +1)
//    i=1,5: (row 16t+g,   k 16s+2c+8, +9) i=3,7: (row 16t+g+8, k 16s+2c+8, +9)
//  Q8_0: 32 code bytes per lane in two 16-byte planes (words 0..3 for t = 0,
//    words 4..7 for t = 1); word 2(2t+s)+h holds bytes (row 16t+g, k0), (row
//    16t+g, k0+1), (row 16t+g+8, k0), (row 16t+g+8, k0+1) with k0 = 16s+2c+8h.
//  Scales: 8 groups of 4 fp16, group g = rows g, g+8, 16+g, 24+g.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mma_init(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, float c0,
                                         float c1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%10,%11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ void mma_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 4-bit codes of one lane -> fp16 pairs (1024 + code, or 1024 + 16 code in the k+8 halves)
__device__ __forceinline__ void q4_frag(uint4 w, uint32_t (&a)[2][2][4]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t x = ws[j], y = x >> 8;
        a[j >> 1][j & 1][0] = (x & 0x000F000Fu) | 0x64006400u;
        a[j >> 1][j & 1][1] = (y & 0x000F000Fu) | 0x64006400u;
        a[j >> 1][j & 1][2] = (x & 0x00F000F0u) | 0x64006400u;
        a[j >> 1][j & 1][3] = (y & 0x00F000F0u) | 0x64006400u;
    }
}

// Q8_0 codes of one lane -> fp16 pairs 1152 + q (offset binary in the mantissa)
__device__ __forceinline__ void q8_frag(uint4 p0, uint4 p1, uint32_t (&a)[2][2][4]) {
    const uint32_t ws[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t x = ws[w] ^ 0x80808080u;
        const int ts = w >> 1, h = w & 1;
        a[ts >> 1][ts & 1][2 * h] = __byte_perm(x, 0x64646464u, 0x5140);
        a[ts >> 1][ts & 1][2 * h + 1] = __byte_perm(x, 0x64646464u, 0x7362);
    }
}

// the two row tiles' exact dots of one record against one 8-position tile:
// d[t][i] = dot(row 16t + g + 8(i>>1), position 2c + (i&1))
__device__ __forceinline__ void record_dots(const uint32_t (&a)[2][2][4], uint4 bf, float2 corr, float (&d)[2][4]) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        mma_init(d[t], a[t][0], bf.x, bf.y, corr.x, corr.y);
        mma_acc(d[t], a[t][1], bf.z, bf.w);
    }
}

// B fragment of one lane for one block and 8-position tile: fp16 activations
// at (position n = g, k = 16s + 2c, +1, 16s + 2c + 8, +9), the k+8 halves
// divided by 16 for the 4-bit format.  `arow` = the position's 32 int8 values
// (nullptr: a padding position).
template <int QT>
__device__ __forceinline__ uint4 b_frag(const int8_t *arow, int c) {
    if (!arow) return make_uint4(0u, 0u, 0u, 0u);
    uint32_t r[4];
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = 16 * s + 2 * c + 8 * h;
            const float sc = (QT == SD_Q4_32 && h == 1) ? 0.0625f : 1.0f;
            const __half lo = __float2half_rn(static_cast<float>(arow[k]) * sc);
            const __half hi = __float2half_rn(static_cast<float>(arow[k + 1]) * sc);
            r[2 * s + h] = static_cast<uint32_t>(__half_as_ushort(lo)) |
                           (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
        }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// accumulator start removing the code offsets: 4-bit -(1032 S_lo + 72 S_hi)
// with S_lo / S_hi the sums of the activations at k % 16 < 8 / >= 8; Q8_0
// -1152 S.  Exact integers (|.| < 2^23).
template <int QT>
__device__ __forceinline__ float dot_corr(const int8_t *arow) {
    if (!arow) return 0.0f;
    const uint4 *p = reinterpret_cast<const uint4 *>(arow);
    const uint4 x0 = p[0], x1 = p[1];
    int lo = 0, hi = 0;
    lo = dp4a(0x01010101, static_cast<int>(x0.x), lo);
    lo = dp4a(0x01010101, static_cast<int>(x0.y), lo);
    hi = dp4a(0x01010101, static_cast<int>(x0.z), hi);
    hi = dp4a(0x01010101, static_cast<int>(x0.w), hi);
    lo = dp4a(0x01010101, static_cast<int>(x1.x), lo);
    lo = dp4a(0x01010101, static_cast<int>(x1.y), lo);
    hi = dp4a(0x01010101, static_cast<int>(x1.z), hi);
    hi = dp4a(0x01010101, static_cast<int>(x1.w), hi);
    const int v = QT == SD_Q4_32 ? -(1032 * lo + 72 * hi) : -1152 * (lo + hi);
    return static_cast<float>(v);
}

// ---------------------------------------------------------------------------
// epilogue of one finished (unit, position): lane = row
// ---------------------------------------------------------------------------
template <int PAIR>
__device__ __forceinline__ void epilogue(const QmmArgs &a, int u, int m, int lane, float v, float vu) {
    if (PAIR) {
        const int64_t F = a.n_out / 2;
        const int64_t n = static_cast<int64_t>(u) * 32 + lane;  // F % 32 == 0 is required
        if (a.y) {
            a.y[m * a.n_out + n] = v;
            a.y[m * a.n_out + F + n] = vu;
        }
        float h = silu_mul(v, vu);
        float d;
        int code = requant_lane(h, d);
        a.q_next[m * a.nq + n] = static_cast<int8_t>(code);
        if (lane == 0) a.s_next[m * (a.nq / 32) + u] = d;
    } else {
        const int64_t n = static_cast<int64_t>(u) * 32 + lane;
        const bool ok = n < a.n_out;
        if (ok && a.residual) v = __fadd_rn(v, a.residual[m * a.n_out + n]);
        if (ok && a.y) a.y[m * a.n_out + n] = v;
        if (a.epi == SD_EPI_REQUANT && static_cast<int64_t>(u) * 32 >= a.col0) {
            float d;
            int code = requant_lane(ok ? v : 0.0f, d);  // n_out % 32 == 0 is required here
            const int64_t c = n - a.col0;
            if (ok) a.q_next[m * a.nq + c] = static_cast<int8_t>(code);
            if (lane == 0) a.s_next[m * (a.nq / 32) + c / 32] = d;
        }
    }
}

// Softmax statistics of one finished 1024-token tile st, then (last tile) the
// per-row fold.  Called by all consumer threads after the tile's logits are
// globally visible.  Warp w handles positions w, w+8, ...
__device__ inline void head_tile_stats(const QmmArgs &a, int st, int lane, int warp) {
    const int64_t V = a.n_out;
    for (int m = warp; m < a.M; m += NCW) {
        float v[32];
        float zmax = -__int_as_float(0x7f800000);
        float bl = -__int_as_float(0x7f800000);
        int bi = 0x7fffffff;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            int64_t e = static_cast<int64_t>(st) * STAT_TILE + lane + 32 * r;
            float z = -__int_as_float(0x7f800000);
            if (e < V) {
                float l = __ldcg(a.y + m * V + e);
                if (l > bl) {
                    bl = l;
                    bi = static_cast<int>(e);
                }
                z = __fdiv_rn(l, a.T);
                zmax = fmaxf(zmax, z);
            }
            v[r] = z;
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
            float ol = __shfl_xor_sync(0xffffffffu, bl, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ol > bl || (ol == bl && oi < bi)) {
                bl = ol;
                bi = oi;
            }
        }
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            int64_t e = static_cast<int64_t>(st) * STAT_TILE + lane + 32 * r;
            v[r] = e < V ? cexpf_canon(__fsub_rn(v[r], zmax)) : 0.0f;
        }
        float s = tree1024_warp(v);
        if (lane == 0) a.st_part[st * MPAD + m] = make_float4(zmax, s, __int_as_float(bi), bl);
    }
}

__device__ inline void head_final_fold(const QmmArgs &a, int lane, int warp) {
    for (int m = warp; m < a.M; m += NCW) {
        float mx = -__int_as_float(0x7f800000);
        float bl = -__int_as_float(0x7f800000);
        int bi = 0x7fffffff;
        for (int t = lane; t < a.n_stiles; t += 32) {
            float4 p = __ldcg(a.st_part + t * MPAD + m);
            mx = fmaxf(mx, p.x);
            int pi = __float_as_int(p.z);
            if (p.w > bl || (p.w == bl && pi < bi)) {
                bl = p.w;
                bi = pi;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            float ol = __shfl_xor_sync(0xffffffffu, bl, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ol > bl || (ol == bl && oi < bi)) {
                bl = ol;
                bi = oi;
            }
        }
        // Z = sequential fold over tiles of s_t * exp(m_t - m); the products in parallel
        float Z = 0.0f;
        for (int t0 = 0; t0 < a.n_stiles; t0 += 32) {
            int t = t0 + lane;
            float e = 0.0f;
            if (t < a.n_stiles) {
                float4 p = __ldcg(a.st_part + t * MPAD + m);
                e = __fmul_rn(p.y, cexpf_canon(__fsub_rn(p.x, mx)));
            }
            int nn = a.n_stiles - t0 < 32 ? a.n_stiles - t0 : 32;
            for (int j = 0; j < nn; ++j) Z = __fadd_rn(Z, __shfl_sync(0xffffffffu, e, j));
        }
        if (lane == 0) {
            a.argmax[m] = bi;
            a.row_max[m] = mx;
            a.row_sumexp[m] = Z;
        }
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int QT, int PAIR, int NT>
__global__ void __launch_bounds__(QMM_THREADS, 1) qmm_kernel(const QmmArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ int s_flag;
    __shared__ volatile int s_abort;   // set by anyone whose bounded wait ran out
    __shared__ volatile int s_cabort;  // set by consumers only, read after a consumer barrier

    constexpr int REC = QT == SD_Q8_0 ? 1088 : 576;  // bytes of one 32-row record
    constexpr int CODE = QT == SD_Q8_0 ? 1024 : 512; // code bytes of a record
    constexpr int ROWS = PAIR ? 64 : 32;
    constexpr int MT = 8 * NT;  // position slots
    const int M = a.M;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lg = lane >> 2, lc = lane & 3;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + a.NS;
    uint8_t *ring = smem + a.off_ring;
    uint4 *bsm = reinterpret_cast<uint4 *>(smem + a.off_act);     // [block][ntile][lane] B fragments
    float *meta = reinterpret_cast<float *>(smem + a.off_meta);   // [block][ntile][corr 8 | d_a 8]
    float *red = reinterpret_cast<float *>(smem + a.off_red);

    const int64_t lo = static_cast<int64_t>(blockIdx.x) * a.W / a.G;
    const int64_t hi = static_cast<int64_t>(blockIdx.x + 1) * a.W / a.G;

    if (tid == 0) {
        for (int i = 0; i < a.NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NCW);
        }
        s_abort = 0;
        s_cabort = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == NCW) {
        // ------------------------------ producer ------------------------------
        pdl_launch_dependents();
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            uint32_t it = 0;
            int64_t g = lo;
            while (g < hi && !s_abort) {
                int s, u, j0, len;
                decode_step(a, g, s, u, j0, len);
                int j1 = static_cast<int>(j0 + (hi - g) < len ? j0 + (hi - g) : len);
                for (int jj = j0; jj < j1 && !s_abort; jj += a.SB) {
                    int n = j1 - jj < a.SB ? j1 - jj : a.SB;
                    int stg = static_cast<int>(it % a.NS);
                    uint32_t ph = (it / a.NS) & 1u;
                    if (!mbar_wait_bounded(&empty[stg], ph ^ 1u, WAIT_NS, &s_abort)) {
                        set_status(a.status, SD_ETIMEOUT);
                        s_abort = 1;
                        break;
                    }
                    uint32_t bytes = static_cast<uint32_t>(n) * a.step_bytes;
                    const uint8_t *src = a.w + (static_cast<int64_t>(u) * a.KB + static_cast<int64_t>(s) * a.KBs + jj) *
                                                   a.step_bytes;
                    mbar_arrive_expect_tx(&full[stg], bytes);
                    bulk_g2s(ring + static_cast<size_t>(stg) * a.SB * a.step_bytes, src, bytes, &full[stg], pol);
                    ++it;
                }
                g += j1 - j0;
            }
            // never leave with copies in flight: wait for the last issued stages
            uint32_t first = it > static_cast<uint32_t>(a.NS) ? it - a.NS : 0u;
            for (uint32_t k = first; k < it; ++k)
                mbar_wait_bounded(&full[k % a.NS], (k / a.NS) & 1u, WAIT_NS);
        }
        return;
    }

    // ------------------------------ consumers ------------------------------
    pdl_wait();
    pdl_launch_dependents();

    uint32_t it = 0;
    int cur_s = -1;
    int64_t g = lo;
    while (g < hi) {
        int s, u, j0, len;
        decode_step(a, g, s, u, j0, len);
        const int j1 = static_cast<int>(j0 + (hi - g) < len ? j0 + (hi - g) : len);

        if (s != cur_s) {
            // stage this split's activations as B fragments + per-(block, position) {corr, d_a}
            named_bar_sync(1, NCW * 32);
            const int64_t K = static_cast<int64_t>(a.KB) * 32;
            const int b0 = s * a.KBs;
            for (int c = tid; c < len * NT * 32; c += NCW * 32) {
                const int jb = c / (NT * 32), rem = c - jb * (NT * 32), nt = rem >> 5, l = rem & 31;
                const int n = nt * 8 + (l >> 2);
                const int8_t *arow = n < M ? a.q + n * K + static_cast<int64_t>(b0 + jb) * 32 : nullptr;
                bsm[(jb * NT + nt) * 32 + l] = b_frag<QT>(arow, l & 3);
            }
            for (int c = tid; c < len * MT; c += NCW * 32) {
                const int jb = c / MT, n = c - jb * MT, nt = n >> 3, p = n & 7;
                const int8_t *arow = n < M ? a.q + n * K + static_cast<int64_t>(b0 + jb) * 32 : nullptr;
                float *mp = meta + (jb * NT + nt) * 16;
                mp[p] = dot_corr<QT>(arow);
                mp[8 + p] = n < M ? a.sc[static_cast<int64_t>(n) * a.KB + b0 + jb] : 0.0f;
            }
            named_bar_sync(1, NCW * 32);
            cur_s = s;
        }

        // acc[nt][t][i]: row 16t + lg + 8(i>>1), position 8nt + 2lc + (i&1); accu: the up rows
        float acc[NT][2][4], accu[PAIR ? NT : 1][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[nt][t][i] = 0.0f;
                    if (PAIR) accu[PAIR ? nt : 0][t][i] = 0.0f;
                }

        bool aborted = false;
        for (int jj = j0; jj < j1; jj += a.SB) {
            const int n = j1 - jj < a.SB ? j1 - jj : a.SB;
            const int stg = static_cast<int>(it % a.NS);
            const uint32_t ph = (it / a.NS) & 1u;
            if (!mbar_wait_bounded(&full[stg], ph, WAIT_NS, &s_abort)) {
                set_status(a.status, SD_ETIMEOUT);
                s_abort = 1;
                aborted = true;
                break;
            }
            const uint8_t *sbase = ring + static_cast<size_t>(stg) * a.SB * a.step_bytes;
            for (int r = warp; r < n; r += NCW) {
                const uint8_t *rec = sbase + static_cast<size_t>(r) * a.step_bytes;
                const int jb = jj + r;
#pragma unroll
                for (int half = 0; half < (PAIR ? 2 : 1); ++half) {
                    const uint8_t *rh = rec + half * REC;
                    uint32_t af[2][2][4];
                    if (QT == SD_Q4_32) {
                        q4_frag(*reinterpret_cast<const uint4 *>(rh + lane * 16), af);
                    } else {
                        q8_frag(*reinterpret_cast<const uint4 *>(rh + lane * 16),
                                *reinterpret_cast<const uint4 *>(rh + 512 + lane * 16), af);
                    }
                    const uint2 sw = *reinterpret_cast<const uint2 *>(rh + CODE + lg * 8);
                    const float2 dw0 = __half22float2(*reinterpret_cast<const __half2 *>(&sw.x));  // rows g, g+8
                    const float2 dw1 = __half22float2(*reinterpret_cast<const __half2 *>(&sw.y));  // rows 16+g, 24+g
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        if (NT == 1 || nt * 8 < M) {
                            const uint4 bf = bsm[(jb * NT + nt) * 32 + lane];
                            const float *mp = meta + (jb * NT + nt) * 16;
                            const float2 corr = *reinterpret_cast<const float2 *>(mp + 2 * lc);
                            const float2 da = *reinterpret_cast<const float2 *>(mp + 8 + 2 * lc);
                            float d[2][4];
                            record_dots(af, bf, corr, d);
                            float (&ac)[2][4] = half ? accu[PAIR ? nt : 0] : acc[nt];
                            const float wr[2][2] = {{dw0.x, dw0.y}, {dw1.x, dw1.y}};
#pragma unroll
                            for (int t = 0; t < 2; ++t)
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    ac[t][i] = __fmaf_rn(d[t][i], __fmul_rn(wr[t][i >> 1], (i & 1) ? da.y : da.x),
                                                         ac[t][i]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stg]);
            ++it;
        }

        // ---- finish the piece: add the 8 warps' partials in warp order ----
        if (aborted) s_cabort = 1;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int m = nt * 8 + 2 * lc + (i & 1), row = 16 * t + lg + 8 * (i >> 1);
                    red[(warp * MT + m) * ROWS + row] = acc[nt][t][i];
                    if (PAIR) red[(warp * MT + m) * ROWS + 32 + row] = accu[PAIR ? nt : 0][t][i];
                }
        named_bar_sync(1, NCW * 32);
        if (s_cabort) return;  // uniform: written only before the barrier above

        const bool direct = (a.KS == 1) && (npieces(a, s, u) == 1);
        bool finish = direct;
        if (!direct) {
            const int piece = static_cast<int>(blockIdx.x) - owner_of(a, unit_start(a, s, u));
            float *pp = a.part + ((static_cast<int64_t>(u) * a.KS + s) * a.P + piece) * (ROWS * MPAD);
            for (int m = warp; m < M; m += NCW) {
                float v = red[(0 * MT + m) * ROWS + lane];
                float vu = PAIR ? red[(0 * MT + m) * ROWS + 32 + lane] : 0.0f;
#pragma unroll
                for (int w2 = 1; w2 < NCW; ++w2) {
                    v = __fadd_rn(v, red[(w2 * MT + m) * ROWS + lane]);
                    if (PAIR) vu = __fadd_rn(vu, red[(w2 * MT + m) * ROWS + 32 + lane]);
                }
                pp[m * ROWS + lane] = v;
                if (PAIR) pp[m * ROWS + 32 + lane] = vu;
            }
            __threadfence();
            named_bar_sync(1, NCW * 32);
            if (tid == 0) {
                int expected = 0;
                for (int s2 = 0; s2 < a.KS; ++s2) expected += npieces(a, s2, u);
                __threadfence();
                unsigned old = atomicAdd(&a.cnt[u], 1u);
                s_flag = (static_cast<int>(old) == expected - 1) ? 1 : 0;
            }
            named_bar_sync(1, NCW * 32);
            finish = s_flag != 0;
            if (finish) __threadfence();
        }

        if (finish) {
            for (int m = warp; m < M; m += NCW) {
                float v, vu = 0.0f;
                if (direct) {
                    v = red[(0 * MT + m) * ROWS + lane];
                    if (PAIR) vu = red[(0 * MT + m) * ROWS + 32 + lane];
#pragma unroll
                    for (int w2 = 1; w2 < NCW; ++w2) {
                        v = __fadd_rn(v, red[(w2 * MT + m) * ROWS + lane]);
                        if (PAIR) vu = __fadd_rn(vu, red[(w2 * MT + m) * ROWS + 32 + lane]);
                    }
                } else {
                    v = 0.0f;
                    bool first = true;
                    for (int s2 = 0; s2 < a.KS; ++s2) {
                        const int np = npieces(a, s2, u);
                        for (int p2 = 0; p2 < np; ++p2) {
                            const float *pp = a.part + ((static_cast<int64_t>(u) * a.KS + s2) * a.P + p2) * (ROWS * MPAD);
                            float x = __ldcg(pp + m * ROWS + lane);
                            float xu = PAIR ? __ldcg(pp + m * ROWS + 32 + lane) : 0.0f;
                            if (first) {
                                v = x;
                                vu = xu;
                                first = false;
                            } else {
                                v = __fadd_rn(v, x);
                                if (PAIR) vu = __fadd_rn(vu, xu);
                            }
                        }
                    }
                }
                epilogue<PAIR>(a, u, m, lane, v, vu);
            }
            if (!direct && tid == 0) a.cnt[u] = 0u;

            if (a.head) {
                __threadfence();
                named_bar_sync(1, NCW * 32);
                const int st = u / (STAT_TILE / 32);
                if (tid == 0) {
                    const int tiles_in_st = (a.NU - st * (STAT_TILE / 32)) < (STAT_TILE / 32)
                                                ? (a.NU - st * (STAT_TILE / 32))
                                                : (STAT_TILE / 32);
                    __threadfence();
                    unsigned old = atomicAdd(&a.st_cnt[st], 1u);
                    s_flag = (static_cast<int>(old) == tiles_in_st - 1) ? 1 : 0;
                }
                named_bar_sync(1, NCW * 32);
                if (s_flag) {
                    __threadfence();
                    head_tile_stats(a, st, lane, warp);
                    __threadfence();
                    named_bar_sync(1, NCW * 32);
                    if (tid == 0) {
                        a.st_cnt[st] = 0u;
                        __threadfence();
                        unsigned old = atomicAdd(a.st_done, 1u);
                        s_flag = (static_cast<int>(old) == a.n_stiles - 1) ? 1 : 0;
                    }
                    named_bar_sync(1, NCW * 32);
                    if (s_flag) {
                        __threadfence();
                        head_final_fold(a, lane, warp);
                        if (tid == 0) *a.st_done = 0u;
                    }
                }
            }
        }
        named_bar_sync(1, NCW * 32);  // red[] and s_flag are reused by the next piece
        g += j1 - j0;
    }
}

// ---------------------------------------------------------------------------
// host side: plan + launch
// ---------------------------------------------------------------------------
struct QmmPlan {
    int32_t KB, NU, KS, KBs, KBlast, G, P, SB, NS;
    int64_t W;
    uint32_t step_bytes;
    size_t ws_part, ws_cnt, ws_stats, ws_total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool make_plan(int qtype, int64_t n_out, int64_t k_in, bool pair, bool head, int sms, QmmPlan &p) {
    if (k_in <= 0 || k_in % 32 || n_out <= 0) return false;
    const int rec = qtype == SD_Q8_0 ? 1088 : 576;
    p.KB = static_cast<int32_t>(k_in / 32);
    if (pair) {
        if (n_out % 64) return false;
        p.NU = static_cast<int32_t>(n_out / 64);
    } else {
        p.NU = static_cast<int32_t>((n_out + 31) / 32);
    }
    p.KS = (p.KB + KB_SPLIT_MAX - 1) / KB_SPLIT_MAX;
    p.KBs = (p.KB + p.KS - 1) / p.KS;
    p.KBlast = p.KB - p.KBs * (p.KS - 1);
    p.W = static_cast<int64_t>(p.NU) * (static_cast<int64_t>(p.KBs) * (p.KS - 1) + p.KBlast);
    p.G = static_cast<int32_t>(p.W < sms ? p.W : sms);
    const int64_t qmin = p.W / p.G;
    int64_t P = (static_cast<int64_t>(p.KBs) - 1) / qmin + 2;
    if (P > p.KBs) P = p.KBs;
    p.P = static_cast<int32_t>(P);
    p.step_bytes = static_cast<uint32_t>(rec * (pair ? 2 : 1));
    p.SB = 0;
    p.NS = 0;
    const int rows = pair ? 64 : 32;
    p.ws_part = align_up(static_cast<size_t>(p.NU) * p.KS * p.P * rows * MPAD * sizeof(float), 256);
    p.ws_cnt = align_up(static_cast<size_t>(p.NU) * sizeof(uint32_t), 256);
    const int64_t nst = (n_out + STAT_TILE - 1) / STAT_TILE;
    p.ws_stats = head ? align_up(static_cast<size_t>(nst) * MPAD * sizeof(float4), 256) +
                            align_up(static_cast<size_t>(nst + 1) * sizeof(uint32_t), 256)
                      : 0;
    p.ws_total = p.ws_part + p.ws_cnt + p.ws_stats;
    return true;
}

// shared-memory layout for NT 8-position tiles; returns total bytes
inline size_t plan_smem(QmmPlan &p, int NT, bool pair, uint32_t &off_ring, uint32_t &off_act, uint32_t &off_meta,
                        uint32_t &off_red) {
    const int rows = pair ? 64 : 32;
    p.SB = p.step_bytes >= 1000 ? NCW : 2 * NCW;  // ~9 KB stages
    const size_t stage = static_cast<size_t>(p.SB) * p.step_bytes;
    const size_t act = static_cast<size_t>(p.KBs) * NT * 512;   // B fragments
    const size_t meta = static_cast<size_t>(p.KBs) * NT * 64;   // corr + d_a per position
    const size_t red = static_cast<size_t>(NCW) * 8 * NT * rows * 4;
    const size_t fixed = 256 + act + meta + red;
    size_t ring = 72 * 1024;
    if (fixed + ring > 220 * 1024) ring = fixed + 2 * stage < 220 * 1024 ? 220 * 1024 - fixed : 2 * stage;
    int ns = static_cast<int>(ring / stage);
    if (ns > 12) ns = 12;
    if (ns < 2) ns = 2;
    p.NS = ns;
    off_ring = 256;
    off_act = static_cast<uint32_t>(align_up(off_ring + ns * stage, 128));
    off_meta = static_cast<uint32_t>(align_up(off_act + act, 16));
    off_red = static_cast<uint32_t>(align_up(off_meta + meta, 16));
    return align_up(off_red + red, 128);
}

template <int QT, int PAIR, int NT>
cudaError_t qmm_launch(QmmArgs a, size_t smem, cudaStream_t s) {
    auto k = qmm_kernel<QT, PAIR, NT>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch(k, dim3(a.G), dim3(QMM_THREADS), smem, s, a);
}

// dispatch on M: one 8-position tile for M <= 8, two above
template <int QT, int PAIR>
cudaError_t qmm_dispatch(QmmArgs a, QmmPlan &p, cudaStream_t s);

}  // namespace sdv
