// sdv_qmatmul.cuh - multi-position quantised matmul (one weight read serves
// all M verify positions), with the requantising, SiLU*mul and head epilogues.
//
// Work decomposition ("stream-K"): the weights of a matrix are 32-row tiles
// (or gate|up tile pairs) x k-blocks.  The k range is cut into KS splits of at
// most 160 blocks so the activations of one split fit in shared memory.  Steps
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

#ifndef SDV_NCW
#define SDV_NCW 8
#endif
constexpr int NCW = SDV_NCW;           // consumer warps
constexpr int QMM_THREADS = (NCW + 1) * 32;
constexpr int KB_SPLIT_MAX = 160;      // blocks per k-split
constexpr int MPAD = 16;               // position stride of workspace partials
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s bound on any in-kernel wait
constexpr int STAT_TILE = 1024;        // vocabulary tile of the softmax statistics
constexpr int WS_UNIT_CNT = 32768;     // workspace counters: units (tiles / tile pairs) per call
constexpr int WS_STAT_CNT = 2048;      // workspace counters: 1024-token statistics tiles
constexpr size_t WS_CNT_BYTES = 160 * 1024;  // >= (WS_UNIT_CNT + WS_STAT_CNT + 1) * 4, 256-aligned

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
    uint32_t off_ring, off_act, off_meta, off_red, off_tmp;
};

// fetch-and-add with release (orders the CTA's prior writes, seen through a bar.sync) and acquire
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

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

// Raw int8 B operand of one lane for one block and 8-position tile: the bytes at
// k = 2c, 2c+1, 2c+8, 2c+9, 16+2c, 17+2c, 24+2c, 25+2c of position g's 32
// activations, as two 32-bit words (pairs in k order).  `arow` nullptr: padding.
__device__ __forceinline__ uint2 b_raw(const int8_t *arow, int c) {
    if (!arow) return make_uint2(0u, 0u);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(arow);
    const int sh = 16 * (c & 1), j = c >> 1;
    const uint32_t p0 = (w[j] >> sh) & 0xFFFFu, p1 = (w[2 + j] >> sh) & 0xFFFFu;
    const uint32_t p2 = (w[4 + j] >> sh) & 0xFFFFu, p3 = (w[6 + j] >> sh) & 0xFFFFu;
    return make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
}

// int8 pair (low 16 bits of x, k order) -> exact fp16 pair; `div16` also scales by 1/16 (exact)
__device__ __forceinline__ uint32_t i8pair_to_h2(uint32_t x, bool div16) {
    const uint32_t u = __byte_perm(x ^ 0x8080u, 0x64646464u, 0x5140);  // (1024 + a + 128) per half
    __half2 h = *reinterpret_cast<const __half2 *>(&u);
    if (div16) h = __hfma2(h, __float2half2_rn(0.0625f), __float2half2_rn(-72.0f));  // (1152 + a)/16 - 72 = a/16
    else h = __hsub2(h, __float2half2_rn(1152.0f));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// fp16 B fragment registers from the raw operand: {s0 k 2c.., s0 k 2c+8.., s1 k 2c.., s1 k 2c+8..};
// the k+8 halves divided by 16 for the 4-bit format
template <int QT>
__device__ __forceinline__ uint4 b_frag_from_raw(uint2 r) {
    const bool d = QT == SD_Q4_32;
    return make_uint4(i8pair_to_h2(r.x, false), i8pair_to_h2(r.x >> 16, d), i8pair_to_h2(r.y, false),
                      i8pair_to_h2(r.y >> 16, d));
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

// Adds `n_done` finished 32-row tiles to statistics tile `st`; the CTA that completes the tile
// computes its statistics, and the CTA that completes the last tile folds them.  Called by all
// consumer threads (bar.sync inside); the finished logits were written before the call.
__device__ __forceinline__ void head_flush(const QmmArgs &a, int st, int n_done, int tid, int lane, int warp,
                                           int &s_flag) {
    if (st < 0 || n_done == 0) return;
    named_bar_sync(1, NCW * 32);
    if (tid == 0) {
        const int tiles_in_st = (a.NU - st * (STAT_TILE / 32)) < (STAT_TILE / 32) ? (a.NU - st * (STAT_TILE / 32))
                                                                                   : (STAT_TILE / 32);
        const unsigned old = atom_add_acq_rel(&a.st_cnt[st], static_cast<uint32_t>(n_done));
        s_flag = (static_cast<int>(old) + n_done == tiles_in_st) ? 1 : 0;
    }
    named_bar_sync(1, NCW * 32);
    if (!s_flag) return;
    head_tile_stats(a, st, lane, warp);
    named_bar_sync(1, NCW * 32);
    if (tid == 0) {
        a.st_cnt[st] = 0u;
        const unsigned old = atom_add_acq_rel(a.st_done, 1u);
        s_flag = (static_cast<int>(old) == a.n_stiles - 1) ? 1 : 0;
    }
    named_bar_sync(1, NCW * 32);
    if (s_flag) {
        head_final_fold(a, lane, warp);
        if (tid == 0) *a.st_done = 0u;
    }
    named_bar_sync(1, NCW * 32);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int QT, int PAIR, int NT>
__global__ void __launch_bounds__(QMM_THREADS, 1) qmm_kernel(const QmmArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ int s_flag;
    __shared__ int s_st_cur, s_st_n;  // head: current statistics tile and tiles finished in it
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
    // B operands of the split: fp16 fragments [block][lane] (one position tile) or raw int8
    // fragments [block][tile][lane] converted at use (two position tiles)
    uint4 *bsm = reinterpret_cast<uint4 *>(smem + a.off_act);
    uint2 *bsm8 = reinterpret_cast<uint2 *>(smem + a.off_act);
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
        s_st_cur = -1;
        s_st_n = 0;
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
            // stage this split's activations straight from global memory: B operands (fp16 fragments,
            // or raw int8 for two position tiles) and per-(block, position) {corr, d_a}
            named_bar_sync(1, NCW * 32);
            const int64_t K = static_cast<int64_t>(a.KB) * 32;
            const int b0 = s * a.KBs;
            const int nitems = len * NT * 32;
            for (int base = tid; base < nitems; base += 4 * NCW * 32) {
                uint2 raw[4];
#pragma unroll
                for (int u4 = 0; u4 < 4; ++u4) {
                    const int c = base + u4 * NCW * 32;
                    raw[u4] = make_uint2(0u, 0u);
                    if (c < nitems) {
                        const int jb = c / (NT * 32), rem = c - jb * (NT * 32), nt = rem >> 5, l = rem & 31;
                        const int n = nt * 8 + (l >> 2);
                        raw[u4] = b_raw(n < M ? a.q + n * K + static_cast<int64_t>(b0 + jb) * 32 : nullptr, l & 3);
                    }
                }
#pragma unroll
                for (int u4 = 0; u4 < 4; ++u4) {
                    const int c = base + u4 * NCW * 32;
                    if (c < nitems) {
                        if (NT == 1) bsm[c] = b_frag_from_raw<QT>(raw[u4]);
                        else bsm8[c] = raw[u4];
                    }
                }
            }
            for (int c = tid; c < len * MT; c += NCW * 32) {
                const int jb = c / MT, n = c - jb * MT, nt = n >> 3, p = n & 7;
                float *mp = meta + (jb * NT + nt) * 16;
                const bool real = n < M;
                mp[p] = dot_corr<QT>(real ? a.q + n * K + static_cast<int64_t>(b0 + jb) * 32 : nullptr);
                mp[8 + p] = real ? a.sc[static_cast<int64_t>(n) * a.KB + b0 + jb] : 0.0f;
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
            // each warp takes steps warp and warp + NCW of the stage; for a gate|up pair the two
            // halves of one step are the two records
            constexpr int RPW = PAIR ? 2 : 2;  // records handled together per warp
            const int r0 = warp, r1 = warp + NCW;
            const int nrec = PAIR ? (r0 < n ? 2 : 0) : ((r0 < n) + (r1 < n));
            if (nrec > 0) {
                const uint8_t *rp[RPW];
                int jbr[RPW];
#pragma unroll
                for (int q = 0; q < RPW; ++q) {
                    if (PAIR) {
                        rp[q] = sbase + static_cast<size_t>(r0) * a.step_bytes + q * REC;
                        jbr[q] = jj + r0;
                    } else {
                        rp[q] = sbase + static_cast<size_t>(q ? r1 : r0) * a.step_bytes;
                        jbr[q] = jj + (q ? r1 : r0);
                    }
                }
                uint32_t af[RPW][2][2][4];
                float2 dwf[RPW][2];
#pragma unroll
                for (int q = 0; q < RPW; ++q) {
                    if (q < nrec) {
                        if (QT == SD_Q4_32) {
                            q4_frag(*reinterpret_cast<const uint4 *>(rp[q] + lane * 16), af[q]);
                        } else {
                            q8_frag(*reinterpret_cast<const uint4 *>(rp[q] + lane * 16),
                                    *reinterpret_cast<const uint4 *>(rp[q] + 512 + lane * 16), af[q]);
                        }
                        const uint2 sw = *reinterpret_cast<const uint2 *>(rp[q] + CODE + lg * 8);
                        dwf[q][0] = __half22float2(*reinterpret_cast<const __half2 *>(&sw.x));  // rows g, g+8
                        dwf[q][1] = __half22float2(*reinterpret_cast<const __half2 *>(&sw.y));  // rows 16+g, 24+g
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if (NT == 1 || nt * 8 < M) {
                        float d[RPW][2][4];
                        float2 da[RPW];
#pragma unroll
                        for (int q = 0; q < RPW; ++q) {
                            if (q < nrec && (q == 0 || !PAIR)) {
                                const int jb = jbr[q];
                                const uint4 bf = NT == 1 ? bsm[jb * 32 + lane]
                                                         : b_frag_from_raw<QT>(bsm8[(jb * NT + nt) * 32 + lane]);
                                const float *mp = meta + (jb * NT + nt) * 16;
                                const float2 corr = *reinterpret_cast<const float2 *>(mp + 2 * lc);
                                da[q] = *reinterpret_cast<const float2 *>(mp + 8 + 2 * lc);
                                record_dots(af[q], bf, corr, d[q]);
                                if (PAIR) {  // the up half shares the step's activations
                                    da[1] = da[0];
                                    record_dots(af[1], bf, corr, d[1]);
                                }
                            }
                        }
#pragma unroll
                        for (int q = 0; q < RPW; ++q) {
                            if (q < nrec) {
                                float (&ac)[2][4] = (PAIR && q == 1) ? accu[PAIR ? nt : 0] : acc[nt];
#pragma unroll
                                for (int t = 0; t < 2; ++t) {
                                    const float w0 = t ? dwf[q][1].x : dwf[q][0].x;
                                    const float w1 = t ? dwf[q][1].y : dwf[q][0].y;
#pragma unroll
                                    for (int i = 0; i < 4; ++i)
                                        ac[t][i] = __fmaf_rn(d[q][t][i], __fmul_rn((i >> 1) ? w1 : w0,
                                                                                   (i & 1) ? da[q].y : da[q].x),
                                                             ac[t][i]);
                                }
                            }
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
            named_bar_sync(1, NCW * 32);  // the partial sums above happen before thread 0's fence
            if (tid == 0) {
                int expected = 0;
                for (int s2 = 0; s2 < a.KS; ++s2) expected += npieces(a, s2, u);
                const unsigned old = atom_add_acq_rel(&a.cnt[u], 1u);
                s_flag = (static_cast<int>(old) == expected - 1) ? 1 : 0;
            }
            named_bar_sync(1, NCW * 32);
            finish = s_flag != 0;  // thread 0 fenced after its atomic; reads below bypass L1
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
                // count finished tiles per 1024-token statistics tile; one counter update per
                // (CTA, statistics tile) run, issued when the run ends
                const int st = u / (STAT_TILE / 32);
                if (st != s_st_cur) {
                    head_flush(a, s_st_cur, s_st_n, tid, lane, warp, s_flag);
                    if (tid == 0) {
                        s_st_cur = st;
                        s_st_n = 0;
                    }
                    named_bar_sync(1, NCW * 32);
                }
                if (tid == 0) s_st_n += 1;
            }
        }
        named_bar_sync(1, NCW * 32);  // red[] and s_flag are reused by the next piece
        g += j1 - j0;
    }
    if (a.head) head_flush(a, s_st_cur, s_st_n, tid, lane, warp, s_flag);
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
    // counters first, at fixed offsets shared by every call: units [0, WS_UNIT_CNT), statistics
    // tiles [WS_UNIT_CNT, WS_UNIT_CNT + WS_STAT_CNT), the statistics "done" counter after them.
    // Each call returns the counters it used to zero, so a workspace can serve calls of any shape.
    if (p.NU > WS_UNIT_CNT) return false;
    const int64_t nst = (n_out + STAT_TILE - 1) / STAT_TILE;
    if (head && nst > WS_STAT_CNT) return false;
    p.ws_cnt = WS_CNT_BYTES;
    p.ws_part = align_up(static_cast<size_t>(p.NU) * p.KS * p.P * rows * MPAD * sizeof(float), 256);
    p.ws_stats = head ? align_up(static_cast<size_t>(nst) * MPAD * sizeof(float4), 256) : 0;
    p.ws_total = p.ws_part + p.ws_cnt + p.ws_stats;
    return true;
}

// shared-memory layout for NT 8-position tiles; returns total bytes
inline size_t plan_smem(QmmPlan &p, int NT, bool pair, uint32_t &off_ring, uint32_t &off_act, uint32_t &off_meta,
                        uint32_t &off_red, uint32_t &off_tmp) {
    const int rows = pair ? 64 : 32;
    p.SB = pair ? NCW : 2 * NCW;  // two records per consumer warp per stage
    const size_t stage = static_cast<size_t>(p.SB) * p.step_bytes;
    const size_t act = static_cast<size_t>(p.KBs) * (NT == 1 ? 512 : 2 * 256);  // fp16 or raw int8 fragments
    const size_t meta = static_cast<size_t>(p.KBs) * NT * 64;   // corr + d_a per position
    const size_t red = static_cast<size_t>(NCW) * 8 * NT * rows * 4;
    const size_t tmp = 0;
    const size_t fixed = 256 + act + meta + red + tmp;
    size_t ring = 96 * 1024;
    if (ring < 4 * stage) ring = 4 * stage;
    if (fixed + ring > 222 * 1024) ring = (222 * 1024 - fixed) / stage * stage;
    if (ring < 2 * stage) ring = 2 * stage;
    int ns = static_cast<int>(ring / stage);
    if (ns > 12) ns = 12;
    if (ns < 2) ns = 2;
    p.NS = ns;
    off_ring = 256;
    off_act = static_cast<uint32_t>(align_up(off_ring + ns * stage, 128));
    off_meta = static_cast<uint32_t>(align_up(off_act + act, 16));
    off_red = static_cast<uint32_t>(align_up(off_meta + meta, 16));
    off_tmp = static_cast<uint32_t>(align_up(off_red + red, 16));
    return align_up(off_tmp + tmp, 128);
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
