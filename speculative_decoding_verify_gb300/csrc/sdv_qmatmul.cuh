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
constexpr uint64_t WAIT_NS = 2000000000ull;   // 2 s bound on any in-kernel wait
constexpr uint64_t KERNEL_NS = 10000000000ull;  // 10 s bound on any launch's loops (self-check)
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
    uint32_t stage_stride;  // bytes between ring slots (>= SB * step_bytes)
    // phase kind inside a pass: 0 matmul (qt, pair), 1 RMSNorm + requant, 2 greedy acceptance
    int32_t kind, qt, pair;
    const float *xin;       // RMSNorm input [M][K] (K = 32 KB)
    const float *norm_w;    // RMSNorm weight [K]
    float eps;
    const int32_t *tokens;  // acceptance inputs / outputs
    const int32_t *parent;
    int32_t *out_tokens;
    int32_t *out_count;
};

constexpr int KIND_MATMUL = 0, KIND_NORM = 1, KIND_ACCEPT = 2;

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
    const unsigned *w = reinterpret_cast<const unsigned *>(arow);
    const int sh = 16 * (c & 1), j = c >> 1;
    const uint32_t p0 = (__ldcg(w + j) >> sh) & 0xFFFFu, p1 = (__ldcg(w + 2 + j) >> sh) & 0xFFFFu;
    const uint32_t p2 = (__ldcg(w + 4 + j) >> sh) & 0xFFFFu, p3 = (__ldcg(w + 6 + j) >> sh) & 0xFFFFu;
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
    const uint4 x0 = __ldcg(p), x1 = __ldcg(p + 1);
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
        if (ok && a.residual) v = __fadd_rn(v, __ldcg(a.residual + m * a.n_out + n));
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
// consumer threads with the same arguments (barriers inside); the finished logits were written
// before the call.
__device__ __forceinline__ void head_flush(const QmmArgs &a, int st, int n_done, int tid, int lane, int warp) {
    if (st < 0 || n_done == 0) return;
    named_bar_sync(1, NCW * 32);  // every thread's logits before thread 0's release
    bool last = false;
    if (tid == 0) {
        const int tiles_in_st = (a.NU - st * (STAT_TILE / 32)) < (STAT_TILE / 32) ? (a.NU - st * (STAT_TILE / 32))
                                                                                   : (STAT_TILE / 32);
        const unsigned old = atom_add_acq_rel(&a.st_cnt[st], static_cast<uint32_t>(n_done));
        last = static_cast<int>(old) + n_done == tiles_in_st;
    }
    if (!bar_any(1, NCW * 32, last)) return;
    head_tile_stats(a, st, lane, warp);
    named_bar_sync(1, NCW * 32);  // the tile's statistics before thread 0's release
    bool fold = false;
    if (tid == 0) {
        a.st_cnt[st] = 0u;
        const unsigned old = atom_add_acq_rel(a.st_done, 1u);
        fold = static_cast<int>(old) == a.n_stiles - 1;
    }
    if (!bar_any(1, NCW * 32, fold)) return;
    head_final_fold(a, lane, warp);
    if (tid == 0) *a.st_done = 0u;
}

// ---------------------------------------------------------------------------
// per-CTA state and shared-memory regions
// ---------------------------------------------------------------------------
// Decisions the consumer threads must take together (abort, "last to arrive", "statistics tile
// complete") travel through bar_any, never through a shared flag.
struct CtaShared {
    volatile int abort;    // set by anyone whose bounded wait ran out; polled by waits
    float inv[16];         // RMSNorm phase: 1 / rms of each row
    uint64_t t0;           // launch start (globaltimer), for the launch-wide time bound
};

// Launch-wide self-check: past KERNEL_NS since the CTA started, record SD_ETIMEOUT and where
// (status[1]: 1 producer, 2 consumer piece loop) and make the caller unwind.
__device__ __forceinline__ bool out_of_time(const CtaShared &cs, int *status, int where) {
    if (gtimer_ns() - cs.t0 <= KERNEL_NS) return false;
    if (status && atomicCAS(status, 0, SD_ETIMEOUT) == 0) status[1] = where;
    return true;
}

struct Smem {
    uint64_t *full, *empty;
    uint8_t *ring;
    uint4 *bsm;   // B operands of the split: fp16 fragments [block][lane] (one position tile)
    uint2 *bsm8;  // ... or raw int8 fragments [block][tile][lane] converted at use (two tiles)
    float *meta;  // [block][tile][corr 8 | d_a 8]
    float *red;   // per-warp partial sums [warp][position][row]; RMSNorm scratch
};

__device__ __forceinline__ Smem smem_regions(uint8_t *smem, const QmmArgs &a) {
    Smem r;
    r.full = reinterpret_cast<uint64_t *>(smem);
    r.empty = r.full + a.NS;
    r.ring = smem + a.off_ring;
    r.bsm = reinterpret_cast<uint4 *>(smem + a.off_act);
    r.bsm8 = reinterpret_cast<uint2 *>(smem + a.off_act);
    r.meta = reinterpret_cast<float *>(smem + a.off_meta);
    r.red = reinterpret_cast<float *>(smem + a.off_red);
    return r;
}

__device__ __forceinline__ void cta_init(const Smem &sm, int NS, CtaShared &cs) {
    for (int i = 0; i < NS; ++i) {
        mbar_init(&sm.full[i], 1);
        mbar_init(&sm.empty[i], NCW);
    }
    cs.abort = 0;
    cs.t0 = gtimer_ns();
    fence_barrier_init();
}

// ---------------------------------------------------------------------------
// producer: stream this CTA's share of one matmul phase through the ring.
// `it` counts stages over the whole launch (slot it % NS, phase parity it / NS).
// ---------------------------------------------------------------------------
__device__ inline void produce_phase(const QmmArgs &a, const Smem &sm, uint32_t &it, CtaShared &cs, uint64_t pol) {
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * a.W / a.G;
    const int64_t hi = static_cast<int64_t>(blockIdx.x + 1) * a.W / a.G;
    int64_t g = lo;
    while (g < hi && !cs.abort) {
        int s, u, j0, len;
        decode_step(a, g, s, u, j0, len);
        const int j1 = static_cast<int>(j0 + (hi - g) < len ? j0 + (hi - g) : len);
        for (int jj = j0; jj < j1 && !cs.abort; jj += a.SB) {
            const int n = j1 - jj < a.SB ? j1 - jj : a.SB;
            const int stg = static_cast<int>(it % a.NS);
            const uint32_t ph = (it / a.NS) & 1u;
            if (out_of_time(cs, a.status, 1)) {
                cs.abort = 1;
                break;
            }
            if (!mbar_wait_bounded(&sm.empty[stg], ph ^ 1u, WAIT_NS, &cs.abort)) {
                set_status(a.status, SD_ETIMEOUT);
                cs.abort = 1;
                break;
            }
            const uint32_t bytes = static_cast<uint32_t>(n) * a.step_bytes;
            const uint8_t *src =
                a.w + (static_cast<int64_t>(u) * a.KB + static_cast<int64_t>(s) * a.KBs + jj) * a.step_bytes;
            mbar_arrive_expect_tx(&sm.full[stg], bytes);
            bulk_g2s(sm.ring + static_cast<size_t>(stg) * a.stage_stride, src, bytes, &sm.full[stg], pol);
            ++it;
        }
        g += j1 - j0;
    }
}

// never leave with copies in flight: wait for the last issued stages
__device__ inline void producer_drain(const Smem &sm, uint32_t it, int NS) {
    const uint32_t first = it > static_cast<uint32_t>(NS) ? it - NS : 0u;
    for (uint32_t k = first; k < it; ++k) mbar_wait_bounded(&sm.full[k % NS], (k / NS) & 1u, WAIT_NS);
}

// ---------------------------------------------------------------------------
// consumers: one matmul phase (staging, stages, piece fixups, epilogues).
// Returns false (the same on every consumer thread) when the phase was abandoned
// after a bounded wait or the launch-wide time bound ran out.
// ---------------------------------------------------------------------------
template <int QT, int PAIR, int NT>
__device__ inline bool consume_phase(const QmmArgs &a, const Smem &sm, uint32_t &it, CtaShared &cs) {
    constexpr int REC = QT == SD_Q8_0 ? 1088 : 576;  // bytes of one 32-row record
    constexpr int CODE = QT == SD_Q8_0 ? 1024 : 512; // code bytes of a record
    constexpr int ROWS = PAIR ? 64 : 32;
    constexpr int MT = 8 * NT;  // position slots
    const int M = a.M;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lg = lane >> 2, lc = lane & 3;
    uint4 *bsm = sm.bsm;
    uint2 *bsm8 = sm.bsm8;
    float *meta = sm.meta;
    float *red = sm.red;

    const int64_t lo = static_cast<int64_t>(blockIdx.x) * a.W / a.G;
    const int64_t hi = static_cast<int64_t>(blockIdx.x + 1) * a.W / a.G;
    int cur_s = -1;
    int st_cur = -1, st_n = 0;  // head: current statistics tile, tiles finished in it (same on all threads)
    int64_t g = lo;
    while (g < hi) {
        // launch-wide self-check: thread 0 decides, the barrier hands the answer to all.  The
        // barrier also ends every use of the previous piece's shared data (stages, red[], B).
        if (bar_any(1, NCW * 32, tid == 0 && out_of_time(cs, a.status, 2))) {
            cs.abort = 1;
            return false;
        }
        int s, u, j0, len;
        decode_step(a, g, s, u, j0, len);
        const int j1 = static_cast<int>(j0 + (hi - g) < len ? j0 + (hi - g) : len);

        if (s != cur_s) {
            // stage this split's activations straight from global memory: B operands (fp16 fragments,
            // or raw int8 for two position tiles) and per-(block, position) {corr, d_a}
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
                mp[8 + p] = real ? __ldcg(a.sc + static_cast<int64_t>(n) * a.KB + b0 + jb) : 0.0f;
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
            const bool ready = mbar_wait_bounded(&sm.full[stg], ph, WAIT_NS, &cs.abort);
            __syncwarp();  // lanes leave the wait one by one; mma.sync below needs the warp converged
            if (!__all_sync(0xffffffffu, ready)) {
                set_status(a.status, SD_ETIMEOUT);
                cs.abort = 1;
                aborted = true;
                break;
            }
            const uint8_t *sbase = sm.ring + static_cast<size_t>(stg) * a.stage_stride;
            // per round each warp takes steps r0 and r0 + NCW (for a gate|up pair, step r0's two halves)
            constexpr int RPW = 2;
            for (int r0 = warp; r0 < n; r0 += (PAIR ? 1 : 2) * NCW) {
                const int r1 = r0 + NCW;
                const int nrec = PAIR ? 2 : (1 + (r1 < n));
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
            if (lane == 0) mbar_arrive(&sm.empty[stg]);
            ++it;
        }

        // ---- finish the piece: add the 8 warps' partials in warp order ----
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
        if (bar_any(1, NCW * 32, aborted)) {
            cs.abort = 1;
            return false;
        }

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
            named_bar_sync(1, NCW * 32);  // the partial sums above happen before thread 0's release
            bool last = false;
            if (tid == 0) {
                int expected = 0;
                for (int s2 = 0; s2 < a.KS; ++s2) expected += npieces(a, s2, u);
                const unsigned old = atom_add_acq_rel(&a.cnt[u], 1u);
                last = static_cast<int>(old) == expected - 1;
            }
            finish = bar_any(1, NCW * 32, last);  // thread 0 acquired with its atomic; reads below bypass L1
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
                if (st != st_cur) {
                    head_flush(a, st_cur, st_n, tid, lane, warp);
                    st_cur = st;
                    st_n = 0;
                }
                ++st_n;
            }
        }
        g += j1 - j0;
    }
    if (a.head) head_flush(a, st_cur, st_n, tid, lane, warp);
    return true;
}

// ---------------------------------------------------------------------------
// consumers: RMSNorm + per-32 requantisation spread over the grid.  Every CTA
// forms the rows' inverse RMS in the canonical order (256 strided partial sums,
// pairwise tree), then requantises its share of the (row, block) items, one
// warp per item -- the same operations as sd_rmsnorm_quant_acts.
// ---------------------------------------------------------------------------
__device__ inline void norm_phase(const QmmArgs &a, const Smem &sm, CtaShared &cs) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int M = a.M;
    const int64_t K = static_cast<int64_t>(a.KB) * 32;
    float *part = sm.red;  // [M][256]
    for (int m = 0; m < M; ++m) {
        const float *xr = a.xin + m * K;
        float s = 0.0f;
        for (int64_t i = tid; i < K; i += 256) {
            const float x = __ldcg(xr + i);
            s = __fadd_rn(s, __fmul_rn(x, x));
        }
        part[m * 256 + tid] = s;
    }
    named_bar_sync(1, NCW * 32);
    for (int stride = 128; stride >= 1; stride >>= 1) {
        if (tid < stride)
            for (int m = 0; m < M; ++m) part[m * 256 + tid] = __fadd_rn(part[m * 256 + tid], part[m * 256 + tid + stride]);
        named_bar_sync(1, NCW * 32);
    }
    if (tid < M) {
        const float mean = __fdiv_rn(part[tid * 256], static_cast<float>(K));
        cs.inv[tid] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.eps)));
    }
    named_bar_sync(1, NCW * 32);
    const int64_t items = static_cast<int64_t>(M) * a.KB;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * items / gridDim.x;
    const int64_t i1 = static_cast<int64_t>(blockIdx.x + 1) * items / gridDim.x;
    for (int64_t it = i0 + warp; it < i1; it += NCW) {
        const int m = static_cast<int>(it / a.KB);
        const int64_t b = it - static_cast<int64_t>(m) * a.KB;
        const float x = __ldcg(a.xin + m * K + b * 32 + lane);
        const float y = __fmul_rn(__fmul_rn(x, cs.inv[m]), a.norm_w[b * 32 + lane]);
        float d;
        const int v = requant_lane(y, d);
        a.q_next[m * K + b * 32 + lane] = static_cast<int8_t>(v);
        if (lane == 0) a.s_next[m * a.KB + b] = d;
    }
}

// greedy acceptance (chain when parent == nullptr, else a tree in BFS order); one thread
__device__ inline void greedy_accept(const int32_t *argmax, const int32_t *tokens, const int32_t *parent, int M,
                                     int32_t *out, int32_t *count) {
    if (!parent) {
        const int K = M - 1;
        int n = 0;
        while (n < K && __ldcg(tokens + n) == __ldcg(argmax + n)) {
            out[n] = tokens[n];
            ++n;
        }
        out[n] = __ldcg(argmax + n);
        *count = n + 1;
        return;
    }
    bool ok[16];
    int depth[16];
    ok[0] = true;
    depth[0] = 0;
    int best = 0;
    for (int i = 1; i < M; ++i) {
        const int p = parent[i];
        ok[i] = false;
        depth[i] = 0;
        if (p < 0 || p >= i) continue;
        depth[i] = depth[p] + 1;
        ok[i] = ok[p] && tokens[i] == __ldcg(argmax + p);
        if (ok[i] && depth[i] > depth[best]) best = i;
    }
    const int d = depth[best];
    for (int i = best, j = d - 1; i != 0; i = parent[i], --j) out[j] = tokens[i];
    out[d] = __ldcg(argmax + best);
    *count = d + 1;
}

// ---------------------------------------------------------------------------
// single-operation kernel (one matmul phase per launch)
// ---------------------------------------------------------------------------
template <int QT, int PAIR, int NT>
__global__ void __launch_bounds__(QMM_THREADS, 1) qmm_kernel(const QmmArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ CtaShared cs;
    const Smem sm = smem_regions(smem, a);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) cta_init(sm, a.NS, cs);
    __syncthreads();
    uint32_t it = 0;
    if (warp == NCW) {
        pdl_launch_dependents();
        if (lane == 0) {
            produce_phase(a, sm, it, cs, policy_evict_first());
            producer_drain(sm, it, a.NS);
        }
        return;
    }
    pdl_wait();
    pdl_launch_dependents();
    (void)consume_phase<QT, PAIR, NT>(a, sm, it, cs);
}

// ---------------------------------------------------------------------------
// persistent verify pass: every phase of the pass in one cooperative launch,
// phases separated by a grid barrier (release / acquire on a global counter,
// bounded wait).  The producer streams weights across phase boundaries.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int NT>
__global__ void __launch_bounds__(QMM_THREADS, 1)
    pass_kernel(const QmmArgs *__restrict__ phases, int n_phases, uint32_t *barrier_ctr) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ CtaShared cs;
    __shared__ QmmArgs sa;  // the current phase, copied from global memory
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const QmmArgs &a0 = phases[0];
    const Smem sm = smem_regions(smem, a0);
    int *status = a0.status;
    if (tid == 0) cta_init(sm, a0.NS, cs);
    __syncthreads();
    uint32_t it = 0;
    if (warp == NCW) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int p = 0; p < n_phases && !cs.abort; ++p)
                if (phases[p].kind == KIND_MATMUL) produce_phase(phases[p], sm, it, cs, pol);
            producer_drain(sm, it, a0.NS);
        }
        return;
    }
    for (int p = 0; p < n_phases; ++p) {
        bool stop = false;
        if (p > 0 && tid == 0) {  // grid barrier: every CTA finished phase p - 1
            const uint32_t target = static_cast<uint32_t>(p) * gridDim.x;
            const uint64_t t0 = gtimer_ns();
            while (ld_acquire(barrier_ctr) < target) {
                if (cs.abort || gtimer_ns() - t0 > WAIT_NS) {
                    set_status(status, SD_ETIMEOUT);
                    stop = true;
                    break;
                }
            }
        }
        {  // copy the phase descriptor into shared memory (constant: may overlap the barrier wait)
            const uint32_t *src = reinterpret_cast<const uint32_t *>(phases + p);
            uint32_t *dst = reinterpret_cast<uint32_t *>(&sa);
            for (int i = tid; i < static_cast<int>(sizeof(QmmArgs) / 4); i += NCW * 32) dst[i] = src[i];
        }
        if (bar_any(1, NCW * 32, stop)) {
            cs.abort = 1;
            return;
        }
        bool ok = true;
        if (sa.kind == KIND_NORM) {
            norm_phase(sa, sm, cs);
        } else if (sa.kind == KIND_ACCEPT) {
            if (blockIdx.x == 0 && tid == 0)
                greedy_accept(sa.argmax, sa.tokens, sa.parent, sa.M, sa.out_tokens, sa.out_count);
        } else if (sa.qt == SD_Q4_32 && sa.pair) {
            ok = consume_phase<SD_Q4_32, 1, NT>(sa, sm, it, cs);
        } else if (sa.qt == SD_Q4_32) {
            ok = consume_phase<SD_Q4_32, 0, NT>(sa, sm, it, cs);
        } else {
            ok = consume_phase<SD_Q8_0, 0, NT>(sa, sm, it, cs);
        }
        if (!ok) return;  // uniform; cs.abort already stops the producer
        named_bar_sync(1, NCW * 32);  // this CTA's writes of phase p before thread 0's release
        if (tid == 0) red_release_add(barrier_ctr, 1u);
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

// steps per stage (~18 KB stages): 32 records of 4-bit, 16 gate|up pairs, 16 Q8_0 records
inline int stage_steps(int qtype, bool pair) { return pair ? 2 * NCW : (qtype == SD_Q8_0 ? 2 * NCW : 4 * NCW); }

// Shared-memory layout for splits of up to `kbs` blocks, NT 8-position tiles, `rows` output
// rows per unit (64 with a gate|up pair) and ring slots of `slot` bytes; returns total bytes.
inline size_t layout_smem(int kbs, int NT, int rows, size_t slot, int &NS, uint32_t &off_ring, uint32_t &off_act,
                          uint32_t &off_meta, uint32_t &off_red) {
    const size_t act = static_cast<size_t>(kbs) * (NT == 1 ? 512 : 2 * 256);  // fp16 or raw int8 fragments
    const size_t meta = static_cast<size_t>(kbs) * NT * 64;                  // corr + d_a per position
    const size_t red = static_cast<size_t>(NCW) * 8 * NT * rows * 4;
    const size_t fixed = 256 + act + meta + red + 3 * 128;
    const size_t budget = 222 * 1024;
    int ns = fixed + 2 * slot <= budget ? static_cast<int>((budget - fixed) / slot) : 2;
    if (ns > 12) ns = 12;
    NS = ns;
    off_ring = 256;
    off_act = static_cast<uint32_t>(align_up(off_ring + ns * slot, 128));
    off_meta = static_cast<uint32_t>(align_up(off_act + act, 128));
    off_red = static_cast<uint32_t>(align_up(off_meta + meta, 128));
    return align_up(off_red + red, 128);
}

// single-operation layout
inline size_t plan_smem(QmmPlan &p, int NT, bool pair, uint32_t &off_ring, uint32_t &off_act, uint32_t &off_meta,
                        uint32_t &off_red, uint32_t &off_tmp) {
    p.SB = stage_steps(p.step_bytes == 1088 ? SD_Q8_0 : SD_Q4_32, pair);
    int ns = 0;
    const size_t total = layout_smem(p.KBs, NT, pair ? 64 : 32, static_cast<size_t>(p.SB) * p.step_bytes, ns, off_ring,
                                     off_act, off_meta, off_red);
    p.NS = ns;
    off_tmp = 0;
    return total;
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
