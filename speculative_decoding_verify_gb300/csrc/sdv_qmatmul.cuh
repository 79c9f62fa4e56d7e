// sdv_qmatmul.cuh - multi-position quantised matmul (one weight read serves
// all M verify positions), with the requantising, SiLU*mul and head epilogues.
//
// Work decomposition ("stream-K"): the weights of a matrix are 32-row tiles
// (or gate|up tile pairs) x k-blocks.  The k range is cut into KS splits of at
// most 160 blocks so the int8 activations of one split fit in shared memory.
// Steps (one record of 32 rows x 32 weights, or a gate|up pair of records) are
// ordered (split, unit, block) and every CTA of a grid of min(#SMs, steps)
// CTAs takes one contiguous, equal share.  A unit whose steps all fall in one
// CTA is finished directly; otherwise each CTA writes its partial sums to the
// workspace and the last one to arrive adds them in (split, piece) order.
// All of this depends on (n_out, k_in, SM count) only, never on M, which
// makes every output row bit-identical whatever the number of positions.
//
// Inside a CTA: warp 8 (one elected lane) streams records with TMA bulk copies
// into a ring of shared-memory stages guarded by mbarriers; warps 0..7 consume
// them, lane r owning row r of the record.  Per record and position the lane
// forms the exact int32 block dot with dp4a (4-bit: sum code*a - 8 sum a, the
// second term preloaded as the chain's start value together with the 2^23+2^22
// bias that turns the int32 into its fp32 value with one subtraction) and adds
// d_w * d_a * dot to its accumulator.  The 8 warps' partials are added in warp
// order at the end of each piece.
#pragma once

#include "sdv_common.cuh"

namespace sdv {

constexpr int NCW = 8;                 // consumer warps
constexpr int QMM_THREADS = (NCW + 1) * 32;
constexpr int KB_SPLIT_MAX = 160;      // blocks per k-split
constexpr int MPAD = 16;               // position stride of workspace partials
constexpr uint64_t WAIT_NS = 2000000000ull;  // 2 s bound on any in-kernel wait
constexpr int STAT_TILE = 1024;        // vocabulary tile of the softmax statistics
constexpr int FP_BIAS_BITS = 0x4B400000;  // bit pattern of 1.5 * 2^23
constexpr float FP_BIAS = 12582912.0f;

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
// block dots of one record row (lane) against one position's activations
// ---------------------------------------------------------------------------

// 4-bit: w = the lane's 16 code bytes; a0/a1 = activation bytes 0..15 / 16..31;
// init = -8 * sum(a) + bias.  Low nibbles are elements 0..15, high nibbles 16..31.
__device__ __forceinline__ int dot_q4(const uint32_t (&lo)[4], const uint32_t (&hi)[4], uint4 a0, uint4 a1, int init) {
    int d = init;
    d = dp4a(static_cast<int>(lo[0]), static_cast<int>(a0.x), d);
    d = dp4a(static_cast<int>(lo[1]), static_cast<int>(a0.y), d);
    d = dp4a(static_cast<int>(lo[2]), static_cast<int>(a0.z), d);
    d = dp4a(static_cast<int>(lo[3]), static_cast<int>(a0.w), d);
    d = dp4a(static_cast<int>(hi[0]), static_cast<int>(a1.x), d);
    d = dp4a(static_cast<int>(hi[1]), static_cast<int>(a1.y), d);
    d = dp4a(static_cast<int>(hi[2]), static_cast<int>(a1.z), d);
    d = dp4a(static_cast<int>(hi[3]), static_cast<int>(a1.w), d);
    return d;
}

__device__ __forceinline__ void unpack_q4(uint4 c, uint32_t (&lo)[4], uint32_t (&hi)[4]) {
    lo[0] = c.x & 0x0F0F0F0Fu;
    lo[1] = c.y & 0x0F0F0F0Fu;
    lo[2] = c.z & 0x0F0F0F0Fu;
    lo[3] = c.w & 0x0F0F0F0Fu;
    hi[0] = (c.x >> 4) & 0x0F0F0F0Fu;
    hi[1] = (c.y >> 4) & 0x0F0F0F0Fu;
    hi[2] = (c.z >> 4) & 0x0F0F0F0Fu;
    hi[3] = (c.w >> 4) & 0x0F0F0F0Fu;
}

__device__ __forceinline__ int dot_q8(uint4 c0, uint4 c1, uint4 a0, uint4 a1, int init) {
    int d = init;
    d = dp4a(static_cast<int>(c0.x), static_cast<int>(a0.x), d);
    d = dp4a(static_cast<int>(c0.y), static_cast<int>(a0.y), d);
    d = dp4a(static_cast<int>(c0.z), static_cast<int>(a0.z), d);
    d = dp4a(static_cast<int>(c0.w), static_cast<int>(a0.w), d);
    d = dp4a(static_cast<int>(c1.x), static_cast<int>(a1.x), d);
    d = dp4a(static_cast<int>(c1.y), static_cast<int>(a1.y), d);
    d = dp4a(static_cast<int>(c1.z), static_cast<int>(a1.z), d);
    d = dp4a(static_cast<int>(c1.w), static_cast<int>(a1.w), d);
    return d;
}

__device__ __forceinline__ float biased_to_float(int d) { return __fsub_rn(__int_as_float(d), FP_BIAS); }

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
template <int QT, int PAIR, int MT, bool EXACT>
__global__ void __launch_bounds__(QMM_THREADS, 1) qmm_kernel(const QmmArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ int s_flag;
    __shared__ volatile int s_abort;   // set by anyone whose bounded wait ran out
    __shared__ volatile int s_cabort;  // set by consumers only, read after a consumer barrier

    constexpr int REC = QT == SD_Q8_0 ? 1088 : 576;  // bytes of one 32-row record
    constexpr int CODE = QT == SD_Q8_0 ? 1024 : 512; // code bytes of a record
    constexpr int ROWS = PAIR ? 64 : 32;
    const int M = EXACT ? MT : a.M;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + a.NS;
    uint8_t *ring = smem + a.off_ring;
    uint8_t *act = smem + a.off_act;
    float2 *meta = reinterpret_cast<float2 *>(smem + a.off_meta);
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
            // stage this split's int8 activations: act[jb][m][32], meta[jb][m] = {d_a, chain start}
            named_bar_sync(1, NCW * 32);
            const int64_t K = static_cast<int64_t>(a.KB) * 32;
            const int b0 = s * a.KBs;
            const int nchunk = len * M * 2;
            for (int c = tid; c < nchunk; c += NCW * 32) {
                int jb = c / (M * 2), rem = c - jb * (M * 2), m = rem >> 1, h = rem & 1;
                uint4 v = *reinterpret_cast<const uint4 *>(a.q + m * K + static_cast<int64_t>(b0 + jb) * 32 + h * 16);
                *reinterpret_cast<uint4 *>(act + (jb * MT + m) * 32 + h * 16) = v;
            }
            for (int c = tid; c < len * M; c += NCW * 32) {
                int jb = c / M, m = c - jb * M;
                float da = a.sc[static_cast<int64_t>(m) * a.KB + b0 + jb];
                int init = FP_BIAS_BITS;
                if (QT == SD_Q4_32) {
                    const uint4 *p = reinterpret_cast<const uint4 *>(a.q + m * K + static_cast<int64_t>(b0 + jb) * 32);
                    uint4 x0 = p[0], x1 = p[1];
                    int sum = 0;
                    sum = dp4a(0x01010101, static_cast<int>(x0.x), sum);
                    sum = dp4a(0x01010101, static_cast<int>(x0.y), sum);
                    sum = dp4a(0x01010101, static_cast<int>(x0.z), sum);
                    sum = dp4a(0x01010101, static_cast<int>(x0.w), sum);
                    sum = dp4a(0x01010101, static_cast<int>(x1.x), sum);
                    sum = dp4a(0x01010101, static_cast<int>(x1.y), sum);
                    sum = dp4a(0x01010101, static_cast<int>(x1.z), sum);
                    sum = dp4a(0x01010101, static_cast<int>(x1.w), sum);
                    init += -8 * sum;
                }
                meta[jb * MT + m] = make_float2(da, __int_as_float(init));
            }
            named_bar_sync(1, NCW * 32);
            cur_s = s;
        }

        float acc[MT], accu[PAIR ? MT : 1];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.0f;
#pragma unroll
        for (int m = 0; m < (PAIR ? MT : 1); ++m) accu[m] = 0.0f;

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
                const uint8_t *ab = act + jb * MT * 32;
                const float2 *mb = meta + jb * MT;
                if (QT == SD_Q4_32) {
                    uint32_t lo4[4], hi4[4], lou[4], hiu[4];
                    unpack_q4(*reinterpret_cast<const uint4 *>(rec + lane * 16), lo4, hi4);
                    const float dw = __half2float(*reinterpret_cast<const __half *>(rec + CODE + lane * 2));
                    float dwu = 0.0f;
                    if (PAIR) {
                        unpack_q4(*reinterpret_cast<const uint4 *>(rec + REC + lane * 16), lou, hiu);
                        dwu = __half2float(*reinterpret_cast<const __half *>(rec + REC + CODE + lane * 2));
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (EXACT || m < M) {
                            const uint4 a0 = *reinterpret_cast<const uint4 *>(ab + m * 32);
                            const uint4 a1 = *reinterpret_cast<const uint4 *>(ab + m * 32 + 16);
                            const float2 mm = mb[m];
                            const int init = __float_as_int(mm.y);
                            acc[m] = __fmaf_rn(__fmul_rn(dw, mm.x), biased_to_float(dot_q4(lo4, hi4, a0, a1, init)), acc[m]);
                            if (PAIR)
                                accu[m] = __fmaf_rn(__fmul_rn(dwu, mm.x), biased_to_float(dot_q4(lou, hiu, a0, a1, init)),
                                                    accu[m]);
                        }
                    }
                } else {
                    const uint4 c0 = *reinterpret_cast<const uint4 *>(rec + lane * 16);
                    const uint4 c1 = *reinterpret_cast<const uint4 *>(rec + 512 + lane * 16);
                    const float dw = __half2float(*reinterpret_cast<const __half *>(rec + CODE + lane * 2));
                    uint4 cu0 = make_uint4(0, 0, 0, 0), cu1 = cu0;
                    float dwu = 0.0f;
                    if (PAIR) {
                        cu0 = *reinterpret_cast<const uint4 *>(rec + REC + lane * 16);
                        cu1 = *reinterpret_cast<const uint4 *>(rec + REC + 512 + lane * 16);
                        dwu = __half2float(*reinterpret_cast<const __half *>(rec + REC + CODE + lane * 2));
                    }
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (EXACT || m < M) {
                            const uint4 a0 = *reinterpret_cast<const uint4 *>(ab + m * 32);
                            const uint4 a1 = *reinterpret_cast<const uint4 *>(ab + m * 32 + 16);
                            const float2 mm = mb[m];
                            const int init = __float_as_int(mm.y);
                            acc[m] = __fmaf_rn(__fmul_rn(dw, mm.x), biased_to_float(dot_q8(c0, c1, a0, a1, init)), acc[m]);
                            if (PAIR)
                                accu[m] = __fmaf_rn(__fmul_rn(dwu, mm.x), biased_to_float(dot_q8(cu0, cu1, a0, a1, init)),
                                                    accu[m]);
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
        for (int m = 0; m < MT; ++m) {
            if (EXACT || m < M) {
                red[(warp * MT + m) * ROWS + lane] = acc[m];
                if (PAIR) red[(warp * MT + m) * ROWS + 32 + lane] = accu[m];
            }
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

// shared-memory layout for MT position slots; returns total bytes
inline size_t plan_smem(QmmPlan &p, int MT, bool pair, uint32_t &off_ring, uint32_t &off_act, uint32_t &off_meta,
                        uint32_t &off_red) {
    const int rows = pair ? 64 : 32;
    p.SB = p.step_bytes >= 1000 ? NCW : 2 * NCW;  // ~9-18 KB stages
    const size_t stage = static_cast<size_t>(p.SB) * p.step_bytes;
    const size_t act = static_cast<size_t>(p.KBs) * MT * 32;
    const size_t meta = static_cast<size_t>(p.KBs) * MT * 8;
    const size_t red = static_cast<size_t>(NCW) * MT * rows * 4;
    const size_t fixed = 256 + act + meta + red;
    // ~72 KB of stages in flight; with M <= 5 the whole CTA stays near 110 KB so the
    // next kernel's CTA can be resident (and prefetching) beside it
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

template <int QT, int PAIR, int MT, bool EXACT>
cudaError_t qmm_launch(QmmArgs a, size_t smem, cudaStream_t s) {
    auto k = qmm_kernel<QT, PAIR, MT, EXACT>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch(k, dim3(a.G), dim3(QMM_THREADS), smem, s, a);
}

// dispatch on M (exact instantiations for 1..8, a guarded 16-slot one above)
template <int QT, int PAIR>
cudaError_t qmm_dispatch(QmmArgs a, QmmPlan &p, cudaStream_t s);

}  // namespace sdv
