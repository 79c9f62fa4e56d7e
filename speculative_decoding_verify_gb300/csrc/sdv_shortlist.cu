// sdv_shortlist.cu - exact shortlist head for greedy verification ("How Kinetic is fast",
// section "Shortlist"): a cheaper copy of the output layer, with a proven bound on each row's
// error, scores every row; the best guaranteed score (the floor) rules out every row whose bound
// cannot reach it; the row tiles holding the remaining rows are scored by the head's own matmul,
// so the chosen token and its score are those of the full head bit for bit.
//
// The copy is the 32-weight 4-bit format of the Q8_0 head's dequantised rows (d = amax / 7.5
// rounded to fp16, code = 8 + round-half-away(w / d) clamped to [0, 15]).  Row r carries
// E_r >= ||w8_r - w4_r||_2 and W_r >= ||w8_r||_2, both rounded up.  With a the dequantised
// activation row of one position, its norm rounded up as A, s_r the copy score the 4-bit matmul
// computes in fp32 and l_r the head's fp32 logit:
//   |l_r - s_r| <= |l_r - exact_r| + |exact_r - s_r| <= B_r = (E_r + gamma (2 W_r + E_r)) A
// (Cauchy-Schwarz for the copy's error; gamma covers the fp32 rounding of the copy score, whose
// terms add up to at most ||w4_r|| ||a|| <= (W_r + E_r) A, and that of the head's logit, whose
// terms add up to at most W_r A).  The floor is F = max_r (s_r - B_r) and row r is a candidate iff
// s_r + B_r >= F; every bound operation is an fp32 operation rounded towards the safe side (A, B_r
// and s_r + B_r up, s_r - B_r down).  A row that is not a candidate has l_r < F <= l_b for the row b
// that set the floor, so the head's argmax (largest logit, lowest index among equals) is a
// candidate, and the argmax over the candidates' logits is the head's.
//
// Per call, six launches: the activation fragments of both matmuls; the copy matmul; the floor
// kernel; the candidate kernel, which marks the 32-row tiles holding a candidate; the Q8_0 head's own
// matmul restricted to the marked tiles (same plan, pieces and arithmetic as sd_head_logits, so those
// logits are its logits bit for bit); the argmax kernel over the marked tiles, whose last CTA also
// sets the next call's mode.  When a call marked more than a quarter of the tiles, the copy pays no
// more: the next calls run in full mode (copy, floor and candidates skipped, every tile marked) and
// try the shortlist again every SL_REPROBE calls.
#include "sdv_qmatmul.cuh"

namespace sdv {

constexpr int SL_THREADS = 256;
constexpr int SL_WARPS = SL_THREADS / 32;
constexpr int SL_MAXM = 16;
// CTAs per SM of the floor, candidate and argmax kernels: about one row per thread on a 152k vocabulary, so
// every thread issues its loads at once instead of walking a slice
constexpr int SL_CTAS_PER_SM = 4;

struct SlBest {
    float v;      // best logit (-inf: none)
    int32_t idx;  // its row (-1: none)
};

constexpr uint32_t SL_REPROBE = 16;  // full-mode calls try the shortlist again every 16 calls

struct ShortlistArgs {
    float *scores;        // copy scores [M][N], then the head's logits of the marked tiles
    const float *bound;   // E_r [N]
    const float *wnorm;   // W_r [N]
    const int8_t *q;      // activations [M][K]
    const float *sc;      // activation scales [M][KB]
    int64_t N, KB;
    int32_t M;
    int32_t G;              // CTAs of the floor, candidate and argmax kernels
    int64_t rows_per_cta;   // multiple of 32
    float gamma;
    float *an;              // [SL_MAXM] activation norms (rounded up), written by the floor kernel
    float *floor_part;      // [SL_MAXM][G]
    float *F;               // [SL_MAXM] floors, written by the floor kernel's last CTA
    SlBest *best_part;      // [SL_MAXM][G]
    uint32_t *ticket;       // [2] CTAs done (floor, argmax); zero between calls
    int *full;              // this call's mode: 1 full head, 0 shortlist
    uint32_t *state;        // [2] calls so far, tiles marked by the last shortlist call (kept across calls)
    uint32_t *umask;        // [NUW] marked 32-row tiles
    uint32_t *nmarked;      // tiles marked in this call
    int32_t *cand;          // [SL_MAXM] candidate rows per position
    int32_t NUW;            // mask words
    uint32_t budget;        // a shortlist call marking more tiles sends the next calls to full mode
    uint8_t *af4, *af8;     // activation fragments for the copy's and the head's matmul
    float *am4, *am8;       // their {corr, d_a} records
    int32_t *argmax;        // [M]
    int32_t *n_cand;        // [M] or nullptr
    int *status;
};

// ---------------------------------------------------------------------------
// load time: the copy, E_r and W_r (one warp per row, lanes over the row's blocks)
// ---------------------------------------------------------------------------

__device__ __forceinline__ double warp_sum_ru(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __dadd_ru(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__global__ void __launch_bounds__(SL_THREADS) shortlist_build_kernel(const uint8_t *src, int64_t N, int64_t KB,
                                                                     uint8_t *dst, float *bound, float *wnorm) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = static_cast<int>(threadIdx.x) & 31;
    const int64_t nwarps = static_cast<int64_t>(gridDim.x) * SL_WARPS;
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * SL_WARPS + threadIdx.x / 32; r < N; r += nwarps) {
        double e2 = 0.0, w2 = 0.0;  // sums of non-negative terms, every operation rounded up
        for (int64_t b = lane; b < KB; b += 32) {
            // a Q8_0 block starts on an even byte: read it as 17 halfwords
            const uint16_t *blk = reinterpret_cast<const uint16_t *>(src + (r * KB + b) * 34);
            const float d8 = __half2float(__ushort_as_half(blk[0]));
            float w[32];
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint16_t v = blk[1 + j];
                w[2 * j] = d8 * static_cast<float>(static_cast<int8_t>(v & 0xFF));  // exact: 11 x 8 bits
                w[2 * j + 1] = d8 * static_cast<float>(static_cast<int8_t>(v >> 8));
                amax = fmaxf(amax, fmaxf(fabsf(w[2 * j]), fabsf(w[2 * j + 1])));
            }
            // d = amax / 7.5 to fp16 (nearest even), held at the largest finite half if it overflows
            const float dq = amax / 7.5f;
            const __half dh = dq < 65520.0f ? __float2half_rn(dq) : __ushort_as_half(static_cast<uint16_t>(0x7BFF));
            const float d = __half2float(dh);
            int c[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                int ci = 8;
                if (d > 0.0f) {
                    const float t = roundf(w[i] / d) + 8.0f;  // roundf: halves away from zero
                    ci = t < 0.0f ? 0 : (t > 15.0f ? 15 : static_cast<int>(t));
                }
                c[i] = ci;
                // w and d (c - 8) carry at most 18 significant bits a few binades apart: the
                // difference is exact in fp64
                const double err = static_cast<double>(w[i]) - static_cast<double>(d) * static_cast<double>(ci - 8);
                e2 = __dadd_ru(e2, __dmul_ru(err, err));
                w2 = __dadd_ru(w2, __dmul_ru(static_cast<double>(w[i]), static_cast<double>(w[i])));
            }
            uint16_t *out = reinterpret_cast<uint16_t *>(dst + (r * KB + b) * 18);
            out[0] = __half_as_ushort(dh);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t lo = static_cast<uint32_t>(c[2 * j] | (c[2 * j + 16] << 4));
                const uint32_t hi = static_cast<uint32_t>(c[2 * j + 1] | (c[2 * j + 17] << 4));
                out[1 + j] = static_cast<uint16_t>(lo | (hi << 8));
            }
        }
        e2 = warp_sum_ru(e2);
        w2 = warp_sum_ru(w2);
        if (lane == 0) {
            bound[r] = __double2float_ru(__dsqrt_ru(e2));
            wnorm[r] = __double2float_ru(__dsqrt_ru(w2));
        }
    }
}

// ---------------------------------------------------------------------------
// verify time
// ---------------------------------------------------------------------------

// C_r = E_r + gamma (2 W_r + E_r), rounded up; B_r = C_r A for a position with norm A
__device__ __forceinline__ float row_coef(const ShortlistArgs &a, int64_t r) {
    const float E = a.bound[r], W = a.wnorm[r];
    return __fadd_ru(E, __fmul_ru(a.gamma, __fadd_ru(__fmul_ru(2.0f, W), E)));
}

__device__ __forceinline__ float warp_sum_ru_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_ru(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ||a_m||_2 of every position, rounded up: per block d_a^2 times the exact integer sum of squared
// codes, summed with upward rounding (the same value in every CTA).  One warp per position.
__device__ void act_norms(const ShortlistArgs &a, float *an) {
    const int warp = static_cast<int>(threadIdx.x) / 32, lane = static_cast<int>(threadIdx.x) & 31;
    const int64_t K = a.KB * 32;
    for (int m = warp; m < a.M; m += SL_WARPS) {
        float t = 0.0f;
        for (int64_t b = lane; b < a.KB; b += 32) {
            const int4 *qa = reinterpret_cast<const int4 *>(a.q + m * K + b * 32);
            const int4 q0 = qa[0], q1 = qa[1];
            int s2 = dp4a(q0.x, q0.x, 0);
            s2 = dp4a(q0.y, q0.y, s2);
            s2 = dp4a(q0.z, q0.z, s2);
            s2 = dp4a(q0.w, q0.w, s2);
            s2 = dp4a(q1.x, q1.x, s2);
            s2 = dp4a(q1.y, q1.y, s2);
            s2 = dp4a(q1.z, q1.z, s2);
            s2 = dp4a(q1.w, q1.w, s2);  // <= 32 * 127^2: exact in fp32
            const float d = a.sc[m * a.KB + b];
            t = __fadd_ru(t, __fmul_ru(__fmul_ru(d, d), static_cast<float>(s2)));
        }
        t = warp_sum_ru_f(t);
        if (lane == 0) an[m] = __fsqrt_ru(t);
    }
    __syncthreads();
}

// Whether this CTA is the grid's last to finish its part.  Every thread fences its stores of
// partial results before the CTA takes its ticket; the last CTA fences again before reading the
// others' partials and puts the counter back to zero for the next call.  Nothing waits.
__device__ __forceinline__ bool last_cta(uint32_t *ticket, int *flag) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const bool last = atomicAdd(ticket, 1u) == gridDim.x - 1;
        if (last) atomicExch(ticket, 0u);
        *flag = last ? 1 : 0;
    }
    __syncthreads();
    const bool last = *flag != 0;
    if (last) __threadfence();
    return last;
}

// the activation fragments of both matmuls (the copy's 4-bit layout, the head's Q8_0 layout), once
// (and this call's tile marks: every tile in full mode, none otherwise; its counters at zero)
__global__ void __launch_bounds__(256) shortlist_act_kernel(const ShortlistArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    act_frag_build<SD_Q4_32>(a.q, a.sc, a.M, static_cast<int>(a.KB), a.af4, a.am4);
    act_frag_build<SD_Q8_0>(a.q, a.sc, a.M, static_cast<int>(a.KB), a.af8, a.am8);
    const uint32_t mark = *a.full ? 0xffffffffu : 0u;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.NUW; i += gridDim.x * blockDim.x) a.umask[i] = mark;
    if (blockIdx.x == gridDim.x - 1) act_norms(a, a.an);  // written to global: the floor and candidate kernels read them
    if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < SL_MAXM) a.cand[threadIdx.x] = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.nmarked = 0;
}

// the floor: per CTA, max over its rows of s_r - B_r (rounded down), per position; the last CTA
// reduces the CTAs' maxima to the floor of each position
__global__ void __launch_bounds__(SL_THREADS, SL_CTAS_PER_SM) shortlist_floor_kernel(const ShortlistArgs a) {
    __shared__ float an[SL_MAXM];
    __shared__ float red[SL_MAXM][SL_WARPS];
    __shared__ int is_last;
    pdl_wait();
    pdl_launch_dependents();
    if (*reinterpret_cast<const volatile int *>(a.full)) return;
    if (static_cast<int>(threadIdx.x) < a.M) an[threadIdx.x] = __ldcg(a.an + threadIdx.x);
    __syncthreads();
    const int warp = static_cast<int>(threadIdx.x) / 32, lane = static_cast<int>(threadIdx.x) & 31;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * a.rows_per_cta;
    const int64_t r1 = min(a.N, r0 + a.rows_per_cta);
    float mx[SL_MAXM];
#pragma unroll
    for (int m = 0; m < SL_MAXM; ++m) mx[m] = -INFINITY;
    for (int64_t r = r0 + threadIdx.x; r < r1; r += SL_THREADS) {
        const float c = row_coef(a, r);
#pragma unroll
        for (int m = 0; m < SL_MAXM; ++m)
            if (m < a.M) mx[m] = fmaxf(mx[m], __fsub_rd(a.scores[m * a.N + r], __fmul_ru(c, an[m])));
    }
#pragma unroll
    for (int m = 0; m < SL_MAXM; ++m) {
        if (m >= a.M) break;
        const float v = warp_max_f(mx[m]);
        if (lane == 0) red[m][warp] = v;
    }
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < a.M) {
        float v = red[threadIdx.x][0];
#pragma unroll
        for (int w = 1; w < SL_WARPS; ++w) v = fmaxf(v, red[threadIdx.x][w]);
        a.floor_part[threadIdx.x * a.G + blockIdx.x] = v;
    }
    if (!last_cta(a.ticket, &is_last)) return;
    for (int m = warp; m < a.M; m += SL_WARPS) {
        float f = -INFINITY;
#pragma unroll 8
        for (int c = lane; c < a.G; c += 32) f = fmaxf(f, __ldcg(a.floor_part + m * a.G + c));
        f = warp_max_f(f);
        if (lane == 0) a.F[m] = f;
    }
}

// (value, index) of the better of two: larger value, lower index among equal values; idx < 0 = none
__device__ __forceinline__ void better(float &v, int32_t &i, float v2, int32_t i2) {
    if (i2 >= 0 && (i < 0 || v2 > v || (v2 == v && i2 < i))) {
        v = v2;
        i = i2;
    }
}

// candidates: per row, the positions whose floor its bound reaches; a row with any marks its 32-row
// tile; per position the candidate count (skipped in full mode, where every tile is marked)
__global__ void __launch_bounds__(SL_THREADS, SL_CTAS_PER_SM) shortlist_cand_kernel(const ShortlistArgs a) {
    __shared__ float F[SL_MAXM], an[SL_MAXM];
    __shared__ int cnt[SL_MAXM];
    pdl_wait();
    pdl_launch_dependents();
    if (*reinterpret_cast<const volatile int *>(a.full)) return;  // full mode: every tile is marked
    const int M = a.M, lane = static_cast<int>(threadIdx.x) & 31;
    if (static_cast<int>(threadIdx.x) < M) {
        F[threadIdx.x] = __ldcg(a.F + threadIdx.x);
        an[threadIdx.x] = __ldcg(a.an + threadIdx.x);
        cnt[threadIdx.x] = 0;
    }
    __syncthreads();
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * a.rows_per_cta;
    const int64_t r1 = min(a.N, r0 + a.rows_per_cta);
    // rows_per_cta is a multiple of 32: a warp's 32 rows are one tile
    for (int64_t g = r0 + (threadIdx.x & ~31u); g < r1; g += SL_THREADS) {
        const int64_t r = g + lane;
        uint32_t cm = 0;
        if (r < r1) {
            const float c = row_coef(a, r);
            for (int m = 0; m < M; ++m)
                if (__fadd_ru(__ldcg(a.scores + m * a.N + r), __fmul_ru(c, an[m])) >= F[m]) cm |= 1u << m;
        }
        const uint32_t any = __ballot_sync(0xffffffffu, cm != 0);
        if (any && lane == 0) {
            const int64_t t = g >> 5;
            const uint32_t bit = 1u << (t & 31);
            if (!(atomicOr(a.umask + (t >> 5), bit) & bit)) atomicAdd(a.nmarked, 1u);
        }
        for (int m = 0; m < M; ++m) {
            const int n = __popc(__ballot_sync(0xffffffffu, (cm >> m) & 1u));
            if (n && lane == 0) atomicAdd(&cnt[m], n);
        }
    }
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < M && cnt[threadIdx.x]) atomicAdd(a.cand + threadIdx.x, cnt[threadIdx.x]);
}

// the argmax over the marked tiles' logits (the head's own), per CTA then by its last CTA; the
// candidate counts (every row in full mode) and the tiles marked, for the next call's mode
__global__ void __launch_bounds__(SL_THREADS, SL_CTAS_PER_SM) shortlist_argmax_kernel(const ShortlistArgs a) {
    __shared__ float wv[SL_WARPS][SL_MAXM];
    __shared__ int32_t wi[SL_WARPS][SL_MAXM];
    __shared__ int is_last;
    pdl_wait();
    pdl_launch_dependents();
    const int M = a.M, warp = static_cast<int>(threadIdx.x) / 32, lane = static_cast<int>(threadIdx.x) & 31;
    float bv[SL_MAXM];
    int32_t bi[SL_MAXM];
#pragma unroll
    for (int m = 0; m < SL_MAXM; ++m) {
        bv[m] = -INFINITY;
        bi[m] = -1;
    }
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * a.rows_per_cta;
    const int64_t r1 = min(a.N, r0 + a.rows_per_cta);
    for (int64_t g = r0 + (threadIdx.x & ~31u); g < r1; g += SL_THREADS) {
        const int64_t t = g >> 5, r = g + lane;
        if (!((__ldcg(a.umask + (t >> 5)) >> (t & 31)) & 1u) || r >= r1) continue;
#pragma unroll
        for (int m = 0; m < SL_MAXM; ++m)
            if (m < M) better(bv[m], bi[m], __ldcg(a.scores + m * a.N + r), static_cast<int32_t>(r));
    }
#pragma unroll
    for (int m = 0; m < SL_MAXM; ++m) {
        if (m >= M) break;
        float v = bv[m];
        int32_t i = bi[m];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) better(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
        if (lane == 0) {
            wv[warp][m] = v;
            wi[warp][m] = i;
        }
    }
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < M) {
        float v = -INFINITY;
        int32_t i = -1;
        for (int w = 0; w < SL_WARPS; ++w) better(v, i, wv[w][threadIdx.x], wi[w][threadIdx.x]);
        a.best_part[threadIdx.x * a.G + blockIdx.x] = SlBest{v, i};
    }
    if (!last_cta(a.ticket + 1, &is_last)) return;
    const bool full = *reinterpret_cast<const volatile int *>(a.full) != 0;
    for (int m = warp; m < M; m += SL_WARPS) {
        float v = -INFINITY;
        int32_t i = -1;
#pragma unroll 8
        for (int c = lane; c < a.G; c += 32) {
            const SlBest *x = a.best_part + m * a.G + c;
            better(v, i, __ldcg(&x->v), __ldcg(&x->idx));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) better(v, i, __shfl_xor_sync(0xffffffffu, v, o), __shfl_xor_sync(0xffffffffu, i, o));
        if (lane == 0) {
            // with finite inputs the row of the head's maximum is always marked
            if (i < 0) set_status(a.status, SD_EDEVICE);
            a.argmax[m] = i;
            if (a.n_cand) a.n_cand[m] = full ? static_cast<int32_t>(a.N) : __ldcg(a.cand + m);
        }
    }
    // the next call's mode: full when the last shortlist call marked more tiles than the budget, except
    // every SL_REPROBE-th call
    if (threadIdx.x == 0) {
        const uint32_t calls = a.state[0] + 1;
        if (!full) a.state[1] = __ldcg(a.nmarked);
        a.state[0] = calls;
        *a.full = a.state[1] > a.budget && calls % SL_REPROBE != 0;
    }
}

struct SlLayout {
    size_t mm, scores, an, F, ticket, floor_part, best_part, full, state, nmarked, cand, umask, af4, af8, total;
    int G, NUW;
    int64_t rows_per_cta;
};

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static bool sl_layout(int64_t vocab, int64_t hidden, SlLayout &L) {
    if (vocab < 1 || vocab > (int64_t(1) << 31) - 1 || hidden <= 0 || hidden % 32) return false;
    // one workspace region serves the copy matmul and then the restricted head matmul
    const size_t mm4 = sd_qmatmul_workspace_bytes(SD_Q4_32, vocab, hidden, SD_EPI_NONE);
    const size_t mm8 = sd_qmatmul_workspace_bytes(SD_Q8_0, vocab, hidden, SD_EPI_NONE);
    if (mm4 == 0 || mm8 == 0) return false;
    const int sms = num_sms();
    if (sms < 1) return false;
    L.G = sms * SL_CTAS_PER_SM;
    L.rows_per_cta = ((vocab + L.G - 1) / L.G + 31) / 32 * 32;
    L.NUW = static_cast<int>(((vocab + 31) / 32 + 31) / 32);
    // the state kept between calls and the counters first, at offsets every shape shares (a workspace
    // may serve calls of several shapes); the matmuls' region next, its own counters at a fixed offset
    L.ticket = 0;
    L.full = 16;
    L.state = 32;
    L.nmarked = 48;
    L.cand = 64;  // SL_MAXM int32
    L.mm = 256;
    L.scores = align256(L.mm + (mm4 > mm8 ? mm4 : mm8));
    L.an = align256(L.scores + sizeof(float) * SL_MAXM * static_cast<size_t>(vocab));
    L.F = align256(L.an + sizeof(float) * SL_MAXM);
    L.floor_part = align256(L.F + sizeof(float) * SL_MAXM);
    L.best_part = align256(L.floor_part + sizeof(float) * SL_MAXM * L.G);
    L.umask = align256(L.best_part + sizeof(SlBest) * SL_MAXM * L.G);
    const size_t afb = static_cast<size_t>(hidden / 32) * af_ws_bytes_per_block(SD_Q8_0);  // either layout fits
    L.af4 = align256(L.umask + sizeof(uint32_t) * static_cast<size_t>(L.NUW));
    L.af8 = align256(L.af4 + afb);
    L.total = align256(L.af8 + afb);
    return true;
}

}  // namespace sdv

using namespace sdv;

extern "C" {

sd_status sd_shortlist_build(const void *head_blocks, int64_t vocab, int64_t hidden, void *copy_blocks, float *bound,
                             float *wnorm, sd_stream_t stream) {
    SD_NVTX("sd_shortlist_build");
    if (!head_blocks || !copy_blocks || !bound || !wnorm) return SD_EINVAL;
    if (!aligned(head_blocks, 16) || !aligned(copy_blocks, 16) || !aligned(bound, 4) || !aligned(wnorm, 4))
        return SD_EINVAL;
    if (vocab < 1 || vocab > (int64_t(1) << 31) - 1 || hidden <= 0 || hidden % 32) return SD_EINVAL;
    const int sms = num_sms();
    if (sms < 1) return SD_ECUDA;
    const int64_t need = (vocab + SL_WARPS - 1) / SL_WARPS;
    const int grid = static_cast<int>(need < int64_t(sms) * 8 ? need : int64_t(sms) * 8);
    return launch(shortlist_build_kernel, dim3(grid), dim3(SL_THREADS), 0, reinterpret_cast<cudaStream_t>(stream),
                  static_cast<const uint8_t *>(head_blocks), vocab, hidden / 32, static_cast<uint8_t *>(copy_blocks),
                  bound, wnorm) == cudaSuccess
               ? SD_OK
               : SD_ECUDA;
}

size_t sd_shortlist_workspace_bytes(int64_t vocab, int64_t hidden) {
    SlLayout L;
    return sl_layout(vocab, hidden, L) ? L.total : 0;
}

sd_status sd_head_shortlist(const void *copy_w, const float *bound, const float *wnorm, const void *head_w,
                            int64_t vocab, int64_t hidden, const int8_t *q, const float *scales, int32_t M,
                            int32_t *argmax, int32_t *n_cand, void *workspace, size_t ws_bytes, sd_stream_t stream) {
    SD_NVTX("sd_head_shortlist");
    if (M < 1) return SD_EINVAL;
    if (M > SL_MAXM) return SD_EUNSUPPORTED;
    if (!copy_w || !bound || !wnorm || !head_w || !q || !scales || !argmax || !workspace) return SD_EINVAL;
    if (!aligned(copy_w, 16) || !aligned(head_w, 16) || !aligned(q, 16) || !aligned(scales, 4) ||
        !aligned(bound, 4) || !aligned(wnorm, 4) || !aligned(argmax, 4) || (n_cand && !aligned(n_cand, 4)) ||
        !aligned(workspace, 256))
        return SD_EINVAL;
    SlLayout L;
    if (!sl_layout(vocab, hidden, L)) return SD_EINVAL;
    if (ws_bytes < L.total) return SD_EINVAL;
    const int64_t KB = hidden / 32;
    int *st = status_ptr();
    if (!st) return SD_ECUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    ShortlistArgs a = {};
    a.scores = reinterpret_cast<float *>(ws + L.scores);
    a.bound = bound;
    a.wnorm = wnorm;
    a.q = q;
    a.sc = scales;
    a.N = vocab;
    a.KB = KB;
    a.M = M;
    a.G = L.G;
    a.rows_per_cta = L.rows_per_cta;
    // fp32 copy score and fp32 head logit: at most KB + 64 rounding steps on any term's path, each
    // <= 2^-24 relative, taken twice over
    a.gamma = static_cast<float>(KB + 64) * 0x1p-23f;
    a.an = reinterpret_cast<float *>(ws + L.an);
    a.floor_part = reinterpret_cast<float *>(ws + L.floor_part);
    a.F = reinterpret_cast<float *>(ws + L.F);
    a.best_part = reinterpret_cast<SlBest *>(ws + L.best_part);
    a.ticket = reinterpret_cast<uint32_t *>(ws + L.ticket);
    a.full = reinterpret_cast<int *>(ws + L.full);
    a.state = reinterpret_cast<uint32_t *>(ws + L.state);
    a.nmarked = reinterpret_cast<uint32_t *>(ws + L.nmarked);
    a.cand = reinterpret_cast<int32_t *>(ws + L.cand);
    a.umask = reinterpret_cast<uint32_t *>(ws + L.umask);
    a.NUW = L.NUW;
    const int64_t NU = (vocab + 31) / 32;
    a.budget = static_cast<uint32_t>(NU / 4 > 0 ? NU / 4 : 1);
    a.af4 = ws + L.af4;
    a.am4 = reinterpret_cast<float *>(ws + L.af4 + static_cast<size_t>(KB) * af_frag_bytes(M));
    a.af8 = ws + L.af8;
    a.am8 = reinterpret_cast<float *>(ws + L.af8 + static_cast<size_t>(KB) * af_frag_bytes(M));
    a.argmax = argmax;
    a.n_cand = n_cand;
    a.status = st;
    const int64_t items = KB * (4 * M + 8 * af_nt(M));
    const int ablocks = static_cast<int>((items + 255) / 256 < 1024 ? (items + 255) / 256 : 1024);
    if (launch(shortlist_act_kernel, dim3(ablocks), dim3(256), 0, s, a) != cudaSuccess) return SD_ECUDA;
    // copy scores of every row: the multi-position matmul over the 4-bit copy (skipped in full mode)
    sd_status rc = qmatmul_restricted(SD_Q4_32, copy_w, vocab, hidden, q, scales, M, a.scores, nullptr, SD_EPI_NONE,
                                      0, nullptr, nullptr, ws + L.mm, L.scores - L.mm, nullptr, a.full, a.af4, a.am4, stream);
    if (rc != SD_OK) return rc;
    if (launch(shortlist_floor_kernel, dim3(L.G), dim3(SL_THREADS), 0, s, a) != cudaSuccess) return SD_ECUDA;
    if (launch(shortlist_cand_kernel, dim3(L.G), dim3(SL_THREADS), 0, s, a) != cudaSuccess) return SD_ECUDA;
    // the head's logits of the marked tiles, by the head's own matmul
    rc = qmatmul_restricted(SD_Q8_0, head_w, vocab, hidden, q, scales, M, a.scores, nullptr, SD_EPI_NONE, 0,
                            nullptr, nullptr, ws + L.mm, L.scores - L.mm, a.umask, nullptr, a.af8, a.am8, stream);
    if (rc != SD_OK) return rc;
    return launch(shortlist_argmax_kernel, dim3(L.G), dim3(SL_THREADS), 0, s, a) == cudaSuccess ? SD_OK : SD_ECUDA;
}

}  // extern "C"
