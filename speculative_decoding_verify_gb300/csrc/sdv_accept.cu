// sdv_accept.cu - greedy and rejection-sampling acceptance of the verify pass.
#include "sdv_common.cuh"

namespace sdv {

constexpr int ATILE = 1024;      // vocabulary tile (same tiles as the head's statistics)
constexpr int MAX_TILES = 2048;  // vocabularies up to 2M tokens
constexpr int ACC_THREADS = 1024;

// ---------------------------------------------------------------------------
// greedy: chain or tree, one thread
// ---------------------------------------------------------------------------
__global__ void accept_greedy_kernel(const int32_t *__restrict__ argmax, const int32_t *__restrict__ tokens,
                                     const int32_t *__restrict__ parent, int M, int32_t *__restrict__ out,
                                     int32_t *__restrict__ count) {
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x != 0) return;
    if (!parent) {
        const int K = M - 1;
        int n = 0;
        while (n < K && tokens[n] == argmax[n]) {
            out[n] = tokens[n];
            ++n;
        }
        out[n] = argmax[n];
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
        ok[i] = ok[p] && tokens[i] == argmax[p];
        if (ok[i] && depth[i] > depth[best]) best = i;
    }
    const int d = depth[best];
    for (int i = best, j = d - 1; i != 0; i = parent[i], --j) out[j] = tokens[i];
    out[d] = argmax[best];
    *count = d + 1;
}

// ---------------------------------------------------------------------------
// rejection sampling, one CTA
// ---------------------------------------------------------------------------
struct SampleArgs {
    const float *logits;
    int64_t V;
    int K;
    const float *row_max;
    const float *row_sumexp;
    const float *q;
    const int32_t *drafts;
    float T;
    uint64_t seed;
    int64_t base_pos;
    int32_t *out;
    int32_t *count;
};

__device__ __forceinline__ float uniform24(uint32_t w) { return __fmul_rn(static_cast<float>(w >> 8), 5.9604644775390625e-08f); }

__device__ __forceinline__ float prob(const SampleArgs &a, int row, int64_t i, float m, float Z) {
    float z = __fdiv_rn(a.logits[row * a.V + i], a.T);
    return __fdiv_rn(cexpf_canon(__fsub_rn(z, m)), Z);
}

// draw weight of token i: mode 0 = p, mode 1 = max(0, p - q) with q a row of
// q (or one-hot at x for a certainty drafter)
__device__ __forceinline__ float draw_w(const SampleArgs &a, int row, int64_t i, float m, float Z, int mode, int x) {
    float p = prob(a, row, i, m, Z);
    if (mode == 0) return p;
    float qi = a.q ? a.q[row * a.V + i] : (i == x ? 1.0f : 0.0f);
    float d = __fsub_rn(p, qi);
    return d > 0.0f ? d : 0.0f;
}

__global__ void __launch_bounds__(ACC_THREADS) accept_sample_kernel(const SampleArgs a) {
    __shared__ float s_tm[MAX_TILES];
    __shared__ float s_ts[MAX_TILES];
    __shared__ float s_m[16], s_Z[16];
    __shared__ int s_row, s_mode, s_x, s_n, s_tile;
    __shared__ float s_u, s_rem;
    pdl_wait();
    pdl_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = ACC_THREADS / 32;
    const int ntiles = static_cast<int>((a.V + ATILE - 1) / ATILE);

    // 1. softmax statistics of rows 0..K (the head's tiles and fold)
    for (int row = 0; row <= a.K; ++row) {
        if (a.row_max) {
            if (tid == 0) {
                s_m[row] = a.row_max[row];
                s_Z[row] = a.row_sumexp[row];
            }
            continue;
        }
        for (int t = warp; t < ntiles; t += nwarps) {
            float v[32];
            float mx = -__int_as_float(0x7f800000);
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                int64_t e = static_cast<int64_t>(t) * ATILE + lane + 32 * r;
                float z = -__int_as_float(0x7f800000);
                if (e < a.V) {
                    z = __fdiv_rn(a.logits[row * a.V + e], a.T);
                    mx = fmaxf(mx, z);
                }
                v[r] = z;
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                int64_t e = static_cast<int64_t>(t) * ATILE + lane + 32 * r;
                v[r] = e < a.V ? cexpf_canon(__fsub_rn(v[r], mx)) : 0.0f;
            }
            float s = tree1024_warp(v);
            if (lane == 0) {
                s_tm[t] = mx;
                s_ts[t] = s;
            }
        }
        __syncthreads();
        if (tid == 0) {
            float m = -__int_as_float(0x7f800000);
            for (int t = 0; t < ntiles; ++t) m = fmaxf(m, s_tm[t]);
            float Z = 0.0f;
            for (int t = 0; t < ntiles; ++t) Z = __fadd_rn(Z, __fmul_rn(s_ts[t], cexpf_canon(__fsub_rn(s_tm[t], m))));
            s_m[row] = m;
            s_Z[row] = Z;
        }
        __syncthreads();
    }
    __syncthreads();

    // 2. accept tests, in order; stop at the first rejection
    if (tid == 0) {
        int n = 0;
        int row = a.K, mode = 0, x = -1;
        float u = 0.0f;
        const uint32_t k0 = static_cast<uint32_t>(a.seed), k1 = static_cast<uint32_t>(a.seed >> 32);
        for (int i = 0; i <= a.K; ++i) {
            const uint64_t pos = static_cast<uint64_t>(a.base_pos + i);
            const uint4 ph = philox4x32_10(make_uint4(static_cast<uint32_t>(pos), static_cast<uint32_t>(pos >> 32), 0u, 0u), k0, k1);
            if (i == a.K) {
                u = uniform24(ph.y);
                break;
            }
            const int xi = a.drafts[i];
            const float px = prob(a, i, xi, s_m[i], s_Z[i]);
            const float qx = a.q ? a.q[i * a.V + xi] : 1.0f;
            if (__fmul_rn(uniform24(ph.x), qx) < px) {
                a.out[n++] = xi;
                continue;
            }
            row = i;
            mode = 1;
            x = xi;
            u = uniform24(ph.y);
            break;
        }
        s_n = n;
        s_row = row;
        s_mode = mode;
        s_x = x;
        s_u = u;
    }
    __syncthreads();

    // 3. inverse-CDF draw on row s_row: tiles, then 32-token chunks, then tokens
    const int row = s_row, x = s_x;
    const float m = s_m[row], Z = s_Z[row];
    for (int pass = 0; pass < 2; ++pass) {
        const int mode = s_mode;
        for (int t = warp; t < ntiles; t += nwarps) {
            float v[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                int64_t e = static_cast<int64_t>(t) * ATILE + lane + 32 * r;
                v[r] = e < a.V ? draw_w(a, row, e, m, Z, mode, x) : 0.0f;
            }
            float s = tree1024_warp(v);
            if (lane == 0) s_ts[t] = s;
        }
        __syncthreads();
        if (tid == 0) {
            float tot = 0.0f;
            for (int t = 0; t < ntiles; ++t) tot = __fadd_rn(tot, s_ts[t]);
            if (!(tot > 0.0f)) {
                s_tile = -1;
                s_mode = 0;  // residual mass zero: draw from p itself
            } else {
                const float target = __fmul_rn(s_u, tot);
                int tsel = -1;
                float C = 0.0f, Cprev = 0.0f;
                for (int t = 0; t < ntiles; ++t) {
                    float Cn = __fadd_rn(C, s_ts[t]);
                    if (Cn > target) {
                        tsel = t;
                        Cprev = C;
                        break;
                    }
                    C = Cn;
                }
                if (tsel < 0) {
                    for (int t = ntiles - 1; t >= 0; --t)
                        if (s_ts[t] > 0.0f) {
                            tsel = t;
                            break;
                        }
                    Cprev = 0.0f;
                    for (int t = 0; t < tsel; ++t) Cprev = __fadd_rn(Cprev, s_ts[t]);
                }
                s_tile = tsel;
                s_rem = __fsub_rn(target, Cprev);
            }
        }
        __syncthreads();
        if (s_tile >= 0 || pass == 1) break;
    }

    if (warp == 0) {
        const int mode = s_mode;
        const int tile = s_tile;
        if (tile < 0) {  // no positive mass at all (non-finite logits): report no token
            if (lane == 0) {
                a.out[s_n] = -1;
                *a.count = s_n + 1;
            }
            return;
        }
        const int64_t i0 = static_cast<int64_t>(tile) * ATILE;
        // chunk sums: lane j adds chunk j's 32 weights in token order
        float c = 0.0f;
        for (int i = 0; i < 32; ++i) {
            int64_t idx = i0 + lane * 32 + i;
            if (idx < a.V) c = __fadd_rn(c, draw_w(a, row, idx, m, Z, mode, x));
        }
        float cs[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) cs[j] = __shfl_sync(0xffffffffu, c, j);
        if (lane == 0) {
            const float rem = s_rem;
            int jsel = -1;
            float D = 0.0f, Dprev = 0.0f;
            for (int j = 0; j < 32; ++j) {
                float Dn = __fadd_rn(D, cs[j]);
                if (Dn > rem) {
                    jsel = j;
                    Dprev = D;
                    break;
                }
                D = Dn;
            }
            if (jsel < 0) {
                for (int j = 31; j >= 0; --j)
                    if (cs[j] > 0.0f) {
                        jsel = j;
                        break;
                    }
                Dprev = 0.0f;
                for (int j = 0; j < jsel; ++j) Dprev = __fadd_rn(Dprev, cs[j]);
            }
            const float rem2 = __fsub_rn(rem, Dprev);
            const int64_t base = i0 + static_cast<int64_t>(jsel) * 32;
            float e = 0.0f;
            int64_t last = -1, pick = -1;
            for (int i = 0; i < 32; ++i) {
                int64_t idx = base + i;
                float wi = idx < a.V ? draw_w(a, row, idx, m, Z, mode, x) : 0.0f;
                e = __fadd_rn(e, wi);
                if (wi > 0.0f) {
                    last = idx;
                    if (e > rem2) {
                        pick = idx;
                        break;
                    }
                }
            }
            if (pick < 0) pick = last;
            a.out[s_n] = static_cast<int32_t>(pick);
            *a.count = s_n + 1;
        }
    }
}

}  // namespace sdv

using namespace sdv;

static inline cudaStream_t cs_(sd_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

extern "C" {

sd_status sd_accept_greedy(const int32_t *argmax, const int32_t *tokens, const int32_t *parent, int32_t M,
                           int32_t *out_tokens, int32_t *out_count, sd_stream_t stream) {
    if (!argmax || !out_tokens || !out_count || M < 1 || M > 16) return SD_EINVAL;
    if (M > 1 && !tokens) return SD_EINVAL;
    return launch(accept_greedy_kernel, dim3(1), dim3(32), 0, cs_(stream), argmax, tokens, parent, static_cast<int>(M),
                  out_tokens, out_count) == cudaSuccess
               ? SD_OK
               : SD_ECUDA;
}

sd_status sd_accept_sample(const float *logits, int64_t vocab, int32_t K, const float *row_max,
                           const float *row_sumexp, const float *q_probs, const int32_t *drafts, float temperature,
                           uint64_t seed, int64_t base_pos, int32_t *out_tokens, int32_t *out_count,
                           sd_stream_t stream) {
    if (!logits || !out_tokens || !out_count || K < 0 || K > 15) return SD_EINVAL;
    if (K > 0 && !drafts) return SD_EINVAL;
    if (vocab < 1 || vocab > static_cast<int64_t>(MAX_TILES) * ATILE) return SD_EINVAL;
    if ((row_max == nullptr) != (row_sumexp == nullptr)) return SD_EINVAL;
    if (!(temperature > 0.0f) || temperature > 3.0e38f) return SD_EINVAL;
    SampleArgs a;
    a.logits = logits;
    a.V = vocab;
    a.K = K;
    a.row_max = row_max;
    a.row_sumexp = row_sumexp;
    a.q = q_probs;
    a.drafts = drafts;
    a.T = temperature;
    a.seed = seed;
    a.base_pos = base_pos;
    a.out = out_tokens;
    a.count = out_count;
    return launch(accept_sample_kernel, dim3(1), dim3(ACC_THREADS), 0, cs_(stream), a) == cudaSuccess ? SD_OK
                                                                                                      : SD_ECUDA;
}

}  // extern "C"
