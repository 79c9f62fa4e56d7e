// sdv_sample.cuh - rejection-sampling acceptance of one verify pass ("Speculative Decoding with
// Open-Weights Models", section "Mathematical Integrity: Rejection Sampling for LLMs": accept a
// draft with probability min(1, p/q), on rejection draw from max(0, p - q)), shared by the
// single-operation kernel and the one-launch pass.
#pragma once
#include "sdv_common.cuh"

namespace sdv {

constexpr int ATILE = 1024;      // vocabulary tile (same tiles as the head's statistics)
constexpr int MAX_TILES = 2048;  // vocabularies up to 2M tokens

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

// Shared state of one acceptance (one CTA).
struct SampleShared {
    float tm[MAX_TILES], ts[MAX_TILES];
    float m[16], Z[16];
    int row, mode, x, n, tile;
    float u, rem;
};

// The acceptance of one CTA's NTH threads (thread index tid, whole warps); `sync` is a barrier over
// exactly those threads.  The statistics come from row_max / row_sumexp when given, else they are
// formed here with the head's tiles and fold.  Tiles go to warps round robin and each tile's sum
// is one warp's tree, so any NTH gives the same bits.
template <int NTH, class Sync>
__device__ void sample_accept(const SampleArgs &a, SampleShared &sh, int tid, Sync sync) {
    float *s_tm = sh.tm, *s_ts = sh.ts, *s_m = sh.m, *s_Z = sh.Z;
    int &s_row = sh.row, &s_mode = sh.mode, &s_x = sh.x, &s_n = sh.n, &s_tile = sh.tile;
    float &s_u = sh.u, &s_rem = sh.rem;
    const int lane = tid & 31, warp = tid >> 5, nwarps = NTH / 32;
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
        sync();
        if (tid == 0) {
            float m = -__int_as_float(0x7f800000);
            for (int t = 0; t < ntiles; ++t) m = fmaxf(m, s_tm[t]);
            float Z = 0.0f;
            for (int t = 0; t < ntiles; ++t) Z = __fadd_rn(Z, __fmul_rn(s_ts[t], cexpf_canon(__fsub_rn(s_tm[t], m))));
            s_m[row] = m;
            s_Z[row] = Z;
        }
        sync();
    }
    sync();

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
    sync();

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
        sync();
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
        sync();
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
