// sdv_topk.cuh - rejection-sampling acceptance against a top-k / top-p filtered target (the sampling
// knobs of "Inside OpenJet Engine", API section: temperature, top-k up to 32, top-p; the rule of
// "Speculative Decoding with Open-Weights Models", section "Mathematical Integrity: Rejection
// Sampling for LLMs", applied to the filtered distribution), shared by the single-operation kernel and
// the one-launch pass.
//
// Row i: z_j = l_j / T (+0, so -0 and +0 are one value).  The candidates are the top_k tokens by z,
// larger z first and the lower token index among equal z; they are found by an MSB-first radix
// select on an order-preserving 32-bit key of z (four 8-bit passes), then gathered in token order
// (block-wide prefix sums, so ties at the k-th key keep the lowest indices) and ranked by one warp.
// With m = z of the first candidate, e_c = cexp(z_c - m); S = their sequential sum; the nucleus is
// the shortest prefix whose running sum reaches top_p * S; p'_c = e_c / (its running sum).  Draft x
// is kept iff u_acc * q(x) < p'(x); a rejection draws from max(0, p'_c - q(c)) over the nucleus in
// candidate order (falling back to p'), a full acceptance draws the bonus token from p' of row K.
#pragma once
#include "sdv_common.cuh"
#include "sdv_sample.cuh"

namespace sdv {

constexpr int TK_MAX = 32;  // largest top_k

struct TopkArgs {
    const float *logits;
    int64_t V;
    int K;
    const float *q;
    const int32_t *drafts;
    float T;
    int top_k;
    float top_p;
    uint64_t seed;
    int64_t base_pos;
    int32_t *out;
    int32_t *count;
};

__device__ __forceinline__ float topk_z(const TopkArgs &a, int row, int64_t j) {
    return __fadd_rn(__fdiv_rn(a.logits[row * a.V + j], a.T), 0.0f);
}

// order-preserving key: a larger z gives a larger key
__device__ __forceinline__ uint32_t topk_key(float z) {
    const uint32_t u = __float_as_uint(z);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// exclusive prefix sum of v over NTH threads (scratch: 32 ints); returns the total in *tot
template <int NTH, class Sync>
__device__ __forceinline__ int block_excl_scan(int v, int *scratch, int *tot, int tid, Sync sync) {
    constexpr int NW = NTH / 32;
    const int lane = tid & 31, warp = tid >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    sync();
    if (warp == 0) {
        int w = lane < NW ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NW) scratch[lane] = w;  // inclusive over warps
    }
    sync();
    const int before = (warp > 0 ? scratch[warp - 1] : 0) + x - v;
    *tot = scratch[NW - 1];
    sync();
    return before;
}

// inverse-CDF draw over n weights in order: the first w > 0 whose running sum exceeds u * W, else the
// last w > 0; -1 when they sum to zero (one thread)
__device__ inline int topk_draw(const float *w, int n, float u) {
    float W = 0.0f;
    for (int c = 0; c < n; ++c) W = __fadd_rn(W, w[c]);
    if (!(W > 0.0f)) return -1;
    const float target = __fmul_rn(u, W);
    float run = 0.0f;
    int last = -1;
    for (int c = 0; c < n; ++c) {
        run = __fadd_rn(run, w[c]);
        if (w[c] > 0.0f) {
            last = c;
            if (run > target) return c;
        }
    }
    return last;
}

// Shared state of one filtered acceptance (one CTA).
struct TopkShared {
    uint32_t hist[256];
    int scratch[32];
    int32_t c_tok[TK_MAX], s_tok[TK_MAX];
    float c_z[TK_MAX], s_p[TK_MAX];
    uint32_t s_prefix;
    int s_need, s_stop, s_n;
};

// The filtered acceptance of one CTA's NTH threads (thread index tid, whole warps, NTH <= 1024);
// `sync` is a barrier over exactly those threads.  Any NTH gives the same bits: the histogram
// counts, the prefix sums and the single-thread decisions do not depend on it.
template <int NTH, class Sync>
__device__ void topk_accept(const TopkArgs &a, TopkShared &sh, int tid, Sync sync) {
    uint32_t *hist = sh.hist;
    int *scratch = sh.scratch;
    int32_t *c_tok = sh.c_tok, *s_tok = sh.s_tok;
    float *c_z = sh.c_z, *s_p = sh.s_p;
    uint32_t &s_prefix = sh.s_prefix;
    int &s_need = sh.s_need, &s_stop = sh.s_stop, &s_n = sh.s_n;
    const int lane = tid & 31, warp = tid >> 5;
    const int keff = a.V < a.top_k ? static_cast<int>(a.V) : a.top_k;
    const int64_t chunk = (a.V + NTH - 1) / NTH;
    const int64_t c0 = tid * chunk < a.V ? tid * chunk : a.V, c1 = c0 + chunk < a.V ? c0 + chunk : a.V;
    if (tid == 0) s_n = 0;
    for (int row = 0; row <= a.K; ++row) {
        // 1. the key of the keff-th largest z: MSB-first radix select, 8 bits per pass
        uint32_t prefix = 0u, mask = 0u;
        int need = keff;
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int b = tid; b < 256; b += NTH) hist[b] = 0u;
            sync();
            for (int64_t j = tid; j < a.V; j += NTH) {
                const uint32_t key = topk_key(topk_z(a, row, j));
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
            sync();
            if (tid == 0) {
                int cum = 0, sel = 0;
                for (int b = 255; b >= 0; --b) {
                    const int c = static_cast<int>(hist[b]);
                    if (cum + c >= need) {
                        sel = b;
                        break;
                    }
                    cum += c;
                }
                s_prefix = prefix | (static_cast<uint32_t>(sel) << shift);
                s_need = need - cum;
            }
            sync();
            prefix = s_prefix;
            need = s_need;
            mask |= 255u << shift;
            sync();
        }
        // 2. gather in token order: every key above the threshold, then the first `need` equal to it
        int ngt = 0, neq = 0;
        for (int64_t j = c0; j < c1; ++j) {
            const uint32_t key = topk_key(topk_z(a, row, j));
            ngt += key > prefix;
            neq += key == prefix;
        }
        int tgt, teq;
        int ogt = block_excl_scan<NTH>(ngt, scratch, &tgt, tid, sync);
        int oeq = block_excl_scan<NTH>(neq, scratch, &teq, tid, sync);
        for (int64_t j = c0; j < c1 && (ngt > 0 || (neq > 0 && oeq < need)); ++j) {
            const float z = topk_z(a, row, j);
            const uint32_t key = topk_key(z);
            if (key > prefix) {
                c_tok[ogt] = static_cast<int32_t>(j);
                c_z[ogt] = z;
                ++ogt;
                --ngt;
            } else if (key == prefix) {
                if (oeq < need) {
                    c_tok[tgt + oeq] = static_cast<int32_t>(j);
                    c_z[tgt + oeq] = z;
                }
                ++oeq;
                --neq;
            }
        }
        sync();
        // 3. rank the keff candidates: larger z first, lower index among equals
        if (warp == 0) {
            if (lane < keff) {
                const float z = c_z[lane];
                const int32_t t = c_tok[lane];
                int r = 0;
                for (int c = 0; c < keff; ++c) r += c_z[c] > z || (c_z[c] == z && c_tok[c] < t);
                s_tok[r] = t;
                s_p[r] = z;
            }
        }
        sync();
        // 4. the nucleus, then this row's decision (one thread)
        if (tid == 0) {
            float e[TK_MAX], w[TK_MAX];
            float S = 0.0f;
            for (int c = 0; c < keff; ++c) {
                e[c] = cexpf_canon(__fsub_rn(s_p[c], s_p[0]));
                S = __fadd_rn(S, e[c]);
            }
            const float goal = __fmul_rn(a.top_p, S);
            int nn = 0;
            float run = 0.0f;
            while (nn < keff) {
                run = __fadd_rn(run, e[nn]);
                ++nn;
                if (run >= goal) break;
            }
            for (int c = 0; c < nn; ++c) e[c] = __fdiv_rn(e[c], run);  // p'
            const uint64_t pos = static_cast<uint64_t>(a.base_pos + row);
            const uint4 ph = philox4x32_10(make_uint4(static_cast<uint32_t>(pos), static_cast<uint32_t>(pos >> 32), 0u, 0u),
                                           static_cast<uint32_t>(a.seed), static_cast<uint32_t>(a.seed >> 32));
            int stop = 1, tok = -1;
            if (row == a.K) {
                const int c = topk_draw(e, nn, uniform24(ph.y));
                tok = s_tok[c];
            } else {
                const int32_t x = a.drafts[row];
                float px = 0.0f;
                for (int c = 0; c < nn; ++c)
                    if (s_tok[c] == x) px = e[c];
                const float qx = a.q ? a.q[row * a.V + x] : 1.0f;
                if (__fmul_rn(uniform24(ph.x), qx) < px) {
                    tok = x;
                    stop = 0;
                } else {
                    for (int c = 0; c < nn; ++c) {
                        const float qc = a.q ? a.q[row * a.V + s_tok[c]] : (s_tok[c] == x ? 1.0f : 0.0f);
                        const float d = __fsub_rn(e[c], qc);
                        w[c] = d > 0.0f ? d : 0.0f;
                    }
                    int c = topk_draw(w, nn, uniform24(ph.y));
                    if (c < 0) c = topk_draw(e, nn, uniform24(ph.y));
                    tok = s_tok[c];
                }
            }
            a.out[s_n] = tok;
            ++s_n;
            s_stop = stop;
            if (stop) *a.count = s_n;
        }
        sync();
        if (s_stop) break;
    }
}

}  // namespace sdv
