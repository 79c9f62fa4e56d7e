/*
 * sdv_oracle.c - plain, slow, obviously correct CPU oracle for the
 * speculative-decoding verify pass.
 *
 * TEST INFRASTRUCTURE ONLY.  The product (the CUDA library) never links,
 * loads or calls this file; only the tests, the smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header, table or constant
 * generator with the CUDA path.
 *
 * Sources (pages on speculative decoding):
 *  - "Inside OpenJet Engine: making speculative decoding pay", section
 *    "One GPU launch for a speculative cycle": GGUF Q8_0 weights, integer
 *    dot products with int8 activations, requantised activations.
 *  - "Speculative Decoding with Open-Weights Models" (micrologics), section
 *    "Mathematical Integrity: Rejection Sampling for LLMs": accept x with
 *    min(1, p(x)/q(x)); on rejection draw from max(0, p - q) renormalised;
 *    and its walkthrough: a bonus token from the last row when all drafts pass.
 *  - "How Kinetic is fast", section "Why the output does not change": greedy
 *    keeps a guess only when it is the model's top token; a certainty drafter
 *    keeps x with probability p(x) and otherwise draws from p without x.
 *    Section "RAD-1": tree drafts, each row seeing only its own path.
 *
 * Where a floating-point result decides an integer (an activation code, an
 * accept decision, a drawn token) the oracle computes it in fp32 in the
 * canonical order the kernels also use, so both sides take the decision in
 * the same precision.  Everything else (the matmul) accumulates in fp64.
 * Build with -ffp-contract=off: every fp32 operation below is one rounding,
 * and fmaf() is used only where the canonical algorithm says "fused".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the following calls (timing on one core); the results do not depend on it. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ */
/* fp16 decode (IEEE 754 binary16 -> binary32, exact)                  */
/* ------------------------------------------------------------------ */
float oracle_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1, exp = (h >> 10) & 0x1F, man = h & 0x3FF;
    float v;
    if (exp == 0) v = ldexpf((float)man, -24);                 /* zero or subnormal */
    else if (exp == 31) v = man ? NAN : INFINITY;
    else v = ldexpf((float)(man | 0x400), exp - 25);           /* 1.m * 2^(e-15) */
    return sign ? -v : v;
}

/* ------------------------------------------------------------------ */
/* Block formats.  Q8_0: fp16 d (little endian) then 32 int8 q; value   */
/* d*q.  4-bit: fp16 d then 16 bytes, byte j = element j (low nibble)   */
/* and element j+16 (high nibble); value d*(code-8).                    */
/* ------------------------------------------------------------------ */
static int block_bytes(int qtype) { return qtype == 0 ? 34 : 18; }

static float block_scale(const uint8_t *blk) { return oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8))); }

/* integer weight of element i (0..31) of one block */
static int block_wq(int qtype, const uint8_t *blk, int i) {
    if (qtype == 0) return (int)(int8_t)blk[2 + i];
    int code = i < 16 ? (blk[2 + i] & 0x0F) : (blk[2 + i - 16] >> 4);
    return code - 8;
}

void oracle_dequant(int qtype, const uint8_t *blocks, int64_t nblocks, float *out) {
    int bb = block_bytes(qtype);
    for (int64_t b = 0; b < nblocks; ++b) {
        const uint8_t *blk = blocks + b * bb;
        float d = block_scale(blk);
        for (int i = 0; i < 32; ++i) out[b * 32 + i] = d * (float)block_wq(qtype, blk, i);
    }
}

/* integer block dot: sum_i wq_i * aq_i over one 32-block (exact in int32) */
static int32_t block_dot(int qtype, const uint8_t *blk, const int8_t *a) {
    int32_t s = 0;
    for (int i = 0; i < 32; ++i) s += block_wq(qtype, blk, i) * (int32_t)a[i];
    return s;
}

/* dots[m][n][b] for weights [N][K/32] blocks and activations q[M][K] */
void oracle_block_dots(int qtype, const uint8_t *w, int64_t N, int64_t K, const int8_t *q, int M, int32_t *dots) {
    int64_t KB = K / 32;
    int bb = block_bytes(qtype);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int m = 0; m < M; ++m)
            for (int64_t b = 0; b < KB; ++b)
                dots[((int64_t)m * N + n) * KB + b] = block_dot(qtype, w + (n * KB + b) * bb, q + (int64_t)m * K + b * 32);
}

/*
 * Multi-position quantised matmul (one weight read serves all M rows):
 *   y[m][n] = residual[m][n] + sum_b d_w[n,b] * d_a[m,b] * dot_b(n, m)
 * accumulated in fp64 and rounded to fp32 once.  absb[m][n] (optional) is the
 * absolute-sum bound |residual| + sum_b |d_w d_a dot_b| used by the tolerance.
 */
void oracle_qmatmul(int qtype, const uint8_t *w, int64_t N, int64_t K, const int8_t *q, const float *scales, int M,
                    const float *residual, float *y, double *absb) {
    int64_t KB = K / 32;
    int bb = block_bytes(qtype);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        for (int m = 0; m < M; ++m) {
            double acc = 0.0, ab = 0.0;
            for (int64_t b = 0; b < KB; ++b) {
                const uint8_t *blk = w + (n * KB + b) * bb;
                int32_t dot = block_dot(qtype, blk, q + (int64_t)m * K + b * 32);
                double t = (double)block_scale(blk) * (double)scales[(int64_t)m * KB + b] * (double)dot;
                acc += t;
                ab += fabs(t);
            }
            if (residual) {
                acc += (double)residual[(int64_t)m * N + n];
                ab += fabs((double)residual[(int64_t)m * N + n]);
            }
            y[(int64_t)m * N + n] = (float)acc;
            if (absb) absb[(int64_t)m * N + n] = ab;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Activation requantisation, per 32-block of a row y:                  */
/*   amax = max |y|, d = amax / 127 (IEEE division),                    */
/*   q = round-half-away-from-zero(y / d) clamped to [-127, 127],       */
/*   q = 0 when d = 0.                                                  */
/* ------------------------------------------------------------------ */
static void requant_row(const float *y, int64_t K, int8_t *q, float *scales) {
    for (int64_t b = 0; b < K / 32; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 32; ++i) {
            float a = fabsf(y[b * 32 + i]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        scales[b] = d;
        for (int i = 0; i < 32; ++i) {
            int v = 0;
            if (d != 0.0f) {
                v = (int)roundf(y[b * 32 + i] / d);
                if (v > 127) v = 127;
                if (v < -127) v = -127;
            }
            q[b * 32 + i] = (int8_t)v;
        }
    }
}

/*
 * RMSNorm + requantisation of M rows (norm_w == NULL: requantisation only).
 * Sum of squares in the canonical order: for each 32-element block, a pairwise
 * tree over its rounded squares x_i*x_i at strides 16, 8, 4, 2, 1 (t[j] +=
 * t[j+s] for j < s); then the same pairwise tree over the K/32 block sums,
 * zero-padded to a power of two of at least 256 slots.  mean = s / K,
 * inv = 1 / sqrt(mean + eps) (correctly rounded division and square root).
 * The normalised row is y = x * inv * w.  Its codes are formed from t = x * w
 * (one rounded multiply): per block c = max|t| / 127 and q = round(t / c), the
 * requantisation above applied to t; the block scale is d = inv * c (one
 * rounded multiply).  In exact arithmetic this is the requantisation of y
 * itself, since the positive row factor inv cancels in y / (max|y| / 127).
 */
void oracle_rmsnorm_quant(const float *x, const float *norm_w, float eps, int M, int64_t K, int8_t *q, float *scales) {
    float *t = (float *)malloc((size_t)K * sizeof(float));
    for (int m = 0; m < M; ++m) {
        const float *xr = x + (int64_t)m * K;
        float *sr = scales + (int64_t)m * (K / 32);
        if (!norm_w) {
            requant_row(xr, K, q + (int64_t)m * K, sr);
            continue;
        }
        const int64_t KB = K / 32;
        int64_t P = 256;
        while (P < KB) P <<= 1;
        float *part = (float *)calloc((size_t)P, sizeof(float));
        for (int64_t b = 0; b < KB; ++b) {
            float sq[32];
            for (int i = 0; i < 32; ++i) sq[i] = xr[b * 32 + i] * xr[b * 32 + i];
            for (int stride = 16; stride >= 1; stride >>= 1)
                for (int j = 0; j < stride; ++j) sq[j] = sq[j] + sq[j + stride];
            part[b] = sq[0];
        }
        for (int64_t stride = P / 2; stride >= 1; stride >>= 1)
            for (int64_t j = 0; j < stride; ++j) part[j] = part[j] + part[j + stride];
        float mean = part[0] / (float)K;
        free(part);
        float inv = 1.0f / sqrtf(mean + eps);
        for (int64_t i = 0; i < K; ++i) t[i] = xr[i] * norm_w[i];
        requant_row(t, K, q + (int64_t)m * K, sr);
        for (int64_t b = 0; b < KB; ++b) sr[b] = inv * sr[b];
    }
    free(t);
}

/* ------------------------------------------------------------------ */
/* Canonical exponential cexp(x), used wherever an exponential feeds an */
/* integer decision.  Cody & Waite argument reduction (W. J. Cody and   */
/* W. Waite, Software Manual for the Elementary Functions, 1980):       */
/*   k = rint(x * log2(e)), r = x - k*ln2 with ln2 split into a 16-bit  */
/*   head (exact times any |k| < 256) and a tail, each applied by one   */
/*   fused multiply-add; e^r by its Taylor series to degree 7 in Horner */
/*   form with fused multiply-adds; scale by 2^k as two exact powers of */
/*   two so that a subnormal result is rounded once.                    */
/* ------------------------------------------------------------------ */
float oracle_cexp(float x) {
    if (x != x) return x;
    if (x > 100.0f) return INFINITY;
    if (x < -104.0f) return 0.0f;
    const float log2e = 1.44269504088896340736f;
    const float ln2_hi = 0.693145751953125f;           /* ln 2 truncated to 16 significant bits */
    const float ln2_lo = 1.42860682030941723212e-6f;   /* ln 2 - ln2_hi */
    float k = rintf(x * log2e);
    float r = fmaf(-k, ln2_hi, x);
    r = fmaf(-k, ln2_lo, r);
    /* 1/n! for n = 7 .. 0 */
    float p = 1.0f / 5040.0f;
    p = fmaf(p, r, 1.0f / 720.0f);
    p = fmaf(p, r, 1.0f / 120.0f);
    p = fmaf(p, r, 1.0f / 24.0f);
    p = fmaf(p, r, 1.0f / 6.0f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int ki = (int)k;
    int k1 = ki / 2, k2 = ki - k1;                      /* both within [-76, 76] */
    return (p * ldexpf(1.0f, k1)) * ldexpf(1.0f, k2);
}

/* ------------------------------------------------------------------ */
/* SiLU gate: h = silu(g) * u with silu(g) = g / (1 + cexp(-g)), each    */
/* operation rounded; h is requantised per 32-block like any activation */
/* ------------------------------------------------------------------ */
void oracle_silu_mul_requant(const float *g, const float *u, int M, int64_t F, int8_t *q, float *scales, float *h_out) {
    float *h = (float *)malloc((size_t)F * sizeof(float));
    for (int m = 0; m < M; ++m) {
        for (int64_t i = 0; i < F; ++i) {
            float gv = g[(int64_t)m * F + i];
            float s = gv / (1.0f + oracle_cexp(-gv));
            h[i] = s * u[(int64_t)m * F + i];
        }
        if (h_out) memcpy(h_out + (int64_t)m * F, h, (size_t)F * sizeof(float));
        requant_row(h, F, q + (int64_t)m * F, scales + (int64_t)m * (F / 32));
    }
    free(h);
}

/* ------------------------------------------------------------------ */
/* Softmax statistics over a vocabulary row, z_i = l_i / T.             */
/* Tiles of 1024 consecutive tokens (the last one shorter).  Per tile:  */
/* m_t = max z, s_t = pairwise tree over 1024 slots (zero padded) of     */
/* cexp(z_i - m_t) at strides 512, 256, ..., 1.  m = max_t m_t and       */
/* Z = sequential fold over t of s_t * cexp(m_t - m).  Argmax is over the */
/* raw logits (temperature free), lowest index among equal maxima.       */
/* p_i = cexp(z_i - m) / Z.                                              */
/* ------------------------------------------------------------------ */
#define TILE 1024

static float tree1024(float *v) {
    for (int s = TILE / 2; s >= 1; s >>= 1)
        for (int j = 0; j < s; ++j) v[j] = v[j] + v[j + s];
    return v[0];
}

static void row_stats(const float *l, int64_t V, float T, float *row_max, float *row_sumexp, int32_t *argmax) {
    int64_t nt = (V + TILE - 1) / TILE;
    float *mt = (float *)malloc((size_t)nt * sizeof(float)), *st = (float *)malloc((size_t)nt * sizeof(float));
    float v[TILE];
    int64_t best = 0;
    float bestv = l[0];
    for (int64_t t = 0; t < nt; ++t) {
        int64_t i0 = t * TILE, n = V - i0 < TILE ? V - i0 : TILE;
        float m = -INFINITY;
        for (int64_t i = 0; i < n; ++i) {
            float z = l[i0 + i] / T;
            if (z > m) m = z;
            if (l[i0 + i] > bestv) { bestv = l[i0 + i]; best = i0 + i; }
        }
        for (int64_t i = 0; i < TILE; ++i) v[i] = i < n ? oracle_cexp(l[i0 + i] / T - m) : 0.0f;
        mt[t] = m;
        st[t] = tree1024(v);
    }
    float m = -INFINITY;
    for (int64_t t = 0; t < nt; ++t) if (mt[t] > m) m = mt[t];
    float Z = 0.0f;
    for (int64_t t = 0; t < nt; ++t) Z = Z + st[t] * oracle_cexp(mt[t] - m);
    if (row_max) *row_max = m;
    if (row_sumexp) *row_sumexp = Z;
    if (argmax) *argmax = (int32_t)best;
    free(mt);
    free(st);
}

void oracle_softmax_stats(const float *logits, int M, int64_t V, float T, float *row_max, float *row_sumexp, int32_t *argmax) {
    for (int m = 0; m < M; ++m)
        row_stats(logits + (int64_t)m * V, V, T, row_max + m, row_sumexp + m, argmax + m);
}

void oracle_softmax_probs(const float *logits, int64_t V, float T, float row_max, float row_sumexp, float *p) {
    for (int64_t i = 0; i < V; ++i) p[i] = oracle_cexp(logits[i] / T - row_max) / row_sumexp;
}

/* ------------------------------------------------------------------ */
/* Greedy acceptance.                                                   */
/* Chain: row 0 holds the current token and rows 1..K the drafts; row i */
/* predicts the token after position i.  n = largest j with             */
/* drafts[i-1] == argmax[i-1] for all i <= j; emit drafts[0..n-1] then  */
/* argmax[n].  Returns the count n + 1.                                 */
/* Tree: node 0 is the root, parent[i] < i.  Node i is accepted when    */
/* its parent is and tokens[i] == argmax[parent[i]].  The deepest       */
/* accepted node (lowest index among equals) ends the emitted path:     */
/* its tokens from the root's child down, then that node's argmax.      */
/* ------------------------------------------------------------------ */
int oracle_accept_greedy_chain(const int32_t *argmax, const int32_t *drafts, int K, int32_t *out) {
    int n = 0;
    while (n < K && drafts[n] == argmax[n]) { out[n] = drafts[n]; ++n; }
    out[n] = argmax[n];
    return n + 1;
}

int oracle_accept_greedy_tree(const int32_t *argmax, const int32_t *tokens, const int32_t *parent, int M, int32_t *out) {
    int *ok = (int *)calloc((size_t)M, sizeof(int)), *depth = (int *)calloc((size_t)M, sizeof(int));
    ok[0] = 1;
    int best = 0;
    for (int i = 1; i < M; ++i) {
        int p = parent[i];
        if (p < 0 || p >= i) continue; /* malformed: not accepted */
        depth[i] = depth[p] + 1;
        ok[i] = ok[p] && tokens[i] == argmax[p];
        if (ok[i] && depth[i] > depth[best]) best = i;
    }
    int d = depth[best];
    for (int i = best, j = d - 1; i != 0; i = parent[i], --j) out[j] = tokens[i];
    out[d] = argmax[best];
    free(ok);
    free(depth);
    return d + 1;
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: */
/* as easy as 1, 2, 3", SC'11).  One round: the two 32x32->64 products  */
/* of counter words 0 and 2 with the round multipliers; the new counter */
/* is (hi(c2*M1) ^ c1 ^ k0, lo(c2*M1), hi(c0*M0) ^ c3 ^ k1, lo(c0*M0)). */
/* The key is bumped by the Weyl constants between rounds.              */
/* ------------------------------------------------------------------ */
void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
        uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c[1] ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c[3] ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
    }
    memcpy(out, c, sizeof(c));
}

/* uniforms of position pos: word 0 -> accept test, word 1 -> residual or bonus draw,
 * u = (word >> 8) * 2^-24 in [0, 1) */
void oracle_uniforms(uint64_t seed, int64_t pos, float *u_acc, float *u_res) {
    uint32_t ctr[4] = {(uint32_t)(uint64_t)pos, (uint32_t)((uint64_t)pos >> 32), 0, 0};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    oracle_philox4x32_10(ctr, key, o);
    *u_acc = (float)(o[0] >> 8) * 5.9604644775390625e-08f;
    *u_res = (float)(o[1] >> 8) * 5.9604644775390625e-08f;
}

/* ------------------------------------------------------------------ */
/* Inverse-CDF draw from unnormalised non-negative weights w[V] with a  */
/* uniform u: S_t = 1024-slot tree sums (as in the softmax tiles),      */
/* S = sequential fold, target = u * S; the first tile whose running    */
/* fold exceeds target (else the last tile with S_t > 0); inside it, 32 */
/* chunks of 32 slots with sequential chunk sums and the same rule;     */
/* inside the chunk, a sequential running sum and the first slot with   */
/* w > 0 where it exceeds the remainder (else the chunk's last slot with */
/* w > 0).  Returns -1 when S is not positive.                          */
/* ------------------------------------------------------------------ */
int32_t oracle_draw_icdf(const float *w, int64_t V, float u) {
    int64_t nt = (V + TILE - 1) / TILE;
    float *S = (float *)malloc((size_t)nt * sizeof(float));
    float v[TILE];
    for (int64_t t = 0; t < nt; ++t) {
        int64_t i0 = t * TILE;
        for (int64_t i = 0; i < TILE; ++i) v[i] = i0 + i < V ? w[i0 + i] : 0.0f;
        S[t] = tree1024(v);
    }
    float tot = 0.0f;
    for (int64_t t = 0; t < nt; ++t) tot = tot + S[t];
    if (!(tot > 0.0f)) { free(S); return -1; }
    float target = u * tot;
    int64_t tsel = -1;
    float C = 0.0f, Cprev = 0.0f;
    for (int64_t t = 0; t < nt; ++t) {
        float Cn = C + S[t];
        if (Cn > target) { tsel = t; Cprev = C; break; }
        C = Cn;
    }
    if (tsel < 0) {
        for (int64_t t = nt - 1; t >= 0; --t) if (S[t] > 0.0f) { tsel = t; break; }
        /* Cprev: the fold up to tile tsel */
        Cprev = 0.0f;
        for (int64_t t = 0; t < tsel; ++t) Cprev = Cprev + S[t];
    }
    free(S);
    float rem = target - Cprev;
    int64_t i0 = tsel * TILE;
    float c[32];
    for (int j = 0; j < 32; ++j) {
        float s = 0.0f;
        for (int i = 0; i < 32; ++i) {
            int64_t idx = i0 + j * 32 + i;
            s = s + (idx < V ? w[idx] : 0.0f);
        }
        c[j] = s;
    }
    int jsel = -1;
    float D = 0.0f, Dprev = 0.0f;
    for (int j = 0; j < 32; ++j) {
        float Dn = D + c[j];
        if (Dn > rem) { jsel = j; Dprev = D; break; }
        D = Dn;
    }
    if (jsel < 0) {
        for (int j = 31; j >= 0; --j) if (c[j] > 0.0f) { jsel = j; break; }
        Dprev = 0.0f;
        for (int j = 0; j < jsel; ++j) Dprev = Dprev + c[j];
    }
    float rem2 = rem - Dprev;
    int64_t base = i0 + (int64_t)jsel * 32;
    float e = 0.0f;
    int64_t last = -1;
    for (int i = 0; i < 32; ++i) {
        int64_t idx = base + i;
        float wi = idx < V ? w[idx] : 0.0f;
        e = e + wi;
        if (wi > 0.0f) {
            last = idx;
            if (e > rem2) return (int32_t)idx;
        }
    }
    return (int32_t)last;
}

/*
 * Rejection-sampling acceptance over K drafts with explicit uniforms
 * (u_acc[i], u_res[i] for i = 0..K).  p_i = softmax(l_i / T) as above;
 * q_i = draft distribution row i, or NULL for a certainty drafter (q one-hot
 * at the draft).  Draft x = drafts[i] is kept iff u_acc[i] * q_i(x) < p_i(x)
 * (equivalent to u < min(1, p/q) because u < 1).  On the first rejection the
 * emitted token is drawn from w = max(0, p_i - q_i) (certainty drafter: p_i
 * with x zeroed) with u_res[i] and the pass stops; if every draft is kept a
 * bonus token is drawn from p_K with u_res[K].  If w sums to zero the draw
 * falls back to p_i.  Returns the count of emitted tokens (kept + 1).
 */
int oracle_accept_sample_u(const float *logits, int64_t V, int K, const float *q_probs, const int32_t *drafts,
                           float T, const float *u_acc, const float *u_res, int32_t *out) {
    float *p = (float *)malloc((size_t)V * sizeof(float)), *w = (float *)malloc((size_t)V * sizeof(float));
    int n = 0;
    for (int i = 0; i <= K; ++i) {
        const float *l = logits + (int64_t)i * V;
        float m, Z;
        row_stats(l, V, T, &m, &Z, NULL);
        oracle_softmax_probs(l, V, T, m, Z, p);
        int32_t tok;
        if (i == K) {
            tok = oracle_draw_icdf(p, V, u_res[i]);
        } else {
            int32_t x = drafts[i];
            float qx = q_probs ? q_probs[(int64_t)i * V + x] : 1.0f;
            if (u_acc[i] * qx < p[x]) { out[n++] = x; continue; }
            for (int64_t j = 0; j < V; ++j) {
                float qj = q_probs ? q_probs[(int64_t)i * V + j] : (j == x ? 1.0f : 0.0f);
                float d = p[j] - qj;
                w[j] = d > 0.0f ? d : 0.0f;
            }
            tok = oracle_draw_icdf(w, V, u_res[i]);
            if (tok < 0) tok = oracle_draw_icdf(p, V, u_res[i]);
        }
        out[n++] = tok;
        break;
    }
    free(p);
    free(w);
    return n;
}

/* The same with the uniforms of positions base_pos .. base_pos + K from
 * Philox4x32-10 keyed by seed (counter = position). */
int oracle_accept_sample(const float *logits, int64_t V, int K, const float *q_probs, const int32_t *drafts,
                         float T, uint64_t seed, int64_t base_pos, int32_t *out) {
    float ua[64], ur[64];
    if (K > 63) return -1;
    for (int i = 0; i <= K; ++i) oracle_uniforms(seed, base_pos + i, &ua[i], &ur[i]);
    return oracle_accept_sample_u(logits, V, K, q_probs, drafts, T, ua, ur, out);
}

/* n_trials independent repetitions at positions base_pos + t*(K+1); writes
 * each trial's count and tokens (row-major [n_trials][K+1]). */
void oracle_accept_sample_trials(const float *logits, int64_t V, int K, const float *q_probs, const int32_t *drafts_per_trial,
                                 float T, uint64_t seed, int64_t base_pos, int64_t n_trials, int32_t *counts, int32_t *tokens) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n_trials; ++t)
        counts[t] = oracle_accept_sample(logits, V, K, q_probs, drafts_per_trial + t * K, T, seed,
                                         base_pos + t * (K + 1), tokens + t * (K + 1));
}

/* ------------------------------------------------------------------ */
/* Rejection sampling against a filtered target (the sampling knobs of  */
/* "Inside OpenJet Engine", API section: temperature, top-k up to 32,   */
/* top-p), read as follows.  Row i: z_j = l_j / T (then z + 0, so that  */
/* -0 and +0 are one value); the candidates are the top_k tokens by z,  */
/* larger z first and, among equal z, the lower token index first.     */
/* With m = z of the first candidate, e_c = cexp(z_c - m) for the       */
/* candidates in that order; S = their sequential sum; the nucleus is   */
/* the shortest prefix of n candidates whose running sum reaches        */
/* top_p * S (n >= 1); S' = the running sum over it; the target is      */
/* p'_c = e_c / S' on the nucleus, 0 elsewhere.  The draft x is kept    */
/* iff u_acc * q(x) < p'(x); on a rejection the token is drawn from     */
/* w_c = max(0, p'_c - q(c)) over the nucleus in candidate order (q     */
/* one-hot at x for a certainty drafter), on a full acceptance from p'  */
/* of row K: W = sequential sum of w, target = u_res * W, the first     */
/* candidate with w > 0 whose running sum exceeds it, else the last one */
/* with w > 0; W not positive falls back to p'.                         */
/* ------------------------------------------------------------------ */

/* candidate j comes before candidate i: larger z, then lower index */
static int cand_before(float zj, int64_t ij, float zi, int64_t ii) { return zj > zi || (zj == zi && ij < ii); }

/* the filtered target of one row: writes up to top_k (token, p') pairs in candidate order; returns n */
int oracle_filter_topk_topp(const float *l, int64_t V, float T, int top_k, float top_p, int32_t *tok, float *prob) {
    int32_t ct[64];
    float cz[64];
    int nc = 0;
    for (int64_t j = 0; j < V; ++j) {
        float z = l[j] / T + 0.0f;
        if (nc == top_k && !cand_before(z, j, cz[nc - 1], ct[nc - 1])) continue;
        int pos = nc < top_k ? nc++ : nc - 1; /* insertion into the sorted list */
        while (pos > 0 && cand_before(z, j, cz[pos - 1], ct[pos - 1])) {
            cz[pos] = cz[pos - 1];
            ct[pos] = ct[pos - 1];
            --pos;
        }
        cz[pos] = z;
        ct[pos] = (int32_t)j;
    }
    float e[64], S = 0.0f;
    for (int c = 0; c < nc; ++c) {
        e[c] = oracle_cexp(cz[c] - cz[0]);
        S = S + e[c];
    }
    const float goal = top_p * S;
    int n = 0;
    float run = 0.0f;
    while (n < nc) {
        run = run + e[n];
        ++n;
        if (run >= goal) break;
    }
    for (int c = 0; c < n; ++c) {
        tok[c] = ct[c];
        prob[c] = e[c] / run;
    }
    return n;
}

/* inverse-CDF draw over n candidate weights in order; -1 if they sum to zero */
static int draw_list(const float *w, int n, float u) {
    float W = 0.0f;
    for (int c = 0; c < n; ++c) W = W + w[c];
    if (!(W > 0.0f)) return -1;
    const float target = u * W;
    float run = 0.0f;
    int last = -1;
    for (int c = 0; c < n; ++c) {
        run = run + w[c];
        if (w[c] > 0.0f) {
            last = c;
            if (run > target) return c;
        }
    }
    return last;
}

int oracle_accept_sample_topk_u(const float *logits, int64_t V, int K, const float *q_probs, const int32_t *drafts,
                                float T, int top_k, float top_p, const float *u_acc, const float *u_res, int32_t *out) {
    int32_t tok[64];
    float p[64], w[64];
    int n = 0;
    for (int i = 0; i <= K; ++i) {
        const int nn = oracle_filter_topk_topp(logits + (int64_t)i * V, V, T, top_k, top_p, tok, p);
        if (i == K) {
            out[n++] = tok[draw_list(p, nn, u_res[i])];
            break;
        }
        const int32_t x = drafts[i];
        float px = 0.0f;
        for (int c = 0; c < nn; ++c)
            if (tok[c] == x) px = p[c];
        const float qx = q_probs ? q_probs[(int64_t)i * V + x] : 1.0f;
        if (u_acc[i] * qx < px) {
            out[n++] = x;
            continue;
        }
        for (int c = 0; c < nn; ++c) {
            const float qc = q_probs ? q_probs[(int64_t)i * V + tok[c]] : (tok[c] == x ? 1.0f : 0.0f);
            const float d = p[c] - qc;
            w[c] = d > 0.0f ? d : 0.0f;
        }
        int c = draw_list(w, nn, u_res[i]);
        if (c < 0) c = draw_list(p, nn, u_res[i]);
        out[n++] = tok[c];
        break;
    }
    return n;
}

int oracle_accept_sample_topk(const float *logits, int64_t V, int K, const float *q_probs, const int32_t *drafts,
                              float T, int top_k, float top_p, uint64_t seed, int64_t base_pos, int32_t *out) {
    float ua[64], ur[64];
    if (K > 63 || top_k < 1 || top_k > 32) return -1;
    for (int i = 0; i <= K; ++i) oracle_uniforms(seed, base_pos + i, &ua[i], &ur[i]);
    return oracle_accept_sample_topk_u(logits, V, K, q_probs, drafts, T, top_k, top_p, ua, ur, out);
}

/* ------------------------------------------------------------------ */
/* Shortlist head ("How Kinetic is fast", section "Shortlist"): a       */
/* smaller copy of the output layer with a proven bound on every row's  */
/* error scores all rows; the best-looking rows are scored exactly,     */
/* which gives a floor, and only rows whose bound reaches the floor are */
/* scored exactly.  Reading: the copy is the 32-weight 4-bit format     */
/* (d = amax / 7.5 rounded to fp16, code = 8 + round-half-away(w / d)   */
/* clamped to [0, 15]) of the Q8_0 head's dequantised weights; the      */
/* bound of row r is E_r = ||w8_r - w4_r||_2 (Cauchy-Schwarz: the copy  */
/* score is within E_r ||a||_2 of the exact one, a the dequantised      */
/* activation row); the floor is F = max_r (s_r - E_r ||a||), s the     */
/* copy scores, and the candidates are the rows with s_r + E_r ||a|| >= F. */
/* Exact scores and the argmax (lowest index among equal maxima) are    */
/* taken over the candidates only.                                      */
/* ------------------------------------------------------------------ */

/* IEEE binary32 -> binary16, round to nearest even; |x| >= 65520 gives infinity */
static uint16_t f32_to_f16_rne_oracle(float x) {
    if (x != x) return 0x7E00u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs((double)x);
    if (a == 0.0) return sign;
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    int e;
    (void)frexp(a, &e);                 /* a = f 2^e, f in [0.5, 1): unit exponent e - 1 */
    int ue = e - 1;
    if (ue < -14) ue = -14;             /* subnormal spacing 2^-24 */
    double q = ldexp(a, 10 - ue);       /* the significand in units of the last place */
    double r = floor(q);
    double frac = q - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    double v = ldexp(r, ue - 10);       /* rounded value */
    (void)frexp(v, &e);
    ue = e - 1;
    if (v < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)ldexp(v, 24));   /* subnormal */
    uint16_t mant = (uint16_t)(ldexp(v, 10 - ue) - 1024.0);
    return (uint16_t)(sign | (uint16_t)((ue + 15) << 10) | mant);
}

/* the 4-bit copy of a Q8_0 matrix [N][K/32], its row bounds E_r and row norms ||w8_r||_2 */
void oracle_shortlist_copy(const uint8_t *q8, int64_t N, int64_t K, uint8_t *q4, float *bound, float *wnorm) {
    int64_t KB = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        double e2 = 0.0, w2 = 0.0;
        for (int64_t b = 0; b < KB; ++b) {
            const uint8_t *blk = q8 + (n * KB + b) * 34;
            uint8_t *out = q4 + (n * KB + b) * 18;
            float w[32], amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                w[i] = block_scale(blk) * (float)block_wq(0, blk, i);
                if (fabsf(w[i]) > amax) amax = fabsf(w[i]);
            }
            /* a scale beyond the largest half (65504) is held there: the copy stays finite */
            const float dq = amax / 7.5f;
            uint16_t d16 = dq < 65520.0f ? f32_to_f16_rne_oracle(dq) : (uint16_t)0x7BFF;
            float d = oracle_f16_to_f32(d16);
            out[0] = (uint8_t)(d16 & 0xFF);
            out[1] = (uint8_t)(d16 >> 8);
            memset(out + 2, 0, 16);
            for (int i = 0; i < 32; ++i) {
                int c = 8;
                if (d > 0.0f) {
                    float t = roundf(w[i] / d) + 8.0f;   /* C99 roundf: halves away from zero */
                    c = t < 0.0f ? 0 : (t > 15.0f ? 15 : (int)t);
                }
                out[2 + (i & 15)] |= (uint8_t)(i < 16 ? c : c << 4);
                double err = (double)w[i] - (double)d * (double)(c - 8);
                e2 += err * err;
                w2 += (double)w[i] * (double)w[i];
            }
        }
        bound[n] = nextafterf((float)sqrt(e2), INFINITY);
        wnorm[n] = nextafterf((float)sqrt(w2), INFINITY);
    }
}

/* exact fp64 score of row n at position m (the definition the shortlist must reproduce) */
static double exact_score(int qtype, const uint8_t *w, int64_t n, int64_t K, const int8_t *q, const float *scales, int m) {
    int64_t KB = K / 32;
    int bb = block_bytes(qtype);
    double acc = 0.0;
    for (int64_t b = 0; b < KB; ++b) {
        const uint8_t *blk = w + (n * KB + b) * bb;
        acc += (double)block_scale(blk) * (double)scales[(int64_t)m * KB + b] *
               (double)block_dot(qtype, blk, q + (int64_t)m * K + b * 32);
    }
    return acc;
}

/* shortlist argmax per position; ncand[m] = candidate rows scored exactly.  Scores in fp64. */
void oracle_shortlist_argmax(const uint8_t *q4, const float *bound, const uint8_t *q8, int64_t N, int64_t K,
                             const int8_t *q, const float *scales, int M, int32_t *argmax, int64_t *ncand) {
    int64_t KB = K / 32;
    double *s = (double *)malloc((size_t)N * sizeof(double));
    for (int m = 0; m < M; ++m) {
        double a2 = 0.0;
        for (int64_t b = 0; b < KB; ++b) {
            double d = scales[(int64_t)m * KB + b];
            for (int i = 0; i < 32; ++i) {
                double v = d * q[(int64_t)m * K + b * 32 + i];
                a2 += v * v;
            }
        }
        const double an = sqrt(a2);
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; ++n) s[n] = exact_score(1, q4, n, K, q, scales, m);
        double F = -INFINITY;
        for (int64_t n = 0; n < N; ++n) {
            double lo = s[n] - (double)bound[n] * an;
            if (lo > F) F = lo;
        }
        int64_t best = -1, nc = 0;
        double bv = -INFINITY;
        for (int64_t n = 0; n < N; ++n) {
            if (s[n] + (double)bound[n] * an < F) continue;
            ++nc;
            double e = exact_score(0, q8, n, K, q, scales, m);
            if (e > bv) { bv = e; best = n; }
        }
        argmax[m] = (int32_t)best;
        ncand[m] = nc;
    }
    free(s);
}

/* ------------------------------------------------------------------ */
/* Decode attention over the K+1 verified positions ("Inside OpenJet    */
/* Engine", section "Cheap drafting, careful state management": split-K */
/* flash decoding of full-attention layers with fp16 K/V and fp32       */
/* accumulation; "How Kinetic is fast", section "Where the guesses come */
/* from": each row of a draft tree sees only its own path; "Speculative */
/* Decoding with Open-Weights Models", section "Engineering the       */
/* Architecture: KV Cache Synchronization": rejected                   */
/* entries are dropped in place).  Reading: the cache holds, per KV     */
/* head, fp16 K and V rows [S_max][D]; the M new positions are appended */
/* at slots L..L+M-1 (fp32 -> fp16, nearest even); query row (i, h)     */
/* sees every committed slot and the new slot L+j iff j is i itself or  */
/* an ancestor of i (chain: j <= i); query head h reads KV head         */
/* h / (H / H_kv); out = sum_j softmax_j(q.k_j / sqrt(D)) v_j.  The     */
/* oracle takes all of it in fp64 from the fp16 values, with no split.  */
/* After acceptance the n entries of the accepted path move to slots    */
/* L..L+n-1 (in path order) and the cache length becomes L+n.           */
/* ------------------------------------------------------------------ */

void oracle_f32_to_f16(const float *x, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_f16_rne_oracle(x[i]);
}

/* k_new, v_new fp32 [M][H_kv][D] -> cache slots [L, L+M) of [H_kv][S_max][D] */
void oracle_kv_append(const float *k_new, const float *v_new, int M, int H_kv, int D, uint16_t *k_cache,
                      uint16_t *v_cache, int64_t S_max, int64_t L) {
    for (int i = 0; i < M; ++i)
        for (int h = 0; h < H_kv; ++h)
            for (int d = 0; d < D; ++d) {
                const int64_t src = ((int64_t)i * H_kv + h) * D + d;
                const int64_t dst = ((int64_t)h * S_max + L + i) * D + d;
                k_cache[dst] = f32_to_f16_rne_oracle(k_new[src]);
                v_cache[dst] = f32_to_f16_rne_oracle(v_new[src]);
            }
}

/* whether new position j is on the path of new position i (parent NULL: a chain) */
static int on_path(const int32_t *parent, int i, int j) {
    if (!parent) return j <= i;
    for (int a = i; a >= 0; a = parent[a])
        if (a == j) return 1;
    return 0;
}

/* q fp32 [M][H][D]; caches fp16 bits [H_kv][S_max][D] holding L + M rows per head;
   out fp64 [M][H][D] */
void oracle_attn_decode(const float *q, const uint16_t *k_cache, const uint16_t *v_cache, int M, int H, int H_kv,
                        int D, int64_t S_max, int64_t L, const int32_t *parent, double *out) {
    const int g = H / H_kv;
    const int64_t NK = L + M;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < M * H; ++r) {
        const int i = r / H, h = r % H, kh = h / g;
        const float *qr = q + (int64_t)r * D;
        double *o = out + (int64_t)r * D;
        double *sc = (double *)malloc((size_t)NK * sizeof(double));
        double mx = -INFINITY;
        for (int64_t j = 0; j < NK; ++j) {
            if (j >= L && !on_path(parent, i, (int)(j - L))) {
                sc[j] = -INFINITY;
                continue;
            }
            const uint16_t *kr = k_cache + ((int64_t)kh * S_max + j) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += (double)qr[d] * (double)oracle_f16_to_f32(kr[d]);
            sc[j] = dot / sqrt((double)D);
            if (sc[j] > mx) mx = sc[j];
        }
        double den = 0.0;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int64_t j = 0; j < NK; ++j) {
            if (sc[j] == -INFINITY) continue;
            const double p = exp(sc[j] - mx);
            den += p;
            const uint16_t *vr = v_cache + ((int64_t)kh * S_max + j) * D;
            for (int d = 0; d < D; ++d) o[d] += p * (double)oracle_f16_to_f32(vr[d]);
        }
        for (int d = 0; d < D; ++d) o[d] /= den;
        free(sc);
    }
}

/* keep the accepted path: slot L+path[t] -> slot L+t for t < n (path increasing, so each move
   reads a slot no earlier move has written) */
void oracle_kv_commit(uint16_t *k_cache, uint16_t *v_cache, int H_kv, int D, int64_t S_max, int64_t L,
                      const int32_t *path, int n) {
    for (int t = 0; t < n; ++t) {
        if (path[t] == t) continue;
        for (int h = 0; h < H_kv; ++h) {
            const int64_t src = ((int64_t)h * S_max + L + path[t]) * D;
            const int64_t dst = ((int64_t)h * S_max + L + t) * D;
            memcpy(k_cache + dst, k_cache + src, (size_t)D * sizeof(uint16_t));
            memcpy(v_cache + dst, v_cache + src, (size_t)D * sizeof(uint16_t));
        }
    }
}

/* ------------------------------------------------------------------ */
/* K-quant formats of the pages' model files (Q4_K_M = Q4_K weights    */
/* with some Q6_K tensors: "Inside OpenJet Engine", section "One GPU    */
/* launch for a speculative cycle" repacks Q6_K; "How Kinetic is fast"  */
/* and "Speculative Decoding with Open-Weights Models" run Q4_K_M).     */
/* The pages print no block layout; the layouts below restate the GGUF  */
/* K-quant formats.  Both hold 256 weights per super-block.             */
/*  Q4_K (144 B): fp16 d, fp16 dmin, 12 bytes of 6-bit scale/min pairs  */
/*   for eight 32-weight sub-blocks, 128 bytes of 4-bit codes.  Pair s:  */
/*   s < 4: scale = b[s] & 63, min = b[s+4] & 63; s >= 4: scale =        */
/*   (b[s+4] & 15) | (b[s-4] >> 6) << 4, min = (b[s+4] >> 4) |          */
/*   (b[s] >> 6) << 4.  Codes: 64-weight chunk c uses bytes 32c..32c+31, */
/*   low nibbles for its first 32 weights, high nibbles for the next 32. */
/*   Weight = d * scale * code - dmin * min.                            */
/*  Q6_K (210 B): 128 bytes ql (low 4 bits), 64 bytes qh (high 2 bits), */
/*   16 int8 scales, fp16 d.  Weight i of half n = i / 128, r = i % 128, */
/*   l = r % 32, k = r / 32: low bits from ql[64n + l + 32 (k & 1)],    */
/*   the low nibble for k < 2 and the high nibble for k >= 2; high bits */
/*   (qh[32n + l] >> 2k) & 3; code = low | high << 4, minus 32.         */
/*   Weight = d * scales[i / 16] * code.                                */
/* With int8 activations per 32-block (q, d_a) the matmul adds, per     */
/* 32-weight activation block, d_a * (d sc dot(code, q) - dmin m sum q) */
/* (Q4_K) or d_a d (sc_lo dot_lo + sc_hi dot_hi) over its two 16-weight */
/* halves (Q6_K): integer dots, then the scales, in fp64.               */
/* ------------------------------------------------------------------ */

enum { OQ4_K = 2, OQ6_K = 3 };

int oracle_kq_block_bytes(int qtype) { return qtype == OQ4_K ? 144 : (qtype == OQ6_K ? 210 : 0); }

static void q4k_scale_min(const uint8_t *b, int s, int *sc, int *mn) {
    if (s < 4) {
        *sc = b[s] & 63;
        *mn = b[s + 4] & 63;
    } else {
        *sc = (b[s + 4] & 15) | ((b[s - 4] >> 6) << 4);
        *mn = (b[s + 4] >> 4) | ((b[s] >> 6) << 4);
    }
}

/* code of weight i (0..255) of a super-block */
static int kq_code(int qtype, const uint8_t *blk, int i) {
    if (qtype == OQ4_K) {
        const int c = i / 64, r = i % 64;
        const uint8_t byte = blk[16 + 32 * c + (r % 32)];
        return r < 32 ? (byte & 15) : (byte >> 4);
    }
    const int n = i / 128, r = i % 128, l = r % 32, k = r / 32;
    const uint8_t lo = blk[64 * n + l + 32 * (k & 1)];
    const int low = k < 2 ? (lo & 15) : (lo >> 4);
    const int high = (blk[128 + 32 * n + l] >> (2 * k)) & 3;
    return (low | (high << 4)) - 32;
}

/* dequantised weights of nblk super-blocks, fp32 */
void oracle_kq_dequant(int qtype, const uint8_t *blocks, int64_t nblk, float *out) {
    const int bb = oracle_kq_block_bytes(qtype);
    for (int64_t n = 0; n < nblk; ++n) {
        const uint8_t *blk = blocks + n * bb;
        for (int i = 0; i < 256; ++i) {
            double v;
            if (qtype == OQ4_K) {
                const double d = oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
                const double dmin = oracle_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
                int sc, mn;
                q4k_scale_min(blk + 4, i / 32, &sc, &mn);
                v = d * sc * kq_code(qtype, blk, i) - dmin * mn;
            } else {
                const double d = oracle_f16_to_f32((uint16_t)(blk[208] | (blk[209] << 8)));
                v = d * (int8_t)blk[192 + i / 16] * kq_code(qtype, blk, i);
            }
            out[n * 256 + i] = (float)v;
        }
    }
}

/* y[m][n] (fp64) = sum over 32-blocks of the factored integer form; w [n_out][k_in/256] blocks,
   q int8 [M][k_in], scales fp32 [M][k_in/32].  absb (nullable) receives the absolute sum of the same
   terms (Q4_K: |d_a| (|d sc dot| + |dmin m sum|); Q6_K: |d_a d| (|sc_lo dot_lo| + |sc_hi dot_hi|)), the
   scale of the rounding error any order of evaluating them in fp32 can make (tolerance reading R5). */
void oracle_kq_matmul(int qtype, const uint8_t *w, int64_t n_out, int64_t k_in, const int8_t *q,
                      const float *scales, int M, double *y, double *absb) {
    const int bb = oracle_kq_block_bytes(qtype);
    const int64_t SB = k_in / 256, KB = k_in / 32;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < n_out; ++n) {
        for (int m = 0; m < M; ++m) {
            double acc = 0.0, ab = 0.0;
            for (int64_t b = 0; b < KB; ++b) {
                const uint8_t *blk = w + (n * SB + b / 8) * bb;
                const int s = (int)(b % 8);  /* 32-weight sub-block within the super-block */
                const int8_t *qa = q + (int64_t)m * k_in + b * 32;
                const double da = scales[(int64_t)m * KB + b];
                if (qtype == OQ4_K) {
                    int64_t dot = 0, sum = 0;
                    for (int i = 0; i < 32; ++i) {
                        dot += (int64_t)kq_code(qtype, blk, 32 * s + i) * qa[i];
                        sum += qa[i];
                    }
                    int sc, mn;
                    q4k_scale_min(blk + 4, s, &sc, &mn);
                    const double d = oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
                    const double dmin = oracle_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
                    acc += da * (d * sc * (double)dot - dmin * mn * (double)sum);
                    ab += fabs(da) * (fabs(d * sc * (double)dot) + fabs(dmin * mn * (double)sum));
                } else {
                    int64_t lo = 0, hi = 0;
                    for (int i = 0; i < 16; ++i) lo += (int64_t)kq_code(qtype, blk, 32 * s + i) * qa[i];
                    for (int i = 16; i < 32; ++i) hi += (int64_t)kq_code(qtype, blk, 32 * s + i) * qa[i];
                    const double d = oracle_f16_to_f32((uint16_t)(blk[208] | (blk[209] << 8)));
                    acc += da * d * ((int8_t)blk[192 + 2 * s] * (double)lo + (int8_t)blk[192 + 2 * s + 1] * (double)hi);
                    ab += fabs(da * d) * (fabs((int8_t)blk[192 + 2 * s] * (double)lo) +
                                          fabs((int8_t)blk[192 + 2 * s + 1] * (double)hi));
                }
            }
            y[(int64_t)m * n_out + n] = acc;
            if (absb) absb[(int64_t)m * n_out + n] = ab;
        }
    }
}

/* The accepted path of the greedy tree rule above as node indices, root first: the nodes whose
   K/V rows the cache keeps ("Speculative Decoding with Open-Weights Models", section
   "Engineering the Architecture: KV Cache Synchronization").  Returns the node count. */
int oracle_accept_greedy_tree_path(const int32_t *argmax, const int32_t *tokens, const int32_t *parent, int M,
                                   int32_t *path) {
    int *ok = (int *)calloc((size_t)M, sizeof(int)), *depth = (int *)calloc((size_t)M, sizeof(int));
    ok[0] = 1;
    int best = 0;
    for (int i = 1; i < M; ++i) {
        const int p = parent[i];
        if (p < 0 || p >= i) continue;
        depth[i] = depth[p] + 1;
        ok[i] = ok[p] && tokens[i] == argmax[p];
        if (ok[i] && depth[i] > depth[best]) best = i;
    }
    const int d = depth[best];
    for (int i = best, j = d; j >= 0; i = parent[i], --j) path[j] = i;
    free(ok);
    free(depth);
    return d + 1;
}
