/*
 * sdgen.c - seeded synthetic inputs for the speculative-decoding verify pass.
 *
 * This file synthesises INPUTS only: normal variates from a counter-based
 * hash, and the offline block quantisation that turns fp32 weights into the
 * GGUF-order block bytes a model file would hold (Q8_0: fp16 d + 32 x int8,
 * 34 B; 4-bit: fp16 d + 16 bytes of nibbles, 18 B).  Nothing of the verify
 * pass itself (dots, matmul, norm, requantisation of activations, softmax,
 * acceptance) lives here.  Both the CUDA path and the CPU oracle consume the
 * bytes this produces; neither is linked into it.
 *
 * Random numbers: element i of a stream keyed by k is a pure function of
 * (k, i).  Bits come from hashing (k, i, attempt) with the SplitMix64 finaliser
 * (Steele, Lea, Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014); the ziggurat method turns them into N(0,1) variates.  Streams
 * can therefore be generated in any chunking and any number of threads with
 * identical results.
 */
#define _GNU_SOURCE
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* 64 random bits number `a` for element i of stream key */
static inline uint64_t draw64(uint64_t key, uint64_t i, uint64_t a) {
    return mix64(key ^ mix64(i * 0x9E3779B97F4A7C15ull + a * 0xD6E8FEB86659FD93ull + 0x632BE59BD9B4E019ull));
}

/* Ziggurat tables for the standard normal, 128 layers (Marsaglia & Tsang,
 * "The Ziggurat Method for Generating Random Variables", J. Stat. Softw. 2000):
 * right edge r = 3.442619855899, layer area v = 9.91256303526217e-3. */
static uint32_t zk[128];
static double zw[128], zf[128];
static pthread_once_t z_once = PTHREAD_ONCE_INIT;

static void zig_setup(void) {
    const double m1 = 2147483648.0;
    double dn = 3.442619855899, tn = dn, vn = 9.91256303526217e-3;
    double q = vn / exp(-0.5 * dn * dn);
    zk[0] = (uint32_t)((dn / q) * m1);
    zk[1] = 0;
    zw[0] = q / m1;
    zw[127] = dn / m1;
    zf[0] = 1.0;
    zf[127] = exp(-0.5 * dn * dn);
    for (int i = 126; i >= 1; --i) {
        dn = sqrt(-2.0 * log(vn / dn + exp(-0.5 * dn * dn)));
        zk[i + 1] = (uint32_t)((dn / tn) * m1);
        tn = dn;
        zf[i] = exp(-0.5 * dn * dn);
        zw[i] = dn / m1;
    }
}

static inline double u53(uint64_t h) { return (double)(h >> 11) * (1.0 / 9007199254740992.0); }

/* N(0,1) variate for element i of stream key; the attempts of the rejection
 * loop draw from (key, i, attempt), so the value is a pure function of (key, i). */
static inline double normal_at(uint64_t key, uint64_t i) {
    uint64_t a = 0;
    for (;;) {
        uint64_t h = draw64(key, i, a++);
        int32_t hz = (int32_t)(uint32_t)h;
        uint32_t iz = (uint32_t)(h >> 32) & 127u;
        uint32_t mag = hz < 0 ? (uint32_t)(-(int64_t)hz) : (uint32_t)hz;
        double x = (double)hz * zw[iz];
        if (mag < zk[iz]) return x;
        if (iz == 0) { /* tail beyond r */
            const double r = 3.442619855899;
            double xt, yt;
            do {
                xt = -log(1.0 - u53(draw64(key, i, a++))) / r;
                yt = -log(1.0 - u53(draw64(key, i, a++)));
            } while (yt + yt < xt * xt);
            return hz > 0 ? r + xt : -r - xt;
        }
        if (zf[iz] + u53(draw64(key, i, a++)) * (zf[iz - 1] - zf[iz]) < exp(-0.5 * x * x)) return x;
    }
}

/* out[j] = mean + std * N_k(start + j), j < n */
void sdgen_normal_f32(uint64_t key, int64_t start, int64_t n, float mean, float std, float *out) {
    pthread_once(&z_once, zig_setup);
    for (int64_t j = 0; j < n; ++j) out[j] = (float)((double)mean + (double)std * normal_at(key, (uint64_t)(start + j)));
}

/* ---- fp16 encode, round to nearest even (IEEE 754 binary16) ---- */
static uint16_t f32_to_f16_rne(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax >= 0x7F800000u) return (uint16_t)(sign | 0x7C00u | (ax > 0x7F800000u ? 0x200u : 0));
    if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* rounds to >= 65520 -> inf */
    if (ax < 0x38800000u) {                                   /* result subnormal or zero */
        if (ax < 0x33000000u) return (uint16_t)sign;          /* < 2^-25: rounds to 0 */
        uint32_t e = ax >> 23, m = (ax & 0x7FFFFFu) | 0x800000u;
        uint32_t shift = 126u - e; /* value = m * 2^(e-150); want units of 2^-24 */
        uint32_t q = m >> shift, rem = m & ((1u << shift) - 1u), half = 1u << (shift - 1u);
        if (rem > half || (rem == half && (q & 1u))) q++;
        return (uint16_t)(sign | q);
    }
    uint32_t e = (ax >> 23) - 112u, m = ax & 0x7FFFFFu;
    uint32_t q = (e << 10) | (m >> 13), rem = m & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (q & 1u))) q++;
    return (uint16_t)(sign | q);
}

/* round half away from zero of an fp32 quotient, evaluated exactly */
static inline int round_half_away(float v) {
    double d = (double)v;
    return (int)(d < 0 ? -floor(-d + 0.5) : floor(d + 0.5));
}

/* One 32-weight block -> GGUF block bytes.
 * Q8_0:  d = amax/127 (fp32 division), q = round(w/d) clamped to +-127, store fp16(d).
 * 4-bit: d = amax/7.5, code = clamp(round(w/d)+8, 0, 15); byte j holds element j in
 *        its low nibble and element j+16 in its high nibble; store fp16(d). */
static void quant_block(int qtype, const float *w, uint8_t *dst) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) { float a = fabsf(w[i]); if (a > amax) amax = a; }
    float d = amax / (qtype == 0 ? 127.0f : 7.5f);
    uint16_t d16 = f32_to_f16_rne(d);
    dst[0] = (uint8_t)(d16 & 0xFF);
    dst[1] = (uint8_t)(d16 >> 8);
    if (qtype == 0) {
        for (int i = 0; i < 32; ++i) {
            int q = 0;
            if (d != 0.0f) { q = round_half_away(w[i] / d); if (q > 127) q = 127; if (q < -127) q = -127; }
            dst[2 + i] = (uint8_t)(int8_t)q;
        }
    } else {
        int code[32];
        for (int i = 0; i < 32; ++i) {
            int c = 8;
            if (d != 0.0f) { c = round_half_away(w[i] / d) + 8; if (c > 15) c = 15; if (c < 0) c = 0; }
            code[i] = c;
        }
        for (int j = 0; j < 16; ++j) dst[2 + j] = (uint8_t)(code[j] | (code[j + 16] << 4));
    }
}

static int64_t block_bytes(int qtype) { return qtype == 0 ? 34 : 18; }

/* quantise an fp32 matrix [n][k] (k % 32 == 0) into GGUF-order blocks [n][k/32] */
void sdgen_quantize(int qtype, const float *w, int64_t n, int64_t k, uint8_t *out) {
    int64_t kb = k / 32, bb = block_bytes(qtype);
    for (int64_t r = 0; r < n; ++r)
        for (int64_t b = 0; b < kb; ++b) quant_block(qtype, w + r * k + b * 32, out + (r * kb + b) * bb);
}

/* ---- fused generate + quantise, multithreaded over fixed row chunks ---- */
typedef struct {
    int qtype;
    uint64_t key;
    int64_t n, k;
    float mean, std;
    uint8_t *out;
    int64_t row0, row1;
} gen_job;

static void *gen_worker(void *arg) {
    gen_job *j = (gen_job *)arg;
    int64_t kb = j->k / 32, bb = block_bytes(j->qtype);
    float *row = (float *)malloc((size_t)j->k * sizeof(float));
    if (!row) return (void *)1;
    for (int64_t r = j->row0; r < j->row1; ++r) {
        sdgen_normal_f32(j->key, r * j->k, j->k, j->mean, j->std, row);
        for (int64_t b = 0; b < kb; ++b) quant_block(j->qtype, row + b * 32, j->out + (r * kb + b) * bb);
    }
    free(row);
    return 0;
}

/* Weights W[n][k] ~ N(mean, std^2) from stream `key` (element r*k+c), quantised
 * into GGUF-order blocks.  The result does not depend on nthreads. */
int sdgen_normal_quantized(int qtype, uint64_t key, int64_t n, int64_t k, float mean, float std,
                           uint8_t *out, int nthreads) {
    if (k % 32 != 0 || n < 0) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = n > 0 ? (int)n : 1;
    pthread_t th[256];
    gen_job jobs[256];
    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (gen_job){qtype, key, n, k, mean, std, out, n * t / nthreads, n * (t + 1) / nthreads};
        if (pthread_create(&th[t], 0, gen_worker, &jobs[t]) != 0) { gen_worker(&jobs[t]); th[t] = 0; }
    }
    for (int t = 0; t < nthreads; ++t) {
        if (th[t]) { void *r = 0; pthread_join(th[t], &r); if (r) rc = 1; }
    }
    return rc;
}

/* raw 32-bit hash stream: out[j] = H_k(start + j) (uniform on [0, 2^32)) */
void sdgen_u32(uint64_t key, int64_t start, int64_t n, uint32_t *out) {
    for (int64_t j = 0; j < n; ++j) {
        uint64_t i = (uint64_t)(start + j);
        out[j] = (uint32_t)(mix64(key ^ mix64(i * 0xD1B54A32D192ED03ull + 0x8CB92BA72F3D8DD7ull)) >> 32);
    }
}
