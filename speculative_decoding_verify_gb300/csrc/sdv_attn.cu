// sdv_attn.cu - decode attention of the verify pass over the K+1 positions ("Inside OpenJet
// Engine", section "Cheap drafting, careful state management": split-K flash decoding of the
// full-attention layers, fp16 K/V with fp32 accumulation; "How Kinetic is fast", section "Where
// the guesses come from": each row of a draft tree sees only its own path; "Speculative Decoding
// with Open-Weights Models", section "Engineering the Architecture: KV Cache Synchronization":
// rejected entries are dropped in place).
//
// Cache: per KV head, fp16 K and V rows [S_max][D]; L committed rows, then the M new positions.
// Query row (i, h) sees every committed row and new row j iff j is on i's path; query head h
// reads KV head h / (H / H_kv); out = softmax(q k^T / sqrt(D)) v.
//
// The context is read once per KV head for all its query rows (M positions x the heads of the
// group, up to 8 per CTA).  It is HBM-bound (about M/2 fp32 multiply-adds per cache byte at
// M = 5), so it runs on the CUDA cores in fp32: a warp takes two keys per step, 16 lanes per key
// with D/16 elements each for q.k (reduced by shuffles), then all 32 lanes with D/32 elements
// each for the running p v; the next pair's K and V are loaded before the current pair is used.
// The keys are split into chunks, one CTA of 4 warps per (chunk, query group, KV head); each CTA
// leaves an unnormalised (max, sum, o) per row and a second kernel combines the chunks.
// Scores are kept in log2 units (q is scaled by log2(e)/sqrt(D) once) and exponentials are exp2f.
#include "sdv_common.cuh"

namespace sdv {

constexpr int AT_TQ = 8;     // query rows per CTA
constexpr int AT_WARPS = 4;  // warps per attention CTA
constexpr int AT_MIN_CHUNK_PAIRS = 32;
constexpr float AT_NEG = -3.402823466e38f;  // running-max start: finite, below every score

struct AttnArgs {
    const float *q;         // [M][H][D]
    const __half *kc, *vc;  // [H_kv][S_max][D]
    const int32_t *parent;  // [M] or nullptr (chain)
    float *part_ml;         // [H_kv][QG][S][AT_TQ][2]: running max (log2 units), sum of exp2
    float *part_o;          // [H_kv][QG][S][AT_TQ][D]: unnormalised output
    float *out;             // [M][H][D]
    int64_t S_max, L, NK;   // NK = L + M keys
    int64_t chunk_pairs;    // key pairs per chunk
    int32_t M, H, H_kv, g;  // g = H / H_kv
    int32_t QG, S;          // query groups per KV head, key chunks
    float qscale;           // log2(e) / sqrt(D)
    int *status;
};

// bit j set: new row L+j is visible to position i (i itself and its ancestors)
__device__ __forceinline__ uint32_t path_mask(const AttnArgs &a, int i) {
    if (!a.parent) return (2u << i) - 1u;
    uint32_t m = 0;
    int x = i;
    for (int step = 0; step <= i && x >= 0; ++step) {
        m |= 1u << x;
        const int p = a.parent[x];
        if (p >= x) {  // parents come before their children; anything else is a bad tree
            set_status(a.status, SD_EDEVICE);
            break;
        }
        x = p;
    }
    return m;
}

template <int D>
struct KvLane {
    static constexpr int DL = D / 16;  // q.k elements per lane (16 lanes per key)
    static constexpr int DV = D / 32;  // p v elements per lane
};

template <int DL>
__device__ __forceinline__ void load_k(const __half *row, int hl, float (&kf)[DL]) {
    if constexpr (DL == 8) {
        const uint4 r = __ldg(reinterpret_cast<const uint4 *>(row + hl * 8));
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[e]));
            kf[2 * e] = f.x;
            kf[2 * e + 1] = f.y;
        }
    } else {
        const uint2 r = __ldg(reinterpret_cast<const uint2 *>(row + hl * 4));
        const uint32_t w[2] = {r.x, r.y};
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[e]));
            kf[2 * e] = f.x;
            kf[2 * e + 1] = f.y;
        }
    }
}

template <int DV>
__device__ __forceinline__ void load_v(const __half *row, int lane, float (&vf)[DV]) {
    if constexpr (DV == 4) {
        const uint2 r = __ldg(reinterpret_cast<const uint2 *>(row + lane * 4));
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
        vf[0] = f0.x;
        vf[1] = f0.y;
        vf[2] = f1.x;
        vf[3] = f1.y;
    } else {
        const uint32_t r = __ldg(reinterpret_cast<const unsigned int *>(row + lane * 2));
        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&r));
        vf[0] = f.x;
        vf[1] = f.y;
    }
}

template <int D>
__global__ void __launch_bounds__(32 * AT_WARPS) attn_partial_kernel(const AttnArgs a) {
    constexpr int DL = KvLane<D>::DL, DV = KvLane<D>::DV;
    __shared__ float sm_m[AT_WARPS][AT_TQ], sm_l[AT_WARPS][AT_TQ];
    __shared__ float sm_o[AT_WARPS][AT_TQ][D];
    pdl_wait();
    pdl_launch_dependents();
    const int sc = blockIdx.x, qg = blockIdx.y, kh = blockIdx.z;
    const int warp = static_cast<int>(threadIdx.x) / 32, lane = static_cast<int>(threadIdx.x) & 31;
    const int half = lane >> 4, hl = lane & 15;
    const int rows = a.M * a.g;

    float qr[AT_TQ][DL];
    uint32_t vis[AT_TQ];
#pragma unroll
    for (int t = 0; t < AT_TQ; ++t) {
        const int tg = qg * AT_TQ + t;
        vis[t] = 0;
#pragma unroll
        for (int e = 0; e < DL; ++e) qr[t][e] = 0.0f;
        if (tg < rows) {
            const int i = tg / a.g, h = kh * a.g + tg % a.g;
            const float *qp = a.q + (static_cast<int64_t>(i) * a.H + h) * D + hl * DL;
#pragma unroll
            for (int e = 0; e < DL; ++e) qr[t][e] = qp[e] * a.qscale;
            vis[t] = path_mask(a, i);
        }
    }

    float m[AT_TQ], l[AT_TQ], o[AT_TQ][DV];
#pragma unroll
    for (int t = 0; t < AT_TQ; ++t) {
        m[t] = AT_NEG;
        l[t] = 0.0f;
#pragma unroll
        for (int e = 0; e < DV; ++e) o[t][e] = 0.0f;
    }

    const int64_t NP = (a.NK + 1) / 2;
    const int64_t p_end = min(NP, (static_cast<int64_t>(sc) + 1) * a.chunk_pairs);
    const __half *kbase = a.kc + static_cast<int64_t>(kh) * a.S_max * D;
    const __half *vbase = a.vc + static_cast<int64_t>(kh) * a.S_max * D;
    int64_t p = static_cast<int64_t>(sc) * a.chunk_pairs + warp;

    // registers of the pair in hand and of the next one
    float kf[DL], vA[DV], vB[DV];
    auto fetch = [&](int64_t pp, float (&k_)[DL], float (&va)[DV], float (&vb)[DV]) {
        const int64_t jA = 2 * pp, jB = jA + 1, jm = jA + half;
        if (jm < a.NK) {
            load_k<DL>(kbase + jm * D, hl, k_);
        } else {
#pragma unroll
            for (int e = 0; e < DL; ++e) k_[e] = 0.0f;
        }
        load_v<DV>(vbase + jA * D, lane, va);
        if (jB < a.NK) {
            load_v<DV>(vbase + jB * D, lane, vb);
        } else {
#pragma unroll
            for (int e = 0; e < DV; ++e) vb[e] = 0.0f;
        }
    };
    if (p < p_end) fetch(p, kf, vA, vB);
    while (p < p_end) {
        const int64_t pn = p + AT_WARPS;
        float kn[DL], vAn[DV], vBn[DV];
        if (pn < p_end) fetch(pn, kn, vAn, vBn);
        const int64_t jA = 2 * p, jB = jA + 1;
#pragma unroll
        for (int t = 0; t < AT_TQ; ++t) {
            float s = 0.0f;
#pragma unroll
            for (int e = 0; e < DL; ++e) s = fmaf(qr[t][e], kf[e], s);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            const float so = __shfl_xor_sync(0xffffffffu, s, 16);
            float sA = half ? so : s, sB = half ? s : so;
            if (jA >= a.L && !((vis[t] >> static_cast<int>(jA - a.L)) & 1u)) sA = -INFINITY;
            if (jB >= a.NK || (jB >= a.L && !((vis[t] >> static_cast<int>(jB - a.L)) & 1u))) sB = -INFINITY;
            const float mn = fmaxf(m[t], fmaxf(sA, sB));
            const float alpha = exp2f(m[t] - mn);
            const float pA = exp2f(sA - mn), pB = exp2f(sB - mn);
            l[t] = fmaf(l[t], alpha, pA + pB);
            m[t] = mn;
#pragma unroll
            for (int e = 0; e < DV; ++e) o[t][e] = fmaf(pB, vB[e], fmaf(pA, vA[e], o[t][e] * alpha));
        }
        if (pn < p_end) {
#pragma unroll
            for (int e = 0; e < DL; ++e) kf[e] = kn[e];
#pragma unroll
            for (int e = 0; e < DV; ++e) {
                vA[e] = vAn[e];
                vB[e] = vBn[e];
            }
        }
        p = pn;
    }

    // the CTA's warps into one (max, sum, o) per row
#pragma unroll
    for (int t = 0; t < AT_TQ; ++t) {
        if (lane == 0) {
            sm_m[warp][t] = m[t];
            sm_l[warp][t] = l[t];
        }
#pragma unroll
        for (int e = 0; e < DV; ++e) sm_o[warp][t][lane * DV + e] = o[t][e];
    }
    __syncthreads();
    const int64_t base = ((static_cast<int64_t>(kh) * a.QG + qg) * a.S + sc) * AT_TQ;
    for (int idx = threadIdx.x; idx < AT_TQ * D; idx += 32 * AT_WARPS) {
        const int t = idx / D, d = idx % D;
        float mx = sm_m[0][t];
#pragma unroll
        for (int w = 1; w < AT_WARPS; ++w) mx = fmaxf(mx, sm_m[w][t]);
        float ov = 0.0f, lv = 0.0f;
#pragma unroll
        for (int w = 0; w < AT_WARPS; ++w) {
            const float f = exp2f(sm_m[w][t] - mx);
            ov = fmaf(sm_o[w][t][d], f, ov);
            lv = fmaf(sm_l[w][t], f, lv);
        }
        a.part_o[(base + t) * D + d] = ov;
        if (d == 0) {
            a.part_ml[(base + t) * 2] = mx;
            a.part_ml[(base + t) * 2 + 1] = lv;
        }
    }
}

// combine the chunks of one (KV head, query group): one warp per query row, lanes over d
template <int D>
__global__ void __launch_bounds__(32 * AT_TQ) attn_combine_kernel(const AttnArgs a) {
    constexpr int DV = KvLane<D>::DV;
    pdl_wait();
    pdl_launch_dependents();
    const int qg = blockIdx.x, kh = blockIdx.y;
    const int t = static_cast<int>(threadIdx.x) / 32, lane = static_cast<int>(threadIdx.x) & 31;
    const int tg = qg * AT_TQ + t;
    if (tg >= a.M * a.g) return;
    const int i = tg / a.g, h = kh * a.g + tg % a.g;
    const int64_t base = (static_cast<int64_t>(kh) * a.QG + qg) * a.S;
    float mx = AT_NEG;
    for (int s = lane; s < a.S; s += 32) mx = fmaxf(mx, a.part_ml[((base + s) * AT_TQ + t) * 2]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float lv = 0.0f, ov[DV];
#pragma unroll
    for (int e = 0; e < DV; ++e) ov[e] = 0.0f;
    for (int s = 0; s < a.S; ++s) {
        const int64_t r = (base + s) * AT_TQ + t;
        const float f = exp2f(a.part_ml[r * 2] - mx);
        lv = fmaf(a.part_ml[r * 2 + 1], f, lv);
#pragma unroll
        for (int e = 0; e < DV; ++e) ov[e] = fmaf(a.part_o[r * D + lane * DV + e], f, ov[e]);
    }
    float *op = a.out + (static_cast<int64_t>(i) * a.H + h) * D + lane * DV;
#pragma unroll
    for (int e = 0; e < DV; ++e) op[e] = ov[e] / lv;
}

// new K/V rows: fp32 [M][H_kv][D] -> fp16 (nearest even) cache slots [L, L+M)
__global__ void kv_append_kernel(const float *k_new, const float *v_new, int32_t M, int32_t H_kv, int32_t D,
                                 __half *kc, __half *vc, int64_t S_max, int64_t L) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t n = static_cast<int64_t>(M) * H_kv * D;
    for (int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < n;
         x += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t d = x % D, h = (x / D) % H_kv, i = x / (static_cast<int64_t>(D) * H_kv);
        const int64_t dst = (h * S_max + L + i) * D + d;
        kc[dst] = __float2half_rn(k_new[x]);
        vc[dst] = __float2half_rn(v_new[x]);
    }
}

constexpr int KC_MAXD = 256;

// keep the accepted path: rows L+path[t] -> L+t, t < n = *count; one CTA per KV head stages the
// rows in shared memory first, so moves whose source another move overwrites stay correct
__global__ void __launch_bounds__(128) kv_commit_kernel(__half *kc, __half *vc, int32_t D, int64_t S_max, int64_t L,
                                                        int32_t M, const int32_t *path, const int32_t *count,
                                                        int *status) {
    __shared__ __half sk[16][KC_MAXD], sv[16][KC_MAXD];
    __shared__ int ok;
    pdl_wait();
    pdl_launch_dependents();
    const int n = *count;
    if (threadIdx.x == 0) {
        int good = n >= 1 && n <= M;
        for (int t = 0; good && t < n; ++t)
            good = path[t] >= 0 && path[t] < M && (t == 0 || path[t] > path[t - 1]);
        ok = good;
        if (!good && blockIdx.x == 0) set_status(status, SD_EDEVICE);
    }
    __syncthreads();
    if (!ok) return;
    const int64_t head = static_cast<int64_t>(blockIdx.x) * S_max;
    for (int x = threadIdx.x; x < n * D; x += blockDim.x) {
        const int t = x / D, d = x % D;
        const int64_t src = (head + L + path[t]) * D + d;
        sk[t][d] = kc[src];
        sv[t][d] = vc[src];
    }
    __syncthreads();
    for (int x = threadIdx.x; x < n * D; x += blockDim.x) {
        const int t = x / D, d = x % D;
        const int64_t dst = (head + L + t) * D + d;
        kc[dst] = sk[t][d];
        vc[dst] = sv[t][d];
    }
}

struct AttnPlan {
    int32_t QG, S;
    int64_t chunk_pairs;
    size_t off_o, total;
};

static bool attn_plan(int32_t M, int32_t H, int32_t H_kv, int32_t D, int64_t L, AttnPlan &p) {
    if (M < 1 || M > 16 || H_kv < 1 || H < H_kv || H % H_kv || (D != 64 && D != 128) || L < 0) return false;
    const int sms = num_sms();
    if (sms < 1) return false;
    const int64_t rows = static_cast<int64_t>(M) * (H / H_kv);
    p.QG = static_cast<int32_t>((rows + AT_TQ - 1) / AT_TQ);
    const int64_t NP = (L + M + 1) / 2;
    // about 4 CTAs (16 warps) per SM over all (chunk, query group, KV head)
    const int64_t per = static_cast<int64_t>(p.QG) * H_kv;
    const int64_t want = (4 * static_cast<int64_t>(sms) + per - 1) / per;
    int64_t cp = (NP + want - 1) / want;
    if (cp < AT_MIN_CHUNK_PAIRS) cp = AT_MIN_CHUNK_PAIRS;
    p.chunk_pairs = cp;
    p.S = static_cast<int32_t>((NP + cp - 1) / cp);  // <= want, whatever the context
    // partials sized for `want` chunks, so one workspace serves every context length
    const size_t nrow = static_cast<size_t>(H_kv) * p.QG * static_cast<size_t>(want) * AT_TQ;
    p.off_o = (nrow * 2 * sizeof(float) + 255) & ~static_cast<size_t>(255);
    p.total = p.off_o + ((nrow * D * sizeof(float) + 255) & ~static_cast<size_t>(255));
    return true;
}

}  // namespace sdv

using namespace sdv;

extern "C" {

size_t sd_attn_workspace_bytes(int32_t M, int32_t H, int32_t H_kv, int32_t D, int64_t L) {
    AttnPlan p;
    return attn_plan(M, H, H_kv, D, L, p) ? p.total : 0;
}

sd_status sd_kv_append(const float *k_new, const float *v_new, int32_t M, int32_t H_kv, int32_t D, void *k_cache,
                       void *v_cache, int64_t S_max, int64_t L, sd_stream_t stream) {
    if (!k_new || !v_new || !k_cache || !v_cache) return SD_EINVAL;
    if (M < 1 || M > 16 || H_kv < 1 || D < 1 || L < 0 || S_max < L + M) return SD_EINVAL;
    if (!aligned(k_new, 4) || !aligned(v_new, 4) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return SD_EINVAL;
    const int64_t n = static_cast<int64_t>(M) * H_kv * D;
    const int grid = static_cast<int>((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    return launch(kv_append_kernel, dim3(grid), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream), k_new, v_new,
                  M, H_kv, D, static_cast<__half *>(k_cache), static_cast<__half *>(v_cache), S_max, L) ==
                   cudaSuccess
               ? SD_OK
               : SD_ECUDA;
}

sd_status sd_attn_decode(const float *q, const void *k_cache, const void *v_cache, int32_t M, int32_t H,
                         int32_t H_kv, int32_t D, int64_t S_max, int64_t L, const int32_t *parent, float *out,
                         void *workspace, size_t ws_bytes, sd_stream_t stream) {
    if (!q || !k_cache || !v_cache || !out || !workspace) return SD_EINVAL;
    if (M < 1 || H_kv < 1 || H < H_kv || H % H_kv || L < 0 || S_max < L + M) return SD_EINVAL;
    if (M > 16 || (D != 64 && D != 128)) return SD_EUNSUPPORTED;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(workspace, 256))
        return SD_EINVAL;
    AttnPlan p;
    if (!attn_plan(M, H, H_kv, D, L, p)) return SD_EINVAL;
    if (ws_bytes < p.total) return SD_EINVAL;
    int *st = status_ptr();
    if (!st) return SD_ECUDA;
    AttnArgs a = {};
    a.q = q;
    a.kc = static_cast<const __half *>(k_cache);
    a.vc = static_cast<const __half *>(v_cache);
    a.parent = parent;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.part_ml = reinterpret_cast<float *>(ws);
    a.part_o = reinterpret_cast<float *>(ws + p.off_o);
    a.out = out;
    a.S_max = S_max;
    a.L = L;
    a.NK = L + M;
    a.chunk_pairs = p.chunk_pairs;
    a.M = M;
    a.H = H;
    a.H_kv = H_kv;
    a.g = H / H_kv;
    a.QG = p.QG;
    a.S = p.S;
    a.qscale = 1.4426950408889634f / sqrtf(static_cast<float>(D));
    a.status = st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const dim3 grid(p.S, p.QG, H_kv);
    cudaError_t e;
    if (D == 128) {
        e = launch(attn_partial_kernel<128>, grid, dim3(32 * AT_WARPS), 0, s, a);
        if (e == cudaSuccess) e = launch(attn_combine_kernel<128>, dim3(p.QG, H_kv), dim3(32 * AT_TQ), 0, s, a);
    } else {
        e = launch(attn_partial_kernel<64>, grid, dim3(32 * AT_WARPS), 0, s, a);
        if (e == cudaSuccess) e = launch(attn_combine_kernel<64>, dim3(p.QG, H_kv), dim3(32 * AT_TQ), 0, s, a);
    }
    return e == cudaSuccess ? SD_OK : SD_ECUDA;
}

sd_status sd_kv_commit(void *k_cache, void *v_cache, int32_t H_kv, int32_t D, int64_t S_max, int64_t L, int32_t M,
                       const int32_t *path, const int32_t *count, sd_stream_t stream) {
    if (!k_cache || !v_cache || !count) return SD_EINVAL;
    if (H_kv < 1 || D < 1 || D > KC_MAXD || M < 1 || M > 16 || L < 0 || S_max < L + M) return SD_EINVAL;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return SD_EINVAL;
    if (!path) return SD_OK;  // a chain keeps its first n rows where they are
    int *st = status_ptr();
    if (!st) return SD_ECUDA;
    return launch(kv_commit_kernel, dim3(H_kv), dim3(128), 0, reinterpret_cast<cudaStream_t>(stream),
                  static_cast<__half *>(k_cache), static_cast<__half *>(v_cache), D, S_max, L, M, path, count, st) ==
                   cudaSuccess
               ? SD_OK
               : SD_ECUDA;
}

}  // extern "C"
