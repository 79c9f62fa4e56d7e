// sdv_qmm_abi.cu - C entry points of the multi-position matmul and the head,
// and the block-dot test hook.
#include "sdv_qmatmul.cuh"

namespace sdv {

// One warp per (tile, block): the matmul's own fragment conversion and
// mma-based exact dots on the repacked record, for every 8-position tile.
template <int QT>
__global__ void block_dots_kernel(const uint8_t *__restrict__ w, int64_t n_out, int32_t KB,
                                  const int8_t *__restrict__ q, int32_t M, int32_t *__restrict__ dots) {
    constexpr int REC = QT == SD_Q8_0 ? 1088 : 576;
    const int64_t tile = blockIdx.x / KB;
    const int b = static_cast<int>(blockIdx.x - tile * KB);
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int64_t K = static_cast<int64_t>(KB) * 32;
    const uint8_t *rec = w + (tile * KB + b) * REC;
    uint32_t af[2][2][4];
    if (QT == SD_Q4_32)
        q4_frag(*reinterpret_cast<const uint4 *>(rec + lane * 16), af);
    else
        q8_frag(*reinterpret_cast<const uint4 *>(rec + lane * 16), *reinterpret_cast<const uint4 *>(rec + 512 + lane * 16),
                af);
    for (int nt = 0; nt * 8 < M; ++nt) {
        const int nb = nt * 8 + g;
        const uint4 bf = b_frag_from_raw<QT>(b_raw(nb < M ? q + nb * K + b * 32 : nullptr, c));
        const int m0 = nt * 8 + 2 * c, m1 = m0 + 1;
        const float2 corr = make_float2(dot_corr<QT>(m0 < M ? q + m0 * K + b * 32 : nullptr),
                                        dot_corr<QT>(m1 < M ? q + m1 * K + b * 32 : nullptr));
        float d[2][4];
        record_dots(af, bf, corr, d);
        for (int t = 0; t < 2; ++t)
            for (int i = 0; i < 4; ++i) {
                const int m = m0 + (i & 1);
                const int64_t n = tile * 32 + 16 * t + g + 8 * (i >> 1);
                if (m < M && n < n_out) dots[(static_cast<int64_t>(m) * n_out + n) * KB + b] = static_cast<int32_t>(d[t][i]);
            }
    }
}

static inline cudaStream_t cs(sd_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

static cudaError_t dispatch(int qtype, bool pair, QmmArgs &a, QmmPlan &p, cudaStream_t s) {
    if (qtype == SD_Q4_32) return pair ? qmm_dispatch<SD_Q4_32, 1>(a, p, s) : qmm_dispatch<SD_Q4_32, 0>(a, p, s);
    if (qtype == SD_Q4_K) return pair ? qmm_dispatch<SD_Q4_K, 1>(a, p, s) : qmm_dispatch<SD_Q4_K, 0>(a, p, s);
    if (qtype == SD_Q6_K) return qmm_dispatch<SD_Q6_K, 0>(a, p, s);
    return qmm_dispatch<SD_Q8_0, 0>(a, p, s);
}

// The call's activation fragments and records go to the workspace's last region (act_frag_kernel).
static void set_af_build(QmmArgs &a, const QmmPlan &p, uint8_t *ws) {
    uint8_t *act = ws + p.ws_cnt + p.ws_part + p.ws_stats;
    a.af_frag = act;
    a.af_meta = reinterpret_cast<const float *>(act + static_cast<size_t>(p.KB) * af_frag_bytes(a.M));
    a.af_build = 1;
}

static bool known_qtype(int q) { return q == SD_Q8_0 || q == SD_Q4_32 || q == SD_Q4_K || q == SD_Q6_K; }

static void fill_plan(QmmArgs &a, const QmmPlan &p) {
    a.GR = p.GR;
    a.GRS = p.GRS;
    a.KB = p.KB;
    a.NU = p.NU;
    a.KS = p.KS;
    a.KBs = p.KBs;
    a.KBlast = p.KBlast;
    a.W = p.W;
    a.G = p.G;
    a.P = p.P;
    a.D = p.D;
    a.R = p.R;
    a.step_bytes = p.step_bytes;
}

}  // namespace sdv

using namespace sdv;

extern "C" {

int64_t sd_debug_schedule(int qtype, int64_t n_out, int64_t k_in, int32_t pair, int32_t head, int32_t sms,
                          int32_t *plan, int32_t *rows, int64_t cap) {
    if (!known_qtype(qtype) || sms < 1 || !plan) return -1;
    QmmPlan p;
    if (!make_plan(qtype, n_out, k_in, pair != 0, head != 0, sms, p)) return -1;
    QmmArgs a = {};
    fill_plan(a, p);
    const int32_t fields[9] = {p.KB, p.NU, p.KS, p.KBs, p.KBlast, p.G, p.P, p.D, p.R};
    for (int i = 0; i < 9; ++i) plan[i] = fields[i];
    int64_t n = 0;
    for (int c = 0; c < p.G; ++c) {
        PieceIter it;
        pieces_begin_cta(a, it, c);
        Piece pc, nx;
        bool have = pieces_next(a, it, pc);
        while (have) {
            const bool more = pieces_next(a, it, nx);
            if (n >= cap || !rows) return -2;
            int32_t *r = rows + 8 * n;
            r[0] = c;
            r[1] = pc.s;
            r[2] = pc.u;
            r[3] = pc.j0;
            r[4] = pc.j1;
            r[5] = pc.first;
            r[6] = pc.np;
            r[7] = more ? 0 : 1;
            ++n;
            pc = nx;
            have = more;
        }
    }
    return n;
}

size_t sd_qmatmul_workspace_bytes(int qtype, int64_t n_out, int64_t k_in, uint32_t epilogue) {
    if (!known_qtype(qtype)) return 0;
    QmmPlan p;
    if (!make_plan(qtype, n_out, k_in, epilogue == SD_EPI_SILU_MUL_REQUANT, false, num_sms(), p)) return 0;
    return p.ws_total;
}

size_t sd_head_workspace_bytes(int64_t vocab, int64_t hidden) {
    QmmPlan p;
    if (!make_plan(SD_Q8_0, vocab, hidden, false, true, num_sms(), p)) return 0;
    return p.ws_total;
}

sd_status sd_qmatmul_multipos(int qtype, const void *w, int64_t n_out, int64_t k_in, const int8_t *q,
                              const float *scales, int32_t M, float *y, const float *residual, uint32_t epilogue,
                              int64_t requant_col0, int8_t *q_next, float *scales_next, void *workspace,
                              size_t ws_bytes, sd_stream_t stream) {
    SD_NVTX("sd_qmatmul_multipos");
    return sdv::qmatmul_restricted(qtype, w, n_out, k_in, q, scales, M, y, residual, epilogue, requant_col0, q_next,
                                   scales_next, workspace, ws_bytes, nullptr, nullptr, nullptr, nullptr, stream);
}

}  // extern "C"

namespace sdv {

sd_status qmatmul_restricted(int qtype, const void *w, int64_t n_out, int64_t k_in, const int8_t *q,
                             const float *scales, int32_t M, float *y, const float *residual, uint32_t epilogue,
                             int64_t requant_col0, int8_t *q_next, float *scales_next, void *workspace,
                             size_t ws_bytes, const uint32_t *unit_mask, const int *skip_if, const uint8_t *af_pre,
                             const float *af_meta_pre, sd_stream_t stream) {
    if (!known_qtype(qtype)) return SD_EINVAL;
    if (M < 1) return SD_EINVAL;
    if (M > 16) return SD_EUNSUPPORTED;
    if (!w || !q || !scales || !workspace) return SD_EINVAL;
    if (!aligned(w, 16) || !aligned(q, 16) || !aligned(scales, 4) || !aligned(workspace, 256)) return SD_EINVAL;
    if (k_in <= 0 || k_in % 32 || n_out <= 0) return SD_EINVAL;
    if ((qtype == SD_Q4_K || qtype == SD_Q6_K) && (k_in % 256 || n_out % 32)) return SD_EINVAL;
    const bool pair = epilogue == SD_EPI_SILU_MUL_REQUANT;
    int64_t nq = 0;
    if (epilogue == SD_EPI_NONE) {
        if (!y) return SD_EINVAL;
    } else if (epilogue == SD_EPI_REQUANT) {
        if (!q_next || !scales_next || n_out % 32 || requant_col0 < 0 || requant_col0 >= n_out ||
            requant_col0 % 32)
            return SD_EINVAL;
        nq = n_out - requant_col0;
    } else if (pair) {
        if (qtype != SD_Q4_32 && qtype != SD_Q4_K) return SD_EUNSUPPORTED;
        if (!q_next || !scales_next || residual || n_out % 64) return SD_EINVAL;
        nq = n_out / 2;
    } else {
        return SD_EINVAL;
    }
    if (y && !aligned(y, 4)) return SD_EINVAL;
    QmmPlan p;
    if (!make_plan(qtype, n_out, k_in, pair, false, num_sms(), p)) return SD_EINVAL;
    if (ws_bytes < p.ws_total) return SD_EINVAL;
    int *st = status_ptr();
    if (!st) return SD_ECUDA;
    QmmArgs a = {};
    fill_plan(a, p);
    a.w = static_cast<const uint8_t *>(w);
    a.n_out = n_out;
    a.q = q;
    a.sc = scales;
    a.M = M;
    a.y = y;
    a.residual = residual;
    a.epi = epilogue;
    a.col0 = requant_col0;
    a.q_next = q_next;
    a.s_next = scales_next;
    a.nq = nq;
    // requantised columns = the last third of the rows in whole 32-row tiles: interleave the thirds
    if (epilogue == SD_EPI_REQUANT && p.NU % 3 == 0 && 3 * requant_col0 == 2 * n_out) a.ilv3 = p.NU / 3;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.cnt = reinterpret_cast<uint32_t *>(ws);
    a.part = reinterpret_cast<float *>(ws + p.ws_cnt);
    set_af_build(a, p, ws);
    if (af_pre) {
        a.af_frag = af_pre;
        a.af_meta = af_meta_pre;
        a.af_build = 0;
    }
    a.unit_mask = unit_mask;
    a.skip_if = skip_if;
    a.status = st;
    return dispatch(qtype, pair, a, p, cs(stream)) == cudaSuccess ? SD_OK : SD_ECUDA;
}

}  // namespace sdv

extern "C" {

sd_status sd_head_logits(const void *w, int64_t vocab, int64_t hidden, const int8_t *q, const float *scales, int32_t M,
                         float temperature, float *logits, int32_t *argmax, float *row_max, float *row_sumexp,
                         void *workspace, size_t ws_bytes, sd_stream_t stream) {
    SD_NVTX("sd_head_logits");
    if (M < 1) return SD_EINVAL;
    if (M > 16) return SD_EUNSUPPORTED;
    if (!w || !q || !scales || !logits || !argmax || !row_max || !row_sumexp || !workspace) return SD_EINVAL;
    if (!aligned(w, 16) || !aligned(q, 16) || !aligned(logits, 16) || !aligned(workspace, 256)) return SD_EINVAL;
    if (!(temperature > 0.0f) || temperature > 3.0e38f) return SD_EINVAL;
    if (hidden <= 0 || hidden % 32 || vocab <= 0) return SD_EINVAL;
    QmmPlan p;
    if (!make_plan(SD_Q8_0, vocab, hidden, false, true, num_sms(), p)) return SD_EINVAL;
    if (ws_bytes < p.ws_total) return SD_EINVAL;
    int *st = status_ptr();
    if (!st) return SD_ECUDA;
    QmmArgs a = {};
    fill_plan(a, p);
    a.w = static_cast<const uint8_t *>(w);
    a.n_out = vocab;
    a.q = q;
    a.sc = scales;
    a.M = M;
    a.y = logits;
    a.epi = SD_EPI_NONE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    a.cnt = reinterpret_cast<uint32_t *>(ws);
    a.st_cnt = a.cnt + WS_UNIT_CNT;
    a.st_done = a.st_cnt + WS_STAT_CNT;
    a.part = reinterpret_cast<float *>(ws + p.ws_cnt);
    const int64_t nst = (vocab + STAT_TILE - 1) / STAT_TILE;
    a.st_part = reinterpret_cast<float4 *>(ws + p.ws_cnt + p.ws_part);
    set_af_build(a, p, ws);
    a.n_stiles = static_cast<int32_t>(nst);
    a.head = 1;
    a.T = temperature;
    a.argmax = argmax;
    a.row_max = row_max;
    a.row_sumexp = row_sumexp;
    a.status = st;
    return dispatch(SD_Q8_0, false, a, p, cs(stream)) == cudaSuccess ? SD_OK : SD_ECUDA;
}

sd_status sd_debug_block_dots(int qtype, const void *w, int64_t n_out, int64_t k_in, const int8_t *q, int32_t M,
                              int32_t *dots, sd_stream_t stream) {
    if ((qtype != SD_Q8_0 && qtype != SD_Q4_32) || !w || !q || !dots || M < 1 || M > 16) return SD_EINVAL;
    if (k_in <= 0 || k_in % 32 || n_out <= 0 || !aligned(w, 16) || !aligned(q, 16)) return SD_EINVAL;
    const int64_t blocks = (n_out + 31) / 32 * (k_in / 32);
    if (blocks > 0x7fffffff) return SD_EINVAL;
    if (qtype == SD_Q4_32)
        block_dots_kernel<SD_Q4_32><<<static_cast<unsigned>(blocks), 32, 0, cs(stream)>>>(
            static_cast<const uint8_t *>(w), n_out, static_cast<int32_t>(k_in / 32), q, M, dots);
    else
        block_dots_kernel<SD_Q8_0><<<static_cast<unsigned>(blocks), 32, 0, cs(stream)>>>(
            static_cast<const uint8_t *>(w), n_out, static_cast<int32_t>(k_in / 32), q, M, dots);
    return cudaGetLastError() == cudaSuccess ? SD_OK : SD_ECUDA;
}

}  // extern "C"
