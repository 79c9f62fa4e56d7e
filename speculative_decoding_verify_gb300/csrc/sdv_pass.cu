// sdv_pass.cu - the whole verify pass of a quantised projection stack as one
// persistent cooperative launch: per layer RMSNorm -> QKV (V requantised in the
// epilogue) -> O (+ residual) -> RMSNorm -> gate|up (SiLU*mul requant) -> down
// (+ residual); then the final RMSNorm, the vocabulary head with fused argmax and
// statistics, and greedy acceptance.  Every phase runs the same device code as
// the single-operation entry points, so the pass equals them bit for bit.
#include <vector>

#include "sdv_qmatmul.cuh"

namespace sdv {

struct PassHeader {
    uint32_t barrier;  // grid-barrier counter, zeroed before every launch
    uint32_t pad[63];
};

static cudaError_t pass_launch(const QmmArgs *phases, int n_phases, uint32_t *ctr, int nt, size_t smem, int grid,
                               cudaStream_t s) {
    void (*k)(const QmmArgs *, int, uint32_t *) = nt == 1 ? pass_kernel<1> : pass_kernel<2>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(ctr, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(QMM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident, or the launch fails
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, phases, n_phases, ctr);
}

}  // namespace sdv

using namespace sdv;

extern "C" {

size_t sd_pass_plan_bytes(int32_t n_layers) {
    if (n_layers < 0) return 0;
    return sizeof(PassHeader) + static_cast<size_t>(6 * n_layers + 3) * sizeof(QmmArgs);
}

size_t sd_pass_workspace_bytes(int64_t hidden, int64_t ffn, int64_t vocab, int32_t wq) {
    const int sms = num_sms();
    size_t best = 0;
    QmmPlan p;
    const int64_t shapes[4][3] = {{3 * hidden, hidden, 0}, {hidden, hidden, 0}, {2 * ffn, hidden, 1}, {hidden, ffn, 0}};
    for (auto &sh : shapes) {
        if (!make_plan(wq, sh[0], sh[1], sh[2] != 0, false, sms, p)) return 0;
        best = p.ws_total > best ? p.ws_total : best;
    }
    if (!make_plan(SD_Q8_0, vocab, hidden, false, true, sms, p)) return 0;
    return p.ws_total > best ? p.ws_total : best;
}

sd_status sd_pass_prepare(const sd_pass_desc *d, void *plan, size_t plan_bytes, sd_pass *out) {
    if (!d || !plan || !out || !aligned(plan, 256)) return SD_EINVAL;
    const int L = d->n_layers;
    const int64_t H = d->hidden, F = d->ffn, V = d->vocab;
    const int M = d->M;
    if (L < 0 || M < 1 || H <= 0 || F <= 0 || V <= 0 || H % 64 || F % 32 || !d->layers) return SD_EINVAL;
    if (M > 16) return SD_EUNSUPPORTED;
    if (d->wq != SD_Q4_32 && d->wq != SD_Q8_0) return SD_EINVAL;
    if (d->wq == SD_Q8_0) return SD_EUNSUPPORTED;  // the SiLU*mul epilogue needs the 4-bit gate|up pairing
    if (plan_bytes < sd_pass_plan_bytes(L)) return SD_EINVAL;
    if (!d->h || !d->qa || !d->sa || !d->qv || !d->sv || !d->qf || !d->sf || !d->final_norm || !d->head ||
        !d->logits || !d->argmax || !d->row_max || !d->row_sumexp || !d->out_tokens || !d->out_count ||
        !d->workspace)
        return SD_EINVAL;
    if (M > 1 && !d->tokens) return SD_EINVAL;
    if (!aligned(d->workspace, 256) || d->ws_bytes < sd_pass_workspace_bytes(H, F, V, d->wq)) return SD_EINVAL;
    if (!(d->temperature > 0.0f)) return SD_EINVAL;
    int *st = status_ptr();
    if (!st) return SD_ECUDA;
    const int sms = num_sms();
    const int NT = M <= 8 ? 1 : 2;

    std::vector<QmmArgs> ph;
    uint8_t *ws = static_cast<uint8_t *>(d->workspace);
    auto base = [&](QmmArgs &a) {
        a = QmmArgs{};
        a.M = M;
        a.status = st;
        a.cnt = reinterpret_cast<uint32_t *>(ws);
        a.st_cnt = a.cnt + WS_UNIT_CNT;
        a.st_done = a.st_cnt + WS_STAT_CNT;
        a.part = reinterpret_cast<float *>(ws + WS_CNT_BYTES);
    };
    auto matmul = [&](int qt, const void *w, int64_t n, int64_t k, bool pair, const int8_t *q, const float *sc,
                      float *y, const float *res, uint32_t epi, int64_t col0, int8_t *qn, float *sn,
                      int64_t nq) -> bool {
        QmmPlan p;
        if (!make_plan(qt, n, k, pair, false, sms, p) || p.G != sms) return false;
        if (!w || !aligned(w, 16)) return false;
        QmmArgs a;
        base(a);
        a.kind = KIND_MATMUL;
        a.qt = qt;
        a.pair = pair ? 1 : 0;
        a.KB = p.KB;
        a.NU = p.NU;
        a.KS = p.KS;
        a.KBs = p.KBs;
        a.KBlast = p.KBlast;
        a.W = p.W;
        a.G = p.G;
        a.P = p.P;
        a.step_bytes = p.step_bytes;
        a.SB = stage_steps(qt, pair);
        a.w = static_cast<const uint8_t *>(w);
        a.n_out = n;
        a.q = q;
        a.sc = sc;
        a.y = y;
        a.residual = res;
        a.epi = epi;
        a.col0 = col0;
        a.q_next = qn;
        a.s_next = sn;
        a.nq = nq;
        ph.push_back(a);
        return true;
    };
    auto norm = [&](const float *x, const float *w, int64_t K, int8_t *q, float *s) {
        QmmArgs a;
        base(a);
        a.kind = KIND_NORM;
        a.KB = static_cast<int32_t>(K / 32);
        a.xin = x;
        a.norm_w = w;
        a.eps = d->eps;
        a.q_next = q;
        a.s_next = s;
        ph.push_back(a);
    };
    for (int l = 0; l < L; ++l) {
        const sd_layer &lw = d->layers[l];
        if (!lw.norm1 || !lw.norm2) return SD_EINVAL;
        norm(d->h, lw.norm1, H, d->qa, d->sa);
        if (!matmul(d->wq, lw.qkv, 3 * H, H, false, d->qa, d->sa, nullptr, nullptr, SD_EPI_REQUANT, 2 * H, d->qv, d->sv,
                    H))
            return SD_EINVAL;
        if (!matmul(d->wq, lw.o, H, H, false, d->qv, d->sv, d->h, d->h, SD_EPI_NONE, 0, nullptr, nullptr, 0))
            return SD_EINVAL;
        norm(d->h, lw.norm2, H, d->qa, d->sa);
        if (!matmul(d->wq, lw.gate_up, 2 * F, H, true, d->qa, d->sa, nullptr, nullptr, SD_EPI_SILU_MUL_REQUANT, 0,
                    d->qf, d->sf, F))
            return SD_EINVAL;
        if (!matmul(d->wq, lw.down, H, F, false, d->qf, d->sf, d->h, d->h, SD_EPI_NONE, 0, nullptr, nullptr, 0))
            return SD_EINVAL;
    }
    norm(d->h, d->final_norm, H, d->qa, d->sa);
    if (!matmul(SD_Q8_0, d->head, V, H, false, d->qa, d->sa, d->logits, nullptr, SD_EPI_NONE, 0, nullptr, nullptr, 0))
        return SD_EINVAL;
    {
        QmmArgs &hd = ph.back();
        const int64_t nst = (V + STAT_TILE - 1) / STAT_TILE;
        QmmPlan p;
        make_plan(SD_Q8_0, V, H, false, true, sms, p);
        hd.head = 1;
        hd.T = d->temperature;
        hd.argmax = d->argmax;
        hd.row_max = d->row_max;
        hd.row_sumexp = d->row_sumexp;
        hd.n_stiles = static_cast<int32_t>(nst);
        hd.st_part = reinterpret_cast<float4 *>(ws + WS_CNT_BYTES + p.ws_part);
    }
    {
        QmmArgs a;
        base(a);
        a.kind = KIND_ACCEPT;
        a.argmax = d->argmax;
        a.tokens = d->tokens;
        a.parent = d->parent;
        a.out_tokens = d->out_tokens;
        a.out_count = d->out_count;
        ph.push_back(a);
    }
    // one shared-memory layout for every phase: the largest split, pair rows, the largest stage
    int kbs = 0;
    size_t slot = 0;
    for (const QmmArgs &a : ph)
        if (a.kind == KIND_MATMUL) {
            kbs = a.KBs > kbs ? a.KBs : kbs;
            const size_t st = static_cast<size_t>(a.SB) * a.step_bytes;
            slot = st > slot ? st : slot;
        }
    int NS = 0;
    uint32_t o_ring, o_act, o_meta, o_red;
    const size_t smem = layout_smem(kbs, NT, 64, slot, NS, o_ring, o_act, o_meta, o_red);
    if (smem > 227 * 1024) return SD_EUNSUPPORTED;
    for (QmmArgs &a : ph) {
        a.NS = NS;
        a.off_ring = o_ring;
        a.off_act = o_act;
        a.off_meta = o_meta;
        a.off_red = o_red;
        a.stage_stride = static_cast<uint32_t>(slot);
    }
    PassHeader hdr = {};
    if (cudaMemcpy(plan, &hdr, sizeof(hdr), cudaMemcpyHostToDevice) != cudaSuccess) return SD_ECUDA;
    if (cudaMemcpy(static_cast<uint8_t *>(plan) + sizeof(PassHeader), ph.data(), ph.size() * sizeof(QmmArgs),
                   cudaMemcpyHostToDevice) != cudaSuccess)
        return SD_ECUDA;
    out->plan = plan;
    out->n_phases = static_cast<int32_t>(ph.size());
    out->nt = NT;
    out->smem_bytes = static_cast<uint32_t>(smem);
    out->grid = sms;
    return SD_OK;
}

sd_status sd_verify_pass(const sd_pass *p, sd_stream_t stream) {
    if (!p || !p->plan || p->n_phases < 1 || (p->nt != 1 && p->nt != 2) || p->grid < 1) return SD_EINVAL;
    uint8_t *plan = static_cast<uint8_t *>(p->plan);
    const QmmArgs *phases = reinterpret_cast<const QmmArgs *>(plan + sizeof(PassHeader));
    uint32_t *ctr = reinterpret_cast<uint32_t *>(plan);
    return pass_launch(phases, p->n_phases, ctr, p->nt, p->smem_bytes, p->grid, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? SD_OK
               : SD_ECUDA;
}

}  // extern "C"
