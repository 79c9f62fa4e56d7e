// sdv_pass.cu - the whole verify pass of a quantised projection stack as one
// persistent cooperative launch: the first RMSNorm; per layer QKV (V requantised
// in the epilogue) -> O (+ residual; the next RMSNorm's codes in the epilogue)
// -> gate|up (SiLU*mul requant) -> down (+ residual; the next RMSNorm's codes);
// then the vocabulary head with fused argmax and statistics, and greedy or
// rejection-sampling acceptance.  An RMSNorm's row factor 1/rms is applied where its codes are
// staged by the next matmul, from block sums of squares the epilogues leave.
// The arithmetic is that of the single-operation entry points, so the pass
// equals them bit for bit.
#include <vector>

#include "sdv_qmatmul.cuh"

namespace sdv {

struct PassHeader {
    uint32_t barrier;  // grid-barrier counter, zeroed before every launch
    uint32_t pad[63];
};

// The plan: the header, the phase table (5 phases per layer, 4 more), then the combine phases' table of
// pieces per (unit, split) (up to PASS_NP_TAB_BYTES entries; a larger shape works them out on the GPU).
constexpr size_t PASS_NP_TAB_BYTES = 16384;
inline size_t pass_np_tab_offset(int n_layers) {
    const size_t end = sizeof(PassHeader) + static_cast<size_t>(5 * n_layers + 4) * sizeof(QmmArgs);
    return (end + 255) / 256 * 256;
}

static cudaError_t pass_launch(const QmmArgs *phases, int n_phases, uint32_t *ctr, uint64_t *trace, int nt,
                               int sample, int kq, size_t smem, int grid, cudaStream_t s) {
    if (kq) return pass_launch_kq(phases, n_phases, ctr, trace, nt, smem, grid, s);
    if (sample) return pass_launch_sampling(phases, n_phases, ctr, trace, nt, smem, grid, s);
    return pass_launch_kernel(nt == 1 ? pass_kernel<1, false> : pass_kernel<2, false>, phases, n_phases, ctr, trace,
                              smem, grid, s);
}

}  // namespace sdv

using namespace sdv;

namespace sdv {

// Workspace of the pass: the matmul counters and partial sums, the head's statistics, the
// activation fragments feeding the QKV / gate|up / head (from the RMSNorm phases), the O
// projection (from the QKV epilogue) and the down projection (from the SiLU epilogue), and the
// per-block sums of squares of the residual stream.  Fragment regions are sized for M = 16.
struct PassWs {
    size_t part, stats, afa_frag, afa_meta, afv_frag, afv_meta, aff_frag, aff_meta, ss, total;
};

static bool pass_ws_layout(int64_t H, int64_t F, int64_t V, int wq, int sms, PassWs &L) {
    QmmPlan p;
    size_t part = 0;
    const int64_t shapes[4][3] = {{3 * H, H, 0}, {H, H, 0}, {2 * F, H, 1}, {H, F, 0}};
    for (auto &sh : shapes) {
        // a K-quant stack's down projection may be Q6_K: the plan (and so the partial sums) is the same
        if (!make_plan(wq, sh[0], sh[1], sh[2] != 0, false, sms, p)) return false;
        part = p.ws_part > part ? p.ws_part : part;
    }
    if (!make_plan(SD_Q8_0, V, H, false, true, sms, p)) return false;
    part = p.ws_part > part ? p.ws_part : part;
    const size_t KBH = static_cast<size_t>(H / 32), KBF = static_cast<size_t>(F / 32);
    const size_t fb = af_frag_bytes(16) > af_frag_bytes(8) ? af_frag_bytes(16) : af_frag_bytes(8);
    const size_t mb = af_meta_bytes_q(16, is_kq(wq) ? SD_Q4_K : SD_Q4_32);
    size_t off = WS_CNT_BYTES;
    L.part = off;
    off += part;
    L.stats = off;
    off += p.ws_stats;
    L.afa_frag = off;
    off += align_up(KBH * fb, 256);
    L.afa_meta = off;
    off += align_up(KBH * mb, 256);
    L.afv_frag = off;
    off += align_up(KBH * fb, 256);
    L.afv_meta = off;
    off += align_up(KBH * mb, 256);
    L.aff_frag = off;
    off += align_up(KBF * fb, 256);
    L.aff_meta = off;
    off += align_up(KBF * mb, 256);
    L.ss = off;
    off += align_up(16 * align_up(KBH, 4) * sizeof(float), 256);
    L.total = off;
    return true;
}

}  // namespace sdv

extern "C" {

size_t sd_pass_plan_bytes(int32_t n_layers) {
    if (n_layers < 0) return 0;
    return pass_np_tab_offset(n_layers) + PASS_NP_TAB_BYTES;
}

size_t sd_pass_workspace_bytes(int64_t hidden, int64_t ffn, int64_t vocab, int32_t wq) {
    if (hidden <= 0 || ffn <= 0 || vocab <= 0 || hidden % 64 || ffn % 32) return 0;
    PassWs L;
    return pass_ws_layout(hidden, ffn, vocab, wq, num_sms(), L) ? L.total : 0;
}

sd_status sd_pass_prepare(const sd_pass_desc *d, void *plan, size_t plan_bytes, sd_pass *out) {
    if (!d || !plan || !out || !aligned(plan, 256)) return SD_EINVAL;
    const int L = d->n_layers;
    const int64_t H = d->hidden, F = d->ffn, V = d->vocab;
    const int M = d->M;
    if (L < 0 || M < 1 || H <= 0 || F <= 0 || V <= 0 || H % 64 || F % 32 || !d->layers) return SD_EINVAL;
    if (M > 16 || H / 32 > PASS_NORM_MAX_KB) return SD_EUNSUPPORTED;
    if (d->wq != SD_Q4_32 && d->wq != SD_Q8_0 && d->wq != SD_Q4_K && d->wq != SD_Q6_K) return SD_EINVAL;
    if (d->wq == SD_Q8_0 || d->wq == SD_Q6_K) return SD_EUNSUPPORTED;  // the SiLU*mul epilogue needs a paired format
    const int wqd = d->wq_down == 0 ? d->wq : d->wq_down;  // the down projections' format
    if (wqd != d->wq && !(d->wq == SD_Q4_K && wqd == SD_Q6_K)) return SD_EUNSUPPORTED;
    const bool kq = is_kq(d->wq);
    if (kq && (H % 256 || F % 256)) return SD_EINVAL;
    if (kq && d->accept != SD_ACCEPT_GREEDY) return SD_EUNSUPPORTED;
    if (plan_bytes < sd_pass_plan_bytes(L)) return SD_EINVAL;
    if (!d->h || !d->qa || !d->sa || !d->qv || !d->sv || !d->qf || !d->sf || !d->final_norm || !d->head ||
        !d->logits || !d->argmax || !d->row_max || !d->row_sumexp || !d->out_tokens || !d->out_count ||
        !d->workspace)
        return SD_EINVAL;
    if (M > 1 && !d->tokens) return SD_EINVAL;
    if (!(d->temperature > 0.0f)) return SD_EINVAL;
    if (d->accept != SD_ACCEPT_GREEDY && d->accept != SD_ACCEPT_SAMPLE) return SD_EINVAL;
    if (d->accept == SD_ACCEPT_SAMPLE &&
        (d->parent || V > static_cast<int64_t>(MAX_TILES) * ATILE || !(d->temperature <= 3.0e38f)))
        return SD_EUNSUPPORTED;  // sampling: chains only, the single-operation call's vocabulary limit
    if (d->accept == SD_ACCEPT_SAMPLE && d->top_k != 0 &&
        (d->top_k < 1 || d->top_k > TK_MAX || !(d->top_p > 0.0f) || d->top_p > 1.0f))
        return SD_EINVAL;
    int *st = status_ptr();
    if (!st) return SD_ECUDA;
    const int sms = num_sms();
    PassWs W;
    if (!pass_ws_layout(H, F, V, d->wq, sms, W)) return SD_EINVAL;
    if (!aligned(d->workspace, 256) || d->ws_bytes < W.total) return SD_EINVAL;
    const int NT = af_nt(M);

    std::vector<QmmArgs> ph;
    ph.reserve(static_cast<size_t>(5 * L + 4));  // pointers returned by matmul() below stay valid
    uint8_t *ws = static_cast<uint8_t *>(d->workspace);
    uint8_t *afa_f = ws + W.afa_frag, *afv_f = ws + W.afv_frag, *aff_f = ws + W.aff_frag;
    float *afa_m = reinterpret_cast<float *>(ws + W.afa_meta), *afv_m = reinterpret_cast<float *>(ws + W.afv_meta),
          *aff_m = reinterpret_cast<float *>(ws + W.aff_meta), *ssb = reinterpret_cast<float *>(ws + W.ss);
    auto base = [&](QmmArgs &a) {
        a = QmmArgs{};
        a.GR = 1;
        a.GRS = 0;
        a.M = M;
        a.status = st;
        a.cnt = reinterpret_cast<uint32_t *>(ws);
        a.st_cnt = a.cnt + WS_UNIT_CNT;
        a.st_done = a.st_cnt + WS_STAT_CNT;
        a.part = reinterpret_cast<float *>(ws + W.part);
    };
    const int ss_ld = static_cast<int>(align_up(static_cast<size_t>(H / 32), 4));
    auto matmul = [&](int qt, const void *w, int64_t n, int64_t k, bool pair, const int8_t *q, const float *sc,
                      const uint8_t *af_f, const float *af_m) -> QmmArgs * {
        QmmPlan p;
        if (!make_plan(qt, n, k, pair, false, sms, p)) return nullptr;  // CTAs past p.G sit the phase out
        if (!w || !aligned(w, 16)) return nullptr;
        QmmArgs a;
        base(a);
        a.kind = KIND_MATMUL;
        a.qt = qt;
        a.pair = pair ? 1 : 0;
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
        a.SB = stage_steps(qt, pair);
        a.w = static_cast<const uint8_t *>(w);
        a.n_out = n;
        a.q = q;
        a.sc = sc;
        a.af_frag = af_f;
        a.af_meta = af_m;
        a.ss_ld = ss_ld;
        a.eps = d->eps;
        ph.push_back(a);
        return &ph.back();
    };
    // input: RMSNorm codes in AF_a, scaled by inv at staging (block sums of squares in ssb)
    auto normed_input = [&](QmmArgs *a) {
        a->af_norm = 1;
        a->ss_in = ssb;
        a->s_norm_out = d->sa;
    };
    // epilogue: residual add into h, block sums of squares, the next RMSNorm's codes into AF_a
    auto residual_out = [&](QmmArgs *a, const float *next_norm, int next_qt) {
        a->y = d->h;
        a->residual = d->h;
        a->ss = ssb;
        a->norm_next = next_norm;
        a->q_next = d->qa;
        a->nq = H;
        a->af_out_frag = afa_f;
        a->af_out_meta = afa_m;
        a->af_out_qt = next_qt;
    };
    {  // the first RMSNorm, on the input rows
        QmmArgs a;
        base(a);
        a.kind = KIND_NORM;
        a.KB = static_cast<int32_t>(H / 32);
        a.xin = d->h;
        a.norm_w = L > 0 ? d->layers[0].norm1 : d->final_norm;
        a.ss = ssb;
        a.ss_ld = ss_ld;
        a.q_next = d->qa;
        a.af_out_frag = afa_f;
        a.af_out_meta = afa_m;
        a.af_out_qt = L > 0 ? d->wq : SD_Q8_0;
        if (!a.norm_w) return SD_EINVAL;
        ph.push_back(a);
    }
    for (int l = 0; l < L; ++l) {
        const sd_layer &lw = d->layers[l];
        if (!lw.norm1 || !lw.norm2) return SD_EINVAL;
        QmmArgs *a = matmul(d->wq, lw.qkv, 3 * H, H, false, d->qa, d->sa, afa_f, afa_m);
        if (!a) return SD_EINVAL;
        normed_input(a);
        a->epi = SD_EPI_REQUANT;
        a->col0 = 2 * H;
        if (a->NU % 3 == 0) a->ilv3 = a->NU / 3;  // V tiles spread over the CTAs, V first
        a->q_next = d->qv;
        a->s_next = d->sv;
        a->nq = H;
        a->af_out_frag = afv_f;
        a->af_out_meta = afv_m;
        a->af_out_qt = d->wq;
        if (!(a = matmul(d->wq, lw.o, H, H, false, d->qv, d->sv, afv_f, afv_m))) return SD_EINVAL;
        residual_out(a, lw.norm2, d->wq);
        if (!(a = matmul(d->wq, lw.gate_up, 2 * F, H, true, d->qa, d->sa, afa_f, afa_m))) return SD_EINVAL;
        normed_input(a);
        a->epi = SD_EPI_SILU_MUL_REQUANT;
        a->q_next = d->qf;
        a->s_next = d->sf;
        a->nq = F;
        a->af_out_frag = aff_f;
        a->af_out_meta = aff_m;
        a->af_out_qt = wqd;
        if (!(a = matmul(wqd, lw.down, H, F, false, d->qf, d->sf, aff_f, aff_m))) return SD_EINVAL;
        const bool lastl = l + 1 == L;
        if (!lastl && !d->layers[l + 1].norm1) return SD_EINVAL;
        residual_out(a, lastl ? d->final_norm : d->layers[l + 1].norm1, lastl ? SD_Q8_0 : d->wq);
        if (a->D == 0 && a->KS > 1) {
            // every unit is shared across k-splits: store partial sums only and finish the units in a
            // combine phase, an equal share per CTA, instead of wherever the last piece lands
            a->defer = 1;
            QmmArgs cmb = *a;
            cmb.kind = KIND_COMBINE;
            ph.push_back(cmb);
        }
    }
    {
        QmmArgs *hd = matmul(SD_Q8_0, d->head, V, H, false, d->qa, d->sa, afa_f, afa_m);
        if (!hd) return SD_EINVAL;
        normed_input(hd);
        hd->y = d->logits;
        hd->head = 1;
        hd->T = d->temperature;
        hd->argmax = d->argmax;
        hd->row_max = d->row_max;
        hd->row_sumexp = d->row_sumexp;
        hd->n_stiles = static_cast<int32_t>((V + STAT_TILE - 1) / STAT_TILE);
        hd->st_part = reinterpret_cast<float4 *>(ws + W.stats);
        // the statistics once the logits are complete: an even spread over the grid instead of
        // wherever a tile's last rows land; the acceptance phase folds them
        hd->defer_stats = 1;
        QmmArgs hs = *hd;
        hs.kind = KIND_HSTATS;
        ph.push_back(hs);
    }
    {
        const QmmArgs &hd = ph[ph.size() - 1];
        QmmArgs a;
        base(a);
        a.kind = KIND_ACCEPT;
        a.defer_stats = 1;
        a.T = hd.T;
        a.n_out = hd.n_out;
        a.n_stiles = hd.n_stiles;
        a.st_part = hd.st_part;
        a.row_max = hd.row_max;
        a.row_sumexp = hd.row_sumexp;
        a.argmax = d->argmax;
        a.tokens = d->tokens;
        a.parent = d->parent;
        a.out_tokens = d->out_tokens;
        a.out_count = d->out_count;
        a.accept_mode = d->accept;
        a.y = d->logits;
        a.q_probs = d->q_probs;
        a.seed = d->seed;
        a.base_pos = d->base_pos;
        a.top_k = d->top_k;
        a.top_p = d->top_p;
        ph.push_back(a);
    }
    // one shared-memory layout for every phase: the largest split, pair rows, the largest stage,
    // and the RMSNorm scratch
    int kbs = 0;
    size_t slot = 0;
    for (const QmmArgs &a : ph)
        if (a.kind == KIND_MATMUL) {
            kbs = a.KBs > kbs ? a.KBs : kbs;
            const size_t sz = static_cast<size_t>(a.SB) * a.step_bytes;
            slot = sz > slot ? sz : slot;
        }
    SmemLayout lay;
    if (!layout_smem(kbs, M, 64, slot, static_cast<size_t>(M) * ss_ld * sizeof(float), lay,
                     kq ? SD_Q4_K : SD_Q4_32))
        return SD_EUNSUPPORTED;
    if (static_cast<size_t>(lay.NS) * slot < sizeof(SampleShared) || static_cast<size_t>(lay.NS) * slot < sizeof(TopkShared))
        return SD_EUNSUPPORTED;  // the sampler's state
    for (QmmArgs &a : ph) apply_layout(a, lay, slot);
    // pieces per (unit, split) of the combine phases, from the host's replay of their schedule: every
    // combine phase of a pass has the same shape, so one table serves all whose schedule matches the first
    std::vector<uint8_t> np_tab;
    const QmmArgs *c0 = nullptr;
    uint8_t *np_dev = static_cast<uint8_t *>(plan) + pass_np_tab_offset(L);
    for (QmmArgs &a : ph) {
        if (a.kind != KIND_COMBINE) continue;
        if (!c0) {
            c0 = &a;
            const size_t n = static_cast<size_t>(a.NU) * np_tab_stride(a.KS);
            if (n > PASS_NP_TAB_BYTES || a.P > 255) break;  // too large: the GPU works them out
            np_tab.assign(n, 0);
            for (int u = 0; u < a.NU; ++u)
                for (int s = 0; s < a.KS; ++s) {
                    int first = 0, np = 0;
                    unit_split_owners(a, s, u, first, np);
                    if (np < 0 || np > a.P) return SD_EINVAL;
                    np_tab[static_cast<size_t>(u) * np_tab_stride(a.KS) + s] = static_cast<uint8_t>(np);
                }
        }
        const bool same = a.NU == c0->NU && a.KS == c0->KS && a.KB == c0->KB && a.KBs == c0->KBs &&
                          a.KBlast == c0->KBlast && a.W == c0->W && a.G == c0->G && a.P == c0->P && a.D == c0->D &&
                          a.R == c0->R && a.GRS == c0->GRS;
        a.np_tab = same ? np_dev : nullptr;
    }
    if (!np_tab.empty() &&
        cudaMemcpy(np_dev, np_tab.data(), np_tab.size(), cudaMemcpyHostToDevice) != cudaSuccess)
        return SD_ECUDA;
    PassHeader hdr = {};
    if (cudaMemcpy(plan, &hdr, sizeof(hdr), cudaMemcpyHostToDevice) != cudaSuccess) return SD_ECUDA;
    if (cudaMemcpy(static_cast<uint8_t *>(plan) + sizeof(PassHeader), ph.data(), ph.size() * sizeof(QmmArgs),
                   cudaMemcpyHostToDevice) != cudaSuccess)
        return SD_ECUDA;
    out->plan = plan;
    out->n_phases = static_cast<int32_t>(ph.size());
    out->nt = NT;
    out->smem_bytes = static_cast<uint32_t>(lay.total);
    out->grid = sms;
    out->accept = d->accept;
    out->kq = kq ? 1 : 0;
    return SD_OK;
}

static sd_status verify_pass_launch(const sd_pass *p, uint64_t *trace, sd_stream_t stream) {
    if (!p || !p->plan || p->n_phases < 1 || (p->nt != 1 && p->nt != 2) || p->grid < 1 ||
        (p->accept != SD_ACCEPT_GREEDY && p->accept != SD_ACCEPT_SAMPLE))
        return SD_EINVAL;
    uint8_t *plan = static_cast<uint8_t *>(p->plan);
    const QmmArgs *phases = reinterpret_cast<const QmmArgs *>(plan + sizeof(PassHeader));
    uint32_t *ctr = reinterpret_cast<uint32_t *>(plan);
    return pass_launch(phases, p->n_phases, ctr, trace, p->nt, p->accept, p->kq, p->smem_bytes, p->grid,
                       reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SD_OK
               : SD_ECUDA;
}

sd_status sd_verify_pass(const sd_pass *p, sd_stream_t stream) {
    SD_NVTX("sd_verify_pass");
    return verify_pass_launch(p, nullptr, stream);
}

size_t sd_pass_trace_bytes(const sd_pass *p) {
    if (!p || p->n_phases < 1 || p->grid < 1) return 0;
    return (static_cast<size_t>(p->grid) + static_cast<size_t>(p->n_phases) * p->grid * TR_SLOTS) * sizeof(uint64_t);
}

sd_status sd_verify_pass_traced(const sd_pass *p, uint64_t *trace, size_t trace_bytes, sd_stream_t stream) {
    SD_NVTX("sd_verify_pass_traced");
    if (!trace || !aligned(trace, 8) || trace_bytes < sd_pass_trace_bytes(p) || sd_pass_trace_bytes(p) == 0)
        return SD_EINVAL;
    return verify_pass_launch(p, trace, stream);
}

}  // extern "C"
