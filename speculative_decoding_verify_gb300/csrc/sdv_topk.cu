// sdv_topk.cu - sd_accept_sample_topk: the filtered rejection-sampling acceptance as one CTA of
// 1024 threads (the rule and its reading are in sdv_topk.cuh).
#include "sdv_topk.cuh"

namespace sdv {

constexpr int TK_THREADS = 1024;

__global__ void __launch_bounds__(TK_THREADS) accept_topk_kernel(const TopkArgs a) {
    __shared__ TopkShared sh;
    pdl_wait();
    pdl_launch_dependents();
    topk_accept<TK_THREADS>(a, sh, static_cast<int>(threadIdx.x), []() { __syncthreads(); });
}

}  // namespace sdv

using namespace sdv;

extern "C" {

sd_status sd_accept_sample_topk(const float *logits, int64_t vocab, int32_t K, const float *q_probs,
                                const int32_t *drafts, float temperature, int32_t top_k, float top_p, uint64_t seed,
                                int64_t base_pos, int32_t *out_tokens, int32_t *out_count, sd_stream_t stream) {
    SD_NVTX("sd_accept_sample_topk");
    if (!logits || !out_tokens || !out_count || K < 0 || K > 15) return SD_EINVAL;
    if (K > 0 && !drafts) return SD_EINVAL;
    if (vocab < 1 || vocab > (int64_t(1) << 31) - 1) return SD_EINVAL;
    if (top_k < 1 || top_k > TK_MAX || !(top_p > 0.0f) || top_p > 1.0f) return SD_EINVAL;
    if (!(temperature > 0.0f) || temperature > 3.0e38f) return SD_EINVAL;
    TopkArgs a;
    a.logits = logits;
    a.V = vocab;
    a.K = K;
    a.q = q_probs;
    a.drafts = drafts;
    a.T = temperature;
    a.top_k = top_k;
    a.top_p = top_p;
    a.seed = seed;
    a.base_pos = base_pos;
    a.out = out_tokens;
    a.count = out_count;
    return launch(accept_topk_kernel, dim3(1), dim3(TK_THREADS), 0, reinterpret_cast<cudaStream_t>(stream), a) ==
                   cudaSuccess
               ? SD_OK
               : SD_ECUDA;
}

}  // extern "C"
