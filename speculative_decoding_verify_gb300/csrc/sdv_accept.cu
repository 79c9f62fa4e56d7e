// sdv_accept.cu - greedy and rejection-sampling acceptance of the verify pass.
#include "sdv_common.cuh"
#include "sdv_sample.cuh"

namespace sdv {

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
// rejection sampling, one CTA of ACC_THREADS threads
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(ACC_THREADS) accept_sample_kernel(const SampleArgs a) {
    __shared__ SampleShared sh;
    pdl_wait();
    pdl_launch_dependents();
    sample_accept<ACC_THREADS>(a, sh, static_cast<int>(threadIdx.x), []() { __syncthreads(); });
}

}  // namespace sdv

using namespace sdv;

static inline cudaStream_t cs_(sd_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

extern "C" {

sd_status sd_accept_greedy(const int32_t *argmax, const int32_t *tokens, const int32_t *parent, int32_t M,
                           int32_t *out_tokens, int32_t *out_count, sd_stream_t stream) {
    SD_NVTX("sd_accept_greedy");
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
    SD_NVTX("sd_accept_sample");
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
