// sdv_noalloc.cu - the multi-position matmul for callers that must not allocate:
// the same kernel as sd_qmatmul_multipos, its scratch taken from one static device
// array of this library instead of a caller workspace.
#include <mutex>

#include "sdv_qmatmul.cuh"

namespace {

// Counters at the front (the kernel returns them to zero), partial sums after them.
static __device__ __align__(256) uint8_t g_noalloc_scratch[SD_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_scratch_addr[64];

// This device's scratch address, looked up once per device with that device current.
sd_status scratch_ptr(void **out) {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return SD_ECUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[d]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SD_ECUDA;
        g_scratch_addr[d] = p;
    }
    *out = g_scratch_addr[d];
    return SD_OK;
}

}  // namespace

extern "C" sd_status sd_qmatmul_multipos_noalloc(int qtype, const void *w, int64_t n_out, int64_t k_in,
                                                 const int8_t *q, const float *scales, int32_t M, float *y,
                                                 const float *residual, uint32_t epilogue, int64_t requant_col0,
                                                 int8_t *q_next, float *scales_next, sd_stream_t stream) {
    SD_NVTX("sd_qmatmul_multipos_noalloc");
    const size_t need = sd_qmatmul_workspace_bytes(qtype, n_out, k_in, epilogue);
    if (need == 0) return SD_EINVAL;
    if (need > SD_NOALLOC_SCRATCH_BYTES) return SD_EUNSUPPORTED;
    void *ws = nullptr;
    const sd_status st = scratch_ptr(&ws);
    if (st != SD_OK) return st;
    // the counters must start at zero; clearing them every call keeps calls independent
    if (cudaMemsetAsync(ws, 0, sdv::WS_CNT_BYTES, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SD_ECUDA;
    return sd_qmatmul_multipos(qtype, w, n_out, k_in, q, scales, M, y, residual, epilogue, requant_col0, q_next,
                               scales_next, ws, SD_NOALLOC_SCRATCH_BYTES, stream);
}
