// sdv_abi.cu - status word, device queries, load-time repack, RMSNorm +
// requantisation, and the test hooks of the verify-pass library.
#include <mutex>

#include "sdv_common.cuh"

namespace sdv {

// One status word per device: a module-scope device variable, so every GPU
// that loads the library holds its own copy.  Host code reaches it through
// cudaGetSymbolAddress, looked up once per device.
static __device__ int g_status_word;

static std::mutex g_mu;
static int *g_status_addr[64];
static int g_sms[64];
static int g_pdl = 1;

static int cur_dev() {
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) return -1;
    return d;
}

int *status_ptr() {
    int d = cur_dev();
    if (d < 0) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_addr[d]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_addr[d] = static_cast<int *>(p);
    }
    return g_status_addr[d];
}

int num_sms() {
    int d = cur_dev();
    if (d < 0) return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sms[d]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 1;
        g_sms[d] = n;
    }
    return g_sms[d];
}

bool pdl_enabled() { return g_pdl != 0; }

// ---------------------------------------------------------------------------
// load-time repack: GGUF blocks -> 32-row tile records (values unchanged)
// ---------------------------------------------------------------------------

// one thread per (record, row): copies the row's code bytes and fp16 scale
__global__ void repack_kernel(int qtype, const uint8_t *__restrict__ src, int64_t n_out, int64_t KB, int pair,
                              int64_t F, uint8_t *__restrict__ dst, int64_t n_records) {
    const int bb = qtype == SD_Q8_0 ? 34 : 18;
    const int rec = qtype == SD_Q8_0 ? 1088 : 576;
    const int code_bytes = qtype == SD_Q8_0 ? 1024 : 512;
    int64_t total = n_records * 32;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        int64_t r_id = i >> 5;
        int row = static_cast<int>(i & 31);
        // record r_id -> (tile, block); pair mode: records come in (gate, up) pairs per (pair j, block b)
        int64_t tile, b;
        int64_t src_row;
        if (pair) {
            int64_t pr = r_id >> 1, half = r_id & 1;
            int64_t j = pr / KB;
            b = pr - j * KB;
            int64_t rr = j * 32 + row;  // row within gate (or up)
            src_row = rr < F ? rr + half * F : -1;
            tile = 0;
        } else {
            tile = r_id / KB;
            b = r_id - tile * KB;
            int64_t rr = tile * 32 + row;
            src_row = rr < n_out ? rr : -1;
        }
        uint8_t *d = dst + r_id * rec;
        const uint8_t *s = src_row >= 0 ? src + (src_row * KB + b) * bb : nullptr;
        if (qtype == SD_Q8_0) {
            for (int e = 0; e < 16; ++e) d[row * 16 + e] = s ? s[2 + e] : 0;
            for (int e = 0; e < 16; ++e) d[512 + row * 16 + e] = s ? s[2 + 16 + e] : 0;
        } else {
            for (int e = 0; e < 16; ++e) d[row * 16 + e] = s ? s[2 + e] : 0;
        }
        d[code_bytes + row * 2 + 0] = s ? s[0] : 0;
        d[code_bytes + row * 2 + 1] = s ? s[1] : 0;
    }
}

}  // namespace sdv

using namespace sdv;

extern "C" {

const char *sd_status_string(sd_status s) {
    switch (s) {
        case SD_OK: return "ok";
        case SD_EINVAL: return "invalid argument";
        case SD_EUNSUPPORTED: return "unsupported";
        case SD_ECUDA: return "CUDA error";
        case SD_ETIMEOUT: return "device wait timed out";
        case SD_EDEVICE: return "device-side check failed";
    }
    return "unknown status";
}

int sd_abi_version(void) { return 1; }

void sd_set_pdl(int enable) { g_pdl = enable ? 1 : 0; }

sd_status sd_device_status(sd_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return SD_ECUDA;
    int *p = status_ptr();
    if (!p) return SD_ECUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SD_ECUDA;
    if (v != 0) {
        int z = 0;
        if (cudaMemcpy(p, &z, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return SD_ECUDA;
    }
    return static_cast<sd_status>(v);
}

size_t sd_repacked_bytes(int qtype, int64_t n_out, int64_t k_in, uint32_t flags) {
    if ((qtype != SD_Q8_0 && qtype != SD_Q4_32) || n_out <= 0 || k_in <= 0 || k_in % 32) return 0;
    int64_t KB = k_in / 32;
    int64_t rec = qtype == SD_Q8_0 ? 1088 : 576;
    if (flags & SD_REPACK_PAIR_GATE_UP) {
        if (n_out % 2) return 0;
        int64_t F = n_out / 2, NP = (F + 31) / 32;
        return static_cast<size_t>(NP * 2 * KB * rec);
    }
    int64_t NT = (n_out + 31) / 32;
    return static_cast<size_t>(NT * KB * rec);
}

sd_status sd_repack_weights(int qtype, const void *src_blocks, int64_t n_out, int64_t k_in, uint32_t flags, void *dst,
                            size_t dst_bytes, sd_stream_t stream) {
    size_t need = sd_repacked_bytes(qtype, n_out, k_in, flags);
    if (!need || !src_blocks || !dst || !aligned(dst, 16) || dst_bytes < need) return SD_EINVAL;
    int64_t KB = k_in / 32;
    int64_t rec = qtype == SD_Q8_0 ? 1088 : 576;
    int64_t n_records = static_cast<int64_t>(need) / rec;
    int pair = (flags & SD_REPACK_PAIR_GATE_UP) ? 1 : 0;
    int64_t threads = n_records * 32;
    int grid = static_cast<int>(threads / 256 + 1 < 65536 ? threads / 256 + 1 : 65536);
    repack_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        qtype, static_cast<const uint8_t *>(src_blocks), n_out, KB, pair, n_out / 2, static_cast<uint8_t *>(dst),
        n_records);
    return cudaGetLastError() == cudaSuccess ? SD_OK : SD_ECUDA;
}

}  // extern "C"
