// sdv_abi.cu - status word, device queries, load-time repack, RMSNorm +
// requantisation, and the test hooks of the verify-pass library.
#include <mutex>

#include "sdv_common.cuh"

namespace sdv {

// One status word per device (plus the location code of a timeout): a module-scope
// device variable, so every GPU that loads the library holds its own copy.  Host
// code reaches it through cudaGetSymbolAddress, looked up once per device.
static __device__ int g_status_word[2];

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

// GGUF code byte / nibble of (row, k) of one block, k in 0..31
__device__ __forceinline__ int q4_code(const uint8_t *blk, int k) {
    return k < 16 ? (blk[2 + k] & 0x0F) : (blk[2 + k - 16] >> 4);
}

// One thread per (record, lane): writes the lane's code bytes in fragment order
// (see sdv_qmatmul.cuh) and, for lanes with c == 0, the group's four scales.
__global__ void repack_kernel(int qtype, const uint8_t *__restrict__ src, int64_t n_out, int64_t KB, int pair,
                              int64_t F, uint8_t *__restrict__ dst, int64_t n_records) {
    const int bb = qtype == SD_Q8_0 ? 34 : 18;
    const int rec = qtype == SD_Q8_0 ? 1088 : 576;
    const int code_bytes = qtype == SD_Q8_0 ? 1024 : 512;
    int64_t total = n_records * 32;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r_id = i >> 5;
        const int lane = static_cast<int>(i & 31), g = lane >> 2, c = lane & 3;
        int64_t row0, b, rows_valid;  // source row of record row 0; rows beyond rows_valid are padding
        if (pair) {
            const int64_t pr = r_id >> 1, half = r_id & 1, j = pr / KB;
            b = pr - j * KB;
            row0 = j * 32 + half * F;
            rows_valid = F - j * 32;  // gate and up halves have F rows each
        } else {
            const int64_t tile = r_id / KB;
            b = r_id - tile * KB;
            row0 = tile * 32;
            rows_valid = n_out - row0;
        }
        auto blk = [&](int rr) -> const uint8_t * {
            return rr < rows_valid ? src + ((row0 + rr) * KB + b) * bb : nullptr;
        };
        uint8_t *d = dst + r_id * rec;
        if (qtype == SD_Q4_32) {
            uint32_t words[4];
            for (int j = 0; j < 4; ++j) {
                const int t = j >> 1, s = j & 1;
                uint32_t wv = 0;
                for (int nib = 0; nib < 8; ++nib) {
                    const int dr = (nib & 2) ? 8 : 0;            // nibbles 2, 3, 6, 7: row + 8
                    const int dk = ((nib & 1) ? 8 : 0) + (nib >> 2);  // 1, 3, 5, 7: k + 8; 4..7: k + 1
                    const uint8_t *bl = blk(16 * t + g + dr);
                    const int code = bl ? q4_code(bl, 16 * s + 2 * c + dk) : 8;
                    wv |= static_cast<uint32_t>(code) << (4 * nib);
                }
                words[j] = wv;
            }
            for (int j = 0; j < 4; ++j)
                for (int e = 0; e < 4; ++e) d[lane * 16 + 4 * j + e] = static_cast<uint8_t>(words[j] >> (8 * e));
        } else {
            for (int w = 0; w < 8; ++w) {
                const int ts = w >> 1, h = w & 1, t = ts >> 1, s = ts & 1;
                const int k0 = 16 * s + 2 * c + 8 * h;
                const uint8_t *bg = blk(16 * t + g), *bg8 = blk(16 * t + g + 8);
                const uint8_t v[4] = {bg ? bg[2 + k0] : (uint8_t)0, bg ? bg[2 + k0 + 1] : (uint8_t)0,
                                      bg8 ? bg8[2 + k0] : (uint8_t)0, bg8 ? bg8[2 + k0 + 1] : (uint8_t)0};
                uint8_t *o = d + (t ? 512 : 0) + lane * 16 + 4 * (w & 3);
                for (int e = 0; e < 4; ++e) o[e] = v[e];
            }
        }
        if (c == 0) {
            const int rr[4] = {g, g + 8, 16 + g, 24 + g};
            for (int e = 0; e < 4; ++e) {
                const uint8_t *bl = blk(rr[e]);
                d[code_bytes + g * 8 + 2 * e] = bl ? bl[0] : 0;
                d[code_bytes + g * 8 + 2 * e + 1] = bl ? bl[1] : 0;
            }
        }
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

int sd_abi_version(void) { return 2; }

void sd_set_pdl(int enable) { g_pdl = enable ? 1 : 0; }

sd_status sd_device_status(sd_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return SD_ECUDA;
    int *p = status_ptr();
    if (!p) return SD_ECUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SD_ECUDA;
    if (v != 0) {
        int z[2] = {0, 0};
        if (cudaMemcpy(p, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return SD_ECUDA;
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
