// sdv_abi.cu - status word, device queries, load-time repack, RMSNorm +
// requantisation, and the test hooks of the verify-pass library.
#include <mutex>
#include <set>
#include <utility>

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

cudaError_t allow_max_dynamic_smem(const void *kernel) {
    const int d = cur_dev();
    if (d < 0) return cudaErrorInvalidDevice;
    static std::mutex mu;
    static std::set<std::pair<const void *, int>> done;
    std::lock_guard<std::mutex> lk(mu);
    if (done.count({kernel, d})) return cudaSuccess;
    int optin = 0;
    cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kernel);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             optin - static_cast<int>(fa.sharedSizeBytes));
    if (e == cudaSuccess) done.insert({kernel, d});
    return e;
}

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

// ---------------------------------------------------------------------------
// K-quant super-blocks (256 weights) -> super-records of 32 rows (values unchanged)
// ---------------------------------------------------------------------------

// code of weight i (0..255) of a Q4_K super-block: 128 code bytes from byte 16, byte 32c + l holding
// weight 64c + l (low nibble) and 64c + 32 + l (high nibble)
__device__ __forceinline__ int q4k_code(const uint8_t *blk, int i) {
    const int c = i >> 6, r = i & 63;
    const uint8_t b = blk[16 + 32 * c + (r & 31)];
    return r < 32 ? (b & 15) : (b >> 4);
}

// 6-bit (scale, min) of sub-block s from the 12 packed bytes at blk + 4
__device__ __forceinline__ void q4k_scale_min_dev(const uint8_t *blk, int s, int &sc, int &mn) {
    const uint8_t *b = blk + 4;
    if (s < 4) {
        sc = b[s] & 63;
        mn = b[s + 4] & 63;
    } else {
        sc = (b[s + 4] & 15) | ((b[s - 4] >> 6) << 4);
        mn = (b[s + 4] >> 4) | ((b[s] >> 6) << 4);
    }
}

// unsigned 6-bit code (0..63) of weight i of a Q6_K super-block: low nibble from the first 128 bytes,
// two high bits from the next 64
__device__ __forceinline__ int q6k_code(const uint8_t *blk, int i) {
    const int n = i >> 7, r = i & 127, l = r & 31, k = r >> 5;
    const uint8_t lo = blk[64 * n + l + 32 * (k & 1)];
    const int low = k < 2 ? (lo & 15) : (lo >> 4);
    const int high = (blk[128 + 32 * n + l] >> (2 * k)) & 3;
    return low | (high << 4);
}

// Where the two high bits of nibble `nib` of code word 2h+e of a lane go in the lane's high-bit word h.
__device__ __forceinline__ int q6k_hi_pos(int e, int nib) {
    // nibbles 0..7 -> bit positions; e = 0: 4, 8, 6, 10, 20, 24, 22, 26; e = 1: 0, 2, 12, 14, 16, 18, 28, 30
    const int p0[8] = {4, 8, 6, 10, 20, 24, 22, 26}, p1[8] = {0, 2, 12, 14, 16, 18, 28, 30};
    return e ? p1[nib] : p0[nib];
}

// One thread per (super-record, lane): the lane's code words of the eight sub-blocks and, for lanes
// with c == 0, its row group's scales and super-block factors.
__global__ void repack_kq_kernel(int qtype, const uint8_t *__restrict__ src, int64_t SBK, int pair, int64_t F,
                                 uint8_t *__restrict__ dst, int64_t n_sr) {
    const int bb = qtype == SD_Q4_K ? 144 : 210;
    const int srb = qtype == SD_Q4_K ? 4736 : 6720;
    const int64_t total = n_sr * 32;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t sr = i >> 5;
        const int lane = static_cast<int>(i & 31), g = lane >> 2, c = lane & 3;
        int64_t row0, j;
        if (pair) {
            const int64_t pr = sr >> 1, half = sr & 1, tp = pr / SBK;
            j = pr - tp * SBK;
            row0 = tp * 32 + half * F;
        } else {
            const int64_t tile = sr / SBK;
            j = sr - tile * SBK;
            row0 = tile * 32;
        }
        auto blk = [&](int rr) -> const uint8_t * { return src + ((row0 + rr) * SBK + j) * bb; };
        uint8_t *d = dst + sr * srb;
        const int rows[4] = {g, g + 8, 16 + g, 24 + g};
        for (int s = 0; s < 8; ++s) {
            uint32_t words[4], hiw[2] = {0u, 0u};
            for (int jw = 0; jw < 4; ++jw) {
                const int t = jw >> 1, sk = jw & 1;
                uint32_t wv = 0;
                for (int nib = 0; nib < 8; ++nib) {
                    const int rr = 16 * t + g + ((nib & 2) ? 8 : 0);
                    const int kk = 32 * s + 16 * sk + 2 * c + ((nib & 1) ? 8 : 0) + (nib >> 2);
                    if (qtype == SD_Q4_K) {
                        wv |= static_cast<uint32_t>(q4k_code(blk(rr), kk)) << (4 * nib);
                    } else {
                        const int code = q6k_code(blk(rr), kk);
                        wv |= static_cast<uint32_t>(code & 15) << (4 * nib);
                        hiw[jw >> 1] |= static_cast<uint32_t>(code >> 4) << q6k_hi_pos(jw & 1, nib);
                    }
                }
                words[jw] = wv;
            }
            const int plane = qtype == SD_Q4_K ? 512 : 768;
            uint8_t *o = d + s * plane + lane * 16;
            for (int jw = 0; jw < 4; ++jw)
                for (int e = 0; e < 4; ++e) o[4 * jw + e] = static_cast<uint8_t>(words[jw] >> (8 * e));
            if (qtype == SD_Q6_K) {
                uint8_t *oh = d + s * plane + 512 + lane * 8;
                for (int h = 0; h < 2; ++h)
                    for (int e = 0; e < 4; ++e) oh[4 * h + e] = static_cast<uint8_t>(hiw[h] >> (8 * e));
            }
            if (c == 0) {
                for (int e = 0; e < 4; ++e) {
                    const uint8_t *bl = blk(rows[e]);
                    if (qtype == SD_Q4_K) {
                        int sc, mn;
                        q4k_scale_min_dev(bl, s, sc, mn);
                        d[4096 + 64 * s + 8 * g + e] = static_cast<uint8_t>(sc);
                        d[4096 + 64 * s + 8 * g + 4 + e] = static_cast<uint8_t>(mn);
                    } else {
                        d[6144 + 64 * s + 8 * g + e] = bl[192 + 2 * s];
                        d[6144 + 64 * s + 8 * g + 4 + e] = bl[192 + 2 * s + 1];
                    }
                }
            }
        }
        if (c == 0) {
            for (int e = 0; e < 4; ++e) {
                const uint8_t *bl = blk(rows[e]);
                if (qtype == SD_Q4_K) {
                    for (int q = 0; q < 4; ++q) d[4608 + 16 * g + 4 * e + q] = bl[q];  // d, dmin
                } else {
                    d[6656 + 8 * g + 2 * e] = bl[208];
                    d[6656 + 8 * g + 2 * e + 1] = bl[209];
                }
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

int sd_abi_version(void) { return 5; }

void sd_set_pdl(int enable) { g_pdl = enable ? 1 : 0; }

sd_status sd_device_status_site(sd_stream_t stream, int32_t *site) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!site) return SD_EINVAL;
    *site = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SD_ECUDA;
    int *p = status_ptr();
    if (!p) return SD_ECUDA;
    int v[2] = {0, 0};
    if (cudaMemcpy(v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return SD_ECUDA;
    if (v[0] != 0 || v[1] != 0) {
        int z[2] = {0, 0};
        if (cudaMemcpy(p, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess) return SD_ECUDA;
    }
    *site = v[1];
    return static_cast<sd_status>(v[0]);
}

int32_t sd_build_flags(void) {
#ifdef SD_DEBUG_BOUNDS
    return SD_BUILD_DEBUG_BOUNDS;
#else
    return 0;
#endif
}

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
    if (qtype == SD_Q4_K || qtype == SD_Q6_K) {
        if (n_out <= 0 || k_in <= 0 || k_in % 256 || n_out % 32) return 0;
        const int64_t srb = qtype == SD_Q4_K ? 4736 : 6720;
        if (flags & SD_REPACK_PAIR_GATE_UP) {
            if (qtype != SD_Q4_K || n_out % 64) return 0;
        }
        return static_cast<size_t>(n_out / 32 * (k_in / 256) * srb);
    }
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
    SD_NVTX("sd_repack_weights");
    size_t need = sd_repacked_bytes(qtype, n_out, k_in, flags);
    if (!need || !src_blocks || !dst || !aligned(dst, 16) || dst_bytes < need) return SD_EINVAL;
    if (qtype == SD_Q4_K || qtype == SD_Q6_K) {
        const int64_t n_sr = static_cast<int64_t>(need) / (qtype == SD_Q4_K ? 4736 : 6720);
        const int64_t threads = n_sr * 32;
        const int grid = static_cast<int>(threads / 256 + 1 < 65536 ? threads / 256 + 1 : 65536);
        repack_kq_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
            qtype, static_cast<const uint8_t *>(src_blocks), k_in / 256, (flags & SD_REPACK_PAIR_GATE_UP) ? 1 : 0,
            n_out / 2, static_cast<uint8_t *>(dst), n_sr);
        return cudaGetLastError() == cudaSuccess ? SD_OK : SD_ECUDA;
    }
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
