/*
 * sdverify.h - C ABI of the GB300 (sm_103a) speculative-decoding verify pass.
 *
 * One verify pass reads block-quantised weights once and serves the current
 * token plus K drafts (M = K+1 positions) with that single read; the full-
 * vocabulary head follows, then greedy or rejection-sampling acceptance.
 *
 * General rules for every call below.
 *  - Pointers are DEVICE pointers unless a parameter says otherwise, owned by
 *    the caller, and must stay valid until the stream has passed the call.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  The return value covers argument validation
 *    (SD_EINVAL / SD_EUNSUPPORTED) and launch errors (SD_ECUDA) only.  Device-
 *    side conditions (a bounded wait that ran out, a bounds check) are recorded
 *    in a per-device status word read by sd_device_status().
 *  - Kernels are launched with programmatic dependent launch: each one may
 *    start streaming its weights while the previous kernel on the stream is
 *    still running, and waits for it before touching any dependent data.
 *  - The library allocates nothing except one status word per device, created
 *    on first use.  Scratch space is passed in as a caller-owned workspace.
 *  - Dimensions: k_in % 32 == 0 (blocks of 32 run along the reduction
 *    dimension), 1 <= M <= 16, n_out >= 1.  Weight, activation and logits
 *    pointers must be 16-byte aligned; workspaces 256-byte aligned.
 *
 * Quantised formats (GGUF order, as read from a model file):
 *  - SD_Q8_0:  per 32 weights, fp16 scale d (little endian) then 32 int8 q;
 *              value d*q; 34 bytes per block.
 *  - SD_Q4_32: per 32 weights, fp16 scale d then 16 bytes; byte j holds
 *              element j in its low nibble and element j+16 in its high
 *              nibble; value d*(code-8); 18 bytes per block.
 * A weight matrix is [n_out rows][k_in/32 blocks] of such blocks.
 * K-quant super-blocks of 256 weights (the GGUF K formats of the Q4_K_M model
 * files the pages run: "Inside OpenJet Engine", section "One GPU launch for a
 * speculative cycle", and "How Kinetic is fast", opening section); a matrix is
 * [n_out rows][k_in/256 super-blocks], n_out % 32 == 0, k_in % 256 == 0:
 *  - SD_Q4_K (144 B): fp16 d, fp16 dmin, 12 bytes of eight 6-bit (scale,
 *              min) pairs (pair s < 4: scale = b[s] & 63, min = b[s+4] & 63;
 *              s >= 4: scale = (b[s+4] & 15) | (b[s-4] >> 6) << 4, min =
 *              (b[s+4] >> 4) | (b[s] >> 6) << 4), 128 bytes of 4-bit codes
 *              (byte 32c + l holds weight 64c + l in its low nibble and 64c +
 *              32 + l in its high one); weight = d scale_s code - dmin min_s
 *              for the 32-weight sub-block s.
 *  - SD_Q6_K (210 B): 128 bytes of low code nibbles, 64 bytes of high 2-bit
 *              pairs, 16 int8 scales, fp16 d; weight i (n = i/128, r = i%128,
 *              l = r%32, k = r/32): low = byte 64n + l + 32(k&1), its low
 *              nibble for k < 2 else its high one; high = (byte 128 + 32n + l
 *              >> 2k) & 3; weight = d scale[i/16] (low | high << 4 - 32).
 */
#ifndef SDVERIFY_H
#define SDVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *sd_stream_t; /* same type as cudaStream_t */

typedef enum {
    SD_OK = 0,
    SD_EINVAL = 1,        /* bad argument: null, misaligned, out-of-range size */
    SD_EUNSUPPORTED = 2,  /* valid but not supported (format, M > 16) */
    SD_ECUDA = 3,         /* a CUDA runtime call or launch failed */
    SD_ETIMEOUT = 4,      /* a bounded device-side wait ran out (from sd_device_status) */
    SD_EDEVICE = 5        /* a device-side check failed (from sd_device_status) */
} sd_status;

typedef enum { SD_Q8_0 = 0, SD_Q4_32 = 1, SD_Q4_K = 2, SD_Q6_K = 3 } sd_qtype;

/* Repack flags */
#define SD_REPACK_PAIR_GATE_UP 1u /* rows [0,F) are gate and [F,2F) are up; store them pairwise */

/* Matmul epilogues */
#define SD_EPI_NONE 0u              /* y = residual + W a */
#define SD_EPI_REQUANT 1u           /* also requantise columns [requant_col0, n_out) into q_next/scales_next */
#define SD_EPI_SILU_MUL_REQUANT 2u  /* gate|up pair: h = silu(g) * u, requantised into q_next/scales_next */

const char *sd_status_string(sd_status s);
int sd_abi_version(void); /* 5: sd_head_shortlist takes the repacked head and returns sd_head_logits' argmax;
                           4: sd_device_status_site and sd_build_flags; 3: sd_pass_desc carries the down
                           projections' format, sd_pass the K-quant flag */

/*
 * Load-time repack ("Inside OpenJet Engine", section "One GPU launch for a
 * speculative cycle": Q8_0 weights are rearranged at load time for aligned
 * access without changing their values).
 *
 * src: GGUF-order blocks [n_out][k_in/32] (device).  dst: dst_bytes >=
 * sd_repacked_bytes(...).  Layout of dst: tiles of 32 rows (the last tile
 * padded with zero scales); per (tile t, block b) one 16-byte-aligned record
 * of the 32 rows' codes followed by their 32 fp16 scales, records ordered
 * (t, b).  Inside a record the codes are placed where lane l = 4g + c of a
 * warp finds its mma.sync m16n8k16 operand fragments (rows 16t'+g and
 * 16t'+g+8, k = 16s+2c, +1, +8, +9 for row half t' and k step s):
 *   SD_Q4_32 (576 B): 16 code bytes per lane; word 2t'+s, nibble i holds
 *     (row 16t'+g + 8*[i&2], k 16s+2c + 8*[i&1] + (i>>2)); then 64 B scales.
 *   SD_Q8_0 (1088 B): two 512-B planes (t' = 0, 1) of 16 bytes per lane; word
 *     2s+h holds (row 16t'+g, k0), (row 16t'+g, k0+1), (row 16t'+g+8, k0),
 *     (row 16t'+g+8, k0+1), k0 = 16s+2c+8h; then 64 B scales.
 *   Scales: 8 groups of 4 fp16, group g = rows g, g+8, 16+g, 24+g.
 * With SD_REPACK_PAIR_GATE_UP (n_out = 2F) the record of gate tile j is
 * followed by the record of up tile j, pairs ordered (j, b).  Values are
 * unchanged; only their places move.
 * K-quants: per (tile, super-block) one super-record of the 32 rows' 256
 * weights, ordered (tile, super-block); 32-weight sub-block s's codes sit in
 * the fragment order above.
 *   SD_Q4_K (4736 B): eight 512-B code planes (sub-block s at 512 s, as
 *     SD_Q4_32); at 4096 + 64 s + 8 g the bytes scale of rows g, g+8, 16+g,
 *     24+g then min of the same rows (sub-block s); at 4608 + 16 g the fp16
 *     (d, dmin) of rows g, g+8, 16+g, 24+g.  The 6-bit fields are stored as
 *     bytes: 32 B per 32 x 256 weights more than the file (2.8 %).
 *   SD_Q6_K (6720 B, the file's bytes): per sub-block s at 768 s, 512 B of low
 *     nibbles (as SD_Q4_32) and 256 B of high bits, 8 B per lane: word h
 *     covers code words 2h, 2h+1; for code word 2h the two high bits of its
 *     nibbles 0, 4, 2, 6, 1, 5, 3, 7 sit at bits 4, 20, 6, 22, 8, 24, 10, 26;
 *     for code word 2h+1 at bits 0, 16, 12, 28, 2, 18, 14, 30; at 6144 + 64 s
 *     + 8 g the int8 scales of rows g, g+8, 16+g, 24+g for weights 0-15 then
 *     16-31 of sub-block s; at 6656 + 8 g the fp16 d of rows g, g+8, 16+g, 24+g.
 *   With SD_REPACK_PAIR_GATE_UP (SD_Q4_K only) the gate super-record of tile
 *   j is followed by the up super-record of tile j.
 * Errors: SD_EINVAL on null/misaligned pointers, k_in % 32 != 0 (K-quants:
 * k_in % 256 != 0 or n_out % 32 != 0; the pair flag with SD_Q6_K), odd n_out
 * with the pair flag, or dst_bytes too small.
 */
size_t sd_repacked_bytes(int qtype, int64_t n_out, int64_t k_in, uint32_t flags);
sd_status sd_repack_weights(int qtype, const void *src_blocks, int64_t n_out, int64_t k_in, uint32_t flags,
                            void *dst, size_t dst_bytes, sd_stream_t stream);

/*
 * RMSNorm fused with per-32-block int8 requantisation of M activation rows
 * ("Inside OpenJet Engine", section "One GPU launch for a speculative cycle":
 * the producing phase requantises activations for the next consumer,
 * including the next RMS normalisation's weight).
 *
 * x: fp32 [M][ldx] (row stride ldx >= K elements).  norm_w: fp32 [K], or NULL
 * for requantisation only.  Out: q int8 [M][K], scales fp32 [M][K/32].
 * Arithmetic (bit-exact contract): s = sum x^2 as, per 32-element block, a
 * pairwise tree over the block's rounded squares (strides 16, 8, 4, 2, 1),
 * then a pairwise tree over the K/32 block sums zero-padded to a power of two
 * of at least 256 slots; inv = 1/sqrt(s/K + eps) correctly rounded.  Codes of
 * the normalised row y = x*inv*w are formed from t = x*w: per block c =
 * amax|t|/127, q = round-half-away(t/c) clamped to +-127 (0 if c=0), scale
 * d = inv*c (in exact arithmetic the requantisation of y, whose row factor
 * cancels in the codes).  Without norm_w: c and q from x, d = c.  With norm_w,
 * K/32 <= 2048 (else SD_EUNSUPPORTED).
 */
sd_status sd_rmsnorm_quant_acts(const float *x, int64_t ldx, const float *norm_w, float eps, int32_t M,
                                int64_t K, int8_t *q, float *scales, sd_stream_t stream);

/*
 * Multi-position quantised matmul: one pass over the repacked weights serves
 * all M positions ("Inside OpenJet Engine", section "One GPU launch for a
 * speculative cycle": integer dot products with int8 activations, weight reads
 * serving multiple verification positions).
 *
 *   y[m][n] = residual[m][n] + sum_b d_w[n,b] * d_a[m,b] * dot_b(n, m)
 *
 * dot_b is the exact int32 dot of one 32-block (4-bit: sum (code-8) a).
 * w: repacked by sd_repack_weights with the same qtype/n_out/k_in (and the
 * pair flag iff epilogue == SD_EPI_SILU_MUL_REQUANT).  q int8 [M][k_in],
 * scales fp32 [M][k_in/32].  y fp32 [M][n_out] (may be NULL for the two
 * requantising epilogues); residual fp32 [M][n_out] or NULL (may alias y).
 * SD_EPI_REQUANT: requant_col0 % 32 == 0; q_next int8 [M][n_out-col0],
 * scales_next fp32 [M][(n_out-col0)/32] receive the per-32 requantisation of
 * y's columns [col0, n_out).  SD_EPI_SILU_MUL_REQUANT: n_out = 2F, F % 32 ==
 * 0; q_next [M][F], scales_next [M][F/32] receive requant(silu(g)*u) with g =
 * columns [0,F), u = [F,2F) and silu(g) = g / (1 + exp(-g)); if y is given it
 * receives g|u.  The reduction order of each output depends on (n_out, k_in,
 * the device's SM count) only, never on M, so a row computed among M
 * positions equals the same row computed alone, bit for bit.
 * workspace: ws_bytes >= sd_qmatmul_workspace_bytes(...), zero-filled by the
 * caller once.  Its first 160 KB are counters at fixed offsets that every call
 * returns to zero; the rest is scratch.  One workspace may therefore serve
 * calls of any shape (sized for the largest), as long as they are ordered on
 * one stream.  After an SD_ETIMEOUT it must be zero-filled again.
 */
size_t sd_qmatmul_workspace_bytes(int qtype, int64_t n_out, int64_t k_in, uint32_t epilogue);
sd_status sd_qmatmul_multipos(int qtype, const void *w, int64_t n_out, int64_t k_in, const int8_t *q,
                              const float *scales, int32_t M, float *y, const float *residual, uint32_t epilogue,
                              int64_t requant_col0, int8_t *q_next, float *scales_next, void *workspace,
                              size_t ws_bytes, sd_stream_t stream);

/*
 * The multi-position matmul without a caller-supplied workspace.  The papers
 * have no counterpart: this is a convenience of this library, not a step of
 * the method.
 *
 * For callers that cannot hand the library device memory: code that runs
 * after a fixed start-up budget has been allocated and may not allocate
 * again, or a host whose allocator the library must not touch.  Arguments and
 * results are those of sd_qmatmul_multipos without `workspace`/`ws_bytes`;
 * the stream-K counters and partial sums live instead in one static device
 * array of SD_NOALLOC_SCRATCH_BYTES per device, inside this library.
 *
 * Allocates nothing: no cudaMalloc/cudaFree, no allocating library routine.
 * The first call on each device looks up that device's scratch address (with
 * the device current) and caches it; make that first call before any stream
 * capture.  Every call clears the scratch's counter region on `stream` before
 * its launch, so no state carries over between calls, including after
 * SD_ETIMEOUT.  Calls whose workspace (sd_qmatmul_workspace_bytes) exceeds
 * SD_NOALLOC_SCRATCH_BYTES are rejected with SD_EUNSUPPORTED before anything
 * is launched (every 27B-shaped projection fits; a 65536 x 17408 one does
 * not).  All calls share the one scratch array: calls that may overlap
 * on the device (different streams, or several host threads) race on it and
 * must be ordered by the caller.
 */
#define SD_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)
sd_status sd_qmatmul_multipos_noalloc(int qtype, const void *w, int64_t n_out, int64_t k_in, const int8_t *q,
                                      const float *scales, int32_t M, float *y, const float *residual,
                                      uint32_t epilogue, int64_t requant_col0, int8_t *q_next, float *scales_next,
                                      sd_stream_t stream);

/*
 * Full-vocabulary output head with fused per-row argmax and softmax
 * statistics ("Inside OpenJet Engine", section "One GPU launch for a
 * speculative cycle": full-vocabulary output head + verification inside the
 * cycle; "How Kinetic is fast", section "Why the output does not change").
 *
 * w: Q8_0 head repacked (vocab rows, hidden = k_in).  Out: logits fp32
 * [M][vocab]; argmax int32 [M] over the raw logits (lowest index on ties);
 * row_max, row_sumexp fp32 [M] of z = logits / temperature: tiles of 1024
 * tokens, per tile m_t = max z and s_t = pairwise tree (strides 512..1, zero
 * padded) of exp(z - m_t); m = max m_t, Z = sequential fold of s_t *
 * exp(m_t - m).  exp is the canonical Cody-Waite/Taylor exponential shared
 * by the acceptance kernel, so these statistics equal what sd_accept_sample
 * recomputes.  Workspace as for the matmul (sd_head_workspace_bytes).
 */
size_t sd_head_workspace_bytes(int64_t vocab, int64_t hidden);
sd_status sd_head_logits(const void *w, int64_t vocab, int64_t hidden, const int8_t *q, const float *scales,
                         int32_t M, float temperature, float *logits, int32_t *argmax, float *row_max,
                         float *row_sumexp, void *workspace, size_t ws_bytes, sd_stream_t stream);

/*
 * Exact shortlist head for greedy verification ("How Kinetic is fast",
 * section "Shortlist": a cheaper copy of the output layer with a proven bound
 * on each row's error scores every row, the best guaranteed score becomes a
 * floor, and only rows whose bound reaches the floor are scored exactly).
 *
 * sd_shortlist_build (load time): head_blocks is the Q8_0 head in GGUF order
 * [vocab][hidden/32] (device, 16-byte aligned).  Writes copy_blocks, the
 * SD_Q4_32 copy in GGUF order (vocab * hidden/32 * 18 bytes): per block d =
 * amax|w|/7.5 rounded to fp16 (nearest even; held at 65504 if larger), code =
 * 8 + round-half-away(w/d) clamped to [0, 15] (8 if d = 0); bound[r] >=
 * ||w8_r - w4_r||_2 and wnorm[r] >= ||w8_r||_2 (fp32, rounded up) of the
 * dequantised rows.  Repack copy_blocks with sd_repack_weights(SD_Q4_32, ...,
 * flags 0) for sd_head_shortlist.  Weights must be finite.
 *
 * sd_head_shortlist (verify time): copy_w the repacked copy, bound / wnorm
 * from the build, head_w the REPACKED Q8_0 head (as for sd_head_logits); q
 * int8 [M][hidden], scales fp32 [M][hidden/32] as for sd_head_logits;
 * 1 <= M <= 16.  argmax int32 [M] receives, per position, sd_head_logits'
 * argmax on the same inputs, bit for bit: the row of the largest fp32 logit
 * of the head's own matmul (lowest index among equal maxima).  The copy's
 * scores and bounds rule rows out; the 32-row tiles holding the remaining
 * candidates are scored by the head's matmul restricted to them (same plan,
 * same arithmetic as sd_head_logits).  n_cand int32 [M] (or NULL) receives
 * the candidate count per position (vocab in full mode).  Full mode: when the
 * previous call's candidates filled more than a quarter of the tiles, the call
 * skips the copy and scores every tile (the full head plus a few empty
 * launches), trying the shortlist again every 16th call.
 * Device-side: a position with no candidate (non-finite inputs only) records
 * SD_EDEVICE in the status word and gets argmax -1.  workspace: ws_bytes >=
 * sd_shortlist_workspace_bytes(vocab, hidden), zero-filled by the caller once
 * and kept between calls (it holds counters that every call returns to zero,
 * and the mode state).
 * Errors: SD_EINVAL on null/misaligned pointers or bad sizes; SD_EUNSUPPORTED
 * for M > 16.
 */
/*
 * Decode attention over the K+1 verified positions ("Inside OpenJet Engine",
 * section "Cheap drafting, careful state management": split-K flash decoding
 * of full-attention layers, fp16 K/V, fp32 accumulation; "How Kinetic is
 * fast", section "Where the guesses come from": each row of a draft tree sees
 * only its own path; "Speculative Decoding with Open-Weights Models", section
 * "Engineering the Architecture: KV Cache Synchronization": rejected entries
 * are dropped in place).
 *
 * Cache layout (per layer, caller-owned, 16-byte aligned): k_cache and
 * v_cache fp16 [H_kv][S_max][D]; rows [0, L) are committed, rows [L, L+M)
 * hold the M = K+1 new positions.
 *
 * sd_kv_append: k_new, v_new fp32 [M][H_kv][D] -> rows [L, L+M), rounded to
 * fp16 (nearest even).  Requires S_max >= L + M.
 *
 * sd_attn_decode: q fp32 [M][H][D] (H a multiple of H_kv; query head h reads
 * KV head h / (H/H_kv)); parent int32 [M] (device) with parent[0] = -1 and
 * parent[i] < i for a draft tree, or NULL for a chain.  out fp32 [M][H][D]:
 *   out[i][h] = sum_j softmax_j(q[i][h] . k_j / sqrt(D)) v_j
 * over the committed rows and the new rows L+j with j on i's path (j = i or
 * an ancestor; chain: j <= i).  fp32 arithmetic from the fp16 cache; keys
 * split into chunks, one partial (max, sum, output) per chunk, then combined.
 * D = 64 or 128, 1 <= M <= 16 (else SD_EUNSUPPORTED).  workspace: ws_bytes >=
 * sd_attn_workspace_bytes(M, H, H_kv, D, L), no initialisation needed; the
 * size for the longest context serves every shorter one (the number of key
 * chunks is capped by the SM count, not the context).  A
 * parent array that is not a tree (parent[i] >= i) records SD_EDEVICE.
 *
 * sd_kv_commit: after acceptance, keep the accepted entries: *count (device,
 * the accepted token count n, 1 <= n <= M) rows; path int32 [M] (device)
 * lists the accepted tree nodes in increasing order (node 0 first), and row
 * L+path[t] moves to row L+t for t < n, in place.  path NULL: a chain, whose
 * first n rows are already in place (nothing is launched).  The cache length
 * becomes L+n.  A count or path out of range records SD_EDEVICE and moves
 * nothing.  D <= 256.  The same call rolls a drafter's own cache back after
 * verification ("Speculative Decoding with Open-Weights Models", section
 * "Engineering the Architecture: KV Cache Synchronization"): its rows for the
 * rejected drafts are dropped and the accepted path is made contiguous, so
 * both caches continue from length L+n.
 */
/*
 * Adaptive draft depth, host only ("Inside OpenJet Engine", section "Cheap
 * drafting, careful state management": a configured depth is cut by one for
 * the cycle after a rejection; "How Kinetic is fast", section "Where the
 * guesses come from": draft length follows recent drafts, and outright misses
 * pause drafting for longer and longer).
 *
 * The state lives in caller memory (HOST pointer); nothing touches a device.
 * sd_depth_init: k_max drafts per cycle (1..15), max_pause >= 0 cycles;
 * k_next = k_max.  Run the next cycle with k_next drafts (0: plain decoding,
 * M = 1), then call sd_depth_update with the number of drafts accepted:
 *   all k_next accepted      -> k_next = k_max, miss count 0
 *   some, not all            -> k_next = max(1, k_max - 1), miss count 0
 *   none (an outright miss)  -> miss count + 1; pause_left =
 *                               min(max_pause, 2^(misses - 1)) cycles with
 *                               k_next = 0 (none if max_pause is 0), then
 *                               k_next = max(1, k_max - 1)
 *   a cycle with k_next = 0  -> pause_left - 1 (accepted is ignored)
 * Errors: SD_EINVAL on a null or uninitialised state, or accepted outside
 * [0, k_next].
 */
typedef struct {
    int32_t k_max;      /* configured depth */
    int32_t max_pause;  /* longest pause, in cycles */
    int32_t k_next;     /* drafts for the next cycle; 0 = no drafting */
    int32_t pause_left; /* cycles without drafts still to run */
    int32_t misses;     /* outright misses in a row */
} sd_depth_state;
sd_status sd_depth_init(sd_depth_state *s, int32_t k_max, int32_t max_pause);
sd_status sd_depth_update(sd_depth_state *s, int32_t accepted);

/*
 * The accepted path of a greedy draft tree as node indices (HOST pointers,
 * no device work): the rule of sd_accept_greedy with a parent array, path
 * int32 [M] receives the accepted nodes root first (node 0, then each
 * accepted draft down to the deepest, lowest index among equals).  Returns
 * the node count n (the accepted token count sd_accept_greedy reports), or -1
 * for null pointers, M outside 1..16, parent[0] != -1 or parent[i] not in
 * [0, i).  Copy path to the device for sd_kv_commit.
 */
int32_t sd_tree_path(const int32_t *argmax, const int32_t *tokens, const int32_t *parent, int32_t M, int32_t *path);

size_t sd_attn_workspace_bytes(int32_t M, int32_t H, int32_t H_kv, int32_t D, int64_t L);
sd_status sd_kv_append(const float *k_new, const float *v_new, int32_t M, int32_t H_kv, int32_t D, void *k_cache,
                       void *v_cache, int64_t S_max, int64_t L, sd_stream_t stream);
sd_status sd_attn_decode(const float *q, const void *k_cache, const void *v_cache, int32_t M, int32_t H, int32_t H_kv,
                         int32_t D, int64_t S_max, int64_t L, const int32_t *parent, float *out, void *workspace,
                         size_t ws_bytes, sd_stream_t stream);
sd_status sd_kv_commit(void *k_cache, void *v_cache, int32_t H_kv, int32_t D, int64_t S_max, int64_t L, int32_t M,
                       const int32_t *path, const int32_t *count, sd_stream_t stream);

sd_status sd_shortlist_build(const void *head_blocks, int64_t vocab, int64_t hidden, void *copy_blocks, float *bound,
                             float *wnorm, sd_stream_t stream);
size_t sd_shortlist_workspace_bytes(int64_t vocab, int64_t hidden);
sd_status sd_head_shortlist(const void *copy_w, const float *bound, const float *wnorm, const void *head_w,
                            int64_t vocab, int64_t hidden, const int8_t *q, const float *scales, int32_t M,
                            int32_t *argmax, int32_t *n_cand, void *workspace, size_t ws_bytes, sd_stream_t stream);

/*
 * Greedy acceptance ("How Kinetic is fast", section "Why the output does not
 * change": keep a guess only when it is the model's top token; section
 * "RAD-1": tree drafts, each row seeing only its own path).
 *
 * parent == NULL (chain): tokens = drafts [M-1]; row i predicts the token
 * after position i.  n = largest j with tokens[i-1] == argmax[i-1] for all
 * i <= j; out_tokens[0..n] = tokens[0..n-1], argmax[n]; *out_count = n+1.
 * parent != NULL (tree, nodes in BFS order, parent[0] = -1, parent[i] < i):
 * tokens [M] (tokens[0] unused).  Node i is accepted when its parent is and
 * tokens[i] == argmax[parent[i]]; the deepest accepted node (lowest index
 * among equals) ends the path; out = the path's tokens, then its argmax.
 * out_tokens: int32 [M]; out_count: int32 [1].
 */
sd_status sd_accept_greedy(const int32_t *argmax, const int32_t *tokens, const int32_t *parent, int32_t M,
                           int32_t *out_tokens, int32_t *out_count, sd_stream_t stream);

/*
 * Rejection-sampling acceptance ("Speculative Decoding with Open-Weights
 * Models", section "Mathematical Integrity: Rejection Sampling for LLMs":
 * accept x with min(1, p(x)/q(x)), on rejection draw from max(0, p-q)
 * renormalised; its walkthrough draws a bonus token from the last row when
 * every draft is kept.  "How Kinetic is fast", section "Why the output does
 * not change": a certainty drafter keeps x with probability p(x) and otherwise
 * draws from p without x).
 *
 * logits fp32 [K+1][vocab]; row_max / row_sumexp from sd_head_logits at the
 * same temperature, or NULL to recompute them identically; q_probs fp32
 * [K][vocab], or NULL for a certainty drafter (q one-hot at the draft);
 * drafts int32 [K].  Uniforms: Philox4x32-10 keyed by seed with counter
 * (position lo, position hi, 0, 0), position = base_pos + row; word 0 ->
 * accept uniform, word 1 -> residual or bonus uniform, u = (w >> 8) * 2^-24.
 * Draft i is kept iff u * q_i(x) < p_i(x).  The residual draw is an inverse
 * CDF over 1024-token tiles, 32-token chunks and single tokens with sequential
 * folds.  K <= 15.  out_tokens int32 [K+1]; *out_count = kept + 1.
 */
sd_status sd_accept_sample(const float *logits, int64_t vocab, int32_t K, const float *row_max,
                           const float *row_sumexp, const float *q_probs, const int32_t *drafts, float temperature,
                           uint64_t seed, int64_t base_pos, int32_t *out_tokens, int32_t *out_count,
                           sd_stream_t stream);

/*
 * The same rule against a filtered target: the sampling knobs of "Inside
 * OpenJet Engine" (API section: temperature, top-k up to 32, top-p), applied in
 * this order (a reading; the page does not fix it).  Row i: z = l / T; the
 * candidates are the top_k tokens by z (larger first, lower index among equal
 * z); with e_c = cexp(z_c - z_first) in that order and S their sequential sum,
 * the nucleus is the shortest prefix whose running sum reaches top_p * S, and
 * the target is p'_c = e_c / (that running sum), 0 outside the nucleus.  The
 * draft x is kept iff u * q(x) < p'(x); a rejection draws from
 * max(0, p'_c - q(c)) over the nucleus in candidate order (p' if that is all
 * zero), a full acceptance draws the bonus token from p' of row K, both by a
 * sequential inverse CDF (the first c with w > 0 whose running sum exceeds
 * u * W).  Uniforms, q_probs, drafts and outputs as in sd_accept_sample.
 * 1 <= top_k <= 32, 0 < top_p <= 1, K <= 15; logits fp32 [K+1][vocab].
 */
sd_status sd_accept_sample_topk(const float *logits, int64_t vocab, int32_t K, const float *q_probs,
                                const int32_t *drafts, float temperature, int32_t top_k, float top_p, uint64_t seed,
                                int64_t base_pos, int32_t *out_tokens, int32_t *out_count, sd_stream_t stream);

/*
 * The whole verify pass in one persistent cooperative launch ("Inside OpenJet
 * Engine", section "One GPU launch for a speculative cycle": one persistent
 * kernel carries the cycle's phases with a software grid barrier between them).
 *
 * Per layer: RMSNorm + requant -> QKV (3H, columns [2H, 3H) requantised in the
 * epilogue) -> O on those codes (+ residual into h) -> RMSNorm + requant ->
 * gate|up (SiLU*mul requant epilogue) -> down (+ residual into h); then the final
 * RMSNorm, the Q8_0 vocabulary head with argmax / statistics, and greedy
 * acceptance (chain, or tree when parent != NULL) or rejection sampling (below).  Every phase runs the same
 * device code as the single-operation calls above, so the pass produces the
 * same bits as issuing those calls one by one.  Between phases the CTAs meet at
 * a grid barrier (release/acquire on a counter in the plan, each wait bounded
 * to 2 s, SD_ETIMEOUT in the status word on expiry); the weight stream never
 * waits for it.
 *
 * sd_layer / sd_pass_desc: device pointers to repacked weights in format wq
 * (SD_Q4_32 or SD_Q4_K; gate_up repacked with SD_REPACK_PAIR_GATE_UP; down in
 * wq_down) and fp32 norm weights [hidden]; the head is Q8_0.  K-quant stacks
 * (hidden and ffn multiples of 256) take greedy acceptance only
 * (SD_EUNSUPPORTED otherwise).  h [M][hidden]
 * is the residual stream (input rows in, final hidden state out); qa/sa
 * [M][hidden], qv/sv [M][hidden], qf/sf [M][ffn] (and [.../32] scales) are
 * activation scratch; logits [M][vocab], argmax/row_max/row_sumexp [M];
 * tokens = drafts [M-1] (chain) or node tokens [M] (tree); out_tokens [M],
 * out_count [1].  workspace: >= sd_pass_workspace_bytes, zero-filled once.
 * accept = SD_ACCEPT_SAMPLE replaces greedy acceptance by the rejection sampling of
 * sd_accept_sample on the pass's own logits and statistics (drafts = tokens
 * [M-1], K = M - 1, temperature, q_probs, seed, base_pos as there; chains only:
 * parent must be NULL, else SD_EUNSUPPORTED); it produces the same tokens as the
 * head followed by sd_accept_sample, or with top_k > 0 by sd_accept_sample_topk.
 * layers is a HOST array read only by sd_pass_prepare.
 * sd_pass_prepare writes the phase table, and the combine phases' pieces per
 * (unit, split) from a host replay of their schedule, into `plan` (device,
 * 256-byte aligned, >= sd_pass_plan_bytes(n_layers), synchronously) and fills
 * `out`; sd_verify_pass launches it on `stream` (capturable in a CUDA graph).
 * The launch runs one CTA per SM; it fails with SD_ECUDA rather than wait if
 * the GPU cannot hold them all at once.
 */
typedef struct {
    const void *qkv, *o, *gate_up, *down;
    const float *norm1, *norm2;
} sd_layer;

typedef struct {
    int32_t n_layers;
    int64_t hidden, ffn, vocab;
    int32_t M;
    int32_t wq; /* SD_Q4_32 */
    float eps;
    float temperature;
    const sd_layer *layers;
    const float *final_norm;
    const void *head; /* Q8_0, repacked */
    float *h;
    int8_t *qa;
    float *sa;
    int8_t *qv;
    float *sv;
    int8_t *qf;
    float *sf;
    float *logits;
    int32_t *argmax;
    float *row_max;
    float *row_sumexp;
    const int32_t *tokens;
    const int32_t *parent;
    int32_t *out_tokens;
    int32_t *out_count;
    void *workspace;
    size_t ws_bytes;
    int32_t accept;        /* SD_ACCEPT_GREEDY (0) or SD_ACCEPT_SAMPLE (1) */
    const float *q_probs;  /* SD_ACCEPT_SAMPLE: drafter probabilities [M-1][vocab], NULL = certainty drafter */
    uint64_t seed;         /* SD_ACCEPT_SAMPLE: Philox key and position of the first draft */
    int64_t base_pos;
    int32_t top_k;         /* SD_ACCEPT_SAMPLE: 0 = unfiltered target (sd_accept_sample), 1..32 = */
    float top_p;           /* the filtered target of sd_accept_sample_topk with top_p in (0, 1] */
    int32_t wq_down;       /* format of the down projections: 0 = wq; SD_Q6_K with wq = SD_Q4_K (the */
                           /* Q4_K_M recipe: Q4_K projections, Q6_K down projections) */
} sd_pass_desc;

typedef enum { SD_ACCEPT_GREEDY = 0, SD_ACCEPT_SAMPLE = 1 } sd_accept_mode;

typedef struct {
    void *plan;
    int32_t n_phases;
    int32_t nt;
    uint32_t smem_bytes;
    int32_t grid;
    int32_t accept; /* the descriptor's acceptance mode */
    int32_t kq;     /* 1 when the stack's weights are K-quants */
} sd_pass;

size_t sd_pass_plan_bytes(int32_t n_layers);
size_t sd_pass_workspace_bytes(int64_t hidden, int64_t ffn, int64_t vocab, int32_t wq);
sd_status sd_pass_prepare(const sd_pass_desc *desc, void *plan, size_t plan_bytes, sd_pass *out);
sd_status sd_verify_pass(const sd_pass *pass, sd_stream_t stream);

/* Tracing (no counterpart on the pages; a profiling aid, since a persistent
 * launch hides its phases from host-side tools): the same pass as
 * sd_verify_pass, plus global-timer stamps (nanoseconds) written into `trace`
 * (device, 8-byte aligned, >= sd_pass_trace_bytes(pass) bytes, caller-owned).
 * Layout, uint64: trace[c] = SM id of CTA c for c < grid; then for phase p and
 * CTA c 12 values at grid + (p * grid + c) * 12.  Global-timer stamps: the phase
 * begins (grid barrier passed), the consumers hold their first activations
 * (matmul phases), the consumers leave the phase, the phase ends, and the
 * producer starts and finishes issuing the phase's weight copies (matmul
 * phases).  Then SM cycles one consumer warp spent in the phase waiting for
 * weight stages, computing records, handing partial sums on, staging a
 * split's activations (the wait for their copy and the RMSNorm row factors
 * included), finishing the CTA's last tile, and in the whole phase.  Values a
 * phase does not reach are left as they were.  Results equal sd_verify_pass's.
 * SD_EINVAL for a null, misaligned or short buffer. */
size_t sd_pass_trace_bytes(const sd_pass *pass);
sd_status sd_verify_pass_traced(const sd_pass *pass, uint64_t *trace, size_t trace_bytes, sd_stream_t stream);

/* Synchronises `stream`, returns and clears the current device's status word
 * (SD_OK, SD_ETIMEOUT or SD_EDEVICE); SD_ECUDA if synchronising failed. */
sd_status sd_device_status(sd_stream_t stream);

/* The same, also returning where the condition was recorded: *site (HOST
 * pointer) = 1 the launch-wide time bound ran out in a producer, 2 in a
 * consumer; >= 100 a bounds check of the debug build failed (the site numbers
 * are listed with the checks in the kernels' sources); 0 otherwise.  SD_EINVAL
 * if site is NULL. */
sd_status sd_device_status_site(sd_stream_t stream, int32_t *site);

/* Build variant: SD_BUILD_DEBUG_BOUNDS set when the library was compiled with
 * SD_DEBUG_BOUNDS: every index the matmul kernels (per call and inside the
 * one-launch pass) compute for a global access or a weight, activation or
 * partial-sum copy is checked against the extent the call's shapes imply; a
 * failed check records SD_EDEVICE with its site and skips the access.  The
 * release build compiles the checks away. */
#define SD_BUILD_DEBUG_BOUNDS 1
int32_t sd_build_flags(void);

/* Programmatic dependent launch on (1, default) or off (0) for later launches. */
void sd_set_pdl(int enable);

/* ---- test hooks (not part of the verify pass) ---- */

/* Per-block int32 dots [M][n_out][k_in/32] from repacked weights, with the
 * same device routine the matmul uses. */
sd_status sd_debug_block_dots(int qtype, const void *w, int64_t n_out, int64_t k_in, const int8_t *q, int32_t M,
                              int32_t *dots, sd_stream_t stream);
/* The matmul's SiLU*mul requantisation applied to given g, u fp32 [M][F]. */
sd_status sd_debug_silu_mul_requant(const float *g, const float *u, int32_t M, int64_t F, int8_t *q, float *scales,
                                    sd_stream_t stream);
/* The canonical exponential on n values. */
sd_status sd_debug_cexp(const float *x, int64_t n, float *y, sd_stream_t stream);
/* Philox4x32-10 words for counters (pos, 0, 0) .. (pos+n-1): out uint32 [n][4]. */
sd_status sd_debug_philox(uint64_t seed, int64_t pos, int64_t n, uint32_t *out, sd_stream_t stream);
/* One CTA waits on an mbarrier that nothing completes, bounded by `limit_ns`
 * nanoseconds of polling (1 .. 10^10); on expiry it records SD_ETIMEOUT in the
 * status word and returns.  Exercises the timeout path without hanging the
 * device: every wait inside the verify kernels is bounded the same way (2 s). */
sd_status sd_debug_wait_timeout(int64_t limit_ns, sd_stream_t stream);

/* The matmul's work partition, replayed on the host with the same code the
 * kernels walk: for each of the `sms` CTAs its pieces in order, as rows of 8
 * int32 {cta, split, unit, j0, j1, first owner, owners, last}; plus the plan
 * {KB, NU, KS, KBs, KBlast, G, P, D, R} in plan[9].  Returns the number of
 * pieces, -1 for a shape the matmul rejects, -2 when cap rows are too few.
 * No GPU is needed. */
int64_t sd_debug_schedule(int qtype, int64_t n_out, int64_t k_in, int32_t pair, int32_t head, int32_t sms,
                          int32_t *plan, int32_t *rows, int64_t cap);

#ifdef __cplusplus
}
#endif
#endif /* SDVERIFY_H */
