// sdv_qmatmul.cuh - multi-position quantised matmul (one weight read serves
// all M verify positions), with the requantising, SiLU*mul, residual and head
// epilogues, and the persistent verify pass built from the same pieces.
//
// Work decomposition: the weights of a matrix are 32-row tiles (or gate|up
// tile pairs; "units") x k-blocks.  The k range is cut into KS splits of at
// most 160 blocks so the activations of one split fit in shared memory.  Steps
// (one record of 32 rows x 32 weights, or a gate|up pair of records) are
// shared out over a grid of min(#SMs, steps) CTAs in equal parts:
//  * with one split and at least as many units as CTAs, each CTA takes D =
//    NU / G whole units, and the R = NU - D G units left over are shared
//    stream-K (each CTA a contiguous equal run of their unit-major steps); a
//    CTA works its shared run first and its whole units last;
//  * otherwise every step is shared stream-K in (split, unit, block) order.
// A unit-split whose steps fall in one CTA is finished directly; otherwise
// each CTA writes its partial sums to the workspace and the last one to
// arrive adds them in (split, piece) order.  All of this depends on (n_out,
// k_in, SM count) only, never on M, which makes every output row
// bit-identical whatever the number of positions.
//
// Inside a CTA three roles run concurrently:
//  * warp 8 (one elected lane) streams records with TMA bulk copies into a
//    ring of shared-memory stages guarded by mbarriers;
//  * warps 0..7 consume them.  Each record's exact int32 block dots come from
//    mma.sync m16n8k16 (f16 operands, f32 accumulate): the weight codes enter
//    as the fp16 values 1024 + code (4-bit, one LOP3 per two values; codes in
//    bits 4..7 of a byte enter as 1024 + 16 code against activations divided
//    by 16) or 1152 + q (Q8_0, one PRMT per two values), activations as exact
//    fp16 integers, and the accumulator starts at minus the offsets'
//    contribution, so it ends at the exact integer dot (every partial sum is
//    an integer below 2^23).  Each lane then adds d_w * d_a * dot for its 8
//    (row, position) results.  At the end of a piece each warp leaves its
//    partial sums in a shared-memory slot and moves on;
//  * warps 9..11 (the finishers, positions split between them) add the 8
//    warps' partials of a piece in warp order, then run the stream-K fixup
//    and the epilogue (residual, block sums of squares, requantisation into
//    the next matmul's activation fragments, head statistics) while the
//    consumers work on the next piece.
#pragma once

#include "sdv_common.cuh"
#include "sdv_sample.cuh"
#include "sdv_topk.cuh"

namespace sdv {

constexpr int NCW = 8;                       // consumer warps
constexpr int NF = 3;                        // finisher warps
constexpr int PRODUCER_WARP = NCW;           // streams the weights
constexpr int FIN_WARP0 = NCW + 1;           // first finisher warp: reductions, fixups, epilogues
constexpr int QMM_THREADS = (NCW + 1 + NF) * 32;
constexpr int CONS_THREADS = NCW * 32;         // named barrier BAR_CONS: consumers
constexpr int WORK_THREADS = (NCW + NF) * 32;  // named barrier BAR_WORK: consumers + finishers
constexpr int FIN_THREADS = NF * 32;           // named barrier BAR_FIN: finishers
constexpr int BAR_CONS = 1, BAR_WORK = 2, BAR_FIN = 3;

constexpr int KB_SPLIT_MAX = 160;      // blocks per k-split
constexpr int MPAD = 16;               // position stride of workspace partials
constexpr int MAX_NS = 10;             // ring stages (mbarrier header room)
constexpr uint64_t WAIT_NS = 2000000000ull;     // 2 s bound on any in-kernel wait
// Bound on any launch's loops (self-check), in SM clock cycles: 10 s at 2.2 GHz, longer at lower
// clocks.  Counted with the SM's cycle counter: reading the global timer costs far more, and
// the check runs once per piece.
constexpr long long KERNEL_CYCLES = 22000000000ll;
constexpr int STAT_TILE = 1024;        // vocabulary tile of the softmax statistics
constexpr int WS_UNIT_CNT = 32768;     // workspace counters: units (tiles / tile pairs) per call
constexpr int WS_STAT_CNT = 2048;      // workspace counters: 1024-token statistics tiles
constexpr size_t WS_CNT_BYTES = 160 * 1024;  // >= (WS_UNIT_CNT + WS_STAT_CNT + 1) * 4, 256-aligned
constexpr int NORM_MAX_KB = 2048;      // RMSNorm rows of at most 65536 elements
constexpr int PASS_NORM_MAX_KB = 1024; // ... inside the verify pass (one warp's 1024-slot tree)

// Shared-memory header: mbarriers at fixed offsets
constexpr uint32_t HDR_FULL = 0, HDR_EMPTY = 8 * MAX_NS, HDR_ACT = 16 * MAX_NS, HDR_AFREE = HDR_ACT + 8,
                   HDR_RFULL = HDR_AFREE + 8, HDR_REMPTY = HDR_RFULL + 16, HDR_FING = HDR_REMPTY + 16,
                   HDR_FINB = HDR_FING + 8, HDR_INV = HDR_FINB + 8, HDR_BYTES = 256;
static_assert(HDR_INV + 8 <= HDR_BYTES, "mbarrier header");

// ---------------------------------------------------------------------------
// Activation fragments ("AF"): a matmul's int8 input laid out for its inner
// loop, written by whoever produces the activations (the RMSNorm phase, the
// requantising epilogues) and copied into shared memory with one bulk copy.
// For K = 32 KB and M positions, NT = 1 (M <= 8) or 2:
//   frag: per block M*4 entries, entry (m, c) at index (jb*M + m)*4 + c holding
//     for position m the k values 2c, 2c+1 | 2c+8, 2c+9 | 16+2c, 17+2c |
//     24+2c, 25+2c: NT = 1 as four fp16 pairs (uint4; for a 4-bit consumer
//     the k+8 pairs divided by 16, exact), NT = 2 as eight raw bytes (uint2).
//   meta: per block 8 NT pairs {corr, d_a} (float2), zero beyond M, where corr
//     is minus the code offsets' contribution: 4-bit -(1032 S_lo + 72 S_hi)
//     with S_lo / S_hi the sums of the codes at k % 16 < 8 / >= 8, Q8_0
//     -1152 (S_lo + S_hi).
// ---------------------------------------------------------------------------
__host__ __device__ __forceinline__ int af_nt(int M) { return M <= 8 ? 1 : 2; }
__host__ __device__ __forceinline__ uint32_t af_frag_bytes(int M) { return af_nt(M) == 1 ? 64u * M : 32u * M; }
__host__ __device__ __forceinline__ uint32_t af_meta_bytes(int M) { return 64u * af_nt(M); }

// K-quant consumers (SD_Q4_K, SD_Q6_K) read a wider {c0, c1, d_a, S} per (block, position): Q4_K the
// offset correction of the raw code dot in c0 and the code sum S of the activations (for the minima);
// Q6_K the corrections of the block's two 16-weight halves in c0, c1.  128 NT bytes per block.
__host__ __device__ constexpr bool is_kq(int qt) { return qt == SD_Q4_K || qt == SD_Q6_K; }
__host__ __device__ __forceinline__ uint32_t af_meta_bytes_q(int M, int qt) {
    return (is_kq(qt) ? 128u : 64u) * af_nt(M);
}
// bytes of one 32-weight step of a matrix (a K-quant super-record holds eight)
__host__ __device__ constexpr int step_bytes_q(int qt) {
    return qt == SD_Q8_0 ? 1088 : (qt == SD_Q4_K ? 592 : (qt == SD_Q6_K ? 840 : 576));
}
constexpr int Q4K_SR = 4736, Q6K_SR = 6720;  // super-record bytes (32 rows x 256 weights)

struct QmmArgs {
    const uint8_t *w;
    int64_t n_out;       // output columns (2F for a gate|up pair)
    int32_t KB;          // k blocks
    int32_t NU;          // units: 32-row tiles, or gate|up tile pairs
    int32_t KS, KBs, KBlast;
    int64_t W;           // total steps
    int32_t G;           // CTAs
    int32_t P;           // max pieces per (unit, split)
    int32_t D, R;        // whole units per CTA and units shared stream-K (D = 0: all shared)
    int32_t defer;       // partial sums only: a KIND_COMBINE phase adds them and runs the epilogue
    int32_t defer_stats; // head: statistics formed by a KIND_HSTATS phase, folded by KIND_ACCEPT
    int32_t SB;          // steps per stage
    int32_t NS;          // stages
    uint32_t step_bytes; // bytes of one step
    const int8_t *q;     // int8 activations [M][K] + scales [M][KB] (staged directly when af_frag is null)
    const float *sc;
    const uint8_t *af_frag;  // activation fragments of the input (bulk-copied when non-null)
    const float *af_meta;
    int32_t M;
    float *y;
    const float *residual;
    float *ss;           // residual epilogue: per-32-block sums of squares of y [M][n_out/32] (nullable)
    uint32_t epi;
    int64_t col0;
    int8_t *q_next;
    float *s_next;
    int64_t nq;          // row width of q_next
    uint8_t *af_out_frag;  // requantising epilogues / RMSNorm: fragments of the next matmul (nullable)
    float *af_out_meta;
    int32_t af_out_qt;     // weight format of that matmul
    const float *norm_next;  // residual epilogue: weight of the next RMSNorm; its codes go to q_next / af_out
    int32_t af_norm;       // the input fragments hold RMSNorm codes: scales are max|x w| / 127, times inv here
    int32_t ss_ld;         // row stride of the block sums of squares (a multiple of 4)
    float *s_norm_out;     // scales inv * c of those codes [M][KB] (nullable)
    float *part;         // workspace partials [NU][KS][P][rows][MPAD]
    uint32_t *cnt;       // workspace counters [NU]
    // head statistics
    int head;
    float T;
    int32_t *argmax;
    float *row_max;
    float *row_sumexp;
    float4 *st_part;     // [n_stiles][MPAD]
    uint32_t *st_cnt;    // [n_stiles]
    uint32_t *st_done;   // [1]
    int32_t n_stiles;
    int *status;
    uint32_t off_ring, off_act, off_meta, off_red, off_ss;
    uint32_t stage_stride;  // bytes between ring slots (>= SB * step_bytes)
    int32_t NRB;            // partial-sum slots between consumers and finisher (1 or 2)
    int32_t rows_p;         // row stride of a slot (rows + 4: conflict-free stores)
    // phase kind inside a pass: KIND_MATMUL (qt, pair), KIND_NORM (RMSNorm + requant), KIND_ACCEPT
    // (statistics fold, then greedy or sampled acceptance), KIND_COMBINE, KIND_HSTATS
    int32_t kind, qt, pair;
    const float *xin;       // RMSNorm input [M][K] (K = 32 KB)
    const float *norm_w;    // RMSNorm weight [K]
    const float *ss_in;     // block sums of squares [M][ss_ld] of the normalised input (af_norm)
    float eps;
    const int32_t *tokens;  // acceptance inputs / outputs
    const int32_t *parent;
    int32_t *out_tokens;
    int32_t *out_count;
    int32_t accept_mode;    // acceptance: 0 greedy, 1 rejection sampling (chain)
    const float *q_probs;   // sampling: drafter probabilities [M-1][n_out] (null: certainty drafter)
    uint64_t seed;          // sampling: Philox key and first position
    int64_t base_pos;
    int32_t top_k;          // sampling: 0 unfiltered, else the top-k / top-p filtered target
    float top_p;
    int32_t ilv3;           // 0, or NU / 3: units taken in threes from the three thirds of the rows (see phys_unit)
    int32_t GR;             // schedule granule in blocks: every piece and split boundary is a multiple (8 for the
                            // 256-weight K-quant super-blocks, else 1)
    int32_t GRS;            // log2 GR (the schedule walk shifts instead of dividing: it runs at every phase start)
    int32_t af_build;       // single-operation calls: act_frag_kernel forms af_frag / af_meta from q / sc first
    // single-operation calls whose work a previous launch decides (read after griddepcontrol.wait):
    const uint32_t *unit_mask;  // bit per row tile: only set tiles are computed (null: all)
    const int *skip_if;         // non-zero: the call does nothing (null: always runs)
    // combine phases: pieces of each (unit, split), [NU][np_tab_stride(KS)] bytes from the host's replay of
    // the schedule (null: worked out here; the walk's divisions cost microseconds after a grid barrier)
    const uint8_t *np_tab;
};

// row stride of np_tab: whole 32-bit words, so up to four splits come in one load
__host__ __device__ __forceinline__ int np_tab_stride(int KS) { return (KS + 3) & ~3; }

constexpr int KIND_MATMUL = 0, KIND_NORM = 1, KIND_ACCEPT = 2, KIND_COMBINE = 3, KIND_HSTATS = 4;

// Optional per-phase trace of the one-launch pass: after the SM ids of the G CTAs, TR_SLOTS values per
// (phase, CTA).  Global-timer nanoseconds: the phase begins (grid barrier passed), the consumers hold
// their first activations, the consumers leave the phase, the phase ends (every role done), and the
// producer starts and finishes issuing the phase's weight copies.  SM cycles spent by consumer warp 0
// in the phase: waiting for weight stages, computing records, handing partial sums to the finishers
// (waiting for a free slot included), staging a split's activations (waiting for their copy, the
// RMSNorm row factors and their scales), the CTA's last tile epilogue, and the whole phase.
constexpr int TR_START = 0, TR_ACT = 1, TR_CONS_END = 2, TR_END = 3, TR_PROD_FIRST = 4, TR_PROD_LAST = 5,
              TR_CYC_WAIT = 6, TR_CYC_COMP = 7, TR_CYC_HAND = 8, TR_CYC_STAGE = 9, TR_CYC_LAST = 10,
              TR_CYC_ALL = 11, TR_SLOTS = 12;

// fetch-and-add with release (orders the writes seen through a barrier) and acquire
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Row tile (32 rows, or a gate|up tile pair) of schedule unit u.  The identity, except for a matmul whose
// requantising epilogue covers the last third of its rows only (the V columns of a fused QKV
// projection): there units are taken in threes, one tile from each third, the requantised one first,
// so every CTA finishes an equal share of requantised tiles and its last unit has no epilogue work.
__host__ __device__ __forceinline__ int phys_unit(const QmmArgs &a, int u) {
    if (!a.ilv3) return u;
    const int r = u % 3, q = u / 3;
    return (r == 0 ? 2 : r - 1) * a.ilv3 + q;
}

// n / d for n >= 0 and d > 0, as a 32-bit division whenever both fit in 32 bits (every schedule
// quantity of a layer-sized matmul does): a 64-bit division is a long instruction sequence on the GPU,
// and the schedule walks sit on the path from a grid barrier to a phase's first copy
__host__ __device__ __forceinline__ int64_t udiv(int64_t n, int64_t d) {
    return ((static_cast<uint64_t>(n) | static_cast<uint64_t>(d)) >> 32) == 0
               ? static_cast<int64_t>(static_cast<uint32_t>(n) / static_cast<uint32_t>(d))
               : n / d;
}

__host__ __device__ __forceinline__ void decode_step(const QmmArgs &a, int64_t g, int &s, int &u, int &j, int &len) {
    int64_t per = static_cast<int64_t>(a.NU) * a.KBs;
    int64_t ss = udiv(g, per);
    if (ss > a.KS - 1) ss = a.KS - 1;
    s = static_cast<int>(ss);
    int64_t rem = g - per * ss;
    len = (s == a.KS - 1) ? a.KBlast : a.KBs;
    u = static_cast<int>(udiv(rem, len));
    j = static_cast<int>(rem - static_cast<int64_t>(u) * len);
}

__host__ __device__ __forceinline__ int64_t unit_start(const QmmArgs &a, int s, int u) {
    int len = (s == a.KS - 1) ? a.KBlast : a.KBs;
    return static_cast<int64_t>(a.NU) * a.KBs * s + static_cast<int64_t>(u) * len;
}

// length of the shared stream-K step sequence
__host__ __device__ __forceinline__ int64_t seq_len(const QmmArgs &a) { return a.D > 0 ? static_cast<int64_t>(a.R) * a.KB : a.W; }

// CTA owning step x of the shared sequence: the CTAs' runs start at floor(c wq / G) granules (wq =
// wseq / GR granules in all), so the owner is the largest c with floor(c wq / G) <= floor(x / GR)
__host__ __device__ __forceinline__ int seq_owner(const QmmArgs &a, int64_t wseq, int64_t x) {
    const int64_t wq = wseq >> a.GRS;
    return wq > 0 ? static_cast<int>(udiv(((x >> a.GRS) + 1) * a.G - 1, wq)) : 0;
}

// CTAs sharing split s of unit u, and the first of them
__host__ __device__ __forceinline__ void unit_split_owners(const QmmArgs &a, int s, int u, int &first, int &np) {
    const int64_t wseq = seq_len(a);
    int64_t st;
    int len;
    if (a.D > 0) {
        st = static_cast<int64_t>(u) * a.KB;
        len = a.KB;
    } else {
        st = unit_start(a, s, u);
        len = (s == a.KS - 1) ? a.KBlast : a.KBs;
    }
    first = seq_owner(a, wseq, st);
    np = seq_owner(a, wseq, st + len - 1) - first + 1;
}

// One piece of a CTA's work: blocks [j0, j1) of split s of unit u, shared by np CTAs from `first` on.
struct Piece {
    int s, u, j0, j1, first, np;
};

struct PieceIter {
    int64_t g, hi;      // cursor in the shared step sequence
    int d_next, d_end;  // whole units still to take
    int cta;            // the CTA walking this schedule
    int mw;             // restricted calls: index of the unit-mask word in mbits (-1: none loaded)
    uint32_t mbits;
};

// The schedule of CTA `cta` (host and device: the host replays it to check the partition).
__host__ __device__ __forceinline__ void pieces_begin_cta(const QmmArgs &a, PieceIter &it, int cta) {
    const int64_t c = cta, wq = seq_len(a) >> a.GRS;
    it.cta = cta;
    it.mw = -1;
    it.mbits = 0;
    if (cta >= a.G) {  // a matmul with fewer granules of work than the grid has CTAs: none for this one
        it.g = it.hi = 0;
        it.d_next = it.d_end = 0;
        return;
    }
    it.g = udiv(c * wq, a.G) << a.GRS;
    it.hi = udiv((c + 1) * wq, a.G) << a.GRS;
    it.d_next = a.D > 0 ? a.R + static_cast<int>(c) * a.D : 0;
    it.d_end = a.D > 0 ? it.d_next + a.D : 0;
}

__device__ __forceinline__ void pieces_begin(const QmmArgs &a, PieceIter &it) {
    pieces_begin_cta(a, it, static_cast<int>(blockIdx.x));
}

// Unit u is computed in this call (a call restricted to a set of row tiles reads them from unit_mask;
// the walk's units mostly increase, so one mask word is loaded per 32 units, not one per piece).
__device__ __forceinline__ bool unit_on(const QmmArgs &a, int u, PieceIter &it) {
    if (!a.unit_mask) return true;
    const int pu = phys_unit(a, u);
    if ((pu >> 5) != it.mw) {
        it.mw = pu >> 5;
        it.mbits = __ldcg(a.unit_mask + it.mw);
    }
    return ((it.mbits >> (pu & 31)) & 1u) != 0u;
}

// The next piece in processing order (shared run first, whole units last); false when done.
__host__ __device__ __forceinline__ bool pieces_next(const QmmArgs &a, PieceIter &it, Piece &p) {
    if (it.g < it.hi) {
        int len;
        if (a.D > 0) {
            p.s = 0;
            len = a.KB;
            p.u = static_cast<int>(udiv(it.g, a.KB));
            p.j0 = static_cast<int>(it.g - static_cast<int64_t>(p.u) * a.KB);
        } else {
            decode_step(a, it.g, p.s, p.u, p.j0, len);
        }
        p.j1 = static_cast<int>(p.j0 + (it.hi - it.g) < len ? p.j0 + (it.hi - it.g) : len);
        it.g += p.j1 - p.j0;
        unit_split_owners(a, p.s, p.u, p.first, p.np);
        return true;
    }
    if (it.d_next < it.d_end) {
        p.s = 0;
        p.u = it.d_next++;
        p.j0 = 0;
        p.j1 = a.KB;
        p.first = it.cta;
        p.np = 1;
        return true;
    }
    return false;
}

// The next piece of a unit this call computes.
__device__ __forceinline__ bool pieces_next_on(const QmmArgs &a, PieceIter &it, Piece &p) {
    while (pieces_next(a, it, p))
        if (unit_on(a, p.u, it)) return true;
    return false;
}

// Whether this CTA has any piece in this phase (past the grid's CTAs, or every piece of a restricted
// call in units it leaves out: none; the roles then sit the phase out).
__device__ inline bool cta_has_work(const QmmArgs &a) {
    if (static_cast<int>(blockIdx.x) >= a.G) return false;
    if (!a.unit_mask) return true;
    PieceIter it;
    pieces_begin(a, it);
    Piece p;
    return pieces_next_on(a, it, p);
}

// ---------------------------------------------------------------------------
// record layout and exact block dots on the tensor cores
//
// Lane l = 4g + c of a warp owns, for a 32-row x 32-weight record, the A
// fragments of mma m16n8k16 for row tiles t = 0, 1 (rows 16t + g, 16t + g + 8)
// and k steps s = 0, 1 (k = 16s + 2c, +1 and 16s + 2c + 8, +9).
//  4-bit: 16 code bytes per lane, word j = 2t + s; nibble i of the word holds
//    i=0,4: (row 16t+g,   k 16s+2c, +1)   i=2,6: (row 16t+g+8, k 16s+2c, +1)
//    i=1,5: (row 16t+g,   k 16s+2c+8, +9) i=3,7: (row 16t+g+8, k 16s+2c+8, +9)
//  Q8_0: 32 code bytes per lane in two 16-byte planes (words 0..3 for t = 0,
//    words 4..7 for t = 1); word 2(2t+s)+h holds bytes (row 16t+g, k0), (row
//    16t+g, k0+1), (row 16t+g+8, k0), (row 16t+g+8, k0+1) with k0 = 16s+2c+8h.
//  Scales: 8 groups of 4 fp16, group g = rows g, g+8, 16+g, 24+g.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mma_init(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, float c0,
                                         float c1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%10,%11};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ void mma_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (x & MASK) | magic as one three-input logic operation (lookup table 0xEA = (a & b) | c), the
// mask as an immediate and the exponent bits in a register: the compiler left to itself splits
// it in two, and this unpack is the integer pipe's largest load in the consumer loop
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "n"(MASK), "r"(magic));
    return r;
}

// 4-bit codes of one lane -> fp16 pairs (1024 + code, or 1024 + 16 code in the k+8 halves)
__device__ __forceinline__ void q4_frag(uint4 w, uint32_t (&a)[2][2][4]) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    const uint32_t magic = 0x64006400u;  // fp16 exponent of 1024 in both halves
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t x = ws[j], y = x >> 8;
        a[j >> 1][j & 1][0] = and_or<0x000F000Fu>(x, magic);
        a[j >> 1][j & 1][1] = and_or<0x000F000Fu>(y, magic);
        a[j >> 1][j & 1][2] = and_or<0x00F000F0u>(x, magic);
        a[j >> 1][j & 1][3] = and_or<0x00F000F0u>(y, magic);
    }
}

// Q8_0 codes of one lane -> fp16 pairs 1152 + q (offset binary in the mantissa)
__device__ __forceinline__ void q8_frag(uint4 p0, uint4 p1, uint32_t (&a)[2][2][4]) {
    const uint32_t ws[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint32_t x = ws[w] ^ 0x80808080u;
        const int ts = w >> 1, h = w & 1;
        a[ts >> 1][ts & 1][2 * h] = __byte_perm(x, 0x64646464u, 0x5140);
        a[ts >> 1][ts & 1][2 * h + 1] = __byte_perm(x, 0x64646464u, 0x7362);
    }
}

// t | (h & MASK) as one three-input logic operation (lookup table 0xF8 = a | (b & c)), the mask as an immediate
template <uint32_t MASK>
__device__ __forceinline__ uint32_t or_masked(uint32_t t, uint32_t h) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xF8;" : "=r"(r) : "r"(t), "n"(MASK), "r"(h));
    return r;
}

// Q6_K codes of one lane -> fp16 pairs 1024 + code (code = low nibble | two high bits << 4, 0..63), or
// 1024 + 16 code in the k+8 halves: the low nibbles are placed as the 4-bit format's, and high-bit word
// h holds the high bits of code words 2h (at 4..11, 20..27) and 2h+1 (at 0..3, 12..19, 28..31) where
// one shift brings each register's pair under the masks 0x00300030 / 0x03000300.
__device__ __forceinline__ void q6_frag(uint4 lo, uint2 hi, uint32_t (&a)[2][2][4]) {
    const uint32_t ws[4] = {lo.x, lo.y, lo.z, lo.w};
    const uint32_t magic = 0x64006400u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t x = ws[j], y = x >> 8, H = (j >> 1) ? hi.y : hi.x;
        const uint32_t ha0 = (j & 1) ? H << 4 : H, ha1 = (j & 1) ? H >> 8 : H >> 2;
        const uint32_t hb0 = (j & 1) ? H << 6 : H, hb1 = (j & 1) ? H >> 6 : H >> 2;
        a[j >> 1][j & 1][0] = or_masked<0x00300030u>(and_or<0x000F000Fu>(x, magic), ha0);
        a[j >> 1][j & 1][1] = or_masked<0x00300030u>(and_or<0x000F000Fu>(y, magic), ha1);
        a[j >> 1][j & 1][2] = or_masked<0x03000300u>(and_or<0x00F000F0u>(x, magic), hb0);
        a[j >> 1][j & 1][3] = or_masked<0x03000300u>(and_or<0x00F000F0u>(y, magic), hb1);
    }
}

// unsigned byte e of x as an exact float (the byte in the mantissa of 2^23)
// 2^23 + byte e of x, exactly (the byte as the low mantissa bits of 2^23)
__device__ __forceinline__ float ubyte_magic(uint32_t x, int e) {
    return __int_as_float(static_cast<int>(__byte_perm(x, 0x4B000000u, 0x7440u | static_cast<uint32_t>(e))));
}
__device__ __forceinline__ float ubyte_f(uint32_t x, int e) { return ubyte_magic(x, e) - 8388608.0f; }

// the two row tiles' exact dots of one record against one 8-position tile:
// d[t][i] = dot(row 16t + g + 8(i>>1), position 2c + (i&1))
__device__ __forceinline__ void record_dots(const uint32_t (&a)[2][2][4], uint4 bf, float2 corr, float (&d)[2][4]) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        mma_init(d[t], a[t][0], bf.x, bf.y, corr.x, corr.y);
        mma_acc(d[t], a[t][1], bf.z, bf.w);
    }
}

// Raw int8 B operand of one lane for one block and 8-position tile: the bytes at
// k = 2c, 2c+1, 2c+8, 2c+9, 16+2c, 17+2c, 24+2c, 25+2c of position g's 32
// activations, as two 32-bit words (pairs in k order).  `arow` nullptr: padding.
__device__ __forceinline__ uint2 b_raw(const int8_t *arow, int c) {
    if (!arow) return make_uint2(0u, 0u);
    const unsigned *w = reinterpret_cast<const unsigned *>(arow);
    const int sh = 16 * (c & 1), j = c >> 1;
    const uint32_t p0 = (__ldcg(w + j) >> sh) & 0xFFFFu, p1 = (__ldcg(w + 2 + j) >> sh) & 0xFFFFu;
    const uint32_t p2 = (__ldcg(w + 4 + j) >> sh) & 0xFFFFu, p3 = (__ldcg(w + 6 + j) >> sh) & 0xFFFFu;
    return make_uint2(p0 | (p1 << 16), p2 | (p3 << 16));
}

// int8 pair (low 16 bits of x, k order) -> exact fp16 pair; `div16` also scales by 1/16 (exact)
__device__ __forceinline__ uint32_t i8pair_to_h2(uint32_t x, bool div16) {
    const uint32_t u = __byte_perm(x ^ 0x8080u, 0x64646464u, 0x5140);  // (1024 + a + 128) per half
    __half2 h = *reinterpret_cast<const __half2 *>(&u);
    if (div16) h = __hfma2(h, __float2half2_rn(0.0625f), __float2half2_rn(-72.0f));  // (1152 + a)/16 - 72 = a/16
    else h = __hsub2(h, __float2half2_rn(1152.0f));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// fp16 B fragment registers from the raw operand: {s0 k 2c.., s0 k 2c+8.., s1 k 2c.., s1 k 2c+8..};
// the k+8 halves divided by 16 for the 4-bit format
template <int QT>
__device__ __forceinline__ uint4 b_frag_from_raw(uint2 r) {
    const bool d = QT != SD_Q8_0;  // the 4-bit and K-quant formats take the k+8 halves as sixteenths
    return make_uint4(i8pair_to_h2(r.x, false), i8pair_to_h2(r.x >> 16, d), i8pair_to_h2(r.y, false),
                      i8pair_to_h2(r.y >> 16, d));
}

// accumulator start removing the code offsets: 4-bit -(1032 S_lo + 72 S_hi)
// with S_lo / S_hi the sums of the activations at k % 16 < 8 / >= 8; Q8_0
// -1152 S.  Exact integers (|.| < 2^23).
template <int QT>
__device__ __forceinline__ float dot_corr(const int8_t *arow) {
    if (!arow) return 0.0f;
    const uint4 *p = reinterpret_cast<const uint4 *>(arow);
    const uint4 x0 = __ldcg(p), x1 = __ldcg(p + 1);
    int lo = 0, hi = 0;
    lo = dp4a(0x01010101, static_cast<int>(x0.x), lo);
    lo = dp4a(0x01010101, static_cast<int>(x0.y), lo);
    hi = dp4a(0x01010101, static_cast<int>(x0.z), hi);
    hi = dp4a(0x01010101, static_cast<int>(x0.w), hi);
    lo = dp4a(0x01010101, static_cast<int>(x1.x), lo);
    lo = dp4a(0x01010101, static_cast<int>(x1.y), lo);
    hi = dp4a(0x01010101, static_cast<int>(x1.z), hi);
    hi = dp4a(0x01010101, static_cast<int>(x1.w), hi);
    const int v = QT == SD_Q4_32 ? -(1032 * lo + 72 * hi) : -1152 * (lo + hi);
    return static_cast<float>(v);
}

// {c0, c1, d_a, S} of a K-quant consumer from the activation code sums of the block's quarters (k 0-7,
// 8-15, 16-23, 24-31; the fragments carry the 8-15 and 24-31 codes as sixteenths).  Q4_K: c0 removes the
// fp16 offsets 1024 and 64 so the dot is sum code * a; S = sum a.  Q6_K: per 16-weight half, c removes
// the offsets and the code bias 32 (1056 = 1024 + 32, 96 = 64 + 32).  Exact integers below 2^24.
template <int QT>
__device__ __forceinline__ float4 kq_meta(const int (&s4)[4], float da) {
    if (QT == SD_Q4_K)
        return make_float4(static_cast<float>(-(1024 * (s4[0] + s4[2]) + 64 * (s4[1] + s4[3]))), 0.0f, da,
                           static_cast<float>(s4[0] + s4[1] + s4[2] + s4[3]));
    return make_float4(static_cast<float>(-(1056 * s4[0] + 96 * s4[1])), static_cast<float>(-(1056 * s4[2] + 96 * s4[3])),
                       da, 0.0f);
}

// ---------------------------------------------------------------------------
// activation fragments: writer
// ---------------------------------------------------------------------------

// two int8 values (or their sixteenths, exact) as an fp16 pair, the first in the low half
__device__ __forceinline__ uint32_t pack_h2(int x0, int x1, float s) {
    __half2 h = __floats2half2_rn(static_cast<float>(x0) * s, static_cast<float>(x1) * s);
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_b4(int x0, int x1, int x2, int x3) {
    return (static_cast<uint32_t>(x0) & 0xFFu) | ((static_cast<uint32_t>(x1) & 0xFFu) << 8) |
           ((static_cast<uint32_t>(x2) & 0xFFu) << 16) | ((static_cast<uint32_t>(x3) & 0xFFu) << 24);
}

// Writes position m of block jb of an activation-fragment buffer (layout above) from one full
// warp whose lane k holds the block's code v and whose scale is d.  qt: weight format of the
// matmul that reads it.  Lanes 0..3 write the fragment entries, lane 0 the {corr, d} pair; the
// writer of the last position also zeroes the pairs of the padding positions M .. 8 NT - 1.
template <bool KQ = false>
__device__ __forceinline__ void af_write(uint8_t *frag, float *meta, int M, int64_t jb, int m, int lane, int v,
                                         float d, int qt) {
    // S_lo + 65536 S_hi in one reduction; |S_lo| <= 16 * 127 < 32768 recovers both exactly
    const int lo = (lane & 8) ? 0 : v;  // k % 16 < 8
    int t = lo + (v - lo) * 65536;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    const int s_hi = (t + 32768) >> 16, s_lo = t - s_hi * 65536;
    const float corr = static_cast<float>(qt == SD_Q4_32 ? -(1032 * s_lo + 72 * s_hi) : -1152 * (s_lo + s_hi));
    const int c = lane & 3, k0 = 2 * c;
    const int e0 = __shfl_sync(0xffffffffu, v, k0), e1 = __shfl_sync(0xffffffffu, v, k0 + 1);
    const int e2 = __shfl_sync(0xffffffffu, v, k0 + 8), e3 = __shfl_sync(0xffffffffu, v, k0 + 9);
    const int e4 = __shfl_sync(0xffffffffu, v, k0 + 16), e5 = __shfl_sync(0xffffffffu, v, k0 + 17);
    const int e6 = __shfl_sync(0xffffffffu, v, k0 + 24), e7 = __shfl_sync(0xffffffffu, v, k0 + 25);
    const int NT = af_nt(M);
    if (lane < 4) {
        const int64_t idx = (jb * M + m) * 4 + c;
        if (NT == 1) {
            const float hs = qt != SD_Q8_0 ? 0.0625f : 1.0f;  // 4-bit and K-quant consumers: k+8 halves / 16
            reinterpret_cast<uint4 *>(frag)[idx] =
                make_uint4(pack_h2(e0, e1, 1.0f), pack_h2(e2, e3, hs), pack_h2(e4, e5, 1.0f), pack_h2(e6, e7, hs));
        } else {
            reinterpret_cast<uint2 *>(frag)[idx] = make_uint2(pack_b4(e0, e1, e2, e3), pack_b4(e4, e5, e6, e7));
        }
    }
    if (KQ && is_kq(qt)) {  // {c0, c1, d, S} from the code sums of the block's four 8-weight quarters
        int x = v;
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        x += __shfl_xor_sync(0xffffffffu, x, 4);
        const int s4[4] = {__shfl_sync(0xffffffffu, x, 0), __shfl_sync(0xffffffffu, x, 8),
                           __shfl_sync(0xffffffffu, x, 16), __shfl_sync(0xffffffffu, x, 24)};
        if (lane == 0) {
            float4 *mp = reinterpret_cast<float4 *>(meta) + jb * 8 * NT;
            mp[m] = qt == SD_Q4_K ? kq_meta<SD_Q4_K>(s4, d) : kq_meta<SD_Q6_K>(s4, d);
            if (m == M - 1)
                for (int p = M; p < 8 * NT; ++p) mp[p] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        return;
    }
    if (lane == 0) {
        float2 *mp = reinterpret_cast<float2 *>(meta) + jb * 8 * NT;
        mp[m] = make_float2(corr, d);
        if (m == M - 1)
            for (int p = M; p < 8 * NT; ++p) mp[p] = make_float2(0.0f, 0.0f);
    }
}

// pairwise tree over the 32 lanes (strides 16, 8, 4, 2, 1); lane 0 holds the sum
__device__ __forceinline__ float tree32(float x, int lane) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const float o = __shfl_down_sync(0xffffffffu, x, s);
        if (lane < s) x = __fadd_rn(x, o);
    }
    return x;
}

// ---------------------------------------------------------------------------
// epilogue of one finished (unit, position), run by the finisher warp: lane = row
// ---------------------------------------------------------------------------
template <int PAIR, bool KQ = false>
__device__ __forceinline__ void epilogue(const QmmArgs &a, int u, int m, int lane, float v, float vu, float res, float nw) {
    // site 106: a position of the call and a row tile of the output
    if (!SD_INB(m >= 0 && m < a.M && u >= 0 && static_cast<int64_t>(u) * 32 < (PAIR ? a.n_out / 2 : a.n_out), a.status,
                106))
        return;
    if (PAIR) {
        const int64_t F = a.n_out / 2;
        const int64_t n = static_cast<int64_t>(u) * 32 + lane;  // F % 32 == 0 is required
        if (a.y) {
            a.y[m * a.n_out + n] = v;
            a.y[m * a.n_out + F + n] = vu;
        }
        const float h = silu_mul(v, vu);
        float d;
        const int code = requant_lane(h, d);
        a.q_next[m * a.nq + n] = static_cast<int8_t>(code);
        if (lane == 0) a.s_next[m * (a.nq / 32) + u] = d;
        if (a.af_out_frag) af_write<KQ>(a.af_out_frag, a.af_out_meta, a.M, u, m, lane, code, d, a.af_out_qt);
    } else {
        const int64_t n = static_cast<int64_t>(u) * 32 + lane;
        const bool ok = n < a.n_out;
        if (ok && a.residual) v = __fadd_rn(v, res);
        if (ok && a.y) a.y[m * a.n_out + n] = v;
        if (a.ss) {  // n_out % 32 == 0 is required here
            const float s = tree32(__fmul_rn(v, v), lane);
            if (lane == 0) a.ss[m * a.ss_ld + u] = s;
        }
        if (a.norm_next) {  // codes of the next RMSNorm from t = v w; its scale waits for inv
            float c;
            const int code = requant_lane(__fmul_rn(v, nw), c);
            a.q_next[m * a.nq + n] = static_cast<int8_t>(code);
            af_write<KQ>(a.af_out_frag, a.af_out_meta, a.M, u, m, lane, code, c, a.af_out_qt);
        }
        if (a.epi == SD_EPI_REQUANT && static_cast<int64_t>(u) * 32 >= a.col0) {
            float d;
            const int code = requant_lane(ok ? v : 0.0f, d);  // n_out % 32 == 0 is required here
            const int64_t c = n - a.col0;
            if (ok) a.q_next[m * a.nq + c] = static_cast<int8_t>(code);
            if (lane == 0) a.s_next[m * (a.nq / 32) + c / 32] = d;
            if (a.af_out_frag)
                af_write<KQ>(a.af_out_frag, a.af_out_meta, a.M, (static_cast<int64_t>(u) * 32 - a.col0) / 32, m, lane, code,
                         d, a.af_out_qt);
        }
    }
}

// ---------------------------------------------------------------------------
// head statistics.  Per operation: the finisher warps (warp f takes positions f, f + NF, ...) of
// the CTA that finishes a 1024-token tile's last 32-row tile form its statistics; the CTA that
// finishes the last statistics tile folds them per row.  In the pass: a statistics phase after
// the logits are complete, (tile, position) items spread over every work warp of the grid, and
// the fold at the start of the acceptance phase.
// ---------------------------------------------------------------------------

// Statistics of tile st for position m (one warp): max of z = l / T, the pairwise-tree sum of
// exp(z - max) and the raw-logit argmax (lowest index on ties).
__device__ inline void head_tile_stats_one(const QmmArgs &a, int st, int m, int lane) {
    const int64_t V = a.n_out;
    const bool unit_t = a.T == 1.0f;  // l / 1 is l exactly
    float v[32];
    float zmax = -__int_as_float(0x7f800000);
    float bl = -__int_as_float(0x7f800000);
    int bi = 0x7fffffff;
    // every load in flight before the first compare; -inf past the vocabulary changes nothing below
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const int64_t e = static_cast<int64_t>(st) * STAT_TILE + lane + 32 * r;
        v[r] = e < V ? __ldcg(a.y + m * V + e) : -__int_as_float(0x7f800000);
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const float l = v[r];
        if (l > bl) {
            bl = l;
            bi = static_cast<int>(static_cast<int64_t>(st) * STAT_TILE + lane + 32 * r);
        }
        const float z = unit_t ? l : __fdiv_rn(l, a.T);
        zmax = fmaxf(zmax, z);
        v[r] = z;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        zmax = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, o));
        const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ol > bl || (ol == bl && oi < bi)) {
            bl = ol;
            bi = oi;
        }
    }
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const int64_t e = static_cast<int64_t>(st) * STAT_TILE + lane + 32 * r;
        v[r] = e < V ? cexpf_canon(__fsub_rn(v[r], zmax)) : 0.0f;
    }
    const float s = tree1024_warp(v);
    // site 107: a statistics tile of the vocabulary and a position of the call
    if (lane == 0 && SD_INB(st >= 0 && st < a.n_stiles && m >= 0 && m < a.M, a.status, 107))
        a.st_part[st * MPAD + m] = make_float4(zmax, s, __int_as_float(bi), bl);
}

__device__ inline void head_tile_stats(const QmmArgs &a, int st, int lane, int f) {
    for (int m = f; m < a.M; m += NF) head_tile_stats_one(a, st, m, lane);
}

// Fold of position m's tile statistics (one warp): argmax, row max and Z = the sequential fold
// over tiles of s_t exp(m_t - max), the products formed in parallel.
__device__ inline void head_final_fold_one(const QmmArgs &a, int m, int lane) {
    float mx = -__int_as_float(0x7f800000);
    float bl = -__int_as_float(0x7f800000);
    int bi = 0x7fffffff;
    if (a.n_stiles <= 256) {  // every tile's statistics in registers at once: one round of loads
        float4 p[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int t = lane + 32 * k;
            p[k] = t < a.n_stiles ? __ldcg(a.st_part + t * MPAD + m)
                                  : make_float4(-__int_as_float(0x7f800000), 0.0f, __int_as_float(0x7fffffff),
                                                -__int_as_float(0x7f800000));
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            mx = fmaxf(mx, p[k].x);
            const int pi = __float_as_int(p[k].z);
            if (p[k].w > bl || (p[k].w == bl && pi < bi)) {
                bl = p[k].w;
                bi = pi;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ol > bl || (ol == bl && oi < bi)) {
                bl = ol;
                bi = oi;
            }
        }
        float Z = 0.0f;  // sequential over tiles, as below
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int t0 = 32 * k;
            if (t0 < a.n_stiles) {
                const float e = t0 + lane < a.n_stiles ? __fmul_rn(p[k].y, cexpf_canon(__fsub_rn(p[k].x, mx))) : 0.0f;
                const int nn = a.n_stiles - t0 < 32 ? a.n_stiles - t0 : 32;
                for (int j = 0; j < nn; ++j) Z = __fadd_rn(Z, __shfl_sync(0xffffffffu, e, j));
            }
        }
        if (lane == 0) {
            a.argmax[m] = bi;
            a.row_max[m] = mx;
            a.row_sumexp[m] = Z;
        }
        return;
    }
    for (int t = lane; t < a.n_stiles; t += 32) {
        const float4 p = __ldcg(a.st_part + t * MPAD + m);
        mx = fmaxf(mx, p.x);
        const int pi = __float_as_int(p.z);
        if (p.w > bl || (p.w == bl && pi < bi)) {
            bl = p.w;
            bi = pi;
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float ol = __shfl_xor_sync(0xffffffffu, bl, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ol > bl || (ol == bl && oi < bi)) {
            bl = ol;
            bi = oi;
        }
    }
    float Z = 0.0f;
    for (int t0 = 0; t0 < a.n_stiles; t0 += 32) {
        const int t = t0 + lane;
        float e = 0.0f;
        if (t < a.n_stiles) {
            const float4 p = __ldcg(a.st_part + t * MPAD + m);
            e = __fmul_rn(p.y, cexpf_canon(__fsub_rn(p.x, mx)));
        }
        const int nn = a.n_stiles - t0 < 32 ? a.n_stiles - t0 : 32;
        for (int j = 0; j < nn; ++j) Z = __fadd_rn(Z, __shfl_sync(0xffffffffu, e, j));
    }
    if (lane == 0) {
        a.argmax[m] = bi;
        a.row_max[m] = mx;
        a.row_sumexp[m] = Z;
    }
}

__device__ inline void head_final_fold(const QmmArgs &a, int lane, int f) {
    for (int m = f; m < a.M; m += NF) head_final_fold_one(a, m, lane);
}

// ---------------------------------------------------------------------------
// per-CTA state and shared-memory regions
// ---------------------------------------------------------------------------

// One piece of a CTA's schedule as the producer publishes it (see produce_phase).
struct QPiece {
    int32_t s, u, j0, j1;
    int32_t first, np;   // CTAs sharing this unit-split, from `first` on
    int32_t expected;    // partial sums the unit waits for (all its splits)
    int32_t last;        // the CTA's last piece of this phase
};
constexpr int PQ_N = 32;  // queue slots: more than the pieces between producer and finishers (NS + NRB + 2)

struct CtaShared {
    volatile int abort;    // set by anyone whose bounded wait ran out; polled by every wait
    int fin_flag;          // finishers: warp 0's decision, published to the other finisher warps
    float inv[16];         // RMSNorm row factors of the current normalised staging
    long long t0;          // launch start (SM cycle counter), for the launch-wide time bound
    QPiece pq[PQ_N];       // the schedule, piece k in slot k % PQ_N
};

// Launch-wide self-check: past KERNEL_CYCLES since the CTA started, record SD_ETIMEOUT and where
// (status[1]: 1 producer, 2 consumer).
__device__ __forceinline__ bool out_of_time(const CtaShared &cs, int *status, int where) {
    if (clock64() - cs.t0 <= KERNEL_CYCLES) return false;
    if (status && atomicCAS(status, 0, SD_ETIMEOUT) == 0) status[1] = where;
    return true;
}

struct Smem {
    uint64_t *full, *empty;    // ring stages
    uint64_t *act_bar;         // the split's activations have landed
    uint64_t *act_free;        // every consumer warp is done with the previous split's activations
    uint64_t *rfull, *rempty;  // partial-sum slots between consumers and finishers
    uint64_t *fin_g, *fin_b;   // finisher rendezvous: gather at warp 0, broadcast back
    uint64_t *inv_bar;         // the RMSNorm row factors of a staging are in CtaShared::inv
    uint8_t *ring;
    uint8_t *act;   // the split's activation fragments
    float *meta;    // the split's {corr, d_a} pairs
    float *red;     // partial-sum slots [NRB][warp][position][rows_p]
    float *ss;      // block sums of squares of a normalised input [M][ss_ld]
};

__device__ __forceinline__ Smem smem_regions(uint8_t *smem, const QmmArgs &a) {
    Smem r;
    r.full = reinterpret_cast<uint64_t *>(smem + HDR_FULL);
    r.empty = reinterpret_cast<uint64_t *>(smem + HDR_EMPTY);
    r.act_bar = reinterpret_cast<uint64_t *>(smem + HDR_ACT);
    r.act_free = reinterpret_cast<uint64_t *>(smem + HDR_AFREE);
    r.rfull = reinterpret_cast<uint64_t *>(smem + HDR_RFULL);
    r.rempty = reinterpret_cast<uint64_t *>(smem + HDR_REMPTY);
    r.fin_g = reinterpret_cast<uint64_t *>(smem + HDR_FING);
    r.fin_b = reinterpret_cast<uint64_t *>(smem + HDR_FINB);
    r.inv_bar = reinterpret_cast<uint64_t *>(smem + HDR_INV);
    r.ring = smem + a.off_ring;
    r.act = smem + a.off_act;
    r.meta = reinterpret_cast<float *>(smem + a.off_meta);
    r.red = reinterpret_cast<float *>(smem + a.off_red);
    r.ss = reinterpret_cast<float *>(smem + a.off_ss);
    return r;
}

// act_arrivals: 1 when activations arrive by bulk copy (plus its bytes), else every consumer thread
__device__ __forceinline__ void cta_init(const Smem &sm, int NS, CtaShared &cs, uint32_t act_arrivals) {
    for (int i = 0; i < NS; ++i) {
        mbar_init(&sm.full[i], 1);
        mbar_init(&sm.empty[i], NCW);
    }
    mbar_init(sm.act_bar, act_arrivals);
    mbar_init(sm.act_free, NCW);
    for (int i = 0; i < 2; ++i) {
        mbar_init(&sm.rfull[i], NCW);
        mbar_init(&sm.rempty[i], NF);
    }
    mbar_init(sm.fin_g, NF);
    mbar_init(sm.fin_b, 1);
    mbar_init(sm.inv_bar, NCW);
    cs.abort = 0;
    cs.t0 = clock64();
    fence_barrier_init();
}

// bounded wait by a whole warp: true when every lane saw the phase complete; on failure the
// status records the timeout and every wait in the CTA gives up from then on
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, CtaShared &cs, int *status) {
    const bool ready = mbar_wait_bounded(bar, parity, WAIT_NS, &cs.abort);
    __syncwarp();  // lanes leave the wait one by one; warp-wide instructions follow
    if (__all_sync(0xffffffffu, ready)) return true;
    set_status(status, SD_ETIMEOUT);
    cs.abort = 1;
    return false;
}

// ---------------------------------------------------------------------------
// producer: stream this CTA's share of one matmul phase through the ring and
// publish its schedule: piece k goes to queue slot k % PQ_N before the first
// stage of that piece is armed, so a consumer that has waited for that stage
// reads it (the stage's mbarrier orders the write).  `it` counts stages over
// the whole launch (slot it % NS, phase parity it / NS), `npub` pieces.
// ---------------------------------------------------------------------------
__device__ inline void produce_phase(const QmmArgs &a, const Smem &sm, uint32_t &it, uint32_t &npub, CtaShared &cs,
                                     uint64_t pol, uint64_t *tslot = nullptr) {
    if (tslot) tslot[TR_PROD_FIRST] = gtimer_ns();
    PieceIter pit;
    pieces_begin(a, pit);
    Piece pc, nx;
    bool have = pieces_next_on(a, pit, pc);
    while (have && !cs.abort) {
        const bool more = pieces_next_on(a, pit, nx);
        {
            QPiece &q = cs.pq[npub % PQ_N];
            q.s = pc.s;
            q.u = pc.u;
            q.j0 = pc.j0;
            q.j1 = pc.j1;
            q.first = pc.first;
            q.np = pc.np;
            int expected = pc.np;
            if (a.KS > 1 && !a.defer) {  // a shared unit waits for the pieces of all its splits (unused
                                         // when a combine phase adds them: the walk is costly)
                expected = 0;
                for (int s2 = 0; s2 < a.KS; ++s2) {
                    int f2, np2;
                    unit_split_owners(a, s2, pc.u, f2, np2);
                    expected += np2;
                }
            }
            q.expected = expected;
            q.last = more ? 0 : 1;
        }
        ++npub;
        const int s = pc.s, u = pc.u, j1 = pc.j1;
        for (int jj = pc.j0; jj < j1 && !cs.abort; jj += a.SB) {
            const int n = j1 - jj < a.SB ? j1 - jj : a.SB;
            const int stg = static_cast<int>(it % a.NS);
            const uint32_t ph = (it / a.NS) & 1u;
            if ((it & 7u) == 0 && out_of_time(cs, a.status, 1)) {  // every 8th stage
                cs.abort = 1;
                break;
            }
            if (!mbar_wait_bounded(&sm.empty[stg], ph ^ 1u, WAIT_NS, &cs.abort)) {
                set_status(a.status, SD_ETIMEOUT);
                cs.abort = 1;
                break;
            }
            const uint32_t bytes = static_cast<uint32_t>(n) * a.step_bytes;
            const uint8_t *src =
                a.w + (static_cast<int64_t>(phys_unit(a, u)) * a.KB + static_cast<int64_t>(s) * a.KBs + jj) *
                          a.step_bytes;
            // site 101: the copy stays inside its unit's k range and its ring stage
            if (!SD_INB(phys_unit(a, u) >= 0 && phys_unit(a, u) < a.NU && s >= 0 && s < a.KS && jj >= 0 &&
                            static_cast<int64_t>(s) * a.KBs + jj + n <= a.KB && bytes <= a.stage_stride,
                        a.status, 101)) {
                cs.abort = 1;
                break;
            }
            mbar_arrive_expect_tx(&sm.full[stg], bytes);
            bulk_g2s(sm.ring + static_cast<size_t>(stg) * a.stage_stride, src, bytes, &sm.full[stg], pol);
            ++it;
        }
        pc = nx;
        have = more;
    }
    if (tslot) tslot[TR_PROD_LAST] = gtimer_ns();
}

// never leave with copies in flight: wait for the last issued stages
__device__ inline void producer_drain(const Smem &sm, uint32_t it, int NS) {
    const uint32_t first = it > static_cast<uint32_t>(NS) ? it - NS : 0u;
    for (uint32_t k = first; k < it; ++k) mbar_wait_bounded(&sm.full[k % NS], (k / NS) & 1u, WAIT_NS);
}

// ---------------------------------------------------------------------------
// consumers: activations of one k-split into shared memory
// ---------------------------------------------------------------------------

// Bulk copy of the split's fragments and {corr, d_a} pairs (consumer thread 0).  The fragments
// were written by generic stores of other CTAs, made visible by the grid barrier's acquire;
// the proxy fence orders that acquire before the copy engine's reads.
__device__ __forceinline__ void stage_issue(const QmmArgs &a, const Smem &sm, int s, int len) {
    const int64_t b0 = static_cast<int64_t>(s) * a.KBs;
    const uint32_t fb = af_frag_bytes(a.M), mb = af_meta_bytes_q(a.M, a.qt);
    const uint32_t nf = static_cast<uint32_t>(len) * fb, nm = static_cast<uint32_t>(len) * mb;
    const uint32_t ns = a.af_norm ? static_cast<uint32_t>(a.M) * a.ss_ld * 4u : 0u;
    // site 102: the split's blocks lie inside the input and fit the activation region (sized for KBs);
    // a skipped copy leaves the consumers' wait to run out
    if (!SD_INB(s >= 0 && s < a.KS && len >= 0 && len <= a.KBs && b0 + len <= a.KB, a.status, 102)) return;
    fence_proxy_async_global();
    fence_proxy_async_shared();
    mbar_arrive_expect_tx(sm.act_bar, nf + nm + ns);
    bulk_g2s_l2keep(sm.act, a.af_frag + b0 * fb, nf, sm.act_bar);
    bulk_g2s_l2keep(sm.meta, reinterpret_cast<const uint8_t *>(a.af_meta) + b0 * mb, nm, sm.act_bar);
    if (ns) bulk_g2s_l2keep(sm.ss, a.ss_in, ns, sm.act_bar);
}

// The same shared-memory contents formed from plain int8 rows and scales (all consumer threads).
template <int QT>
__device__ inline void stage_rows(const QmmArgs &a, const Smem &sm, int s, int len, int tid) {
    const int M = a.M, NT = af_nt(M);
    const int64_t K = static_cast<int64_t>(a.KB) * 32;
    const int b0 = s * a.KBs;
    const int nitems = len * M * 4;  // (block, position, c)
    for (int base = tid; base < nitems; base += 4 * CONS_THREADS) {
        uint2 raw[4];
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
            const int it = base + u4 * CONS_THREADS;
            raw[u4] = make_uint2(0u, 0u);
            if (it < nitems) {
                const int jb = it / (M * 4), rem = it - jb * M * 4, m = rem >> 2, c = rem & 3;
                raw[u4] = b_raw(a.q + m * K + static_cast<int64_t>(b0 + jb) * 32, c);
            }
        }
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) {
            const int it = base + u4 * CONS_THREADS;
            if (it < nitems) {
                if (NT == 1) reinterpret_cast<uint4 *>(sm.act)[it] = b_frag_from_raw<QT>(raw[u4]);
                else reinterpret_cast<uint2 *>(sm.act)[it] = raw[u4];
            }
        }
    }
    const int P8 = 8 * NT;
    for (int it = tid; it < len * P8; it += CONS_THREADS) {
        const int jb = it / P8, m = it - jb * P8;
        const bool real = m < M;
        const float da = real ? __ldcg(a.sc + static_cast<int64_t>(m) * a.KB + b0 + jb) : 0.0f;
        if constexpr (is_kq(QT)) {
            // the activations' code sums over k 0-7, 8-15, 16-23, 24-31 of the block
            int s4[4] = {0, 0, 0, 0};
            if (real) {
                const uint4 *p = reinterpret_cast<const uint4 *>(a.q + m * K + static_cast<int64_t>(b0 + jb) * 32);
                const uint4 x0 = __ldcg(p), x1 = __ldcg(p + 1);
                s4[0] = dp4a(0x01010101, static_cast<int>(x0.y), dp4a(0x01010101, static_cast<int>(x0.x), 0));
                s4[1] = dp4a(0x01010101, static_cast<int>(x0.w), dp4a(0x01010101, static_cast<int>(x0.z), 0));
                s4[2] = dp4a(0x01010101, static_cast<int>(x1.y), dp4a(0x01010101, static_cast<int>(x1.x), 0));
                s4[3] = dp4a(0x01010101, static_cast<int>(x1.w), dp4a(0x01010101, static_cast<int>(x1.z), 0));
            }
            reinterpret_cast<float4 *>(sm.meta)[it] = kq_meta<QT>(s4, da);
        } else {
            const float corr = dot_corr<QT>(real ? a.q + m * K + static_cast<int64_t>(b0 + jb) * 32 : nullptr);
            reinterpret_cast<float2 *>(sm.meta)[it] = make_float2(corr, da);
        }
    }
}

// Inverse RMS of row m from its block sums of squares (whole warp; the result is broadcast):
// the pairwise tree over the zero-padded power of two of at least 256 slots.  Slots past
// K/32 are zeros, so the tree over 256 slots (8 per lane) and the one over 1024 slots (32 per
// lane) give the same sum when K/32 <= 256 (their extra levels add exact zeros).
__device__ __forceinline__ float warp_row_inv(const QmmArgs &a, const Smem &sm, int m, int lane) {
    const float *row = sm.ss + m * a.ss_ld;
    float sum;
    if (a.KB <= 256) {
        float v[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int slot = lane + 32 * r;
            v[r] = slot < a.KB ? row[slot] : 0.0f;
        }
#pragma unroll
        for (int h = 4; h >= 1; h >>= 1)
#pragma unroll
            for (int r = 0; r < h; ++r) v[r] = __fadd_rn(v[r], v[r + h]);
        float x = v[0];
#pragma unroll
        for (int st = 16; st >= 1; st >>= 1) {
            const float o = __shfl_down_sync(0xffffffffu, x, st);
            if (lane < st) x = __fadd_rn(x, o);
        }
        sum = x;
    } else {
        float v[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const int slot = lane + 32 * r;
            v[r] = slot < a.KB ? row[slot] : 0.0f;
        }
        sum = tree1024_warp(v);
    }
    const float mean = __fdiv_rn(sum, static_cast<float>(a.KB) * 32.0f);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, a.eps)));
    return __shfl_sync(0xffffffffu, inv, 0);
}

// The four fp16 row scales of a lane's group (rows g, g+8, 16+g, 24+g) as pairs (w, w), ready to
// multiply a lane's two positions at once.
__device__ __forceinline__ void row_scale_pairs(uint2 sw, float2 (&wr)[4]) {
    const __half2 h01 = *reinterpret_cast<const __half2 *>(&sw.x), h23 = *reinterpret_cast<const __half2 *>(&sw.y);
    wr[0] = __half22float2(__low2half2(h01));
    wr[1] = __half22float2(__high2half2(h01));
    wr[2] = __half22float2(__low2half2(h23));
    wr[3] = __half22float2(__high2half2(h23));
}

// steps one call of stage_compute covers when full: 32 records of 4-bit, 16 gate|up pairs or Q8_0 records
__host__ __device__ constexpr int sub_steps(int qtype, int pair) { return pair ? 2 * NCW : (qtype == SD_Q8_0 ? 2 * NCW : 4 * NCW); }

// ---------------------------------------------------------------------------
// consumers: the records of one stage (sub-step).  Warp w takes steps w, w + 8, ...;
// acc[nt][t][i] holds row 16t + g + 8(i>>1), position 8nt + 2c + (i&1)
// (accu: the up rows of a gate|up pair).
// ---------------------------------------------------------------------------
template <int QT, int PAIR, int NT, bool FULL>
__device__ __forceinline__ void stage_compute(const uint8_t *sbase, int n, int jb0, const uint8_t *act,
                                              const float *meta, int M, int warp, int lane, const float2 (&inv)[NT],
                                              float (&acc)[NT][2][4], float (&accu)[PAIR ? NT : 1][2][4]) {
    constexpr int REC = QT == SD_Q8_0 ? 1088 : 576;   // bytes of one 32-row record
    constexpr int CODE = QT == SD_Q8_0 ? 1024 : 512;  // code bytes of a record
    constexpr int STEP = PAIR ? 2 * REC : REC;
    constexpr int RPW = (PAIR || QT == SD_Q8_0) ? 2 : 4;  // steps per warp in a full stage
    const int lg = lane >> 2, lc = lane & 3;
    const uint4 *act4 = reinterpret_cast<const uint4 *>(act);
    const uint2 *act2 = reinterpret_cast<const uint2 *>(act);
    const float4 *meta4 = reinterpret_cast<const float4 *>(meta);
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int r = warp + NCW * i;
        if (!FULL && r >= n) break;
        const uint8_t *rp = sbase + r * STEP;
        const int jb = jb0 + r;
        uint32_t af[2][2][4], afu[2][2][4];
        float2 wr[4], ur[4];  // scales of rows g, g+8, 16+g, 24+g, each as a pair (w, w)
        if (QT == SD_Q4_32) q4_frag(*reinterpret_cast<const uint4 *>(rp + lane * 16), af);
        else q8_frag(*reinterpret_cast<const uint4 *>(rp + lane * 16), *reinterpret_cast<const uint4 *>(rp + 512 + lane * 16), af);
        row_scale_pairs(*reinterpret_cast<const uint2 *>(rp + CODE + lg * 8), wr);
        if (PAIR) {
            q4_frag(*reinterpret_cast<const uint4 *>(rp + REC + lane * 16), afu);
            row_scale_pairs(*reinterpret_cast<const uint2 *>(rp + REC + CODE + lg * 8), ur);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            uint4 bf;
            if (NT == 1) {
                // lanes of padding positions (lg >= M) read whatever fragment follows in shared memory
                // (the next block's, or the {corr, d_a} pairs after the last block): their columns of the
                // product are never stored
                bf = act4[jb * 4 * M + lane];
            } else {
                const uint2 raw = 8 * nt + lg < M ? act2[jb * 4 * M + 32 * nt + lane] : make_uint2(0u, 0u);
                bf = b_frag_from_raw<QT>(raw);
            }
            const float4 mt = meta4[(jb * NT + nt) * 4 + lc];  // corr(p), d_a(p), corr(p+1), d_a(p+1); p = 8nt+2c
            const float2 corr = make_float2(mt.x, mt.z);
            const float2 da = fmul2_rn(inv[nt], make_float2(mt.y, mt.w));  // exact when inv = 1
            float d[2][4];
            record_dots(af, bf, corr, d);
            // acc(row, p), acc(row, p+1) += dot * (w_row * d_a): two fp32 roundings per element, as pairs
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float2 r = ffma2_rn(make_float2(d[t][2 * h], d[t][2 * h + 1]), fmul2_rn(wr[2 * t + h], da),
                                              make_float2(acc[nt][t][2 * h], acc[nt][t][2 * h + 1]));
                    acc[nt][t][2 * h] = r.x;
                    acc[nt][t][2 * h + 1] = r.y;
                }
            if (PAIR) {
                record_dots(afu, bf, corr, d);
#pragma unroll
                for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        float(&au)[2][4] = accu[PAIR ? nt : 0];
                        const float2 r = ffma2_rn(make_float2(d[t][2 * h], d[t][2 * h + 1]),
                                                  fmul2_rn(ur[2 * t + h], da),
                                                  make_float2(au[t][2 * h], au[t][2 * h + 1]));
                        au[t][2 * h] = r.x;
                        au[t][2 * h + 1] = r.y;
                    }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// consumers, K-quant formats: the records of one sub-step.  Steps come in whole super-records (eight
// 32-weight sub-blocks of 32 rows); record r = warp + 8i of a sub-step is sub-block `warp` of
// super-record i, so each warp always takes the same sub-block.  Accumulators as stage_compute's.
//  Q4_K: dot = sum code * a exactly (the activations' {c0} removes the code offset); per (row,
//    position) acc += d_a (d sc dot - dmin m S), S the activations' code sum.
//  Q6_K: the two 16-weight halves' dots (code - 32) a separately (corrections c0, c1); acc += (d d_a)
//    (sc_lo dot_lo + sc_hi dot_hi), whose integer part is exact below 2^24.
// ---------------------------------------------------------------------------
template <int QT, int PAIR, int NT, bool FULL>
__device__ __forceinline__ void stage_compute_kq(const uint8_t *sbase, int n, int jb0, const uint8_t *act,
                                                 const float *meta, int M, int warp, int lane,
                                                 const float2 (&inv)[NT], float (&acc)[NT][2][4],
                                                 float (&accu)[PAIR ? NT : 1][2][4]) {
    constexpr int SR = QT == SD_Q4_K ? Q4K_SR : Q6K_SR;
    constexpr int PSR = PAIR ? 2 * SR : SR;           // a gate|up pair of super-records
    constexpr int RPW = PAIR ? 2 : 4;                 // records per warp in a full sub-step
    const int lg = lane >> 2, lc = lane & 3;
    const uint4 *act4 = reinterpret_cast<const uint4 *>(act);
    const uint2 *act2 = reinterpret_cast<const uint2 *>(act);
    const float4 *meta4 = reinterpret_cast<const float4 *>(meta);
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int r = warp + NCW * i;
        if (!FULL && r >= n) break;
        const int jb = jb0 + r;
#pragma unroll
        for (int half = 0; half < (PAIR ? 2 : 1); ++half) {
            const uint8_t *srp = sbase + i * PSR + half * SR;
            uint32_t af[2][2][4];
            float f1[4], f2[4];  // per row g, g+8, 16+g, 24+g: Q4_K d sc, dmin m; Q6_K sc_lo, sc_hi
            float dq[4];         // Q6_K: d per row
            if (QT == SD_Q4_K) {
                q4_frag(*reinterpret_cast<const uint4 *>(srp + warp * 512 + lane * 16), af);
                const uint2 scm = *reinterpret_cast<const uint2 *>(srp + 4096 + 64 * warp + 8 * lg);
                const uint4 dd = *reinterpret_cast<const uint4 *>(srp + 4608 + 16 * lg);
                const uint32_t dw[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 dm = __half22float2(*reinterpret_cast<const __half2 *>(&dw[e]));  // d, dmin
                    // (scale, min) of row e: each byte under the exponent of 2^23, less 2^23 (exact), as a pair
                    const float2 sm = fadd2_rn(make_float2(ubyte_magic(scm.x, e), ubyte_magic(scm.y, e)),
                                               make_float2(-8388608.0f, -8388608.0f));
                    const float2 pr = fmul2_rn(dm, sm);  // exact: 11 x 6 bits
                    f1[e] = pr.x;
                    f2[e] = pr.y;
                }
            } else {
                q6_frag(*reinterpret_cast<const uint4 *>(srp + warp * 768 + lane * 16),
                        *reinterpret_cast<const uint2 *>(srp + warp * 768 + 512 + lane * 8), af);
                const uint2 scb = *reinterpret_cast<const uint2 *>(srp + 6144 + 64 * warp + 8 * lg);
                const uint2 dh = *reinterpret_cast<const uint2 *>(srp + 6656 + 8 * lg);
                const float2 d01 = __half22float2(*reinterpret_cast<const __half2 *>(&dh.x));
                const float2 d23 = __half22float2(*reinterpret_cast<const __half2 *>(&dh.y));
                dq[0] = d01.x;
                dq[1] = d01.y;
                dq[2] = d23.x;
                dq[3] = d23.y;
#pragma unroll
                for (int e = 0; e < 4; ++e) {  // int8 scales: the biased byte less 2^23 + 128, exact
                    const float2 sc = fadd2_rn(make_float2(ubyte_magic(scb.x ^ 0x80808080u, e),
                                                           ubyte_magic(scb.y ^ 0x80808080u, e)),
                                               make_float2(-8388736.0f, -8388736.0f));
                    f1[e] = sc.x;
                    f2[e] = sc.y;
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                uint4 bf;
                if (NT == 1) {
                    bf = act4[jb * 4 * M + lane];  // padding lanes read neighbouring fragments; never stored
                } else {
                    const uint2 raw = 8 * nt + lg < M ? act2[jb * 4 * M + 32 * nt + lane] : make_uint2(0u, 0u);
                    bf = b_frag_from_raw<QT>(raw);
                }
                const float4 m0 = meta4[(jb * NT + nt) * 8 + 2 * lc], m1 = meta4[(jb * NT + nt) * 8 + 2 * lc + 1];
                const float2 da = fmul2_rn(inv[nt], make_float2(m0.z, m1.z));
                float(&ac)[2][4] = half ? accu[PAIR ? nt : 0] : acc[nt];
                if (QT == SD_Q4_K) {
                    float d[2][4];
                    record_dots(af, bf, make_float2(m0.x, m1.x), d);
                    const float2 ns = make_float2(-m0.w, -m1.w);
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int e = 2 * t + h;
                            const float2 v = ffma2_rn(make_float2(d[t][2 * h], d[t][2 * h + 1]),
                                                      make_float2(f1[e], f1[e]), fmul2_rn(ns, make_float2(f2[e], f2[e])));
                            const float2 r2 = ffma2_rn(v, da, make_float2(ac[t][2 * h], ac[t][2 * h + 1]));
                            ac[t][2 * h] = r2.x;
                            ac[t][2 * h + 1] = r2.y;
                        }
                } else {
                    float dl[2][4], dh2[2][4];
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        mma_init(dl[t], af[t][0], bf.x, bf.y, m0.x, m1.x);
                        mma_init(dh2[t], af[t][1], bf.z, bf.w, m0.y, m1.y);
                    }
#pragma unroll
                    for (int t = 0; t < 2; ++t)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int e = 2 * t + h;
                            const float2 v = ffma2_rn(make_float2(dh2[t][2 * h], dh2[t][2 * h + 1]),
                                                      make_float2(f2[e], f2[e]),
                                                      fmul2_rn(make_float2(dl[t][2 * h], dl[t][2 * h + 1]),
                                                               make_float2(f1[e], f1[e])));
                            const float2 r2 = ffma2_rn(v, fmul2_rn(make_float2(dq[e], dq[e]), da),
                                                       make_float2(ac[t][2 * h], ac[t][2 * h + 1]));
                            ac[t][2 * h] = r2.x;
                            ac[t][2 * h + 1] = r2.y;
                        }
                }
            }
        }
    }
}

// The k-split of the CTA's first piece in a matmul phase whose activations arrive as fragments, or -1
// (not such a phase, or no piece here).  A function of the descriptor alone when the call is not
// restricted, so the one-launch pass walks it while it waits at the grid barrier.
constexpr int SPLIT_LATER = -2;  // restricted call: its unit mask may only be read after the barrier
__device__ inline int first_split(const QmmArgs &a) {
    if (a.kind != KIND_MATMUL || !a.af_frag) return -1;
    PieceIter pit;
    pieces_begin(a, pit);
    Piece pc;
    return pieces_next_on(a, pit, pc) ? pc.s : -1;
}

// Thread 0, right after the grid barrier of a matmul phase whose activations arrive as fragments:
// start the bulk copy of the CTA's first k-split s at once (consume_phase then only waits for it).
// Returns whether it issued the copy.
__device__ inline bool issue_first_split(const QmmArgs &a, const Smem &sm, uint32_t act_it, CtaShared &cs, int s) {
    if (s == SPLIT_LATER) s = first_split(a);
    if (s < 0) return false;
    if (act_it > 0 && !mbar_wait_bounded(sm.act_free, (act_it - 1) & 1u, WAIT_NS, &cs.abort)) {
        set_status(a.status, SD_ETIMEOUT);
        cs.abort = 1;
        return false;
    }
    stage_issue(a, sm, s, (s == a.KS - 1) ? a.KBlast : a.KBs);
    return true;
}

// first_split where it may run before the barrier, SPLIT_LATER where it may not
__device__ __forceinline__ int first_split_early(const QmmArgs &a) { return a.unit_mask ? SPLIT_LATER : first_split(a); }

// The CTA's last piece of a phase, when it is a whole tile finished here (one split, one piece) and no
// statistics are formed inline: its epilogue runs on the consumer warps, a position each, instead of
// waiting in the finishers' queue; the sums over the consumer warps are added in the same order.
__device__ __forceinline__ bool last_by_consumers(const QmmArgs &a, const QPiece &pc) {
    return pc.last && a.KS == 1 && pc.np == 1 && !(a.head && !a.defer_stats);
}

// ---------------------------------------------------------------------------
// consumers: one matmul phase.  `it` counts ring stages, `pk` pieces (their
// partial-sum slots and queue entries), `act_it` activation stagings and
// `nrm_it` those of RMSNorm codes, all over the whole launch.  Every wait is bounded; a warp whose wait fails marks the
// CTA aborted and leaves, and every other wait then gives up at once, so all
// roles reach the phase-end barrier.  Returns false on an abandoned phase.
// ---------------------------------------------------------------------------
template <int QT, int PAIR, int NT>
__device__ inline bool consume_phase(const QmmArgs &a, const Smem &sm, uint32_t &it, uint32_t &pk, uint32_t &act_it,
                                     uint32_t &nrm_it, CtaShared &cs, bool pre_issued = false,
                                     uint64_t *tslot = nullptr) {
    if (!cta_has_work(a)) return true;  // no work for this CTA in this phase
    const int M = a.M;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lg = lane >> 2, lc = lane & 3;
    // descriptor fields the loops use, in registers (the descriptor may sit in shared memory, and
    // every mbarrier operation below is a compiler memory barrier)
    const int SB = a.SB, rows_p = a.rows_p;
    const uint32_t NS = static_cast<uint32_t>(a.NS), NRB = static_cast<uint32_t>(a.NRB), sstride = a.stage_stride;
    uint32_t stg = it % NS, sph = (it / NS) & 1u;  // ring slot and phase parity of stage `it`
    int cur_s = -1;
    const bool tr = tslot != nullptr && threadIdx.x == 0;  // consumer warp 0 keeps the cycle accounts
    long long c_wait = 0, c_comp = 0, c_hand = 0, c_stage = 0, c_last = 0, c0 = 0;
    const long long c_start = tr ? clock64() : 0;
    float2 inv[NT];  // RMSNorm row factors of this lane's positions 8nt + 2c, +1 (1 when not normalised)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) inv[nt] = make_float2(1.0f, 1.0f);
    // launch-wide self-check, once per phase (a clock read per piece measured 0.45 % of the pass); every
    // wait below is bounded on its own
    if (out_of_time(cs, a.status, 2)) cs.abort = 1;
    for (;;) {
        // the next piece's descriptor rides with its first stage
        if (tr) c0 = clock64();
        if (!warp_wait(&sm.full[stg], sph, cs, a.status)) return false;
        if (tr) c_wait += clock64() - c0;
        const QPiece pc = cs.pq[pk % PQ_N];
        const int s = pc.s, j0 = pc.j0, j1 = pc.j1;

        if (s != cur_s) {
            if (tr) c0 = clock64();
            const int len = (s == a.KS - 1) ? a.KBlast : a.KBs;
            if (cur_s >= 0 && lane == 0) mbar_arrive(sm.act_free);  // done with the previous split
            if (a.af_frag) {
                bool issued = pre_issued && cur_s < 0;  // the phase's first copy, issued at the grid barrier
                if (tid == 0 && !issued) {
                    if (act_it > 0 && !mbar_wait_bounded(sm.act_free, (act_it - 1) & 1u, WAIT_NS, &cs.abort)) {
                        set_status(a.status, SD_ETIMEOUT);
                        cs.abort = 1;
                    } else {
                        stage_issue(a, sm, s, len);
                        issued = true;
                    }
                }
                if (!warp_wait(sm.act_bar, act_it & 1u, cs, a.status)) {
                    // a copy may still be landing: thread 0 waits for it before the CTA can end
                    if (tid == 0 && issued) mbar_wait_bounded(sm.act_bar, act_it & 1u, WAIT_NS);
                    return false;
                }
            } else {
                if (act_it > 0 && !warp_wait(sm.act_free, (act_it - 1) & 1u, cs, a.status)) return false;
                stage_rows<QT>(a, sm, s, len, tid);
                mbar_arrive(sm.act_bar);  // every consumer thread: its share is written
                if (!warp_wait(sm.act_bar, act_it & 1u, cs, a.status)) return false;
            }
            ++act_it;
            if (tslot && cur_s < 0 && threadIdx.x == 0) tslot[TR_ACT] = gtimer_ns();
            if (a.af_norm) {
                // the row factors, one warp per row (warp w: rows w, w + 8), published through
                // inv_bar; applied to the block scales as they are loaded: d_a = inv * max|x w| / 127
                for (int m = warp; m < M; m += NCW) {
                    const float r = warp_row_inv(a, sm, m, lane);
                    if (lane == 0) cs.inv[m] = r;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.inv_bar);
                if (!warp_wait(sm.inv_bar, nrm_it & 1u, cs, a.status)) return false;
                ++nrm_it;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int p0 = 8 * nt + 2 * lc;
                    inv[nt] = make_float2(p0 < M ? cs.inv[p0] : 1.0f, p0 + 1 < M ? cs.inv[p0 + 1] : 1.0f);
                }
                // the CTA holding the split's first step writes the scales out (warp w: blocks w, w+8, ...)
                int first = 0, np = 1;
                if (a.D == 0) unit_split_owners(a, s, 0, first, np);
                if (a.s_norm_out && static_cast<int>(blockIdx.x) == first) {
                    const int b0 = s * a.KBs;
                    const float2 *mp = reinterpret_cast<const float2 *>(sm.meta);
                    for (int it2 = warp * 32 + lane; it2 < len * M; it2 += CONS_THREADS) {
                        const int jb = it2 / M, m = it2 - jb * M;
                        a.s_norm_out[static_cast<int64_t>(m) * a.KB + b0 + jb] =
                            __fmul_rn(cs.inv[m], mp[jb * 8 * NT + m].y);
                    }
                }
            }
            cur_s = s;
            if (tr) c_stage += clock64() - c0;
        }

        float acc[NT][2][4], accu[PAIR ? NT : 1][2][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[nt][t][e] = 0.0f;
                    accu[PAIR ? nt : 0][t][e] = 0.0f;
                }

        for (int jj = j0; jj < j1; jj += SB) {
            const int n = j1 - jj < SB ? j1 - jj : SB;
            if (tr) c0 = clock64();
            if (jj != j0 && !warp_wait(&sm.full[stg], sph, cs, a.status)) return false;
            if (tr) {
                const long long c1 = clock64();
                c_wait += c1 - c0;
                c0 = c1;
            }
            const uint8_t *sbase = sm.ring + static_cast<size_t>(stg) * sstride;
            const uint32_t done = stg;
            ++it;
            if (++stg == NS) {
                stg = 0;
                sph ^= 1u;
            }
            constexpr int SUB = sub_steps(QT, PAIR);
            constexpr int STEP = step_bytes_q(QT) * (PAIR ? 2 : 1);
            for (int off = 0; off < n; off += SUB) {
                const int nn = n - off < SUB ? n - off : SUB;
                if constexpr (is_kq(QT)) {
                    if (nn == SUB)
                        stage_compute_kq<QT, PAIR, NT, true>(sbase + off * STEP, nn, jj + off, sm.act, sm.meta, M,
                                                             warp, lane, inv, acc, accu);
                    else
                        stage_compute_kq<QT, PAIR, NT, false>(sbase + off * STEP, nn, jj + off, sm.act, sm.meta, M,
                                                              warp, lane, inv, acc, accu);
                } else {
                    if (nn == SUB)
                        stage_compute<QT, PAIR, NT, true>(sbase + off * STEP, nn, jj + off, sm.act, sm.meta, M, warp,
                                                          lane, inv, acc, accu);
                    else
                        stage_compute<QT, PAIR, NT, false>(sbase + off * STEP, nn, jj + off, sm.act, sm.meta, M, warp,
                                                           lane, inv, acc, accu);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[done]);
            if (tr) c_comp += clock64() - c0;
        }

        // hand the piece's partial sums to the finishers
        if (tr) c0 = clock64();
        const uint32_t b = pk % NRB, use = pk / NRB;
        ++pk;
        if (!warp_wait(&sm.rempty[b], (use & 1u) ^ 1u, cs, a.status)) return false;
        float *rb = sm.red + (static_cast<size_t>(b) * NCW + warp) * M * rows_p;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int m = nt * 8 + 2 * lc + (e & 1), row = 16 * t + lg + 8 * (e >> 1);
                    if (m < M) {
                        rb[m * rows_p + row] = acc[nt][t][e];
                        if (PAIR) rb[m * rows_p + 32 + row] = accu[PAIR ? nt : 0][t][e];
                    }
                }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.rfull[b]);
        if (tr) c_hand += clock64() - c0;
        if (last_by_consumers(a, pc)) {
            // the CTA's last tile: every consumer warp's partial sums, then a position per warp
            if (tr) c0 = clock64();
            if (!warp_wait(&sm.rfull[b], use & 1u, cs, a.status)) return false;
            const int up = phys_unit(a, pc.u);
            const float *rb0 = sm.red + static_cast<size_t>(b) * NCW * M * rows_p;
            const size_t wstride = static_cast<size_t>(M) * rows_p;
            for (int m = warp; m < M; m += NCW) {
                float v = rb0[m * rows_p + lane], vu = PAIR ? rb0[m * rows_p + 32 + lane] : 0.0f;
#pragma unroll
                for (int w2 = 1; w2 < NCW; ++w2) {
                    v = __fadd_rn(v, rb0[w2 * wstride + m * rows_p + lane]);
                    if (PAIR) vu = __fadd_rn(vu, rb0[w2 * wstride + m * rows_p + 32 + lane]);
                }
                float res = 0.0f, nw = 0.0f;
                if (!PAIR) {
                    const int64_t n = static_cast<int64_t>(up) * 32 + lane;
                    const bool nok = n < a.n_out;
                    res = (a.residual && nok) ? __ldcg(a.residual + m * a.n_out + n) : 0.0f;
                    if (a.norm_next && nok) nw = __ldg(a.norm_next + n);
                }
                epilogue<PAIR, is_kq(QT)>(a, up, m, lane, v, vu, res, nw);
            }
            if (tr) c_last += clock64() - c0;
        }
        if (pc.last) break;
    }
    if (lane == 0) mbar_arrive(sm.act_free);  // done with this phase's last split
    if (tr) {
        tslot[TR_CONS_END] = gtimer_ns();
        tslot[TR_CYC_WAIT] = static_cast<uint64_t>(c_wait);
        tslot[TR_CYC_COMP] = static_cast<uint64_t>(c_comp);
        tslot[TR_CYC_HAND] = static_cast<uint64_t>(c_hand);
        tslot[TR_CYC_STAGE] = static_cast<uint64_t>(c_stage);
        tslot[TR_CYC_LAST] = static_cast<uint64_t>(c_last);
        tslot[TR_CYC_ALL] = static_cast<uint64_t>(clock64() - c_start);
    }
    return !cs.abort;
}

// ---------------------------------------------------------------------------
// finisher warps (warp f takes positions f, f + NF, ...): rendezvous through
// mbarriers (every wait bounded).  fin_sync: each finisher warp arrives;
// warp 0 waits for all, lane 0 decides, and the decision reaches the others.
// ---------------------------------------------------------------------------
template <class Leader>
__device__ __forceinline__ bool fin_sync(const Smem &sm, CtaShared &cs, uint32_t &fin_it, int f, int lane, int *status,
                                         Leader leader) {
    const uint32_t ph = fin_it & 1u;
    ++fin_it;
    __syncwarp();
    if (lane == 0) mbar_arrive(sm.fin_g);
    if (f == 0) {
        if (!warp_wait(sm.fin_g, ph, cs, status)) return false;
        int d = 0;
        if (lane == 0) d = leader() ? 1 : 0;
        if (lane == 0) {
            cs.fin_flag = d;
            mbar_arrive(sm.fin_b);
        }
        return __shfl_sync(0xffffffffu, d, 0) != 0;
    }
    if (!warp_wait(sm.fin_b, ph, cs, status)) return false;
    return cs.fin_flag != 0;
}

// Adds `n_done` finished 32-row tiles to statistics tile `st`; the CTA that completes the tile
// forms its statistics, the CTA that completes the last tile folds them.  Every finisher warp
// calls it with the same arguments; the finished logits were written before the call.
__device__ inline void head_flush(const QmmArgs &a, const Smem &sm, CtaShared &cs, uint32_t &fin_it, int st,
                                  int n_done, int lane, int f) {
    if (st < 0 || n_done == 0 || cs.abort) return;
    const bool last = fin_sync(sm, cs, fin_it, f, lane, a.status, [&]() {
        const int left = a.NU - st * (STAT_TILE / 32);
        const int tiles_in_st = left < STAT_TILE / 32 ? left : STAT_TILE / 32;
        const unsigned old = atom_add_acq_rel(&a.st_cnt[st], static_cast<uint32_t>(n_done));
        return static_cast<int>(old) + n_done == tiles_in_st;
    });
    if (!last || cs.abort) return;
    head_tile_stats(a, st, lane, f);
    const bool fold = fin_sync(sm, cs, fin_it, f, lane, a.status, [&]() {
        a.st_cnt[st] = 0u;
        const unsigned old = atom_add_acq_rel(a.st_done, 1u);
        return static_cast<int>(old) == a.n_stiles - 1;
    });
    if (!fold || cs.abort) return;
    head_final_fold(a, lane, f);
    if (f == 0 && lane == 0) *a.st_done = 0u;
}

// One matmul phase of the finisher warps.  For each piece, in the consumers' order: add the 8
// consumer warps' partial sums (warp order), then finish the unit directly, or store the partial
// and, if this CTA arrived last, add all partials in (split, piece) order and finish it.
template <int PAIR, int NT, bool KQ = false>
__device__ inline bool finish_phase(const QmmArgs &a, const Smem &sm, uint32_t &pk, uint32_t &fin_it, CtaShared &cs,
                                    int f) {
    constexpr int ROWS = PAIR ? 64 : 32;
    constexpr int FIN_MPW = (8 * NT + NF - 1) / NF;  // positions per finisher warp at most
    constexpr int CH = 8;                            // partial sums loaded together
    constexpr int FKS = 8, FP = 4;                   // splits x pieces held at once when all splits share
    if (!cta_has_work(a)) return true;  // no work for this CTA in this phase
    const int M = a.M;
    const int lane = threadIdx.x & 31;
    int st_cur = -1, st_n = 0;  // head: current statistics tile and tiles finished in it
    for (;;) {
        const uint32_t b = pk % static_cast<uint32_t>(a.NRB), use = pk / static_cast<uint32_t>(a.NRB);
        const uint32_t slot = pk % PQ_N;
        ++pk;
        if (!warp_wait(&sm.rfull[b], use & 1u, cs, a.status)) return false;
        const QPiece pc = cs.pq[slot];
        if (last_by_consumers(a, pc)) {  // the consumers finish this tile
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.rempty[b]);
            break;
        }
        const int s = pc.s, u = pc.u;
        const bool direct = (a.KS == 1) && (pc.np == 1);
        // values the epilogue needs, in flight while the partial sums are added
        float res[FIN_MPW], nw = 0.0f;
        const int up = phys_unit(a, u);  // the row tile of this unit
        if (!PAIR) {
            const int64_t n = static_cast<int64_t>(up) * 32 + lane;
            const bool nok = n < a.n_out;
#pragma unroll
            for (int i = 0; i < FIN_MPW; ++i) {
                const int m = f + NF * i;
                res[i] = (a.residual && nok && m < M) ? __ldcg(a.residual + m * a.n_out + n) : 0.0f;
            }
            if (a.norm_next && nok) nw = __ldg(a.norm_next + n);
        }
        // this warp's positions: the 8 consumer warps' partial sums, added in warp order
        float v[FIN_MPW], vu[FIN_MPW];
        {
            const float *rb = sm.red + static_cast<size_t>(b) * NCW * M * a.rows_p;
            const size_t wstride = static_cast<size_t>(M) * a.rows_p;
#pragma unroll
            for (int i = 0; i < FIN_MPW; ++i) {
                const int m = f + NF * i;
                v[i] = vu[i] = 0.0f;
                if (m < M) {
                    v[i] = rb[m * a.rows_p + lane];
                    if (PAIR) vu[i] = rb[m * a.rows_p + 32 + lane];
#pragma unroll
                    for (int w2 = 1; w2 < NCW; ++w2) {
                        v[i] = __fadd_rn(v[i], rb[w2 * wstride + m * a.rows_p + lane]);
                        if (PAIR) vu[i] = __fadd_rn(vu[i], rb[w2 * wstride + m * a.rows_p + 32 + lane]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.rempty[b]);  // the slot is free again
        }
        bool finish = direct;
        if (!direct) {
            // site 103: this CTA's partial-sum slot of (unit, split) exists
            const int slot_c = static_cast<int>(blockIdx.x) - pc.first;
            if (!SD_INB(u >= 0 && u < a.NU && s >= 0 && s < a.KS && slot_c >= 0 && slot_c < a.P && pc.np <= a.P, a.status,
                        103)) {
                cs.abort = 1;
                return false;
            }
            float *pp = a.part + ((static_cast<int64_t>(u) * a.KS + s) * a.P + slot_c) * (ROWS * MPAD);
#pragma unroll
            for (int i = 0; i < FIN_MPW; ++i) {
                const int m = f + NF * i;
                if (m < M) {
                    pp[m * ROWS + lane] = v[i];
                    if (PAIR) pp[m * ROWS + 32 + lane] = vu[i];
                }
            }
            if (a.defer) {  // the combine phase after the grid barrier adds them up
                if (pc.last) break;
                continue;
            }
            // every finisher's partial sums before the release in the counter update
            finish = fin_sync(sm, cs, fin_it, f, lane, a.status, [&]() {
                // site 104: one counter per unit, inside the workspace's counter region
                if (!SD_INB(u < WS_UNIT_CNT && pc.expected >= 1 && pc.expected <= a.KS * a.P, a.status, 104))
                    return false;
                const unsigned old = atom_add_acq_rel(&a.cnt[u], 1u);
                return static_cast<int>(old) == pc.expected - 1;
            });
            if (cs.abort) return false;
            if (finish && !PAIR && a.KS > 1 && a.KS <= FKS && a.P <= FP) {
                // every partial sum of the unit in one round of loads per position, added in
                // (split, piece) order as in the chunked walk below
                int npa[FKS];
#pragma unroll
                for (int s2 = 0; s2 < FKS; ++s2) {
                    int f2;
                    npa[s2] = 0;
                    if (s2 < a.KS) unit_split_owners(a, s2, u, f2, npa[s2]);
                    if (!SD_INB(npa[s2] >= 0 && npa[s2] <= a.P, a.status, 105)) npa[s2] = 0;
                }
#pragma unroll
                for (int i = 0; i < FIN_MPW; ++i) {
                    const int m = f + NF * i;
                    v[i] = 0.0f;
                    if (m < M) {
                        float x[FKS][FP];
#pragma unroll
                        for (int s2 = 0; s2 < FKS; ++s2) {
                            const float *qs = a.part + (static_cast<int64_t>(u) * a.KS + s2) * a.P * (ROWS * MPAD) +
                                              m * ROWS + lane;
#pragma unroll
                            for (int c = 0; c < FP; ++c) x[s2][c] = c < npa[s2] ? __ldcg(qs + c * (ROWS * MPAD)) : 0.0f;
                        }
                        bool first = true;
#pragma unroll
                        for (int s2 = 0; s2 < FKS; ++s2)
#pragma unroll
                            for (int c = 0; c < FP; ++c)
                                if (c < npa[s2]) {
                                    v[i] = first ? x[s2][c] : __fadd_rn(v[i], x[s2][c]);
                                    first = false;
                                }
                    }
                }
                if (f == 0 && lane == 0) a.cnt[u] = 0u;
            } else if (finish) {  // the acquire in the counter update orders the loads below
#pragma unroll
                for (int i = 0; i < FIN_MPW; ++i) v[i] = vu[i] = 0.0f;
                bool first = true;
                for (int s2 = 0; s2 < a.KS; ++s2) {
                    int f2, np;
                    if (a.KS == 1) np = pc.np;
                    else unit_split_owners(a, s2, u, f2, np);
                    if (!SD_INB(np >= 0 && np <= a.P, a.status, 105)) np = 0;  // site 105: pieces per split
                    const float *qs = a.part + (static_cast<int64_t>(u) * a.KS + s2) * a.P * (ROWS * MPAD);
                    for (int c0 = 0; c0 < np; c0 += CH) {
                        // a chunk of pieces: every load in flight together, then added in piece order
                        float x[CH][FIN_MPW], xu[CH][FIN_MPW];
#pragma unroll
                        for (int c = 0; c < CH; ++c)
#pragma unroll
                            for (int i = 0; i < FIN_MPW; ++i) {
                                const int m = f + NF * i;
                                const bool in = c0 + c < np && m < M;
                                const float *q = qs + static_cast<int64_t>(c0 + c) * (ROWS * MPAD) + m * ROWS + lane;
                                x[c][i] = in ? __ldcg(q) : 0.0f;
                                xu[c][i] = (PAIR && in) ? __ldcg(q + 32) : 0.0f;
                            }
#pragma unroll
                        for (int c = 0; c < CH; ++c) {
                            if (c0 + c < np) {
#pragma unroll
                                for (int i = 0; i < FIN_MPW; ++i) {
                                    v[i] = first ? x[c][i] : __fadd_rn(v[i], x[c][i]);
                                    if (PAIR) vu[i] = first ? xu[c][i] : __fadd_rn(vu[i], xu[c][i]);
                                }
                                first = false;
                            }
                        }
                    }
                }
                if (f == 0 && lane == 0) a.cnt[u] = 0u;
            }
        }
        if (finish) {
#pragma unroll
            for (int i = 0; i < FIN_MPW; ++i) {
                const int m = f + NF * i;
                if (m < M) epilogue<PAIR, KQ>(a, up, m, lane, v[i], vu[i], res[i], nw);
            }
        }
        if (finish && a.head && !a.defer_stats) {  // the same decisions on every finisher warp
            const int st = up / (STAT_TILE / 32);
            if (st != st_cur) {
                head_flush(a, sm, cs, fin_it, st_cur, st_n, lane, f);
                st_cur = st;
                st_n = 0;
            }
            ++st_n;
        }
        if (pc.last) break;
    }
    if (a.head && !a.defer_stats) head_flush(a, sm, cs, fin_it, st_cur, st_n, lane, f);
    return !cs.abort;
}

// ---------------------------------------------------------------------------
// consumers: the pass's first RMSNorm, on the input rows.  One warp per
// 32-element block, all positions: the block's sum of squares (pairwise tree
// over its squares) and its codes from t = x w (c = max|t| / 127), written as
// int8 codes and as the next matmul's activation fragments holding {corr, c};
// that matmul multiplies c by each row's inverse RMS when it stages them.
// Later RMSNorms are formed the same way in the residual epilogues.
// ---------------------------------------------------------------------------
template <bool KQ = false>
__device__ inline void norm_phase(const QmmArgs &a) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int M = a.M, KB = a.KB;
    const int64_t K = static_cast<int64_t>(KB) * 32;
    const int b0 = static_cast<int>(udiv(static_cast<int64_t>(blockIdx.x) * KB, gridDim.x));
    const int b1 = static_cast<int>(udiv(static_cast<int64_t>(blockIdx.x + 1) * KB, gridDim.x));
    for (int b = b0 + warp; b < b1; b += NCW) {
        for (int m = 0; m < M; ++m) {
            const int64_t i = m * K + static_cast<int64_t>(b) * 32 + lane;
            const float x = __ldcg(a.xin + i);
            const float sq = tree32(__fmul_rn(x, x), lane);
            if (lane == 0) a.ss[m * a.ss_ld + b] = sq;
            float c;
            const int v = requant_lane(__fmul_rn(x, a.norm_w[static_cast<int64_t>(b) * 32 + lane]), c);
            a.q_next[i] = static_cast<int8_t>(v);
            af_write<KQ>(a.af_out_frag, a.af_out_meta, M, b, m, lane, v, c, a.af_out_qt);
        }
    }
}

// ---------------------------------------------------------------------------
// deferred fixup of a matmul whose units are all shared (several k-splits):
// after the grid barrier every CTA finishes an equal share of the units.  Work
// warp w (consumers and finishers, 0..10) takes (unit, position) items w,
// w + 11, ...: the partial sums in (split, piece) order, then the epilogue.
// ---------------------------------------------------------------------------
template <bool KQ = false>
__device__ inline void combine_phase(const QmmArgs &a, int widx) {
    constexpr int ROWS = 32, CH = 8, NWW = NCW + NF;
    constexpr int CKS = 4, CP = 4;  // splits and pieces per split held in registers at once
    const int lane = threadIdx.x & 31, M = a.M;
    const int u0 = static_cast<int>(udiv(static_cast<int64_t>(blockIdx.x) * a.NU, gridDim.x));
    const int u1 = static_cast<int>(udiv(static_cast<int64_t>(blockIdx.x + 1) * a.NU, gridDim.x));
    const int items = (u1 - u0) * M;
    for (int i = widx; i < items; i += NWW) {
        const int u = u0 + i / M, m = i - (i / M) * M, up = phys_unit(a, u);
        const int64_t n = static_cast<int64_t>(up) * 32 + lane;
        const bool nok = n < a.n_out;
        const float res = (a.residual && nok) ? __ldcg(a.residual + m * a.n_out + n) : 0.0f;
        const float nw = (a.norm_next && nok) ? __ldg(a.norm_next + n) : 0.0f;
        float v = 0.0f;
        bool first = true;
        if (a.KS <= CKS && a.P <= CP) {  // every partial sum of the unit in one round of loads
            // every slot the unit has (P per split) is loaded while the pieces per split are worked
            // out; slots past a split's pieces are never added
            int np[CKS];
            float x[CKS][CP];
            static_assert(CKS <= 4, "one table word per unit");
            const uint32_t npw = a.np_tab ? __ldg(reinterpret_cast<const uint32_t *>(a.np_tab) + u) : 0u;
#pragma unroll
            for (int s2 = 0; s2 < CKS; ++s2) {
                const float *qs = a.part + (static_cast<int64_t>(u) * a.KS + s2) * a.P * (ROWS * MPAD) + m * ROWS + lane;
#pragma unroll
                for (int c = 0; c < CP; ++c) x[s2][c] = (s2 < a.KS && c < a.P) ? __ldcg(qs + c * (ROWS * MPAD)) : 0.0f;
            }
#pragma unroll
            for (int s2 = 0; s2 < CKS; ++s2) {
                int f2;
                np[s2] = 0;
                if (s2 < a.KS) {
                    if (a.np_tab) np[s2] = static_cast<int>((npw >> (8 * s2)) & 255u);
                    else unit_split_owners(a, s2, u, f2, np[s2]);
                }
                if (!SD_INB(np[s2] >= 0 && np[s2] <= a.P, a.status, 108)) np[s2] = 0;  // site 108: pieces per split
            }
#pragma unroll
            for (int s2 = 0; s2 < CKS; ++s2)
#pragma unroll
                for (int c = 0; c < CP; ++c)
                    if (c < np[s2]) {  // (split, piece) order, as in the chunked walk below
                        v = first ? x[s2][c] : __fadd_rn(v, x[s2][c]);
                        first = false;
                    }
            epilogue<0, KQ>(a, up, m, lane, v, 0.0f, res, nw);
            continue;
        }
        for (int s2 = 0; s2 < a.KS; ++s2) {
            int f2, np;
            if (a.np_tab) np = __ldg(a.np_tab + static_cast<int64_t>(u) * np_tab_stride(a.KS) + s2);
            else unit_split_owners(a, s2, u, f2, np);
            if (!SD_INB(np >= 0 && np <= a.P, a.status, 108)) np = 0;
            const float *qs = a.part + (static_cast<int64_t>(u) * a.KS + s2) * a.P * (ROWS * MPAD) + m * ROWS + lane;
            for (int c0 = 0; c0 < np; c0 += CH) {
                float x[CH];
#pragma unroll
                for (int c = 0; c < CH; ++c) x[c] = c0 + c < np ? __ldcg(qs + static_cast<int64_t>(c0 + c) * (ROWS * MPAD)) : 0.0f;
#pragma unroll
                for (int c = 0; c < CH; ++c)
                    if (c0 + c < np) {
                        v = first ? x[c] : __fadd_rn(v, x[c]);
                        first = false;
                    }
            }
        }
        epilogue<0, KQ>(a, up, m, lane, v, 0.0f, res, nw);
    }
}

// greedy acceptance (chain when parent == nullptr, else a tree in BFS order); one thread
__device__ inline void greedy_accept(const int32_t *argmax, const int32_t *tokens, const int32_t *parent, int M,
                                     int32_t *out, int32_t *count) {
    if (!parent) {
        const int K = M - 1;
        int n = 0;
        while (n < K && __ldcg(tokens + n) == __ldcg(argmax + n)) {
            out[n] = tokens[n];
            ++n;
        }
        out[n] = __ldcg(argmax + n);
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
        ok[i] = ok[p] && tokens[i] == __ldcg(argmax + p);
        if (ok[i] && depth[i] > depth[best]) best = i;
    }
    const int d = depth[best];
    for (int i = best, j = d - 1; i != 0; i = parent[i], --j) out[j] = tokens[i];
    out[d] = __ldcg(argmax + best);
    *count = d + 1;
}

// ---------------------------------------------------------------------------
// single-operation calls: the activation fragments and {corr, d_a} records of plain int8 rows, for
// the whole k range, formed once per call into the workspace (the same bytes stage_rows forms in
// shared memory), so that each CTA stages a split with one bulk copy instead of latency-bound row
// loads.  Items (block, position, c) of the fragments, then (block, position slot) of the records.
// ---------------------------------------------------------------------------
template <int QT>
__device__ inline void act_frag_build(const int8_t *q, const float *sc, int M, int KB, uint8_t *frag, float *meta) {
    const int NT = af_nt(M), P8 = 8 * NT;
    const int64_t K = static_cast<int64_t>(KB) * 32;
    const int64_t nfrag = static_cast<int64_t>(KB) * M * 4, nmeta = static_cast<int64_t>(KB) * P8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < nfrag + nmeta; it += stride) {
        if (it < nfrag) {
            const int64_t jb = it / (M * 4);
            const int rem = static_cast<int>(it - jb * M * 4), m = rem >> 2, c = rem & 3;
            const uint2 raw = b_raw(q + m * K + jb * 32, c);
            if (NT == 1) reinterpret_cast<uint4 *>(frag)[it] = b_frag_from_raw<QT>(raw);
            else reinterpret_cast<uint2 *>(frag)[it] = raw;
        } else {
            const int64_t i2 = it - nfrag, jb = i2 / P8;
            const int m = static_cast<int>(i2 - jb * P8);
            const bool real = m < M;
            const float da = real ? __ldg(sc + static_cast<int64_t>(m) * KB + jb) : 0.0f;
            if constexpr (is_kq(QT)) {
                int s4[4] = {0, 0, 0, 0};
                if (real) {
                    const uint4 *p = reinterpret_cast<const uint4 *>(q + m * K + jb * 32);
                    const uint4 x0 = __ldg(p), x1 = __ldg(p + 1);
                    s4[0] = dp4a(0x01010101, static_cast<int>(x0.y), dp4a(0x01010101, static_cast<int>(x0.x), 0));
                    s4[1] = dp4a(0x01010101, static_cast<int>(x0.w), dp4a(0x01010101, static_cast<int>(x0.z), 0));
                    s4[2] = dp4a(0x01010101, static_cast<int>(x1.y), dp4a(0x01010101, static_cast<int>(x1.x), 0));
                    s4[3] = dp4a(0x01010101, static_cast<int>(x1.w), dp4a(0x01010101, static_cast<int>(x1.z), 0));
                }
                reinterpret_cast<float4 *>(meta)[i2] = kq_meta<QT>(s4, da);
            } else {
                const float corr = dot_corr<QT>(real ? q + m * K + jb * 32 : nullptr);
                reinterpret_cast<float2 *>(meta)[i2] = make_float2(corr, da);
            }
        }
    }
}

template <int QT>
__global__ void __launch_bounds__(256) act_frag_kernel(const QmmArgs a) {
    pdl_wait();
    pdl_launch_dependents();  // the matmul's producer may start streaming weights
    if (a.skip_if && *reinterpret_cast<const volatile int *>(a.skip_if) != 0) return;
    act_frag_build<QT>(a.q, a.sc, a.M, a.KB, const_cast<uint8_t *>(a.af_frag), const_cast<float *>(a.af_meta));
}

// ---------------------------------------------------------------------------
// single-operation kernel (one matmul phase per launch)
// ---------------------------------------------------------------------------
template <int QT, int PAIR, int NT>
__global__ void __launch_bounds__(QMM_THREADS, 1) qmm_kernel(const QmmArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ CtaShared cs;
    const Smem sm = smem_regions(smem, a);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) cta_init(sm, a.NS, cs, a.af_frag ? 1u : static_cast<uint32_t>(CONS_THREADS));
    __syncthreads();
    if (a.skip_if || a.unit_mask) {  // written by the previous launch: every role waits for it
        pdl_wait();
        if (a.skip_if && *reinterpret_cast<const volatile int *>(a.skip_if) != 0) {
            pdl_launch_dependents();
            return;
        }
    }
    uint32_t it = 0, pk = 0, act_it = 0, nrm_it = 0, fin_it = 0;
    if (warp == PRODUCER_WARP) {
        pdl_launch_dependents();
        if (lane == 0) {
            uint32_t npub = 0;
            produce_phase(a, sm, it, npub, cs, policy_evict_first());
            producer_drain(sm, it, a.NS);
        }
        return;
    }
    // the first split walked before the wait for the previous launch (unless the call is restricted)
    const int s0 = tid == 0 ? first_split_early(a) : -1;
    pdl_wait();
    pdl_launch_dependents();
    if (warp >= FIN_WARP0) {
        (void)finish_phase<PAIR, NT>(a, sm, pk, fin_it, cs, warp - FIN_WARP0);
    } else {
        // the first split's activations are copied while the first weight stage is still in flight
        const bool pre = tid == 0 && issue_first_split(a, sm, act_it, cs, s0);
        (void)consume_phase<QT, PAIR, NT>(a, sm, it, pk, act_it, nrm_it, cs, pre);
    }
}

// Single-operation calls with several k-splits: the matmul leaves every unit's partial sums, and this
// launch adds them in (split, piece) order and runs the epilogue, each CTA an equal share of the units
// (the one-launch pass's combine phase, as its own launch).
static __global__ void __launch_bounds__(WORK_THREADS) qmm_combine_kernel(const QmmArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    combine_phase<false>(a, static_cast<int>(threadIdx.x) >> 5);
}

// ---------------------------------------------------------------------------
// persistent verify pass: every phase of the pass in one cooperative launch,
// phases separated by a grid barrier (release / acquire on a global counter,
// bounded wait).  The producer streams weights, and publishes the schedule,
// across phase boundaries.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Rejection-sampling acceptance by every work warp of one CTA (work-thread index wtid); `scratch`
// (the weight ring, idle by then) holds the shared state.
__device__ __forceinline__ void pass_sample_accept(const QmmArgs &sa, uint8_t *scratch, int wtid) {
    SampleArgs g;
    g.logits = sa.y;
    g.V = sa.n_out;
    g.K = sa.M - 1;
    g.row_max = sa.row_max;
    g.row_sumexp = sa.row_sumexp;
    g.q = sa.q_probs;
    g.drafts = sa.tokens;
    g.T = sa.T;
    g.seed = sa.seed;
    g.base_pos = sa.base_pos;
    g.out = sa.out_tokens;
    g.count = sa.out_count;
    sample_accept<WORK_THREADS>(g, *reinterpret_cast<SampleShared *>(scratch), wtid,
                                []() { named_bar_sync(BAR_WORK, WORK_THREADS); });
}

// SAMPLE: the acceptance phase may run rejection sampling (a separate instantiation, so that the
// greedy pass's code and register allocation stay those of the matmul loops alone)
// The same against the top-k / top-p filtered target.
__device__ __forceinline__ void pass_topk_accept(const QmmArgs &sa, uint8_t *scratch, int wtid) {
    TopkArgs g;
    g.logits = sa.y;
    g.V = sa.n_out;
    g.K = sa.M - 1;
    g.q = sa.q_probs;
    g.drafts = sa.tokens;
    g.T = sa.T;
    g.top_k = sa.top_k;
    g.top_p = sa.top_p;
    g.seed = sa.seed;
    g.base_pos = sa.base_pos;
    g.out = sa.out_tokens;
    g.count = sa.out_count;
    topk_accept<WORK_THREADS>(g, *reinterpret_cast<TopkShared *>(scratch), wtid,
                              []() { named_bar_sync(BAR_WORK, WORK_THREADS); });
}

// KQ: the stack's projections are K-quants (Q4_K, Q6_K) instead of the 32-weight 4-bit format; a separate
// instantiation, so each pass carries the consumer loops of its own formats only
template <int NT, bool SAMPLE, bool KQ = false>
__global__ void __launch_bounds__(QMM_THREADS, 1)
    pass_kernel(const QmmArgs *__restrict__ phases, int n_phases, uint32_t *barrier_ctr, uint64_t *trace) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ CtaShared cs;
    __shared__ QmmArgs sa;  // the current phase, copied from global memory
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const QmmArgs &a0 = phases[0];
    const Smem sm = smem_regions(smem, a0);
    int *status = a0.status;
    if (tid == 0) cta_init(sm, a0.NS, cs, 1u);
    __syncthreads();
    uint32_t it = 0, pk = 0, act_it = 0, nrm_it = 0, fin_it = 0;
    const int G = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
    // this CTA's stamps of phase p (nullptr when not tracing)
    auto tslot = [&](int p) -> uint64_t * {
        return trace ? trace + G + (static_cast<int64_t>(p) * G + cta) * TR_SLOTS : nullptr;
    };
    if (trace && tid == 0) {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        trace[cta] = smid;
    }
    if (warp == PRODUCER_WARP) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            uint32_t npub = 0;
            for (int p = 0; p < n_phases && !cs.abort; ++p)
                if (phases[p].kind == KIND_MATMUL) produce_phase(phases[p], sm, it, npub, cs, pol, tslot(p));
            producer_drain(sm, it, a0.NS);
        }
        return;
    }
    for (int p = 0; p < n_phases; ++p) {
        // the phase descriptor into shared memory before the grid barrier: it is constant, and every
        // work thread left the previous one at the phase-end barrier
        if (warp < NCW) {
            const uint32_t *src = reinterpret_cast<const uint32_t *>(phases + p);
            uint32_t *dst = reinterpret_cast<uint32_t *>(&sa);
            for (int i = tid; i < static_cast<int>(sizeof(QmmArgs) / 4); i += CONS_THREADS) dst[i] = src[i];
            named_bar_sync(BAR_CONS, CONS_THREADS);
        }
        bool stop = false, pre = false;
        if (tid == 0) {
            const int s0 = first_split_early(sa);  // walked while the other CTAs finish phase p - 1
            if (p > 0) {  // grid barrier: every CTA finished phase p - 1
                const uint32_t target = static_cast<uint32_t>(p) * gridDim.x;
                const uint64_t t0 = gtimer_ns();
                while (ld_acquire(barrier_ctr) < target) {
                    if (cs.abort || gtimer_ns() - t0 > WAIT_NS) {
                        set_status(status, SD_ETIMEOUT);
                        stop = true;
                        break;
                    }
                }
            }
            if (!stop) pre = issue_first_split(sa, sm, act_it, cs, s0);
            if (trace) tslot(p)[TR_START] = gtimer_ns();
        }
        if (bar_any(BAR_WORK, WORK_THREADS, stop)) {
            cs.abort = 1;
            return;
        }
        bool ok = true;
        if (sa.kind == KIND_NORM) {
            if (warp < NCW) norm_phase<KQ>(sa);
        } else if (sa.kind == KIND_ACCEPT) {
            if (blockIdx.x == 0) {  // the deferred fold (one warp per position), then the acceptance
                if (sa.defer_stats) {
                    for (int m = warp < NCW ? warp : warp - 1; m < sa.M; m += NCW + NF) head_final_fold_one(sa, m, lane);
                    named_bar_sync(BAR_WORK, WORK_THREADS);
                }
                if (SAMPLE && sa.accept_mode == 1) {
                    if constexpr (SAMPLE) {
                        if (sa.top_k > 0) pass_topk_accept(sa, sm.ring, (warp < NCW ? warp : warp - 1) * 32 + lane);
                        else pass_sample_accept(sa, sm.ring, (warp < NCW ? warp : warp - 1) * 32 + lane);
                    }
                } else if (tid == 0) {
                    greedy_accept(sa.argmax, sa.tokens, sa.parent, sa.M, sa.out_tokens, sa.out_count);
                }
            }
        } else if (sa.kind == KIND_COMBINE) {
            combine_phase<KQ>(sa, warp < NCW ? warp : warp - 1);
        } else if (sa.kind == KIND_HSTATS) {  // (tile, position) items over every work warp of the grid
            constexpr int NWW = NCW + NF;
            const int n_items = sa.n_stiles * sa.M;
            for (int i = (warp < NCW ? warp : warp - 1) * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x);
                 i < n_items; i += static_cast<int>(gridDim.x) * NWW)
                head_tile_stats_one(sa, i / sa.M, i % sa.M, lane);
        } else if (warp >= FIN_WARP0) {
            const int f = warp - FIN_WARP0;
            ok = sa.pair ? finish_phase<1, NT, KQ>(sa, sm, pk, fin_it, cs, f) : finish_phase<0, NT, KQ>(sa, sm, pk, fin_it, cs, f);
        } else if (KQ && sa.qt == SD_Q4_K && sa.pair) {
            if constexpr (KQ) ok = consume_phase<SD_Q4_K, 1, NT>(sa, sm, it, pk, act_it, nrm_it, cs, pre, tslot(p));
        } else if (KQ && sa.qt == SD_Q4_K) {
            if constexpr (KQ) ok = consume_phase<SD_Q4_K, 0, NT>(sa, sm, it, pk, act_it, nrm_it, cs, pre, tslot(p));
        } else if (KQ && sa.qt == SD_Q6_K) {
            if constexpr (KQ) ok = consume_phase<SD_Q6_K, 0, NT>(sa, sm, it, pk, act_it, nrm_it, cs, pre, tslot(p));
        } else if (!KQ && sa.qt == SD_Q4_32 && sa.pair) {
            if constexpr (!KQ) ok = consume_phase<SD_Q4_32, 1, NT>(sa, sm, it, pk, act_it, nrm_it, cs, pre, tslot(p));
        } else if (!KQ && sa.qt == SD_Q4_32) {
            if constexpr (!KQ) ok = consume_phase<SD_Q4_32, 0, NT>(sa, sm, it, pk, act_it, nrm_it, cs, pre, tslot(p));
        } else {
            ok = consume_phase<SD_Q8_0, 0, NT>(sa, sm, it, pk, act_it, nrm_it, cs, pre, tslot(p));
        }
        // every write of phase p (consumers and finishers) before thread 0's release
        if (bar_any(BAR_WORK, WORK_THREADS, !ok)) {
            cs.abort = 1;
            return;
        }
        if (tid == 0) {
            if (trace) tslot(p)[TR_END] = gtimer_ns();
            red_release_add(barrier_ctr, 1u);
        }
    }
}

// One cooperative launch of a pass kernel: every CTA resident at once, or the launch fails.
inline cudaError_t pass_launch_kernel(void (*k)(const QmmArgs *, int, uint32_t *, uint64_t *), const QmmArgs *phases,
                                      int n_phases, uint32_t *ctr, uint64_t *trace, size_t smem, int grid,
                                      cudaStream_t s) {
    cudaError_t e = allow_max_dynamic_smem(k);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(ctr, 0, sizeof(uint32_t), s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(QMM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, phases, n_phases, ctr, trace);
}

// the sampling instantiations, compiled in their own translation unit (sdv_pass_sample.cu)
cudaError_t pass_launch_sampling(const QmmArgs *phases, int n_phases, uint32_t *ctr, uint64_t *trace, int nt,
                                 size_t smem, int grid, cudaStream_t s);
// the K-quant instantiations (greedy acceptance), in sdv_pass_kq.cu
cudaError_t pass_launch_kq(const QmmArgs *phases, int n_phases, uint32_t *ctr, uint64_t *trace, int nt, size_t smem,
                           int grid, cudaStream_t s);

// ---------------------------------------------------------------------------
// host side: plan + launch
// ---------------------------------------------------------------------------
struct QmmPlan {
    int32_t KB, NU, KS, KBs, KBlast, G, P, D, R, SB, NS, NRB, rows_p, GR, GRS;
    int64_t W;
    uint32_t step_bytes;
    size_t ws_part, ws_cnt, ws_stats, ws_act, ws_total;
};

// Workspace bytes per k block of the activation fragments and {corr, d_a} records a single-operation
// call forms (the largest over M = 1..16).
inline size_t af_ws_bytes_per_block(int qtype) {
    size_t mx = 0;
    for (int M = 1; M <= 16; ++M) {
        const size_t b = af_frag_bytes(M) + af_meta_bytes_q(M, qtype);
        mx = b > mx ? b : mx;
    }
    return mx;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool make_plan(int qtype, int64_t n_out, int64_t k_in, bool pair, bool head, int sms, QmmPlan &p) {
    if (k_in <= 0 || k_in % 32 || n_out <= 0) return false;
    const int GR = is_kq(qtype) ? 8 : 1;  // K-quants: pieces never split a 256-weight super-block
    if (GR > 1 && (k_in % 256 || n_out % 32)) return false;
    const int rec = step_bytes_q(qtype);
    p.GR = GR;
    p.GRS = GR == 8 ? 3 : 0;
    p.KB = static_cast<int32_t>(k_in / 32);
    if (pair) {
        if (n_out % 64) return false;
        p.NU = static_cast<int32_t>(n_out / 64);
    } else {
        p.NU = static_cast<int32_t>((n_out + 31) / 32);
    }
    p.KS = (p.KB + KB_SPLIT_MAX - 1) / KB_SPLIT_MAX;
    p.KBs = ((p.KB + p.KS - 1) / p.KS + GR - 1) / GR * GR;
    p.KS = (p.KB + p.KBs - 1) / p.KBs;
    p.KBlast = p.KB - p.KBs * (p.KS - 1);
    p.W = static_cast<int64_t>(p.NU) * (static_cast<int64_t>(p.KBs) * (p.KS - 1) + p.KBlast);
    p.G = static_cast<int32_t>(p.W / GR < sms ? p.W / GR : sms);
    // whole units per CTA when there is one split and at least one unit per CTA; the rest shared
    p.D = (p.KS == 1 && p.NU >= p.G) ? p.NU / p.G : 0;
    p.R = p.D > 0 ? p.NU - p.D * p.G : 0;
    const int64_t wseq = p.D > 0 ? static_cast<int64_t>(p.R) * p.KB : p.W;
    const int64_t qmin = wseq / GR / p.G * GR;  // the shortest run, a whole number of granules
    int64_t P = qmin > 0 ? (static_cast<int64_t>(p.KBs) - 1) / qmin + 2 : p.KBs / GR;
    if (P > p.KBs / GR) P = p.KBs / GR;
    p.P = static_cast<int32_t>(P);
    const int64_t shared_units = p.D > 0 ? p.R : p.NU;  // units that may need partial sums
    p.step_bytes = static_cast<uint32_t>(rec * (pair ? 2 : 1));
    p.SB = 0;
    p.NS = 0;
    p.NRB = 0;
    p.rows_p = 0;
    const int rows = pair ? 64 : 32;
    // counters first, at fixed offsets shared by every call: units [0, WS_UNIT_CNT), statistics
    // tiles [WS_UNIT_CNT, WS_UNIT_CNT + WS_STAT_CNT), the statistics "done" counter after them.
    // Each call returns the counters it used to zero, so a workspace can serve calls of any shape.
    if (p.NU > WS_UNIT_CNT) return false;
    const int64_t nst = (n_out + STAT_TILE - 1) / STAT_TILE;
    if (head && nst > WS_STAT_CNT) return false;
    p.ws_cnt = WS_CNT_BYTES;
    p.ws_part = align_up(static_cast<size_t>(shared_units) * p.KS * p.P * rows * MPAD * sizeof(float), 256);
    p.ws_stats = head ? align_up(static_cast<size_t>(nst) * MPAD * sizeof(float4), 256) : 0;
    p.ws_act = align_up(static_cast<size_t>(p.KB) * af_ws_bytes_per_block(qtype), 256);
    p.ws_total = p.ws_part + p.ws_cnt + p.ws_stats + p.ws_act;
    return true;
}

// steps per stage (~36 KB stages, one mbarrier wait per 64 records): 64 records of 4-bit, 32
// gate|up pairs, 32 Q8_0 records.  The consumers take a stage in sub-steps of sub_steps().
inline int stage_steps(int qtype, bool pair) {
    if (qtype == SD_Q6_K) return 4 * NCW;  // 4 super-records, 26.9 KB
    return pair ? 4 * NCW : (qtype == SD_Q8_0 ? 4 * NCW : 8 * NCW);
}

struct SmemLayout {
    int NS, NRB, rows_p;
    uint32_t off_ring, off_act, off_meta, off_red, off_ss;
    size_t total;
};


// Shared memory for splits of up to `kbs` blocks, M positions, `rows` output rows per unit (64
// with a gate|up pair), ring slots of `slot` bytes and `ss` bytes of block sums of squares.
// Returns false when not even two ring stages fit.
inline bool layout_smem(int kbs, int M, int rows, size_t slot, size_t ss, SmemLayout &L, int meta_qt = SD_Q4_32) {
    const size_t act = static_cast<size_t>(kbs) * af_frag_bytes(M);
    const size_t meta = static_cast<size_t>(kbs) * af_meta_bytes_q(M, meta_qt);
    L.rows_p = rows + 4;
    L.NRB = M <= 8 ? 2 : 1;
    const size_t red = static_cast<size_t>(L.NRB) * NCW * M * L.rows_p * sizeof(float);
    const size_t fixed = HDR_BYTES + act + meta + red + ss + 4 * 128;
    const size_t budget = 222 * 1024;
    if (fixed + 2 * slot > budget) return false;
    int ns = static_cast<int>((budget - fixed) / slot);
    if (ns > MAX_NS) ns = MAX_NS;
    L.NS = ns;
    L.off_ring = HDR_BYTES;
    L.off_act = static_cast<uint32_t>(align_up(L.off_ring + ns * slot, 128));
    L.off_meta = static_cast<uint32_t>(align_up(L.off_act + act, 128));
    L.off_red = static_cast<uint32_t>(align_up(L.off_meta + meta, 128));
    L.off_ss = static_cast<uint32_t>(align_up(L.off_red + red, 128));
    L.total = align_up(L.off_ss + ss, 128);
    return true;
}

inline void apply_layout(QmmArgs &a, const SmemLayout &L, size_t slot) {
    a.NS = L.NS;
    a.NRB = L.NRB;
    a.rows_p = L.rows_p;
    a.off_ring = L.off_ring;
    a.off_act = L.off_act;
    a.off_meta = L.off_meta;
    a.off_red = L.off_red;
    a.off_ss = L.off_ss;
    a.stage_stride = static_cast<uint32_t>(slot);
}

template <int QT, int PAIR, int NT>
cudaError_t qmm_launch(QmmArgs a, size_t smem, cudaStream_t s) {
    auto k = qmm_kernel<QT, PAIR, NT>;
    cudaError_t e = allow_max_dynamic_smem(k);
    if (e != cudaSuccess) return e;
    return launch(k, dim3(a.G), dim3(QMM_THREADS), smem, s, a);
}

// Lays out shared memory for one single-operation call and launches it (one 8-position tile
// for M <= 8, two above).  Returns cudaErrorInvalidValue when the layout does not fit.
template <int QT, int PAIR>
cudaError_t qmm_dispatch(QmmArgs a, QmmPlan &p, cudaStream_t s) {  // instantiated in sdv_qmm_q4*.cu, sdv_qmm_q8.cu
    p.SB = stage_steps(QT, PAIR != 0);
    const size_t slot = static_cast<size_t>(p.SB) * p.step_bytes;
    SmemLayout L;
    if (!layout_smem(p.KBs, a.M, PAIR ? 64 : 32, slot, 0, L, QT)) return cudaErrorInvalidValue;
    a.SB = p.SB;
    apply_layout(a, L, slot);
    a.kind = KIND_MATMUL;
    a.qt = QT;
    a.pair = PAIR;
    if (a.af_build) {
        const int64_t items = static_cast<int64_t>(a.KB) * (4 * a.M + 8 * af_nt(a.M));
        const int64_t blocks = (items + 255) / 256;
        const cudaError_t e = launch(act_frag_kernel<QT>, dim3(static_cast<unsigned>(blocks < 1024 ? blocks : 1024)),
                                     dim3(256), 0, s, a);
        if (e != cudaSuccess) return e;
    }
    // several k-splits (no gate|up pairing, not the head): the partial sums are added by a second launch
    // spread over the grid rather than by the last split to finish each unit, whose fixups would run
    // one after another on the finisher warps
    a.defer = (!PAIR && !a.head && a.KS > 1) ? 1 : 0;
    cudaError_t e = af_nt(a.M) == 1 ? qmm_launch<QT, PAIR, 1>(a, L.total, s) : qmm_launch<QT, PAIR, 2>(a, L.total, s);
    if (e == cudaSuccess && a.defer) e = launch(qmm_combine_kernel, dim3(a.G), dim3(WORK_THREADS), 0, s, a);
    return e;
}

extern template cudaError_t qmm_dispatch<SD_Q4_32, 0>(QmmArgs, QmmPlan &, cudaStream_t);
extern template cudaError_t qmm_dispatch<SD_Q4_32, 1>(QmmArgs, QmmPlan &, cudaStream_t);
extern template cudaError_t qmm_dispatch<SD_Q8_0, 0>(QmmArgs, QmmPlan &, cudaStream_t);
extern template cudaError_t qmm_dispatch<SD_Q4_K, 0>(QmmArgs, QmmPlan &, cudaStream_t);
extern template cudaError_t qmm_dispatch<SD_Q4_K, 1>(QmmArgs, QmmPlan &, cudaStream_t);
extern template cudaError_t qmm_dispatch<SD_Q6_K, 0>(QmmArgs, QmmPlan &, cudaStream_t);

}  // namespace sdv
