"""CPU oracle for the speculative-decoding verify pass -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may
import this package.  The product path (``speculative_decoding_verify_gb300``)
never does, and shares no code with it.

Every function is a thin numpy wrapper over ``sdv_oracle.c`` (plain C, built with
``-O2 -ffp-contract=off``, OpenMP over output rows only).  Each one follows the
page passage cited in the C source:

* block dequant / integer block dots / multi-position matmul (fp64 accumulate):
  "Inside OpenJet Engine", section "One GPU launch for a speculative cycle";
* RMSNorm + per-32 int8 requantisation, SiLU*mul requantisation: same section
  (the producer requantises activations for the next consumer);
* softmax statistics, greedy chain/tree acceptance: "How Kinetic is fast",
  sections "RAD-1" and "Why the output does not change";
* rejection sampling and the certainty drafter: "Speculative Decoding with
  Open-Weights Models", section "Mathematical Integrity: Rejection Sampling for
  LLMs", and "How Kinetic is fast", section "Why the output does not change";
* the same against a top-k / top-p filtered target (the sampling knobs of
  "Inside OpenJet Engine", API section; the filtering order is a reading);
* Philox4x32-10: Salmon et al., SC'11;
* the 4-bit shortlist copy and its exact argmax: "How Kinetic is fast",
  section "Shortlist";
* decode attention over the K+1 positions with a tree mask, the fp16 KV append
  and the in-place commit of the accepted path: "Inside OpenJet Engine",
  section "Cheap drafting, careful state management"; "How Kinetic is fast",
  section "Where the guesses come from"; "Speculative Decoding with
  Open-Weights Models", section "Engineering the Architecture: KV Cache
  Synchronization";
* the adaptive draft depth: "Inside OpenJet Engine", section "Cheap drafting,
  careful state management", and "How Kinetic is fast", section "Where the
  guesses come from";
* Q4_K / Q6_K super-blocks and their matmul: the GGUF K-quant formats the
  pages' model files use (no page prints a block).

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_pins.py`` against something other than itself.  The
free-running 64-layer stack composition (``stack_pass``) is pinned only through
its stages; its end-to-end float output is "parity unpinned".  The K-quant
decoders are pinned to their stated layout, but their agreement with real GGUF
files is "parity unpinned" (no model file is available).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsdv_oracle.so")
_lock = threading.Lock()
_lib = None

Q8_0 = 0
Q4_32 = 1
BLOCK_BYTES = {Q8_0: 34, Q4_32: 18}

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_F = ctypes.c_float


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "sdv_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
                               "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _get():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            sig = {
                "oracle_num_threads": ([], _I),
                "oracle_set_num_threads": ([_I], None),
                "oracle_f16_to_f32": ([ctypes.c_uint16], _F),
                "oracle_dequant": ([_I, _P, _I64, _P], None),
                "oracle_block_dots": ([_I, _P, _I64, _I64, _P, _I, _P], None),
                "oracle_qmatmul": ([_I, _P, _I64, _I64, _P, _P, _I, _P, _P, _P], None),
                "oracle_rmsnorm_quant": ([_P, _P, _F, _I, _I64, _P, _P], None),
                "oracle_cexp": ([_F], _F),
                "oracle_silu_mul_requant": ([_P, _P, _I, _I64, _P, _P, _P], None),
                "oracle_softmax_stats": ([_P, _I, _I64, _F, _P, _P, _P], None),
                "oracle_softmax_probs": ([_P, _I64, _F, _F, _F, _P], None),
                "oracle_accept_greedy_chain": ([_P, _P, _I, _P], _I),
                "oracle_accept_greedy_tree": ([_P, _P, _P, _I, _P], _I),
                "oracle_philox4x32_10": ([_P, _P, _P], None),
                "oracle_uniforms": ([ctypes.c_uint64, _I64, _P, _P], None),
                "oracle_draw_icdf": ([_P, _I64, _F], ctypes.c_int32),
                "oracle_accept_sample_u": ([_P, _I64, _I, _P, _P, _F, _P, _P, _P], _I),
                "oracle_accept_sample": ([_P, _I64, _I, _P, _P, _F, ctypes.c_uint64, _I64, _P], _I),
                "oracle_accept_sample_trials": ([_P, _I64, _I, _P, _P, _F, ctypes.c_uint64, _I64, _I64, _P, _P],
                                                None),
                "oracle_filter_topk_topp": ([_P, _I64, _F, _I, _F, _P, _P], _I),
                "oracle_accept_sample_topk_u": ([_P, _I64, _I, _P, _P, _F, _I, _F, _P, _P, _P], _I),
                "oracle_accept_sample_topk": ([_P, _I64, _I, _P, _P, _F, _I, _F, ctypes.c_uint64, _I64, _P], _I),
                "oracle_shortlist_copy": ([_P, _I64, _I64, _P, _P, _P], None),
                "oracle_f32_to_f16": ([_P, _I64, _P], None),
                "oracle_kq_block_bytes": ([_I], _I),
                "oracle_accept_greedy_tree_path": ([_P, _P, _P, _I, _P], _I),
                "oracle_kq_dequant": ([_I, _P, _I64, _P], None),
                "oracle_kq_matmul": ([_I, _P, _I64, _I64, _P, _P, _I, _P, _P], None),
                "oracle_kv_append": ([_P, _P, _I, _I, _I, _P, _P, _I64, _I64], None),
                "oracle_attn_decode": ([_P, _P, _P, _I, _I, _I, _I, _I64, _I64, _P, _P], None),
                "oracle_kv_commit": ([_P, _P, _I, _I, _I64, _I64, _P, _I], None),
                "oracle_shortlist_argmax": ([_P, _P, _P, _I64, _I64, _P, _P, _I, _P, _P], None),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


def num_threads() -> int:
    return _get().oracle_num_threads()


def set_num_threads(n: int):
    """Threads of the calls that follow (for timing on one core); results do not depend on it."""
    _get().oracle_set_num_threads(int(n))


def f16_to_f32(bits: int) -> float:
    return float(_get().oracle_f16_to_f32(bits))


def dequant(qtype: int, blocks: np.ndarray, n_out: int, k_in: int) -> np.ndarray:
    blocks, p = _c(blocks, np.uint8)
    assert blocks.size == n_out * (k_in // 32) * BLOCK_BYTES[qtype]
    out = np.empty((n_out, k_in), dtype=np.float32)
    _get().oracle_dequant(qtype, p, n_out * (k_in // 32), out.ctypes.data)
    return out


def block_dots(qtype: int, w: np.ndarray, n_out: int, k_in: int, q: np.ndarray) -> np.ndarray:
    w, pw = _c(w, np.uint8)
    q, pq = _c(q, np.int8)
    M = q.shape[0]
    out = np.empty((M, n_out, k_in // 32), dtype=np.int32)
    _get().oracle_block_dots(qtype, pw, n_out, k_in, pq, M, out.ctypes.data)
    return out


def qmatmul(qtype: int, w: np.ndarray, n_out: int, k_in: int, q: np.ndarray, scales: np.ndarray,
            residual: np.ndarray | None = None):
    """Returns (y fp32 [M][n_out], absbound fp64 [M][n_out])."""
    w, pw = _c(w, np.uint8)
    q, pq = _c(q, np.int8)
    scales, ps = _c(scales, np.float32)
    M = q.shape[0]
    assert q.shape == (M, k_in) and scales.shape == (M, k_in // 32)
    pr = None
    if residual is not None:
        residual, pr = _c(residual, np.float32)
        assert residual.shape == (M, n_out)
    y = np.empty((M, n_out), dtype=np.float32)
    ab = np.empty((M, n_out), dtype=np.float64)
    _get().oracle_qmatmul(qtype, pw, n_out, k_in, pq, ps, M, pr, y.ctypes.data, ab.ctypes.data)
    return y, ab


def rmsnorm_quant(x: np.ndarray, norm_w: np.ndarray | None, eps: float = 1e-6):
    """Returns (q int8 [M][K], scales fp32 [M][K/32]); norm_w None = requantise only."""
    x, px = _c(x, np.float32)
    M, K = x.shape
    pw = None
    if norm_w is not None:
        norm_w, pw = _c(norm_w, np.float32)
    q = np.empty((M, K), dtype=np.int8)
    s = np.empty((M, K // 32), dtype=np.float32)
    _get().oracle_rmsnorm_quant(px, pw, eps, M, K, q.ctypes.data, s.ctypes.data)
    return q, s


def cexp(x) -> np.ndarray:
    f = _get().oracle_cexp
    x = np.asarray(x, dtype=np.float32)
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.float32).reshape(x.shape)


def silu_mul_requant(g: np.ndarray, u: np.ndarray):
    """Returns (q int8 [M][F], scales fp32 [M][F/32], h fp32 [M][F])."""
    g, pg = _c(g, np.float32)
    u, pu = _c(u, np.float32)
    M, F = g.shape
    q = np.empty((M, F), dtype=np.int8)
    s = np.empty((M, F // 32), dtype=np.float32)
    h = np.empty((M, F), dtype=np.float32)
    _get().oracle_silu_mul_requant(pg, pu, M, F, q.ctypes.data, s.ctypes.data, h.ctypes.data)
    return q, s, h


def softmax_stats(logits: np.ndarray, T: float = 1.0):
    """Returns (row_max [M], row_sumexp [M], argmax [M])."""
    logits, pl = _c(logits, np.float32)
    M, V = logits.shape
    m = np.empty(M, dtype=np.float32)
    z = np.empty(M, dtype=np.float32)
    a = np.empty(M, dtype=np.int32)
    _get().oracle_softmax_stats(pl, M, V, T, m.ctypes.data, z.ctypes.data, a.ctypes.data)
    return m, z, a


def softmax_probs(logits_row: np.ndarray, T: float = 1.0) -> np.ndarray:
    l, pl = _c(logits_row.reshape(1, -1), np.float32)
    m, z, _ = softmax_stats(l, T)
    p = np.empty(l.shape[1], dtype=np.float32)
    _get().oracle_softmax_probs(pl, l.shape[1], T, float(m[0]), float(z[0]), p.ctypes.data)
    return p


def accept_greedy_chain(argmax: np.ndarray, drafts: np.ndarray) -> np.ndarray:
    argmax, pa = _c(argmax, np.int32)
    drafts, pd = _c(drafts, np.int32)
    K = drafts.size
    assert argmax.size == K + 1
    out = np.empty(K + 1, dtype=np.int32)
    n = _get().oracle_accept_greedy_chain(pa, pd, K, out.ctypes.data)
    return out[:n].copy()


def accept_greedy_tree(argmax: np.ndarray, tokens: np.ndarray, parent: np.ndarray) -> np.ndarray:
    argmax, pa = _c(argmax, np.int32)
    tokens, pt = _c(tokens, np.int32)
    parent, pp = _c(parent, np.int32)
    M = tokens.size
    out = np.empty(M, dtype=np.int32)
    n = _get().oracle_accept_greedy_tree(pa, pt, pp, M, out.ctypes.data)
    return out[:n].copy()


def accept_greedy_tree_path(argmax: np.ndarray, tokens: np.ndarray, parent: np.ndarray) -> np.ndarray:
    """Node indices of the accepted path (root first) under the greedy tree rule."""
    argmax, pa = _c(argmax, np.int32)
    tokens, pt = _c(tokens, np.int32)
    parent, pp = _c(parent, np.int32)
    M = tokens.size
    out = np.empty(M, dtype=np.int32)
    n = _get().oracle_accept_greedy_tree_path(pa, pt, pp, M, out.ctypes.data)
    return out[:n].copy()


def philox4x32_10(ctr, key) -> np.ndarray:
    c, pc = _c(np.array(ctr, dtype=np.uint32), np.uint32)
    k, pk = _c(np.array(key, dtype=np.uint32), np.uint32)
    out = np.empty(4, dtype=np.uint32)
    _get().oracle_philox4x32_10(pc, pk, out.ctypes.data)
    return out


def uniforms(seed: int, pos: int):
    a = ctypes.c_float()
    r = ctypes.c_float()
    _get().oracle_uniforms(seed, pos, ctypes.byref(a), ctypes.byref(r))
    return a.value, r.value


def draw_icdf(w: np.ndarray, u: float) -> int:
    w, pw = _c(w, np.float32)
    return int(_get().oracle_draw_icdf(pw, w.size, u))


def accept_sample_u(logits, q_probs, drafts, T, u_acc, u_res) -> np.ndarray:
    logits, pl = _c(logits, np.float32)
    K1, V = logits.shape
    K = K1 - 1
    pq = None
    if q_probs is not None:
        q_probs, pq = _c(q_probs, np.float32)
        assert q_probs.shape == (K, V)
    drafts, pd = _c(drafts, np.int32)
    ua, pua = _c(u_acc, np.float32)
    ur, pur = _c(u_res, np.float32)
    out = np.empty(K + 1, dtype=np.int32)
    n = _get().oracle_accept_sample_u(pl, V, K, pq, pd, T, pua, pur, out.ctypes.data)
    return out[:n].copy()


def accept_sample(logits, q_probs, drafts, T: float, seed: int, base_pos: int) -> np.ndarray:
    logits, pl = _c(logits, np.float32)
    K1, V = logits.shape
    K = K1 - 1
    pq = None
    if q_probs is not None:
        q_probs, pq = _c(q_probs, np.float32)
        assert q_probs.shape == (K, V)
    drafts, pd = _c(drafts, np.int32)
    out = np.empty(K + 1, dtype=np.int32)
    n = _get().oracle_accept_sample(pl, V, K, pq, pd, T, seed, base_pos, out.ctypes.data)
    return out[:n].copy()


def filter_topk_topp(logits_row, T: float, top_k: int, top_p: float):
    """The filtered target of one row: (tokens, probabilities) of the nucleus in candidate order."""
    l, pl = _c(np.asarray(logits_row).reshape(-1), np.float32)
    tok = np.empty(64, dtype=np.int32)
    prob = np.empty(64, dtype=np.float32)
    n = _get().oracle_filter_topk_topp(pl, l.size, T, top_k, top_p, tok.ctypes.data, prob.ctypes.data)
    return tok[:n].copy(), prob[:n].copy()


def accept_sample_topk_u(logits, q_probs, drafts, T, top_k, top_p, u_acc, u_res) -> np.ndarray:
    logits, pl = _c(logits, np.float32)
    K1, V = logits.shape
    K = K1 - 1
    pq = None
    if q_probs is not None:
        q_probs, pq = _c(q_probs, np.float32)
        assert q_probs.shape == (K, V)
    drafts, pd = _c(drafts, np.int32)
    ua, pua = _c(u_acc, np.float32)
    ur, pur = _c(u_res, np.float32)
    out = np.empty(K + 1, dtype=np.int32)
    n = _get().oracle_accept_sample_topk_u(pl, V, K, pq, pd, T, top_k, top_p, pua, pur, out.ctypes.data)
    return out[:n].copy()


def accept_sample_topk(logits, q_probs, drafts, T: float, top_k: int, top_p: float, seed: int,
                       base_pos: int) -> np.ndarray:
    logits, pl = _c(logits, np.float32)
    K1, V = logits.shape
    K = K1 - 1
    pq = None
    if q_probs is not None:
        q_probs, pq = _c(q_probs, np.float32)
        assert q_probs.shape == (K, V)
    drafts, pd = _c(drafts, np.int32)
    out = np.empty(K + 1, dtype=np.int32)
    n = _get().oracle_accept_sample_topk(pl, V, K, pq, pd, T, top_k, top_p, seed, base_pos, out.ctypes.data)
    assert n > 0
    return out[:n].copy()


def shortlist_copy(q8_blocks, N: int, K: int):
    """4-bit copy of a Q8_0 matrix with its row error bounds and row norms: (q4 blocks, bound, wnorm)."""
    w, pw = _c(np.asarray(q8_blocks).reshape(-1), np.uint8)
    q4 = np.zeros(N * (K // 32) * 18, dtype=np.uint8)
    bound = np.empty(N, dtype=np.float32)
    wnorm = np.empty(N, dtype=np.float32)
    _get().oracle_shortlist_copy(pw, N, K, q4.ctypes.data, bound.ctypes.data, wnorm.ctypes.data)
    return q4, bound, wnorm


def shortlist_argmax(q4_blocks, bound, q8_blocks, N: int, K: int, q, scales):
    """Argmax per position through the shortlist (fp64 scores) and the count of rows scored exactly."""
    w4, p4 = _c(np.asarray(q4_blocks).reshape(-1), np.uint8)
    bd, pb = _c(bound, np.float32)
    w8, p8 = _c(np.asarray(q8_blocks).reshape(-1), np.uint8)
    q, pq = _c(q, np.int8)
    sc, ps = _c(scales, np.float32)
    M = q.shape[0]
    am = np.empty(M, dtype=np.int32)
    nc = np.empty(M, dtype=np.int64)
    _get().oracle_shortlist_argmax(p4, pb, p8, N, K, pq, ps, M, am.ctypes.data, nc.ctypes.data)
    return am, nc


Q4_K, Q6_K = 2, 3   # 256-weight K-quant super-blocks (144 and 210 bytes)


def kq_dequant(qtype: int, blocks, n_out: int, k_in: int) -> np.ndarray:
    """K-quant super-blocks [n_out][k_in/256] -> fp32 [n_out][k_in]."""
    blocks, p = _c(np.asarray(blocks).reshape(-1), np.uint8)
    bb = _get().oracle_kq_block_bytes(qtype)
    assert k_in % 256 == 0 and blocks.size == n_out * (k_in // 256) * bb
    out = np.empty((n_out, k_in), dtype=np.float32)
    _get().oracle_kq_dequant(qtype, p, n_out * (k_in // 256), out.ctypes.data)
    return out


def kq_matmul(qtype: int, blocks, n_out: int, k_in: int, q, scales, with_bound: bool = False):
    """fp64 [M][n_out]: per 32-weight block, the integer dots times the scales (factored form).
    with_bound: also the absolute sum of the same terms [M][n_out] (the tolerance scale, reading R5)."""
    blocks, pw = _c(np.asarray(blocks).reshape(-1), np.uint8)
    q, pq = _c(q, np.int8)
    sc, ps = _c(scales, np.float32)
    M = q.shape[0]
    y = np.empty((M, n_out), dtype=np.float64)
    ab = np.empty((M, n_out), dtype=np.float64)
    _get().oracle_kq_matmul(qtype, pw, n_out, k_in, pq, ps, M, y.ctypes.data, ab.ctypes.data)
    return (y, ab) if with_bound else y


def f32_to_f16(x) -> np.ndarray:
    """fp32 -> fp16 bits (uint16), nearest even."""
    x, px = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _get().oracle_f32_to_f16(px, x.size, out.ctypes.data)
    return out


def kv_append(k_new, v_new, k_cache, v_cache, L: int):
    """Write fp32 [M][H_kv][D] rows into slots [L, L+M) of the fp16-bit caches [H_kv][S_max][D] (in place)."""
    k_new, pk = _c(k_new, np.float32)
    v_new, pv = _c(v_new, np.float32)
    M, H_kv, D = k_new.shape
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    S_max = k_cache.shape[1]
    assert L + M <= S_max
    _get().oracle_kv_append(pk, pv, M, H_kv, D, k_cache.ctypes.data, v_cache.ctypes.data, S_max, L)


def attn_decode(q, k_cache, v_cache, L: int, parent=None) -> np.ndarray:
    """q fp32 [M][H][D]; caches fp16 bits [H_kv][S_max][D] with L committed + M new rows.  fp64 [M][H][D]."""
    q, pq = _c(q, np.float32)
    M, H, D = q.shape
    k_cache, pk = _c(k_cache, np.uint16)
    v_cache, pv = _c(v_cache, np.uint16)
    H_kv, S_max, D2 = k_cache.shape
    assert D2 == D and H % H_kv == 0 and L + M <= S_max
    pp = None
    if parent is not None:
        parent, pp = _c(parent, np.int32)
    out = np.empty((M, H, D), dtype=np.float64)
    _get().oracle_attn_decode(pq, pk, pv, M, H, H_kv, D, S_max, L, pp, out.ctypes.data)
    return out


def kv_commit(k_cache, v_cache, L: int, path):
    """Move the accepted path's rows to slots [L, L+n) (in place)."""
    path, pp = _c(path, np.int32)
    H_kv, S_max, D = k_cache.shape
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    _get().oracle_kv_commit(k_cache.ctypes.data, v_cache.ctypes.data, H_kv, D, S_max, L, pp, path.size)


def accept_sample_trials(logits, q_probs, drafts_per_trial, T: float, seed: int, base_pos: int):
    """Independent repetitions at positions base_pos + t*(K+1).  Returns (counts [n], tokens [n][K+1])."""
    logits, pl = _c(logits, np.float32)
    K1, V = logits.shape
    K = K1 - 1
    pq = None
    if q_probs is not None:
        q_probs, pq = _c(q_probs, np.float32)
    d, pd = _c(drafts_per_trial, np.int32)
    n = d.shape[0]
    counts = np.empty(n, dtype=np.int32)
    toks = np.full((n, K + 1), -1, dtype=np.int32)
    _get().oracle_accept_sample_trials(pl, V, K, pq, pd, T, seed, base_pos, n, counts.ctypes.data,
                                       toks.ctypes.data)
    return counts, toks


# ---------------------------------------------------------------------------
# Composition of the 27B-shaped projection stack (attention omitted).
# Per layer: RMSNorm -> requant -> QKV; O takes the requantised V slice (the
# output of attention whose only key is the token itself); residual add after
# O and after down; RMSNorm -> gate|up -> SiLU*mul -> requant -> down.  A final
# RMSNorm feeds the vocabulary head.
# ---------------------------------------------------------------------------

def stack_layer(h: np.ndarray, wts: dict, norm1: np.ndarray, norm2: np.ndarray, hidden: int, ffn: int,
                wq: int = Q4_32, eps: float = 1e-6, trace: dict | None = None) -> np.ndarray:
    M = h.shape[0]
    q1, s1 = rmsnorm_quant(h, norm1, eps)
    qkv, _ = qmatmul(wq, wts["qkv"], 3 * hidden, hidden, q1, s1)
    qv, sv = rmsnorm_quant(np.ascontiguousarray(qkv[:, 2 * hidden:]), None)
    h2, _ = qmatmul(wq, wts["o"], hidden, hidden, qv, sv, residual=h)
    q3, s3 = rmsnorm_quant(h2, norm2, eps)
    gu, _ = qmatmul(wq, wts["gate_up"], 2 * ffn, hidden, q3, s3)
    q4, s4, _ = silu_mul_requant(np.ascontiguousarray(gu[:, :ffn]), np.ascontiguousarray(gu[:, ffn:]))
    h3, _ = qmatmul(wq, wts["down"], hidden, ffn, q4, s4, residual=h2)
    if trace is not None:
        trace.update(q1=q1, s1=s1, qkv=qkv, qv=qv, sv=sv, h2=h2, q3=q3, s3=s3, gu=gu, q4=q4, s4=s4, h3=h3)
    return h3


def head(h: np.ndarray, final_norm: np.ndarray, head_w: np.ndarray, vocab: int, hidden: int, T: float = 1.0,
         eps: float = 1e-6, head_q: int = Q8_0):
    """Returns (logits, argmax, row_max, row_sumexp)."""
    q, s = rmsnorm_quant(h, final_norm, eps)
    logits, _ = qmatmul(head_q, head_w, vocab, hidden, q, s)
    m, z, a = softmax_stats(logits, T)
    return logits, a, m, z


# ---------------------------------------------------------------------------
# adaptive draft depth (plain Python: a few integers per cycle)
# ---------------------------------------------------------------------------

def depth_policy(k_max: int, max_pause: int, cycles):
    """Drafts per cycle under the adaptive-depth reading: "Inside OpenJet Engine", section "Cheap
    drafting, careful state management" (a configured depth is cut by one for the cycle after a
    rejection) and "How Kinetic is fast", section "Where the guesses come from" (draft length
    follows recent drafts; after drafts that miss outright, drafting pauses for longer and
    longer).

    cycles: the accepted-draft count of each cycle, in order (ignored for a cycle that drafted
    nothing).  Returns the depth used by each cycle, starting at k_max:
      all drafts accepted        -> next depth k_max, miss count 0
      some but not all accepted  -> next depth max(1, k_max - 1), miss count 0
      none accepted (a miss)     -> miss count + 1, then min(max_pause, 2^(misses - 1)) cycles
                                    without drafts (none if max_pause is 0), then depth
                                    max(1, k_max - 1)
    """
    reduced = max(1, k_max - 1)
    k, pause, misses = k_max, 0, 0
    used = []
    for acc in cycles:
        used.append(k)
        if k == 0:
            pause = max(0, pause - 1)
            k = 0 if pause > 0 else reduced
        elif acc == k:
            misses, k = 0, k_max
        elif acc > 0:
            misses, k = 0, reduced
        else:
            misses = min(misses + 1, 31)
            pause = min(max_pause, 2 ** (misses - 1))
            k = 0 if pause > 0 else reduced
    return used
