"""GB300 (sm_103a) speculative-decoding verify pass: thin Python binding.

Every function marshals torch tensors (device memory owned by the caller) into
the C ABI of ``libsdverify.so`` (declared in ``include/sdverify.h``) and calls
it on the current CUDA stream.  All arithmetic runs in the library's kernels;
there is no CPU or PyTorch fallback: if the library is missing, ``lib()``
raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# SDV_DEBUG_BOUNDS=1 selects the bounds-checked build of the same sources (build.build(debug_bounds=True))
DEBUG_BOUNDS = os.environ.get("SDV_DEBUG_BOUNDS", "") == "1"
LIB_PATH = os.path.join(HERE, "libsdverify_dbg.so" if DEBUG_BOUNDS else "libsdverify.so")

Q8_0 = 0
Q4_32 = 1
Q4_K = 2
Q6_K = 3
BLOCK_BYTES = {Q8_0: 34, Q4_32: 18}
SUPER_BLOCK_BYTES = {Q4_K: 144, Q6_K: 210}  # K-quant super-blocks of 256 weights
REPACK_PAIR_GATE_UP = 1
EPI_NONE = 0
EPI_REQUANT = 1
EPI_SILU_MUL_REQUANT = 2

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "device wait timed out",
          5: "device-side check failed"}

_lib = None


class SdLayer(ctypes.Structure):
    _fields_ = [("qkv", ctypes.c_void_p), ("o", ctypes.c_void_p), ("gate_up", ctypes.c_void_p),
                ("down", ctypes.c_void_p), ("norm1", ctypes.c_void_p), ("norm2", ctypes.c_void_p)]


class SdPassDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int64), ("ffn", ctypes.c_int64),
                ("vocab", ctypes.c_int64), ("M", ctypes.c_int32), ("wq", ctypes.c_int32), ("eps", ctypes.c_float),
                ("temperature", ctypes.c_float), ("layers", ctypes.POINTER(SdLayer)),
                ("final_norm", ctypes.c_void_p), ("head", ctypes.c_void_p), ("h", ctypes.c_void_p),
                ("qa", ctypes.c_void_p), ("sa", ctypes.c_void_p), ("qv", ctypes.c_void_p), ("sv", ctypes.c_void_p),
                ("qf", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("logits", ctypes.c_void_p),
                ("argmax", ctypes.c_void_p), ("row_max", ctypes.c_void_p), ("row_sumexp", ctypes.c_void_p),
                ("tokens", ctypes.c_void_p), ("parent", ctypes.c_void_p), ("out_tokens", ctypes.c_void_p),
                ("out_count", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("ws_bytes", ctypes.c_size_t),
                ("accept", ctypes.c_int32), ("q_probs", ctypes.c_void_p), ("seed", ctypes.c_uint64),
                ("base_pos", ctypes.c_int64), ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float),
                ("wq_down", ctypes.c_int32)]

ACCEPT_GREEDY, ACCEPT_SAMPLE = 0, 1


class SdPass(ctypes.Structure):
    _fields_ = [("plan", ctypes.c_void_p), ("n_phases", ctypes.c_int32), ("nt", ctypes.c_int32),
                ("smem_bytes", ctypes.c_uint32), ("grid", ctypes.c_int32), ("accept", ctypes.c_int32),
                ("kq", ctypes.c_int32)]


class SdDepthState(ctypes.Structure):
    _fields_ = [("k_max", ctypes.c_int32), ("max_pause", ctypes.c_int32), ("k_next", ctypes.c_int32),
                ("pause_left", ctypes.c_int32), ("misses", ctypes.c_int32)]


class SdError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({code})")
        self.code = code


def lib():
    """Load libsdverify.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with speculative_decoding_verify_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I, I32, I64, U32, U64, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int32, ctypes.c_int64,
                                           ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t)
        sig = {
            "sd_status_string": ([I], ctypes.c_char_p),
            "sd_abi_version": ([], I),
            "sd_repacked_bytes": ([I, I64, I64, U32], SZ),
            "sd_repack_weights": ([I, P, I64, I64, U32, P, SZ, P], I),
            "sd_rmsnorm_quant_acts": ([P, I64, P, F, I32, I64, P, P, P], I),
            "sd_qmatmul_workspace_bytes": ([I, I64, I64, U32], SZ),
            "sd_qmatmul_multipos": ([I, P, I64, I64, P, P, I32, P, P, U32, I64, P, P, P, SZ, P], I),
            "sd_qmatmul_multipos_noalloc": ([I, P, I64, I64, P, P, I32, P, P, U32, I64, P, P, P], I),
            "sd_head_workspace_bytes": ([I64, I64], SZ),
            "sd_head_logits": ([P, I64, I64, P, P, I32, F, P, P, P, P, P, SZ, P], I),
            "sd_tree_path": ([P, P, P, I32, P], I32),
            "sd_depth_init": ([ctypes.POINTER(SdDepthState), I32, I32], I),
            "sd_depth_update": ([ctypes.POINTER(SdDepthState), I32], I),
            "sd_device_status_site": ([P, ctypes.POINTER(I32)], I),
            "sd_build_flags": ([], I32),
            "sd_attn_workspace_bytes": ([I32, I32, I32, I32, I64], SZ),
            "sd_kv_append": ([P, P, I32, I32, I32, P, P, I64, I64, P], I),
            "sd_attn_decode": ([P, P, P, I32, I32, I32, I32, I64, I64, P, P, P, SZ, P], I),
            "sd_kv_commit": ([P, P, I32, I32, I64, I64, I32, P, P, P], I),
            "sd_shortlist_build": ([P, I64, I64, P, P, P, P], I),
            "sd_shortlist_workspace_bytes": ([I64, I64], SZ),
            "sd_head_shortlist": ([P, P, P, P, I64, I64, P, P, I32, P, P, P, SZ, P], I),
            "sd_accept_greedy": ([P, P, P, I32, P, P, P], I),
            "sd_accept_sample": ([P, I64, I32, P, P, P, P, F, U64, I64, P, P, P], I),
            "sd_accept_sample_topk": ([P, I64, I32, P, P, F, I32, F, U64, I64, P, P, P], I),
            "sd_device_status": ([P], I),
            "sd_set_pdl": ([I], None),
            "sd_debug_block_dots": ([I, P, I64, I64, P, I32, P, P], I),
            "sd_debug_silu_mul_requant": ([P, P, I32, I64, P, P, P], I),
            "sd_debug_cexp": ([P, I64, P, P], I),
            "sd_debug_philox": ([U64, I64, I64, P, P], I),
            "sd_debug_wait_timeout": ([I64, P], I),
            "sd_debug_schedule": ([I, I64, I64, I32, I32, I32, P, P, I64], I64),
            "sd_pass_plan_bytes": ([I32], SZ),
            "sd_pass_workspace_bytes": ([I64, I64, I64, I32], SZ),
            "sd_pass_prepare": ([ctypes.POINTER(SdPassDesc), P, SZ, ctypes.POINTER(SdPass)], I),
            "sd_verify_pass": ([ctypes.POINTER(SdPass), P], I),
            "sd_pass_trace_bytes": ([ctypes.POINTER(SdPass)], ctypes.c_size_t),
            "sd_verify_pass_traced": ([ctypes.POINTER(SdPass), P, ctypes.c_size_t, P], I),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(code: int, what: str):
    if code != 0:
        raise SdError(code, what)


def _dev(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor")


# ---------------------------------------------------------------------------
# verify-pass calls
# ---------------------------------------------------------------------------

def repacked_bytes(qtype: int, n_out: int, k_in: int, pair: bool = False) -> int:
    return int(lib().sd_repacked_bytes(qtype, n_out, k_in, REPACK_PAIR_GATE_UP if pair else 0))


def repack_weights(qtype: int, src: torch.Tensor, n_out: int, k_in: int, pair: bool = False,
                   out: torch.Tensor | None = None) -> torch.Tensor:
    """GGUF-order blocks (uint8 CUDA tensor) -> repacked records (uint8 CUDA tensor)."""
    _dev(src, torch.uint8, "src")
    nb = repacked_bytes(qtype, n_out, k_in, pair)
    if nb == 0:
        raise ValueError("bad repack shape")
    if out is None:
        out = torch.empty(nb, dtype=torch.uint8, device=src.device)
    _check(lib().sd_repack_weights(qtype, _p(src), n_out, k_in, REPACK_PAIR_GATE_UP if pair else 0, _p(out),
                                   out.numel(), _stream()), "sd_repack_weights")
    return out


def rmsnorm_quant_acts(x: torch.Tensor, norm_w: torch.Tensor | None, q: torch.Tensor, scales: torch.Tensor,
                       eps: float = 1e-6, K: int | None = None, ldx: int | None = None):
    M = x.shape[0]
    K = K if K is not None else x.shape[1]
    ldx = ldx if ldx is not None else x.stride(0)
    _check(lib().sd_rmsnorm_quant_acts(_p(x), ldx, _p(norm_w), eps, M, K, _p(q), _p(scales), _stream()),
           "sd_rmsnorm_quant_acts")


def qmatmul_workspace_bytes(qtype: int, n_out: int, k_in: int, epilogue: int = EPI_NONE) -> int:
    return int(lib().sd_qmatmul_workspace_bytes(qtype, n_out, k_in, epilogue))


def head_workspace_bytes(vocab: int, hidden: int) -> int:
    return int(lib().sd_head_workspace_bytes(vocab, hidden))


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """Zero-filled workspace (the calls leave its counters at zero again)."""
    return torch.zeros(max(256, (nbytes + 255) // 256 * 256), dtype=torch.uint8, device=device or "cuda")


def qmatmul_multipos(qtype: int, w: torch.Tensor, n_out: int, k_in: int, q: torch.Tensor, scales: torch.Tensor,
                     ws: torch.Tensor, y: torch.Tensor | None = None, residual: torch.Tensor | None = None,
                     epilogue: int = EPI_NONE, requant_col0: int = 0, q_next: torch.Tensor | None = None,
                     scales_next: torch.Tensor | None = None):
    M = q.shape[0]
    _check(lib().sd_qmatmul_multipos(qtype, _p(w), n_out, k_in, _p(q), _p(scales), M, _p(y), _p(residual), epilogue,
                                     requant_col0, _p(q_next), _p(scales_next), _p(ws), ws.numel(), _stream()),
           "sd_qmatmul_multipos")


def qmatmul_multipos_noalloc(qtype: int, w: torch.Tensor, n_out: int, k_in: int, q: torch.Tensor,
                             scales: torch.Tensor, y: torch.Tensor | None = None, residual: torch.Tensor | None = None,
                             epilogue: int = EPI_NONE, requant_col0: int = 0, q_next: torch.Tensor | None = None,
                             scales_next: torch.Tensor | None = None):
    """sd_qmatmul_multipos with the library's static scratch instead of a workspace (allocates nothing)."""
    M = q.shape[0]
    _check(lib().sd_qmatmul_multipos_noalloc(qtype, _p(w), n_out, k_in, _p(q), _p(scales), M, _p(y), _p(residual),
                                             epilogue, requant_col0, _p(q_next), _p(scales_next), _stream()),
           "sd_qmatmul_multipos_noalloc")


def head_logits(w: torch.Tensor, vocab: int, hidden: int, q: torch.Tensor, scales: torch.Tensor, ws: torch.Tensor,
                logits: torch.Tensor, argmax: torch.Tensor, row_max: torch.Tensor, row_sumexp: torch.Tensor,
                temperature: float = 1.0):
    M = q.shape[0]
    _check(lib().sd_head_logits(_p(w), vocab, hidden, _p(q), _p(scales), M, temperature, _p(logits), _p(argmax),
                                _p(row_max), _p(row_sumexp), _p(ws), ws.numel(), _stream()), "sd_head_logits")


def tree_path(argmax, tokens, parent):
    """Accepted nodes of a greedy draft tree, root first (host int32 arrays in, numpy out)."""
    import numpy as np
    a = np.ascontiguousarray(argmax, dtype=np.int32).reshape(-1)
    t = np.ascontiguousarray(tokens, dtype=np.int32).reshape(-1)
    p = np.ascontiguousarray(parent, dtype=np.int32).reshape(-1)
    # sd_tree_path reads M entries of each array: refuse mismatched lengths before the call
    if not (a.size == t.size == p.size) or not 1 <= t.size <= 16:
        raise SdError(1, f"sd_tree_path: argmax, tokens and parent need one equal length in 1..16 "
                         f"(got {a.size}, {t.size}, {p.size})")
    out = np.empty(t.size, dtype=np.int32)
    n = lib().sd_tree_path(a.ctypes.data, t.ctypes.data, p.ctypes.data, t.size, out.ctypes.data)
    if n < 0:
        raise SdError(1, "sd_tree_path")
    return out[:n].copy()


class DepthPolicy:
    """Adaptive draft depth (host only): ``k`` is the number of drafts to run this cycle (0: plain
    decoding); call ``update(accepted)`` after the cycle."""

    def __init__(self, k_max: int, max_pause: int = 64):
        self.state = SdDepthState()
        _check(lib().sd_depth_init(ctypes.byref(self.state), k_max, max_pause), "sd_depth_init")

    @property
    def k(self) -> int:
        return int(self.state.k_next)

    def update(self, accepted: int) -> int:
        _check(lib().sd_depth_update(ctypes.byref(self.state), accepted), "sd_depth_update")
        return self.k


def attn_workspace_bytes(M: int, H: int, H_kv: int, D: int, L: int) -> int:
    return int(lib().sd_attn_workspace_bytes(M, H, H_kv, D, L))


def kv_append(k_new: torch.Tensor, v_new: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, L: int):
    """k_new, v_new fp32 [M][H_kv][D] -> rows [L, L+M) of the fp16 caches [H_kv][S_max][D]."""
    M, H_kv, D = k_new.shape
    _check(lib().sd_kv_append(_p(k_new), _p(v_new), M, H_kv, D, _p(k_cache), _p(v_cache), k_cache.shape[1], L,
                              _stream()), "sd_kv_append")


def attn_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, L: int, out: torch.Tensor,
                ws: torch.Tensor, parent: torch.Tensor | None = None):
    """q fp32 [M][H][D] over the fp16 caches [H_kv][S_max][D] (L committed rows + M new) -> out [M][H][D]."""
    M, H, D = q.shape
    H_kv, S_max, _ = k_cache.shape
    _check(lib().sd_attn_decode(_p(q), _p(k_cache), _p(v_cache), M, H, H_kv, D, S_max, L, _p(parent), _p(out),
                                _p(ws), ws.numel(), _stream()), "sd_attn_decode")


def kv_commit(k_cache: torch.Tensor, v_cache: torch.Tensor, L: int, M: int, count: torch.Tensor,
              path: torch.Tensor | None = None):
    """Keep the accepted path's rows (count[0] of them) at rows [L, L+count)."""
    H_kv, S_max, D = k_cache.shape
    _check(lib().sd_kv_commit(_p(k_cache), _p(v_cache), H_kv, D, S_max, L, M, _p(path), _p(count), _stream()),
           "sd_kv_commit")


def shortlist_build(head_blocks: torch.Tensor, vocab: int, hidden: int):
    """4-bit copy of a GGUF-order Q8_0 head with its row error bounds and row norms:
    (copy blocks in GGUF order, bound fp32 [vocab], wnorm fp32 [vocab])."""
    dev = head_blocks.device
    copy = torch.empty(vocab * (hidden // 32) * 18, dtype=torch.uint8, device=dev)
    bound = torch.empty(vocab, dtype=torch.float32, device=dev)
    wnorm = torch.empty(vocab, dtype=torch.float32, device=dev)
    _check(lib().sd_shortlist_build(_p(head_blocks), vocab, hidden, _p(copy), _p(bound), _p(wnorm), _stream()),
           "sd_shortlist_build")
    return copy, bound, wnorm


def shortlist_workspace_bytes(vocab: int, hidden: int) -> int:
    return int(lib().sd_shortlist_workspace_bytes(vocab, hidden))


def head_shortlist(copy_w: torch.Tensor, bound: torch.Tensor, wnorm: torch.Tensor, head_w: torch.Tensor,
                   vocab: int, hidden: int, q: torch.Tensor, scales: torch.Tensor, ws: torch.Tensor,
                   argmax: torch.Tensor, n_cand: torch.Tensor | None = None):
    """argmax = sd_head_logits' argmax on the repacked Q8_0 head head_w; ws zero-filled once and kept."""
    M = q.shape[0]
    _check(lib().sd_head_shortlist(_p(copy_w), _p(bound), _p(wnorm), _p(head_w), vocab, hidden, _p(q),
                                   _p(scales), M, _p(argmax), _p(n_cand), _p(ws), ws.numel(), _stream()),
           "sd_head_shortlist")


def accept_greedy(argmax: torch.Tensor, tokens: torch.Tensor | None, parent: torch.Tensor | None, M: int,
                  out_tokens: torch.Tensor, out_count: torch.Tensor):
    _check(lib().sd_accept_greedy(_p(argmax), _p(tokens), _p(parent), M, _p(out_tokens), _p(out_count), _stream()),
           "sd_accept_greedy")


def accept_sample(logits: torch.Tensor, K: int, drafts: torch.Tensor | None, out_tokens: torch.Tensor,
                  out_count: torch.Tensor, q_probs: torch.Tensor | None = None, row_max: torch.Tensor | None = None,
                  row_sumexp: torch.Tensor | None = None, temperature: float = 1.0, seed: int = 0, base_pos: int = 0):
    V = logits.shape[1]
    _check(lib().sd_accept_sample(_p(logits), V, K, _p(row_max), _p(row_sumexp), _p(q_probs), _p(drafts),
                                  temperature, seed, base_pos, _p(out_tokens), _p(out_count), _stream()),
           "sd_accept_sample")


def accept_sample_topk(logits: torch.Tensor, K: int, drafts: torch.Tensor | None, out_tokens: torch.Tensor,
                       out_count: torch.Tensor, top_k: int, top_p: float = 1.0, q_probs: torch.Tensor | None = None,
                       temperature: float = 1.0, seed: int = 0, base_pos: int = 0):
    V = logits.shape[1]
    _check(lib().sd_accept_sample_topk(_p(logits), V, K, _p(q_probs), _p(drafts), temperature, top_k, top_p, seed,
                                       base_pos, _p(out_tokens), _p(out_count), _stream()),
           "sd_accept_sample_topk")


def device_status() -> int:
    return int(lib().sd_device_status(_stream()))


def device_status_site() -> tuple[int, int]:
    """(status, site): the status word and where it was recorded (0 none, 1/2 a time bound,
    >= 100 a bounds check of the debug build); both cleared."""
    site = ctypes.c_int32(0)
    st = int(lib().sd_device_status_site(_stream(), ctypes.byref(site)))
    return st, int(site.value)


def build_flags() -> int:
    return int(lib().sd_build_flags())


def set_pdl(enable: bool):
    lib().sd_set_pdl(1 if enable else 0)


def pass_plan_bytes(n_layers: int) -> int:
    return int(lib().sd_pass_plan_bytes(n_layers))


def pass_workspace_bytes(hidden: int, ffn: int, vocab: int, wq: int = Q4_32) -> int:
    return int(lib().sd_pass_workspace_bytes(hidden, ffn, vocab, wq))


def pass_prepare(desc: SdPassDesc, plan: torch.Tensor) -> SdPass:
    out = SdPass()
    _check(lib().sd_pass_prepare(ctypes.byref(desc), _p(plan), plan.numel(), ctypes.byref(out)), "sd_pass_prepare")
    return out


def verify_pass(p: SdPass):
    _check(lib().sd_verify_pass(ctypes.byref(p), _stream()), "sd_verify_pass")


def pass_trace_bytes(p: SdPass) -> int:
    return int(lib().sd_pass_trace_bytes(ctypes.byref(p)))


def verify_pass_traced(p: SdPass, trace: torch.Tensor):
    """sd_verify_pass with per-phase global-timer stamps into `trace` (int64 CUDA tensor of at least
    pass_trace_bytes(p) bytes): SM ids of the grid's CTAs, then 6 stamps per (phase, CTA)."""
    _check(lib().sd_verify_pass_traced(ctypes.byref(p), _p(trace), trace.numel() * trace.element_size(), _stream()),
           "sd_verify_pass_traced")


# ---------------------------------------------------------------------------
# test hooks
# ---------------------------------------------------------------------------

def debug_block_dots(qtype: int, w: torch.Tensor, n_out: int, k_in: int, q: torch.Tensor) -> torch.Tensor:
    M = q.shape[0]
    dots = torch.empty((M, n_out, k_in // 32), dtype=torch.int32, device=q.device)
    _check(lib().sd_debug_block_dots(qtype, _p(w), n_out, k_in, _p(q), M, _p(dots), _stream()), "sd_debug_block_dots")
    return dots


def debug_silu_mul_requant(g: torch.Tensor, u: torch.Tensor):
    M, F = g.shape
    q = torch.empty((M, F), dtype=torch.int8, device=g.device)
    s = torch.empty((M, F // 32), dtype=torch.float32, device=g.device)
    _check(lib().sd_debug_silu_mul_requant(_p(g), _p(u), M, F, _p(q), _p(s), _stream()), "sd_debug_silu_mul_requant")
    return q, s


def debug_cexp(x: torch.Tensor) -> torch.Tensor:
    y = torch.empty_like(x)
    _check(lib().sd_debug_cexp(_p(x), x.numel(), _p(y), _stream()), "sd_debug_cexp")
    return y


def debug_philox(seed: int, pos: int, n: int, device="cuda") -> torch.Tensor:
    out = torch.empty((n, 4), dtype=torch.int32, device=device)
    _check(lib().sd_debug_philox(seed, pos, n, _p(out), _stream()), "sd_debug_philox")
    return out


def debug_wait_timeout(limit_ns: int):
    _check(lib().sd_debug_wait_timeout(limit_ns, _stream()), "sd_debug_wait_timeout")
