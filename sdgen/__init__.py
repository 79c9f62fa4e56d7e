"""Seeded synthetic inputs for the speculative-decoding verify pass.

Every tensor is a pure function of a small integer key, so any one of them can
be regenerated on its own, in any order and on any number of threads.  The
module holds input synthesis only -- normal variates, the offline Q8_0 / 4-bit
block quantisation a model file would already contain, draft tokens and draft
distributions -- and none of the verify pass's arithmetic.  Both the CUDA path
and the CPU oracle consume what it produces.

Workload recipes (shapes, distributions) follow the synthetic configurations
of the verify-pass benchmark: weights N(0, 0.02), hidden rows N(0, 1), norm
weights 1 + N(0, 0.1), eps 1e-6, hidden 5120, FFN 17408, vocabulary 151936.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsdgen.so")
_lock = threading.Lock()
_lib = None

Q8_0 = 0
Q4_32 = 1
BLOCK_BYTES = {Q8_0: 34, Q4_32: 18}

HIDDEN = 5120
FFN = 17408
VOCAB = 151936
EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile libsdgen.so next to this file (gcc, no FMA contraction)."""
    src = os.path.join(_HERE, "sdgen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _get():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            lib.sdgen_normal_f32.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_float, ctypes.c_float, ctypes.c_void_p]
            lib.sdgen_normal_f32.restype = None
            lib.sdgen_quantize.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_void_p]
            lib.sdgen_quantize.restype = None
            lib.sdgen_normal_quantized.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_int64,
                                                   ctypes.c_int64, ctypes.c_float, ctypes.c_float,
                                                   ctypes.c_void_p, ctypes.c_int]
            lib.sdgen_normal_quantized.restype = ctypes.c_int
            lib.sdgen_u32.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
            lib.sdgen_u32.restype = None
            _lib = lib
    return _lib


def key(*ids: int) -> int:
    """Pack up to four small non-negative ids (config, layer, tensor, seed) into a 64-bit stream key."""
    k = 0x5D5EED
    for i in ids:
        k = (k * 0x100000001B3 + (int(i) & 0xFFFFFFFF) + 1) & 0xFFFFFFFFFFFFFFFF
    return k


def nthreads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal(k: int, shape, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    _get().sdgen_normal_f32(k, 0, n, mean, std, out.ctypes.data)
    return out.reshape(shape)


def quantize(qtype: int, w: np.ndarray) -> np.ndarray:
    """fp32 [n][k] -> GGUF-order blocks, uint8 [n][k/32 * block_bytes]."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    assert k % 32 == 0
    out = np.empty((n, k // 32 * BLOCK_BYTES[qtype]), dtype=np.uint8)
    _get().sdgen_quantize(qtype, w.ctypes.data, n, k, out.ctypes.data)
    return out


def quantized_normal(qtype: int, k: int, n_out: int, k_in: int, std: float = 0.02,
                     out: np.ndarray | None = None) -> np.ndarray:
    """Weights W[n_out][k_in] ~ N(0, std^2) from stream k, quantised to GGUF-order blocks."""
    if out is None:
        out = np.empty((n_out, k_in // 32 * BLOCK_BYTES[qtype]), dtype=np.uint8)
    assert out.flags.c_contiguous and out.nbytes == n_out * (k_in // 32) * BLOCK_BYTES[qtype]
    rc = _get().sdgen_normal_quantized(qtype, k, n_out, k_in, 0.0, std, out.ctypes.data, nthreads())
    if rc:
        raise RuntimeError("sdgen: generation failed")
    return out


def pinned_quantized_normal(qtype: int, k: int, n_out: int, k_in: int, std: float = 0.02):
    """Same as quantized_normal, written straight into a pinned torch uint8 tensor."""
    import torch
    t = torch.empty((n_out, k_in // 32 * BLOCK_BYTES[qtype]), dtype=torch.uint8, pin_memory=True)
    rc = _get().sdgen_normal_quantized(qtype, k, n_out, k_in, 0.0, std, t.data_ptr(), nthreads())
    if rc:
        raise RuntimeError("sdgen: generation failed")
    return t


def u32(k: int, n: int) -> np.ndarray:
    """n raw 32-bit hashes of stream k."""
    out = np.empty(n, dtype=np.uint32)
    _get().sdgen_u32(k, 0, n, out.ctypes.data)
    return out


def uniform_tokens(k: int, n: int, vocab: int) -> np.ndarray:
    """n tokens uniform over [0, vocab) from stream k."""
    return ((u32(k, n).astype(np.uint64) * np.uint64(vocab)) >> np.uint64(32)).astype(np.int32)


def uniforms(k: int, n: int) -> np.ndarray:
    """n float64 uniforms in [0, 1) on a 2^-32 grid from stream k."""
    return u32(k, n).astype(np.float64) * (1.0 / 4294967296.0)


# ---------------------------------------------------------------------------
# Workload recipes
# ---------------------------------------------------------------------------

def drafts_p(k: int, target_argmax: np.ndarray, vocab: int, p_match: float = 0.75) -> np.ndarray:
    """Draft d_i (i = 1..K) equals argmax of row i-1 with probability p_match, else is
    uniform over the vocabulary (which may coincide with the argmax)."""
    K = len(target_argmax)
    u = uniforms(key(k, 1), K)
    rnd = uniform_tokens(key(k, 2), K, vocab)
    return np.where(u < p_match, target_argmax, rnd).astype(np.int32)


def norm_weight(k: int, n: int) -> np.ndarray:
    return normal(k, (n,), std=0.1, mean=1.0)


class StackSpec:
    """27B-shaped dense projection stack: per layer RMSNorm -> QKV (H -> 3H) -> O (H -> H)
    -> RMSNorm -> gate|up (H -> 2F) -> SiLU*mul -> down (F -> H); then a final RMSNorm and
    a Q8_0 vocabulary head.  Attention and recurrent mixers are omitted."""

    def __init__(self, layers=64, hidden=HIDDEN, ffn=FFN, vocab=VOCAB, wq=Q4_32, head_q=Q8_0, seed=0):
        self.layers, self.hidden, self.ffn, self.vocab = layers, hidden, ffn, vocab
        self.wq, self.head_q, self.seed = wq, head_q, seed

    # (name, n_out, k_in)
    def matrices(self):
        H, F = self.hidden, self.ffn
        return [("qkv", 3 * H, H), ("o", H, H), ("gate_up", 2 * F, H), ("down", H, F)]

    def weight_key(self, layer: int, name: str) -> int:
        idx = {"qkv": 0, "o": 1, "gate_up": 2, "down": 3, "head": 4}[name]
        return key(4, self.seed, layer, idx)

    def norm_key(self, layer: int, which: int) -> int:
        return key(4, self.seed, layer, 10 + which)

    def weights(self, layer: int, name: str) -> np.ndarray:
        for nm, n, k in self.matrices():
            if nm == name:
                return quantized_normal(self.wq, self.weight_key(layer, name), n, k)
        raise KeyError(name)

    def head(self) -> np.ndarray:
        return quantized_normal(self.head_q, self.weight_key(0, "head"), self.vocab, self.hidden)

    def norms(self, layer: int):
        return norm_weight(self.norm_key(layer, 0), self.hidden), norm_weight(self.norm_key(layer, 1), self.hidden)

    def final_norm(self) -> np.ndarray:
        return norm_weight(self.norm_key(self.layers, 2), self.hidden)

    def hidden_in(self, M: int) -> np.ndarray:
        return normal(key(4, self.seed, 999, 0), (M, self.hidden))

    def weight_bytes(self) -> int:
        bb = BLOCK_BYTES[self.wq]
        per_layer = sum(n * (k // 32) * bb for _, n, k in self.matrices())
        return self.layers * per_layer + self.vocab * (self.hidden // 32) * BLOCK_BYTES[self.head_q]


def tree16(k: int):
    """16-node draft tree: root, complete binary tree of depth 3 (15 nodes), plus one node
    hanging below the first depth-3 leaf in BFS order.  Returns parent[16] (BFS order,
    parent[0] = -1) and depth[16]."""
    parent = [-1]
    for i in range(1, 15):
        parent.append((i - 1) // 2)
    parent.append(7)  # first depth-3 leaf in BFS order is node 7
    depth = [0] * 16
    for i in range(1, 16):
        depth[i] = depth[parent[i]] + 1
    return np.array(parent, dtype=np.int32), np.array(depth, dtype=np.int32)


KQ_BLOCK_BYTES = {2: 144, 3: 210}   # Q4_K, Q6_K super-blocks of 256 weights


def random_kq_blocks(qtype: int, k: int, n_out: int, k_in: int, d_scale: float = 1e-3) -> np.ndarray:
    """Seeded K-quant super-blocks [n_out][k_in/256]: random code and scale bytes (every byte
    pattern is a valid block), with the fp16 scale fields set to finite values in
    [d_scale, 2 d_scale)."""
    assert k_in % 256 == 0
    bb = KQ_BLOCK_BYTES[qtype]
    nblk = n_out * (k_in // 256)
    raw = u32(k, (nblk * bb + 3) // 4).view(np.uint8)[:nblk * bb].reshape(nblk, bb).copy()
    d = (d_scale * (1.0 + u32(key(k, 1), 2 * nblk).astype(np.float64) / 2.0 ** 32)).astype(np.float16)
    d = d.view(np.uint8).reshape(nblk, 2, 2)
    if qtype == 2:
        raw[:, 0:2] = d[:, 0]
        raw[:, 2:4] = d[:, 1]
    else:
        raw[:, 208:210] = d[:, 0]
    return raw.reshape(n_out, -1)
