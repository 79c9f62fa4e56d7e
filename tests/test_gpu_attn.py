"""GPU parity of the decode attention over the K+1 positions against the oracle: the fp16 append
and the commit of the accepted path bit-exact; attention outputs within a tolerance derived from
the fp32 arithmetic, for chains and trees, grouped query heads, D = 64 and 128, an empty context,
contexts that leave a ragged last chunk and an odd key count, and a 32k-row context."""
import numpy as np
import pytest
import torch

import oracle
import sdgen
from _util import cuda, host, status_ok

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def sdv():
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    import speculative_decoding_verify_gb300 as m
    m.lib()
    return m


def make_cache(seed, H_kv, S_max, D, L, scale=1.0):
    kc = np.zeros((H_kv, S_max, D), np.uint16)
    vc = np.zeros((H_kv, S_max, D), np.uint16)
    if L:  # seeded inputs, stored as fp16 (numpy's nearest-even conversion)
        kc[:, :L] = (sdgen.normal(sdgen.key(seed, 0), (H_kv, L, D)) * scale).astype(np.float16).view(np.uint16)
        vc[:, :L] = sdgen.normal(sdgen.key(seed, 1), (H_kv, L, D)).astype(np.float16).view(np.uint16)
    return kc, vc


def tolerance(q, kc, vc, L, parent, H_kv):
    """Per output element: (2 delta + 8 (NK + 16) u) * sum_j P_j |v_j| + 1e-30, with delta the
    fp32 rounding of a score in exp2 units, ln2 (D + 3) u max_j sum_d |q_d k_d| log2(e) / sqrt(D),
    plus 4 u for exp2f; P the exact probabilities (numpy, fp64)."""
    M, H, D = q.shape
    g = H // H_kv
    NK = L + M
    K = kc.view(np.float16).astype(np.float64)
    V = vc.view(np.float16).astype(np.float64)
    tol = np.zeros((M, H, D))
    for h in range(H):
        kh = h // g
        qh = q[:, h].astype(np.float64)
        S = qh @ K[kh, :NK].T / np.sqrt(D)
        mask = np.zeros((M, NK))
        for i in range(M):
            if parent is None:
                path = set(range(i + 1))
            else:
                path, a = set(), i
                while a >= 0:
                    path.add(a)
                    a = int(parent[a])
            for j in range(M):
                if j not in path:
                    mask[i, L + j] = -np.inf
        P = np.exp(S + mask - (S + mask).max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        A = P @ np.abs(V[kh, :NK])
        absdot = (np.abs(qh) @ np.abs(K[kh, :NK]).T).max(axis=1) / np.sqrt(D) * np.log2(np.e)
        delta = np.log(2) * (D + 3) * U * absdot + 4 * U
        tol[:, h] = (2 * delta[:, None] + 8 * (NK + 16) * U) * A + 1e-30
    return tol


def run(sdv, q, kc, vc, L, parent=None, new=None):
    """Append the new rows (if given) on the GPU and run the attention; returns out and caches."""
    M, H, D = q.shape
    H_kv = kc.shape[0]
    kd, vd = cuda(kc.view(np.float16)), cuda(vc.view(np.float16))
    if new is not None:
        sdv.kv_append(cuda(new[0]), cuda(new[1]), kd, vd, L)
    out = torch.full((M, H, D), float("nan"), dtype=torch.float32, device="cuda")
    ws = sdv.workspace(sdv.attn_workspace_bytes(M, H, H_kv, D, L))
    par = cuda(np.asarray(parent, np.int32)) if parent is not None else None
    sdv.attn_decode(cuda(q), kd, vd, L, out, ws, par)
    torch.cuda.synchronize()
    status_ok()
    return host(out), host(kd).view(np.uint16), host(vd).view(np.uint16)


CASES = [
    # (H_kv, H, D, L, M, tree)
    (4, 4, 128, 1000, 5, False),
    (4, 4, 128, 1000, 5, True),
    (2, 8, 128, 777, 5, False),      # grouped heads, odd key count
    (2, 6, 64, 300, 4, True),        # D = 64
    (3, 3, 128, 0, 5, True),         # no committed context
    (1, 16, 128, 5000, 16, False),   # 16 positions x 16 heads of a group: two query groups
    (8, 8, 128, 63, 1, False),       # one position
    # contexts of 1024..16384 keys: the chunks of a (query group, KV head) merged in one cluster
    (40, 40, 128, 4096, 5, False),   # the 27B-shaped layer at a short context
    (2, 6, 64, 2000, 4, True),       # D = 64, tree
    (4, 4, 128, 1019, 5, False),     # 1024 keys: the smallest clustered context
    (2, 2, 128, 16379, 5, True),     # 16384 keys: the largest
]


@pytest.mark.parametrize("H_kv,H,D,L,M,tree", CASES)
def test_attention_matches_oracle(sdv, H_kv, H, D, L, M, tree):
    seed = 100 + L + M + H
    S_max = L + M + 13
    kc, vc = make_cache(seed, H_kv, S_max, D, L)
    k_new = sdgen.normal(sdgen.key(seed, 2), (M, H_kv, D))
    v_new = sdgen.normal(sdgen.key(seed, 3), (M, H_kv, D))
    q = sdgen.normal(sdgen.key(seed, 4), (M, H, D))
    parent = None
    if tree:
        parent = np.array([-1] + [int(x) for x in (np.arange(1, M) - 1) // 2], np.int32)  # a binary tree
    out, kd, vd = run(sdv, q, kc, vc, L, parent, new=(k_new, v_new))
    oracle.kv_append(k_new, v_new, kc, vc, L)
    assert np.array_equal(kd, kc) and np.array_equal(vd, vc)   # the append, bit for bit
    ref = oracle.attn_decode(q, kc, vc, L, parent)
    tol = tolerance(q, kc, vc, L, parent, H_kv)
    err = np.abs(out.astype(np.float64) - ref)
    assert np.all(err <= tol), f"worst {(err / tol).max():.3g}x of the bound"


def test_attention_sharp_scores_and_masked_chunks(sdv):
    """Scaled keys make the softmax sharp (scores up to about 100 in exp2 units); a 2-position
    tree whose second row sees only one new key; chunks that hold no visible key for a row."""
    H_kv, H, D, L, M = 2, 2, 128, 3000, 6
    kc, vc = make_cache(7, H_kv, L + M, D, L, scale=4.0)
    k_new = sdgen.normal(sdgen.key(7, 2), (M, H_kv, D)) * 4.0
    v_new = sdgen.normal(sdgen.key(7, 3), (M, H_kv, D))
    q = sdgen.normal(sdgen.key(7, 4), (M, H, D)) * 2.0
    parent = np.array([-1, 0, 0, 1, 1, 2], np.int32)
    out, _, _ = run(sdv, q, kc, vc, L, parent, new=(k_new, v_new))
    oracle.kv_append(k_new, v_new, kc, vc, L)
    ref = oracle.attn_decode(q, kc, vc, L, parent)
    tol = tolerance(q, kc, vc, L, parent, H_kv)
    assert np.all(np.abs(out - ref) <= tol)


@pytest.mark.parametrize("path,count", [([0, 2, 5], 3), ([0, 1, 2, 3, 4, 5], 6), ([0], 1), ([0, 3, 4], 3)])
def test_commit_moves_the_accepted_path(sdv, path, count):
    H_kv, D, L, M = 3, 128, 50, 6
    S_max = L + M
    kc, vc = make_cache(11, H_kv, S_max, D, L + M)
    kd, vd = cuda(kc.view(np.float16)), cuda(vc.view(np.float16))
    p = np.zeros(M, np.int32)
    p[:len(path)] = path
    sdv.kv_commit(kd, vd, L, M, cuda(np.array([count], np.int32)), cuda(p))
    torch.cuda.synchronize()
    status_ok()
    oracle.kv_commit(kc, vc, L, np.array(path, np.int32))
    assert np.array_equal(host(kd).view(np.uint16), kc) and np.array_equal(host(vd).view(np.uint16), vc)


def test_tree_attention_then_commit_then_chain(sdv):
    """Tree attention of node 5, then the commit of its path on the GPU, then chain attention of the
    path's queries over the committed cache: the last row equals node 5's output (same arithmetic
    up to the chunking, checked against the oracle's tolerance on each side)."""
    H_kv, H, D, L, M = 2, 4, 128, 1500, 6
    kc, vc = make_cache(12, H_kv, L + M, D, L)
    k_new = sdgen.normal(sdgen.key(12, 2), (M, H_kv, D))
    v_new = sdgen.normal(sdgen.key(12, 3), (M, H_kv, D))
    q = sdgen.normal(sdgen.key(12, 4), (M, H, D))
    parent = np.array([-1, 0, 0, 2, 2, 3], np.int32)
    kd, vd = cuda(kc.view(np.float16)), cuda(vc.view(np.float16))
    sdv.kv_append(cuda(k_new), cuda(v_new), kd, vd, L)
    out = torch.empty((M, H, D), dtype=torch.float32, device="cuda")
    ws = sdv.workspace(sdv.attn_workspace_bytes(M, H, H_kv, D, L))
    sdv.attn_decode(cuda(q), kd, vd, L, out, ws, cuda(parent))
    path = np.array([0, 2, 3, 5, 0, 0], np.int32)
    sdv.kv_commit(kd, vd, L, M, cuda(np.array([4], np.int32)), cuda(path))
    qc = np.ascontiguousarray(q[[0, 2, 3, 5]])
    out2 = torch.empty((4, H, D), dtype=torch.float32, device="cuda")
    ws2 = sdv.workspace(sdv.attn_workspace_bytes(4, H, H_kv, D, L))
    sdv.attn_decode(cuda(qc), kd, vd, L, out2, ws2)
    torch.cuda.synchronize()
    status_ok()
    oracle.kv_append(k_new, v_new, kc, vc, L)
    ref = oracle.attn_decode(q, kc, vc, L, parent)[5]
    tol = tolerance(q, kc, vc, L, parent, H_kv)[5]
    assert np.all(np.abs(host(out)[5] - ref) <= tol)
    assert np.all(np.abs(host(out2)[3] - ref) <= tol)


def test_attention_long_context(sdv):
    """40 heads of 128 over a 32768-row context at M = 5 (the 27B-shaped attention of one layer)."""
    H_kv, H, D, L, M = 40, 40, 128, 32768, 5
    kc, vc = make_cache(13, H_kv, L + M, D, L)
    k_new = sdgen.normal(sdgen.key(13, 2), (M, H_kv, D))
    v_new = sdgen.normal(sdgen.key(13, 3), (M, H_kv, D))
    q = sdgen.normal(sdgen.key(13, 4), (M, H, D))
    out, _, _ = run(sdv, q, kc, vc, L, None, new=(k_new, v_new))
    oracle.kv_append(k_new, v_new, kc, vc, L)
    ref = oracle.attn_decode(q, kc, vc, L)
    tol = tolerance(q, kc, vc, L, None, H_kv)
    err = np.abs(out - ref)
    assert np.all(err <= tol), f"worst {(err / tol).max():.3g}x of the bound"
