"""GPU parity of the exact shortlist head ("How Kinetic is fast", section "Shortlist"):
sd_shortlist_build against the oracle's copy (bytes bit-exact, bounds valid and tight), and
sd_head_shortlist's argmax against the oracle's (bit-exact: both take the exact scores in fp64 in
block order), on random heads where the bound prunes nothing, on heads with one row per position
that stands out (the bound prunes nearly everything), with exact ties, with two rows whose copies
are equal byte for byte, and at the full 151936 x 5120 head."""
import numpy as np
import pytest
import torch

import oracle
import sdgen
from _util import acts, cuda, host, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    import speculative_decoding_verify_gb300 as m
    m.lib()
    return m


def gpu_build(sdv, w8, N, K):
    hb = cuda(np.asarray(w8, dtype=np.uint8).reshape(-1))
    copy, bound, wnorm = sdv.shortlist_build(hb, N, K)
    torch.cuda.synchronize()
    status_ok()
    return hb, copy, bound, wnorm


def gpu_shortlist(sdv, w8, N, K, q, s, built=None, ws=None):
    hb, copy, bound, wnorm = built if built is not None else gpu_build(sdv, w8, N, K)
    cw = sdv.repack_weights(sdv.Q4_32, copy, N, K)
    if ws is None:
        ws = sdv.workspace(sdv.shortlist_workspace_bytes(N, K))
    M = q.shape[0]
    am = torch.full((M,), -2, dtype=torch.int32, device="cuda")
    nc = torch.full((M,), -2, dtype=torch.int32, device="cuda")
    sdv.head_shortlist(cw, bound, wnorm, hb, N, K, cuda(q), cuda(s), ws, am, nc)
    torch.cuda.synchronize()
    status_ok()
    return host(am), host(nc)


def true_norms(w8, q4, N, K):
    a = oracle.dequant(oracle.Q8_0, w8, N, K).astype(np.float64).reshape(N, K)
    b = oracle.dequant(oracle.Q4_32, q4, N, K).astype(np.float64).reshape(N, K)
    return np.sqrt(((a - b) ** 2).sum(axis=1)), np.sqrt((a ** 2).sum(axis=1))


def with_edge_blocks(w8, N, K):
    """A zero block (d = 0), a block whose amax / 7.5 overflows fp16 (scale held at 65504), and a
    block with the smallest subnormal scale."""
    rows = np.asarray(w8, dtype=np.uint8).reshape(N, K // 32, 34).copy()
    rows[0, 0] = 0
    rows[1, 0, :2] = np.frombuffer(np.float16(65504.0).tobytes(), dtype=np.uint8)
    rows[1, 0, 2:] = np.arange(-127, 129, 8)[:32].astype(np.int8).view(np.uint8)
    rows[2, 1, :2] = np.array([1, 0], dtype=np.uint8)  # fp16 0x0001 = 2^-24
    return rows.reshape(-1)


@pytest.mark.parametrize("N,K", [(1000, 1024), (33, 64), (4096, 5120), (1, 32)])
def test_shortlist_build_matches_oracle(sdv, N, K):
    w8 = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(80, N), N, K)
    if N >= 3 and K >= 64:
        w8 = with_edge_blocks(w8, N, K)
    _, copy, bound, wnorm = gpu_build(sdv, w8, N, K)
    q4_o, bound_o, wnorm_o = oracle.shortlist_copy(w8, N, K)
    assert np.array_equal(host(copy), q4_o)
    e, wn = true_norms(w8, q4_o, N, K)
    g_b, g_w = host(bound).astype(np.float64), host(wnorm).astype(np.float64)
    # rounded up: never below the fp64 norm, at most one fp32 step above it
    assert np.all(g_b >= e) and np.all(g_b <= e * (1 + 2.5e-7) + 1e-44)
    assert np.all(g_w >= wn) and np.all(g_w <= wn * (1 + 2.5e-7) + 1e-44)


def planted(w8, N, K, q, s, rows_for):
    """Row rows_for[m] follows position m's activations: the winner stands out by far."""
    M = q.shape[0]
    a = (q.astype(np.float64).reshape(M, K // 32, 32) * s[:, :, None]).reshape(M, K)
    rows = np.asarray(w8, dtype=np.uint8).reshape(N, -1).copy()
    for m, r in enumerate(rows_for):
        blk = sdgen.quantize(oracle.Q8_0, (a[m] / np.abs(a[m]).max() * 0.1).astype(np.float32)[None, :])
        rows[r] = np.asarray(blk).reshape(-1)
    return rows.reshape(-1)


def check(sdv, w8, N, K, q, s, max_cand=None):
    am, nc = gpu_shortlist(sdv, w8, N, K, q, s)
    q4, bound, _ = oracle.shortlist_copy(w8, N, K)
    am_o, _ = oracle.shortlist_argmax(q4, bound, w8, N, K, q, s)
    assert list(am) == list(am_o)
    assert np.all(nc >= 1) and np.all(nc <= N)
    if max_cand is not None:
        assert np.all(nc <= max_cand), nc
    return am, nc


@pytest.mark.parametrize("N,K,M", [(5000, 1024, 5), (3000, 512, 16), (4096, 1024, 1), (1, 32, 5), (77, 32, 3)])
def test_shortlist_argmax_random(sdv, N, K, M):
    w8 = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(81, N), N, K)
    q, s = acts(sdgen.key(81, N + 1), M, K)
    check(sdv, w8, N, K, q, s)


@pytest.mark.parametrize("N,K,M", [(5000, 1024, 5), (3000, 512, 16)])
def test_shortlist_argmax_planted_winners_prune(sdv, N, K, M):
    w8 = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(82, N), N, K)
    q, s = acts(sdgen.key(82, N + 1), M, K)
    rows_for = [(97 * m + 13) % N for m in range(M)]
    w8 = planted(w8, N, K, q, s, rows_for)
    am, _ = check(sdv, w8, N, K, q, s, max_cand=N // 100)
    assert list(am) == rows_for


def test_shortlist_argmax_ties_take_the_lower_index(sdv):
    N, K, M = 4096, 1024, 3
    w8 = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(83), N, K)
    q, s = acts(sdgen.key(83, 1), M, K)
    q4, bound, _ = oracle.shortlist_copy(w8, N, K)
    top = int(oracle.shortlist_argmax(q4, bound, w8, N, K, q, s)[0][0])
    rows = np.asarray(w8).reshape(N, -1).copy()
    for dup in (7, N - 1):          # one copy below, one above the winner
        if dup != top:
            rows[dup] = rows[top]
    w8 = rows.reshape(-1)
    am, _ = check(sdv, w8, N, K, q, s)
    assert am[0] == min(7, top)


def test_shortlist_argmax_when_the_copy_ranks_the_winner_second(sdv):
    """Rows whose 4-bit copies are equal byte for byte, the lower one an int8 step worse exactly."""
    N, K, M = 1024, 512, 1
    w8 = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(84), N, K)
    q, s = acts(sdgen.key(84, 1), M, K)
    q4, bound, _ = oracle.shortlist_copy(w8, N, K)
    top = int(oracle.shortlist_argmax(q4, bound, w8, N, K, q, s)[0][0])
    lo = 3 if top != 3 else 4
    rows = np.asarray(w8).reshape(N, K // 32, 34).copy()
    a = q.astype(np.int64).reshape(K)
    copy_top = oracle.shortlist_copy(rows[top].reshape(-1), 1, K)[0]
    found = False
    for b in range(K // 32):
        v = rows[top, b, 2:].view(np.int8).astype(np.int64)
        for j in range(32):
            if a[b * 32 + j] == 0 or abs(v[j]) == np.abs(v).max():
                continue
            w = v.copy()
            w[j] -= 1 if a[b * 32 + j] > 0 else -1
            if abs(w[j]) >= np.abs(v).max():
                continue
            cand = rows[top].copy()
            cand[b, 2:] = w.astype(np.int8).view(np.uint8)
            if np.array_equal(oracle.shortlist_copy(cand.reshape(-1), 1, K)[0], copy_top):
                rows[lo] = cand
                found = True
                break
        if found:
            break
    assert found
    am, nc = check(sdv, rows.reshape(-1), N, K, q, s)
    assert am[0] == top and nc[0] >= 2


def test_shortlist_workspace_reused_across_calls(sdv):
    """One workspace, calls of two shapes in a row: the copy matmul's counters return to zero."""
    K = 1024
    big = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(85), 6000, K)
    ws = sdv.workspace(sdv.shortlist_workspace_bytes(6000, K))
    for N, M, seed in ((6000, 5, 1), (2500, 3, 2), (6000, 5, 3)):
        w8 = np.asarray(big).reshape(6000, -1)[:N].reshape(-1)
        q, s = acts(sdgen.key(85, seed), M, K)
        am, _ = gpu_shortlist(sdv, w8, N, K, q, s, ws=ws)
        q4, bound, _ = oracle.shortlist_copy(w8, N, K)
        assert list(am) == list(oracle.shortlist_argmax(q4, bound, w8, N, K, q, s)[0])


@pytest.mark.parametrize("peaked", [False, True])
def test_shortlist_full_vocabulary_head(sdv, peaked):
    """The 151936 x 5120 head over 5 positions."""
    N, K, M = 151936, 5120, 5
    w8 = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(86), N, K)
    q, s = acts(sdgen.key(86, 1), M, K)
    rows_for = [151935, 0, 77777, 4096, 100000]
    if peaked:
        w8 = planted(w8, N, K, q, s, rows_for)
    am, nc = check(sdv, w8, N, K, q, s, max_cand=N // 1000 if peaked else None)
    if peaked:
        assert list(am) == rows_for
