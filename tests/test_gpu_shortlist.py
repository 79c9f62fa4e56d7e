"""GPU parity of the exact shortlist head ("How Kinetic is fast", section "Shortlist": every
exact score comes from the layer's own kernel, so the chosen token is the full layer's):
sd_shortlist_build against the oracle's copy (bytes bit-exact, bounds valid and tight), and
sd_head_shortlist's argmax equal to sd_head_logits' argmax on the same inputs, bit for bit, on
random heads where the bound prunes nothing, on heads with one row per position that stands out
(the bound prunes nearly everything; there the token is also the oracle's), with exact ties, with
two rows whose copies are equal byte for byte, across the full-mode switch and its retries, and at
the full 151936 x 5120 head."""
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


def head_argmax(sdv, head, N, K, q, s):
    """sd_head_logits' argmax: the reference the shortlist must reproduce."""
    M = q.shape[0]
    ws = sdv.workspace(sdv.head_workspace_bytes(N, K))
    logits = torch.empty((M, N), dtype=torch.float32, device="cuda")
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    rm = torch.empty(M, dtype=torch.float32, device="cuda")
    rs = torch.empty(M, dtype=torch.float32, device="cuda")
    sdv.head_logits(head, N, K, cuda(q), cuda(s), ws, logits, am, rm, rs)
    torch.cuda.synchronize()
    status_ok()
    return host(am)


def gpu_shortlist(sdv, w8, N, K, q, s, built=None, ws=None):
    """(shortlist argmax, candidate counts, sd_head_logits' argmax)."""
    hb, copy, bound, wnorm = built if built is not None else gpu_build(sdv, w8, N, K)
    cw = sdv.repack_weights(sdv.Q4_32, copy, N, K)
    head = sdv.repack_weights(sdv.Q8_0, hb, N, K)
    if ws is None:
        ws = sdv.workspace(sdv.shortlist_workspace_bytes(N, K))
    M = q.shape[0]
    am = torch.full((M,), -2, dtype=torch.int32, device="cuda")
    nc = torch.full((M,), -2, dtype=torch.int32, device="cuda")
    sdv.head_shortlist(cw, bound, wnorm, head, N, K, cuda(q), cuda(s), ws, am, nc)
    torch.cuda.synchronize()
    status_ok()
    return host(am), host(nc), head_argmax(sdv, head, N, K, q, s)


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


def check(sdv, w8, N, K, q, s, max_cand=None, ws=None):
    am, nc, am_h = gpu_shortlist(sdv, w8, N, K, q, s, ws=ws)
    assert list(am) == list(am_h)
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
    # equal exact scores: the head's fp32 sums of the tied rows may differ in the last bit (their tiles
    # are summed in different pieces), and the shortlist follows the head
    assert am[0] in (7, top, N - 1)


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
        am, _, am_h = gpu_shortlist(sdv, w8, N, K, q, s, ws=ws)
        assert list(am) == list(am_h)


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


def test_shortlist_full_mode_and_its_retries(sdv):
    """A random head fills every tile with candidates, so the next calls run in full mode (every row
    counted); on a peaked head the 16th call tries the shortlist again and stays with it."""
    N, K, M = 5000, 1024, 5
    w8 = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(87), N, K)
    q, s = acts(sdgen.key(87, 1), M, K)
    ws = sdv.workspace(sdv.shortlist_workspace_bytes(N, K))
    am, nc = check(sdv, w8, N, K, q, s, ws=ws)                 # call 0: shortlist, nearly all candidates
    am, nc = check(sdv, w8, N, K, q, s, ws=ws)                 # call 1: full mode
    assert list(nc) == [N] * M
    rows_for = [(97 * m + 13) % N for m in range(M)]
    pk = planted(w8, N, K, q, s, rows_for)
    for call in range(2, 18):
        am, nc = check(sdv, pk, N, K, q, s, ws=ws)
        assert list(am) == rows_for
        if call < 16:
            assert list(nc) == [N] * M, call               # still full mode
        else:
            assert np.all(nc <= N // 100), (call, nc)      # retried at call 16, kept at 17
