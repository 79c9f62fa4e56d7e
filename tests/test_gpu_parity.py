"""GPU parity: every ABI call against the CPU oracle on the same seeded inputs,
at sizes the oracle finishes in seconds that still span many tiles, several
k-splits and ragged tails.  Integer and index results must be bit-exact; fp32
results within 1e-5 of the absolute-sum bound; every output batch-invariant."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import sdgen
from _util import acts, assert_close, cuda, host, status_ok, unpack_repacked

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def sdv():
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    import speculative_decoding_verify_gb300 as m
    m.lib()
    return m


def gpu_qmm(sdv, qtype, blocks, n, k, q, s, residual=None, epi=0, col0=0, want_y=True, ws=None):
    pair = epi == sdv.EPI_SILU_MUL_REQUANT
    w = sdv.repack_weights(qtype, cuda(blocks).reshape(-1), n, k, pair)
    torch.cuda.synchronize()
    M = q.shape[0]
    if ws is None:
        ws = sdv.workspace(sdv.qmatmul_workspace_bytes(qtype, n, k, epi))
    y = torch.full((M, n), float("nan"), dtype=torch.float32, device="cuda") if want_y else None
    res = cuda(residual) if residual is not None else None
    qn = sn = None
    if epi == sdv.EPI_REQUANT:
        qn = torch.zeros((M, n - col0), dtype=torch.int8, device="cuda")
        sn = torch.zeros((M, (n - col0) // 32), dtype=torch.float32, device="cuda")
    elif pair:
        qn = torch.zeros((M, n // 2), dtype=torch.int8, device="cuda")
        sn = torch.zeros((M, n // 64), dtype=torch.float32, device="cuda")
    sdv.qmatmul_multipos(qtype, w, n, k, cuda(q), cuda(s), ws, y=y, residual=res, epilogue=epi, requant_col0=col0,
                         q_next=qn, scales_next=sn)
    status_ok()
    return (host(y) if y is not None else None), (host(qn) if qn is not None else None), \
        (host(sn) if sn is not None else None), ws


# ---------------------------------------------------------------------------
# repack
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("qtype", [oracle.Q8_0, oracle.Q4_32])
@pytest.mark.parametrize("shape,pair", [((64, 64), False), ((1000, 96), False), ((33, 32), False),
                                        ((2 * 96, 64), True), ((2 * 50, 32), True)])
def test_repack_roundtrip_bytes_unchanged(sdv, qtype, shape, pair):
    n, k = shape
    blocks = sdgen.quantized_normal(qtype, sdgen.key(100, n, k, qtype), n, k)
    out = sdv.repack_weights(qtype, cuda(blocks).reshape(-1), n, k, pair)
    status_ok()
    assert out.numel() == sdv.repacked_bytes(qtype, n, k, pair)
    back = unpack_repacked(qtype, host(out), n, k, pair)
    assert np.array_equal(back, blocks)


# ---------------------------------------------------------------------------
# integer work: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("qtype", [oracle.Q8_0, oracle.Q4_32])
def test_block_dots_bit_exact(sdv, qtype):
    n, k, M = 100, 192, 7
    blocks = sdgen.quantized_normal(qtype, sdgen.key(101, qtype), n, k)
    q, _ = acts(sdgen.key(102), M, k, 3.0)
    q[0, :32] = 127
    q[1, :32] = -127
    w = sdv.repack_weights(qtype, cuda(blocks).reshape(-1), n, k)
    g = host(sdv.debug_block_dots(qtype, w, n, k, cuda(q)))
    status_ok()
    assert np.array_equal(g, oracle.block_dots(qtype, blocks, n, k, q))


@pytest.mark.parametrize("K", [1024, 5120, 17408])
@pytest.mark.parametrize("M", [1, 5, 16])
@pytest.mark.parametrize("with_norm", [True, False])
def test_rmsnorm_quant_bit_exact(sdv, K, M, with_norm):
    x = sdgen.normal(sdgen.key(103, K, M), (M, K))
    x[0, :64] *= 1000.0
    if M > 1:
        x[1, 32:64] = 0.0
    w = sdgen.norm_weight(sdgen.key(104, K), K) if with_norm else None
    q = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    s = torch.zeros((M, K // 32), dtype=torch.float32, device="cuda")
    sdv.rmsnorm_quant_acts(cuda(x), cuda(w) if w is not None else None, q, s, 1e-6)
    status_ok()
    qo, so = oracle.rmsnorm_quant(x, w, 1e-6)
    assert np.array_equal(host(q), qo)
    assert np.array_equal(host(s).view(np.uint32), so.view(np.uint32))


def test_rmsnorm_strided_rows(sdv):
    M, K, ld = 5, 512, 1536
    x = sdgen.normal(sdgen.key(105), (M, ld))
    q = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    s = torch.zeros((M, K // 32), dtype=torch.float32, device="cuda")
    xd = cuda(x)
    sdv.rmsnorm_quant_acts(xd[:, 1024:], None, q, s, 1e-6, K=K, ldx=ld)
    status_ok()
    qo, so = oracle.rmsnorm_quant(np.ascontiguousarray(x[:, 1024:]), None)
    assert np.array_equal(host(q), qo) and np.array_equal(host(s), so)


def test_cexp_bit_exact(sdv):
    xs = np.concatenate([np.linspace(-110.0, 95.0, 400001, dtype=np.float32),
                         sdgen.normal(sdgen.key(106), (100000,)) * 10,
                         np.array([0.0, -0.0, 1e-30, -1e-30, 88.72, 88.73, -103.97, -104.0, -87.3], np.float32)])
    g = host(sdv.debug_cexp(cuda(xs)))
    status_ok()
    o = oracle.cexp(xs)
    assert np.array_equal(g.view(np.uint32), o.view(np.uint32))


def test_philox_matches_oracle_and_kat(sdv):
    kat = json.load(open(os.path.join(GOLDEN, "philox4x32_10_kat.json")))["vectors"][0]
    g0 = host(sdv.debug_philox(0, 0, 1)).view(np.uint32)[0]
    assert [f"{int(v):08x}" for v in g0] == kat["out"]
    for seed, pos in ((0, 0), (0xDEADBEEF12345678, 1 << 33), (7, -5)):
        g = host(sdv.debug_philox(seed, pos, 500)).view(np.uint32)
        for i in range(0, 500, 37):
            p = (pos + i) & 0xFFFFFFFFFFFFFFFF
            o = oracle.philox4x32_10([p & 0xFFFFFFFF, p >> 32, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
            assert np.array_equal(g[i], o)
    status_ok()


def test_silu_mul_requant_bit_exact(sdv):
    M, F = 5, 17408
    g = sdgen.normal(sdgen.key(107), (M, F)) * 3
    u = sdgen.normal(sdgen.key(108), (M, F))
    g[0, :6] = [0.0, 95.0, -95.0, 1e-30, 20.0, -20.0]
    qg, sg = sdv.debug_silu_mul_requant(cuda(g), cuda(u))
    status_ok()
    qo, so, _ = oracle.silu_mul_requant(g, u)
    assert np.array_equal(host(qg), qo)
    assert np.array_equal(host(sg).view(np.uint32), so.view(np.uint32))


# ---------------------------------------------------------------------------
# multi-position matmul
# ---------------------------------------------------------------------------

SHAPES = [(1024, 1024), (1000, 320), (96, 17408), (4096, 1024), (200, 5120)]


@pytest.mark.parametrize("qtype", [oracle.Q8_0, oracle.Q4_32])
@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("M", [1, 3, 5, 8, 11, 16])
def test_qmatmul_vs_oracle(sdv, qtype, shape, M):
    n, k = shape
    blocks = sdgen.quantized_normal(qtype, sdgen.key(110, n, k, qtype), n, k)
    q, s = acts(sdgen.key(111, k, M), M, k)
    y, _, _, ws = gpu_qmm(sdv, qtype, blocks, n, k, q, s)
    yo, ab = oracle.qmatmul(qtype, blocks, n, k, q, s)
    assert_close(y, yo, ab, f"qmm q{qtype} {shape} M={M}")
    # a second call on the same workspace (its counters must be back at zero) gives the same bits
    y2, _, _, _ = gpu_qmm(sdv, qtype, blocks, n, k, q, s, ws=ws)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("qtype", [oracle.Q8_0, oracle.Q4_32])
def test_qmatmul_residual_in_place(sdv, qtype):
    n, k, M = 640, 2048, 5
    blocks = sdgen.quantized_normal(qtype, sdgen.key(112, qtype), n, k)
    q, s = acts(sdgen.key(113), M, k)
    r = sdgen.normal(sdgen.key(114), (M, n)) * 5
    w = sdv.repack_weights(qtype, cuda(blocks).reshape(-1), n, k)
    ws = sdv.workspace(sdv.qmatmul_workspace_bytes(qtype, n, k))
    h = cuda(r)
    sdv.qmatmul_multipos(qtype, w, n, k, cuda(q), cuda(s), ws, y=h, residual=h)
    status_ok()
    yo, ab = oracle.qmatmul(qtype, blocks, n, k, q, s, residual=r)
    assert_close(host(h), yo, ab, "in-place residual")


def test_one_workspace_serves_mixed_shapes(sdv):
    """Calls of different shapes (different unit counts and k splits) share one workspace."""
    M = 5
    shapes = [(3 * 256, 320, 4), (640, 5120, 3), (96, 17408, 2), (4000, 1024, 1), (640, 5120, 3)]
    ws = sdv.workspace(max(sdv.qmatmul_workspace_bytes(oracle.Q4_32, n, k) for n, k, _ in shapes))
    for n, k, key in shapes:
        blocks = sdgen.quantized_normal(oracle.Q4_32, sdgen.key(140, key), n, k)
        q, s = acts(sdgen.key(141, k), M, k)
        r = sdgen.normal(sdgen.key(142, n), (M, n))
        y, _, _, _ = gpu_qmm(sdv, oracle.Q4_32, blocks, n, k, q, s, residual=r, ws=ws)
        yo, ab = oracle.qmatmul(oracle.Q4_32, blocks, n, k, q, s, residual=r)
        assert_close(y, yo, ab, f"shared workspace {n}x{k}")


def test_requant_epilogue(sdv):
    """QKV-like: the last third of the columns is requantised in the epilogue.  The codes equal the
    standalone requantisation kernel applied to the same GPU outputs; the outputs match the oracle."""
    H, M = 256, 5
    n, k, col0 = 3 * H, H, 2 * H
    blocks = sdgen.quantized_normal(oracle.Q4_32, sdgen.key(115), n, k)
    q, s = acts(sdgen.key(116), M, k)
    y, qn, sn, _ = gpu_qmm(sdv, oracle.Q4_32, blocks, n, k, q, s, epi=sdv.EPI_REQUANT, col0=col0)
    yo, ab = oracle.qmatmul(oracle.Q4_32, blocks, n, k, q, s)
    assert_close(y, yo, ab, "requant epilogue y")
    qq = torch.zeros((M, n - col0), dtype=torch.int8, device="cuda")
    ss = torch.zeros((M, (n - col0) // 32), dtype=torch.float32, device="cuda")
    yd = cuda(y)
    sdv.rmsnorm_quant_acts(yd[:, col0:], None, qq, ss, K=n - col0, ldx=n)
    status_ok()
    assert np.array_equal(host(qq), qn) and np.array_equal(host(ss), sn)
    # and against the oracle's own codes: only values on a rounding boundary may differ, by one step
    qo, so = oracle.rmsnorm_quant(np.ascontiguousarray(yo[:, col0:]), None)
    assert np.abs(qo.astype(int) - qn.astype(int)).max() <= 1
    assert (qo != qn).mean() < 1e-3


@pytest.mark.parametrize("F,k", [(256, 256), (2048, 1024), (512, 17408)])
def test_silu_epilogue(sdv, F, k):
    M = 5
    n = 2 * F
    blocks = sdgen.quantized_normal(oracle.Q4_32, sdgen.key(117, F, k), n, k)
    q, s = acts(sdgen.key(118, k), M, k)
    y, qn, sn, _ = gpu_qmm(sdv, oracle.Q4_32, blocks, n, k, q, s, epi=sdv.EPI_SILU_MUL_REQUANT)
    yo, ab = oracle.qmatmul(oracle.Q4_32, blocks, n, k, q, s)
    assert_close(y, yo, ab, "gate|up")
    qd, sd = sdv.debug_silu_mul_requant(cuda(y[:, :F]), cuda(y[:, F:]))
    status_ok()
    assert np.array_equal(host(qd), qn) and np.array_equal(host(sd), sn)
    qo, so, _ = oracle.silu_mul_requant(np.ascontiguousarray(yo[:, :F]), np.ascontiguousarray(yo[:, F:]))
    assert np.abs(qo.astype(int) - qn.astype(int)).max() <= 1
    assert (qo != qn).mean() < 1e-3


@pytest.mark.parametrize("qtype,epi", [(oracle.Q8_0, 0), (oracle.Q4_32, 0), (oracle.Q4_32, 1), (oracle.Q4_32, 2)])
@pytest.mark.parametrize("shape", [(1024, 1024), (512, 17408)])
def test_batch_invariance(sdv, qtype, epi, shape):
    """A row computed among 16 positions equals the same row computed alone, bit for bit."""
    n, k = shape
    if epi == 1:
        col0 = n // 2
    else:
        col0 = 0
    blocks = sdgen.quantized_normal(qtype, sdgen.key(119, n, k, qtype), n, k)
    q, s = acts(sdgen.key(120, k), 16, k)
    y16, q16, s16, _ = gpu_qmm(sdv, qtype, blocks, n, k, q, s, epi=epi, col0=col0)
    for m in range(16):
        y1, q1, s1, _ = gpu_qmm(sdv, qtype, blocks, n, k, q[m:m + 1], s[m:m + 1], epi=epi, col0=col0)
        assert np.array_equal(y1.view(np.uint32), y16[m:m + 1].view(np.uint32))
        if q1 is not None:
            assert np.array_equal(q1, q16[m:m + 1]) and np.array_equal(s1, s16[m:m + 1])


# ---------------------------------------------------------------------------
# head with fused argmax and softmax statistics
# ---------------------------------------------------------------------------

def gpu_head(sdv, blocks, V, H, q, s, T=1.0):
    w = sdv.repack_weights(oracle.Q8_0, cuda(blocks).reshape(-1), V, H)
    M = q.shape[0]
    ws = sdv.workspace(sdv.head_workspace_bytes(V, H))
    logits = torch.zeros((M, V), dtype=torch.float32, device="cuda")
    am = torch.zeros(M, dtype=torch.int32, device="cuda")
    rm = torch.zeros(M, dtype=torch.float32, device="cuda")
    rz = torch.zeros(M, dtype=torch.float32, device="cuda")
    sdv.head_logits(w, V, H, cuda(q), cuda(s), ws, logits, am, rm, rz, T)
    status_ok()
    return host(logits), host(am), host(rm), host(rz)


@pytest.mark.parametrize("V,H,T,M", [(4096, 1024, 1.0, 5), (3000, 512, 0.7, 3), (40000, 1024, 1.0, 16)])
def test_head_vs_oracle(sdv, V, H, T, M):
    blocks = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(121, V, H), V, H)
    q, s = acts(sdgen.key(122, H), M, H)
    lg, am, rm, rz = gpu_head(sdv, blocks, V, H, q, s, T)
    lo, ab = oracle.qmatmul(oracle.Q8_0, blocks, V, H, q, s)
    assert_close(lg, lo, ab, "head logits")
    # argmax: the lowest index of the GPU logits' maximum; a near-tie within tolerance may pick another
    # index than the oracle, but never a logit outside the tolerance of the oracle maximum
    assert np.array_equal(am, np.argmax(lg, axis=1))
    om = oracle.softmax_stats(lo, T)
    tol = 1e-5 * ab.max(axis=1) + 1e-6
    for m in range(M):
        assert lo[m, am[m]] >= lo[m].max() - 2 * tol[m]
    assert np.array_equal(rm, (lg / np.float32(T)).max(axis=1))
    assert np.all(np.abs(rz / om[1] - 1) <= 2 * tol / T + 1e-6)


def test_head_batch_invariance(sdv):
    V, H = 4096, 1024
    blocks = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(123), V, H)
    q, s = acts(sdgen.key(124), 16, H)
    lg, am, rm, rz = gpu_head(sdv, blocks, V, H, q, s)
    for m in (0, 7, 15):
        l1, a1, r1, z1 = gpu_head(sdv, blocks, V, H, q[m:m + 1], s[m:m + 1])
        assert np.array_equal(l1.view(np.uint32), lg[m:m + 1].view(np.uint32))
        assert a1[0] == am[m] and r1[0] == rm[m] and z1[0] == rz[m]


def test_head_repeated_calls_identical(sdv):
    """Many back-to-back head calls at 16 positions (every consumer warp busy in the epilogue, so
    the CTA's warps reach the statistics bookkeeping in varying order) return identical results."""
    V, H, M = 4096, 512, 16
    blocks = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(125), V, H)
    q, s = acts(sdgen.key(126), M, H)
    w = sdv.repack_weights(oracle.Q8_0, cuda(blocks).reshape(-1), V, H)
    ws = sdv.workspace(sdv.head_workspace_bytes(V, H))
    qd, sd = cuda(q), cuda(s)
    outs = []
    for _ in range(40):
        lg = torch.zeros((M, V), dtype=torch.float32, device="cuda")
        am = torch.zeros(M, dtype=torch.int32, device="cuda")
        rm = torch.zeros(M, dtype=torch.float32, device="cuda")
        rz = torch.zeros(M, dtype=torch.float32, device="cuda")
        sdv.head_logits(w, V, H, qd, sd, ws, lg, am, rm, rz, 1.0)
        outs.append((lg, am, rm, rz))
    status_ok()
    for o in outs[1:]:
        for x, y in zip(o, outs[0]):
            assert torch.equal(x, y)


# ---------------------------------------------------------------------------
# acceptance: bit-exact when fed the oracle's logits
# ---------------------------------------------------------------------------

def test_accept_greedy_bit_exact(sdv):
    g = json.load(open(os.path.join(GOLDEN, "rad1_worked_example.json")))
    cases = [(np.array(c["argmax"]), np.array(c["drafts"]), None) for c in g["cases"].values()]
    rng = np.random.default_rng(130)
    for _ in range(200):
        K = int(rng.integers(0, 16))
        cases.append((rng.integers(0, 3, K + 1), rng.integers(0, 3, K), None))
    parent, _ = sdgen.tree16(0)
    for _ in range(200):
        cases.append((rng.integers(0, 3, 16), rng.integers(0, 3, 16), parent))
    outs = []
    for am, tok, par in cases:
        M = len(am)
        ot = torch.full((M,), -7, dtype=torch.int32, device="cuda")
        oc = torch.zeros(1, dtype=torch.int32, device="cuda")
        sdv.accept_greedy(cuda(am.astype(np.int32)), cuda(tok.astype(np.int32)) if len(tok) else None,
                          cuda(par) if par is not None else None, M, ot, oc)
        outs.append((ot, oc))
    status_ok()
    for (am, tok, par), (ot, oc) in zip(cases, outs):
        ref = oracle.accept_greedy_chain(am, tok) if par is None else oracle.accept_greedy_tree(am, tok, par)
        n = int(host(oc)[0])
        assert list(host(ot)[:n]) == list(ref)


@pytest.mark.parametrize("certainty", [False, True])
@pytest.mark.parametrize("stats", ["given", "recomputed"])
def test_accept_sample_bit_exact_small_vocab(sdv, certainty, stats):
    V, K = 16, 3
    l = sdgen.normal(sdgen.key(131), (K + 1, V)) * 1.5
    qp = None if certainty else np.stack(
        [oracle.softmax_probs(l[i] + sdgen.normal(sdgen.key(132, i), (V,))) for i in range(K)])
    m, z, _ = oracle.softmax_stats(l, 1.0)
    ld = cuda(l)
    qd = cuda(qp) if qp is not None else None
    rmd, rzd = (cuda(m), cuda(z)) if stats == "given" else (None, None)
    rng = np.random.default_rng(133)
    runs = []
    for t in range(300):
        dr = rng.integers(0, V, K).astype(np.int32)
        ot = torch.full((K + 1,), -7, dtype=torch.int32, device="cuda")
        oc = torch.zeros(1, dtype=torch.int32, device="cuda")
        sdv.accept_sample(ld, K, cuda(dr), ot, oc, q_probs=qd, row_max=rmd, row_sumexp=rzd, seed=99,
                          base_pos=t * (K + 1))
        runs.append((dr, ot, oc))
    status_ok()
    for t, (dr, ot, oc) in enumerate(runs):
        ref = oracle.accept_sample(l, qp, dr, 1.0, 99, t * (K + 1))
        n = int(host(oc)[0])
        assert list(host(ot)[:n]) == list(ref), t


@pytest.mark.parametrize("certainty", [False, True])
def test_accept_sample_bit_exact_full_vocab(sdv, certainty):
    V, K = 151936, 4
    l = sdgen.normal(sdgen.key(134), (K + 1, V)) * 3
    qp = None if certainty else np.stack(
        [oracle.softmax_probs(l[i] + sdgen.normal(sdgen.key(135, i), (V,))) for i in range(K)])
    rng = np.random.default_rng(136)
    ld = cuda(l)
    qd = cuda(qp) if qp is not None else None
    for t in range(12):
        # half of the drafts are the row's argmax (likely kept), half are random (likely rejected)
        dr = np.where(rng.random(K) < 0.5, np.argmax(l[:K], axis=1), rng.integers(0, V, K)).astype(np.int32)
        ot = torch.full((K + 1,), -7, dtype=torch.int32, device="cuda")
        oc = torch.zeros(1, dtype=torch.int32, device="cuda")
        sdv.accept_sample(ld, K, cuda(dr), ot, oc, q_probs=qd, temperature=1.0, seed=5 + t, base_pos=1000 * t)
        ref = oracle.accept_sample(l, qp, dr, 1.0, 5 + t, 1000 * t)
        status_ok()
        n = int(host(oc)[0])
        assert list(host(ot)[:n]) == list(ref), t


def test_bounded_wait_reports_timeout(sdv):
    assert sdv.device_status() == 0
    sdv.debug_wait_timeout(2_000_000)  # 2 ms
    assert sdv.device_status() == 4    # SD_ETIMEOUT, and the word is cleared
    assert sdv.device_status() == 0


# ---------------------------------------------------------------------------
# rejection sampling against a top-k / top-p filtered target
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("certainty", [False, True])
@pytest.mark.parametrize("top_k,top_p", [(1, 1.0), (5, 0.8), (20, 0.95), (32, 1.0), (32, 0.3)])
def test_accept_sample_topk_bit_exact_small_vocab(sdv, certainty, top_k, top_p):
    V, K = 64, 3
    l = sdgen.normal(sdgen.key(150), (K + 1, V)) * 1.5
    l[:, 7] = l[:, 9] = l.max(axis=1)  # ties at the top, broken by the lower index
    qp = None if certainty else np.stack(
        [oracle.softmax_probs(l[i] + sdgen.normal(sdgen.key(151, i), (V,))) for i in range(K)])
    ld = cuda(l)
    qd = cuda(qp) if qp is not None else None
    rng = np.random.default_rng(152)
    runs = []
    for t in range(120):
        am = np.argmax(l[:K], axis=1)
        dr = np.where(rng.random(K) < 0.5, am, rng.integers(0, V, K)).astype(np.int32)
        ot = torch.full((K + 1,), -7, dtype=torch.int32, device="cuda")
        oc = torch.zeros(1, dtype=torch.int32, device="cuda")
        sdv.accept_sample_topk(ld, K, cuda(dr), ot, oc, top_k, top_p, q_probs=qd, temperature=0.9, seed=31,
                               base_pos=t * (K + 1))
        runs.append((dr, ot, oc))
    status_ok()
    for t, (dr, ot, oc) in enumerate(runs):
        ref = oracle.accept_sample_topk(l, qp, dr, 0.9, top_k, top_p, 31, t * (K + 1))
        n = int(host(oc)[0])
        assert list(host(ot)[:n]) == list(ref), t


@pytest.mark.parametrize("certainty", [False, True])
def test_accept_sample_topk_bit_exact_full_vocab(sdv, certainty):
    V, K = 151936, 4
    l = sdgen.normal(sdgen.key(153), (K + 1, V)) * 3
    qp = None if certainty else np.stack(
        [oracle.softmax_probs(l[i] + sdgen.normal(sdgen.key(154, i), (V,))) for i in range(K)])
    ld = cuda(l)
    qd = cuda(qp) if qp is not None else None
    rng = np.random.default_rng(155)
    for t in range(8):
        # the drafts: a row's best token (likely kept), its second best, or a random one (rejected)
        order = np.argsort(-l[:K], axis=1, kind="stable")
        pick = rng.integers(0, 3, K)
        dr = np.where(pick == 0, order[:, 0], np.where(pick == 1, order[:, 1], rng.integers(0, V, K))).astype(np.int32)
        ot = torch.full((K + 1,), -7, dtype=torch.int32, device="cuda")
        oc = torch.zeros(1, dtype=torch.int32, device="cuda")
        sdv.accept_sample_topk(ld, K, cuda(dr), ot, oc, 20, 0.95, q_probs=qd, temperature=1.0, seed=9 + t,
                               base_pos=500 * t)
        ref = oracle.accept_sample_topk(l, qp, dr, 1.0, 20, 0.95, 9 + t, 500 * t)
        status_ok()
        n = int(host(oc)[0])
        assert list(host(ot)[:n]) == list(ref), t


def test_accept_sample_topk_argument_checks(sdv):
    l = torch.zeros((2, 8), dtype=torch.float32, device="cuda")
    d = torch.zeros(1, dtype=torch.int32, device="cuda")
    ot = torch.zeros(2, dtype=torch.int32, device="cuda")
    oc = torch.zeros(1, dtype=torch.int32, device="cuda")
    for k, p in ((0, 1.0), (33, 1.0), (4, 0.0), (4, 1.5)):
        with pytest.raises(sdv.SdError):
            sdv.accept_sample_topk(l, 1, d, ot, oc, k, p)


@pytest.mark.parametrize("K", [0, 2])
def test_accept_sample_topk_vocab_smaller_than_k(sdv, K):
    """top_k = 32 over an 8-token vocabulary: every token is a candidate; K = 0 draws the bonus token only."""
    V = 8
    l = sdgen.normal(sdgen.key(156), (K + 1, V)) * 2
    ld = cuda(l)
    rng = np.random.default_rng(157)
    for t in range(40):
        dr = rng.integers(0, V, K).astype(np.int32)
        ot = torch.full((K + 1,), -7, dtype=torch.int32, device="cuda")
        oc = torch.zeros(1, dtype=torch.int32, device="cuda")
        sdv.accept_sample_topk(ld, K, cuda(dr) if K else None, ot, oc, 32, 0.5, temperature=1.3, seed=t, base_pos=3 * t)
        ref = oracle.accept_sample_topk(l, None, dr, 1.3, 32, 0.5, t, 3 * t)
        status_ok()
        n = int(host(oc)[0])
        assert list(host(ot)[:n]) == list(ref), t


def test_accept_sample_topk_many_ties(sdv):
    """Integer-valued logits with many exact ties and signed zeros: candidates, nucleus and draws
    bit-exact against the oracle."""
    rng = np.random.default_rng(158)
    for trial in range(24):
        V, K = int(rng.integers(1, 3000)), int(rng.integers(0, 4))
        l = rng.integers(-4, 5, (K + 1, V)).astype(np.float32)
        l[rng.random((K + 1, V)) < 0.1] = -0.0
        T = float(rng.choice([1.0, 0.5, 2.0]))
        k, p = int(rng.choice([1, 3, 20, 32])), float(rng.choice([1.0, 0.9, 0.5]))
        dr = rng.integers(0, V, K).astype(np.int32)
        ot = torch.full((K + 1,), -7, dtype=torch.int32, device="cuda")
        oc = torch.zeros(1, dtype=torch.int32, device="cuda")
        sdv.accept_sample_topk(cuda(l), K, cuda(dr) if K else None, ot, oc, k, p, temperature=T, seed=trial,
                               base_pos=7 * trial)
        ref = oracle.accept_sample_topk(l, None, dr, T, k, p, trial, 7 * trial)
        status_ok()
        n = int(host(oc)[0])
        assert list(host(ot)[:n]) == list(ref), trial
