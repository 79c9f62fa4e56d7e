"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each test fixes an oracle function to an independent truth: a numpy library
routine applied to integer codes the test chose itself, a closed form, the
worked example on the Kinetic page, published Philox known-answer vectors,
exact enumeration of the acceptance rule over its uniform grid, or a large
Monte-Carlo run.  A plausible mistake in the oracle (a swapped nibble, a
dropped residual, a wrong comparison, a wrong Philox word) fails one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import sdgen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# helpers: pack chosen integer codes into GGUF block bytes (format definition)
# ---------------------------------------------------------------------------

def pack_blocks(qtype, wq, d16):
    """wq int [N][K] (Q8_0: -127..127; 4-bit: -8..7), d16 float16 [N][K/32] -> block bytes."""
    N, K = wq.shape
    KB = K // 32
    bb = oracle.BLOCK_BYTES[qtype]
    out = np.zeros((N, KB, bb), dtype=np.uint8)
    out[:, :, 0:2] = d16.astype(np.float16).view(np.uint8).reshape(N, KB, 2)
    w = wq.reshape(N, KB, 32)
    if qtype == oracle.Q8_0:
        out[:, :, 2:] = w.astype(np.int8).view(np.uint8)
    else:
        code = (w + 8).astype(np.uint8)
        out[:, :, 2:] = code[:, :, :16] | (code[:, :, 16:] << 4)
    return out.reshape(N, KB * bb)


def rand_case(rng, qtype, N, K, M):
    lim = 127 if qtype == oracle.Q8_0 else 8
    wq = rng.integers(-lim, lim if qtype == oracle.Q4_32 else lim + 1, size=(N, K))
    d16 = (rng.random((N, K // 32)) * 1e-3 + 1e-5).astype(np.float16)
    aq = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    sa = (rng.random((M, K // 32)) * 0.05 + 1e-3).astype(np.float32)
    return wq, d16, aq, sa


# ---------------------------------------------------------------------------
# fp16 decode
# ---------------------------------------------------------------------------

def test_f16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(b)) for b in bits[::7]], dtype=np.float32)
    r = ref[::7]
    nan = np.isnan(r)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), r[~nan].view(np.uint32))


# ---------------------------------------------------------------------------
# block dots and dequant: numpy integer matmul on codes the test chose
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("qtype", [oracle.Q8_0, oracle.Q4_32])
def test_block_dots_match_numpy_integer_matmul(qtype):
    rng = np.random.default_rng(1)
    N, K, M = 37, 256, 5
    wq, d16, aq, _ = rand_case(rng, qtype, N, K, M)
    blocks = pack_blocks(qtype, wq, d16)
    dots = oracle.block_dots(qtype, blocks, N, K, aq)
    KB = K // 32
    ref = np.einsum("nbi,mbi->mnb", wq.reshape(N, KB, 32).astype(np.int64),
                    aq.reshape(M, KB, 32).astype(np.int64))
    assert np.array_equal(dots, ref)
    bound = 516128 if qtype == oracle.Q8_0 else 32 * 8 * 127
    assert np.abs(dots).max() <= bound


def test_block_dots_extremes_and_q4_identity():
    # extremes: every product at its maximum magnitude
    N, K = 2, 32
    wq8 = np.full((N, K), 127)
    wq8[1] = -127
    a = np.full((1, K), -127, dtype=np.int8)
    blk = pack_blocks(oracle.Q8_0, wq8, np.ones((N, 1), np.float16))
    assert list(oracle.block_dots(oracle.Q8_0, blk, N, K, a)[0, :, 0]) == [-516128, 516128]
    # 4-bit: sum (code-8) a == sum code*a - 8 sum a
    rng = np.random.default_rng(2)
    wq = rng.integers(-8, 8, size=(3, 64))
    aq = rng.integers(-127, 128, size=(2, 64)).astype(np.int8)
    blk = pack_blocks(oracle.Q4_32, wq, np.ones((3, 2), np.float16))
    dots = oracle.block_dots(oracle.Q4_32, blk, 3, 64, aq).astype(np.int64)
    code = (wq + 8).reshape(3, 2, 32).astype(np.int64)
    a = aq.reshape(2, 2, 32).astype(np.int64)
    alt = np.einsum("nbi,mbi->mnb", code, a) - 8 * a.sum(axis=2)[:, None, :]
    assert np.array_equal(dots, alt)


@pytest.mark.parametrize("qtype", [oracle.Q8_0, oracle.Q4_32])
def test_dequant_matches_codes_times_fp16_scale(qtype):
    rng = np.random.default_rng(3)
    wq, d16, _, _ = rand_case(rng, qtype, 9, 128, 1)
    v = oracle.dequant(qtype, pack_blocks(qtype, wq, d16), 9, 128)
    ref = (np.repeat(d16.astype(np.float32), 32, axis=1).astype(np.float64) * wq).astype(np.float32)
    assert np.array_equal(v, ref)


@pytest.mark.parametrize("qtype", [oracle.Q8_0, oracle.Q4_32])
def test_generator_roundtrip_error_bound(qtype):
    # weights ~ N(0, 0.02) quantised by the generator: |w - dequant| <= d/2 (plus fp16 rounding of d)
    N, K = 64, 512
    k = sdgen.key(99, qtype)
    w = sdgen.normal(k, (N, K), std=0.02)
    blocks = sdgen.quantize(qtype, w)
    assert np.array_equal(blocks, sdgen.quantized_normal(qtype, k, N, K, std=0.02))
    v = oracle.dequant(qtype, blocks, N, K)
    amax = np.abs(w.reshape(N, K // 32, 32)).max(axis=2)
    d = amax / (127.0 if qtype == oracle.Q8_0 else 7.5)
    lev = 127 if qtype == oracle.Q8_0 else 8
    bound = np.repeat(d * 0.5 + amax * 2.0 ** -11 * (lev / (lev - 1)) + 1e-12, 32, axis=1)
    assert np.all(np.abs(w - v) <= bound)


# ---------------------------------------------------------------------------
# multi-position matmul: numpy float64 matmul of dequantised operands
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("qtype", [oracle.Q8_0, oracle.Q4_32])
@pytest.mark.parametrize("with_residual", [False, True])
def test_qmatmul_matches_numpy_float64(qtype, with_residual):
    rng = np.random.default_rng(4)
    N, K, M = 45, 320, 5
    wq, d16, aq, sa = rand_case(rng, qtype, N, K, M)
    blocks = pack_blocks(qtype, wq, d16)
    res = rng.standard_normal((M, N)).astype(np.float32) if with_residual else None
    y, ab = oracle.qmatmul(qtype, blocks, N, K, aq, sa, residual=res)
    W = oracle.dequant(qtype, blocks, N, K).astype(np.float64)
    A = aq.astype(np.float64) * np.repeat(sa.astype(np.float64), 32, axis=1)
    ref = A @ W.T
    absref = np.abs(A) @ np.abs(W).T
    if res is not None:
        ref = ref + res
        absref = absref + np.abs(res)
    assert np.all(np.abs(y.astype(np.float64) - ref) <= 2.0 ** -24 * np.abs(ref) + 1e-12 * absref + 1e-30)
    assert np.all(ab >= np.abs(y) * (1 - 1e-6))
    # the absolute bound is >= the per-block absolute sum, and equals it for sign-aligned data
    assert np.all(ab <= absref * (1 + 1e-12) + 1e-30)


# ---------------------------------------------------------------------------
# RMSNorm + requantisation
# ---------------------------------------------------------------------------

def test_rmsnorm_constant_row_closed_form():
    K = 1024
    c = 0.5  # c*c and all partial sums are exact, so mean == c*c exactly
    x = np.full((1, K), c, dtype=np.float32)
    w = sdgen.norm_weight(sdgen.key(5), K)
    q, s = oracle.rmsnorm_quant(x, w, 1e-6)
    inv = np.float32(1.0) / np.sqrt(np.float32(c * c) + np.float32(1e-6), dtype=np.float32)
    y = (np.float32(c) * inv) * w
    closed = w.astype(np.float64) * c / math.sqrt(c * c + 1e-6)
    assert np.all(np.abs(y - closed) <= 4 * np.spacing(np.abs(closed).astype(np.float32)))
    yb = y.reshape(1, K // 32, 32)
    # block scale: max|y| / 127 in closed form, reached within three roundings (inv, /127, *inv)
    d_closed = np.abs(closed.reshape(1, K // 32, 32)).max(axis=2) / 127.0
    assert np.all(np.abs(s - d_closed) <= 3 * np.spacing(d_closed.astype(np.float32)))
    # codes: the block's largest |w| maps to +-127, every value within half a step of y
    qb = q.reshape(1, K // 32, 32).astype(np.int32)
    wb = np.abs(w.reshape(1, K // 32, 32))
    assert np.all(np.abs(np.take_along_axis(qb, wb.argmax(axis=2)[..., None], axis=2)) == 127)
    deq = qb.astype(np.float64) * s[..., None]
    assert np.all(np.abs(deq - closed.reshape(1, K // 32, 32)) <= s[..., None] * (0.5 + 1e-5))


@pytest.mark.parametrize("c", [0.5, -4.0, 2.0 ** -20])
def test_rmsnorm_power_of_two_row_normalises_to_w_exactly(c):
    """Closed form with every step exact: a constant row x = c = +-2^k with eps = 0 has mean square
    c^2 (exact partial sums), inv = 1/|c| (a power of two), so the normalised row is sign(c) w
    exactly; its block scales are exactly fl(max|w| / 127) and its codes the requantisation of
    sign(c) w.  A wrong divisor of the mean, a missing square root or a misplaced row factor
    changes the scales."""
    K = 5120
    x = np.full((2, K), c, dtype=np.float32)
    w = sdgen.norm_weight(sdgen.key(5, 1), K)
    q, s = oracle.rmsnorm_quant(x, w, 0.0)
    yn = (np.sign(c) * w).astype(np.float32)
    qr, sr = oracle.rmsnorm_quant(np.vstack([yn, yn]), None)  # requantisation alone of sign(c) w
    d = (np.abs(w.reshape(K // 32, 32)).max(axis=1) / np.float32(127.0)).astype(np.float32)
    assert np.array_equal(s[0], d) and np.array_equal(s[1], d)
    assert np.array_equal(sr[0], d)
    assert np.array_equal(q, qr)
    assert np.all(np.abs(q.reshape(2, K // 32, 32)).max(axis=2) == 127)


def test_rmsnorm_codes_equal_the_plain_definition_except_at_ties():
    """Reading R4 forms the codes from t = x w and the scale as inv max|t| / 127; the plain
    definition requantises y = (x inv) w.  On the bench's input rows at the RMSNorm sites of the
    oracle's own pass: live on the first four layers, and from the stored statistics of all 129
    sites of the 64-layer stack (tests/golden/make_rmsnorm_ties.py, which calls only the oracle).
    Every code that differs differs by one step and sits within TIE of a half-integer of the plain
    quotient; scales agree within 4 fp32 ulps (the two orders' few roundings)."""
    import json
    import os

    from _rmsnorm_ties import TIE, compare_site, stack_sites
    spec = sdgen.StackSpec()
    live = [dict(compare_site(x, w, sdgen.EPS), site=n) for n, x, w in stack_sites(spec, 5, 4)]
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "rmsnorm_ties_27b_stack_m5.json")))
    sites = g["sites"]
    assert len(sites) == 2 * spec.layers + 1 and g["tie_band"] == TIE
    assert live == sites[:len(live)]  # the stored statistics are those of the current oracle
    for r in live + sites:
        assert r["max_step"] <= 1, r
        assert r["max_tie_distance_of_differing"] <= TIE, r
        assert r["max_scale_ulps"] <= 4.0, r
    assert g["total_differing"] == sum(r["differing"] for r in sites)
    assert g["tie_rate"] < 1e-5


@pytest.mark.parametrize("K", [1024, 5120, 17408])
def test_rmsnorm_quant_vs_float64_definition(K):
    M = 3
    x = sdgen.normal(sdgen.key(6, K), (M, K))
    x[1] *= 40.0
    x[2, :32] = 0.0  # an all-zero block: d = 0, q = 0
    w = sdgen.norm_weight(sdgen.key(7, K), K)
    q, s = oracle.rmsnorm_quant(x, w, 1e-6)
    x64 = x.astype(np.float64)
    y = x64 / np.sqrt((x64 ** 2).mean(axis=1, keepdims=True) + 1e-6) * w
    deq = q.astype(np.float64) * np.repeat(s.astype(np.float64), 32, axis=1)
    tol = np.repeat(s.astype(np.float64), 32, axis=1) * 0.5 + np.abs(y) * 1e-6 + 1e-30
    assert np.all(np.abs(deq - y) <= tol)
    qb = np.abs(q.reshape(M, K // 32, 32).astype(np.int32)).max(axis=2)
    assert np.all((qb == 127) | (s == 0))
    # requantise-only mode is the identity norm
    q2, s2 = oracle.rmsnorm_quant(x, None)
    deq2 = q2.astype(np.float64) * np.repeat(s2.astype(np.float64), 32, axis=1)
    assert np.all(np.abs(deq2 - x64) <= np.repeat(s2, 32, axis=1) * 0.5 * (1 + 1e-6) + 1e-30)


# ---------------------------------------------------------------------------
# canonical exponential
# ---------------------------------------------------------------------------

def test_cexp_within_2ulp_of_fp64_exp():
    xs = np.concatenate([np.linspace(-103.9, 88.7, 200001, dtype=np.float32),
                         np.float32(np.random.default_rng(8).standard_normal(20000) * 5)])
    got = oracle.cexp(xs).astype(np.float64)
    ref = np.exp(xs.astype(np.float64))
    fin = np.isfinite(got) & (ref < 3.0e38) & (ref > 1.2e-38)
    ulp = np.spacing(ref[fin].astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(got[fin] - ref[fin]) / ulp) <= 2.0
    assert oracle.cexp([0.0])[0] == 1.0
    assert oracle.cexp([-200.0])[0] == 0.0 and np.isinf(oracle.cexp([120.0])[0])
    # subnormal range is rounded once: within one subnormal step
    xs2 = np.linspace(-103.0, -88.0, 2001, dtype=np.float32)
    got2 = oracle.cexp(xs2).astype(np.float64)
    assert np.all(np.abs(got2 - np.exp(xs2.astype(np.float64))) <= 2.0 ** -149 * 2 + np.exp(xs2.astype(np.float64)) * 2.5e-7)


def test_silu_mul_requant_vs_float64():
    M, F = 2, 1024
    g = sdgen.normal(sdgen.key(9), (M, F)) * 4
    u = sdgen.normal(sdgen.key(10), (M, F))
    g[0, :8] = [0.0, -0.0, 90.0, -90.0, 1e-30, -1e-30, 20.0, -20.0]
    q, s, h = oracle.silu_mul_requant(g, u)
    g64 = g.astype(np.float64)
    ref = g64 / (1 + np.exp(-g64)) * u
    assert np.all(np.abs(h - ref) <= 4 * np.spacing(np.abs(ref).astype(np.float32)) + 1e-37)
    deq = q.astype(np.float64) * np.repeat(s.astype(np.float64), 32, axis=1)
    assert np.all(np.abs(deq - h) <= np.repeat(s, 32, axis=1) * 0.5 * (1 + 1e-6) + 1e-30)


# ---------------------------------------------------------------------------
# softmax statistics and argmax
# ---------------------------------------------------------------------------

def test_softmax_uniform_logits():
    V = 151936
    l = np.full((2, V), 3.25, dtype=np.float32)
    m, z, a = oracle.softmax_stats(l, 1.0)
    assert list(m) == [3.25, 3.25] and list(z) == [float(V)] * 2 and list(a) == [0, 0]
    p = oracle.softmax_probs(l[0])
    assert np.all(p == np.float32(1.0) / np.float32(V))


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_softmax_stats_vs_float64(T):
    V = 151936
    l = sdgen.normal(sdgen.key(11), (3, V)) * 3
    l[1, 777] = l[1].max() + 1.0
    l[1, 99999] = l[1, 777]  # tie: lowest index wins
    l[2, V - 1] = 40.0       # maximum in the short last tile
    m, z, a = oracle.softmax_stats(l, T)
    zz = l.astype(np.float64) / T
    mref = zz.max(axis=1)
    zref = np.exp(zz - mref[:, None]).sum(axis=1)
    assert np.array_equal(m, (l / np.float32(T)).max(axis=1))
    assert np.all(np.abs(z - zref) <= 1e-5 * zref)
    assert list(a) == list(np.argmax(l, axis=1)) and a[1] == 777 and a[2] == V - 1
    p = oracle.softmax_probs(l[0], T)
    pref = np.exp(zz[0] - mref[0]) / zref[0]
    assert abs(p.astype(np.float64).sum() - 1.0) < 1e-4
    assert np.all(np.abs(p - pref) <= 1e-5 * pref + 1e-12)


# ---------------------------------------------------------------------------
# greedy acceptance
# ---------------------------------------------------------------------------

def test_worked_example_rad1():
    g = json.load(open(os.path.join(GOLDEN, "rad1_worked_example.json")))
    for case in g["cases"].values():
        kept = oracle.accept_greedy_chain(np.array(case["argmax"]), np.array(case["drafts"]))
        assert list(kept) == case["kept"]
        assert len(kept) - 1 == case["accepted"]


def test_greedy_chain_edges():
    am = np.array([5, 6, 7, 8], dtype=np.int32)
    assert list(oracle.accept_greedy_chain(am[:1], np.array([], np.int32))) == [5]          # K = 0
    assert list(oracle.accept_greedy_chain(am, np.array([5, 6, 7]))) == [5, 6, 7, 8]        # all kept + bonus
    assert list(oracle.accept_greedy_chain(am, np.array([4, 6, 7]))) == [5]                 # first rejected
    assert list(oracle.accept_greedy_chain(am, np.array([5, 6, 0]))) == [5, 6, 7]           # last rejected


def test_greedy_tree_chain_special_case_and_example():
    rng = np.random.default_rng(12)
    for _ in range(200):
        K = int(rng.integers(0, 8))
        am = rng.integers(0, 4, size=K + 1).astype(np.int32)
        dr = rng.integers(0, 4, size=K).astype(np.int32)
        chain = oracle.accept_greedy_chain(am, dr)
        tokens = np.concatenate([[9], dr]).astype(np.int32)
        parent = np.arange(-1, K, dtype=np.int32)
        assert list(oracle.accept_greedy_tree(am, tokens, parent)) == list(chain)
    # 16-node tree: root, binary depth 3, spine below node 7.  Argmax chain along 0->1->3->7->15.
    parent, depth = sdgen.tree16(0)
    am = np.arange(100, 116, dtype=np.int32)
    tokens = np.full(16, 1, dtype=np.int32)
    tokens[1], tokens[3], tokens[7], tokens[15] = am[0], am[1], am[3], am[7]
    tokens[2] = am[0]          # a sibling that also matches the root's argmax
    tokens[5] = am[2]          # ... and its child too (depth 2), shorter than the main path
    kept = oracle.accept_greedy_tree(am, tokens, parent)
    assert list(kept) == [am[0], am[1], am[3], am[7], am[15]]
    # equal-depth tie: lowest BFS index wins
    tokens2 = np.full(16, 1, dtype=np.int32)
    tokens2[1], tokens2[2] = am[0], am[0]
    tokens2[3], tokens2[5] = am[1], am[2]
    assert list(oracle.accept_greedy_tree(am, tokens2, parent)) == [am[0], am[1], am[3]]


def test_drafted_greedy_equals_plain_greedy_toy_model():
    """A toy deterministic model: embedding -> 2-layer stack -> head.  Decoding with
    drafts verified in one batched pass gives exactly the plain greedy sequence."""
    Vt, H, F, L = 256, 64, 96, 2
    E = sdgen.normal(sdgen.key(20), (Vt, H))
    wts = []
    for l in range(L):
        wts.append(dict(qkv=sdgen.quantized_normal(sdgen.Q4_32, sdgen.key(21, l), 3 * H, H, std=0.2),
                        o=sdgen.quantized_normal(sdgen.Q4_32, sdgen.key(22, l), H, H, std=0.2),
                        gate_up=sdgen.quantized_normal(sdgen.Q4_32, sdgen.key(23, l), 2 * F, H, std=0.2),
                        down=sdgen.quantized_normal(sdgen.Q4_32, sdgen.key(24, l), H, F, std=0.2)))
    n1 = [sdgen.norm_weight(sdgen.key(25, l), H) for l in range(L)]
    n2 = [sdgen.norm_weight(sdgen.key(26, l), H) for l in range(L)]
    fn = sdgen.norm_weight(sdgen.key(27), H)
    hw = sdgen.quantized_normal(sdgen.Q8_0, sdgen.key(28), Vt, H, std=0.2)

    def argmax_rows(tokens):
        h = E[np.asarray(tokens)]
        for l in range(L):
            h = oracle.stack_layer(h, wts[l], n1[l], n2[l], H, F)
        return oracle.head(h, fn, hw, Vt, H)[1]

    t0, steps = 3, 24
    plain = [t0]
    for _ in range(steps):
        plain.append(int(argmax_rows([plain[-1]])[0]))
    rng = np.random.default_rng(29)
    out = [t0]
    K = 4
    while len(out) < steps + 1:
        cur = out[-1]
        # noisy drafter: the true next token with prob 0.75, else random
        drafts = []
        prev = cur
        for _ in range(K):
            nxt = int(argmax_rows([prev])[0]) if rng.random() < 0.75 else int(rng.integers(0, Vt))
            drafts.append(nxt)
            prev = nxt
        am = argmax_rows([cur] + drafts)
        out.extend(int(t) for t in oracle.accept_greedy_chain(am, np.array(drafts, np.int32)))
    assert out[:steps + 1] == plain


# ---------------------------------------------------------------------------
# Philox4x32-10
# ---------------------------------------------------------------------------

def test_philox_known_answer_vectors():
    g = json.load(open(os.path.join(GOLDEN, "philox4x32_10_kat.json")))
    for v in g["vectors"]:
        out = oracle.philox4x32_10([int(x, 16) for x in v["ctr"]], [int(x, 16) for x in v["key"]])
        assert [f"{int(x):08x}" for x in out] == v["out"]


def test_philox_uniforms_properties():
    n = 200000
    ua = np.empty(n)
    ur = np.empty(n)
    for i in range(n):
        ua[i], ur[i] = oracle.uniforms(1234, i)
    for u in (ua, ur):
        assert u.min() >= 0.0 and u.max() < 1.0
        assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))
        h, _ = np.histogram(u, bins=64, range=(0, 1))
        chi2 = ((h - n / 64) ** 2 / (n / 64)).sum()
        assert chi2 < 120  # 63 dof; p ~ 1e-5
    assert abs(np.corrcoef(ua, ur)[0, 1]) < 0.01
    assert abs(np.corrcoef(ua[:-1], ua[1:])[0, 1]) < 0.01


# ---------------------------------------------------------------------------
# rejection sampling: exact enumeration over the uniform grid + Monte Carlo
# ---------------------------------------------------------------------------

def _grid_law(fn, n_bits=24):
    """Exact law of fn(u) over the uniform grid u = k 2^-24 (k < 2^24) for fn piecewise
    constant in u with few pieces: binary-search the breakpoints."""
    N = 1 << n_bits
    law = {}
    k = 0
    while k < N:
        tok = fn(k / N)
        lo, hi = k, N
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if fn(mid / N) == tok:
                lo = mid
            else:
                hi = mid
        law[tok] = law.get(tok, 0) + (hi - k)
        k = hi
    return {t: c / N for t, c in law.items()}


@pytest.mark.parametrize("certainty", [False, True])
def test_rejection_sampling_exact_law(certainty):
    """Emitted-token law of one verified draft, enumerated exactly over the uniforms,
    equals the target distribution p (the rejection-sampling guarantee)."""
    V = 16
    l = sdgen.normal(sdgen.key(40), (2, V)) * 1.5
    p = oracle.softmax_probs(l[0]).astype(np.float64)
    qrow = None if certainty else oracle.softmax_probs(l[0] + sdgen.normal(sdgen.key(41), (V,)))
    qfull = None if certainty else qrow[None, :]
    top = 1.0 - 2.0 ** -24
    for x in range(V) if certainty else [None]:
        law = np.zeros(V)
        for xd in ([x] if certainty else range(V)):
            dr = np.array([xd], np.int32)
            qx = 1.0 if certainty else float(qrow[xd])
            acc = _grid_law(lambda u: len(oracle.accept_sample_u(l, qfull, dr, 1.0, [u, 0.0], [0.0, 0.0])) == 2)
            pacc = acc.get(True, 0.0)
            assert abs(pacc - min(1.0, p[xd] / qx)) <= 2.0 ** -23
            weight = 1.0 if certainty else qx
            law[xd] += weight * pacc
            if pacc < 1.0:
                res = _grid_law(lambda u: int(oracle.accept_sample_u(l, qfull, dr, 1.0, [top, 0.0], [u, 0.0])[0]))
                qv = np.eye(V)[xd] if certainty else qrow.astype(np.float64)
                w = np.maximum(0.0, p - qv)
                r = w / w.sum()
                for t, pr in res.items():
                    assert abs(pr - r[t]) <= 2e-6
                    law[t] += weight * (1 - pacc) * pr
        assert np.all(np.abs(law - p) <= 4e-6), np.abs(law - p).max()


@pytest.mark.parametrize("certainty", [False, True])
def test_rejection_sampling_monte_carlo_1e6(certainty):
    V, K, n = 16, 2, 1_000_000
    l = sdgen.normal(sdgen.key(50), (K + 1, V)) * 1.5
    if certainty:
        q = None
        # a fixed certainty draft per row (the drafter's single guess)
        drafts = np.tile(np.array([3, 11], np.int32), (n, 1))
    else:
        q = np.stack([oracle.softmax_probs(l[i] + sdgen.normal(sdgen.key(51, i), (V,))) for i in range(K)])
        # drafts sampled from q (input synthesis, independent of the verify uniforms)
        u = sdgen.uniforms(sdgen.key(52), n * K).reshape(n, K)
        cdf = np.cumsum(q.astype(np.float64), axis=1)
        drafts = np.stack([np.minimum(np.searchsorted(cdf[i] / cdf[i, -1], u[:, i], side="right"), V - 1)
                           for i in range(K)], axis=1).astype(np.int32)
    counts, toks = oracle.accept_sample_trials(l, q, drafts, 1.0, seed=777, base_pos=0)
    assert np.all((counts >= 1) & (counts <= K + 1))
    p0 = oracle.softmax_probs(l[0]).astype(np.float64)
    p1 = oracle.softmax_probs(l[1]).astype(np.float64)
    for p, sel in ((p0, toks[:, 0]), (p1, toks[counts >= 2, 1])):
        N = sel.size
        freq = np.bincount(sel, minlength=V) / N
        sigma = np.sqrt(p * (1 - p) / N)
        assert np.all(np.abs(freq - p) <= 3 * sigma + 1e-12), (freq - p) / sigma
        chi2 = (((freq - p) * N) ** 2 / (p * N)).sum()
        assert chi2 < 45  # 15 dof: p ~ 1e-4


# ---------------------------------------------------------------------------
# rejection sampling against a top-k / top-p filtered target
# ---------------------------------------------------------------------------

def test_filter_topk_topp_worked_example():
    """z = (1, 3, 2, 3, -1): ties broken by index, closed-form probabilities, the nucleus cut."""
    l = np.array([1.0, 3.0, 2.0, 3.0, -1.0], np.float32)
    tok, p = oracle.filter_topk_topp(l, 1.0, 3, 1.0)
    assert list(tok) == [1, 3, 2]
    e = np.exp(np.array([0.0, 0.0, -1.0]))
    np.testing.assert_allclose(p, e / e.sum(), rtol=4e-7)
    tok, p = oracle.filter_topk_topp(l, 1.0, 3, 0.5)  # 1/2.37 < 0.5 <= 2/2.37: two candidates
    assert list(tok) == [1, 3] and list(p) == [0.5, 0.5]
    tok, p = oracle.filter_topk_topp(l, 1.0, 5, 1e-9)  # the nucleus is never empty
    assert list(tok) == [1] and list(p) == [1.0]


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_filter_without_cuts_is_the_softmax(T):
    V = 16
    l = sdgen.normal(sdgen.key(60), (V,)) * 2
    tok, p = oracle.filter_topk_topp(l, T, V, 1.0)
    z = l.astype(np.float32) / np.float32(T)
    assert list(tok) == list(np.lexsort((np.arange(V), -z)))
    ref = np.exp(z.astype(np.float64) - z.max())
    ref /= ref.sum()
    np.testing.assert_allclose(p, ref[tok], rtol=1e-6)


def test_filter_nucleus_is_the_shortest_prefix():
    V = 64
    l = sdgen.normal(sdgen.key(61), (V,)) * 3
    for top_p in (0.3, 0.6, 0.9, 0.99):
        tok, p = oracle.filter_topk_topp(l, 1.0, 32, top_p)
        full_tok, full_p = oracle.filter_topk_topp(l, 1.0, 32, 1.0)
        assert list(tok) == list(full_tok[:tok.size])
        c = np.cumsum(full_p.astype(np.float64))
        n = tok.size
        assert c[n - 1] >= top_p - 1e-6 and (n == 1 or c[n - 2] < top_p + 1e-6)
        np.testing.assert_allclose(p.sum(), 1.0, rtol=1e-6)


def test_topk1_is_greedy_chain():
    """With top_k = 1 the target is one-hot at the argmax, so any uniforms give the greedy chain rule."""
    V, K = 64, 4
    l = sdgen.normal(sdgen.key(62), (K + 1, V)) * 2
    am = np.argmax(l, axis=1).astype(np.int32)
    rng = np.random.default_rng(63)
    for t in range(40):
        drafts = np.where(rng.random(K) < 0.7, am[:K], rng.integers(0, V, K)).astype(np.int32)
        q = oracle.softmax_probs(l[0] + 0.0)[None, :].repeat(K, 0) if t % 2 else None
        got = oracle.accept_sample_topk(l, q, drafts, 1.0, 1, 1.0, seed=t, base_pos=100 * t)
        assert list(got) == list(oracle.accept_greedy_chain(am, drafts)), t


@pytest.mark.parametrize("certainty", [False, True])
def test_filtered_rejection_sampling_exact_law(certainty):
    """Emitted-token law of one verified draft, enumerated exactly over the uniforms, equals the
    filtered target p' (top_k = 5, top_p = 0.8): the rejection-sampling guarantee for p'."""
    V = 12
    l = sdgen.normal(sdgen.key(64), (2, V)) * 1.5
    tok, pk = oracle.filter_topk_topp(l[0], 1.0, 5, 0.8)
    p = np.zeros(V)
    p[tok] = pk
    qrow = None if certainty else oracle.softmax_probs(l[0] + sdgen.normal(sdgen.key(65), (V,)))
    qfull = None if certainty else qrow[None, :]
    top = 1.0 - 2.0 ** -24
    for x in (range(V) if certainty else [None]):
        law = np.zeros(V)
        for xd in ([x] if certainty else range(V)):
            dr = np.array([xd], np.int32)
            qx = 1.0 if certainty else float(qrow[xd])
            acc = _grid_law(lambda u: len(oracle.accept_sample_topk_u(l, qfull, dr, 1.0, 5, 0.8, [u, 0.0],
                                                                     [0.0, 0.0])) == 2)
            pacc = acc.get(True, 0.0)
            assert abs(pacc - min(1.0, p[xd] / qx)) <= 2.0 ** -23
            weight = 1.0 if certainty else qx
            law[xd] += weight * pacc
            if pacc < 1.0:
                res = _grid_law(lambda u: int(oracle.accept_sample_topk_u(l, qfull, dr, 1.0, 5, 0.8, [top, 0.0],
                                                                          [u, 0.0])[0]))
                qv = np.eye(V)[xd] if certainty else qrow.astype(np.float64)
                w = np.maximum(0.0, p - qv)
                r = w / w.sum() if w.sum() > 0 else p
                for t, pr in res.items():
                    assert abs(pr - r[t]) <= 2e-6
                    law[t] += weight * (1 - pacc) * pr
        if certainty:
            # a certainty drafter's draft x: the law is p' whatever x is
            assert np.all(np.abs(law - p) <= 4e-6), np.abs(law - p).max()
    if not certainty:
        assert np.all(np.abs(law - p) <= 4e-6), np.abs(law - p).max()


def test_filter_candidates_match_a_stable_sort_with_many_ties():
    """Integer-valued logits (many exact ties, -0 and +0 among them): the candidate order is a stable
    sort of z descending, for every top_k, and the probabilities follow the closed form."""
    rng = np.random.default_rng(66)
    for trial in range(30):
        V = int(rng.integers(1, 200))
        l = rng.integers(-4, 5, V).astype(np.float32)
        l[rng.random(V) < 0.1] = -0.0
        T = float(rng.choice([1.0, 0.5, 2.0]))
        z = (l / np.float32(T) + np.float32(0.0)).astype(np.float32)
        order = np.lexsort((np.arange(V), -z))
        for k in (1, 2, 7, 32):
            tok, p = oracle.filter_topk_topp(l, T, k, 1.0)
            kk = min(k, V)
            assert list(tok) == list(order[:tok.size]), (trial, k)
            # the nucleus at top_p = 1: the shortest prefix whose fp32 running sum reaches the total
            # (a tail too small to move the sum is left out; its mass is below 2^-24 of the total)
            e32 = [oracle.cexp(float(z[i] - z[order[0]])) for i in order[:kk]]
            S = np.float32(0.0)
            for x in e32:
                S = np.float32(S + np.float32(x))
            run, n = np.float32(0.0), 0
            while n < kk:
                run = np.float32(run + np.float32(e32[n]))
                n += 1
                if run >= S:
                    break
            assert tok.size == n, (trial, k)
            e = np.exp(z[tok].astype(np.float64) - z[tok[0]])
            np.testing.assert_allclose(p, e / e.sum(), rtol=2e-6)


# ---------------------------------------------------------------------------
# shortlist head: 4-bit copy with per-row error bounds, exact argmax over the candidates
# ---------------------------------------------------------------------------

def _shortlist_case(seed, N=4096, K=1024, M=3):
    w8 = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(seed, 1), N, K)
    x = sdgen.normal(sdgen.key(seed, 2), (M, K))
    q, s = oracle.rmsnorm_quant(x, None)
    return w8, q, s


def _exact_scores(w8, N, K, q, s):
    dots = oracle.block_dots(oracle.Q8_0, w8, N, K, q).astype(np.float64)  # [M][N][KB]
    d = oracle.dequant(oracle.Q8_0, w8, N, K).reshape(N, K // 32, 32)
    dw = np.array([[oracle.f16_to_f32(int(v)) for v in row] for row in
                   np.asarray(w8).reshape(N, K // 32, 34)[:, :, :2].copy().view(np.uint16)[:, :, 0]])
    del d
    return (dots * dw[None] * s.astype(np.float64)[:, None, :]).sum(axis=2)


def test_shortlist_copy_error_is_half_a_step_and_bounded():
    N, K = 256, 512
    w8 = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(70), N, K)
    q4, bound, wnorm = oracle.shortlist_copy(w8, N, K)
    a = oracle.dequant(oracle.Q8_0, w8, N, K).astype(np.float64)
    b = oracle.dequant(oracle.Q4_32, q4, N, K).astype(np.float64)
    d4 = np.asarray(q4).reshape(N, K // 32, 18)[:, :, :2].copy().view(np.uint16)[:, :, 0]
    step = np.vectorize(lambda h: oracle.f16_to_f32(int(h)))(d4).astype(np.float64)
    # d = amax / 7.5 in fp32, rounded to fp16 to nearest even (numpy's conversion)
    amax = np.abs(oracle.dequant(oracle.Q8_0, w8, N, K).reshape(N, K // 32, 32)).max(axis=2).astype(np.float32)
    assert np.array_equal(d4, (amax / np.float32(7.5)).astype(np.float16).view(np.uint16))
    # codes: 8 + round-half-away(w / d) of the fp32 quotient, clamped to [0, 15] (8 where d == 0)
    d32 = step.astype(np.float32)[:, :, None]
    wq = a.astype(np.float32).reshape(N, K // 32, 32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (wq / d32).astype(np.float64)
    want = np.where(d32 > 0, np.clip(np.sign(t) * np.floor(np.abs(t) + 0.5) + 8, 0, 15), 8).astype(np.uint8)
    nib = np.asarray(q4).reshape(N, K // 32, 18)[:, :, 2:]
    got = np.concatenate([nib & 15, nib >> 4], axis=2)
    assert np.array_equal(got, want)
    err = (a - b).reshape(N, K // 32, 32)
    # half a step, plus the fp16 rounding of d at the clamped extreme: |w| <= amax <= 7.5 d (1 + 2^-10)
    assert np.all(np.abs(err) <= 0.5 * step[:, :, None] + 7.5 * step[:, :, None] * 2.0 ** -10)
    e = np.sqrt((err.reshape(N, K) ** 2).sum(axis=1))
    assert np.all(bound >= e) and np.all(bound <= e * (1 + 1e-6) + 1e-30)
    assert np.allclose(wnorm, np.sqrt((a ** 2).sum(axis=1)), rtol=1e-6)


def test_shortlist_bound_holds_for_every_row():
    N, K, M = 2048, 1024, 3
    w8, q, s = _shortlist_case(71, N, K, M)
    q4, bound, _ = oracle.shortlist_copy(w8, N, K)
    exact = _exact_scores(w8, N, K, q, s)
    dots4 = oracle.block_dots(oracle.Q4_32, q4, N, K, q).astype(np.float64)
    d4 = np.asarray(q4).reshape(N, K // 32, 18)[:, :, :2].copy().view(np.uint16)[:, :, 0]
    dw4 = np.vectorize(lambda h: oracle.f16_to_f32(int(h)))(d4).astype(np.float64)
    copy = (dots4 * dw4[None] * s.astype(np.float64)[:, None, :]).sum(axis=2)
    an = np.sqrt(((q.astype(np.float64).reshape(M, K // 32, 32) * s[:, :, None]) ** 2).sum(axis=(1, 2)))
    assert np.all(np.abs(exact - copy) <= bound[None, :] * an[:, None] * (1 + 1e-9))


def test_shortlist_argmax_is_the_full_argmax_with_ties():
    N, K, M = 4096, 1024, 3
    w8, q, s = _shortlist_case(72, N, K, M)
    exact = _exact_scores(w8, N, K, q, s)
    # a duplicate of position 0's best row at a lower index: equal scores, the lower index must win
    top = int(np.argmax(exact[0]))
    rows = np.asarray(w8).reshape(N, -1).copy()
    dup = 5 if top != 5 else 6
    rows[dup] = rows[top]
    w8 = rows.reshape(-1)
    exact = _exact_scores(w8, N, K, q, s)
    q4, bound, _ = oracle.shortlist_copy(w8, N, K)
    am, nc = oracle.shortlist_argmax(q4, bound, w8, N, K, q, s)
    ref = [int(np.flatnonzero(exact[m] == exact[m].max())[0]) for m in range(M)]
    assert list(am) == ref and am[0] == min(dup, top)
    assert np.all(nc >= 1)


def test_shortlist_scores_few_rows_when_the_winner_stands_out():
    """Random rows leave every row within the worst-case bound of the best (the bound grows like
    ||err|| ||a||, the spread of random scores like their root-mean-square), so nothing is skipped;
    a row aligned with the activations, as in a peaked output distribution, lets the shortlist skip
    almost all of them."""
    N, K, M = 4096, 1024, 2
    w8, q, s = _shortlist_case(73, N, K, M)
    a = (q.astype(np.float64).reshape(M, K // 32, 32) * s[:, :, None]).reshape(M, K)
    # rows 100 and 2000 follow positions 0 and 1's activations (requantised as Q8_0 blocks)
    planted = {0: 100, 1: 2000}
    rows = np.asarray(w8).reshape(N, -1).copy()
    for m, r in planted.items():
        blk = sdgen.quantize(oracle.Q8_0, (a[m] / np.abs(a[m]).max() * 0.1).astype(np.float32)[None, :])
        rows[r] = np.asarray(blk).reshape(-1)
    w8 = rows.reshape(-1)
    q4, bound, _ = oracle.shortlist_copy(w8, N, K)
    am, nc = oracle.shortlist_argmax(q4, bound, w8, N, K, q, s)
    exact = _exact_scores(w8, N, K, q, s)
    assert list(am) == [int(np.argmax(exact[m])) for m in range(M)] == [100, 2000]
    assert np.all(nc <= N // 100), nc


def test_shortlist_finds_the_exact_winner_when_the_copy_ranks_it_second():
    """Two rows whose 4-bit copies are equal byte for byte, the lower-index one a single int8 step
    worse in exact arithmetic: the copy alone would pick the lower index, the exact scores of the
    candidates must pick the other."""
    N, K, M = 1024, 512, 1
    w8, q, s = _shortlist_case(74, N, K, M)
    exact = _exact_scores(w8, N, K, q, s)
    top = int(np.argmax(exact[0]))
    lo = 3 if top != 3 else 4
    rows = np.asarray(w8).reshape(N, K // 32, 34).copy()
    a = q.astype(np.int64).reshape(K)
    copy_top = np.asarray(oracle.shortlist_copy(rows[top].reshape(-1), 1, K)[0]).copy()
    done = False
    for b in range(K // 32):
        v = rows[top, b, 2:].view(np.int8).astype(np.int64)
        for j in range(32):
            aj = a[b * 32 + j]
            if aj == 0 or abs(v[j]) == np.abs(v).max():
                continue
            w = v.copy()
            w[j] -= 1 if aj > 0 else -1
            if abs(w[j]) >= np.abs(v).max():
                continue
            cand = rows[top].copy()
            cand[b, 2:] = w.astype(np.int8).view(np.uint8)
            if np.array_equal(np.asarray(oracle.shortlist_copy(cand.reshape(-1), 1, K)[0]), copy_top):
                rows[lo] = cand
                done = True
                break
        if done:
            break
    assert done
    w8 = rows.reshape(-1)
    exact = _exact_scores(w8, N, K, q, s)
    q4, bound, _ = oracle.shortlist_copy(w8, N, K)
    assert np.array_equal(np.asarray(q4).reshape(N, -1)[lo], np.asarray(q4).reshape(N, -1)[top])
    assert exact[0, lo] < exact[0, top] == exact[0].max()
    am, nc = oracle.shortlist_argmax(q4, bound, w8, N, K, q, s)
    assert int(am[0]) == top and nc[0] >= 2


# ---------------------------------------------------------------------------
# decode attention over the K+1 positions, fp16 KV append, commit of the accepted path
# ---------------------------------------------------------------------------

def _f16(a):
    return np.asarray(a, dtype=np.float32).astype(np.float16).view(np.uint16)


def _caches(H_kv, S_max, D):
    return np.zeros((H_kv, S_max, D), dtype=np.uint16), np.zeros((H_kv, S_max, D), dtype=np.uint16)


def test_f16_conversion_is_numpys_nearest_even():
    x = np.concatenate([sdgen.normal(sdgen.key(90), (4096,)) * s for s in (1e-6, 1e-3, 1.0, 300.0, 3e4)])
    x = np.concatenate([x, np.float32([65504.0, 65519.0, 65520.0, -7e4, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                                       0.0, -0.0, np.inf])])
    with np.errstate(over="ignore"):
        want = x.astype(np.float32).astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f32_to_f16(x), want)


def test_attention_one_hot_keys_closed_form():
    """Keys alpha e_j, query beta e_2: score alpha beta / sqrt(D) at key 2, 0 elsewhere, so the
    output is (e^s v_2 + sum_{j != 2} v_j) / (e^s + n - 1); the scale 1/sqrt(D) is what is pinned."""
    H_kv, D, L, M = 1, 64, 12, 1
    kc, vc = _caches(H_kv, 32, D)
    alpha, beta = 2.0, 3.0
    for j in range(L + M):
        kc[0, j] = _f16(alpha * np.eye(D)[j])
        vc[0, j] = _f16(np.full(D, float(j)))
    q = np.zeros((M, 1, D), np.float32)
    q[0, 0, 2] = beta
    out = oracle.attn_decode(q, kc, vc, L)
    s = alpha * beta / np.sqrt(D)
    n = L + M
    want = (np.exp(s) * 2.0 + (sum(range(n)) - 2.0)) / (np.exp(s) + n - 1)
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-13)


def test_attention_chain_and_tree_masks_count_the_visible_keys():
    """Equal keys: the output is the mean of the visible values.  Value of slot j is j, so the
    mean names the visible set: committed 0..L-1 plus the path of position i."""
    H_kv, D, L, M = 1, 32, 7, 5
    kc, vc = _caches(H_kv, 16, D)
    for j in range(L + M):
        kc[0, j] = _f16(np.full(D, 0.5))
        vc[0, j] = _f16(np.full(D, float(j)))
    q = sdgen.normal(sdgen.key(91), (M, 1, D))
    chain = oracle.attn_decode(q, kc, vc, L)
    for i in range(M):
        vis = list(range(L)) + [L + j for j in range(i + 1)]
        np.testing.assert_allclose(chain[i, 0], np.mean(vis), rtol=1e-13)
    parent = np.array([-1, 0, 0, 1, 2], np.int32)  # node 3 under 1, node 4 under 2
    tree = oracle.attn_decode(q, kc, vc, L, parent)
    paths = {0: [0], 1: [0, 1], 2: [0, 2], 3: [0, 1, 3], 4: [0, 2, 4]}
    for i in range(M):
        vis = list(range(L)) + [L + j for j in paths[i]]
        np.testing.assert_allclose(tree[i, 0], np.mean(vis), rtol=1e-13)


def test_attention_grouped_heads_read_their_kv_head():
    """H = 3 H_kv: query head h reads KV head h // 3 (constant values per KV head)."""
    H_kv, H, D, L, M = 2, 6, 32, 9, 3
    kc, vc = _caches(H_kv, 16, D)
    rng = sdgen.normal(sdgen.key(92), (H_kv, L + M, D))
    for h in range(H_kv):
        kc[h, :L + M] = _f16(rng[h])
        vc[h, :L + M] = _f16(np.full((L + M, D), 10.0 * (h + 1)))
    q = sdgen.normal(sdgen.key(92, 1), (M, H, D))
    out = oracle.attn_decode(q, kc, vc, L)
    for h in range(H):
        np.testing.assert_allclose(out[:, h], 10.0 * (h // 3 + 1), rtol=1e-13)


def test_attention_matches_a_dense_softmax_with_explicit_mask():
    """Brute force by matrices: S = Q K^T / sqrt(D) + mask, softmax rows, times V (numpy, fp64)."""
    H_kv, H, D, L, M = 2, 4, 64, 40, 5
    S_max = 64
    kc, vc = _caches(H_kv, S_max, D)
    kc[:, :L] = _f16(sdgen.normal(sdgen.key(93), (H_kv, L, D)))
    vc[:, :L] = _f16(sdgen.normal(sdgen.key(93, 1), (H_kv, L, D)))
    k_new = sdgen.normal(sdgen.key(93, 2), (M, H_kv, D))
    v_new = sdgen.normal(sdgen.key(93, 3), (M, H_kv, D))
    oracle.kv_append(k_new, v_new, kc, vc, L)
    assert np.array_equal(kc[:, L:L + M], _f16(k_new.transpose(1, 0, 2)))
    q = sdgen.normal(sdgen.key(93, 4), (M, H, D)) * 2.0
    parent = np.array([-1, 0, 1, 0, 3], np.int32)
    out = oracle.attn_decode(q, kc, vc, L, parent)
    Kf = kc.view(np.float16).astype(np.float64)
    Vf = vc.view(np.float16).astype(np.float64)
    anc = [[0], [0, 1], [0, 1, 2], [0, 3], [0, 3, 4]]
    for h in range(H):
        kh = h // (H // H_kv)
        S = q[:, h].astype(np.float64) @ Kf[kh, :L + M].T / np.sqrt(D)
        mask = np.full((M, L + M), -np.inf)
        mask[:, :L] = 0
        for i in range(M):
            mask[i, [L + j for j in anc[i]]] = 0
        P = np.exp(S + mask - (S + mask).max(axis=1, keepdims=True))
        P /= P.sum(axis=1, keepdims=True)
        np.testing.assert_allclose(out[:, h], P @ Vf[kh, :L + M], rtol=1e-12, atol=1e-14)


def test_commit_then_chain_equals_tree_attention():
    """Attention of tree node i before the commit equals chain attention of the last position
    after the commit of i's path: the commit keeps exactly the path's entries, in order."""
    H_kv, H, D, L, M = 2, 2, 32, 20, 6
    kc, vc = _caches(H_kv, 32, D)
    kc[:, :L + M] = _f16(sdgen.normal(sdgen.key(94), (H_kv, L + M, D)))
    vc[:, :L + M] = _f16(sdgen.normal(sdgen.key(94, 1), (H_kv, L + M, D)))
    q = sdgen.normal(sdgen.key(94, 2), (M, H, D))
    parent = np.array([-1, 0, 0, 2, 2, 3], np.int32)
    tree = oracle.attn_decode(q, kc, vc, L, parent)
    path = np.array([0, 2, 3, 5], np.int32)   # node 5's path
    kc2, vc2 = kc.copy(), vc.copy()
    oracle.kv_commit(kc2, vc2, L, path)
    n = path.size
    assert np.array_equal(kc2[:, L:L + n], kc[:, L + path]) and np.array_equal(vc2[:, :L], vc[:, :L])
    # chain over the committed n entries: query rows 0..n-1 take the path's queries
    qc = q[path]
    chain = oracle.attn_decode(qc, kc2[:, :L + n].copy(), vc2[:, :L + n].copy(), L)
    np.testing.assert_allclose(chain[n - 1], tree[5], rtol=1e-13)
    np.testing.assert_allclose(chain[1], tree[2], rtol=1e-13)


def test_attention_is_stable_for_large_scores():
    """A key scoring 1e4 above the rest takes all the weight (no overflow in the softmax)."""
    H_kv, D, L, M = 1, 32, 30, 1
    kc, vc = _caches(H_kv, 32, D)
    kc[0, :L + M] = _f16(np.ones((L + M, D)) * 0.01)
    kc[0, 17] = _f16(np.ones(D) * 100.0)
    vc[0, :L + M] = _f16(sdgen.normal(sdgen.key(95), (L + M, D)))
    q = np.full((M, 1, D), 20.0, np.float32)
    out = oracle.attn_decode(q, kc, vc, L)
    np.testing.assert_allclose(out[0, 0], vc[0, 17].view(np.float16).astype(np.float64), rtol=1e-12)


# ---------------------------------------------------------------------------
# adaptive draft depth
# ---------------------------------------------------------------------------

def test_depth_cut_by_one_for_the_cycle_after_a_rejection():
    """A configured depth of four runs three drafts in the cycle after a rejection, and four again
    after that cycle's drafts are all accepted."""
    assert oracle.depth_policy(4, 64, [4, 2, 3, 4]) == [4, 4, 3, 4]
    # a rejection at 4 (1 of 4), all 3 of the cut cycle accepted -> 4 again, and so on
    assert oracle.depth_policy(4, 64, [1, 3, 1, 3, 3]) == [4, 3, 4, 3, 4]
    # rejections in a row keep the cut depth
    assert oracle.depth_policy(4, 64, [2, 1, 2, 3]) == [4, 3, 3, 3]
    assert oracle.depth_policy(1, 64, [0, 0, 1]) == [1, 0, 1]


def test_outright_misses_pause_drafting_for_longer_and_longer():
    """Misses in a row: pauses of 1, 2, 4, 8 cycles; each resumption drafts at the cut depth."""
    used = oracle.depth_policy(4, 64, [0] * 40)
    drafted = [i for i, k in enumerate(used) if k > 0]
    gaps = [b - a - 1 for a, b in zip(drafted, drafted[1:])]
    assert gaps[:4] == [1, 2, 4, 8]
    assert all(used[i] == 3 for i in drafted[1:])
    # a hit resets the streak (the miss after it pauses 1 cycle, not 4); paused cycles accept nothing
    assert oracle.depth_policy(4, 64, [0, 0, 0, 0, 0, 2, 0, 0, 0]) == [4, 0, 3, 0, 0, 3, 3, 0, 3]
    # the cap holds
    used = oracle.depth_policy(2, 3, [0] * 30)
    drafted = [i for i, k in enumerate(used) if k > 0]
    assert max(b - a - 1 for a, b in zip(drafted, drafted[1:])) == 3
    assert oracle.depth_policy(4, 0, [0, 0, 2]) == [4, 3, 3]


# ---------------------------------------------------------------------------
# K-quant formats (Q4_K, Q6_K): layouts pinned by packing known fields, the matmul by the
# dense product of the dequantised weights
# ---------------------------------------------------------------------------

def _pack_q4k(d, dmin, sc, mn, codes):
    """One Q4_K super-block from its fields: sc, mn 6-bit [8]; codes 4-bit [256]."""
    b = np.zeros(144, np.uint8)
    b[0:2] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    b[2:4] = np.frombuffer(np.float16(dmin).tobytes(), np.uint8)
    s = np.zeros(12, np.int64)
    for j in range(4):
        s[j] = sc[j] | ((sc[j + 4] >> 4) << 6)          # scale j, top bits of scale j+4
        s[j + 4] = mn[j] | ((mn[j + 4] >> 4) << 6)      # min j, top bits of min j+4
        s[j + 8] = (sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4)
    b[4:16] = s
    for c in range(4):
        lo, hi = codes[64 * c:64 * c + 32], codes[64 * c + 32:64 * c + 64]
        b[16 + 32 * c:48 + 32 * c] = np.asarray(lo) | (np.asarray(hi) << 4)
    return b


def _pack_q6k(d, scales, codes):
    """One Q6_K super-block: scales int8 [16]; codes 6-bit unsigned [256] (weight = code - 32)."""
    b = np.zeros(210, np.uint8)
    codes = np.asarray(codes, np.int64)
    for n in range(2):
        for l in range(32):
            q = [codes[128 * n + 32 * k + l] for k in range(4)]
            b[64 * n + l] = (q[0] & 15) | ((q[2] & 15) << 4)
            b[64 * n + l + 32] = (q[1] & 15) | ((q[3] & 15) << 4)
            b[128 + 32 * n + l] = (q[0] >> 4) | ((q[1] >> 4) << 2) | ((q[2] >> 4) << 4) | ((q[3] >> 4) << 6)
    b[192:208] = np.asarray(scales, np.int8).view(np.uint8)
    b[208:210] = np.frombuffer(np.float16(d).tobytes(), np.uint8)
    return b


def test_q4k_layout_from_known_fields():
    u = sdgen.u32(sdgen.key(96), 8 + 8 + 256)
    sc, mn, codes = u[:8] % 64, u[8:16] % 64, u[16:] % 16
    b = _pack_q4k(0.5, 0.25, sc, mn, codes)
    w = oracle.kq_dequant(oracle.Q4_K, b, 1, 256)[0]
    want = 0.5 * np.repeat(sc, 32) * codes - 0.25 * np.repeat(mn, 32)
    assert np.array_equal(w, want.astype(np.float32))
    # every 6-bit field reaches its top value
    b = _pack_q4k(1.0, 1.0, [63] * 8, [63] * 8, [15] * 256)
    assert np.all(oracle.kq_dequant(oracle.Q4_K, b, 1, 256) == 63 * 15 - 63)


def test_q6k_layout_from_known_fields():
    u = sdgen.u32(sdgen.key(97), 16 + 256)
    scales = (u[:16] % 256).astype(np.int64) - 128
    codes = u[16:] % 64
    b = _pack_q6k(0.125, scales, codes)
    w = oracle.kq_dequant(oracle.Q6_K, b, 1, 256)[0]
    want = 0.125 * np.repeat(scales, 16) * (codes.astype(np.int64) - 32)
    assert np.array_equal(w, want.astype(np.float32))


@pytest.mark.parametrize("qtype", [2, 3])
def test_kq_matmul_factored_form_equals_dense_product(qtype):
    """The per-block integer form (Q4_K: d sc dot - dmin m sum) against the fp64 product of the
    dequantised weights with the dequantised activations."""
    N, K, M = 96, 1024, 5
    w = sdgen.random_kq_blocks(qtype, sdgen.key(98, qtype), N, K)
    q, s = oracle.rmsnorm_quant(sdgen.normal(sdgen.key(98, 9), (M, K)), None)
    y = oracle.kq_matmul(qtype, w, N, K, q, s)
    W = oracle.kq_dequant(qtype, w, N, K).astype(np.float64)
    A = (q.astype(np.float64).reshape(M, K // 32, 32) * s[:, :, None]).reshape(M, K)
    ref = A @ W.T
    absb = np.abs(A) @ np.abs(W).T
    # the dequantised weights are fp32 roundings of the exact values (at most 2^-24 relative)
    assert np.all(np.abs(y - ref) <= 2.0 ** -23 * absb + 1e-300)


def test_kq_matmul_reduces_to_the_32_weight_formats():
    """Q4_K with every scale 1, min 8 and dmin = d is Q4_32 (d (code - 8)); Q6_K with every scale 1
    is Q8_0 with codes in [-32, 31].  Same weights, so the same matmul as the brute-force-pinned
    32-weight path, whose fp64 sums come back rounded to fp32: equal to the fp32 rounding of the
    K-quant path's fp64 sums (one rounding step either way at a rounding boundary)."""
    N, K, M = 24, 512, 3
    q, s = oracle.rmsnorm_quant(sdgen.normal(sdgen.key(99, 1), (M, K)), None)
    u = sdgen.u32(sdgen.key(99, 2), N * K)
    d = np.float16(0.0123)
    # 4-bit
    codes4 = (u % 16).reshape(N, K // 256, 256)
    q4k = np.stack([np.concatenate([_pack_q4k(d, d, [1] * 8, [8] * 8, codes4[n, j]) for j in range(K // 256)])
                    for n in range(N)])
    q432 = np.zeros((N, K // 32, 18), np.uint8)
    q432[:, :, 0:2] = np.frombuffer(d.tobytes(), np.uint8)
    c = codes4.reshape(N, K // 32, 32)
    q432[:, :, 2:] = c[:, :, :16] | (c[:, :, 16:] << 4)
    y_k = oracle.kq_matmul(oracle.Q4_K, q4k, N, K, q, s)
    y_32, _ = oracle.qmatmul(oracle.Q4_32, q432.reshape(-1), N, K, q, s)
    assert np.all(np.abs(y_k.astype(np.float32) - y_32) <= np.spacing(np.abs(y_32)))
    # 6-bit
    codes6 = (u // 16 % 64).reshape(N, K // 256, 256)
    q6k = np.stack([np.concatenate([_pack_q6k(d, [1] * 16, codes6[n, j]) for j in range(K // 256)])
                    for n in range(N)])
    q80 = np.zeros((N, K // 32, 34), np.uint8)
    q80[:, :, 0:2] = np.frombuffer(d.tobytes(), np.uint8)
    q80[:, :, 2:] = (codes6.reshape(N, K // 32, 32).astype(np.int64) - 32).astype(np.int8).view(np.uint8)
    y_k = oracle.kq_matmul(oracle.Q6_K, q6k, N, K, q, s)
    y_8, _ = oracle.qmatmul(oracle.Q8_0, q80.reshape(-1), N, K, q, s)
    assert np.all(np.abs(y_k.astype(np.float32) - y_8) <= np.spacing(np.abs(y_8)))


def test_tree_path_names_the_accepted_tokens():
    """The accepted path's nodes carry exactly the tokens the pinned tree rule emits (the last
    emitted token is the argmax after the path's end), on random trees with repeated tokens."""
    u = sdgen.u32(sdgen.key(100), 200 * 64)
    for t in range(200):
        M = 2 + t % 15
        r = u[t * 64:(t + 1) * 64]
        parent = np.array([-1] + [int(r[i] % i) for i in range(1, M)], np.int32)
        argmax = (r[16:16 + M] % 3).astype(np.int32)        # three tokens: many matches and ties
        tokens = (r[32:32 + M] % 3).astype(np.int32)
        path = oracle.accept_greedy_tree_path(argmax, tokens, parent)
        out = oracle.accept_greedy_tree(argmax, tokens, parent)
        assert path[0] == 0 and len(path) == len(out)
        assert all(parent[path[i]] == path[i - 1] for i in range(1, len(path)))
        assert list(tokens[path[1:]]) + [argmax[path[-1]]] == list(out)


@pytest.mark.parametrize("qtype", [oracle.Q4_K, oracle.Q6_K])
def test_kq_matmul_bound_is_the_absolute_sum(qtype):
    """The tolerance scale returned with the K-quant product is the absolute sum of its terms: at least
    |y| everywhere, and equal to y when every weight and activation is non-negative (no cancellation).
    Q4_K with zero minima and Q6_K with codes >= 32 and positive scales make every term >= 0."""
    N, K, M = 8, 512, 3
    w = sdgen.random_kq_blocks(qtype, sdgen.key(190, qtype), N, K).reshape(N, K // 256, -1)
    q, s = oracle.rmsnorm_quant(np.abs(sdgen.normal(sdgen.key(191), (M, K))), None)
    y, ab = oracle.kq_matmul(qtype, w, N, K, q, s, with_bound=True)
    assert np.all(ab >= np.abs(y) * (1 - 1e-12))
    w2 = w.copy()
    if qtype == oracle.Q4_K:
        w2[..., 4:16] &= 0x3F                    # sub-blocks 0-3: minima 0 (bytes 4-7: scales, 8-11: minima)
        w2[..., 8:12] = 0
        w2[..., 12:16] &= 0x0F                   # sub-blocks 4-7: minima 0
        w2[..., 4:8] &= 0x3F                     # and the high bits of the minima of 4-7
    else:
        w2[..., 128:192] = 0xAA                  # high bits 2 for every code: codes 32..47
        w2[..., 192:208] = 5                     # positive scales
    y2, ab2 = oracle.kq_matmul(qtype, w2, N, K, q, s, with_bound=True)
    assert np.all(y2 >= 0)
    assert np.allclose(ab2, y2, rtol=1e-12, atol=0)
