"""GPU parity at the full workload sizes.

* Layer-sized matmuls (hidden 5120, FFN 17408; Q8_0 and 4-bit): every output
  of an M = 8 run against the oracle, and rows of M = 1, 2, 3, 5 runs bit-equal
  to the M = 8 rows (batch invariance carries the parity over).
* The 5120 x 151936 Q8_0 head at K+1 = 5: logits, argmax and statistics against
  the oracle; greedy and rejection-sampling acceptance (general drafter and
  certainty drafter) bit-exact when fed the oracle's logits.
* The 64-layer stack as one CUDA graph of per-operation launches: stage-wise
  parity on three layers with oracle inputs, every row of the pass bit-equal
  to that row run alone, the chain/tree acceptance rule on the pass's own
  argmax, and the free-running divergence from the oracle's own 64-layer pass
  (reported; its float parity is unpinned).
* The same stack as the one persistent launch the bench times (its deferred
  down-projection combine and head-statistics phases exist only at these
  widths): every output bit-equal to the per-operation pass, at M = 5 (chain)
  and M = 16 (tree), and with rejection-sampling acceptance (against the
  per-operation pass + sd_accept_sample and the oracle's rule).
"""
import numpy as np
import pytest
import torch

import oracle
import sdgen
from _util import acts, assert_close, cuda, host, status_ok

pytestmark = pytest.mark.gpu

H, F, V = sdgen.HIDDEN, sdgen.FFN, sdgen.VOCAB


@pytest.fixture(scope="module")
def sdv():
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    import speculative_decoding_verify_gb300 as m
    m.lib()
    return m


def norm_acts(key, M, K):
    """RMSNorm'd + requantised N(0,1) rows with norm weights 1 + N(0, 0.1) (oracle, as GPU input)."""
    x = sdgen.normal(sdgen.key(key, 0), (M, K))
    w = sdgen.norm_weight(sdgen.key(key, 1), K)
    return oracle.rmsnorm_quant(x, w, sdgen.EPS)


# ---------------------------------------------------------------------------
# layer-sized matmuls
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("qtype", [oracle.Q8_0, oracle.Q4_32])
@pytest.mark.parametrize("n,k", [(5120, 5120), (17408, 5120), (5120, 17408)])
def test_layer_matmuls(sdv, qtype, n, k):
    blocks = sdgen.quantized_normal(qtype, sdgen.key(2, n, k, qtype), n, k)
    w = sdv.repack_weights(qtype, cuda(blocks).reshape(-1), n, k)
    ws = sdv.workspace(sdv.qmatmul_workspace_bytes(qtype, n, k))
    q, s = norm_acts(200 + k, 8, k)
    qd, sd = cuda(q), cuda(s)
    y8 = torch.zeros((8, n), dtype=torch.float32, device="cuda")
    sdv.qmatmul_multipos(qtype, w, n, k, qd, sd, ws, y=y8)
    status_ok()
    yo, ab = oracle.qmatmul(qtype, blocks, n, k, q, s)
    assert_close(host(y8), yo, ab, f"{n}x{k} q{qtype}")
    for M in (1, 2, 3, 5):
        y = torch.zeros((M, n), dtype=torch.float32, device="cuda")
        sdv.qmatmul_multipos(qtype, w, n, k, qd[:M], sd[:M], ws, y=y)
        status_ok()
        assert np.array_equal(host(y).view(np.uint32), host(y8)[:M].view(np.uint32))


# ---------------------------------------------------------------------------
# full-vocabulary head + acceptance
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def head_case(sdv):
    M = 5
    blocks = sdgen.quantized_normal(oracle.Q8_0, sdgen.key(3, 0), V, H)
    w = sdv.repack_weights(oracle.Q8_0, cuda(blocks).reshape(-1), V, H)
    q, s = norm_acts(300, M, H)
    lo, ab = oracle.qmatmul(oracle.Q8_0, blocks, V, H, q, s)
    return dict(M=M, blocks=blocks, w=w, q=q, s=s, lo=lo, ab=ab)


def test_head_full_vocab(sdv, head_case):
    c = head_case
    M = c["M"]
    ws = sdv.workspace(sdv.head_workspace_bytes(V, H))
    lg = torch.zeros((M, V), dtype=torch.float32, device="cuda")
    am = torch.zeros(M, dtype=torch.int32, device="cuda")
    rm = torch.zeros(M, dtype=torch.float32, device="cuda")
    rz = torch.zeros(M, dtype=torch.float32, device="cuda")
    sdv.head_logits(c["w"], V, H, cuda(c["q"]), cuda(c["s"]), ws, lg, am, rm, rz, 1.0)
    status_ok()
    g = host(lg)
    assert_close(g, c["lo"], c["ab"], "head logits")
    assert np.array_equal(host(am), np.argmax(g, axis=1))
    mo, zo, ao = oracle.softmax_stats(c["lo"], 1.0)
    tol = 1e-5 * c["ab"].max(axis=1) + 1e-6
    for m in range(M):
        assert c["lo"][m, host(am)[m]] >= c["lo"][m].max() - 2 * tol[m]
    assert np.array_equal(host(rm), g.max(axis=1))
    assert np.all(np.abs(host(rz) / zo - 1) <= 2 * tol + 1e-6)
    # the same workspace again (its counters are back at zero): identical bits
    lg2 = torch.zeros_like(lg)
    sdv.head_logits(c["w"], V, H, cuda(c["q"]), cuda(c["s"]), ws, lg2, am, rm, rz, 1.0)
    status_ok()
    assert torch.equal(lg.view(torch.int32), lg2.view(torch.int32))


def test_head_greedy_accept_p075(sdv, head_case):
    c = head_case
    M = c["M"]
    _, _, ao = oracle.softmax_stats(c["lo"])
    for t in range(8):
        drafts = sdgen.drafts_p(sdgen.key(3, 10 + t), ao[:M - 1], V)
        ot = torch.zeros(M, dtype=torch.int32, device="cuda")
        oc = torch.zeros(1, dtype=torch.int32, device="cuda")
        sdv.accept_greedy(cuda(ao), cuda(drafts), None, M, ot, oc)
        status_ok()
        ref = oracle.accept_greedy_chain(ao, drafts)
        assert list(host(ot)[:int(host(oc)[0])]) == list(ref)


@pytest.mark.parametrize("certainty", [False, True])
def test_head_rejection_sampling(sdv, head_case, certainty):
    """q = softmax(target logits + N(0,1) noise), drafts ~ q (or a certainty drafter proposing them),
    T = 1, Philox keyed by (seed, position): the GPU's kept tokens equal the oracle's, bit for bit."""
    c = head_case
    M = c["M"]
    K = M - 1
    lo = c["lo"]
    noise = sdgen.normal(sdgen.key(3, 20), (K, V))
    qp = np.stack([oracle.softmax_probs(lo[i] + noise[i]) for i in range(K)])
    m, z, _ = oracle.softmax_stats(lo)
    ld, qd = cuda(lo), cuda(qp)
    cdf = np.cumsum(qp.astype(np.float64), axis=1)
    for t in range(10):
        u = sdgen.uniforms(sdgen.key(3, 30, t), K)
        drafts = np.array([min(np.searchsorted(cdf[i] / cdf[i, -1], u[i], side="right"), V - 1) for i in range(K)],
                          dtype=np.int32)
        ot = torch.full((M,), -7, dtype=torch.int32, device="cuda")
        oc = torch.zeros(1, dtype=torch.int32, device="cuda")
        given = t % 2 == 0
        sdv.accept_sample(ld, K, cuda(drafts), ot, oc, q_probs=None if certainty else qd,
                          row_max=cuda(m) if given else None, row_sumexp=cuda(z) if given else None,
                          temperature=1.0, seed=1234, base_pos=77 + 5 * t)
        status_ok()
        ref = oracle.accept_sample(lo, None if certainty else qp, drafts, 1.0, 1234, 77 + 5 * t)
        assert list(host(ot)[:int(host(oc)[0])]) == list(ref), t


# ---------------------------------------------------------------------------
# the 64-layer stack, as the bench runs it
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def stack_env(sdv):
    from speculative_decoding_verify_gb300.verify_pass import VerifyStack, repack_matrix
    spec = sdgen.StackSpec()
    layers, norms = [], []
    for l in range(spec.layers):
        lw = {}
        for name, n, k in spec.matrices():
            b = sdgen.pinned_quantized_normal(spec.wq, spec.weight_key(l, name), n, k)
            lw[name] = repack_matrix(spec.wq, b, n, k, pair=(name == "gate_up"))
        layers.append(lw)
        n1, n2 = spec.norms(l)
        norms.append((cuda(n1), cuda(n2)))
    hb = sdgen.pinned_quantized_normal(spec.head_q, spec.weight_key(0, "head"), V, H)
    head = repack_matrix(spec.head_q, hb, V, H)
    fn = cuda(spec.final_norm())

    def make(M, parent=None):
        return VerifyStack(layers, norms, fn, head, H, F, V, M, tree_parent=parent)

    return dict(spec=spec, make=make, layers=layers, norms=norms)


@pytest.mark.parametrize("layer", [0, 31, 63])
def test_stack_stagewise_parity(sdv, stack_env, layer):
    """Each stage of layer l, fed the oracle's input of that stage."""
    spec = stack_env["spec"]
    st = stack_env["make"](5)
    wts = {name: spec.weights(layer, name) for name, _, _ in spec.matrices()}
    n1, n2 = spec.norms(layer)
    h = sdgen.normal(sdgen.key(5, layer), (5, H)) * 2
    tr = {}
    oracle.stack_layer(h, wts, n1, n2, H, F, spec.wq, trace=tr)
    lw = stack_env["layers"][layer]
    # 1. RMSNorm + requant: bit-exact
    st.h.copy_(cuda(h))
    sdv.rmsnorm_quant_acts(st.h, stack_env["norms"][layer][0], st.qa, st.sa, sdgen.EPS)
    status_ok()
    assert np.array_equal(host(st.qa), tr["q1"]) and np.array_equal(host(st.sa), tr["s1"])
    # 2. QKV with the V columns requantised in the epilogue
    y = torch.zeros((5, 3 * H), dtype=torch.float32, device="cuda")
    sdv.qmatmul_multipos(spec.wq, lw["qkv"], 3 * H, H, st.qa, st.sa, st.ws, y=y, epilogue=sdv.EPI_REQUANT,
                         requant_col0=2 * H, q_next=st.qv, scales_next=st.sv)
    status_ok()
    assert_close(host(y), tr["qkv"], oracle.qmatmul(spec.wq, wts["qkv"], 3 * H, H, tr["q1"], tr["s1"])[1], "qkv")
    qq = torch.zeros((5, H), dtype=torch.int8, device="cuda")
    ss = torch.zeros((5, H // 32), dtype=torch.float32, device="cuda")
    sdv.rmsnorm_quant_acts(y[:, 2 * H:], None, qq, ss, K=H, ldx=3 * H)
    status_ok()
    assert torch.equal(qq, st.qv) and torch.equal(ss, st.sv)
    # 3. O + residual, fed the oracle's requantised V
    st.h.copy_(cuda(h))
    sdv.qmatmul_multipos(spec.wq, lw["o"], H, H, cuda(tr["qv"]), cuda(tr["sv"]), st.ws, y=st.h, residual=st.h)
    status_ok()
    assert_close(host(st.h), tr["h2"], oracle.qmatmul(spec.wq, wts["o"], H, H, tr["qv"], tr["sv"], residual=h)[1],
                 "o")
    # 4. second RMSNorm, fed the oracle's h2: bit-exact
    sdv.rmsnorm_quant_acts(cuda(tr["h2"]), stack_env["norms"][layer][1], st.qa, st.sa, sdgen.EPS)
    status_ok()
    assert np.array_equal(host(st.qa), tr["q3"]) and np.array_equal(host(st.sa), tr["s3"])
    # 5. gate|up with SiLU*mul requant; g|u against the oracle, the codes against the GPU's own requant of g|u
    gu = torch.zeros((5, 2 * F), dtype=torch.float32, device="cuda")
    sdv.qmatmul_multipos(spec.wq, lw["gate_up"], 2 * F, H, cuda(tr["q3"]), cuda(tr["s3"]), st.ws, y=gu,
                         epilogue=sdv.EPI_SILU_MUL_REQUANT, q_next=st.qf, scales_next=st.sf)
    status_ok()
    assert_close(host(gu), tr["gu"], oracle.qmatmul(spec.wq, wts["gate_up"], 2 * F, H, tr["q3"], tr["s3"])[1],
                 "gate_up")
    qd, sd = sdv.debug_silu_mul_requant(gu[:, :F].contiguous(), gu[:, F:].contiguous())
    status_ok()
    assert torch.equal(qd, st.qf) and torch.equal(sd, st.sf)
    assert (host(st.qf) != tr["q4"]).mean() < 1e-3
    # 6. down + residual, fed the oracle's codes
    st.h.copy_(cuda(tr["h2"]))
    sdv.qmatmul_multipos(spec.wq, lw["down"], H, F, cuda(tr["q4"]), cuda(tr["s4"]), st.ws, y=st.h, residual=st.h)
    status_ok()
    assert_close(host(st.h), tr["h3"],
                 oracle.qmatmul(spec.wq, wts["down"], H, F, tr["q4"], tr["s4"], residual=tr["h2"])[1], "down")


def run_graph(st, h_in):
    st.h.copy_(h_in)
    st.capture()
    st.h.copy_(h_in)
    st.replay()
    torch.cuda.synchronize()


def test_stack_pass_batch_invariant_and_accept(sdv, stack_env):
    """The graph-captured pass at M = 5: every row bit-equal to that row alone (M = 1), the chain rule on
    the pass's own argmax, and the free-running divergence from the oracle's 64-layer pass (reported)."""
    spec = stack_env["spec"]
    M = 5
    h0 = cuda(spec.hidden_in(M))
    st = stack_env["make"](M)
    st.h.copy_(h0)
    st.run()
    torch.cuda.synchronize()
    am0 = host(st.argmax)
    drafts = sdgen.drafts_p(sdgen.key(4, 7), am0[:M - 1], V)
    st.tokens[:M - 1].copy_(cuda(drafts))
    run_graph(st, h0)
    status_ok()
    lg5, am5 = host(st.logits), host(st.argmax)
    assert np.array_equal(am5, am0)
    n = int(host(st.out_count)[0])
    kept = list(host(st.out_tokens)[:n])
    # chain rule on the pass's own argmax
    j = 0
    while j < M - 1 and drafts[j] == am5[j]:
        j += 1
    assert kept == list(drafts[:j]) + [am5[j]]
    for m in range(M):
        s1 = stack_env["make"](1)
        run_graph(s1, h0[m:m + 1])
        status_ok()
        assert np.array_equal(host(s1.logits).view(np.uint32), lg5[m:m + 1].view(np.uint32))
        assert int(host(s1.argmax)[0]) == am5[m]
        del s1
    # free-running comparison with the oracle (reported, not gated beyond a sanity bound)
    h = spec.hidden_in(M)
    for l in range(spec.layers):
        wts = {name: spec.weights(l, name) for name, _, _ in spec.matrices()}
        n1, n2 = spec.norms(l)
        h = oracle.stack_layer(h, wts, n1, n2, H, F, spec.wq)
    lo, ao, _, _ = oracle.head(h, spec.final_norm(), spec.head(), V, H)
    rel = np.abs(lg5 - lo).max() / np.abs(lo).max()
    agree = int((ao == am5).sum())
    print(f"\nfree-running 64-layer pass vs oracle: max |dlogit| / max|logit| = {rel:.3e}, "
          f"argmax agreement {agree}/{M}")
    # requantisation codes that land on a rounding boundary differ by one step between fp32
    # reduction orders and the difference compounds over 64 random layers: reported, loosely bounded
    assert rel < 0.25


def test_tree_pass_batch_invariant(sdv, stack_env):
    """The 16-node draft tree (root, binary tree of depth 3, one spine node) as M = 16 rows through the
    64-layer stack and head.  Tree tokens are uniform over the vocabulary except along the path
    0 -> 1 -> 3 -> 7 -> 15, which follows the ORACLE's argmax chain of its own 64-layer pass.
    Checks: every one of the 16 rows' logits bit-equal that row run alone (M = 1); the pass's
    acceptance equals the tree rule on the pass's own argmax; and sd_accept_greedy fed the oracle's
    argmax accepts exactly what the oracle's tree rule accepts (the whole path plus its bonus)."""
    spec = stack_env["spec"]
    parent, depth = sdgen.tree16(0)
    M = 16
    emb = sdgen.normal(sdgen.key(6, 0), (M, H))
    # the oracle's own 64-layer pass over the 16 rows: its argmax chain lays out the accepted path
    h = emb.copy()
    for l in range(spec.layers):
        wts = {name: spec.weights(l, name) for name, _, _ in spec.matrices()}
        n1, n2 = spec.norms(l)
        h = oracle.stack_layer(h, wts, n1, n2, H, F, spec.wq)
    _, ao, _, _ = oracle.head(h, spec.final_norm(), spec.head(), V, H)
    tokens = sdgen.uniform_tokens(sdgen.key(6, 1), M, V)
    path = (1, 3, 7, 15)
    for child in path:
        tokens[child] = ao[parent[child]]
    tokens = tokens.astype(np.int32)
    ref = oracle.accept_greedy_tree(ao, tokens, parent)
    assert list(ref) == [tokens[c] for c in path] + [ao[15]]

    st = stack_env["make"](M, parent=cuda(parent))
    hin = cuda(emb)
    st.tokens.copy_(cuda(tokens))
    run_graph(st, hin)
    status_ok()
    lg, am = host(st.logits), host(st.argmax)
    n = int(host(st.out_count)[0])
    assert list(host(st.out_tokens)[:n]) == list(oracle.accept_greedy_tree(am, tokens, parent))
    print(f"\ntree pass vs oracle argmax: {int((am == ao).sum())}/{M} rows agree")

    # config-5 acceptance, integer work fed the oracle's argmax: bit-exact against the oracle's rule
    ot = torch.full((M,), -1, dtype=torch.int32, device="cuda")
    oc = torch.zeros(1, dtype=torch.int32, device="cuda")
    sdv.accept_greedy(cuda(ao.astype(np.int32)), cuda(tokens), cuda(parent), M, ot, oc)
    status_ok()
    assert list(host(ot)[:int(host(oc)[0])]) == list(ref)

    # every row of the M = 16 pass bit-equal to that row alone (one M = 1 stack, reused)
    s1 = stack_env["make"](1)
    for m in range(M):
        run_graph(s1, hin[m:m + 1])
        status_ok()
        assert np.array_equal(host(s1.logits).view(np.uint32), lg[m:m + 1].view(np.uint32)), m
        assert int(host(s1.argmax)[0]) == am[m]
    del s1


@pytest.mark.parametrize("M", [5, 16])
def test_stack_fused_pass_equals_per_op_pass(sdv, stack_env, M):
    """The one-launch pass against the per-operation pass on the 64-layer stack: hidden rows, logits,
    statistics, requantised activations and the accepted tokens, all bit-equal."""
    spec = stack_env["spec"]
    parent = cuda(sdgen.tree16(0)[0]) if M == 16 else None
    h0 = cuda(spec.hidden_in(M)) if M == 5 else cuda(sdgen.normal(sdgen.key(6, 2), (M, H)))
    a = stack_env["make"](M, parent)
    a.h.copy_(h0)
    a.run()
    torch.cuda.synchronize()
    am = host(a.argmax)
    # drafts: the pass's own argmax for the first two, then a miss
    tokens = np.array([am[i] if i < 2 else (am[i] + 1) % V for i in range(M)], np.int32)
    if M == 16:
        tokens = np.roll(tokens, 1)  # node i's draft is judged against its parent's argmax
    a.tokens.copy_(cuda(tokens))
    b = stack_env["make"](M, parent)
    b.tokens.copy_(cuda(tokens))
    a.h.copy_(h0)
    a.run()
    b.h.copy_(h0)
    b.run_fused()
    status_ok()
    for name in ("h", "logits", "argmax", "row_max", "row_sumexp", "qa", "sa", "qv", "sv", "qf", "sf"):
        x, y = getattr(a, name), getattr(b, name)
        assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x,
                           y.view(torch.int32) if y.dtype == torch.float32 else y), name
    n = int(host(a.out_count)[0])
    assert n >= 1 and int(host(b.out_count)[0]) == n
    assert torch.equal(a.out_tokens[:n], b.out_tokens[:n])


def test_stack_fused_pass_sampled_acceptance(sdv, stack_env):
    """The 64-layer one-launch pass ending in rejection sampling (certainty drafter, T = 0.7) against
    the per-operation pass followed by sd_accept_sample, and the oracle's rule on its logits."""
    spec = stack_env["spec"]
    M, T = 5, 0.7
    h0 = cuda(spec.hidden_in(M))
    a, b = stack_env["make"](M), stack_env["make"](M)
    a.h.copy_(h0)
    a.run()
    torch.cuda.synchronize()
    am = host(a.argmax)
    drafts = np.array([am[0], am[1], (am[2] + 5) % V, am[3]], np.int32)
    for st in (a, b):
        st.h.copy_(h0)
        st.tokens[:M - 1].copy_(cuda(drafts))
    for l in range(spec.layers):
        a.layer(l)
    a.head(T)
    a.accept_sampled(T, 77, 4096)
    b.prepare_fused(temperature=T, sample=True, seed=77, base_pos=4096)
    b.run_fused()
    status_ok()
    for name in ("logits", "row_max", "row_sumexp"):
        x, y = getattr(a, name), getattr(b, name)
        assert torch.equal(x.view(torch.int32), y.view(torch.int32)), name
    n = int(host(a.out_count)[0])
    assert int(host(b.out_count)[0]) == n
    assert torch.equal(a.out_tokens[:n], b.out_tokens[:n])
    assert list(host(b.out_tokens)[:n]) == list(oracle.accept_sample(host(b.logits), None, drafts, T, 77, 4096))


def test_stack_fused_pass_filtered_sampling(sdv, stack_env):
    """The 64-layer one-launch pass with top_k = 20, top_p = 0.95 (T = 1) against the oracle's rule on
    its own logits and the per-operation pass + sd_accept_sample_topk."""
    spec = stack_env["spec"]
    M = 5
    h0 = cuda(spec.hidden_in(M))
    a, b = stack_env["make"](M), stack_env["make"](M)
    a.h.copy_(h0)
    a.run()
    torch.cuda.synchronize()
    am = host(a.argmax)
    drafts = np.array([am[0], am[1], am[2], (am[3] + 9) % V], np.int32)
    for st in (a, b):
        st.h.copy_(h0)
        st.tokens[:M - 1].copy_(cuda(drafts))
    for l in range(spec.layers):
        a.layer(l)
    a.head(1.0)
    a.accept_sampled(1.0, 123, 77, top_k=20, top_p=0.95)
    b.prepare_fused(temperature=1.0, sample=True, seed=123, base_pos=77, top_k=20, top_p=0.95)
    b.run_fused()
    status_ok()
    n = int(host(a.out_count)[0])
    assert int(host(b.out_count)[0]) == n
    assert torch.equal(a.out_tokens[:n], b.out_tokens[:n])
    assert list(host(b.out_tokens)[:n]) == list(oracle.accept_sample_topk(host(b.logits), None, drafts, 1.0, 20, 0.95,
                                                                        123, 77))
