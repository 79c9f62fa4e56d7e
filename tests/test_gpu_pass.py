"""The one-launch verify pass equals the per-operation pipeline bit for bit.

sd_verify_pass runs every phase (RMSNorm + requant, the four projections with
their epilogues, the head with statistics, greedy acceptance) in one persistent
cooperative launch.  Each phase is the same device code as the single-operation
calls, so the final hidden state, logits, argmax, statistics and accepted tokens
must match issuing those calls one by one, for chain and tree acceptance and
for one and two 8-position tiles.  The per-operation pipeline itself is checked
against the oracle stage by stage elsewhere; here it is also checked end to end
on a small stack.
"""
import numpy as np
import pytest
import torch

import oracle
import sdgen
from _util import assert_close, cuda, host, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    import speculative_decoding_verify_gb300 as m
    m.lib()
    return m


def small_stack(sdv, L=3, H=512, F=1024, V=4096, seed=0):
    from speculative_decoding_verify_gb300.verify_pass import repack_matrix
    spec = sdgen.StackSpec(layers=L, hidden=H, ffn=F, vocab=V, seed=seed)
    layers, norms, host_w = [], [], []
    for l in range(L):
        lw, hw = {}, {}
        for name, n, k in spec.matrices():
            b = spec.weights(l, name)
            hw[name] = b
            lw[name] = repack_matrix(spec.wq, b, n, k, pair=(name == "gate_up"))
        layers.append(lw)
        host_w.append(hw)
        n1, n2 = spec.norms(l)
        norms.append((cuda(n1), cuda(n2)))
    head_b = spec.head()
    head = repack_matrix(spec.head_q, head_b, V, H)
    return spec, layers, norms, host_w, head, head_b


def make(sdv, env, M, parent=None):
    from speculative_decoding_verify_gb300.verify_pass import VerifyStack
    spec, layers, norms, _, head, _ = env
    return VerifyStack(layers, norms, cuda(spec.final_norm()), head, spec.hidden, spec.ffn, spec.vocab, M,
                       tree_parent=parent)


def run_both(sdv, env, M, tokens, parent=None, h_in=None):
    spec = env[0]
    h0 = cuda(h_in if h_in is not None else spec.hidden_in(M))
    a = make(sdv, env, M, cuda(parent) if parent is not None else None)
    b = make(sdv, env, M, cuda(parent) if parent is not None else None)
    for st in (a, b):
        st.h.copy_(h0)
        st.tokens[:len(tokens)].copy_(cuda(np.asarray(tokens, np.int32)))
    a.run()
    b.run_fused()
    status_ok()
    return a, b


def same(x, y):
    return torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x,
                       y.view(torch.int32) if y.dtype == torch.float32 else y)


@pytest.mark.parametrize("M", [1, 5, 16])
def test_fused_pass_equals_pipeline(sdv, M):
    env = small_stack(sdv)
    spec = env[0]
    # drafts: the pipeline's own argmax for the first two, a miss after
    probe = make(sdv, env, M)
    probe.h.copy_(cuda(spec.hidden_in(M)))
    probe.run()
    am = host(probe.argmax)
    drafts = np.array([am[i] if i < 2 else (am[i] + 1) % spec.vocab for i in range(M - 1)], np.int32)
    a, b = run_both(sdv, env, M, drafts)
    for name in ("h", "logits", "argmax", "row_max", "row_sumexp", "qa", "sa", "qv", "sv", "qf", "sf"):
        assert same(getattr(a, name), getattr(b, name)), name
    n = int(host(a.out_count)[0])
    assert int(host(b.out_count)[0]) == n
    assert torch.equal(a.out_tokens[:n], b.out_tokens[:n])
    if M >= 4:
        assert n == 3  # two drafts kept, the third rejected, one correction


def test_fused_pass_tree(sdv):
    env = small_stack(sdv, seed=1)
    spec = env[0]
    parent, _ = sdgen.tree16(0)
    M = 16
    probe = make(sdv, env, M, cuda(parent))
    h_in = sdgen.normal(sdgen.key(7, 1), (M, spec.hidden))
    probe.h.copy_(cuda(h_in))
    probe.run()
    am = host(probe.argmax)
    tokens = sdgen.uniform_tokens(sdgen.key(7, 2), M, spec.vocab)
    for child in (2, 5, 11):  # 0 -> 2 -> 5 -> 11 follows the argmax
        tokens[child] = am[parent[child]]
    a, b = run_both(sdv, env, M, tokens, parent=parent, h_in=h_in)
    assert same(a.logits, b.logits)
    n = int(host(b.out_count)[0])
    assert list(host(b.out_tokens)[:n]) == [tokens[2], tokens[5], tokens[11], am[11]]
    assert torch.equal(a.out_tokens[:n], b.out_tokens[:n])


def test_pipeline_small_stack_vs_oracle(sdv):
    """The per-operation pipeline on a small stack against the oracle's composition: every stage's
    codes are float-derived, so this is checked loosely (logits within a few percent, argmax of
    the oracle reached within its tolerance); the bit-exact contract is per stage."""
    env = small_stack(sdv, seed=2)
    spec, _, _, host_w, _, head_b = env
    M = 5
    st = make(sdv, env, M)
    h = spec.hidden_in(M)
    st.h.copy_(cuda(h))
    st.run()
    status_ok()
    for l in range(spec.layers):
        n1, n2 = spec.norms(l)
        h = oracle.stack_layer(h, host_w[l], n1, n2, spec.hidden, spec.ffn, spec.wq)
    lo, ao, _, _ = oracle.head(h, spec.final_norm(), head_b, spec.vocab, spec.hidden)
    lg = host(st.logits)
    assert np.abs(lg - lo).max() <= 0.05 * np.abs(lo).max()
    assert (host(st.argmax) == ao).mean() >= 0.6


def test_fused_pass_rejects_bad_plans(sdv):
    import ctypes
    env = small_stack(sdv, L=1)
    st = make(sdv, env, 5)
    st.prepare_fused()
    bad = sdv.SdPass()
    bad.plan = None
    assert sdv.lib().sd_verify_pass(ctypes.byref(bad), None) == 1


@pytest.mark.parametrize("certainty", [False, True])
@pytest.mark.parametrize("M", [1, 5])
def test_fused_pass_sampled_acceptance(sdv, M, certainty):
    """The one-launch pass ending in rejection sampling against the per-operation pass followed by
    sd_accept_sample (bit-equal tokens, logits and statistics), and against the oracle's rule on
    the pass's own logits."""
    env = small_stack(sdv, seed=3)
    spec = env[0]
    V, K, T = spec.vocab, M - 1, 0.8
    h0 = cuda(spec.hidden_in(M))
    probe = make(sdv, env, M)
    probe.h.copy_(h0)
    probe.run()
    am = host(probe.argmax)
    lg = host(probe.logits)
    qp = None if certainty or K == 0 else np.stack(
        [oracle.softmax_probs(lg[i] / T + sdgen.normal(sdgen.key(140, i), (V,))) for i in range(K)]).astype(np.float32)
    qd = cuda(qp) if qp is not None else None
    rng = np.random.default_rng(141)
    a, b = make(sdv, env, M), make(sdv, env, M)
    for t in range(6):
        drafts = np.where(rng.random(K) < 0.6, am[:K], rng.integers(0, V, K)).astype(np.int32)
        seed, base = 1000 + t, 17 * t
        for st in (a, b):
            st.h.copy_(h0)
            if K:
                st.tokens[:K].copy_(cuda(drafts))
        for l in range(spec.layers):
            a.layer(l)
        a.head(T)
        a.accept_sampled(T, seed, base, q_probs=qd)
        b.prepare_fused(temperature=T, sample=True, seed=seed, base_pos=base, q_probs=qd)
        b.run_fused()
        status_ok()
        for name in ("logits", "argmax", "row_max", "row_sumexp"):
            assert same(getattr(a, name), getattr(b, name)), name
        n = int(host(a.out_count)[0])
        assert int(host(b.out_count)[0]) == n and n >= 1
        assert torch.equal(a.out_tokens[:n], b.out_tokens[:n])
        ref = oracle.accept_sample(host(b.logits), qp, drafts, T, seed, base)
        assert list(host(b.out_tokens)[:n]) == list(ref), t


def test_fused_pass_sampling_rejects_trees(sdv):
    env = small_stack(sdv, L=1)
    parent, _ = sdgen.tree16(0)
    st = make(sdv, env, 16, cuda(parent))
    with pytest.raises(sdv.SdError) as e:
        st.prepare_fused(sample=True)
    assert e.value.code == 2  # SD_EUNSUPPORTED


@pytest.mark.parametrize("top_k,top_p,certainty", [(1, 1.0, True), (20, 0.95, False), (32, 0.6, True)])
def test_fused_pass_filtered_sampling(sdv, top_k, top_p, certainty):
    """The one-launch pass ending in rejection sampling against the top-k / top-p filtered target,
    against the per-operation pass + sd_accept_sample_topk and the oracle's rule on its logits."""
    env = small_stack(sdv, seed=4)
    spec = env[0]
    M, V, T = 5, spec.vocab, 0.9
    K = M - 1
    h0 = cuda(spec.hidden_in(M))
    probe = make(sdv, env, M)
    probe.h.copy_(h0)
    probe.run()
    am, lg = host(probe.argmax), host(probe.logits)
    qp = None if certainty else np.stack(
        [oracle.softmax_probs(lg[i] / T + sdgen.normal(sdgen.key(142, i), (V,))) for i in range(K)]).astype(np.float32)
    qd = cuda(qp) if qp is not None else None
    rng = np.random.default_rng(143)
    a, b = make(sdv, env, M), make(sdv, env, M)
    for t in range(5):
        drafts = np.where(rng.random(K) < 0.7, am[:K], rng.integers(0, V, K)).astype(np.int32)
        seed, base = 2000 + t, 11 * t
        for st in (a, b):
            st.h.copy_(h0)
            st.tokens[:K].copy_(cuda(drafts))
        for l in range(spec.layers):
            a.layer(l)
        a.head(T)
        a.accept_sampled(T, seed, base, q_probs=qd, top_k=top_k, top_p=top_p)
        b.prepare_fused(temperature=T, sample=True, seed=seed, base_pos=base, q_probs=qd, top_k=top_k, top_p=top_p)
        b.run_fused()
        status_ok()
        assert same(a.logits, b.logits)
        n = int(host(a.out_count)[0])
        assert int(host(b.out_count)[0]) == n and n >= 1
        assert torch.equal(a.out_tokens[:n], b.out_tokens[:n])
        ref = oracle.accept_sample_topk(host(b.logits), qp, drafts, T, top_k, top_p, seed, base)
        assert list(host(b.out_tokens)[:n]) == list(ref), t
        if top_k == 1:  # the greedy chain rule on the pass's argmax
            assert list(ref) == list(oracle.accept_greedy_chain(host(b.argmax), drafts))
