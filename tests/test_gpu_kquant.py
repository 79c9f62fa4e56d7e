"""K-quant formats (Q4_K, Q6_K super-blocks of 256 weights) on the GPU, against the oracle.

* The load-time repack moves bytes only: the super-records unpack (tests/_util.py restates the
  documented layout) to the input super-blocks byte for byte, with and without the gate|up pairing.
* The multi-position matmul over the repacked weights equals the oracle's factored fp64 product
  within the fp32 tolerance (1e-5 of the absolute sum of the terms, reading R5) at the 27B-shaped
  widths (5120 and 17408) and on small and ragged shapes, for M = 1, 5 and 16.
* Batch invariance: rows computed among M positions equal the same rows computed alone, bit for bit.
* Epilogues: the V-requantising QKV shape, a residual projection, and the SiLU*mul gate|up pair,
  whose codes equal the library's own requantisation of the pair's outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import sdgen
from _util import acts, assert_close, cuda, host, status_ok, unpack_kq_repacked

pytestmark = pytest.mark.gpu

Q4_K, Q6_K = oracle.Q4_K, oracle.Q6_K


@pytest.fixture(scope="module")
def sdv():
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    import speculative_decoding_verify_gb300 as m
    m.lib()
    return m


def blocks(qtype, key, n, k):
    return sdgen.random_kq_blocks(qtype, sdgen.key(180, key, qtype, n, k), n, k)


@pytest.mark.parametrize("qtype,n,k,pair", [(Q4_K, 64, 512, False), (Q6_K, 64, 512, False), (Q4_K, 128, 768, True),
                                            (Q4_K, 5120, 5120, False), (Q6_K, 5120, 17408, False)])
def test_kq_repack_roundtrip_bytes_unchanged(sdv, qtype, n, k, pair):
    b = blocks(qtype, 1, n, k)
    w = sdv.repack_weights(qtype, cuda(b).reshape(-1), n, k, pair)
    status_ok()
    assert w.numel() == n // 32 * (k // 256) * (4736 if qtype == Q4_K else 6720)
    assert np.array_equal(unpack_kq_repacked(qtype, host(w), n, k, pair), b.reshape(n, -1))


def test_kq_repack_rejects_bad_shapes(sdv):
    L = sdv.lib()
    assert L.sd_repacked_bytes(Q4_K, 5120, 5000, 0) == 0      # k_in % 256
    assert L.sd_repacked_bytes(Q6_K, 100, 512, 0) == 0        # n_out % 32
    assert L.sd_repacked_bytes(Q6_K, 128, 512, 1) == 0        # no gate|up pairing for Q6_K
    assert L.sd_repacked_bytes(Q4_K, 128, 512, 1) == 128 // 32 * (512 // 256) * 4736  # pairs: same bytes


def run_mm(sdv, qtype, w, n, k, q, s, **kw):
    M = q.shape[0]
    ws = sdv.workspace(sdv.qmatmul_workspace_bytes(qtype, n, k, kw.get("epilogue", 0)))
    y = torch.full((M, n), float("nan"), dtype=torch.float32, device="cuda")
    sdv.qmatmul_multipos(qtype, w, n, k, cuda(q), cuda(s), ws, y=y, **kw)
    status_ok()
    return host(y)


SHAPES = [(Q4_K, 32, 256), (Q4_K, 96, 512), (Q6_K, 64, 768), (Q4_K, 4800, 2560), (Q6_K, 160, 17408),
          (Q4_K, 5120, 5120), (Q4_K, 17408, 5120), (Q6_K, 5120, 17408), (Q4_K, 5120, 17408), (Q6_K, 5120, 5120)]


@pytest.mark.parametrize("qtype,n,k", SHAPES)
@pytest.mark.parametrize("M", [1, 5, 16])
def test_kq_matmul_vs_oracle(sdv, qtype, n, k, M):
    b = blocks(qtype, 2, n, k)
    w = sdv.repack_weights(qtype, cuda(b).reshape(-1), n, k)
    q, s = acts(sdgen.key(181, k, M), M, k)
    yo, ab = oracle.kq_matmul(qtype, b, n, k, q, s, with_bound=True)
    g = run_mm(sdv, qtype, w, n, k, q, s)
    assert_close(g, yo, ab, f"{'Q4_K' if qtype == Q4_K else 'Q6_K'} {n}x{k} M={M}")


@pytest.mark.parametrize("qtype,n,k", [(Q4_K, 5120, 5120), (Q6_K, 5120, 17408), (Q4_K, 96, 512)])
def test_kq_rows_equal_rows_alone(sdv, qtype, n, k):
    b = blocks(qtype, 3, n, k)
    w = sdv.repack_weights(qtype, cuda(b).reshape(-1), n, k)
    q, s = acts(sdgen.key(182, k), 16, k)
    y16 = run_mm(sdv, qtype, w, n, k, q, s)
    y8 = run_mm(sdv, qtype, w, n, k, q[:8], s[:8])
    for M in (1, 2, 3, 5):
        yM = run_mm(sdv, qtype, w, n, k, q[:M], s[:M])
        assert np.array_equal(yM.view(np.uint32), y8[:M].view(np.uint32)), M
    for m in (0, 7, 8, 15):  # the two-tile (M > 8) path: each row alone
        y1 = run_mm(sdv, qtype, w, n, k, q[m:m + 1], s[m:m + 1])
        assert np.array_equal(y1.view(np.uint32), y16[m:m + 1].view(np.uint32)), m


def test_kq_epilogues(sdv):
    H, F, M = 512, 1024, 5
    # QKV-shaped Q4_K with the V columns requantised
    b = blocks(Q4_K, 4, 3 * H, H)
    w = sdv.repack_weights(Q4_K, cuda(b).reshape(-1), 3 * H, H)
    q, s = acts(sdgen.key(183, 1), M, H)
    qn = torch.zeros((M, H), dtype=torch.int8, device="cuda")
    sn = torch.zeros((M, H // 32), dtype=torch.float32, device="cuda")
    y = run_mm(sdv, Q4_K, w, 3 * H, H, q, s, epilogue=sdv.EPI_REQUANT, requant_col0=2 * H, q_next=qn, scales_next=sn)
    yo, ab = oracle.kq_matmul(Q4_K, b, 3 * H, H, q, s, with_bound=True)
    assert_close(y, yo, ab, "qkv")
    qq = torch.zeros_like(qn)
    ss = torch.zeros_like(sn)
    sdv.rmsnorm_quant_acts(cuda(y[:, 2 * H:]), None, qq, ss, K=H)
    status_ok()
    assert torch.equal(qq, qn) and torch.equal(ss, sn)
    # Q6_K residual projection
    b6 = blocks(Q6_K, 5, H, F)
    w6 = sdv.repack_weights(Q6_K, cuda(b6).reshape(-1), H, F)
    q6, s6 = acts(sdgen.key(183, 2), M, F)
    r = sdgen.normal(sdgen.key(183, 3), (M, H))
    yr = torch.from_numpy(r).cuda()
    ws = sdv.workspace(sdv.qmatmul_workspace_bytes(Q6_K, H, F))
    sdv.qmatmul_multipos(Q6_K, w6, H, F, cuda(q6), cuda(s6), ws, y=yr, residual=yr)
    status_ok()
    yo6, ab6 = oracle.kq_matmul(Q6_K, b6, H, F, q6, s6, with_bound=True)
    assert_close(host(yr), yo6 + r, ab6 + np.abs(r), "residual")
    # Q4_K gate|up pair with the SiLU*mul requantisation
    bg = blocks(Q4_K, 6, 2 * F, H)
    wg = sdv.repack_weights(Q4_K, cuda(bg).reshape(-1), 2 * F, H, pair=True)
    qf = torch.zeros((M, F), dtype=torch.int8, device="cuda")
    sf = torch.zeros((M, F // 32), dtype=torch.float32, device="cuda")
    gu = run_mm(sdv, Q4_K, wg, 2 * F, H, q, s, epilogue=sdv.EPI_SILU_MUL_REQUANT, q_next=qf, scales_next=sf)
    yog, abg = oracle.kq_matmul(Q4_K, bg, 2 * F, H, q, s, with_bound=True)
    assert_close(gu, yog, abg, "gate|up")
    gq, gs = sdv.debug_silu_mul_requant(torch.from_numpy(np.ascontiguousarray(gu[:, :F])).cuda(),
                                        torch.from_numpy(np.ascontiguousarray(gu[:, F:])).cuda())
    status_ok()
    assert torch.equal(gq, qf) and torch.equal(gs, sf)


# ---------------------------------------------------------------------------
# the one-launch pass over a K-quant stack (Q4_K projections, Q6_K down projections, Q8_0 head)
# ---------------------------------------------------------------------------

def kq_stack(sdv, L=3, H=512, F=1024, V=4096):
    from speculative_decoding_verify_gb300.verify_pass import repack_matrix
    spec = sdgen.StackSpec(layers=L, hidden=H, ffn=F, vocab=V, seed=3)
    layers, norms = [], []
    for l in range(L):
        lw = {}
        for name, n, k in spec.matrices():
            qt = Q6_K if name == "down" else Q4_K
            # small super-block scales keep weights near the 0.02 of the other stacks
            b = sdgen.random_kq_blocks(qt, sdgen.key(184, l, n, k), n, k, d_scale=2e-5)
            lw[name] = repack_matrix(qt, b, n, k, pair=(name == "gate_up"))
        layers.append(lw)
        n1, n2 = spec.norms(l)
        norms.append((cuda(n1), cuda(n2)))
    head = repack_matrix(spec.head_q, spec.head(), V, H)
    return spec, layers, norms, head


def kq_make(env, M, parent=None):
    from speculative_decoding_verify_gb300.verify_pass import VerifyStack
    spec, layers, norms, head = env
    return VerifyStack(layers, norms, cuda(spec.final_norm()), head, spec.hidden, spec.ffn, spec.vocab, M,
                       wq=Q4_K, wq_down=Q6_K, tree_parent=parent)


@pytest.mark.parametrize("M", [1, 5, 16])
def test_kq_fused_pass_equals_pipeline(sdv, M):
    """The K-quant pass as one launch against the same calls issued one by one: hidden rows, logits,
    statistics, every requantised activation and the accepted tokens, bit for bit (chain; a tree at
    M = 16)."""
    env = kq_stack(sdv)
    spec = env[0]
    parent = cuda(sdgen.tree16(0)[0]) if M == 16 else None
    h0 = cuda(sdgen.normal(sdgen.key(185, M), (M, spec.hidden)))
    a, b = kq_make(env, M, parent), kq_make(env, M, parent)
    a.h.copy_(h0)
    a.run()
    torch.cuda.synchronize()
    am = host(a.argmax)
    tokens = np.array([am[i] if i < 2 else (am[i] + 1) % spec.vocab for i in range(M)], np.int32)
    if M == 16:
        tokens = np.roll(tokens, 1)
    for st in (a, b):
        st.h.copy_(h0)
        st.tokens[:M].copy_(cuda(tokens))
    a.run()
    b.run_fused()
    status_ok()
    assert b.fused.kq == 1
    for name in ("h", "logits", "argmax", "row_max", "row_sumexp", "qa", "sa", "qv", "sv", "qf", "sf"):
        x, y = getattr(a, name), getattr(b, name)
        assert torch.equal(x.view(torch.int32) if x.dtype == torch.float32 else x,
                           y.view(torch.int32) if y.dtype == torch.float32 else y), name
    assert np.isfinite(host(b.logits)).all()
    n = int(host(a.out_count)[0])
    assert n >= 1 and int(host(b.out_count)[0]) == n
    assert torch.equal(a.out_tokens[:n], b.out_tokens[:n])


def test_kq_pass_rejects_sampling_and_bad_widths(sdv):
    env = kq_stack(sdv, L=1)
    st = kq_make(env, 5)
    with pytest.raises(sdv.SdError):
        st.prepare_fused(sample=True)
