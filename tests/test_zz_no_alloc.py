"""The allocation-free matmul entry point (sd_qmatmul_multipos_noalloc) against
the workspace entry point (sd_qmatmul_multipos) and the oracle.

Collected last on purpose: it must pass after every other test has run in the
same process, and alone in a fresh one (its fixture builds and loads the
library itself).  It runs the same kernel on the same work plan as the
workspace call -- only the address of the scratch differs -- so its outputs
must equal that call's bit for bit, on two calls in a row (the static scratch
comes back usable).  A call beyond the scratch's size is refused, not launched.
"""
import numpy as np
import pytest
import torch

import oracle
import sdgen
from _util import acts, assert_close, cuda, host, status_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sdv():
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    import speculative_decoding_verify_gb300 as m
    m.lib()
    return m


def outputs(sdv, M, n, k, epi, col0):
    y = torch.full((M, n), float("nan"), dtype=torch.float32, device="cuda")
    qn = sn = None
    if epi == sdv.EPI_REQUANT:
        qn = torch.zeros((M, n - col0), dtype=torch.int8, device="cuda")
        sn = torch.zeros((M, (n - col0) // 32), dtype=torch.float32, device="cuda")
    elif epi == sdv.EPI_SILU_MUL_REQUANT:
        qn = torch.zeros((M, n // 2), dtype=torch.int8, device="cuda")
        sn = torch.zeros((M, n // 64), dtype=torch.float32, device="cuda")
    return y, qn, sn


# (n_out, k_in, epilogue, requant_col0): a residual projection split over k, a V-requant, a gate|up pair,
# and the 27B-shaped down projection (17408 -> 5120)
CASES = [(640, 17408, 0, 0), (3 * 512, 512, 1, 1024), (2 * 1024, 512, 2, 0), (5120, 17408, 0, 0)]


@pytest.mark.parametrize("n,k,epi,col0", CASES)
def test_noalloc_equals_workspace_call_twice(sdv, n, k, epi, col0):
    M = 5
    qt = oracle.Q4_32
    pair = epi == sdv.EPI_SILU_MUL_REQUANT
    blocks = sdgen.quantized_normal(qt, sdgen.key(170, n, k), n, k)
    q, s = acts(sdgen.key(171, k), M, k)
    r = sdgen.normal(sdgen.key(172, n), (M, n)) if epi == 0 else None
    w = sdv.repack_weights(qt, cuda(blocks).reshape(-1), n, k, pair)
    qd, sd = cuda(q), cuda(s)
    res = cuda(r) if r is not None else None

    # the existing entry point with its own workspace
    ws = sdv.workspace(sdv.qmatmul_workspace_bytes(qt, n, k, epi))
    y0, qn0, sn0 = outputs(sdv, M, n, k, epi, col0)
    sdv.qmatmul_multipos(qt, w, n, k, qd, sd, ws, y=y0, residual=res, epilogue=epi, requant_col0=col0,
                         q_next=qn0, scales_next=sn0)
    status_ok()
    yo, ab = oracle.qmatmul(qt, blocks, n, k, q, s, residual=r)

    for _ in range(2):  # two calls in a row on the one static scratch
        y1, qn1, sn1 = outputs(sdv, M, n, k, epi, col0)
        sdv.qmatmul_multipos_noalloc(qt, w, n, k, qd, sd, y=y1, residual=res, epilogue=epi, requant_col0=col0,
                                     q_next=qn1, scales_next=sn1)
        status_ok()
        # same kernel, same plan, same reduction order: identical bits, not merely within tolerance
        assert np.array_equal(host(y1).view(np.uint32), host(y0).view(np.uint32)), f"noalloc vs workspace {n}x{k}"
        assert_close(host(y1), yo, ab, f"noalloc vs oracle {n}x{k}")
        if qn1 is not None:
            assert np.array_equal(host(qn1), host(qn0)) and np.array_equal(host(sn1), host(sn0))


def test_noalloc_rejects_calls_beyond_its_scratch(sdv):
    # fewer 32-row units than SMs and thirteen k-splits: every unit is shared across CTAs, whose
    # partial sums (several MB) do not fit the static scratch
    N, K, M = 4800, 65536, 5
    assert sdv.qmatmul_workspace_bytes(oracle.Q4_32, N, K, 0) > (4 << 20)  # SD_NOALLOC_SCRATCH_BYTES
    q = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    s = torch.zeros((M, K // 32), dtype=torch.float32, device="cuda")
    w = torch.zeros(16, dtype=torch.uint8, device="cuda")  # never read: the call is refused first
    y = torch.zeros((M, 16), dtype=torch.float32, device="cuda")
    rc = sdv.lib().sd_qmatmul_multipos_noalloc(oracle.Q4_32, sdv._p(w), N, K, sdv._p(q), sdv._p(s), M, sdv._p(y),
                                               None, 0, 0, None, None, sdv._stream())
    assert rc == 2  # SD_EUNSUPPORTED
    status_ok()
