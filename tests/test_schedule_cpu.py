"""The matmul's work partition, replayed on the host with the kernels' own schedule code
(sd_debug_schedule, no GPU): every (split, unit, block) step is processed by exactly one CTA, each
piece names the CTAs that share its unit-split, pieces never cross a unit-split, each CTA's work is
within one step of the mean (stream-K balance), and every CTA ends on a piece flagged last."""
import ctypes

import numpy as np
import pytest

Q8_0, Q4_32, Q4_K, Q6_K = 0, 1, 2, 3


@pytest.fixture(scope="module")
def L():
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    import speculative_decoding_verify_gb300 as sdv
    return sdv.lib()


def schedule(L, qtype, n_out, k_in, pair=False, head=False, sms=152):
    plan = np.zeros(9, np.int32)
    cap = 1 << 16
    rows = np.zeros((cap, 8), np.int32)
    n = L.sd_debug_schedule(qtype, n_out, k_in, int(pair), int(head), sms, plan.ctypes.data, rows.ctypes.data, cap)
    assert n > 0, n
    return dict(zip("KB NU KS KBs KBlast G P D R".split(), plan.tolist())), rows[:n]


SHAPES = [
    # the 27B-shaped projections and head
    (Q4_32, 3 * 5120, 5120, False, False), (Q4_32, 5120, 5120, False, False), (Q4_32, 2 * 17408, 5120, True, False),
    (Q4_32, 5120, 17408, False, False), (Q8_0, 151936, 5120, False, True),
    # small, ragged and tall-k shapes, fewer units than CTAs
    (Q4_32, 512, 512, False, False), (Q8_0, 33, 64, False, False), (Q4_32, 1024, 1024, True, False),
    (Q4_32, 640, 17408, False, False), (Q8_0, 4096, 1024, False, True), (Q4_32, 65536, 17408, False, False),
    (Q4_32, 32, 32, False, False), (Q8_0, 100, 2048, False, False),
    # K-quant super-blocks: every piece a whole number of 256-weight super-blocks
    (Q4_K, 3 * 5120, 5120, False, False), (Q4_K, 2 * 17408, 5120, True, False), (Q6_K, 5120, 17408, False, False),
    (Q4_K, 32, 256, False, False), (Q6_K, 640, 17408, False, False), (Q4_K, 4800, 2560, False, False),
]


@pytest.mark.parametrize("qtype,n_out,k_in,pair,head", SHAPES)
@pytest.mark.parametrize("sms", [152, 7])
def test_partition_covers_every_step_once(L, qtype, n_out, k_in, pair, head, sms):
    p, rows = schedule(L, qtype, n_out, k_in, pair, head, sms)
    KB, NU, KS, KBs, KBlast, G = p["KB"], p["NU"], p["KS"], p["KBs"], p["KBlast"], p["G"]
    assert NU == (n_out // 64 if pair else (n_out + 31) // 32) and KB == k_in // 32
    assert KBs * (KS - 1) + KBlast == KB and 1 <= KBlast <= KBs
    seen = {}
    owners = {}
    work = np.zeros(G, np.int64)
    gr = 8 if qtype in (Q4_K, Q6_K) else 1
    assert KBs % gr == 0 and KBlast % gr == 0
    for cta, s, u, j0, j1, first, np_, last in rows:
        ln = KBlast if s == KS - 1 else KBs
        assert 0 <= s < KS and 0 <= u < NU and 0 <= j0 < j1 <= ln  # never crosses a unit-split
        assert j0 % gr == 0 and j1 % gr == 0                       # nor a K-quant super-block
        assert first <= cta < first + np_
        key = (s, u)
        owners.setdefault(key, set()).add(int(cta))
        prev = seen.setdefault(key, [])
        prev.append((j0, j1, first, np_))
        work[cta] += j1 - j0
    assert set(seen) == {(s, u) for s in range(KS) for u in range(NU)}
    for (s, u), segs in seen.items():
        ln = KBlast if s == KS - 1 else KBs
        segs.sort()
        assert segs[0][0] == 0 and segs[-1][1] == ln
        assert all(a[1] == b[0] for a, b in zip(segs, segs[1:]))  # contiguous, no overlap
        firsts = {x[2] for x in segs}
        nps = {x[3] for x in segs}
        assert len(firsts) == 1 and len(nps) == 1                 # one answer per unit-split
        f, n = firsts.pop(), nps.pop()
        assert owners[(s, u)] == set(range(f, f + n))             # exactly the CTAs that hold a piece
    W = KB * NU
    assert work.sum() == W
    # balance: the shared steps split evenly, whole units in equal numbers
    assert work.max() - work.min() <= (KB if p["D"] > 0 else gr) + gr
    # every CTA has work, and its last piece is the one flagged last
    ctas = rows[:, 0]
    assert set(ctas.tolist()) == set(range(G))
    for c in range(G):
        flags = rows[ctas == c, 7]
        assert flags[-1] == 1 and flags[:-1].sum() == 0


def test_rejected_shapes(L):
    plan = np.zeros(9, np.int32)
    rows = np.zeros((4, 8), np.int32)
    assert L.sd_debug_schedule(Q4_32, 5120, 100, 0, 0, 152, plan.ctypes.data, rows.ctypes.data, 4) == -1
    assert L.sd_debug_schedule(Q4_32, 5120, 5120, 0, 0, 152, plan.ctypes.data, rows.ctypes.data, 4) == -2
