"""The library's host-side cycle helpers (host code in libsdverify.so) against the oracle: the
adaptive draft depth (sd_depth_init / sd_depth_update) step for step on seeded acceptance
sequences, and the accepted tree path (sd_tree_path) on seeded random trees, plus their argument
checks.  No GPU: both run on the host."""
import ctypes

import numpy as np
import pytest

import oracle
import sdgen


@pytest.fixture(scope="module")
def sdv():
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    import speculative_decoding_verify_gb300 as m
    m.lib()
    return m


def drive(sdv, k_max, max_pause, hit_rate, n, seed):
    """Run n cycles; each drafted token is accepted with probability hit_rate until the first
    rejection.  Returns the depths used and the accepted counts fed back."""
    u = sdgen.u32(sdgen.key(9, seed), n * 16).reshape(n, 16) / 2.0 ** 32
    pol = sdv.DepthPolicy(k_max, max_pause)
    used, accs = [], []
    for c in range(n):
        k = pol.k
        acc = 0
        while acc < k and u[c, acc] < hit_rate:
            acc += 1
        used.append(k)
        accs.append(acc)
        pol.update(acc)
    return used, accs


@pytest.mark.parametrize("k_max,max_pause,hit_rate", [(4, 64, 0.7), (4, 64, 0.2), (1, 8, 0.5), (15, 3, 0.9),
                                                      (3, 0, 0.3), (7, 64, 0.02)])
def test_depth_matches_oracle(sdv, k_max, max_pause, hit_rate):
    used, accs = drive(sdv, k_max, max_pause, hit_rate, 400, k_max * 100 + max_pause)
    assert used == oracle.depth_policy(k_max, max_pause, accs)
    assert all(0 <= k <= k_max for k in used)


def test_depth_argument_checks(sdv):
    L = sdv.lib()
    st = sdv.SdDepthState()
    assert L.sd_depth_init(ctypes.byref(st), 0, 4) == 1
    assert L.sd_depth_init(ctypes.byref(st), 16, 4) == 1
    assert L.sd_depth_init(ctypes.byref(st), 4, -1) == 1
    assert L.sd_depth_init(None, 4, 4) == 1
    assert L.sd_depth_init(ctypes.byref(st), 4, 4) == 0 and st.k_next == 4
    assert L.sd_depth_update(ctypes.byref(st), 5) == 1     # more accepted than drafted
    assert L.sd_depth_update(ctypes.byref(st), -1) == 1
    assert st.k_next == 4                                   # a rejected call changes nothing
    assert L.sd_depth_update(ctypes.byref(st), 2) == 0 and st.k_next == 3


def test_tree_path_matches_oracle(sdv):
    u = sdgen.u32(sdgen.key(101), 300 * 64)
    for t in range(300):
        M = 1 + t % 16
        r = u[t * 64:(t + 1) * 64]
        parent = np.array([-1] + [int(r[i] % i) for i in range(1, M)], np.int32)
        argmax = (r[16:16 + M] % 3).astype(np.int32)
        tokens = (r[32:32 + M] % 3).astype(np.int32)
        assert list(sdv.tree_path(argmax, tokens, parent)) == list(
            oracle.accept_greedy_tree_path(argmax, tokens, parent))


def test_tree_path_rejects_malformed_trees(sdv):
    with pytest.raises(sdv.SdError):
        sdv.tree_path([0, 0], [0, 0], [-1, 1])      # a node as its own parent
    with pytest.raises(sdv.SdError):
        sdv.tree_path([0, 0], [0, 0], [0, 0])       # no root
    with pytest.raises(sdv.SdError):
        sdv.tree_path([0] * 17, [0] * 17, [-1] + list(range(16)))


def test_tree_path_rejects_arrays_of_unequal_length(sdv):
    """The C call reads M entries of each array: shorter argmax or parent arrays are refused on the host."""
    with pytest.raises(sdv.SdError):
        sdv.tree_path([0], [0, 0, 0], [-1, 0, 0])   # argmax shorter than tokens
    with pytest.raises(sdv.SdError):
        sdv.tree_path([0, 0, 0], [0, 0, 0], [-1, 0])  # parent shorter than tokens
    with pytest.raises(sdv.SdError):
        sdv.tree_path([], [], [])                     # empty tree
