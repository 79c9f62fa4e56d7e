"""Where the oracle's RMSNorm codes may differ from the plain definition, and by how much.

The oracle (reading R4) forms the codes of an RMSNorm from t = x*w and the block
scale as inv * max|t| / 127.  The plain definition normalises first, y =
(x*inv)*w (two rounded multiplies), and requantises y: d = max|y| / 127, q =
round-half-away(y / d).  In exact arithmetic the two give the same codes (the
positive row factor inv cancels in y / d); in fp32 they can differ by one step
only where the plain quotient y / d lies within a few roundings of a half-integer.

``compare_site`` measures that on one norm site: the number of codes, how many
differ, the largest distance of a differing code's plain quotient from the
nearest half-integer, and the largest scale difference in fp32 ulps.  It is test
infrastructure (the RMSNorm pin and the script that writes the stored
statistics of the 64-layer stack call it), not a product path.
"""
from __future__ import annotations

import numpy as np

import oracle

# A code is "at a rounding tie" when its plain quotient is within TIE of k + 1/2: the two
# orders differ by at most about six fp32 roundings of a quotient of magnitude <= 127.5,
# under 5e-5 absolute; twice that is the band.
TIE = 1e-4


def plain_rmsnorm_quant(x: np.ndarray, w: np.ndarray, eps: float):
    """The plain definition in fp32: inv from the float64 mean square (rounded once to fp32),
    y = (x inv) w with two rounded multiplies, then the per-32 requantisation of y."""
    x = np.asarray(x, np.float32)
    w = np.asarray(w, np.float32)
    M, K = x.shape
    ms = (x.astype(np.float64) ** 2).mean(axis=1)
    inv = (1.0 / np.sqrt(ms + eps)).astype(np.float32)
    y = (x * inv[:, None]).astype(np.float32) * w[None, :]
    y = y.astype(np.float32)
    yb = y.reshape(M, K // 32, 32)
    d = (np.abs(yb).max(axis=2) / np.float32(127.0)).astype(np.float32)
    safe = np.where(d == 0, np.float32(1.0), d)
    quot = (yb / safe[..., None]).astype(np.float32).astype(np.float64)  # one IEEE fp32 division
    q = np.sign(quot) * np.floor(np.abs(quot) + 0.5)  # half away from zero, exact in float64
    q = np.clip(q, -127, 127)
    q = np.where(d[..., None] == 0, 0, q)
    exact_quot = yb.astype(np.float64) / np.where(d == 0, 1.0, d.astype(np.float64))[..., None]
    return q.reshape(M, K).astype(np.int8), d, exact_quot.reshape(M, K)


def compare_site(x: np.ndarray, w: np.ndarray, eps: float) -> dict:
    qo, so = oracle.rmsnorm_quant(x, w, eps)
    qp, sp, quot = plain_rmsnorm_quant(x, w, eps)
    diff = qo != qp
    frac = np.abs(quot) - np.floor(np.abs(quot))
    tie_dist = np.abs(frac - 0.5)
    step = np.abs(qo.astype(np.int32) - qp.astype(np.int32))
    ulp = np.spacing(np.maximum(np.abs(sp), np.float32(1e-30))).astype(np.float64)
    scale_ulps = np.abs(so.astype(np.float64) - sp.astype(np.float64)) / ulp
    return {
        "codes": int(qo.size),
        "differing": int(diff.sum()),
        "max_step": int(step.max()) if step.size else 0,
        "max_tie_distance_of_differing": float(tie_dist[diff].max()) if diff.any() else 0.0,
        "max_scale_ulps": float(scale_ulps.max()) if scale_ulps.size else 0.0,
    }


def stack_sites(spec, M: int, layers: int):
    """(name, x, w) of each RMSNorm site of the oracle's own pass over the first `layers` layers
    of the stack (two per layer: before QKV and before gate|up; then the final norm when all
    layers are run), on the stack's input rows."""
    h = spec.hidden_in(M)
    for l in range(layers):
        wts = {name: spec.weights(l, name) for name, _, _ in spec.matrices()}
        n1, n2 = spec.norms(l)
        tr = {}
        h_next = oracle.stack_layer(h, wts, n1, n2, spec.hidden, spec.ffn, spec.wq, trace=tr)
        yield f"layer{l}.norm1", h, n1
        yield f"layer{l}.norm2", tr["h2"], n2
        h = h_next
    if layers == spec.layers:
        yield "final_norm", h, spec.final_norm()
