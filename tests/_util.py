"""Shared helpers of the GPU tests: moving seeded inputs to the device, running
one ABI call, unpacking the repacked layout, and the float tolerance."""
import numpy as np
import torch

import oracle
import sdgen

RTOL = 1e-5  # |gpu - oracle| <= RTOL * (|residual| + sum_b |d_w d_a dot_b|) + 1 ulp of the oracle value


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def acts(key, M, K, scale=1.0):
    """Seeded int8 activations + scales: normal rows requantised by the oracle."""
    x = sdgen.normal(key, (M, K)) * scale
    return oracle.rmsnorm_quant(x, None)


def assert_close(g, o, absb, what=""):
    g = np.asarray(g, dtype=np.float64)
    o32 = np.asarray(o, dtype=np.float32)
    err = np.abs(g - o32.astype(np.float64))
    bound = RTOL * np.asarray(absb, dtype=np.float64) + np.spacing(np.abs(o32)).astype(np.float64)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst {(err / bound).max():.3g}x"
    return float((err / np.maximum(np.abs(o32), 1e-30)).max())


def unpack_repacked(qtype, buf, n_out, k_in, pair=False):
    """Inverse of the documented repack layout -> GGUF-order blocks [n_out][k_in/32 * bb]."""
    buf = np.asarray(buf, dtype=np.uint8)
    KB = k_in // 32
    bb = oracle.BLOCK_BYTES[qtype]
    rec = 1088 if qtype == oracle.Q8_0 else 576
    code = 1024 if qtype == oracle.Q8_0 else 512
    out = np.zeros((n_out, KB, bb), dtype=np.uint8)
    if pair:
        F = n_out // 2
        nt = (F + 31) // 32
        recs = buf.reshape(nt, KB, 2, rec)
    else:
        nt = (n_out + 31) // 32
        recs = buf.reshape(nt, KB, 1, rec)
    for t in range(nt):
        for h in range(recs.shape[2]):
            r = recs[t, :, h, :]                   # [KB][rec]
            rows = np.arange(32) + t * 32
            if pair:
                rows = rows + h * (n_out // 2)
                valid = (np.arange(32) + t * 32) < n_out // 2
            else:
                valid = rows < n_out
            for i in np.nonzero(valid)[0]:
                n = rows[i]
                out[n, :, 0] = r[:, code + 2 * i]
                out[n, :, 1] = r[:, code + 2 * i + 1]
                if qtype == oracle.Q8_0:
                    out[n, :, 2:18] = r[:, i * 16:(i + 1) * 16]
                    out[n, :, 18:34] = r[:, 512 + i * 16:512 + (i + 1) * 16]
                else:
                    out[n, :, 2:18] = r[:, i * 16:(i + 1) * 16]
    return out.reshape(n_out, KB * bb)


def status_ok():
    import speculative_decoding_verify_gb300 as sdv
    torch.cuda.synchronize()
    st = sdv.device_status()
    assert st == 0, f"device status {st}"
