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
    """Inverse of the documented repack layout -> GGUF-order blocks [n_out][k_in/32 * bb].

    Record = 32 rows x one 32-weight block; lane l = 4g + c holds the A fragments of
    mma m16n8k16 for rows 16t+g (+8) and k 16s+2c (+1, +8, +9).  4-bit: word 2t+s of the
    lane's 16 bytes, nibble i at (row 16t+g+8[i&2], k 16s+2c+8[i&1]+(i>>2)).  Q8_0:
    plane t (512 B each), word 2s+h holds (row 16t+g, k0), (.., k0+1), (row 16t+g+8, k0),
    (.., k0+1) with k0 = 16s+2c+8h.  Scales: group g = rows g, g+8, 16+g, 24+g."""
    buf = np.asarray(buf, dtype=np.uint8)
    KB = k_in // 32
    bb = oracle.BLOCK_BYTES[qtype]
    rec = 1088 if qtype == oracle.Q8_0 else 576
    code_b = 1024 if qtype == oracle.Q8_0 else 512
    halves = 2 if pair else 1
    rows_per = n_out // 2 if pair else n_out
    nt = (rows_per + 31) // 32
    recs = buf.reshape(nt, KB, halves, rec)
    vals = np.zeros((nt, halves, 32, KB, 32), dtype=np.int32)   # [tile][half][row][block][k]: code or q
    dsc = np.zeros((nt, halves, 32, KB, 2), dtype=np.uint8)
    for lane in range(32):
        g, c = lane >> 2, lane & 3
        if qtype == oracle.Q4_32:
            words = recs[:, :, :, lane * 16:(lane + 1) * 16].reshape(nt, KB, halves, 4, 4).astype(np.uint32)
            words = (words[..., 0] | (words[..., 1] << 8) | (words[..., 2] << 16) | (words[..., 3] << 24))
            for j in range(4):
                t, s_ = j >> 1, j & 1
                for i in range(8):
                    row = 16 * t + g + (8 if i & 2 else 0)
                    k = 16 * s_ + 2 * c + (8 if i & 1 else 0) + (i >> 2)
                    vals[:, :, row, :, k] = ((words[:, :, :, j] >> (4 * i)) & 0xF).transpose(0, 2, 1)
        else:
            for t in range(2):
                plane = recs[:, :, :, t * 512 + lane * 16:t * 512 + (lane + 1) * 16].reshape(nt, KB, halves, 4, 4)
                for wq in range(4):
                    s_, h = wq >> 1, wq & 1
                    k0 = 16 * s_ + 2 * c + 8 * h
                    for e, (dr, dk) in enumerate(((0, 0), (0, 1), (8, 0), (8, 1))):
                        vals[:, :, 16 * t + g + dr, :, k0 + dk] = plane[:, :, :, wq, e].astype(np.int8).transpose(0, 2, 1)
        if c == 0:
            for e, row in enumerate((g, g + 8, 16 + g, 24 + g)):
                off = code_b + g * 8 + 2 * e
                dsc[:, :, row, :, :] = recs[:, :, :, off:off + 2].transpose(0, 2, 1, 3)
    out = np.zeros((n_out, KB, bb), dtype=np.uint8)
    for h in range(halves):
        blockrows = np.arange(nt * 32)
        valid = blockrows < rows_per
        v = vals[:, h].reshape(nt * 32, KB, 32)[valid]
        d = dsc[:, h].reshape(nt * 32, KB, 2)[valid]
        r0 = h * rows_per
        out[r0:r0 + rows_per, :, 0:2] = d
        if qtype == oracle.Q8_0:
            out[r0:r0 + rows_per, :, 2:] = v.astype(np.int8).view(np.uint8)
        else:
            out[r0:r0 + rows_per, :, 2:] = (v[:, :, :16] | (v[:, :, 16:] << 4)).astype(np.uint8)
    return out.reshape(n_out, KB * bb)


def status_ok():
    import speculative_decoding_verify_gb300 as sdv
    torch.cuda.synchronize()
    st = sdv.device_status()
    assert st == 0, f"device status {st}"


def unpack_kq_repacked(qtype, buf, n_out, k_in, pair=False):
    """Inverse of the documented K-quant super-record layout -> GGUF super-blocks [n_out][k_in/256 * bb]
    (Q4_K 144 B: d, dmin, 12 packed (scale, min) bytes, 128 code bytes; Q6_K 210 B: 128 low-nibble
    bytes, 64 high-bit bytes, 16 int8 scales, d).  Codes: sub-block s plane, lane l = 4g + c, word j =
    2t+s' holds nibble i at (row 16t+g+8[i&2], weight 32s + 16s'+2c+8[i&1]+(i>>2)); Q6_K high bits of
    word j at the documented positions of the lane's high-bit word j//2."""
    buf = np.asarray(buf, dtype=np.uint8)
    SBK = k_in // 256
    q4 = qtype == oracle.Q4_K
    srb, bb, plane = (4736, 144, 512) if q4 else (6720, 210, 768)
    halves = 2 if pair else 1
    rows_per = n_out // 2 if pair else n_out
    nt = rows_per // 32
    sr = buf.reshape(nt, SBK, halves, srb)
    code = np.zeros((nt, halves, 32, SBK, 256), dtype=np.int32)  # unsigned codes (Q6_K: 0..63)
    p0 = [4, 8, 6, 10, 20, 24, 22, 26]
    p1 = [0, 2, 12, 14, 16, 18, 28, 30]

    def u32(a):
        a = a.astype(np.uint32)
        return a[..., 0] | (a[..., 1] << 8) | (a[..., 2] << 16) | (a[..., 3] << 24)

    for s in range(8):
        for lane in range(32):
            g, c = lane >> 2, lane & 3
            base = s * plane + lane * 16
            words = u32(sr[..., base:base + 16].reshape(nt, SBK, halves, 4, 4))
            if not q4:
                hb = s * plane + 512 + lane * 8
                hw = u32(sr[..., hb:hb + 8].reshape(nt, SBK, halves, 2, 4))
            for j in range(4):
                t, sk = j >> 1, j & 1
                for i in range(8):
                    row = 16 * t + g + (8 if i & 2 else 0)
                    k = 32 * s + 16 * sk + 2 * c + (8 if i & 1 else 0) + (i >> 2)
                    v = (words[..., j] >> (4 * i)) & 0xF
                    if not q4:
                        pos = (p1 if j & 1 else p0)[i]
                        v = v | (((hw[..., j >> 1] >> pos) & 3) << 4)
                    code[:, :, row, :, k] = v.transpose(0, 2, 1)
    out = np.zeros((nt, halves, 32, SBK, bb), dtype=np.uint8)
    for g in range(8):
        for e, row in enumerate((g, g + 8, 16 + g, 24 + g)):
            if q4:
                sc = np.stack([sr[..., 4096 + 64 * s + 8 * g + e] for s in range(8)], -1).astype(np.int32)
                mn = np.stack([sr[..., 4096 + 64 * s + 8 * g + 4 + e] for s in range(8)], -1).astype(np.int32)
                b = np.zeros(sc.shape[:-1] + (12,), dtype=np.int32)
                for s in range(4):
                    b[..., s] = (sc[..., s] & 63) | ((sc[..., s + 4] >> 4) << 6)
                    b[..., s + 4] = (mn[..., s] & 63) | ((mn[..., s + 4] >> 4) << 6)
                    b[..., s + 8] = (sc[..., s + 4] & 15) | ((mn[..., s + 4] & 15) << 4)
                dd = sr[..., 4608 + 16 * g + 4 * e:4608 + 16 * g + 4 * e + 4]
                out[:, :, row, :, 0:4] = dd.transpose(0, 2, 1, 3)
                out[:, :, row, :, 4:16] = b.astype(np.uint8).transpose(0, 2, 1, 3)
            else:
                scs = np.stack([sr[..., 6144 + 64 * s + 8 * g + 4 * h + e] for s in range(8) for h in range(2)], -1)
                out[:, :, row, :, 192:208] = scs.transpose(0, 2, 1, 3)
                out[:, :, row, :, 208:210] = sr[..., 6656 + 8 * g + 2 * e:6656 + 8 * g + 2 * e + 2].transpose(0, 2, 1, 3)
    # codes into the file's order
    i = np.arange(256)
    if q4:
        cidx, r = i // 64, i % 64
        byte = 16 + 32 * cidx + (r % 32)
        for hi in (0, 1):
            sel = (r >= 32) == bool(hi)
            vals = code[..., sel] << (4 * hi)
            out[..., byte[sel]] |= vals.astype(np.uint8)
    else:
        n_, r = i // 128, i % 128
        l, kq = r % 32, r // 32
        lo_byte = 64 * n_ + l + 32 * (kq & 1)
        hi_byte = 128 + 32 * n_ + l
        for sel_k in range(4):
            sel = kq == sel_k
            lo = code[..., sel] & 15
            out[..., lo_byte[sel]] |= (lo << (4 if sel_k >= 2 else 0)).astype(np.uint8)
            out[..., hi_byte[sel]] |= ((code[..., sel] >> 4) << (2 * sel_k)).astype(np.uint8)
    o = out.reshape(nt, halves, 32, SBK * bb)
    res = np.zeros((n_out, SBK * bb), dtype=np.uint8)
    for h in range(halves):
        res[h * rows_per:(h + 1) * rows_per] = o[:, h].reshape(rows_per, SBK * bb)
    return res
