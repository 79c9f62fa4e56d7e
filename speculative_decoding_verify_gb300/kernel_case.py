"""Run one verify-pass kernel on one seeded layer-sized case, for profiling.

    python -m speculative_decoding_verify_gb300.kernel_case --case gate_up --M 5 --reps 3

Cases: qkv (4-bit 5120->15360, requant epilogue), o (4-bit 5120->5120 + residual),
gate_up (4-bit 5120->2x17408, SiLU*mul requant), down (4-bit 17408->5120 + residual),
head (Q8_0 5120->151936 with argmax/statistics), rmsnorm (M x 5120), and pass:
the one-launch verify pass over --layers 27B-shaped 4-bit layers plus the head.
Prints the mean event-timed duration per launch and the weight-stream GB/s.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import sdgen  # noqa: E402

import speculative_decoding_verify_gb300 as sdv  # noqa: E402

H, F, V = sdgen.HIDDEN, sdgen.FFN, sdgen.VOCAB
CASES = {
    "qkv": (sdv.Q4_32, 3 * H, H, sdv.EPI_REQUANT),
    "o": (sdv.Q4_32, H, H, sdv.EPI_NONE),
    "gate_up": (sdv.Q4_32, 2 * F, H, sdv.EPI_SILU_MUL_REQUANT),
    "down": (sdv.Q4_32, H, F, sdv.EPI_NONE),
    "head": (sdv.Q8_0, V, H, None),
}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", default="gate_up", choices=list(CASES) + ["rmsnorm", "pass"])
    ap.add_argument("--layers", type=int, default=4)
    ap.add_argument("--M", type=int, default=5)
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args()
    sdv.lib()
    M = a.M
    dev = "cuda"
    if a.case == "pass":
        from speculative_decoding_verify_gb300.verify_pass import VerifyStack, repack_matrix
        spec = sdgen.StackSpec(layers=a.layers, hidden=H, ffn=F, vocab=V, seed=0)
        layers, norms = [], []
        for l in range(a.layers):
            lw = {}
            for name, n, k in spec.matrices():
                blocks = sdgen.pinned_quantized_normal(spec.wq, spec.weight_key(l, name), n, k)
                lw[name] = repack_matrix(spec.wq, blocks, n, k, pair=(name == "gate_up"), device=dev)
            layers.append(lw)
            norms.append(tuple(torch.from_numpy(x).to(dev) for x in spec.norms(l)))
        hb = sdgen.pinned_quantized_normal(spec.head_q, spec.weight_key(0, "head"), V, H)
        head = repack_matrix(spec.head_q, hb, V, H, device=dev)
        stack = VerifyStack(layers, norms, torch.from_numpy(spec.final_norm()).to(dev), head, H, F, V, M)
        h0 = torch.from_numpy(spec.hidden_in(M)).to(dev)
        stack.prepare_fused()

        def run():
            stack.h.copy_(h0)
            stack.run_fused()
        nbytes = spec.weight_bytes()
    elif a.case == "rmsnorm":
        x = torch.from_numpy(sdgen.normal(sdgen.key(9, 0), (M, H))).to(dev)
        w = torch.from_numpy(sdgen.norm_weight(sdgen.key(9, 1), H)).to(dev)
        q = torch.zeros((M, H), dtype=torch.int8, device=dev)
        s = torch.zeros((M, H // 32), dtype=torch.float32, device=dev)
        run = lambda: sdv.rmsnorm_quant_acts(x, w, q, s)  # noqa: E731
        nbytes = 0
    else:
        qtype, n, k, epi = CASES[a.case]
        blocks = sdgen.pinned_quantized_normal(qtype, sdgen.key(9, 2, n, k), n, k)
        w = sdv.repack_weights(qtype, blocks.to(dev).reshape(-1), n, k, pair=(epi == sdv.EPI_SILU_MUL_REQUANT))
        xq = torch.from_numpy(sdgen.normal(sdgen.key(9, 3), (M, k))).to(dev)
        q = torch.zeros((M, k), dtype=torch.int8, device=dev)
        s = torch.zeros((M, k // 32), dtype=torch.float32, device=dev)
        sdv.rmsnorm_quant_acts(xq, None, q, s)
        nbytes = n * (k // 32) * sdv.BLOCK_BYTES[qtype]
        if a.case == "head":
            ws = sdv.workspace(sdv.head_workspace_bytes(n, k))
            lg = torch.zeros((M, n), dtype=torch.float32, device=dev)
            am = torch.zeros(M, dtype=torch.int32, device=dev)
            rm = torch.zeros(M, dtype=torch.float32, device=dev)
            rz = torch.zeros(M, dtype=torch.float32, device=dev)
            run = lambda: sdv.head_logits(w, n, k, q, s, ws, lg, am, rm, rz)  # noqa: E731
        else:
            ws = sdv.workspace(sdv.qmatmul_workspace_bytes(qtype, n, k, epi))
            y = torch.zeros((M, n), dtype=torch.float32, device=dev)
            if epi == sdv.EPI_REQUANT:
                qn = torch.zeros((M, n - 2 * H), dtype=torch.int8, device=dev)
                sn = torch.zeros((M, (n - 2 * H) // 32), dtype=torch.float32, device=dev)
                run = lambda: sdv.qmatmul_multipos(qtype, w, n, k, q, s, ws, y=y, epilogue=epi,  # noqa: E731
                                                   requant_col0=2 * H, q_next=qn, scales_next=sn)
            elif epi == sdv.EPI_SILU_MUL_REQUANT:
                qn = torch.zeros((M, n // 2), dtype=torch.int8, device=dev)
                sn = torch.zeros((M, n // 64), dtype=torch.float32, device=dev)
                run = lambda: sdv.qmatmul_multipos(qtype, w, n, k, q, s, ws, epilogue=epi,  # noqa: E731
                                                   q_next=qn, scales_next=sn)
            else:
                run = lambda: sdv.qmatmul_multipos(qtype, w, n, k, q, s, ws, y=y, residual=y)  # noqa: E731
    torch.cuda.synchronize()
    run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.reps):
        run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / a.reps
    st = sdv.device_status()
    gbs = nbytes / (ms * 1e-3) / 1e9 if nbytes else 0.0
    print(f"case={a.case} M={M} reps={a.reps} ms_per_launch={ms:.4f} weight_bytes={nbytes} GB/s={gbs:.1f} status={st}")
    if st != 0:
        sys.exit(1)


if __name__ == "__main__":
    main()
