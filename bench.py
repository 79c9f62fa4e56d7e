"""Benchmark of the speculative-decoding verify pass on GB300.

Workload (default): the 27B-shaped dense projection stack -- 64 layers of
RMSNorm -> 4-bit QKV 5120->15360 -> O 5120->5120 (+residual) -> RMSNorm ->
4-bit gate|up 5120->2x17408 -> SiLU*mul -> requant -> down 17408->5120
(+residual) -- then a final RMSNorm, the 5120x151936 Q8_0 head with fused
argmax/softmax statistics and greedy acceptance of K = 4 drafts (M = K+1 = 5
positions).  Weights N(0, 0.02) block-quantised, hidden rows N(0, 1), synthetic
and seeded.  One step = one verify pass; its 14.23 GB of weights are read from
HBM once per step (far above the 129 MB L2, so no step reuses another's data).

Prints one JSON line: metric = weight-stream GB/s of the pass (value), with
verified positions/s, the HBM fraction, the dominant kernel's roofline, the
clocks seen during the timed region, an end-to-end figure through host buffers
and the CPU oracle's throughput on a bounded sample of the same work.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "weight-stream GB/s (% of HBM peak) per verify pass at K+1=5; verified pos/s"
METRIC_TREE = "weight-stream GB/s (% of HBM peak) per tree verify pass at M=16; verified pos/s"
NOMINAL_HBM_GBS = 8000.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            return out
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(f)
            except Exception:
                pass
        os.unlink(self.path)
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for nm, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        out.update(sm_mhz=sm[len(sm) // 2] if sm else None, sm_max_mhz=max(mx) if mx else None,
                   reasons=sorted(reasons), samples=len(rows))
        return out


# ---------------------------------------------------------------------------
# model construction
# ---------------------------------------------------------------------------
def build_stack(spec, M, device, timings, tree_parent=None):
    import numpy as np
    import torch

    import sdgen
    from speculative_decoding_verify_gb300.verify_pass import VerifyStack, repack_matrix

    t0 = time.time()
    layers, norms = [], []
    for l in range(spec.layers):
        lw = {}
        for name, n, k in spec.matrices():
            blocks = sdgen.pinned_quantized_normal(spec.wq, spec.weight_key(l, name), n, k)
            lw[name] = repack_matrix(spec.wq, blocks, n, k, pair=(name == "gate_up"), device=device)
        layers.append(lw)
        n1, n2 = spec.norms(l)
        norms.append((torch.from_numpy(n1).to(device), torch.from_numpy(n2).to(device)))
        if l % 16 == 15:
            log(f"  layers 0..{l} resident ({time.time() - t0:.0f} s)")
    hb = sdgen.pinned_quantized_normal(spec.head_q, spec.weight_key(0, "head"), spec.vocab, spec.hidden)
    head = repack_matrix(spec.head_q, hb, spec.vocab, spec.hidden, device=device)
    fn = torch.from_numpy(spec.final_norm()).to(device)
    timings["build_s"] = time.time() - t0
    return VerifyStack(layers, norms, fn, head, spec.hidden, spec.ffn, spec.vocab, M, wq=spec.wq,
                       head_q=spec.head_q, device=device, tree_parent=tree_parent)


# The translation units of pass_kernel and the headers they include.
PASS_KERNEL_SOURCES = ("sdv_common.cuh", "sdv_pass.cu", "sdv_pass_sample.cu", "sdv_qmatmul.cuh", "sdv_sample.cuh",
                       "sdv_topk.cuh")


def kernel_source_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "speculative_decoding_verify_gb300", "csrc")
    for f in PASS_KERNEL_SOURCES:
        h.update(open(os.path.join(d, f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(name="pass_kernel_traffic.txt"):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, if it was taken
    on the current kernel source."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line:
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return float(kv["dram_bytes_per_full_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------------------
# per-kernel durations of one eagerly launched pass (CUDA events on the stream)
# ---------------------------------------------------------------------------
def profile_pass(stack):
    import torch

    from speculative_decoding_verify_gb300 import (EPI_NONE, EPI_REQUANT, EPI_SILU_MUL_REQUANT, accept_greedy,
                                                   head_logits, qmatmul_multipos, rmsnorm_quant_acts)
    s = torch.cuda.current_stream()
    ev = []

    def mark(kind, nbytes):
        e = torch.cuda.Event(enable_timing=True)
        e.record(s)
        ev.append((kind, nbytes, e))

    H, F, V, wq = stack.H, stack.F, stack.V, stack.wq
    bb = 18
    first = torch.cuda.Event(enable_timing=True)
    first.record(s)
    for l in range(len(stack.layers)):
        w = stack.layers[l]
        n1, n2 = stack.norms[l]
        rmsnorm_quant_acts(stack.h, n1, stack.qa, stack.sa, stack.eps)
        mark("rmsnorm_quant", 0)
        qmatmul_multipos(wq, w["qkv"], 3 * H, H, stack.qa, stack.sa, stack.ws, epilogue=EPI_REQUANT,
                         requant_col0=2 * H, q_next=stack.qv, scales_next=stack.sv)
        mark("qmm_q4", 3 * H * H // 32 * bb)
        qmatmul_multipos(wq, w["o"], H, H, stack.qv, stack.sv, stack.ws, y=stack.h, residual=stack.h)
        mark("qmm_q4", H * H // 32 * bb)
        rmsnorm_quant_acts(stack.h, n2, stack.qa, stack.sa, stack.eps)
        mark("rmsnorm_quant", 0)
        qmatmul_multipos(wq, w["gate_up"], 2 * F, H, stack.qa, stack.sa, stack.ws, epilogue=EPI_SILU_MUL_REQUANT,
                         q_next=stack.qf, scales_next=stack.sf)
        mark("qmm_q4", 2 * F * H // 32 * bb)
        qmatmul_multipos(wq, w["down"], H, F, stack.qf, stack.sf, stack.ws, y=stack.h, residual=stack.h)
        mark("qmm_q4", H * F // 32 * bb)
    rmsnorm_quant_acts(stack.h, stack.final_norm, stack.qa, stack.sa, stack.eps)
    mark("rmsnorm_quant", 0)
    head_logits(stack.head_w, V, H, stack.qa, stack.sa, stack.ws, stack.logits, stack.argmax, stack.row_max,
                stack.row_sumexp)
    mark("head_q8", V * H // 32 * 34)
    accept_greedy(stack.argmax, stack.tokens, stack.parent, stack.M, stack.out_tokens, stack.out_count)
    mark("accept_greedy", 0)
    torch.cuda.synchronize()
    out = {}
    prev = first
    for kind, nb, e in ev:
        ms = prev.elapsed_time(e)
        d = out.setdefault(kind, {"launches": 0, "ms": 0.0, "bytes": 0})
        d["launches"] += 1
        d["ms"] += ms
        d["bytes"] += nb
        prev = e
    return out


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the same work
# ---------------------------------------------------------------------------
def oracle_sample(spec, M, budget_s=12.0, max_layers=64):
    import numpy as np

    import oracle
    import sdgen

    oracle.build()
    h = spec.hidden_in(M)
    nbytes = 0
    t_total = 0.0
    layers = 0
    for l in range(max_layers):
        wts = {name: spec.weights(l, name) for name, _, _ in spec.matrices()}
        n1, n2 = spec.norms(l)
        t0 = time.time()
        h = oracle.stack_layer(h, wts, n1, n2, spec.hidden, spec.ffn, spec.wq)
        t_total += time.time() - t0
        nbytes += sum(w.nbytes for w in wts.values())
        layers += 1
        if t_total > budget_s:
            break
    cores = oracle.num_threads()
    # the same oracle on one host core, over layer 0 only
    wts = {name: spec.weights(0, name) for name, _, _ in spec.matrices()}
    n1, n2 = spec.norms(0)
    one = sum(w.nbytes for w in wts.values())
    oracle.set_num_threads(1)
    try:
        t0 = time.time()
        oracle.stack_layer(spec.hidden_in(M), wts, n1, n2, spec.hidden, spec.ffn, spec.wq)
        t1 = time.time() - t0
    finally:
        oracle.set_num_threads(cores)
    return {"value": nbytes / t_total / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{layers} layer(s) of the 64-layer stack at M={M} (all four 4-bit matrices, "
                      f"{nbytes / 1e6:.0f} MB of weights, {nbytes / spec.weight_bytes():.1%} of the pass's bytes; "
                      f"the Q8_0 head is not in the sample), {t_total:.1f} s",
            "single_core": {"value": one / t1 / 1e9, "unit": "GB/s", "cores": 1,
                            "sample": f"layer 0 ({one / 1e6:.0f} MB), {t1:.2f} s; x 64 layers: about "
                                      f"{t1 * 64:.0f} s per pass without the head (extrapolated)"}}


def reference_arm(args, spec, M):
    """The oracle timed as the reference implementation on the host cores."""
    import numpy as np

    import oracle
    import sdgen

    oracle.build()
    # one step = the oracle's multi-position matmul over a 3584 x 5120 slice of layer 0's O projection
    # (10.3 MB of 4-bit weights) -- a bounded sample of the pass's weight stream
    n, k = 3584, spec.hidden
    w = sdgen.quantized_normal(spec.wq, spec.weight_key(0, "o"), spec.hidden, k)[:n].copy()
    q, s = oracle.rmsnorm_quant(spec.hidden_in(M), None)
    for _ in range(args.warmup):
        oracle.qmatmul(spec.wq, w, n, k, q, s)
    t0 = time.time()
    for _ in range(args.steps):
        oracle.qmatmul(spec.wq, w, n, k, q, s)
    dt = time.time() - t0
    v = w.nbytes * args.steps / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {"workload": "verify pass weight stream (64-layer 27B-shaped 4-bit stack + Q8_0 head), "
                                   "sampled: 3584x5120 slice of one 4-bit projection per step", "M": M},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{args.steps} steps of a 3584x5120 4-bit projection at M={M}"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
def max_over_ranks(x: float, dist, device) -> float:
    """The largest of every rank's x: the job's time is that of its slowest replica (x itself when the
    job has one rank)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rates(weight_bytes: int, M: int, ms: float, world: int):
    """Whole-job rates of `world` replicas that each stream `weight_bytes` and verify M positions per
    step of `ms` milliseconds (the slowest replica's): (GB/s, positions/s)."""
    return weight_bytes / (ms * 1e-3) / 1e9 * world, M / (ms * 1e-3) * world


def shortlist_bench(args, local):
    """The exact shortlist head against the full Q8_0 head on the 5120 x 151936 head over M positions:
    device time per call (CUDA events, one stream, the 826 MB head and its 438 MB copy far above L2;
    back-to-back calls, so an unpeaked head runs in the shortlist's full mode with a shortlist try
    every 16th call), candidate counts, and whether both give the same argmax.  Three heads: random rows (N(0, 0.02),
    the bound prunes nothing), and the same head with one row per position aligned with that
    position's activations, mildly (a few hundred rows stay candidates) or strongly (a peaked output
    distribution, where the bound prunes every other row).  Prints one JSON line."""
    import numpy as np
    import torch

    import sdgen
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    sdgen.build()
    import speculative_decoding_verify_gb300 as sdv

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    spec = sdgen.StackSpec(layers=0)
    N, K, M = spec.vocab, spec.hidden, args.M
    KB = K // 32
    hb_host = sdgen.pinned_quantized_normal(spec.head_q, spec.weight_key(0, "head"), N, K)
    hb = hb_host.to(dev).reshape(-1)
    x = torch.from_numpy(spec.hidden_in(M)).to(dev)
    q = torch.empty((M, K), dtype=torch.int8, device=dev)
    sc = torch.empty((M, KB), dtype=torch.float32, device=dev)
    sdv.rmsnorm_quant_acts(x, None, q, sc)
    torch.cuda.synchronize()

    def plant(scale):
        """Rows 151935, 77776, ... follow positions 0, 1, ...: their activations / max * scale (the
        random rows have std 0.02; at 0.1 the row's score stands far out, at 0.012 it is a few
        standard deviations above the best random row)."""
        a = (q.cpu().numpy().astype(np.float64).reshape(M, KB, 32) * sc.cpu().numpy()[:, :, None]).reshape(M, K)
        rows = [(151935 + 77777 * m) % N for m in range(M)]
        for m, r in enumerate(rows):
            sl = slice(r * KB * 34, (r + 1) * KB * 34)
            blk = sdgen.quantize(spec.head_q, (a[m] / np.abs(a[m]).max() * scale).astype(np.float32)[None, :])
            hb[sl].copy_(torch.from_numpy(np.ascontiguousarray(blk).reshape(-1)))
        torch.cuda.synchronize()
        return rows

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        if sdv.device_status() != 0:
            raise RuntimeError("device status after the timed calls")
        return e0.elapsed_time(e1) / args.steps

    cases = {}
    for case, scale in (("random", None), ("mild", 0.012), ("peaked", 0.1)):
        planted = plant(scale) if scale else None
        head = sdv.repack_weights(spec.head_q, hb, N, K)
        copy, bound, wnorm = sdv.shortlist_build(hb, N, K)
        cw = sdv.repack_weights(sdv.Q4_32, copy, N, K)
        del copy
        ws_h = sdv.workspace(sdv.head_workspace_bytes(N, K), device=dev)
        ws_s = sdv.workspace(sdv.shortlist_workspace_bytes(N, K), device=dev)
        logits = torch.empty((M, N), dtype=torch.float32, device=dev)
        am_h = torch.empty(M, dtype=torch.int32, device=dev)
        rmax = torch.empty(M, dtype=torch.float32, device=dev)
        rsum = torch.empty(M, dtype=torch.float32, device=dev)
        am_s = torch.empty(M, dtype=torch.int32, device=dev)
        nc = torch.empty(M, dtype=torch.int32, device=dev)
        full_ms = timed(lambda: sdv.head_logits(head, N, K, q, sc, ws_h, logits, am_h, rmax, rsum))
        short_ms = timed(lambda: sdv.head_shortlist(cw, bound, wnorm, head, N, K, q, sc, ws_s, am_s, nc))
        cases[case] = {"full_head_ms": round(full_ms, 4), "shortlist_ms": round(short_ms, 4),
                       "speedup": round(full_ms / short_ms, 3), "candidates_last_call": nc.cpu().tolist(),
                       "argmax_shortlist": am_s.cpu().tolist(), "argmax_full_head_fp32": am_h.cpu().tolist(),
                       "same_argmax": am_s.cpu().tolist() == am_h.cpu().tolist(), "planted_rows": planted}
        del head, cw, ws_h, ws_s, logits
        torch.cuda.empty_cache()
        log(f"shortlist {case}: full head {full_ms:.4f} ms, shortlist {short_ms:.4f} ms, "
            f"candidates {cases[case]['candidates_last_call']}")
    head_bytes = N * KB * 34
    copy_bytes = N * KB * 18
    print(json.dumps({
        "metric": "exact greedy head: ms per call, shortlist vs full Q8_0 head", "unit": "ms",
        "value": cases["peaked"]["shortlist_ms"], "higher_is_better": False, "steps": args.steps,
        "warmup": args.warmup, "n_gpus": 1, "dtype": "int8 dot / fp32 copy scores / fp64 exact scores",
        "data": "synthetic", "config": {"workload": f"Q8_0 head {N}x{K}, M={M}",
                                        "l2": "inputs larger than L2 (head 826 MB, copy 438 MB)"},
        "algorithmic_bytes": {"full_head": head_bytes, "shortlist_copy": copy_bytes + 8 * N,
                              "per_exact_row": KB * 34},
        "cases": cases}))


def attention_bench(args, local):
    """Decode attention of one 27B-shaped layer (40 heads of 128, one KV head per query head) over
    the K+1 positions at contexts of 4096 and 32768 rows: device time per call (CUDA events around
    the call's two launches, enqueued while the device still runs a short sleep so that host-side
    marshalling is not counted; L2 flushed by a write and cleaned by a read of two buffers larger
    than L2 before each call), the fp16 K and V rows read once per call as the algorithmic bytes,
    against the measured copy peak.  Prints one JSON line."""
    import numpy as np
    import torch

    import sdgen
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    sdgen.build()
    import speculative_decoding_verify_gb300 as sdv

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    H_kv = H = 40
    D, M = 128, args.M
    peak, peak_kind = measured_peaks()
    cases = {}
    for L in (4096, 32768):
        S_max = L + M
        kc = torch.from_numpy(sdgen.normal(sdgen.key(6, L), (H_kv, S_max, D)).astype(np.float16)).to(dev)
        vc = torch.from_numpy(sdgen.normal(sdgen.key(6, L + 1), (H_kv, S_max, D)).astype(np.float16)).to(dev)
        q = torch.from_numpy(sdgen.normal(sdgen.key(6, L + 2), (M, H, D))).to(dev)
        out = torch.empty((M, H, D), dtype=torch.float32, device=dev)
        ws = sdv.workspace(sdv.attn_workspace_bytes(M, H, H_kv, D, L), device=dev)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # larger than L2
        evict = torch.ones(256 << 20, dtype=torch.uint8, device=dev)
        for _ in range(args.warmup):
            sdv.attn_decode(q, kc, vc, L, out, ws)
        torch.cuda.synchronize()
        times = []
        for _ in range(args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush.fill_(1)
            # reading a second buffer larger than L2 writes the flush's dirty lines back before the
            # timed region, so the call neither finds its inputs in L2 nor pays for that write-back
            evict.sum()
            # the device idles about 0.1 ms while the host enqueues the call: the events see the call's
            # device time, not the binding's host overhead
            torch.cuda._sleep(200000)
            e0.record()
            sdv.attn_decode(q, kc, vc, L, out, ws)
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        if sdv.device_status() != 0:
            raise RuntimeError("device status after the timed calls")
        ms = float(np.median(times))
        nbytes = 2 * H_kv * (L + M) * D * 2
        gbs = nbytes / ms / 1e6
        cases[str(L)] = {"ms": round(ms, 4), "kv_bytes": nbytes, "GB/s": round(gbs, 1),
                         "frac_of_peak": round(gbs / peak, 3)}
        log(f"attention L={L}: {ms:.4f} ms, {gbs:.0f} GB/s ({gbs / peak:.1%} of the {peak_kind} copy peak)")
        del kc, vc, flush, evict
        torch.cuda.empty_cache()
    print(json.dumps({
        "metric": "decode attention over K+1 positions: KV GB/s per call", "unit": "GB/s",
        "value": cases["32768"]["GB/s"], "higher_is_better": True, "steps": args.steps, "warmup": args.warmup,
        "n_gpus": 1, "dtype": "fp16 K/V, fp32 arithmetic", "data": "synthetic",
        "config": {"workload": f"attention 40x128 heads, M={M}, contexts 4096 and 32768",
                   "l2": "between timed calls a 256 MB buffer written, then another 256 MB read: L2 holds "
                         "neither inputs nor dirty lines when a call starts"},
        "peak_gbs": peak, "peak_kind": peak_kind, "cases": cases}))


def write_trace(path, stack, h_dev, sdv):
    """One traced pass (the same launch as the timed one, with per-phase stamps) -> .npz with the SM id
    of each CTA, the stamps [phase][cta][6] relative to the earliest stamp, and each phase's kind."""
    import numpy as np
    import torch

    p = stack.fused
    n = sdv.pass_trace_bytes(p) // 8
    tr = torch.zeros(n, dtype=torch.int64, device=h_dev.device)
    stack.h.copy_(h_dev)
    sdv.verify_pass_traced(p, tr)
    torch.cuda.synchronize()
    t = tr.cpu().numpy()
    G, P = p.grid, p.n_phases
    smid = t[:G].copy()
    raw = t[G:G + P * G * 12].reshape(P, G, 12)
    st = raw[:, :, :6].astype(np.float64)
    t0 = st[st > 0].min()
    st = np.where(st > 0, st - t0, np.nan)
    np.savez(path, smid=smid, stamps=st, cycles=raw[:, :, 6:].astype(np.float64))
    log(f"trace: {P} phases x {G} CTAs written to {path}")


def kquant_bench(args, local):
    """The one-launch verify pass over the 64-layer 27B-shaped stack in the Q4_K_M recipe: Q4_K QKV, O
    and gate|up, Q6_K down projections, the Q8_0 5120 x 151936 head, greedy acceptance at M positions.
    Weights are seeded random super-blocks (every byte pattern is a valid block; the fp16 scales are
    set so the weights stay near the other stacks' 0.02).  Algorithmic bytes are the file's: 144 B
    (Q4_K) and 210 B (Q6_K) per 256 weights.  Prints one JSON line like the default pass."""
    import numpy as np
    import torch

    import oracle
    import sdgen
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    sdgen.build()
    import speculative_decoding_verify_gb300 as sdv
    from speculative_decoding_verify_gb300.verify_pass import VerifyStack, repack_matrix

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    M, Lyr = args.M, args.layers
    spec = sdgen.StackSpec(layers=Lyr)
    H, F, V = spec.hidden, spec.ffn, spec.vocab
    fmt = {"qkv": sdv.Q4_K, "o": sdv.Q4_K, "gate_up": sdv.Q4_K, "down": sdv.Q6_K}
    d_scale = 2e-5

    def kq_blocks(l, name, n, k):
        return sdgen.random_kq_blocks(fmt[name], sdgen.key(7, l, n, k), n, k, d_scale=d_scale)

    t0 = time.time()
    layers, norms = [], []
    for l in range(Lyr):
        lw = {}
        for name, n, k in spec.matrices():
            lw[name] = repack_matrix(fmt[name], kq_blocks(l, name, n, k), n, k, pair=(name == "gate_up"), device=dev)
        layers.append(lw)
        n1, n2 = spec.norms(l)
        norms.append((torch.from_numpy(n1).to(dev), torch.from_numpy(n2).to(dev)))
        if l % 16 == 15:
            log(f"  K-quant layers 0..{l} resident ({time.time() - t0:.0f} s)")
    hb = sdgen.pinned_quantized_normal(spec.head_q, spec.weight_key(0, "head"), V, H)
    head = repack_matrix(spec.head_q, hb, V, H, device=dev)
    build_s = time.time() - t0
    stack = VerifyStack(layers, norms, torch.from_numpy(spec.final_norm()).to(dev), head, H, F, V, M, wq=sdv.Q4_K,
                        wq_down=sdv.Q6_K, device=dev)
    per_layer = sum(n * (k // 256) * sdv.SUPER_BLOCK_BYTES[fmt[name]] for name, n, k in spec.matrices())
    wbytes = Lyr * per_layer + V * (H // 32) * 34
    h0 = torch.from_numpy(spec.hidden_in(M)).to(dev)
    stack.h.copy_(h0)
    stack.run_fused()
    torch.cuda.synchronize()
    am = stack.argmax.cpu().numpy()
    drafts = sdgen.drafts_p(sdgen.key(4, 8), am[:M - 1], V)
    stack.tokens[:M - 1].copy_(torch.from_numpy(drafts))
    if sdv.device_status() != 0:
        raise RuntimeError("device status after the first pass")
    h_dev = h0.clone()

    def body():
        stack.h.copy_(h_dev)
        stack.run_fused()

    g_stream = torch.cuda.Stream()
    g_stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(g_stream):
        body()
    torch.cuda.current_stream().wait_stream(g_stream)
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        body()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        gr.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        gr.replay()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    if sdv.device_status() != 0:
        raise RuntimeError("device status after the timed region")
    # end to end through host buffers
    h_host = torch.from_numpy(spec.hidden_in(M)).pin_memory()
    d_host = torch.from_numpy(np.ascontiguousarray(drafts)).pin_memory()
    out_host = torch.zeros(M, dtype=torch.int32).pin_memory()
    cnt_host = torch.zeros(1, dtype=torch.int32).pin_memory()
    n_e2e = max(10, args.steps // 4)
    t1 = time.perf_counter()
    for _ in range(n_e2e):
        h_dev.copy_(h_host, non_blocking=True)
        stack.tokens[:M - 1].copy_(d_host, non_blocking=True)
        gr.replay()
        out_host.copy_(stack.out_tokens, non_blocking=True)
        cnt_host.copy_(stack.out_count, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    e2e_ms = (time.perf_counter() - t1) / n_e2e * 1e3
    peak, peak_kind = measured_peaks()
    gbs = wbytes / (ms * 1e-3) / 1e9
    if args.trace:
        write_trace(args.trace, stack, h_dev, sdv)
    del stack, gr, layers
    torch.cuda.empty_cache()
    # CPU baseline: the oracle's K-quant matmuls over a bounded sample of the stack's layers
    oracle.build()
    q, sc = oracle.rmsnorm_quant(spec.hidden_in(M), None)
    qf, sf = oracle.rmsnorm_quant(sdgen.normal(sdgen.key(7, 999), (M, F)), None)
    nb, tt, nl = 0, 0.0, 0
    for l in range(Lyr):
        for name, n, k in spec.matrices():
            blk = kq_blocks(l, name, n, k)
            t2 = time.time()
            oracle.kq_matmul(fmt[name], blk, n, k, qf if k == F else q, sf if k == F else sc)
            tt += time.time() - t2
            nb += blk.nbytes
        nl += 1
        if tt > 10.0:
            break
    line = {"metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8 activations, 4/6-bit K-quant codes", "data": "synthetic (seeded random K-quant super-blocks)",
            "config": {"workload": f"verify pass: {Lyr}-layer 27B-shaped Q4_K_M-style stack (Q4_K QKV/O/gate|up, "
                                   f"Q6_K down) + 5120x151936 Q8_0 head + greedy accept, K+1={M}",
                       "M": M, "layers": Lyr, "weight_bytes_per_pass": wbytes,
                       "l2": "inputs larger than L2: weights streamed per step far above the 129 MB L2",
                       "mode": "fused (one persistent launch per pass)"},
            "pos_per_s": M / (ms * 1e-3), "hbm_frac_of_measured": gbs / peak,
            "roofline": {"bound": "hbm", "kernel": "pass_kernel<K-quant> (one launch per pass)", "achieved": gbs,
                         "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                         "algorithmic_bytes_per_launch": wbytes, "avg_launch_ms": ms,
                         "note": "the repacked Q4_K records hold their 6-bit scales as bytes: 2.8 % above the file"},
            "clocks": clk,
            "e2e": {"value": wbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h_host.numel() * 4 + d_host.numel() * 4,
                    "d2h_bytes_per_step": out_host.numel() * 4 + cnt_host.numel() * 4},
            "gpu_launches": args.steps, "build_s": build_s,
            "cpu_baseline": {"value": nb / tt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{nl} layer(s) of the K-quant stack at M={M} (QKV, O, gate|up, down: "
                                       f"{nb / 1e6:.0f} MB, {nb / wbytes:.1%} of the pass's bytes; head not "
                                       f"sampled), {tt:.1f} s"}}
    print(json.dumps(line), flush=True)


CASES = ("qkv", "o", "gate_up", "down", "head", "rmsnorm", "pass")


def case_bench(args, local):
    """One kernel on one seeded layer-sized case, for profiling: qkv (4-bit 5120->15360, V requant
    epilogue), o (4-bit 5120->5120 + residual), gate_up (4-bit 5120->2x17408, SiLU*mul requant),
    down (4-bit 17408->5120 + residual), head (Q8_0 5120->151936 with argmax and statistics),
    rmsnorm (M x 5120), or pass (the one-launch pass over --layers layers plus the head).  Runs
    --steps launches after one untimed launch and prints one line: mean event-timed duration per
    launch and weight-stream GB/s."""
    import numpy as np
    import torch

    import sdgen
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    sdgen.build()
    import speculative_decoding_verify_gb300 as sdv

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    H, F, V = sdgen.HIDDEN, sdgen.FFN, sdgen.VOCAB
    M = args.M
    mats = {"qkv": (sdv.Q4_32, 3 * H, H, sdv.EPI_REQUANT), "o": (sdv.Q4_32, H, H, sdv.EPI_NONE),
            "gate_up": (sdv.Q4_32, 2 * F, H, sdv.EPI_SILU_MUL_REQUANT), "down": (sdv.Q4_32, H, F, sdv.EPI_NONE),
            "head": (sdv.Q8_0, V, H, None)}
    if args.case == "pass":
        spec = sdgen.StackSpec(layers=args.layers)
        stack = build_stack(spec, M, dev, {})
        h0 = torch.from_numpy(spec.hidden_in(M)).to(dev)
        stack.prepare_fused()

        def run():
            stack.h.copy_(h0)
            stack.run_fused()
        nbytes = spec.weight_bytes()
    elif args.case == "rmsnorm":
        x = torch.from_numpy(sdgen.normal(sdgen.key(9, 0), (M, H))).to(dev)
        w = torch.from_numpy(sdgen.norm_weight(sdgen.key(9, 1), H)).to(dev)
        q = torch.zeros((M, H), dtype=torch.int8, device=dev)
        sc = torch.zeros((M, H // 32), dtype=torch.float32, device=dev)
        run = lambda: sdv.rmsnorm_quant_acts(x, w, q, sc)  # noqa: E731
        nbytes = 0
    else:
        qtype, n, k, epi = mats[args.case]
        blocks = sdgen.pinned_quantized_normal(qtype, sdgen.key(9, 2, n, k), n, k)
        w = sdv.repack_weights(qtype, blocks.to(dev).reshape(-1), n, k, pair=(epi == sdv.EPI_SILU_MUL_REQUANT))
        xq = torch.from_numpy(sdgen.normal(sdgen.key(9, 3), (M, k))).to(dev)
        q = torch.zeros((M, k), dtype=torch.int8, device=dev)
        sc = torch.zeros((M, k // 32), dtype=torch.float32, device=dev)
        sdv.rmsnorm_quant_acts(xq, None, q, sc)
        nbytes = n * (k // 32) * sdv.BLOCK_BYTES[qtype]
        y = torch.zeros((M, n), dtype=torch.float32, device=dev)
        if args.case == "head":
            ws = sdv.workspace(sdv.head_workspace_bytes(n, k), dev)
            am = torch.zeros(M, dtype=torch.int32, device=dev)
            rm = torch.zeros(M, dtype=torch.float32, device=dev)
            rz = torch.zeros(M, dtype=torch.float32, device=dev)
            run = lambda: sdv.head_logits(w, n, k, q, sc, ws, y, am, rm, rz)  # noqa: E731
        else:
            ws = sdv.workspace(sdv.qmatmul_workspace_bytes(qtype, n, k, epi), dev)
            if epi == sdv.EPI_REQUANT:
                qn = torch.zeros((M, n - 2 * H), dtype=torch.int8, device=dev)
                sn = torch.zeros((M, (n - 2 * H) // 32), dtype=torch.float32, device=dev)
                run = lambda: sdv.qmatmul_multipos(qtype, w, n, k, q, sc, ws, y=y, epilogue=epi,  # noqa: E731
                                                   requant_col0=2 * H, q_next=qn, scales_next=sn)
            elif epi == sdv.EPI_SILU_MUL_REQUANT:
                qn = torch.zeros((M, n // 2), dtype=torch.int8, device=dev)
                sn = torch.zeros((M, n // 64), dtype=torch.float32, device=dev)
                run = lambda: sdv.qmatmul_multipos(qtype, w, n, k, q, sc, ws, epilogue=epi,  # noqa: E731
                                                   q_next=qn, scales_next=sn)
            else:
                run = lambda: sdv.qmatmul_multipos(qtype, w, n, k, q, sc, ws, y=y, residual=y)  # noqa: E731
    torch.cuda.synchronize()
    run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    st = sdv.device_status()
    gbs = nbytes / (ms * 1e-3) / 1e9 if nbytes else 0.0
    print(f"case={args.case} M={M} launches={args.steps} ms_per_launch={ms:.4f} weight_bytes={nbytes} "
          f"GB/s={gbs:.1f} status={st}", flush=True)
    if st != 0:
        raise SystemExit(1)


SKINNY_SHAPES = (("QKV/O-like 5120x5120", 5120, 5120), ("FFN up/gate 5120->17408", 17408, 5120),
                 ("FFN down 17408->5120", 5120, 17408))


def skinny_bench(args, local):
    """Layer-sized skinny matmuls: each shape x M in {1, 2, 3, 5, 8} x {Q8_0, 4-bit}, one
    sd_qmatmul_multipos call per step over activations formed by the fused RMSNorm + int8 requant
    (weight 1 + N(0, 0.1), eps 1e-6) of N(0, 1) rows.  The weights rotate over copies totalling at
    least 1 GB, so no call finds its matrix in L2.  Device time of back-to-back calls (CUDA events
    around the loop).  Prints one JSON line: the aggregate weight-stream GB/s over all cases, and
    each case."""
    import numpy as np
    import torch

    import sdgen
    from speculative_decoding_verify_gb300 import build as b
    b.build()
    sdgen.build()
    import speculative_decoding_verify_gb300 as sdv
    from speculative_decoding_verify_gb300.verify_pass import repack_matrix

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    peak, peak_kind = measured_peaks()
    rotate_bytes = 1 << 30
    cases = []
    tot_bytes, tot_ms = 0, 0.0
    for qt, qname in ((sdv.Q8_0, "Q8_0"), (sdv.Q4_32, "4-bit")):
        for sname, n, k in SKINNY_SHAPES:
            blocks = sdgen.pinned_quantized_normal(qt, sdgen.key(21, qt, n, k), n, k)
            w0 = repack_matrix(qt, blocks, n, k, device=dev)
            nbytes = n * (k // 32) * sdv.BLOCK_BYTES[qt]
            copies = [w0] + [w0.clone() for _ in range(max(1, -(-rotate_bytes // w0.numel())) - 1)]
            ws = sdv.workspace(sdv.qmatmul_workspace_bytes(qt, n, k), device=dev)
            nw = torch.from_numpy(sdgen.norm_weight(sdgen.key(22, k), k)).to(dev)
            for M in (1, 2, 3, 5, 8):
                x = torch.from_numpy(sdgen.normal(sdgen.key(23, k, M), (M, k))).to(dev)
                q = torch.empty((M, k), dtype=torch.int8, device=dev)
                sc = torch.empty((M, k // 32), dtype=torch.float32, device=dev)
                sdv.rmsnorm_quant_acts(x, nw, q, sc, eps=1e-6)
                y = torch.empty((M, n), dtype=torch.float32, device=dev)
                for i in range(args.warmup):
                    sdv.qmatmul_multipos(qt, copies[i % len(copies)], n, k, q, sc, ws, y=y)
                torch.cuda.synchronize()
                reps = max(args.steps, 2 * len(copies))
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for i in range(reps):
                    sdv.qmatmul_multipos(qt, copies[i % len(copies)], n, k, q, sc, ws, y=y)
                e1.record()
                torch.cuda.synchronize()
                if sdv.device_status() != 0:
                    raise RuntimeError(f"device status after {qname} {sname} M={M}")
                ms = e0.elapsed_time(e1) / reps
                gbs = nbytes / (ms * 1e-3) / 1e9
                cases.append({"format": qname, "shape": sname, "n_out": n, "k_in": k, "M": M,
                              "weight_bytes": nbytes, "us_per_call": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                              "frac_of_peak": round(gbs / peak, 3), "copies": len(copies)})
                tot_bytes += nbytes
                tot_ms += ms
                log(f"{qname} {sname} M={M}: {ms * 1e3:.1f} us, {gbs:.0f} GB/s ({gbs / peak:.1%})")
            del copies, w0, ws
            torch.cuda.empty_cache()
    agg = tot_bytes / (tot_ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": "weight-stream GB/s of layer-sized skinny matmuls (aggregate over shapes x M x formats)",
        "value": agg, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8 activations, Q8_0 / 4-bit codes",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) rows through RMSNorm + requant)",
        "config": {"workload": "layer-sized skinny matmuls: 5120x5120, 5120->17408, 17408->5120 in Q8_0 and 4-bit, "
                               "M in {1,2,3,5,8}, one sd_qmatmul_multipos call per step",
                   "l2": "weights rotated over copies of at least 1 GB per shape (larger than L2)"},
        "roofline": {"bound": "hbm", "kernel": "qmm_kernel (multi-position matmul, one launch per call)",
                     "achieved": agg, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": agg / peak,
                     "traffic": None, "algorithmic_bytes_per_launch": "each case's weight_bytes",
                     "avg_launch_ms": tot_ms / len(cases)},
        "gpu_launches": sum(max(args.steps, 2 * c["copies"]) for c in cases),
        "cases": cases}), flush=True)


def run_probe(name, extra):
    """Build probes/<name> for sm_103a into _build/probes and run it; its table goes to stdout."""
    import subprocess

    from speculative_decoding_verify_gb300 import build as b
    src = os.path.join(ROOT, "probes", {"consumer": "consumer_loop_probe.cu", "tcgen05": "tcgen05_probe.cu"}[name])
    out_dir = os.path.join(ROOT, "_build", "probes")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, name)
    cmd = [b.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-I",
           os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "speculative_decoding_verify_gb300", "csrc"), src,
           "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise SystemExit(f"probe build failed:\n{r.stderr[-3000:]}")
    r = subprocess.run([exe] + list(extra))
    if r.returncode != 0:
        raise SystemExit(r.returncode)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=64)
    ap.add_argument("--M", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--fused-only", action="store_true",
                    help="time only the one-launch pass (no per-operation graph, no eager per-kernel breakdown)")
    ap.add_argument("--mode", default="fused", choices=["fused", "graph"],
                    help="fused: the whole pass as one persistent launch; graph: one CUDA graph of per-op launches")
    ap.add_argument("--attention", action="store_true",
                    help="instead of the pass: time the decode attention over the K+1 positions (own JSON line)")
    ap.add_argument("--shortlist", action="store_true",
                    help="instead of the pass: time the exact shortlist head against the full head (own JSON line)")
    ap.add_argument("--kquant", action="store_true",
                    help="instead of the default stack: the Q4_K_M-style K-quant stack (own JSON line)")
    ap.add_argument("--trace", default=None, metavar="FILE",
                    help="after the timed region, run one traced pass and write its per-phase, per-CTA "
                         "global-timer stamps (numpy .npz) to FILE")
    ap.add_argument("--config", type=int, default=4, choices=(2, 4, 5),
                    help="2: layer-sized skinny matmuls (own JSON line); 4: the 64-layer verify pass at K+1=5 "
                         "(default); 5: the same stack verifying a 16-node draft tree (M=16)")
    ap.add_argument("--probe", default=None, choices=("consumer", "tcgen05"),
                    help="instead of the pass: build and run a design microbenchmark from probes/ (prints its table)")
    ap.add_argument("--probe-args", default="400", help="arguments of the probe program (consumer: iterations [filter])")
    ap.add_argument("--case", default=None, choices=CASES,
                    help="instead of the pass: run one kernel on one layer-sized case --steps times, for profiling")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    import sdgen
    spec = sdgen.StackSpec(layers=args.layers)
    M = args.M

    if args.impl == "reference":
        if rank == 0:
            reference_arm(args, spec, M)
        return
    if args.probe:
        run_probe(args.probe, args.probe_args.split())
        return
    if args.case:
        case_bench(args, local)
        return
    if args.kquant:
        kquant_bench(args, local)
        return
    if args.shortlist:
        shortlist_bench(args, local)
        return
    if args.attention:
        attention_bench(args, local)
        return
    if args.config == 2:
        skinny_bench(args, local)
        return
    tree = args.config == 5
    if tree:
        M = args.M = 16

    import numpy as np
    import torch

    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(device))

    from speculative_decoding_verify_gb300 import build as b
    if rank == 0 or world == 1:
        b.build()
    if dist:
        dist.barrier()
    sdgen.build()
    import speculative_decoding_verify_gb300 as sdv
    sdv.lib()
    if args.no_pdl:
        sdv.set_pdl(False)

    timings = {}
    log(f"[rank {rank}] building the {spec.layers}-layer stack ({spec.weight_bytes() / 1e9:.2f} GB of weights)")
    parent_np = sdgen.tree16(0)[0] if tree else None
    stack = build_stack(spec, M, device, timings,
                        tree_parent=torch.from_numpy(parent_np).to(device) if tree else None)
    h0 = torch.from_numpy(spec.hidden_in(M)).to(device)

    # drafts: the target's argmax with probability 0.75 per position, else uniform (from an untimed pass);
    # a tree: uniform tokens except along the path 0-1-3-7-15, which follows the argmax chain
    stack.h.copy_(h0)
    if args.fused_only:
        stack.run_fused()
    else:
        stack.run()
    torch.cuda.synchronize()
    am = stack.argmax.cpu().numpy()
    if tree:
        drafts = sdgen.uniform_tokens(sdgen.key(4, 8), M, spec.vocab).astype(np.int32)
        for child in (1, 3, 7, 15):
            drafts[child] = am[parent_np[child]]
    else:
        drafts = sdgen.drafts_p(sdgen.key(4, 7), am[:M - 1], spec.vocab)
    stack.tokens[:len(drafts)].copy_(torch.from_numpy(drafts))
    if sdv.device_status() != 0:
        raise RuntimeError("device status after the first pass")

    # the timed step: copy the input rows into the residual stream, then the pass -- as one persistent
    # launch (fused) or as one CUDA graph of per-operation launches (graph); both are timed, the
    # selected mode is the headline
    h_dev = torch.empty_like(h0)
    h_dev.copy_(h0)
    stack.prepare_fused()

    def body_graph():
        stack.h.copy_(h_dev)
        stack.run()

    def body_fused():
        stack.h.copy_(h_dev)
        stack.run_fused()

    def capture(body):
        g_stream = torch.cuda.Stream()
        g_stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(g_stream):
            body()
        torch.cuda.current_stream().wait_stream(g_stream)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            body()
        torch.cuda.synchronize()
        return gr

    if args.fused_only:
        args.mode = "fused"
        graphs = {"fused": capture(body_fused)}
    else:
        graphs = {"graph": capture(body_graph), "fused": capture(body_fused)}

    def time_mode(gr, steps, sample_clocks=False):
        for _ in range(args.warmup):
            gr.replay()
        torch.cuda.synchronize()
        clocks = ClockSampler(local) if sample_clocks else None
        if clocks:
            clocks.start()
            time.sleep(0.3)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            gr.replay()
        e1.record()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        return e0.elapsed_time(e1) / steps, (clocks.stop() if clocks else None)

    other = "graph" if args.mode == "fused" else "fused"
    ms_other = time_mode(graphs[other], max(10, args.steps // 4))[0] if other in graphs else None
    ms, clk = time_mode(graphs[args.mode], args.steps, sample_clocks=True)
    graph = graphs[args.mode]
    kept = int(stack.out_count.cpu()[0])
    if sdv.device_status() != 0:
        raise RuntimeError("device status after the timed region")
    ms = max_over_ranks(ms, dist, device)

    wbytes = spec.weight_bytes()
    gbs, pos_s = job_rates(wbytes, M, ms, world)

    # end to end through the ABI with host buffers: H2D of the input rows and drafts, the pass, D2H of the
    # accepted tokens and their count, every step
    h_host = torch.from_numpy(spec.hidden_in(M)).pin_memory()
    d_host = torch.from_numpy(np.ascontiguousarray(drafts)).pin_memory()
    out_host = torch.zeros(M, dtype=torch.int32).pin_memory()
    cnt_host = torch.zeros(1, dtype=torch.int32).pin_memory()
    e2e_steps = max(10, args.steps // 4)

    def e2e_step():
        h_dev.copy_(h_host, non_blocking=True)
        stack.tokens[:d_host.numel()].copy_(d_host, non_blocking=True)
        graph.replay()
        out_host.copy_(stack.out_tokens, non_blocking=True)
        cnt_host.copy_(stack.out_count, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
        torch.cuda.current_stream().synchronize()
    e2e_ms = (time.perf_counter() - t0) / e2e_steps * 1e3
    e2e_ms = max_over_ranks(e2e_ms, dist, device)
    h2d = h_host.numel() * 4 + d_host.numel() * 4
    d2h = out_host.numel() * 4 + cnt_host.numel() * 4

    if args.trace and rank == 0:
        write_trace(args.trace, stack, h_dev, sdv)

    # per-kernel durations of the per-operation pipeline (one eagerly launched pass, events between launches)
    prof = None
    if not args.fused_only:
        stack.h.copy_(h_dev)
        prof = profile_pass(stack)
        prof_total = sum(v["ms"] for v in prof.values())
    peak, peak_kind = measured_peaks()
    if args.mode == "fused":
        # one persistent launch per pass: the pass kernel is the step's only kernel of this library (the step
        # also copies the 100 KB of input rows), so its launch duration is the timed region's per-step time
        kms = ms
        achieved = wbytes / (kms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "pass_kernel (one persistent launch per verify pass)",
                "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                "traffic": committed_traffic(), "algorithmic_bytes_per_launch": wbytes, "avg_launch_ms": kms,
                "launches_per_pass": 1}
    else:
        q4 = prof["qmm_q4"]
        achieved = q4["bytes"] / (q4["ms"] * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": "qmm_kernel<Q4_32> (4-bit multi-position matmul)",
                "achieved": achieved, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                "traffic": None,
                "algorithmic_bytes_per_launch": q4["bytes"] / q4["launches"],
                "avg_launch_ms": q4["ms"] / q4["launches"], "launches_per_pass": q4["launches"],
                "share_of_eager_pass": q4["ms"] / prof_total}
    if prof:
        roof["per_op_pipeline_eager"] = {k: {"launches": v["launches"], "ms": round(v["ms"], 4),
                                             "share": round(v["ms"] / prof_total, 4)} for k, v in prof.items()}

    line = {"metric": METRIC_TREE if tree else METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) hidden rows)",
            "config": {"workload": ("tree verify pass: 16-node draft tree (root, binary depth 3, one spine node) "
                                    "as M=16 rows through the 64-layer 27B-shaped 4-bit stack + 5120x151936 Q8_0 "
                                    "head + greedy tree accept") if tree else
                                   ("verify pass: 64-layer 27B-shaped 4-bit projection stack + 5120x151936 "
                                    "Q8_0 head + greedy accept, K+1=5"),
                       "M": M, "layers": spec.layers, "hidden": spec.hidden, "ffn": spec.ffn, "vocab": spec.vocab,
                       "weight_bytes_per_pass": wbytes, "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                       "l2": "inputs larger than L2: 14.2 GB of weights streamed per step vs 129 MB L2",
                       "pdl": not args.no_pdl, "mode": args.mode,
                       "modes": {"fused": "one persistent cooperative launch per pass",
                                 "graph": "one CUDA graph of 387 per-operation launches per pass"}},
            "pos_per_s": pos_s, "hbm_frac_of_measured": gbs / world / peak,
            "hbm_frac_of_nominal_8TBps": gbs / world / NOMINAL_HBM_GBS,
            "accepted_tokens_last_pass": kept,
            "roofline": roof, "clocks": clk,
            "e2e": {"value": wbytes / (e2e_ms * 1e-3) / 1e9 * world, "unit": "GB/s", "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": (1 if args.mode == "fused" else stack.launches_per_pass()) * args.steps,
            f"{other}_ms_per_step": ms_other, f"{other}_GBps": wbytes / (ms_other * 1e-3) / 1e9 if ms_other else None,
            "build_s": timings.get("build_s")}

    del stack, graph, graphs
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = oracle_sample(spec, M)
        except Exception as ex:  # the baseline is reported, never required
            line["cpu_baseline"] = {"value": None, "error": str(ex)[:200]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
