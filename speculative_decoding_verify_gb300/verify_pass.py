"""The verify pass of a dense quantised projection stack, driven through the C ABI.

Per layer (attention and recurrent mixers omitted): RMSNorm + requant -> QKV
(H -> 3H, the V columns requantised in the matmul epilogue) -> O (+ residual)
-> RMSNorm + requant -> gate|up (H -> 2F, SiLU*mul + requant epilogue) -> down
(+ residual); then a final RMSNorm, the vocabulary head with fused argmax and
softmax statistics, and greedy (chain or tree) acceptance.  One weight read per
matrix serves all M = K+1 positions.  ``capture()`` records the whole pass as
one CUDA graph; launches inside it use programmatic dependent launch so each
kernel streams its weights while the previous one finishes.
"""
from __future__ import annotations

import torch

import ctypes

from . import (ACCEPT_GREEDY, ACCEPT_SAMPLE, EPI_NONE, EPI_REQUANT, EPI_SILU_MUL_REQUANT, Q4_32, Q8_0, SdLayer,
               SdPassDesc, accept_greedy, accept_sample, accept_sample_topk, head_logits, head_workspace_bytes, pass_plan_bytes, pass_prepare, pass_workspace_bytes,
               qmatmul_multipos, qmatmul_workspace_bytes, repack_weights, rmsnorm_quant_acts, verify_pass,
               workspace)


class VerifyStack:
    """Device-resident weights + activation buffers for one M."""

    def __init__(self, layers, norms, final_norm, head_w, hidden: int, ffn: int, vocab: int, M: int,
                 wq: int = Q4_32, head_q: int = Q8_0, eps: float = 1e-6, tree_parent: torch.Tensor | None = None,
                 device="cuda", wq_down: int | None = None):
        """layers: list of dicts {qkv, o, gate_up, down} of REPACKED uint8 CUDA tensors (gate_up repacked with
        the gate|up pairing).  norms: list of (norm1, norm2) fp32 CUDA tensors [hidden].  wq: format of the
        projections (Q4_32 or Q4_K); wq_down: of the down projections (default wq; Q6_K with Q4_K)."""
        assert head_q == Q8_0
        self.layers, self.norms, self.final_norm, self.head_w = layers, norms, final_norm, head_w
        self.H, self.F, self.V, self.M, self.wq, self.eps = hidden, ffn, vocab, M, wq, eps
        self.wq_down = wq if wq_down is None else wq_down
        H, F, V = hidden, ffn, vocab
        f32 = dict(dtype=torch.float32, device=device)
        i8 = dict(dtype=torch.int8, device=device)
        i32 = dict(dtype=torch.int32, device=device)
        self.h = torch.zeros((M, H), **f32)
        self.qa = torch.zeros((M, H), **i8)
        self.sa = torch.zeros((M, H // 32), **f32)
        self.qv = torch.zeros((M, H), **i8)
        self.sv = torch.zeros((M, H // 32), **f32)
        self.qf = torch.zeros((M, F), **i8)
        self.sf = torch.zeros((M, F // 32), **f32)
        self.logits = torch.zeros((M, V), **f32)
        self.argmax = torch.zeros(M, **i32)
        self.row_max = torch.zeros(M, **f32)
        self.row_sumexp = torch.zeros(M, **f32)
        self.tokens = torch.zeros(max(M, 1), **i32)   # drafts (chain) or node tokens (tree)
        self.parent = tree_parent
        self.out_tokens = torch.zeros(M, **i32)
        self.out_count = torch.zeros(1, **i32)
        ws = max(qmatmul_workspace_bytes(wq, 3 * H, H, EPI_REQUANT),
                 qmatmul_workspace_bytes(wq, H, H, EPI_NONE),
                 qmatmul_workspace_bytes(wq, 2 * F, H, EPI_SILU_MUL_REQUANT),
                 qmatmul_workspace_bytes(self.wq_down, H, F, EPI_NONE),
                 head_workspace_bytes(V, H), pass_workspace_bytes(H, F, V, wq))
        self.ws = workspace(ws, device)
        self.graph = None
        self.fused = None

    # -- the pass -------------------------------------------------------------
    def layer(self, l: int):
        H, F, wq = self.H, self.F, self.wq
        w = self.layers[l]
        n1, n2 = self.norms[l]
        rmsnorm_quant_acts(self.h, n1, self.qa, self.sa, self.eps)
        qmatmul_multipos(wq, w["qkv"], 3 * H, H, self.qa, self.sa, self.ws, epilogue=EPI_REQUANT,
                         requant_col0=2 * H, q_next=self.qv, scales_next=self.sv)
        qmatmul_multipos(wq, w["o"], H, H, self.qv, self.sv, self.ws, y=self.h, residual=self.h)
        rmsnorm_quant_acts(self.h, n2, self.qa, self.sa, self.eps)
        qmatmul_multipos(wq, w["gate_up"], 2 * F, H, self.qa, self.sa, self.ws, epilogue=EPI_SILU_MUL_REQUANT,
                         q_next=self.qf, scales_next=self.sf)
        qmatmul_multipos(self.wq_down, w["down"], H, F, self.qf, self.sf, self.ws, y=self.h, residual=self.h)

    def head(self, temperature: float = 1.0):
        rmsnorm_quant_acts(self.h, self.final_norm, self.qa, self.sa, self.eps)
        head_logits(self.head_w, self.V, self.H, self.qa, self.sa, self.ws, self.logits, self.argmax, self.row_max,
                    self.row_sumexp, temperature)

    def accept(self):
        accept_greedy(self.argmax, self.tokens, self.parent, self.M, self.out_tokens, self.out_count)

    def accept_sampled(self, temperature: float, seed: int, base_pos: int = 0, q_probs=None, top_k: int = 0,
                       top_p: float = 1.0):
        """Rejection-sampling acceptance of the drafts self.tokens[:M-1] on this pass's logits and statistics
        (top_k > 0: against the top-k / top-p filtered target)."""
        drafts = self.tokens if self.M > 1 else None
        if top_k > 0:
            accept_sample_topk(self.logits, self.M - 1, drafts, self.out_tokens, self.out_count, top_k, top_p,
                               q_probs=q_probs, temperature=temperature, seed=seed, base_pos=base_pos)
            return
        accept_sample(self.logits, self.M - 1, drafts, self.out_tokens, self.out_count,
                      q_probs=q_probs, row_max=self.row_max, row_sumexp=self.row_sumexp, temperature=temperature,
                      seed=seed, base_pos=base_pos)

    def run(self):
        """One verify pass over self.h (input hidden rows) and self.tokens (drafts); an NVTX range per
        layer, for the head and for the acceptance (each library call inside has its own)."""
        nvtx = torch.cuda.nvtx
        for l in range(len(self.layers)):
            nvtx.range_push(f"layer {l}")
            self.layer(l)
            nvtx.range_pop()
        nvtx.range_push("head")
        self.head()
        nvtx.range_pop()
        nvtx.range_push("accept")
        self.accept()
        nvtx.range_pop()

    # -- the same pass as one persistent cooperative launch -----------------------
    def prepare_fused(self, temperature: float = 1.0, sample: bool = False, seed: int = 0, base_pos: int = 0,
                      q_probs=None, top_k: int = 0, top_p: float = 1.0):
        """Build the phase table of the one-launch pass over this stack's buffers; `sample` ends it with
        rejection-sampling acceptance (temperature, seed, base_pos, q_probs as in accept_sample)
        instead of greedy acceptance."""
        self._q_probs = q_probs
        L = len(self.layers)
        arr = (SdLayer * max(L, 1))()
        for l in range(L):
            w = self.layers[l]
            n1, n2 = self.norms[l]
            arr[l] = SdLayer(w["qkv"].data_ptr(), w["o"].data_ptr(), w["gate_up"].data_ptr(), w["down"].data_ptr(),
                             n1.data_ptr(), n2.data_ptr())
        self._layer_arr = arr
        p = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        d = SdPassDesc(L, self.H, self.F, self.V, self.M, self.wq, self.eps, temperature,
                       ctypes.cast(arr, ctypes.POINTER(SdLayer)), p(self.final_norm), p(self.head_w), p(self.h),
                       p(self.qa), p(self.sa), p(self.qv), p(self.sv), p(self.qf), p(self.sf), p(self.logits),
                       p(self.argmax), p(self.row_max), p(self.row_sumexp), p(self.tokens), p(self.parent),
                       p(self.out_tokens), p(self.out_count), p(self.ws), self.ws.numel(),
                       ACCEPT_SAMPLE if sample else ACCEPT_GREEDY, p(q_probs), seed, base_pos, top_k, top_p,
                       0 if self.wq_down == self.wq else self.wq_down)
        self._plan = torch.zeros(pass_plan_bytes(L), dtype=torch.uint8, device=self.h.device)
        self.fused = pass_prepare(d, self._plan)
        return self.fused

    def run_fused(self):
        """One verify pass (layers, head, acceptance) as a single cooperative launch."""
        if self.fused is None:
            self.prepare_fused()
        verify_pass(self.fused)

    def capture(self):
        """Record run() as one CUDA graph (replayed by replay())."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run()  # warm-up outside capture: sets kernel attributes, loads modules
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        self.graph = g
        return g

    def replay(self):
        self.graph.replay()

    def launches_per_pass(self) -> int:
        return 6 * len(self.layers) + 3


def repack_matrix(qtype: int, blocks_host, n_out: int, k_in: int, pair: bool = False, device="cuda"):
    """Upload GGUF-order blocks (numpy uint8 or pinned torch tensor) and repack them on the device."""
    if not isinstance(blocks_host, torch.Tensor):
        blocks_host = torch.from_numpy(blocks_host)
    src = blocks_host.to(device, non_blocking=True).reshape(-1)
    out = repack_weights(qtype, src, n_out, k_in, pair)
    torch.cuda.current_stream().synchronize()  # weights must be resident before any pass reads them
    del src
    return out
