"""A Llama-style dense decoder whose every step runs through libbi.

The model is the serving scenario of "Reproducible LLM Inference - Batch
Invariance, the Cost of Determinism, and Where Bitwise Identity Is Actually
Required" (§5-§6): a pre-norm transformer decoder over a paged KV cache,
stepped by a continuous-batching scheduler, whose tokens must not depend on
which other requests share a step.  Each layer is

    y   = RMSNorm(h) * w_attn                       bi_rmsnorm / bi_add_rmsnorm
    qkv = y W_qkv^T                                  bi_gemm
    q, k, v = RoPE(qkv split), at each token's position   bi_rope_qkv
    K/V cache <- k, v                                bi_kv_write
    a   = attention(q, cache)                        bi_attn_decode / bi_attn_prefill_chunk
    h  += a W_o^T;  y = RMSNorm(h) * w_mlp            bi_gemm, bi_add_rmsnorm
    h  += (silu(y W_gate^T) * y W_up^T) W_down^T      bi_gemm_swiglu, bi_gemm

followed by a final RMSNorm, the LM-head GEMM on the rows that need a token
and bi_sample (greedy at temperature 0, seeded Gumbel-max above).  Weights are
random (no trained checkpoint is needed for invariance); the shapes default to
Llama-3-8B's.  PyTorch only owns memory; every arithmetic step is a libbi call.

A step's tokens are ordered decode rows first (one token per sequence, run by
the decode kernel) and prefill chunks after them (the chunked-prefill kernel),
so both attention kernels write contiguous slices of one output.  The two
kernels give bit-identical results for the same position, so which one serves
a token never changes its bytes.

Decode-only steps can be replayed from CUDA graphs (``use_graphs``): a step
is a few hundred short launches, so at small batch the host, not the GPU, sets
its pace ("Reproducible LLM Inference - Batch Invariance, the Cost of
Determinism, and Where Bitwise Identity Is Actually Required", §8.5: graphs
recover much of what deterministic mode costs).  Every call takes its shapes
from host arguments that are fixed per (batch size, KV-length bucket) and
reads lengths, positions and page tables on the device, so a captured step
replays the same kernels on the step's uploaded arrays.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import _binding as bi
from . import synth


@dataclass(frozen=True)
class DecoderConfig:
    layers: int = 32
    hidden: int = 4096
    heads: int = 32
    kv_heads: int = 8
    head_dim: int = 128
    ffn: int = 14336
    vocab: int = 128256
    rope_theta: float = 500000.0
    eps: float = 1e-5
    page_size: int = 16
    split_size: int = 256
    init_std: float = 0.02

    @property
    def qkv_dim(self) -> int:
        return (self.heads + 2 * self.kv_heads) * self.head_dim


LLAMA3_8B = DecoderConfig()
"""Llama-3-8B's shapes: 32 layers, hidden 4096, 32 query / 8 KV heads of 128,
MLP 14336, vocabulary 128256, RoPE theta 500000."""

TINY = DecoderConfig(layers=2, hidden=256, heads=4, kv_heads=2, head_dim=64, ffn=512, vocab=512,
                     rope_theta=10000.0, split_size=64)
"""A two-layer decoder small enough for the fp64 oracle."""


# Below one full 128-row tile the fused SwiGLU epilogue is slower than the
# two-kernel form: its element work falls on the few warps that own valid
# rows, after the tile's last MMA, with nothing to overlap (GB300, gate/up
# 2 x 14336 by 4096: 55 against 50 us at 16 rows, 53 against 54 at 128, 90
# against 99 at 512, 1.05 against 1.21 ms at 8192).
SWIGLU_FUSE_MIN_ROWS = 128


class DecoderWeights:
    """Random bf16 weights N(0, init_std^2), norm weights 1.  Linear weights
    are [out, in] (the GEMM's W [N, K]); the q/k/v and gate/up projections are
    stacked into one matrix each, the gate/up one in blocks of 128 features
    (the block's gate rows, then its up rows: the layout bi_gemm_swiglu reads,
    so the SwiGLU product comes out of the GEMM epilogue).  ``gen_device`` is
    where the numbers are drawn (CPU for configurations an oracle also reads,
    the GPU for speed)."""

    def __init__(self, cfg: DecoderConfig, seed: int, device, gen_device=None):
        gd = device if gen_device is None else gen_device
        H, s = cfg.hidden, cfg.init_std

        def draw(shape, k):
            return synth.normal_bf16(shape, seed * 100003 + k, std=s, device=gd).to(device)

        self.embed = draw((cfg.vocab, H), 1)
        self.lm_head = draw((cfg.vocab, H), 2)
        self.final_norm = torch.ones(H, dtype=torch.bfloat16, device=device)
        self.attn_norm, self.mlp_norm, self.wqkv, self.wo, self.wgu, self.wdown = ([] for _ in
                                                                                    range(6))
        for layer in range(cfg.layers):
            k = 16 * (layer + 1)
            self.attn_norm.append(torch.ones(H, dtype=torch.bfloat16, device=device))
            self.mlp_norm.append(torch.ones(H, dtype=torch.bfloat16, device=device))
            self.wqkv.append(draw((cfg.qkv_dim, H), k + 1))
            self.wo.append(draw((H, cfg.heads * cfg.head_dim), k + 2))
            self.wgu.append(draw((2 * cfg.ffn, H), k + 3))
            self.wdown.append(draw((H, cfg.ffn), k + 4))


@dataclass
class StepPlan:
    """One forward step, built on the host by the scheduler.

    tokens, pos, row_seq [T]: the step's tokens, their absolute positions and
      the row of ``table`` (the sequence) each belongs to; decode tokens
      first (rows 0 .. n_dec-1 of both), then the prefill chunks.
    table [n_seq, max_blocks], kv_lens [n_seq]: page table rows and KV lengths
      after this step's tokens are written.
    cu_q [n_pre + 1], q_start [n_pre]: the prefill chunks (offsets relative to
      the first prefill token; n_pre = n_seq - n_dec).
    sample_rows [n_s]: the token rows whose logits choose a next token, with
      temperature, seed and counter (the position being chosen) per row.
    """
    tokens: np.ndarray
    pos: np.ndarray
    row_seq: np.ndarray
    table: np.ndarray
    kv_lens: np.ndarray
    n_dec: int
    cu_q: np.ndarray
    q_start: np.ndarray
    sample_rows: np.ndarray
    temperature: np.ndarray
    seed: np.ndarray
    counter: np.ndarray


class _Pack:
    """Packs a step's small host arrays into one pinned buffer (16-byte
    aligned pieces) and moves it to the device with one copy."""

    def __init__(self, nbytes: int, device):
        self.host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
        self.dev = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.off = 0
        self.views = []
        self.copied = None   # event after the last upload's copy

    def add(self, a: np.ndarray, dtype):
        if self.off == 0 and self.copied is not None:
            self.copied.synchronize()      # the host buffer is free again
        a = np.ascontiguousarray(a)
        n = a.nbytes
        if self.off + n > self.host.numel():
            raise ValueError("step plan larger than the planned buffer")
        if n:
            self.host[self.off:self.off + n].numpy()[:] = a.view(np.uint8).reshape(-1)
        self.views.append((self.off, a.shape, dtype))
        self.off = (self.off + n + 15) // 16 * 16

    def upload(self):
        if self.off:
            self.dev[:self.off].copy_(self.host[:self.off], non_blocking=True)
            self.copied = torch.cuda.Event()
            self.copied.record()
        out = []
        for off, shape, dtype in self.views:
            n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            out.append(self.dev[off:off + n].view(dtype).view(shape))
        self.off, self.views = 0, []
        return out


class Decoder:
    """The decoder on one GPU: weights, a paged KV cache of ``num_pages``
    pages per layer, and activation buffers for up to ``max_tokens`` tokens and
    ``max_seqs`` sequences per step.  ``mode`` selects the batch-invariant
    kernels (default) or their batch-variant versions for every call."""

    def __init__(self, cfg: DecoderConfig, weights: DecoderWeights, *, num_pages: int,
                 max_tokens: int, max_seqs: int, max_blocks: int, device,
                 mode: int = bi.INVARIANT, use_graphs: bool = False,
                 graph_kv_bucket: int = 1024, max_graphs: int = 32):
        self.cfg, self.w, self.mode, self.device = cfg, weights, mode, device
        self.max_tokens, self.max_seqs, self.max_blocks = max_tokens, max_seqs, max_blocks
        c = cfg
        self.kv = torch.zeros(c.layers, 2, num_pages, c.kv_heads, c.page_size, c.head_dim,
                              dtype=torch.bfloat16, device=device)
        self.num_pages = num_pages
        T, H, bf = max_tokens, c.hidden, torch.bfloat16

        def buf(*shape, dtype=bf):
            return torch.empty(*shape, dtype=dtype, device=device)

        self.h, self.y, self.qkv = buf(T, H), buf(T, H), buf(T, c.qkv_dim)
        self.q, self.k, self.v = (buf(T, c.heads, c.head_dim), buf(T, c.kv_heads, c.head_dim),
                                  buf(T, c.kv_heads, c.head_dim))
        self.att, self.o = buf(T, c.heads, c.head_dim), buf(T, H)
        self.act, self.delta = buf(T, c.ffn), buf(T, H)
        # the gate/up projection of steps below SWIGLU_FUSE_MIN_ROWS tokens
        self.gu = buf(min(T, SWIGLU_FUSE_MIN_ROWS - 1), 2 * c.ffn)
        self.ys, self.logits = buf(max_seqs, H), buf(max_seqs, c.vocab)
        self.tokens_out = buf(max_seqs, dtype=torch.int32)
        self.tokens_host = torch.empty(max_seqs, dtype=torch.int32, pin_memory=True)
        self.ws = None
        words = 4 * T + max_seqs * (max_blocks + 8) + 64
        self.pack = _Pack(4 * words + 8 * 2 * max_seqs + 16 * 16, device)
        self.sm_scale = c.head_dim ** -0.5
        # decode-step graphs: captured on the second step of a shape, kept
        # (at most max_graphs, oldest dropped) per (decode rows, KV bucket)
        self.use_graphs = use_graphs and mode == bi.INVARIANT
        self.graph_kv_bucket = graph_kv_bucket
        self.max_graphs = max_graphs
        self.graphs, self.seen = {}, set()
        self.graph_replays = 0
        # when a list, eager steps append (layer, name, copy) of every stored
        # activation: the residual stream, each norm's output, q/k/v, the
        # attention output, the projections and the logits (-1: outside the
        # layers); for checking a step stage by stage
        self.capture = None
        if self.use_graphs:
            # the decode workspace at its largest, so that no captured step
            # ever sees it move
            ctx = max_blocks * c.page_size
            self._workspace(bi.bi_attn_decode_workspace_size(
                max_seqs, c.heads, c.kv_heads, c.head_dim, ctx, c.split_size, mode))

    # workspace: one growing device buffer shared by all calls of a step (the
    # calls run in stream order, so they never overlap)
    def _workspace(self, nbytes: int):
        if nbytes == 0:
            return None
        if nbytes == 2 ** 64 - 1:
            raise bi.BiError(bi.ERR_CUDA, "workspace size query")
        if self.ws is None or self.ws.numel() * 4 < nbytes:
            self.ws = torch.empty((nbytes + 15) // 16 * 4, dtype=torch.float32,
                                  device=self.device)
        return self.ws

    def _ws_norm(self, M):
        return self._workspace(bi.bi_rmsnorm_workspace_size(M, self.cfg.hidden, self.mode))

    def _gemm(self, A, W, C):
        ws = None
        if self.mode != bi.INVARIANT:
            ws = self._workspace(bi.bi_gemm_workspace_size(A.shape[0], W.shape[0], A.shape[1],
                                                           self.mode))
        bi.bi_gemm(A, W, C, self.mode, 0, ws)

    def _gemm_swiglu(self, A, W, out):
        """out = SwiGLU of the gate/up projection A W^T: in the GEMM epilogue
        from SWIGLU_FUSE_MIN_ROWS rows on, else as the GEMM then the SwiGLU
        kernel (the same bytes either way)."""
        T = A.shape[0]
        if T < SWIGLU_FUSE_MIN_ROWS:
            gu = self.gu[:T]
            self._gemm(A, W, gu)
            bi.bi_silu_mul(gu, out, block=128)
            return
        ws = None
        if self.mode != bi.INVARIANT:
            ws = self._workspace(bi.bi_gemm_workspace_size(T, W.shape[0], A.shape[1], self.mode))
        bi.bi_gemm_swiglu(A, W, out, self.mode, 0, ws)

    def step(self, plan: StepPlan) -> np.ndarray:
        """Run one forward step; returns the chosen tokens of plan.sample_rows
        (host int32)."""
        c = self.cfg
        T, n_seq, n_dec = len(plan.tokens), len(plan.kv_lens), plan.n_dec
        n_pre, n_s = n_seq - n_dec, len(plan.sample_rows)
        if T == 0 or T > self.max_tokens or n_seq > self.max_seqs or n_s > self.max_seqs:
            raise ValueError("step outside the decoder's buffers")
        if plan.table.shape[1] != self.max_blocks:
            raise ValueError("page table width differs from max_blocks")
        p = self.pack
        p.add(plan.tokens.astype(np.int32), torch.int32)
        p.add(plan.pos.astype(np.int32), torch.int32)
        p.add(plan.row_seq.astype(np.int32), torch.int32)
        p.add(plan.table.astype(np.int32), torch.int32)
        p.add(plan.kv_lens.astype(np.int32), torch.int32)
        p.add(plan.cu_q.astype(np.int32), torch.int32)
        p.add(plan.q_start.astype(np.int32), torch.int32)
        p.add(plan.sample_rows.astype(np.int32), torch.int32)
        p.add(plan.temperature.astype(np.float32), torch.float32)
        p.add(plan.seed.astype(np.uint64).view(np.int64), torch.int64)
        p.add(plan.counter.astype(np.uint64).view(np.int64), torch.int64)
        views = p.upload()
        kv_max = int(plan.kv_lens.max())
        max_q = int(np.diff(plan.cu_q).max()) if n_pre else 0
        if self.use_graphs and n_pre == 0:
            bucket = min(-(-kv_max // self.graph_kv_bucket) * self.graph_kv_bucket,
                         self.max_blocks * c.page_size)
            key = (n_dec, bucket)
            g = self.graphs.get(key)
            if g is None and key in self.seen:
                if len(self.graphs) >= self.max_graphs:
                    self.graphs.pop(next(iter(self.graphs)))
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    self._forward(T, n_dec, n_pre, n_s, views, bucket, max_q)
                self.graphs[key] = g
            self.seen.add(key)
            if g is not None:
                g.replay()
                self.graph_replays += 1
            else:
                self._forward(T, n_dec, n_pre, n_s, views, bucket, max_q)
        else:
            self._forward(T, n_dec, n_pre, n_s, views, kv_max, max_q)
        if n_s == 0:
            return np.empty(0, np.int32)
        out = self.tokens_host[:n_s]
        out.copy_(self.tokens_out[:n_s])      # synchronous: the step's one read-back
        return out.numpy().copy()

    def _forward(self, T, n_dec, n_pre, n_s, views, kv_max, max_q):
        """Enqueue one step's kernels (no host synchronisation, no allocation
        once the workspace has its size); kv_max is a host bound on the KV
        lengths."""
        c, w, mode = self.cfg, self.w, self.mode
        (tok, pos, row_seq, table, kv_lens, cu_q, q_start, rows, temp, seed, counter) = views
        keep = self.capture is not None and not torch.cuda.is_current_stream_capturing()
        cap = self._keep if keep else (lambda *a: None)
        h, y = self.h[:T], self.y[:T]
        bi.bi_gather_rows(w.embed, tok, h)
        bi.bi_rmsnorm(h, w.attn_norm[0], y, c.eps, mode, self._ws_norm(T))
        delta = self.delta[:T]
        for layer in range(c.layers):
            if layer:
                bi.bi_add_rmsnorm(delta, h, w.attn_norm[layer], y, c.eps, mode, self._ws_norm(T))
            cap(layer, "h", h)
            cap(layer, "y_attn", y)
            qkv = self.qkv[:T]
            self._gemm(y, w.wqkv[layer], qkv)
            q, k, v = self.q[:T], self.k[:T], self.v[:T]
            bi.bi_rope_qkv(qkv, pos, c.heads, c.kv_heads, c.head_dim, c.rope_theta, q, k, v)
            cap(layer, "qkv", qkv)
            cap(layer, "q", q)
            cap(layer, "k", k)
            cap(layer, "v", v)
            kc, vc = self.kv[layer, 0], self.kv[layer, 1]
            bi.bi_kv_write(k, v, row_seq, pos, kc, vc, table)
            att = self.att[:T]
            if n_dec:
                ws = self._workspace(bi.bi_attn_decode_workspace_size(
                    n_dec, c.heads, c.kv_heads, c.head_dim, kv_max, c.split_size, mode))
                bi.bi_attn_decode(q[:n_dec], kc, vc, table[:n_dec], kv_lens[:n_dec], att[:n_dec],
                                  max_kv_len=kv_max, split_size=c.split_size,
                                  sm_scale=self.sm_scale, mode=mode, workspace=ws)
            if n_pre:
                bi.bi_attn_prefill_chunk(q[n_dec:], cu_q, q_start, kc, vc, table[n_dec:],
                                         kv_lens[n_dec:], att[n_dec:],
                                         max_q_len=max_q,
                                         max_kv_len=kv_max, split_size=c.split_size,
                                         sm_scale=self.sm_scale, mode=mode)
            cap(layer, "att", att)
            o = self.o[:T]
            self._gemm(att.view(T, c.heads * c.head_dim), w.wo[layer], o)
            cap(layer, "o", o)
            bi.bi_add_rmsnorm(o, h, w.mlp_norm[layer], y, c.eps, mode, self._ws_norm(T))
            cap(layer, "h_mid", h)
            cap(layer, "y_mlp", y)
            act = self.act[:T]
            self._gemm_swiglu(y, w.wgu[layer], act)
            if T < SWIGLU_FUSE_MIN_ROWS:
                cap(layer, "gate_up", self.gu[:T])
            cap(layer, "act", act)
            self._gemm(act, w.wdown[layer], delta)
            cap(layer, "delta", delta)
        bi.bi_add_rmsnorm(delta, h, w.final_norm, y, c.eps, mode, self._ws_norm(T))
        cap(-1, "h", h)
        cap(-1, "y_final", y)
        if n_s == 0:
            return
        ys, logits = self.ys[:n_s], self.logits[:n_s]
        bi.bi_gather_rows(y, rows, ys)
        self._gemm(ys, w.lm_head, logits)
        cap(-1, "logits", logits)
        bi.bi_sample(logits, temp, seed, counter, self.tokens_out[:n_s])

    def _keep(self, layer, name, t):
        self.capture.append((layer, name, t.clone()))
