"""fp64 oracle of a whole bf16 decoder forward pass (TEST INFRASTRUCTURE ONLY).

The model is a pre-norm Llama-style decoder whose activations are stored in
bf16 between operations, as a serving engine stores them.  This module states
that definition with the oracle's own operations, each evaluated in float64
from bf16 inputs and its result rounded once to bf16 (round to nearest, ties
to even) where the model stores it:

    h_0 = embed[tokens]
    per layer:  y = RMSNorm(h) * w_attn;  qkv = y W_qkv^T;  q, k = RoPE;  v
                a = causal softmax attention (1/sqrt(D) scale, GQA head groups)
                h = bf16(h + a W_o^T);  y = RMSNorm(h) * w_mlp
                h = bf16(h + (silu(y W_gate^T) * y W_up^T) W_down^T)
    logits = (RMSNorm(h) * w_final) W_lm^T        (float64, not rounded)

W_gate and W_up are stacked into one weight in blocks of 128 features: rows
256b .. 256b+127 are the gate rows of features 128b .. 128b+127 and the next
128 rows the up rows of the same features.

Sources: "Reproducible LLM Inference - Batch Invariance, the Cost of
Determinism, and Where Bitwise Identity Is Actually Required" (§5.3-5.5: the
three reductions; §6: the serving loop) and "Your Answer Depends on Who Else
Is in the Batch" ("A Concrete Example": RMSNorm).  The layer arrangement
around them (pre-norm, RoPE, SwiGLU) is the Llama family's, which the pages
name as the models served but do not spell out.
"""
from __future__ import annotations

import numpy as np

from . import add_bf16, attention, gather_rows, gemm, rmsnorm, rope_qkv, silu_mul


def to_bf16(x) -> np.ndarray:
    """float64 -> bf16 bit patterns (uint16), round to nearest, ties to even,
    at 8 significant bits (normal range; zero stays zero)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m 2^e, 1/2 <= |m| < 1
    q = np.ldexp(np.rint(m * 256.0), e - 8)  # rint rounds half to even
    return (q.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def gate_up_halves(gu) -> np.ndarray:
    """[T, 2F] projection in the blocked gate/up column order -> [T, 2F] with
    all gate columns first, then all up columns (silu_mul's layout)."""
    gu = np.asarray(gu)
    T, F2 = gu.shape
    blocks = gu.reshape(T, F2 // 256, 2, 128)
    return np.concatenate([blocks[:, :, 0, :].reshape(T, -1), blocks[:, :, 1, :].reshape(T, -1)],
                          axis=1)


def forward_logits(weights, cfg, tokens) -> np.ndarray:
    """Logits [T, vocab] (float64) of every position of one sequence whose
    tokens (int, length T) start at position 0.  ``weights`` holds CPU bf16
    tensors shaped like the GPU model's (embed, lm_head, final_norm and per
    layer attn_norm, mlp_norm, wqkv, wo, wgu, wdown)."""
    tok = np.asarray(tokens, dtype=np.int64)
    T = len(tok)
    Hq, Hkv, D, P = cfg.heads, cfg.kv_heads, cfg.head_dim, cfg.page_size
    pos = np.arange(T)
    npages = -(-T // P)
    table = np.arange(npages, dtype=np.int32)[None, :]
    h = gather_rows(weights.embed, tok)
    for layer in range(cfg.layers):
        y = to_bf16(rmsnorm(h, weights.attn_norm[layer], cfg.eps))
        qkv = to_bf16(gemm(y, weights.wqkv[layer]))
        q, k, v = rope_qkv(qkv, pos, Hq, Hkv, D, cfg.rope_theta)
        qb, kb, vb = to_bf16(q), to_bf16(k), to_bf16(v)
        # the sequence's keys and values in pages 0, 1, ... of a private cache
        kc = np.zeros((npages * P, Hkv, D), np.uint16)
        vc = np.zeros((npages * P, Hkv, D), np.uint16)
        kc[:T], vc[:T] = kb, vb
        kc = np.ascontiguousarray(kc.reshape(npages, P, Hkv, D).transpose(0, 2, 1, 3))
        vc = np.ascontiguousarray(vc.reshape(npages, P, Hkv, D).transpose(0, 2, 1, 3))
        a = attention(qb, np.zeros(T, np.int32), pos + 1, kc, vc, table, D ** -0.5)
        o = to_bf16(gemm(to_bf16(a).reshape(T, Hq * D), weights.wo[layer]))
        h = add_bf16(o, h)
        y = to_bf16(rmsnorm(h, weights.mlp_norm[layer], cfg.eps))
        act = to_bf16(silu_mul(gate_up_halves(to_bf16(gemm(y, weights.wgu[layer])))))
        d = to_bf16(gemm(act, weights.wdown[layer]))
        h = add_bf16(d, h)
    y = to_bf16(rmsnorm(h, weights.final_norm, cfg.eps))
    return gemm(y, weights.lm_head)

