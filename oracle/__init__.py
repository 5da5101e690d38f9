"""fp64 CPU oracle for the batch-invariant reduction kernels.

TEST INFRASTRUCTURE ONLY.  This package is imported by ``tests/``, by
``__graft_entry__.smoke()`` and by the CPU-baseline leg of ``bench.py``;
nothing in the product path (the ``invariant_bi_rmsnorm_02_gb300`` package and
its CUDA library) may import, link or call it, and it imports nothing from
there.  The arithmetic lives in ``oracle.c`` (plain C, double precision, one
POSIX thread per slice of independent rows); this module only compiles it with
gcc and marshals numpy / torch-CPU arrays through ctypes.

Every function states the plain definition it computes, citing the page:

* [P1] "Reproducible LLM Inference - Batch Invariance, the Cost of Determinism,
  and Where Bitwise Identity Is Actually Required" (hidekazu-konishi.com)
* [P3] "Your Answer Depends on Who Else Is in the Batch" (praveentn.live)

Inputs are bf16 tensors (torch, CPU) or numpy uint16 arrays holding bf16 bit
patterns; outputs are numpy float64 arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_i32 = ctypes.c_int
_dbl = ctypes.c_double
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, no fast-math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_default_threads.restype = _i32
            lib.oracle_rmsnorm.argtypes = [_vp, _vp, _i64, _i64, _dbl, _vp, _vp, _i32]
            lib.oracle_rmsnorm.restype = _i32
            lib.oracle_add_bf16.argtypes = [_vp, _vp, _i64, _vp]
            lib.oracle_add_bf16.restype = _i32
            lib.oracle_gemm.argtypes = [_vp, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _i32]
            lib.oracle_gemm.restype = _i32
            lib.oracle_attention.argtypes = [_vp, _i64, _i32, _i32, _vp, _vp, _vp, _vp,
                                             _i32, _i32, _i64, _vp, _i32, _dbl, _vp, _i32]
            lib.oracle_attention.restype = _i32
            lib.oracle_attention_splits.argtypes = [_vp, _i64, _i32, _i32, _vp, _vp, _vp,
                                                    _vp, _i32, _i32, _i64, _vp, _i32, _dbl,
                                                    _i64, _i64, _vp, _i32]
            lib.oracle_attention_splits.restype = _i32
            lib.oracle_split_starts_fixed_size.argtypes = [_i64, _i64, _vp, _i64]
            lib.oracle_split_starts_fixed_size.restype = _i64
            lib.oracle_split_starts_fixed_count.argtypes = [_i64, _i64, _vp, _i64]
            lib.oracle_split_starts_fixed_count.restype = _i64
            lib.oracle_philox4x64.argtypes = [_vp, _vp, _vp]
            lib.oracle_philox4x64.restype = None
            lib.oracle_sample_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, _i64, _i64,
                                                  _vp]
            lib.oracle_sample_uniform.restype = _i32
            lib.oracle_sample_scores.argtypes = [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _i32]
            lib.oracle_sample_scores.restype = _i32
            _lib = lib
    return _lib


def default_threads() -> int:
    """Number of host threads the oracle uses when nthreads <= 0."""
    return int(_load().oracle_default_threads())


def _bits(t) -> np.ndarray:
    """bf16 tensor (torch) or uint16 array -> contiguous uint16 bit patterns."""
    if isinstance(t, np.ndarray):
        if t.dtype != np.uint16:
            raise TypeError("numpy input must hold bf16 bit patterns as uint16")
        return np.ascontiguousarray(t)
    import torch
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor, got %s" % t.dtype)
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32arr(a) -> np.ndarray:
    if not isinstance(a, np.ndarray):
        a = a.detach().cpu().numpy() if hasattr(a, "detach") else np.asarray(a)
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a: np.ndarray) -> int:
    return a.ctypes.data if a is not None else None


def rmsnorm(x, w, eps: float, nthreads: int = 0, return_mean_sq: bool = False):
    """RMSNorm of each row of x [M,H] (P3 "A Concrete Example"; RMSNorm per
    Zhang & Sennrich, cited by P3):  y = x / sqrt(mean(x^2) + eps) * w."""
    xb, wb = _bits(x), _bits(w)
    M, H = xb.shape
    if wb.shape != (H,):
        raise ValueError("w must be [H]")
    y = np.empty((M, H), np.float64)
    ms = np.empty((M,), np.float64)
    rc = _load().oracle_rmsnorm(_p(xb), _p(wb), M, H, float(eps), _p(y), _p(ms), nthreads)
    if rc:
        raise RuntimeError("oracle_rmsnorm failed: %d" % rc)
    return (y, ms) if return_mean_sq else y


def add_bf16(x, r) -> np.ndarray:
    """The bf16 residual stream after an add: round_bf16(float32(x) + float32(r))
    element by element; returns the uint16 bit patterns, shape of x."""
    xb, rb = _bits(x), _bits(r)
    if xb.shape != rb.shape:
        raise ValueError("x and r differ in shape")
    h = np.empty(xb.shape, np.uint16)
    rc = _load().oracle_add_bf16(_p(xb), _p(rb), xb.size, _p(h))
    if rc:
        raise RuntimeError("oracle_add_bf16 failed: %d" % rc)
    return h


def add_rmsnorm(x, r, w, eps: float, nthreads: int = 0):
    """Pre-norm step of a decoder layer: h = add_bf16(x, r), y = rmsnorm(h, w).
    Returns (h as uint16 bf16 bits, y float64)."""
    h = add_bf16(x, r)
    return h, rmsnorm(h, w, eps, nthreads)


def gemm(A, W, rows=None, nthreads: int = 0) -> np.ndarray:
    """C[i,n] = sum_k A[i,k] W[n,k] (P1 §3.3), A [M,K], W [N,K].  With
    ``rows`` only those rows of A are computed (result [len(rows), N])."""
    ab, wb = _bits(A), _bits(W)
    M, K = ab.shape
    N, K2 = wb.shape
    if K != K2:
        raise ValueError("inner dimensions differ")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nr = M if r is None else len(r)
    C = np.empty((nr, N), np.float64)
    rc = _load().oracle_gemm(_p(ab), _p(wb), M, N, K, _p(r), 0 if r is None else len(r),
                             _p(C), nthreads)
    if rc:
        raise RuntimeError("oracle_gemm failed: %d" % rc)
    return C


def attention(q, row_seq, row_nkeys, k_cache, v_cache, block_table, scale: float,
              nthreads: int = 0, split_size: int = 0, split_count: int = 0) -> np.ndarray:
    """Softmax attention of each query row over keys 0..row_nkeys[r]-1 of its
    sequence, read through the page table (P1 §5.5).

    q: [R, Hq, D] bf16; k_cache/v_cache: [num_pages, Hkv, page, D] bf16;
    block_table: [B, max_blocks] int32.  Decode passes one row per request with
    n = kv length; causal prefill one row per token with n = position + 1.
    With split_size or split_count the same result is evaluated split by split
    and merged in index order (the split statement, P1 §4.3 and §5.5)."""
    qb = _bits(q)
    kb, vb = _bits(k_cache), _bits(v_cache)
    R, Hq, D = qb.shape
    num_pages, Hkv, page, D2 = kb.shape
    if D2 != D or vb.shape != kb.shape:
        raise ValueError("cache shape mismatch")
    rs, rn, bt = _i32arr(row_seq), _i32arr(row_nkeys), _i32arr(block_table)
    if rs.shape != (R,) or rn.shape != (R,) or bt.ndim != 2:
        raise ValueError("row_seq/row_nkeys must be [R]; block_table [B, max_blocks]")
    out = np.empty((R, Hq, D), np.float64)
    lib = _load()
    if split_size or split_count:
        rc = lib.oracle_attention_splits(_p(qb), R, Hq, D, _p(rs), _p(rn), _p(kb), _p(vb),
                                         Hkv, page, num_pages, _p(bt), bt.shape[1],
                                         float(scale), split_size, split_count, _p(out),
                                         nthreads)
    else:
        rc = lib.oracle_attention(_p(qb), R, Hq, D, _p(rs), _p(rn), _p(kb), _p(vb), Hkv,
                                  page, num_pages, _p(bt), bt.shape[1], float(scale),
                                  _p(out), nthreads)
    if rc:
        raise RuntimeError("oracle_attention failed: %d" % rc)
    return out


def decode_attention(q, k_cache, v_cache, block_table, kv_lens, scale: float,
                     nthreads: int = 0) -> np.ndarray:
    """Decode: request b's single query [B, Hq, D] over its kv_lens[b] keys."""
    kl = _i32arr(kv_lens)
    B = kl.shape[0]
    return attention(q, np.arange(B, dtype=np.int32), kl, k_cache, v_cache, block_table,
                     scale, nthreads)


def prefill_attention(q, seq, positions, k_cache, v_cache, block_table, scale: float,
                      nthreads: int = 0) -> np.ndarray:
    """Causal prefill: the token at absolute position p of sequence ``seq``
    attends to keys 0..p (P1 §5.5: the reduction for a token must not depend
    on how its sequence is chunked).  q: [T, Hq, D]; positions: [T]."""
    pos = _i32arr(positions)
    s = np.full(pos.shape, seq, np.int32) if np.isscalar(seq) else _i32arr(seq)
    return attention(q, s, pos + 1, k_cache, v_cache, block_table, scale, nthreads)


def split_starts_fixed_size(L: int, S: int) -> list:
    """Chunk starts (plus the end L) of the fixed split-SIZE plan (P1 §5.5)."""
    cap = L // max(S, 1) + 3
    buf = np.zeros(cap, np.int64)
    n = _load().oracle_split_starts_fixed_size(L, S, _p(buf), cap)
    if n < 0:
        raise ValueError("bad split plan arguments")
    return [int(v) for v in buf[: n + 1]]


def split_starts_fixed_count(L: int, count: int) -> list:
    """Chunk starts (plus the end L) of the fixed split-COUNT plan (P3)."""
    cap = count + 1
    buf = np.zeros(cap, np.int64)
    n = _load().oracle_split_starts_fixed_count(L, count, _p(buf), cap)
    if n < 0:
        raise ValueError("bad split plan arguments")
    return [int(v) for v in buf[: n + 1]]


# --------------------------------------------------------------------------
# seeded sampling
# --------------------------------------------------------------------------
def philox4x64(counter, key) -> np.ndarray:
    """Philox4x64-10 (Salmon et al., SC 2011) of a 4-word counter under a
    2-word key: the four 64-bit output words."""
    c = np.ascontiguousarray(counter, dtype=np.uint64)
    k = np.ascontiguousarray(key, dtype=np.uint64)
    if c.shape != (4,) or k.shape != (2,):
        raise ValueError("counter has 4 words, key 2")
    out = np.empty(4, np.uint64)
    _load().oracle_philox4x64(_p(c), _p(k), _p(out))
    return out


def sample_uniform(seed: int, step: int, v0: int, n: int) -> np.ndarray:
    """The uniforms in (0, 1) of vocabulary entries v0 .. v0+n-1 for one
    (seed, step) -- the random numbers behind the Gumbel noise."""
    u = np.empty(n, np.float64)
    rc = _load().oracle_sample_uniform(int(seed), int(step), int(v0), int(n), _p(u))
    if rc:
        raise RuntimeError("oracle_sample_uniform failed: %d" % rc)
    return u


def sample(logits, temperature, seed, step, nthreads: int = 0):
    """Seeded Gumbel-max sampling (P1 §9.3; §9.2 for temperature 0): for each
    row b, token = argmax_v score[b, v] with score = z / T_b - log(-log(u))
    when T_b > 0 and score = z otherwise; ties go to the lowest index.
    logits [B, V] bf16; temperature float32 [B]; seed, step uint64 [B].
    Returns (tokens int64 [B], scores float64 [B, V])."""
    zb = _bits(logits)
    B, V = zb.shape
    T = np.ascontiguousarray(np.asarray(temperature, dtype=np.float32).reshape(B))
    sd = np.ascontiguousarray(np.asarray(seed, dtype=np.uint64).reshape(B))
    st = np.ascontiguousarray(np.asarray(step, dtype=np.uint64).reshape(B))
    scores = np.empty((B, V), np.float64)
    rc = _load().oracle_sample_scores(_p(zb), B, V, _p(T), _p(sd), _p(st), _p(scores), nthreads)
    if rc:
        raise RuntimeError("oracle_sample_scores failed: %d" % rc)
    return np.argmax(scores, axis=1).astype(np.int64), scores


# --------------------------------------------------------------------------
# element-wise decoder-layer steps (numpy, float64)
# --------------------------------------------------------------------------
def _widen(t) -> np.ndarray:
    """bf16 (torch tensor or uint16 bits) -> float64, exactly."""
    b = _bits(t).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def gather_rows(src, idx) -> np.ndarray:
    """Row gather (token embedding lookup): the bf16 bit patterns of
    src[idx[i], :] for each i."""
    return _bits(src)[np.asarray(idx, dtype=np.int64)]


def rope(x, pos, theta: float) -> np.ndarray:
    """Rotary position embedding of x [T, H, D] at positions pos [T], in the
    rotate-half arrangement of the Llama family (the pages fix no positional
    encoding): pair i < D/2 of a head holds elements i and i + D/2 and turns
    by the angle pos * theta^(-2i/D) (counter-clockwise, element i as the real
    part)."""
    xv = _widen(x)
    D = xv.shape[-1]
    half = D // 2
    i = np.arange(half, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * theta ** (-2.0 * i / D)
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = xv[..., :half], xv[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_qkv(qkv, pos, Hq: int, Hkv: int, D: int, theta: float):
    """Split a stacked QKV projection [T, (Hq + 2 Hkv) D] into q, k, v and
    rotate q and k (see rope); v is returned unrotated (float64)."""
    T = qkv.shape[0]
    bits = _bits(qkv).reshape(T, Hq + 2 * Hkv, D)
    q = rope(bits[:, :Hq], pos, theta)
    k = rope(bits[:, Hq:Hq + Hkv], pos, theta)
    v = _widen(bits[:, Hq + Hkv:])
    return q, k, v


def silu_mul(gate_up) -> np.ndarray:
    """SwiGLU product of a stacked [T, 2F] gate/up projection:
    silu(g) * u with silu(g) = g / (1 + exp(-g)) (float64)."""
    gu = _widen(gate_up)
    F = gu.shape[1] // 2
    g, u = gu[:, :F], gu[:, F:]
    return g / (1.0 + np.exp(-g)) * u
