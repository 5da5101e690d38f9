"""Thin ctypes binding over libbi.so (the C ABI in include/bi.h).

The functions named ``bi_*`` mirror the C entry points one to one: they take
torch tensors that already live on the GPU, pass their device pointers and the
current CUDA stream, and raise ``BiError`` on a non-OK status.  The short
names (``rmsnorm``, ``gemm``, ``attn_decode``, ``attn_prefill_chunk``,
``kv_write``) additionally allocate the outputs and the workspace with torch.
No arithmetic of the method happens here; every step runs in the CUDA
kernels, and a missing library is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbi.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_BOUNDS, ERR_TIMEOUT = range(7)
INVARIANT, VARIANT = 0, 1
NOALLOC_SCRATCH_BYTES = 32 << 20   # BI_NOALLOC_SCRATCH_BYTES in include/bi.h

__all__ = [
    "BiError", "INVARIANT", "VARIANT", "LIB_PATH", "load", "library_path", "OK",
    "ERR_INVALID_ARG", "ERR_UNSUPPORTED", "ERR_WORKSPACE", "ERR_CUDA", "ERR_DEVICE_BOUNDS",
    "ERR_TIMEOUT",
    "bi_rmsnorm", "bi_rmsnorm_workspace_size", "bi_gemm", "bi_gemm_workspace_size",
    "bi_gemm_variant_splits", "bi_attn_decode", "bi_attn_decode_workspace_size",
    "bi_attn_prefill_chunk", "bi_kv_write", "bi_check_device_errors", "bi_status_string",
    "bi_version", "bi_attn_decode_noalloc", "bi_selftest_wait_timeout", "bi_add_rmsnorm",
    "bi_sample", "bi_gather_rows", "bi_rope_qkv", "bi_silu_mul", "bi_gemm_swiglu",
    "NOALLOC_SCRATCH_BYTES", "rmsnorm", "add_rmsnorm", "gemm", "gemm_swiglu",
    "swiglu_interleave", "attn_decode", "attn_prefill_chunk", "kv_write", "sample",
    "gather_rows", "rope_qkv", "silu_mul", "EXPORTED_SYMBOLS",
]

# every function include/bi.h declares
EXPORTED_SYMBOLS = (
    "bi_rmsnorm", "bi_rmsnorm_workspace_size", "bi_gemm", "bi_gemm_workspace_size",
    "bi_gemm_variant_splits", "bi_attn_decode", "bi_attn_decode_workspace_size",
    "bi_attn_prefill_chunk", "bi_kv_write", "bi_check_device_errors", "bi_status_string",
    "bi_version", "bi_attn_decode_noalloc", "bi_selftest_wait_timeout", "bi_add_rmsnorm",
    "bi_sample", "bi_gather_rows", "bi_rope_qkv", "bi_silu_mul", "bi_gemm_swiglu",
)


class BiError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, _status_text(status), status))


_lock = threading.Lock()
_lib = None

_vp, _i64, _i32, _f32, _sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                             ctypes.c_size_t)


def library_path() -> str:
    return LIB_PATH


def load(build_if_missing: bool = True):
    """Load libbi.so (building it with nvcc first if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            if not build_if_missing:
                raise RuntimeError("libbi.so is not built (run the package's build step)")
            from . import build as _build
            _build.build()
        import torch.cuda  # noqa: F401  (loads the CUDA runtime torch ships)
        lib = ctypes.CDLL(LIB_PATH)
        sig = {
            "bi_rmsnorm": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _f32, _i32, _vp, _sz, _vp]),
            "bi_add_rmsnorm": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _f32, _i32, _vp, _sz,
                                      _vp]),
            "bi_rmsnorm_workspace_size": (_sz, [_i64, _i64, _i32]),
            "bi_gemm": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _vp, _sz, _vp]),
            "bi_gemm_workspace_size": (_sz, [_i64, _i64, _i64, _i32, _i32]),
            "bi_gemm_variant_splits": (_i32, [_i64, _i64, _i64, _i32]),
            "bi_gemm_swiglu": (_i32, [_vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _vp, _sz,
                                      _vp]),
            "bi_attn_decode": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                      _i32, _i64, _i32, _i32, _i32, _f32, _i32, _i32, _vp, _sz,
                                      _vp]),
            "bi_attn_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                                    _i32]),
            "bi_attn_prefill_chunk": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                             _i32, _i32, _i32, _i32, _i64, _i32, _i64, _i32,
                                             _i32, _i32, _f32, _i32, _i32, _vp, _sz, _vp]),
            "bi_kv_write": (_i32, [_vp, _vp, _vp, _vp, _i64, _vp, _vp, _vp, _i32, _i32, _i32,
                                   _i64, _i32, _vp]),
            "bi_attn_decode_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                              _i32, _i32, _i32, _i64, _i32, _i32, _i32, _f32,
                                              _vp]),
            "bi_sample": (_i32, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
            "bi_gather_rows": (_i32, [_vp, _i64, _i64, _vp, _i64, _vp, _vp]),
            "bi_rope_qkv": (_i32, [_vp, _vp, _i64, _i32, _i32, _i32, ctypes.c_double, _vp, _vp,
                                   _vp, _vp]),
            "bi_silu_mul": (_i32, [_vp, _i64, _i64, _i64, _vp, _vp]),
            "bi_check_device_errors": (_i32, [_vp]),
            "bi_selftest_wait_timeout": (_i32, [ctypes.c_uint32, _vp]),
            "bi_status_string": (ctypes.c_char_p, [_i32]),
            "bi_version": (ctypes.c_char_p, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _status_text(status: int) -> str:
    try:
        return load().bi_status_string(status).decode()
    except Exception:  # pragma: no cover - library not loadable
        return "status"


def _check(status: int, what: str) -> None:
    if status != OK:
        raise BiError(status, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _ws(workspace):
    if workspace is None:
        return None, 0
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


# ---------------------------------------------------------------- raw entry points
def bi_rmsnorm(x, w, y, eps, mode=INVARIANT, workspace=None, stream=None, y_f32=None):
    M, H = x.shape
    wp, wb = _ws(workspace)
    _check(load().bi_rmsnorm(_ptr(x, torch.bfloat16, "x"), _ptr(w, torch.bfloat16, "w"),
                             _ptr(y, torch.bfloat16, "y"), _ptr(y_f32, torch.float32, "y_f32"),
                             M, H, float(eps), int(mode), wp, wb, _stream(stream)),
           "bi_rmsnorm")


def bi_add_rmsnorm(x, residual, w, y, eps, mode=INVARIANT, workspace=None, stream=None,
                   y_f32=None):
    """residual <- bf16(x + residual); y <- RMSNorm(residual) * w (include/bi.h)."""
    M, H = x.shape
    if tuple(residual.shape) != (M, H) or tuple(y.shape) != (M, H):
        raise ValueError("x, residual and y must have the same shape")
    wp, wb = _ws(workspace)
    _check(load().bi_add_rmsnorm(_ptr(x, torch.bfloat16, "x"),
                                 _ptr(residual, torch.bfloat16, "residual"),
                                 _ptr(w, torch.bfloat16, "w"), _ptr(y, torch.bfloat16, "y"),
                                 _ptr(y_f32, torch.float32, "y_f32"), M, H, float(eps),
                                 int(mode), wp, wb, _stream(stream)), "bi_add_rmsnorm")


def bi_rmsnorm_workspace_size(M, H, mode=INVARIANT) -> int:
    return int(load().bi_rmsnorm_workspace_size(M, H, int(mode)))


def bi_gemm(A, W, C, mode=INVARIANT, variant_splits=0, workspace=None, stream=None):
    M, K = A.shape
    N = W.shape[0]
    wp, wb = _ws(workspace)
    _check(load().bi_gemm(_ptr(A, torch.bfloat16, "A"), _ptr(W, torch.bfloat16, "W"),
                          _ptr(C, torch.bfloat16, "C"), M, N, K, int(mode), int(variant_splits),
                          wp, wb, _stream(stream)), "bi_gemm")


def bi_gemm_workspace_size(M, N, K, mode=INVARIANT, variant_splits=0) -> int:
    return int(load().bi_gemm_workspace_size(M, N, K, int(mode), int(variant_splits)))


def bi_gemm_variant_splits(M, N, K, num_sms) -> int:
    return int(load().bi_gemm_variant_splits(M, N, K, int(num_sms)))


def bi_gemm_swiglu(A, W, out, mode=INVARIANT, variant_splits=0, workspace=None, stream=None):
    M, K = A.shape
    F = W.shape[0] // 2
    if W.shape[0] % 2 or tuple(out.shape) != (M, F):
        raise ValueError("W must be [2F, K] and out [M, F]")
    wp, wb = _ws(workspace)
    _check(load().bi_gemm_swiglu(_ptr(A, torch.bfloat16, "A"), _ptr(W, torch.bfloat16, "W"),
                                 _ptr(out, torch.bfloat16, "out"), M, F, K, int(mode),
                                 int(variant_splits), wp, wb, _stream(stream)), "bi_gemm_swiglu")


def bi_attn_decode(q, k_cache, v_cache, block_table, kv_lens, out, out_f32=None, *,
                   max_kv_len, split_size, sm_scale, mode=INVARIANT, variant_splits=0,
                   workspace=None, stream=None):
    B, Hq, D = q.shape
    num_pages, Hkv, page, D2 = k_cache.shape
    wp, wb = _ws(workspace)
    _check(load().bi_attn_decode(
        _ptr(q, torch.bfloat16, "q"), _ptr(k_cache, torch.bfloat16, "k_cache"),
        _ptr(v_cache, torch.bfloat16, "v_cache"), _ptr(block_table, torch.int32, "block_table"),
        _ptr(kv_lens, torch.int32, "kv_lens"), _ptr(out, torch.bfloat16, "out"),
        _ptr(out_f32, torch.float32, "out_f32"), B, Hq, Hkv, D, page, num_pages,
        block_table.shape[1], int(max_kv_len), int(split_size), float(sm_scale), int(mode),
        int(variant_splits), wp, wb, _stream(stream)), "bi_attn_decode")


def bi_attn_decode_noalloc(q, k_cache, v_cache, block_table, kv_lens, out, out_f32=None, *,
                           max_kv_len, split_size, sm_scale, stream=None):
    """Decode without a workspace argument (scratch from the library's fixed
    array); for callers that cannot allocate device memory."""
    B, Hq, D = q.shape
    num_pages, Hkv, page, _ = k_cache.shape
    _check(load().bi_attn_decode_noalloc(
        _ptr(q, torch.bfloat16, "q"), _ptr(k_cache, torch.bfloat16, "k_cache"),
        _ptr(v_cache, torch.bfloat16, "v_cache"), _ptr(block_table, torch.int32, "block_table"),
        _ptr(kv_lens, torch.int32, "kv_lens"), _ptr(out, torch.bfloat16, "out"),
        _ptr(out_f32, torch.float32, "out_f32"), B, Hq, Hkv, D, page, num_pages,
        block_table.shape[1], int(max_kv_len), int(split_size), float(sm_scale),
        _stream(stream)), "bi_attn_decode_noalloc")


def bi_attn_decode_workspace_size(B, Hq, Hkv, D, max_kv_len, split_size, mode=INVARIANT,
                                  variant_splits=0) -> int:
    return int(load().bi_attn_decode_workspace_size(B, Hq, Hkv, D, max_kv_len, split_size,
                                                    int(mode), int(variant_splits)))


def bi_attn_prefill_chunk(q, cu_q, q_start_pos, k_cache, v_cache, block_table, kv_lens, out,
                          out_f32=None, *, max_q_len, max_kv_len, split_size, sm_scale,
                          mode=INVARIANT, variant_splits=0, workspace=None, stream=None):
    total_q, Hq, D = q.shape
    num_pages, Hkv, page, _ = k_cache.shape
    B = kv_lens.shape[0]
    wp, wb = _ws(workspace)
    _check(load().bi_attn_prefill_chunk(
        _ptr(q, torch.bfloat16, "q"), _ptr(cu_q, torch.int32, "cu_q"),
        _ptr(q_start_pos, torch.int32, "q_start_pos"), _ptr(k_cache, torch.bfloat16, "k_cache"),
        _ptr(v_cache, torch.bfloat16, "v_cache"), _ptr(block_table, torch.int32, "block_table"),
        _ptr(kv_lens, torch.int32, "kv_lens"), _ptr(out, torch.bfloat16, "out"),
        _ptr(out_f32, torch.float32, "out_f32"), B, Hq, Hkv, D, page, num_pages,
        block_table.shape[1], total_q, int(max_q_len), int(max_kv_len), int(split_size),
        float(sm_scale), int(mode), int(variant_splits), wp, wb, _stream(stream)),
        "bi_attn_prefill_chunk")


def bi_kv_write(k_new, v_new, seq, pos, k_cache, v_cache, block_table, stream=None):
    n, Hkv, D = k_new.shape
    num_pages, _, page, _ = k_cache.shape
    _check(load().bi_kv_write(
        _ptr(k_new, torch.bfloat16, "k_new"), _ptr(v_new, torch.bfloat16, "v_new"),
        _ptr(seq, torch.int32, "seq"), _ptr(pos, torch.int32, "pos"), n,
        _ptr(k_cache, torch.bfloat16, "k_cache"), _ptr(v_cache, torch.bfloat16, "v_cache"),
        _ptr(block_table, torch.int32, "block_table"), Hkv, D, page, num_pages,
        block_table.shape[1], _stream(stream)), "bi_kv_write")


def bi_sample(logits, temperature, seed, step, tokens, stream=None):
    """tokens[b] <- the token of row b of logits (include/bi.h).  seed and step
    are int64 tensors whose bits are read as uint64."""
    B, V = logits.shape
    for t, name in ((temperature, "temperature"), (seed, "seed"), (step, "step"),
                    (tokens, "tokens")):
        if tuple(t.shape) != (B,):
            raise ValueError("%s must have shape [B]" % name)
    _check(load().bi_sample(_ptr(logits, torch.bfloat16, "logits"), B, V,
                            _ptr(temperature, torch.float32, "temperature"),
                            _ptr(seed, torch.int64, "seed"), _ptr(step, torch.int64, "step"),
                            _ptr(tokens, torch.int32, "tokens"), _stream(stream)), "bi_sample")


def bi_gather_rows(src, idx, dst, stream=None):
    rows, H = src.shape
    n = idx.shape[0]
    if tuple(dst.shape) != (n, H):
        raise ValueError("dst must be [len(idx), H]")
    _check(load().bi_gather_rows(_ptr(src, torch.bfloat16, "src"), rows, H,
                                 _ptr(idx, torch.int32, "idx"), n,
                                 _ptr(dst, torch.bfloat16, "dst"), _stream(stream)),
           "bi_gather_rows")


def bi_rope_qkv(qkv, pos, Hq, Hkv, D, theta, q, k, v, stream=None):
    T = qkv.shape[0]
    if qkv.shape[1] != (Hq + 2 * Hkv) * D or pos.shape != (T,):
        raise ValueError("qkv must be [T, (Hq + 2 Hkv) D] and pos [T]")
    if q.shape != (T, Hq, D) or k.shape != (T, Hkv, D) or v.shape != (T, Hkv, D):
        raise ValueError("q, k, v must be [T, H, D]")
    _check(load().bi_rope_qkv(_ptr(qkv, torch.bfloat16, "qkv"), _ptr(pos, torch.int32, "pos"), T,
                              Hq, Hkv, D, float(theta), _ptr(q, torch.bfloat16, "q"),
                              _ptr(k, torch.bfloat16, "k"), _ptr(v, torch.bfloat16, "v"),
                              _stream(stream)), "bi_rope_qkv")


def bi_silu_mul(gate_up, out, block=None, stream=None):
    """block: features per gate/up block (None: F, i.e. the gate half then
    the up half; 128: the layout bi_gemm writes with bi_gemm_swiglu's
    weight)."""
    T, F2 = gate_up.shape
    if F2 % 2 or tuple(out.shape) != (T, F2 // 2):
        raise ValueError("gate_up must be [T, 2F] and out [T, F]")
    blk = F2 // 2 if block is None else int(block)
    _check(load().bi_silu_mul(_ptr(gate_up, torch.bfloat16, "gate_up"), T, F2 // 2, blk,
                              _ptr(out, torch.bfloat16, "out"), _stream(stream)), "bi_silu_mul")


def bi_check_device_errors(stream=None) -> int:
    return int(load().bi_check_device_errors(_stream(stream)))


def bi_selftest_wait_timeout(timeout_us: int, stream=None) -> int:
    """Launch the bounded-wait diagnostic (see include/bi.h); returns the
    launch status, the recorded one comes from bi_check_device_errors."""
    return int(load().bi_selftest_wait_timeout(int(timeout_us), _stream(stream)))


def bi_status_string(status: int) -> str:
    return load().bi_status_string(int(status)).decode()


def bi_version() -> str:
    return load().bi_version().decode()


# ---------------------------------------------------------- allocating helpers
def _workspace(nbytes: int, device) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    if nbytes == 2 ** 64 - 1:
        raise BiError(ERR_CUDA, "workspace size query")
    return torch.empty((nbytes + 15) // 16 * 4, dtype=torch.float32, device=device)


def rmsnorm(x, w, eps=1e-6, mode=INVARIANT, want_f32=False, stream=None):
    y = torch.empty_like(x)
    y32 = torch.empty(x.shape, dtype=torch.float32, device=x.device) if want_f32 else None
    ws = _workspace(bi_rmsnorm_workspace_size(x.shape[0], x.shape[1], mode), x.device)
    bi_rmsnorm(x, w, y, eps, mode, ws, stream, y_f32=y32)
    return (y, y32) if want_f32 else y


def add_rmsnorm(x, residual, w, eps=1e-6, mode=INVARIANT, want_f32=False, stream=None):
    """Updates residual in place (residual <- bf16(x + residual)) and returns
    RMSNorm(residual) * w (and its fp32 values with want_f32)."""
    y = torch.empty_like(x)
    y32 = torch.empty(x.shape, dtype=torch.float32, device=x.device) if want_f32 else None
    ws = _workspace(bi_rmsnorm_workspace_size(x.shape[0], x.shape[1], mode), x.device)
    bi_add_rmsnorm(x, residual, w, y, eps, mode, ws, stream, y_f32=y32)
    return (y, y32) if want_f32 else y


def gemm(A, W, mode=INVARIANT, variant_splits=0, stream=None):
    C = torch.empty(A.shape[0], W.shape[0], dtype=torch.bfloat16, device=A.device)
    ws = _workspace(bi_gemm_workspace_size(A.shape[0], W.shape[0], A.shape[1], mode,
                                           variant_splits), A.device)
    bi_gemm(A, W, C, mode, variant_splits, ws, stream)
    return C


def attn_decode(q, k_cache, v_cache, block_table, kv_lens, *, max_kv_len, split_size,
                sm_scale=None, mode=INVARIANT, variant_splits=0, want_f32=False, stream=None):
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    sm_scale = D ** -0.5 if sm_scale is None else sm_scale
    out = torch.empty_like(q)
    out32 = torch.empty(q.shape, dtype=torch.float32, device=q.device) if want_f32 else None
    ws = _workspace(bi_attn_decode_workspace_size(B, Hq, Hkv, D, max_kv_len, split_size, mode,
                                                  variant_splits), q.device)
    bi_attn_decode(q, k_cache, v_cache, block_table, kv_lens, out, out32,
                   max_kv_len=max_kv_len, split_size=split_size, sm_scale=sm_scale, mode=mode,
                   variant_splits=variant_splits, workspace=ws, stream=stream)
    return (out, out32) if want_f32 else out


def attn_prefill_chunk(q, cu_q, q_start_pos, k_cache, v_cache, block_table, kv_lens, *,
                       max_q_len, max_kv_len, split_size, sm_scale=None, mode=INVARIANT,
                       variant_splits=0, want_f32=False, stream=None):
    D = q.shape[2]
    sm_scale = D ** -0.5 if sm_scale is None else sm_scale
    out = torch.empty_like(q)
    out32 = torch.empty(q.shape, dtype=torch.float32, device=q.device) if want_f32 else None
    bi_attn_prefill_chunk(q, cu_q, q_start_pos, k_cache, v_cache, block_table, kv_lens, out,
                          out32, max_q_len=max_q_len, max_kv_len=max_kv_len,
                          split_size=split_size, sm_scale=sm_scale, mode=mode,
                          variant_splits=variant_splits, stream=stream)
    return (out, out32) if want_f32 else out


def sample(logits, temperature, seed, step, stream=None):
    """One token per row: seeded Gumbel-max at temperature > 0, argmax at 0."""
    tokens = torch.empty(logits.shape[0], dtype=torch.int32, device=logits.device)
    bi_sample(logits, temperature, seed, step, tokens, stream)
    return tokens


def gather_rows(src, idx, stream=None):
    dst = torch.empty(idx.shape[0], src.shape[1], dtype=src.dtype, device=src.device)
    bi_gather_rows(src, idx, dst, stream)
    return dst


def rope_qkv(qkv, pos, Hq, Hkv, D, theta=500000.0, stream=None):
    T = qkv.shape[0]
    q = torch.empty(T, Hq, D, dtype=qkv.dtype, device=qkv.device)
    k = torch.empty(T, Hkv, D, dtype=qkv.dtype, device=qkv.device)
    v = torch.empty(T, Hkv, D, dtype=qkv.dtype, device=qkv.device)
    bi_rope_qkv(qkv, pos, Hq, Hkv, D, theta, q, k, v, stream)
    return q, k, v


def gemm_swiglu(A, W, mode=INVARIANT, variant_splits=0, stream=None):
    out = torch.empty(A.shape[0], W.shape[0] // 2, dtype=torch.bfloat16, device=A.device)
    ws = _workspace(bi_gemm_workspace_size(A.shape[0], W.shape[0], A.shape[1], mode,
                                           variant_splits), A.device)
    bi_gemm_swiglu(A, W, out, mode, variant_splits, ws, stream)
    return out


def swiglu_interleave(F: int) -> np.ndarray:
    """Row order of bi_gemm_swiglu's weight: entry r is the row of a [gate;
    up] stacked weight (gate rows 0..F-1, up rows F..2F-1) that goes to row r
    (blocks of 128 features, the gate rows of a block before its up rows)."""
    if F % 128:
        raise ValueError("F must be a multiple of 128")
    j = np.arange(2 * F)
    blk, r = j // 256, j % 256
    return np.where(r < 128, blk * 128 + r, F + blk * 128 + (r - 128)).astype(np.int32)


def silu_mul(gate_up, block=None, stream=None):
    out = torch.empty(gate_up.shape[0], gate_up.shape[1] // 2, dtype=gate_up.dtype,
                      device=gate_up.device)
    bi_silu_mul(gate_up, out, block, stream)
    return out


def kv_write(k_new, v_new, seq, pos, k_cache, v_cache, block_table, stream=None):
    bi_kv_write(k_new, v_new, seq, pos, k_cache, v_cache, block_table, stream)
