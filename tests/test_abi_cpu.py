"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/bi.h declares, sizes workspaces by host
arithmetic, and rejects bad arguments before it touches the device."""
import ctypes
import os
import re

import pytest

import invariant_bi_rmsnorm_02_gb300 as bi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bi.h")


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(bi_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return bi.load()


def test_header_lists_the_entry_points():
    names = header_functions()
    for n in ("bi_rmsnorm", "bi_gemm", "bi_attn_decode", "bi_attn_prefill_chunk"):
        assert n in names
    assert sorted(bi.EXPORTED_SYMBOLS) == names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings_and_version(lib):
    assert bi.bi_status_string(0) == "ok"
    for s in range(1, 7):
        assert bi.bi_status_string(s) not in ("ok", "unknown status")
    assert bi.bi_status_string(99) == "unknown status"
    assert re.fullmatch(r"\d+\.\d+\.\d+", bi.bi_version())


def test_workspace_sizes_are_host_arithmetic(lib):
    assert bi.bi_rmsnorm_workspace_size(8192, 4096, bi.INVARIANT) == 0
    assert bi.bi_rmsnorm_workspace_size(3, 4096, bi.VARIANT) == 3 * 64 * 4
    assert bi.bi_gemm_workspace_size(8192, 6144, 4096, bi.INVARIANT) == 0
    assert bi.bi_gemm_workspace_size(1, 6144, 4096, bi.VARIANT, 4) == 4 * 6144 * 4
    # decode: unit list + split partials, each area rounded up to 256 bytes
    up = lambda x: (x + 255) // 256 * 256

    def dec(B, Hq, D, S_max):
        E = S_max + (S_max & 1)   # {m, l} rows padded to an even count
        return 256 + up(16 * B * S_max) + up(8 * B * Hq * E) + 4 * B * Hq * S_max * D
    assert bi.bi_attn_decode_workspace_size(64, 32, 8, 128, 32768, 256, bi.INVARIANT) == \
        dec(64, 32, 128, 128)
    assert bi.bi_attn_decode_workspace_size(8, 4, 2, 64, 512, 64, bi.VARIANT, 5) == \
        dec(8, 4, 64, 5)
    assert bi.bi_attn_decode_workspace_size(3, 5, 5, 64, 64 * 7, 64, bi.INVARIANT) == \
        dec(3, 5, 64, 7)
    assert bi.bi_attn_decode_workspace_size(3, 4, 2, 64, 0, 64, bi.INVARIANT) == 0


def test_gemm_variant_split_count(lib):
    # split-K only when the tiles cover at most a quarter of the SMs, then
    # until the slices cover them, at least 4 k-blocks per slice; the tiles
    # are the kernel's: 128 x 64 for at most 64 rows when those fit in one
    # wave (and K is at least four whole 64-column groups), else 128 x 256
    assert bi.bi_gemm_variant_splits(8192, 6144, 4096, 152) == 1
    assert bi.bi_gemm_variant_splits(1, 6144, 4096, 152) == 1     # 96 narrow tiles: no split
    assert bi.bi_gemm_variant_splits(64, 6144, 4096, 152) == 1
    assert bi.bi_gemm_variant_splits(65, 6144, 4096, 152) == 8    # 24 wide tiles
    assert bi.bi_gemm_variant_splits(128, 6144, 4096, 152) == 8
    assert bi.bi_gemm_variant_splits(256, 6144, 4096, 152) == 1   # 48 tiles: no split
    assert bi.bi_gemm_variant_splits(1, 14336, 4096, 152) == 1    # 224 narrow > 152: 56 wide
    assert bi.bi_gemm_variant_splits(1, 14336, 4096, 256) == 1    # 224 narrow tiles fit
    assert bi.bi_gemm_variant_splits(1, 512, 256, 152) == 1       # K = 4 k-blocks
    assert bi.bi_gemm_variant_splits(1, 2048, 4096, 152) == 8     # 32 narrow tiles
    assert bi.bi_gemm_variant_splits(1, 512, 4096, 152) == 16     # 8 narrow tiles
    assert bi.bi_gemm_variant_splits(1, 6144, 4000, 152) == 8     # K not whole groups: 24 wide


def _call_rms(lib, x, w, y, M, H, eps=1e-6, mode=0, ws=None, wsb=0):
    return lib.bi_rmsnorm(x, w, y, None, M, H, eps, mode, ws, wsb, None)


def test_rmsnorm_argument_checks(lib):
    p = 1 << 20  # a 16-byte aligned fake address: never dereferenced on these paths
    assert _call_rms(lib, p, p, p, 4, 7) == bi.ERR_UNSUPPORTED
    assert _call_rms(lib, p, p, p, 4, 4 * 65536) == bi.ERR_UNSUPPORTED
    assert _call_rms(lib, p, p, p, -1, 4096) == bi.ERR_INVALID_ARG
    assert _call_rms(lib, None, p, p, 4, 4096) == bi.ERR_INVALID_ARG
    assert _call_rms(lib, p + 2, p, p, 4, 4096) == bi.ERR_INVALID_ARG
    assert _call_rms(lib, p, p, p, 4, 4096, mode=7) == bi.ERR_INVALID_ARG
    assert _call_rms(lib, p, p, p, 4, 4096, eps=-1.0) == bi.ERR_INVALID_ARG
    assert _call_rms(lib, None, None, None, 0, 4096) == bi.OK  # empty batch: no-op


def test_gemm_argument_checks(lib):
    p = 1 << 20
    g = lambda *a: lib.bi_gemm(*a)
    assert g(p, p, p, 4, 100, 64, 0, 0, None, 0, None) == bi.ERR_UNSUPPORTED   # N % 8
    assert g(p, p, p, 4, 128, 60, 0, 0, None, 0, None) == bi.ERR_UNSUPPORTED   # K % 8
    assert g(p, p, p, 4, 0, 64, 0, 0, None, 0, None) == bi.ERR_INVALID_ARG
    assert g(p, None, p, 4, 128, 64, 0, 0, None, 0, None) == bi.ERR_INVALID_ARG
    assert g(p, p, p + 8, 4, 128, 64, 0, 0, None, 0, None) == bi.ERR_INVALID_ARG
    assert g(None, None, None, 0, 128, 64, 0, 0, None, 0, None) == bi.OK


def test_gemm_swiglu_argument_checks(lib):
    p = 1 << 20
    g = lambda *a: lib.bi_gemm_swiglu(*a)
    assert g(p, p, p, 4, 192, 64, 0, 0, None, 0, None) == bi.ERR_UNSUPPORTED   # F % 128
    assert g(p, p, p, 4, 128, 60, 0, 0, None, 0, None) == bi.ERR_UNSUPPORTED   # K % 8
    assert g(p, p, p, 4, 0, 64, 0, 0, None, 0, None) == bi.ERR_INVALID_ARG
    assert g(p, p, p, 4, 128, 64, 5, 0, None, 0, None) == bi.ERR_INVALID_ARG   # mode
    assert g(p, None, p, 4, 128, 64, 0, 0, None, 0, None) == bi.ERR_INVALID_ARG
    assert g(p, p, p + 8, 4, 128, 64, 0, 0, None, 0, None) == bi.ERR_INVALID_ARG
    # variant with an explicit split count and no workspace: refused, host-side
    assert g(p, p, p, 4, 128, 256, 1, 2, None, 0, None) == bi.ERR_WORKSPACE
    assert g(None, None, None, 0, 128, 64, 0, 0, None, 0, None) == bi.OK


def test_silu_mul_argument_checks(lib):
    p = 1 << 20
    f = lambda T, F, block, out=p: lib.bi_silu_mul(p, T, F, block, out, None)
    assert f(4, 256, 0) == bi.ERR_INVALID_ARG
    assert f(4, 256, 12) == bi.ERR_UNSUPPORTED          # block % 8
    assert f(4, 384, 256) == bi.ERR_UNSUPPORTED         # F % block
    assert f(4, 256, 128, out=p + 4) == bi.ERR_INVALID_ARG
    assert f(0, 256, 128) == bi.OK


def _decode(lib, **kw):
    p = 1 << 20
    a = dict(q=p, k=p, v=p, bt=p, kl=p, out=p, o32=None, B=2, Hq=4, Hkv=2, D=64, page=16,
             npages=8, maxblk=4, maxkv=64, S=64, scale=0.125, mode=0, vs=0, ws=p, wsb=1 << 20)
    a.update(kw)
    return lib.bi_attn_decode(a["q"], a["k"], a["v"], a["bt"], a["kl"], a["out"], a["o32"],
                              a["B"], a["Hq"], a["Hkv"], a["D"], a["page"], a["npages"],
                              a["maxblk"], a["maxkv"], a["S"], a["scale"], a["mode"], a["vs"],
                              a["ws"], a["wsb"], None)


def test_attention_argument_checks(lib):
    assert _decode(lib, D=96) == bi.ERR_UNSUPPORTED
    assert _decode(lib, Hq=6, Hkv=4) == bi.ERR_UNSUPPORTED
    assert _decode(lib, Hq=34, Hkv=2) == bi.ERR_UNSUPPORTED       # group of 17 > 16
    assert _decode(lib, page=32) == bi.ERR_UNSUPPORTED
    assert _decode(lib, S=100) == bi.ERR_UNSUPPORTED
    assert _decode(lib, q=None) == bi.ERR_INVALID_ARG
    assert _decode(lib, out=(1 << 20) + 4) == bi.ERR_INVALID_ARG
    assert _decode(lib, npages=0) == bi.ERR_INVALID_ARG
    assert _decode(lib, scale=0.0) == bi.ERR_INVALID_ARG          # the scale must be > 0
    assert _decode(lib, scale=-0.125) == bi.ERR_INVALID_ARG
    assert _decode(lib, scale=float("inf")) == bi.ERR_INVALID_ARG
    assert _decode(lib, scale=float("nan")) == bi.ERR_INVALID_ARG
    assert _decode(lib, B=0) == bi.OK


def _prefill(lib, **kw):
    p = 1 << 20
    a = dict(q=p, cu=p, st=p, k=p, v=p, bt=p, kl=p, out=p, o32=None, B=1, Hq=4, Hkv=2, D=64,
             page=16, npages=8, maxblk=4, tq=16, mq=16, maxkv=64, S=64, scale=0.125, mode=0,
             vs=0)
    a.update(kw)
    return lib.bi_attn_prefill_chunk(a["q"], a["cu"], a["st"], a["k"], a["v"], a["bt"], a["kl"],
                                     a["out"], a["o32"], a["B"], a["Hq"], a["Hkv"], a["D"],
                                     a["page"], a["npages"], a["maxblk"], a["tq"], a["mq"],
                                     a["maxkv"], a["S"], a["scale"], a["mode"], a["vs"], None, 0,
                                     None)


def test_prefill_argument_checks(lib):
    # every rejection happens on the host, before any device call
    assert _prefill(lib, D=96) == bi.ERR_UNSUPPORTED
    assert _prefill(lib, S=100) == bi.ERR_UNSUPPORTED
    assert _prefill(lib, q=None) == bi.ERR_INVALID_ARG
    assert _prefill(lib, tq=-1) == bi.ERR_INVALID_ARG
    assert _prefill(lib, mq=-1) == bi.ERR_INVALID_ARG
    assert _prefill(lib, scale=0.0) == bi.ERR_INVALID_ARG         # the scale must be > 0
    assert _prefill(lib, scale=float("nan")) == bi.ERR_INVALID_ARG
    assert _prefill(lib, cu=None) == bi.ERR_INVALID_ARG
    assert _prefill(lib, st=None) == bi.ERR_INVALID_ARG
    assert _prefill(lib, B=0) == bi.OK
    assert _prefill(lib, tq=0) == bi.OK                           # nothing to do


def test_binding_rejects_host_tensors():
    import torch
    x = torch.zeros(2, 64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        bi.bi_rmsnorm(x, x[0], x, 1e-6)


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "invariant_bi_rmsnorm_02_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "liboracle" not in text, f


@pytest.mark.parametrize("F", [128, 256, 1024, 14336])
def test_swiglu_interleave_inverts_the_oracle_layout(F):
    """bi.swiglu_interleave (the row order bi_gemm_swiglu's weight takes) and
    the oracle's reading of that layout (gate_up_halves) undo each other."""
    import numpy as np
    from oracle.decoder import gate_up_halves
    perm = bi.swiglu_interleave(F)
    assert sorted(perm.tolist()) == list(range(2 * F))
    x = np.random.default_rng(F).standard_normal((3, 2 * F))
    assert np.array_equal(gate_up_halves(x[:, perm]), x)


def test_swiglu_interleave_rejects_unaligned_widths():
    with pytest.raises(ValueError):
        bi.swiglu_interleave(192)
