"""Element-wise decoder-layer steps on the GPU through the C ABI (row gather,
rotary embedding fused with the QKV split, SwiGLU product) against the fp64
oracle, with tolerances derived from their fp32 arithmetic."""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_02_gb300 as bi
import oracle
from invariant_bi_rmsnorm_02_gb300 import synth
from gpu_util import bf16_half_ulp, check_close, f64, same_bytes

pytestmark = pytest.mark.gpu


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def test_gather_rows_exact_and_bounds_checked(cuda):
    src = synth.normal_bf16((1000, 4096), 11000, device=cuda)
    idx = torch.tensor([5, 999, 0, 5, 512], dtype=torch.int32, device=cuda)
    got = bi.gather_rows(src, idx)
    assert bi.bi_check_device_errors() == bi.OK
    assert np.array_equal(bits(got), oracle.gather_rows(src.cpu(), idx.cpu().numpy()))
    bad = torch.tensor([1, 1000, -1], dtype=torch.int32, device=cuda)
    out = bi.gather_rows(src, bad)
    assert bi.bi_check_device_errors() == bi.ERR_DEVICE_BOUNDS
    assert same_bytes(out[0], src[1]) and (bits(out[1:]) == 0).all()


def rope_bound(g, x1, x2):
    # one bf16 rounding of the output, plus the fp32 rotation: sine and cosine
    # of the fp64-reduced angle (a few ulp), two products and a sum
    return bf16_half_ulp(g) + 2.0 ** -20 * (np.abs(x1) + np.abs(x2)) + 1e-30


@pytest.mark.parametrize("T,Hq,Hkv,D,theta", [(37, 32, 8, 128, 500000.0), (5, 4, 2, 64, 10000.0),
                                              (1, 8, 8, 16, 1e6)])
def test_rope_qkv_matches_oracle(cuda, T, Hq, Hkv, D, theta):
    qkv = synth.normal_bf16((T, (Hq + 2 * Hkv) * D), 11100 + D, device=cuda)
    pos = synth.uniform_int(T, 0, 131072, 11101 + T).to(torch.int32)
    pos[0] = 0
    q, k, v = bi.rope_qkv(qkv, pos.to(cuda), Hq, Hkv, D, theta)
    assert bi.bi_check_device_errors() == bi.OK
    rq, rk, rv = oracle.rope_qkv(qkv.cpu(), pos.numpy(), Hq, Hkv, D, theta)
    x = f64(qkv).reshape(T, Hq + 2 * Hkv, D)
    half = D // 2
    for got, ref, xin, name in ((q, rq, x[:, :Hq], "q"), (k, rk, x[:, Hq:Hq + Hkv], "k")):
        g = f64(got)
        # each output element's pair partner, for the bound
        x1 = np.concatenate([xin[..., :half], xin[..., half:]], axis=-1)
        x2 = np.concatenate([xin[..., half:], xin[..., :half]], axis=-1)
        check_close(g, ref, rope_bound(g, x1, x2), "rope %s T=%d D=%d" % (name, T, D))
    assert np.array_equal(f64(v), rv)
    assert np.array_equal(f64(q)[0], x[0, :Hq])          # position 0 is the identity


def test_rope_rows_are_independent_of_the_batch(cuda):
    Hq, Hkv, D = 32, 8, 128
    qkv = synth.normal_bf16((300, (Hq + 2 * Hkv) * D), 11200, device=cuda)
    pos = synth.uniform_int(300, 0, 8192, 11201).to(torch.int32).to(cuda)
    q, k, v = bi.rope_qkv(qkv, pos, Hq, Hkv, D)
    for a, b in ((0, 1), (17, 18), (299, 300), (100, 164)):
        q1, k1, v1 = bi.rope_qkv(qkv[a:b].contiguous(), pos[a:b].contiguous(), Hq, Hkv, D)
        assert same_bytes(q1, q[a:b]) and same_bytes(k1, k[a:b]) and same_bytes(v1, v[a:b])


@pytest.mark.parametrize("T,F", [(1, 14336), (5, 14336), (64, 8), (3, 1000)])
def test_silu_mul_matches_oracle(cuda, T, F):
    gu = synth.normal_bf16((T, 2 * F), 11300 + F, std=2.0, device=cuda)
    out = bi.silu_mul(gu)
    assert bi.bi_check_device_errors() == bi.OK
    r = oracle.silu_mul(gu.cpu())
    g = f64(out)
    # one bf16 rounding, plus expf (2 ulp), the add, the division and the
    # product in fp32
    check_close(g, r, bf16_half_ulp(g) + 2.0 ** -20 * np.abs(r) + 1e-30, "silu_mul")
    if T > 1:
        assert same_bytes(bi.silu_mul(gu[1:2].contiguous()), out[1:2])
    assert same_bytes(bi.silu_mul(gu, block=F), out)        # block = F: the halves layout


@pytest.mark.parametrize("T,F,block", [(3, 14336, 128), (70, 384, 128), (2, 64, 8),
                                       (5, 96, 32)])
def test_silu_mul_blocked_layout_matches_oracle(cuda, T, F, block):
    gu = synth.normal_bf16((T, 2 * F), 11400 + F + block, std=2.0, device=cuda)
    out = bi.silu_mul(gu, block=block)
    assert bi.bi_check_device_errors() == bi.OK
    # the oracle reads the stacked halves: gather block b's gate and up
    # columns (2 block b .. and block after) into them
    x = gu.cpu().view(torch.int16).numpy().view(np.uint16).reshape(T, F // block, 2, block)
    halves = np.concatenate([x[:, :, 0, :].reshape(T, F), x[:, :, 1, :].reshape(T, F)], axis=1)
    r = oracle.silu_mul(halves)
    g = f64(out)
    check_close(g, r, bf16_half_ulp(g) + 2.0 ** -20 * np.abs(r) + 1e-30, "silu_mul blocked")
    # the same elements through the halves layout: identical bytes
    h = torch.from_numpy(halves.view(np.int16)).view(torch.bfloat16).to(cuda)
    assert same_bytes(bi.silu_mul(h), out)
