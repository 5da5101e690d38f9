"""The gate/up projection with the SwiGLU product in the GEMM epilogue
(bi_gemm_swiglu) on the GPU: the same bytes as the GEMM followed by the
standalone SwiGLU kernel, in both modes; parity with the fp64 oracle; bitwise
batch invariance over M."""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_02_gb300 as bi
import oracle
from invariant_bi_rmsnorm_02_gb300 import synth
from oracle.decoder import gate_up_halves, to_bf16
from gpu_util import check_close, f64, first_divergence, same_bytes

pytestmark = pytest.mark.gpu


def unfused(A, W, mode, splits=0):
    """bi_gemm into [M, 2F], then bi_silu_mul on the blocked layout, and on
    the columns put in gate-then-up order: the two-kernel forms of the fused
    call (they must agree)."""
    F = W.shape[0] // 2
    C = bi.gemm(A, W, mode, splits)
    perm = torch.from_numpy(bi.swiglu_interleave(F)).long().to(C.device)
    halves = torch.empty_like(C)
    halves[:, perm] = C
    blocked = bi.silu_mul(C, block=128)
    assert same_bytes(blocked, bi.silu_mul(halves))
    return blocked


@pytest.mark.parametrize("M,F,K", [(1, 128, 64), (3, 384, 256), (130, 256, 200),
                                   (257, 1024, 512), (64, 3584, 4096)])
@pytest.mark.parametrize("mode,splits", [(bi.INVARIANT, 0), (bi.VARIANT, 0), (bi.VARIANT, 3)])
def test_gemm_swiglu_equals_gemm_then_silu(cuda, M, F, K, mode, splits):
    A = synth.normal_bf16((M, K), 5000 + M + F, device=cuda)
    W = synth.normal_bf16((2 * F, K), 5001 + K, std=0.05, device=cuda)
    got = bi.gemm_swiglu(A, W, mode, splits)
    want = unfused(A, W, mode, splits)
    assert bi.bi_check_device_errors() == bi.OK
    assert same_bytes(got, want), first_divergence(got, want)


@pytest.mark.parametrize("M,F,K", [(5, 256, 256), (129, 512, 320)])
def test_gemm_swiglu_matches_oracle(cuda, M, F, K):
    A = synth.normal_bf16((M, K), 5100 + M)
    W = synth.normal_bf16((2 * F, K), 5101 + F, std=0.05)
    got = f64(bi.gemm_swiglu(A.to(cuda), W.to(cuda)))
    assert bi.bi_check_device_errors() == bi.OK
    gu = gate_up_halves(oracle.gemm(A, W))
    r = oracle.silu_mul(to_bf16(gu))
    g, u = gu[:, :F], gu[:, F:]
    sig = 1.0 / (1.0 + np.exp(-g))
    # g and u are rounded to bf16 from an fp32 sum on the GPU and from the
    # fp64 sum in the oracle: they differ by the fp32 sum's worst-case error
    # (K 2^-24 sum_k |a_k w_k|) plus one bf16 step (2^-7 relative); the
    # product moves by |d silu/dg| <= 1.1 times the first, |silu(g)| times
    # the second, and is rounded once more
    e = gate_up_halves(K * 2.0 ** -24 * (np.abs(f64(A)) @ np.abs(f64(W)).T))
    dg = 2.0 ** -7 * np.abs(g) + e[:, :F]
    du = 2.0 ** -7 * np.abs(u) + e[:, F:]
    bound = (1.1 * dg * (np.abs(u) + du) + np.abs(g * sig) * du + 2.0 ** -7 * np.abs(r)
             + 1e-30)
    check_close(got, r, bound, "gemm_swiglu %dx%dx%d" % (M, F, K))
    rb = torch.from_numpy(r).to(torch.bfloat16).double().numpy()
    agree = float((got == rb).mean())
    assert agree > 0.9, "only %.3f of outputs equal bf16(oracle)" % agree


def test_gemm_swiglu_rows_do_not_depend_on_the_batch(cuda):
    F, K = 512, 1024
    A = synth.normal_bf16((300, K), 5200, device=cuda)
    W = synth.normal_bf16((2 * F, K), 5201, std=0.05, device=cuda)
    full = bi.gemm_swiglu(A, W)
    for M in (1, 3, 17, 128, 129):
        part = bi.gemm_swiglu(A[:M].contiguous(), W)
        assert same_bytes(part, full[:M]), M
    idx = torch.tensor([299, 5, 130], device=cuda)
    assert same_bytes(bi.gemm_swiglu(A[idx].contiguous(), W), full[idx])
    assert bi.bi_check_device_errors() == bi.OK


def test_gemm_swiglu_rejects_unsupported_shapes(cuda):
    A = torch.zeros(4, 64, dtype=torch.bfloat16, device=cuda)
    W = torch.zeros(2 * 192, 64, dtype=torch.bfloat16, device=cuda)   # F = 192: not 128-aligned
    out = torch.zeros(4, 192, dtype=torch.bfloat16, device=cuda)
    with pytest.raises(bi.BiError) as e:
        bi.bi_gemm_swiglu(A, W, out)
    assert e.value.status == bi.ERR_UNSUPPORTED
    # variant mode, two slices of K = 256 (four k-blocks), no workspace
    Av = torch.zeros(4, 256, dtype=torch.bfloat16, device=cuda)
    Wv = torch.zeros(256, 256, dtype=torch.bfloat16, device=cuda)
    outv = torch.zeros(4, 128, dtype=torch.bfloat16, device=cuda)
    with pytest.raises(bi.BiError) as e:
        bi.bi_gemm_swiglu(Av, Wv, outv, bi.VARIANT, 2)
    assert e.value.status == bi.ERR_WORKSPACE
