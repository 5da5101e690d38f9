"""bf16 GEMM (tcgen05) on the GPU through the C ABI: parity with the fp64
oracle, exact special cases, bitwise batch invariance over M, and split-K
(the batch-variant mode) as a negative control."""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_02_gb300 as bi
import oracle
from invariant_bi_rmsnorm_02_gb300 import synth
from gpu_util import check_close, f64, first_divergence, same_bytes

pytestmark = pytest.mark.gpu


def gemm_bound(A, W, r, rows=None):
    """The stated tolerance: 1e-2 relative per element, plus the textbook
    worst-case error of an fp32 sum of K products, K * 2^-24 * sum_k |a_k w_k|,
    which only matters where the sum cancels to near zero."""
    a = np.abs(f64(A) if rows is None else f64(A)[rows])
    w = np.abs(f64(W))
    K = a.shape[1]
    return 1e-2 * np.abs(r) + K * 2.0 ** -24 * (a @ w.T)


def rounding_agreement(g, r):
    """Fraction of outputs equal to the oracle rounded once to bf16."""
    rb = torch.from_numpy(r).to(torch.bfloat16).to(torch.float64).numpy()
    return float((g == rb).mean())


def run_parity(cuda, M, N, K, mode, seed, splits=0):
    A = synth.normal_bf16((M, K), seed)
    W = synth.normal_bf16((N, K), seed + 1, std=0.02)
    C = bi.gemm(A.to(cuda), W.to(cuda), mode, splits)
    assert bi.bi_check_device_errors() == bi.OK
    r = oracle.gemm(A, W)
    g = f64(C)
    check_close(g, r, gemm_bound(A, W, r), "gemm %dx%dx%d mode=%d" % (M, N, K, mode))
    agree = rounding_agreement(g, r)
    assert agree > 0.95, "only %.3f of outputs equal bf16(oracle)" % agree
    return C


@pytest.mark.parametrize("M,N,K", [(1, 512, 256), (8, 512, 256), (3, 6144, 512),
                                   (130, 768, 320), (257, 1024, 1024), (64, 264, 72),
                                   (129, 256, 64), (200, 520, 136),
                                   # small batches over wide weights: narrow tiles with a
                                   # partial last tile or 64 rows of A, and the wide
                                   # tiles a weight too wide for one wave of them takes
                                   (5, 4104, 256), (7, 6152, 256), (40, 9216, 512),
                                   (2, 14336, 256)])
def test_gemm_matches_oracle(cuda, M, N, K):
    run_parity(cuda, M, N, K, bi.INVARIANT, 3000 + M + N + K)


@pytest.mark.parametrize("M,N,K,splits", [(1, 512, 256, 0), (3, 6144, 512, 0),
                                          (16, 1024, 1024, 4), (130, 768, 320, 3)])
def test_gemm_variant_matches_oracle(cuda, M, N, K, splits):
    run_parity(cuda, M, N, K, bi.VARIANT, 3100 + M + N + K, splits)


def test_gemm_identity_weight_is_exact(cuda):
    A = synth.normal_bf16((300, 256), 3200, device=cuda)
    W = torch.eye(256, dtype=torch.bfloat16, device=cuda)
    assert same_bytes(bi.gemm(A, W), A)


def test_gemm_small_integers_are_exact(cuda):
    g = torch.Generator().manual_seed(5)
    A = torch.randint(-2, 3, (77, 1024), generator=g)
    W = torch.randint(-2, 3, (512, 1024), generator=g)
    C = bi.gemm(A.to(torch.bfloat16).to(cuda), W.to(torch.bfloat16).to(cuda))
    want = (A @ W.T)  # |sum| <= 4096, but bf16 holds integers up to 256 exactly
    small = want.abs() <= 256
    got = C.cpu().to(torch.float64)
    assert torch.equal(got[small], want[small].to(torch.float64))
    wb = want.to(torch.float64).to(torch.bfloat16).to(torch.float64)
    assert torch.equal(got, wb)   # integer sums are exact in fp32: one rounding to bf16


@pytest.mark.parametrize("N", [6144, 14336])
def test_gemm_full_size_sampled(cuda, N):
    M, K = 8192, 4096
    A = synth.normal_bf16((M, K), 3300, device=cuda)
    W = synth.normal_bf16((N, K), 3301, std=0.02, device=cuda)
    C = bi.gemm(A, W)
    rows = np.array([0, 1, 127, 128, 255, 4095, 4096, 8190, 8191])
    Ac, Wc = A.cpu(), W.cpu()
    r = oracle.gemm(Ac, Wc, rows=rows)
    g = f64(C[torch.from_numpy(rows).to(cuda)])
    check_close(g, r, gemm_bound(Ac, Wc, r, rows), "gemm 8192x%dx4096 sample" % N)
    assert rounding_agreement(g, r) > 0.95


def test_gemm_batch_invariance_over_m(cuda):
    # every row of C has the same bytes at every M (1..256, 1024, 8192), in any
    # position and beside any neighbours
    K, N = 4096, 6144
    A = synth.normal_bf16((8192, K), 3400, device=cuda)
    W = synth.normal_bf16((N, K), 3401, std=0.02, device=cuda)
    full = bi.gemm(A, W)
    for M in list(range(1, 257)) + [300, 1024, 4097]:
        C = bi.gemm(A[:M].contiguous(), W)
        assert same_bytes(C, full[:M]), (M, first_divergence(C, full[:M]))
    perm = torch.randperm(512, generator=torch.Generator().manual_seed(4)).to(cuda)
    assert same_bytes(bi.gemm(A[perm].contiguous(), W), full[perm])
    other = synth.normal_bf16((77, K), 3402, device=cuda)
    other[50] = A[3]
    assert same_bytes(bi.gemm(other, W)[50], full[3])


def test_gemm_last_round_rows_match_small_batches(cuda):
    # at 8192 rows the QKV projection's last round of 128 x 256 tiles (the
    # last rows in raster order) runs on a few SMs while the others are done:
    # every row there, and elsewhere, has the bytes of a small batch
    K, N = 4096, 6144
    A = synth.normal_bf16((8192, K), 3450, device=cuda)
    W = synth.normal_bf16((N, K), 3451, std=0.02, device=cuda)
    full = bi.gemm(A, W)
    assert bi.bi_check_device_errors() == bi.OK
    for r0 in (0, 4096, 7680, 7936):
        part = bi.gemm(A[r0:r0 + 256].contiguous(), W)
        assert same_bytes(part, full[r0:r0 + 256]), (r0, first_divergence(part, full[r0:r0 + 256]))
    # the same rows again at 8192, run to run
    assert same_bytes(bi.gemm(A, W), full)


def test_gemm_batch_invariance_mlp_up(cuda):
    K, N = 4096, 14336
    A = synth.normal_bf16((1024, K), 3500, device=cuda)
    W = synth.normal_bf16((N, K), 3501, std=0.02, device=cuda)
    full = bi.gemm(A, W)
    for M in (1, 3, 16, 64, 256):
        assert same_bytes(bi.gemm(A[:M].contiguous(), W), full[:M]), M


@pytest.mark.parametrize("N", [4096, 9216])
def test_gemm_batch_invariance_wide_weights(cuda, N):
    # small batches run the narrow 64-column tiles, a 1024-row batch 128 x
    # 256 ones: every row has the same bytes in both
    K = 4096
    A = synth.normal_bf16((1024, K), 3550 + N, device=cuda)
    W = synth.normal_bf16((N, K), 3551 + N, std=0.02, device=cuda)
    full = bi.gemm(A, W)
    for M in (1, 3, 16, 33, 64):
        assert same_bytes(bi.gemm(A[:M].contiguous(), W), full[:M]), M
    assert bi.bi_check_device_errors() == bi.OK


def test_gemm_run_to_run(cuda):
    A = synth.normal_bf16((1000, 4096), 3600, device=cuda)
    W = synth.normal_bf16((6144, 4096), 3601, std=0.02, device=cuda)
    ref = bi.gemm(A, W)
    for _ in range(10):
        assert same_bytes(bi.gemm(A, W), ref)


def test_gemm_split_k_is_not_batch_invariant(cuda):
    # negative control: split-K picks its slice count from M, so row bytes
    # move with the batch size; the harness must see it (65 to 128 rows: 24
    # tiles of 128 x 256, which the variant cuts into 8 slices of K)
    K, N = 4096, 6144
    A = synth.normal_bf16((1024, K), 3700, device=cuda)
    W = synth.normal_bf16((N, K), 3701, std=0.02, device=cuda)
    ref = bi.gemm(A, W, bi.VARIANT)          # M = 1024: no split
    differing_rows = 0
    for M in (65, 100, 128):
        C = bi.gemm(A[:M].contiguous(), W, bi.VARIANT)
        differing_rows += int((C.view(torch.int16) != ref[:M].view(torch.int16)).any(1).sum())
    assert differing_rows > 0
    inv = bi.gemm(A[:16].contiguous(), W, bi.INVARIANT)
    assert same_bytes(inv, bi.gemm(A, W, bi.INVARIANT)[:16])


def test_gemm_empty_batch(cuda):
    A = torch.empty(0, 256, dtype=torch.bfloat16, device=cuda)
    W = torch.zeros(512, 256, dtype=torch.bfloat16, device=cuda)
    assert bi.gemm(A, W).shape == (0, 512)
