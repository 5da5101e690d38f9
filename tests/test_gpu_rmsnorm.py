"""RMSNorm on the GPU through the C ABI: parity with the fp64 oracle, bitwise
batch invariance, and the batch-variant mode as a negative control."""
import math

import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_02_gb300 as bi
import oracle
from invariant_bi_rmsnorm_02_gb300 import synth
from gpu_util import bf16_half_ulp, check_close, f64, same_bytes

pytestmark = pytest.mark.gpu
EPS = 1e-6


def rms_bound(g, r, H):
    """Tolerance: the stated 1e-2 relative bound, and a tighter one derived from
    the arithmetic -- one bf16 rounding of the output plus the fp32 error of a
    sum of H squares and a few roundings (H + 8 units of 2^-24, relative)."""
    stated = 1e-2 * np.abs(r) + 1e-30
    derived = bf16_half_ulp(g) + np.abs(r) * (H + 8) * 2.0 ** -24
    return np.minimum(stated, derived) + 1e-30


@pytest.mark.parametrize("M,H", [(1, 256), (8, 256), (3, 4096), (300, 4096), (5, 8),
                                 (7, 1000), (2, 12288), (33, 520)])
@pytest.mark.parametrize("mode", [bi.INVARIANT, bi.VARIANT])
def test_rmsnorm_matches_oracle(cuda, M, H, mode):
    x = synth.normal_bf16((M, H), 2000 + M + H)
    w = synth.normal_bf16((H,), 2001 + H, std=0.1, mean=1.0)
    y = bi.rmsnorm(x.to(cuda), w.to(cuda), EPS, mode)
    assert bi.bi_check_device_errors() == bi.OK
    r = oracle.rmsnorm(x, w, EPS)
    g = f64(y)
    check_close(g, r, rms_bound(g, r, H), "rmsnorm M=%d H=%d mode=%d" % (M, H, mode))


def test_rmsnorm_full_size_sampled(cuda):
    # the Llama-shaped workload at its largest batch: 8192 x 4096
    M, H = 8192, 4096
    x = synth.normal_bf16((M, H), 2100, device=cuda)
    w = synth.normal_bf16((H,), 2101, std=0.1, mean=1.0, device=cuda)
    y = bi.rmsnorm(x, w, EPS)
    rows = np.array([0, 1, 127, 128, 4095, 4096, 8190, 8191])
    r = oracle.rmsnorm(x[rows].cpu(), w.cpu(), EPS)
    g = f64(y[rows])
    check_close(g, r, rms_bound(g, r, H), "rmsnorm 8192x4096 sample")


def test_rmsnorm_constant_row_and_zero_row(cuda):
    H = 4096
    x = torch.zeros(3, H, dtype=torch.bfloat16)
    x[0] = 0.5
    x[2] = -3.0
    w = torch.ones(H, dtype=torch.bfloat16)
    y = f64(bi.rmsnorm(x.to(cuda), w.to(cuda), EPS))
    assert (y[1] == 0).all()
    for i, c in ((0, 0.5), (2, -3.0)):
        want = c / math.sqrt(c * c + EPS)
        assert np.abs(y[i] - want).max() <= 2.0 ** -8 * abs(want)


def test_rmsnorm_batch_invariance_sweep(cuda):
    # every row's bytes are the same at every batch size 1..256, in any position
    H = 4096
    x = synth.normal_bf16((256, H), 2200, device=cuda)
    w = synth.normal_bf16((H,), 2201, std=0.1, mean=1.0, device=cuda)
    full = bi.rmsnorm(x, w, EPS)
    for M in range(1, 257):
        assert same_bytes(bi.rmsnorm(x[:M].contiguous(), w, EPS), full[:M]), M
    perm = torch.randperm(256, generator=torch.Generator().manual_seed(3)).to(cuda)
    assert same_bytes(bi.rmsnorm(x[perm].contiguous(), w, EPS), full[perm])
    # other neighbours: row 0 among fresh random rows
    other = synth.normal_bf16((100, H), 2202, device=cuda)
    other[37] = x[0]
    assert same_bytes(bi.rmsnorm(other, w, EPS)[37], full[0])
    # large batches too
    big = synth.normal_bf16((8192, H), 2203, device=cuda)
    big[:256] = x
    yb = bi.rmsnorm(big, w, EPS)
    assert same_bytes(yb[:256], full)
    for M in (1024, 3000, 8191):
        assert same_bytes(bi.rmsnorm(big[:M].contiguous(), w, EPS), yb[:M])


def test_rmsnorm_run_to_run(cuda):
    x = synth.normal_bf16((64, 4096), 2300, device=cuda)
    w = synth.normal_bf16((4096,), 2301, device=cuda)
    ref = bi.rmsnorm(x, w, EPS)
    for _ in range(10):
        assert same_bytes(bi.rmsnorm(x, w, EPS), ref)


def worked_example_rows(n, H=4096):
    """The crafted rows of the worked RMSNorm example: one coordinate with
    square 1, the rest with square ~3e-8 (plus a small per-row jitter)."""
    x = torch.full((n, H), math.sqrt(3e-8), dtype=torch.float32)
    x[:, 0] = 1.0
    x[:, 1:] *= 1 + 0.01 * torch.arange(n, dtype=torch.float32)[:, None] / n
    return x.to(torch.bfloat16)


def test_rmsnorm_variant_is_not_batch_invariant(cuda):
    # negative control: the split-row variant reduces a row in 32 chunks at
    # M = 1 and in one block at M = 1024.  The two orders round the fp32 sum
    # of squares differently in a good share of rows; that shows in the fp32
    # output (y_f32) and only rarely survives the bf16 rounding, since a
    # bf16 square has at most 16 significant bits.  The invariant kernel's
    # bytes never move, in either output.
    H, R = 4096, 256
    x = synth.normal_bf16((R, H), 2400, device=cuda)
    w = torch.ones(H, dtype=torch.bfloat16, device=cuda)
    big = torch.cat([x, synth.normal_bf16((1024 - R, H), 2401, device=cuda)])
    inv_ref, inv_ref32 = bi.rmsnorm(big, w, EPS, bi.INVARIANT, want_f32=True)
    var_ref, var_ref32 = bi.rmsnorm(big, w, EPS, bi.VARIANT, want_f32=True)  # no split
    differing = 0
    for i in range(R):
        row = x[i:i + 1].contiguous()
        yi, yi32 = bi.rmsnorm(row, w, EPS, bi.INVARIANT, want_f32=True)
        assert same_bytes(yi, inv_ref[i:i + 1]) and same_bytes(yi32, inv_ref32[i:i + 1]), i
        yv, yv32 = bi.rmsnorm(row, w, EPS, bi.VARIANT, want_f32=True)
        differing += int(not same_bytes(yv32, var_ref32[i:i + 1]))
    assert differing > 0, "variant mode unexpectedly batch-invariant"
    # the worked example's crafted rows stay within tolerance in both modes
    xc = worked_example_rows(8).to(cuda)
    r = oracle.rmsnorm(xc.cpu(), w.cpu(), EPS)
    for mode in (bi.INVARIANT, bi.VARIANT):
        g = f64(bi.rmsnorm(xc, w, EPS, mode))
        check_close(g, r, rms_bound(g, r, H), "worked example mode=%d" % mode)


def test_rmsnorm_f32_output_is_the_unrounded_result(cuda):
    x = synth.normal_bf16((64, 4096), 2500, device=cuda)
    w = synth.normal_bf16((4096,), 2501, std=0.1, mean=1.0, device=cuda)
    for M, mode in ((64, bi.INVARIANT), (1, bi.VARIANT), (64, bi.VARIANT)):
        y, y32 = bi.rmsnorm(x[:M].contiguous(), w, EPS, mode, want_f32=True)
        assert same_bytes(y, y32.to(torch.bfloat16))
        assert same_bytes(bi.rmsnorm(x[:M].contiguous(), w, EPS, mode), y)


def test_rmsnorm_empty_batch(cuda):
    x = torch.empty(0, 4096, dtype=torch.bfloat16, device=cuda)
    w = torch.ones(4096, dtype=torch.bfloat16, device=cuda)
    assert bi.rmsnorm(x, w).shape == (0, 4096)


@pytest.mark.parametrize("H", [256, 4096])
@pytest.mark.parametrize("mode", [bi.INVARIANT, bi.VARIANT])
def test_rmsnorm_exact_row_is_bit_exact(cuda, H, mode):
    # entries +-1/2, +-1, +-2 in counts 4:3:1 have mean square exactly 1: every
    # partial sum of squares is a multiple of 1/4 (exact in fp32), rsqrt(1) = 1
    # and each output is a weight times a power of two, so with eps = 0 the
    # kernel's result is the exact value, bit for bit, in any reduction order
    n_half, n_one, n_two = H // 2, 3 * H // 8, H // 8
    mags = np.concatenate([np.full(n_half, 0.5), np.full(n_one, 1.0), np.full(n_two, 2.0)])
    g = np.random.default_rng(H + 17 * mode)
    rows = []
    for _ in range(6):
        rows.append(g.permutation(mags) * g.choice([-1.0, 1.0], H))
    x = torch.tensor(np.stack(rows), dtype=torch.float32).to(torch.bfloat16)
    assert float((x.double() ** 2).mean(dim=1).max()) == 1.0
    w = synth.normal_bf16((H,), 2600 + H, std=0.1, mean=1.0)
    y = bi.rmsnorm(x.to(cuda), w.to(cuda), 0.0, mode)
    want = torch.from_numpy(oracle.rmsnorm(x, w, 0.0)).to(torch.bfloat16)
    assert same_bytes(y.cpu(), want)
    assert same_bytes(want.float(), (x.float() * w.float()).to(torch.bfloat16).float())
