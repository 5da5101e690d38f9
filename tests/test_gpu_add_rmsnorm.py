"""Residual add fused with RMSNorm on the GPU through the C ABI: the updated
residual stream equals the oracle's bf16 add bit for bit, the normalised
output matches the fp64 oracle, the fused kernel equals a separate bf16 add
followed by RMSNorm byte for byte, and both are batch-invariant."""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_02_gb300 as bi
import oracle
from invariant_bi_rmsnorm_02_gb300 import synth
from gpu_util import check_close, f64, same_bytes
from test_gpu_rmsnorm import rms_bound

pytestmark = pytest.mark.gpu
EPS = 1e-6


def bits(t):
    return t.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("M,H", [(1, 256), (8, 4096), (300, 4096), (5, 8), (7, 1000),
                                 (2, 12288), (33, 520)])
@pytest.mark.parametrize("mode", [bi.INVARIANT, bi.VARIANT])
def test_add_rmsnorm_matches_oracle(cuda, M, H, mode):
    x = synth.normal_bf16((M, H), 9200 + M + H)
    r = synth.normal_bf16((M, H), 9300 + M + H)
    w = synth.normal_bf16((H,), 9400 + H, std=0.1, mean=1.0)
    res = r.to(cuda)
    y = bi.add_rmsnorm(x.to(cuda), res, w.to(cuda), EPS, mode)
    assert bi.bi_check_device_errors() == bi.OK
    h_want, y_want = oracle.add_rmsnorm(x, r, w, EPS)
    assert np.array_equal(bits(res), h_want), "residual stream M=%d H=%d" % (M, H)
    g = f64(y)
    check_close(g, y_want, rms_bound(g, y_want, H), "add_rmsnorm M=%d H=%d mode=%d" % (M, H, mode))


@pytest.mark.parametrize("mode", [bi.INVARIANT, bi.VARIANT])
def test_add_rmsnorm_equals_add_then_rmsnorm(cuda, mode):
    # the fused step is exactly a bf16 add followed by bi_rmsnorm, both outputs
    for M, H in ((1, 4096), (64, 4096), (1000, 4096), (3, 12288), (9, 520)):
        x = synth.normal_bf16((M, H), 9500 + M, device=cuda)
        r = synth.normal_bf16((M, H), 9501 + M, device=cuda)
        w = synth.normal_bf16((H,), 9502, std=0.1, mean=1.0, device=cuda)
        h = (x.float() + r.float()).to(torch.bfloat16)
        y_sep, y32_sep = bi.rmsnorm(h, w, EPS, mode, want_f32=True)
        res = r.clone()
        y, y32 = bi.add_rmsnorm(x, res, w, EPS, mode, want_f32=True)
        assert same_bytes(res, h), (M, H)
        assert same_bytes(y, y_sep) and same_bytes(y32, y32_sep), (M, H)


def test_add_rmsnorm_batch_invariance(cuda):
    H = 4096
    x = synth.normal_bf16((512, H), 9600, device=cuda)
    r = synth.normal_bf16((512, H), 9601, device=cuda)
    w = synth.normal_bf16((H,), 9602, std=0.1, mean=1.0, device=cuda)
    res_full = r.clone()
    y_full, y32_full = bi.add_rmsnorm(x, res_full, w, EPS, want_f32=True)
    for M in list(range(1, 33)) + [100, 255, 256, 511]:
        res = r[:M].clone()
        y, y32 = bi.add_rmsnorm(x[:M].contiguous(), res, w, EPS, want_f32=True)
        assert same_bytes(y, y_full[:M]) and same_bytes(y32, y32_full[:M]), M
        assert same_bytes(res, res_full[:M]), M
    perm = torch.randperm(512, generator=torch.Generator().manual_seed(5)).to(cuda)
    res = r[perm].contiguous()
    y = bi.add_rmsnorm(x[perm].contiguous(), res, w, EPS)
    assert same_bytes(y, y_full[perm]) and same_bytes(res, res_full[perm])
    # the fused kernel's rows equal the plain invariant RMSNorm of the sum
    assert same_bytes(bi.rmsnorm(res_full, w, EPS), y_full)


def test_add_rmsnorm_input_untouched_and_residual_in_place(cuda):
    H = 2048
    x = synth.normal_bf16((16, H), 9700, device=cuda)
    r = synth.normal_bf16((16, H), 9701, device=cuda)
    w = torch.ones(H, dtype=torch.bfloat16, device=cuda)
    x0, res = x.clone(), r.clone()
    ptr = res.data_ptr()
    bi.add_rmsnorm(x, res, w, EPS)
    assert same_bytes(x, x0)
    assert res.data_ptr() == ptr
    # x = -residual: the stream becomes +0 and the normalised row is 0
    res2 = (-x).contiguous()
    y = bi.add_rmsnorm(x, res2, w, EPS)
    assert (bits(res2) == 0).all() and (f64(y) == 0).all()


def test_add_rmsnorm_full_size_sampled(cuda):
    # the Llama-shaped workload at its largest batch: 8192 x 4096
    M, H = 8192, 4096
    x = synth.normal_bf16((M, H), 9800, device=cuda)
    r = synth.normal_bf16((M, H), 9801, device=cuda)
    w = synth.normal_bf16((H,), 9802, std=0.1, mean=1.0, device=cuda)
    res = r.clone()
    y = bi.add_rmsnorm(x, res, w, EPS)
    rows = np.array([0, 1, 127, 4096, 8191])
    h_want, y_want = oracle.add_rmsnorm(x[rows].cpu(), r[rows].cpu(), w.cpu(), EPS)
    assert np.array_equal(bits(res[rows]), h_want)
    g = f64(y[rows])
    check_close(g, y_want, rms_bound(g, y_want, H), "add_rmsnorm 8192x4096 sample")


def test_add_rmsnorm_empty_and_rejected_shapes(cuda):
    x = torch.empty(0, 4096, dtype=torch.bfloat16, device=cuda)
    assert bi.add_rmsnorm(x, x.clone(), torch.ones(4096, dtype=torch.bfloat16, device=cuda)).shape == (0, 4096)
    xo = torch.zeros(2, 12, dtype=torch.bfloat16, device=cuda)   # H not a multiple of 8
    with pytest.raises(bi.BiError):
        bi.add_rmsnorm(xo, xo.clone(), torch.ones(12, dtype=torch.bfloat16, device=cuda))
