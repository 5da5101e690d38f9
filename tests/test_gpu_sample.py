"""Next-token selection on the GPU through the C ABI: greedy argmax and seeded
Gumbel-max sampling against the fp64 oracle, ties, invariance to the batch
around a request, and the draw distribution."""
import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_02_gb300 as bi
import oracle
from invariant_bi_rmsnorm_02_gb300 import synth
from gpu_util import same_bytes

pytestmark = pytest.mark.gpu
VOCAB = 128256   # the Llama-3 vocabulary


def u64(vals, dev):
    """uint64 values as the int64 tensor whose bits the library reads."""
    a = np.asarray(vals, dtype=np.uint64).view(np.int64)
    return torch.from_numpy(a.copy()).to(dev)


def check_tokens(got, logits, T, seed, step):
    """got must be the oracle's token, or -- at temperature > 0 only -- a
    token whose exact score is within the fp32 error of both scores (a near
    tie the kernel's fp32 arithmetic may resolve either way).  Returns the
    number of near ties taken."""
    want, scores = oracle.sample(logits.cpu(), T, seed, step)
    got = got.cpu().numpy().astype(np.int64)
    ties = 0
    for b in np.nonzero(got != want)[0]:
        assert T[b] > 0, ("greedy row differs", b, got[b], want[b])
        z = logits[b].float().cpu().numpy().astype(np.float64)

        def err(v):
            # fp32 score z * (1/T) + G: the reciprocal, the product, two logf
            # (1 ulp each) and the sum, bounded with a factor 4 of margin
            s = scores[b, v]
            return 2.0 ** -21 * (abs(z[v] / T[b]) + abs(s - z[v] / T[b]) + abs(s) + 1.0)

        gap = scores[b, want[b]] - scores[b, got[b]]
        assert 0 <= gap <= err(want[b]) + err(got[b]), ("row", b, got[b], want[b], gap)
        ties += 1
    return ties


def test_sample_matches_oracle_full_vocab(cuda):
    B, V = 128, VOCAB
    logits = synth.normal_bf16((B, V), 9990, std=2.0, device=cuda)
    T = np.array([0.0, 0.6, 1.0, 1.7] * (B // 4), np.float32)
    g = np.random.default_rng(9991)
    seed = g.integers(0, 2 ** 63, B, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    step = g.integers(0, 5000, B, dtype=np.uint64)
    tok = bi.sample(logits, torch.from_numpy(T).to(cuda), u64(seed, cuda), u64(step, cuda))
    assert bi.bi_check_device_errors() == bi.OK
    assert check_tokens(tok, logits, T, seed, step) <= 2


@pytest.mark.parametrize("V", [1, 7, 8, 9, 1000, 4097, 32000])
def test_sample_shapes_match_oracle(cuda, V):
    B = 24
    logits = synth.normal_bf16((B, V), 10000 + V, device=cuda)
    T = np.array([0.0, 0.8, 1.3] * (B // 3), np.float32)
    seed = np.arange(B, dtype=np.uint64) * np.uint64(7919)
    step = np.arange(B, dtype=np.uint64) + np.uint64(V)
    tok = bi.sample(logits, torch.from_numpy(T).to(cuda), u64(seed, cuda), u64(step, cuda))
    assert check_tokens(tok, logits, T, seed, step) <= 1


def test_greedy_ties_signed_zero_and_special_values(cuda):
    V = 1000
    z = torch.full((7, V), -1.0)
    z[0, [17, 400, 999]] = 2.5                  # three-way tie: lowest index
    z[1, 3] = -0.0
    z[1, 5] = 0.0                               # -0 == +0: index 3
    z[2] = float("-inf")                        # every entry -inf: index 0
    z[3, 10] = float("nan")
    z[3, 11] = 7.0                              # a NaN counts as -inf
    z[4, V - 1] = 1.0                           # the last entry
    z[5] = float("-inf")
    z[5, 300] = float("nan")                    # NaN and -inf tie: lowest index
    z[5, 301:] = float("nan")
    z[5, :300] = float("nan")
    z[5, 299] = float("-inf")
    z[6] = float("nan")                         # every entry NaN: index 0
    logits = z.to(torch.bfloat16).to(cuda)
    T = torch.zeros(7, device=cuda)
    tok = bi.sample(logits, T, u64([1] * 7, cuda), u64([0] * 7, cuda))
    assert tok.cpu().tolist() == [17, 3, 0, 11, V - 1, 0, 0]
    # a negative or NaN temperature is greedy too
    T2 = torch.tensor([-1.0, float("nan"), 0.0, -0.0, -5.0, 0.0, -2.0], device=cuda)
    assert same_bytes(bi.sample(logits, T2, u64([9] * 7, cuda), u64([4] * 7, cuda)), tok)
    # the same rows at an odd 2-byte offset take the per-entry load path
    store = torch.empty(7 * V + 1, dtype=torch.bfloat16, device=cuda)
    shifted = store[1:].view(7, V)
    shifted.copy_(logits)
    assert same_bytes(bi.sample(shifted, T, u64([1] * 7, cuda), u64([0] * 7, cuda)), tok)


def test_sample_is_batch_invariant_and_repeatable(cuda):
    B, V = 256, VOCAB
    logits = synth.normal_bf16((B, V), 10100, device=cuda)
    T = torch.full((B,), 0.9, device=cuda)
    T[::5] = 0.0
    seed = u64(np.arange(B, dtype=np.uint64) * np.uint64(2654435761), cuda)
    step = u64(np.arange(B, dtype=np.uint64) % np.uint64(97), cuda)
    full = bi.sample(logits, T, seed, step)
    for _ in range(3):
        assert same_bytes(bi.sample(logits, T, seed, step), full)
    for b in (0, 1, 77, 255):
        one = bi.sample(logits[b:b + 1].contiguous(), T[b:b + 1].contiguous(),
                        seed[b:b + 1].contiguous(), step[b:b + 1].contiguous())
        assert int(one[0]) == int(full[b]), b
    perm = torch.randperm(B, generator=torch.Generator().manual_seed(11)).to(cuda)
    got = bi.sample(logits[perm].contiguous(), T[perm].contiguous(), seed[perm].contiguous(),
                    step[perm].contiguous())
    assert same_bytes(got, full[perm])
    # rows stored at an odd 2-byte offset take the scalar load path: same tokens
    store = torch.empty(B * V + 1, dtype=torch.bfloat16, device=cuda)
    shifted = store[1:].view(B, V)
    shifted.copy_(logits)
    assert shifted.data_ptr() % 16 != 0
    assert same_bytes(bi.sample(shifted, T, seed, step), full)
    # the seed and the step both move the draw
    other_seed = bi.sample(logits, T, u64(np.arange(B, dtype=np.uint64) + np.uint64(5), cuda),
                           step)
    other_step = bi.sample(logits, T, seed, u64(np.arange(B, dtype=np.uint64) + np.uint64(1000),
                                                   cuda))
    sampled = (T > 0).cpu()
    assert (other_seed.cpu() != full.cpu())[sampled].any()
    assert (other_step.cpu() != full.cpu())[sampled].any()
    # greedy rows ignore seed and step
    assert same_bytes(other_seed.cpu()[~sampled], full.cpu()[~sampled])


def test_gumbel_max_draws_follow_softmax_on_gpu(cuda):
    # one row of logits sampled at 60000 steps: the token frequencies follow
    # softmax(z / T), and every draw is the oracle's
    zvals = [0.0, 1.0, 2.0, -1.0, 1.0, 0.5]
    z = torch.tensor(zvals, dtype=torch.float32).to(torch.bfloat16)
    T, n = 0.8, 60000
    logits = z.repeat(n, 1).to(cuda)
    Tt = torch.full((n,), T, device=cuda)
    seed = np.full(n, 123456789, np.uint64)
    step = np.arange(n, dtype=np.uint64)
    tok = bi.sample(logits, Tt, u64(seed, cuda), u64(step, cuda))
    assert check_tokens(tok, logits, np.full(n, T, np.float32), seed, step) <= 3
    p = np.exp(np.array(zvals) / T)
    p /= p.sum()
    freq = np.bincount(tok.cpu().numpy(), minlength=6) / n
    assert np.all(np.abs(freq - p) < 5 * np.sqrt(p * (1 - p) / n)), (freq, p)


def test_sample_empty_and_rejected(cuda):
    e = torch.empty(0, 10, dtype=torch.bfloat16, device=cuda)
    z = torch.empty(0, device=cuda)
    i = torch.empty(0, dtype=torch.int64, device=cuda)
    assert bi.sample(e, z, i, i).shape == (0,)
    big = torch.zeros(65536, 8, dtype=torch.bfloat16, device=cuda)
    T = torch.zeros(65536, device=cuda)
    s = torch.zeros(65536, dtype=torch.int64, device=cuda)
    with pytest.raises(bi.BiError):
        bi.sample(big, T, s, s)
    assert bi.bi_check_device_errors() == bi.OK
