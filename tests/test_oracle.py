"""Pins for the fp64 oracle: each test ties the oracle to something other
than itself -- numbers printed on the pages (tests/golden), closed forms,
invariants of the mathematics, special cases that reduce to a library routine,
and brute force on tiny inputs written independently here with math.fsum.
CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from invariant_bi_rmsnorm_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf(x):
    """python/numpy values -> bf16 tensor (exact when the values are bf16)."""
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float64).numpy()


# --------------------------------------------------------------------------
# RMSNorm
# --------------------------------------------------------------------------
def test_rmsnorm_hand_worked():
    # x = [3, 4]: mean of squares 12.5, root 3.5355339..., eps 0, w = 1
    y = oracle.rmsnorm(bf([[3.0, 4.0]]), bf([1.0, 1.0]), 0.0)
    assert y[0, 0] == pytest.approx(0.8485281374238571, abs=1e-15)
    assert y[0, 1] == pytest.approx(1.1313708498984762, abs=1e-15)
    # the weight multiplies element-wise: w = [2, -0.5]
    y = oracle.rmsnorm(bf([[3.0, 4.0]]), bf([2.0, -0.5]), 0.0)
    assert y[0, 0] == pytest.approx(1.6970562748477142, abs=1e-15)
    assert y[0, 1] == pytest.approx(-0.5656854249492381, abs=1e-15)


@pytest.mark.parametrize("c", [0.5, -3.0, 1e-3, 100.0])
def test_rmsnorm_constant_row_closed_form(c):
    # a constant row has mean square c^2: y = c / sqrt(c^2 + eps) * w
    H, eps = 4096, 1e-6
    w = synth.normal_bf16((H,), 7, std=0.1, mean=1.0)
    cb = float(bf([c])[0])
    y = oracle.rmsnorm(bf(np.full((1, H), c)), w, eps)
    expect = cb / math.sqrt(cb * cb + eps) * f64(w)
    np.testing.assert_allclose(y[0], expect, rtol=1e-14, atol=0)


def test_rmsnorm_unit_rms_and_scale_invariance():
    # with w = 1 and eps = 0 every output row has mean square exactly 1, and
    # scaling a row by a power of two leaves it unchanged
    x = synth.normal_bf16((5, 256), 11)
    one = torch.ones(256, dtype=torch.bfloat16)
    y = oracle.rmsnorm(x, one, 0.0)
    np.testing.assert_allclose((y ** 2).mean(axis=1), 1.0, rtol=1e-13)
    y2 = oracle.rmsnorm((x.float() * 8).to(torch.bfloat16), one, 0.0)
    np.testing.assert_allclose(y2, y, rtol=1e-14)


def test_rmsnorm_brute_force_fsum():
    rng = np.random.default_rng(3)
    for H in (1, 2, 3, 7, 16):
        x = bf(rng.standard_normal((4, H)))
        w = bf(rng.standard_normal(H))
        eps = 1e-6
        y = oracle.rmsnorm(x, w, eps)
        xs, ws = f64(x), f64(w)
        for i in range(4):
            inv = 1.0 / math.sqrt(math.fsum(v * v for v in xs[i]) / H + eps)
            for j in range(H):
                assert y[i, j] == pytest.approx(xs[i, j] * inv * ws[j], rel=1e-14, abs=1e-300)


def test_rmsnorm_worked_example_exact_total():
    # one coordinate with square 1.0, 4095 with square ~3e-8: the exact total
    # printed on the page is 1.00012285.  Our bf16 row can only approximate
    # sqrt(3e-8) to bf16's relative half-spacing (<= 2^-8), so the total may
    # move by at most 4095 * 3e-8 * 2 * 2^-8 ~ 9.6e-7.
    g = golden("rmsnorm_worked_example.json")
    H = g["H"]
    row = np.full((1, H), math.sqrt(g["small_square"]), dtype=np.float32)
    row[0, 0] = math.sqrt(g["large_square"])
    _, ms = oracle.rmsnorm(bf(row), bf(np.ones(H)), 1e-6, return_mean_sq=True)
    assert abs(ms[0] * H - g["exact_total"]) <= 1e-6


def test_rmsnorm_dropped_eps_or_mean_is_detected():
    # eps matters where the mean square is tiny: x = 1e-3 constant, eps 1e-6
    # gives 1e-3 / sqrt(1e-6 + 1e-6) = 0.70710678...
    H = 64
    xb = bf(np.full((1, H), 2.0 ** -10))
    v = 2.0 ** -10
    y = oracle.rmsnorm(xb, bf(np.ones(H)), v * v)
    np.testing.assert_allclose(y[0], 1 / math.sqrt(2.0), rtol=1e-15)


# --------------------------------------------------------------------------
# fp32 worked examples on the pages (pins the fp32 emulation the GPU tests
# use to explain order effects)
# --------------------------------------------------------------------------
def test_absorption_example():
    g = golden("absorption.json")
    one = np.float32(g["large"])
    small = np.float32(g["small"])
    acc = one
    for _ in range(g["count"]):
        acc = np.float32(acc + small)
    assert float(acc) == g["sequential_fp32"]
    s = np.float32(0)
    for _ in range(g["count"]):
        s = np.float32(s + small)
    first = np.float32(s + one)
    assert abs(float(first) - g["small_first_fp32"]) <= g["printed_digits_abs"]
    ulps = (float(first) - 1.0) / 2.0 ** -23
    assert abs(ulps - g["ulp_distance_approx"]) <= 1.0
    assert float(np.spacing(np.float32(1.0))) / 2 == pytest.approx(g["half_ulp_at_one"], rel=1e-2)


def _tree_f32(vals):
    vals = [np.float32(v) for v in vals]
    while len(vals) > 1:
        vals = [np.float32(vals[i] + vals[i + 1]) for i in range(0, len(vals), 2)]
    return vals[0]


def test_rmsnorm_worked_example_fp32_orders():
    g = golden("rmsnorm_worked_example.json")
    sq = [np.float32(g["large_square"])] + [np.float32(g["small_square"])] * (g["H"] - 1)
    acc = np.float32(0)
    for v in sq:                       # one block per row, sequential from index 1
        acc = np.float32(acc + v)
    assert abs(float(acc) - g["sequential_fp32_total"]) <= g["printed_digits_abs"]
    L = g["split_block_len"]
    blocks = []
    for b in range(g["split_blocks"]):
        chunk = sq[b * L:(b + 1) * L]
        if b == 0:                      # the 127 small values meet first
            blocks.append(np.float32(chunk[0] + _tree_f32(chunk[1:] + [np.float32(0)])))
        else:
            blocks.append(_tree_f32(chunk))
    assert abs(float(blocks[0]) - g["split_block0_fp32"]) <= g["printed_digits_abs"]
    assert float(blocks[1]) == pytest.approx(g["split_other_block_fp32"], rel=2e-3)
    total = _tree_f32(blocks)
    assert abs(float(total) - g["split_fp32_total"]) <= g["printed_digits_abs"]
    assert float(total) - float(acc) == pytest.approx(g["difference"], rel=1e-3)


# --------------------------------------------------------------------------
# GEMM
# --------------------------------------------------------------------------
def test_gemm_identity_weight():
    A = synth.normal_bf16((9, 64), 21)
    W = torch.eye(64, dtype=torch.bfloat16)
    np.testing.assert_array_equal(oracle.gemm(A, W), f64(A))


def test_gemm_small_integers_match_integer_matmul():
    rng = np.random.default_rng(5)
    A = rng.integers(-2, 3, size=(13, 40))
    W = rng.integers(-2, 3, size=(24, 40))
    C = oracle.gemm(bf(A), bf(W))
    np.testing.assert_array_equal(C, (A.astype(np.int64) @ W.T.astype(np.int64)).astype(np.float64))


def test_gemm_brute_force_nonsquare():
    # W is [N, K]: a transposed operand would read the wrong elements
    rng = np.random.default_rng(6)
    A = bf(rng.standard_normal((3, 7)))
    W = bf(rng.standard_normal((5, 7)))
    C = oracle.gemm(A, W)
    a, w = f64(A), f64(W)
    for i in range(3):
        for n in range(5):
            assert C[i, n] == pytest.approx(math.fsum(a[i, k] * w[n, k] for k in range(7)), rel=1e-14, abs=1e-14)


def test_gemm_rank_one_closed_form():
    a = bf(np.linspace(-2, 2, 6))
    b = bf(np.linspace(0.5, 3, 4))
    K = 96
    A = a[:, None].expand(6, K).contiguous()
    W = b[:, None].expand(4, K).contiguous()
    C = oracle.gemm(A, W)
    np.testing.assert_allclose(C, K * np.outer(f64(a), f64(b)), rtol=1e-15)


def test_gemm_row_sample_matches_full():
    A = synth.normal_bf16((17, 48), 31)
    W = synth.normal_bf16((20, 48), 32, std=0.02)
    full = oracle.gemm(A, W)
    rows = np.array([16, 0, 5])
    np.testing.assert_array_equal(oracle.gemm(A, W, rows=rows), full[rows])


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------
def _dense_cache(K, V, page=4):
    """K, V [L, Hkv, D] bf16 -> a paged cache with a reversed page order."""
    L, Hkv, D = K.shape
    npg = -(-L // page)
    kc = torch.zeros(npg, Hkv, page, D, dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    bt = torch.zeros(1, npg, dtype=torch.int32)
    for blk in range(npg):
        phys = npg - 1 - blk
        bt[0, blk] = phys
        n = min(page, L - blk * page)
        kc[phys, :, :n] = K[blk * page: blk * page + n].transpose(0, 1)
        vc[phys, :, :n] = V[blk * page: blk * page + n].transpose(0, 1)
    return kc, vc, bt


def _brute_attention(q, K, V, n, scale, G):
    """independent statement with math.exp / math.fsum, tiny inputs only"""
    qf, kf, vf = f64(q), f64(K), f64(V)
    Hq, D = qf.shape
    out = np.zeros((Hq, D))
    for h in range(Hq):
        s = [scale * math.fsum(qf[h, d] * kf[t, h // G, d] for d in range(D)) for t in range(n)]
        mx = max(s)
        e = [math.exp(v - mx) for v in s]
        den = math.fsum(e)
        for d in range(D):
            out[h, d] = math.fsum(e[t] * vf[t, h // G, d] for t in range(n)) / den
    return out


def test_attention_brute_force_decode_and_causal():
    Hq, Hkv, D, L = 4, 2, 8, 11
    q = synth.normal_bf16((L, Hq, D), 41)
    K = synth.normal_bf16((L, Hkv, D), 42)
    V = synth.normal_bf16((L, Hkv, D), 43)
    kc, vc, bt = _dense_cache(K, V)
    scale = 1 / math.sqrt(D)
    dec = oracle.decode_attention(q[-1:], kc, vc, bt, [L], scale)
    np.testing.assert_allclose(dec[0], _brute_attention(q[-1], K, V, L, scale, 2), rtol=1e-12, atol=1e-14)
    pre = oracle.prefill_attention(q, 0, np.arange(L), kc, vc, bt, scale)
    for p in range(L):
        np.testing.assert_allclose(pre[p], _brute_attention(q[p], K, V, p + 1, scale, 2),
                                   rtol=1e-12, atol=1e-14)


def test_attention_single_key_returns_v():
    q = synth.normal_bf16((1, 4, 64), 51)
    K = synth.normal_bf16((1, 2, 64), 52)
    V = synth.normal_bf16((1, 2, 64), 53)
    kc, vc, bt = _dense_cache(K, V, page=16)
    out = oracle.decode_attention(q, kc, vc, bt, [1], 0.125)
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], f64(V[0, h // 2]))


def test_attention_identical_keys_gives_mean_of_v():
    L, D = 37, 64
    k = synth.normal_bf16((1, 1, D), 61)
    K = k.expand(L, 1, D).contiguous()
    V = synth.normal_bf16((L, 1, D), 62)
    q = synth.normal_bf16((1, 1, D), 63)
    kc, vc, bt = _dense_cache(K, V, page=16)
    out = oracle.decode_attention(q, kc, vc, bt, [L], 1 / 8)
    np.testing.assert_allclose(out[0, 0], f64(V[:, 0]).mean(axis=0), rtol=0, atol=1e-14)


def test_attention_dominant_key_selects_its_value():
    L, D = 20, 64
    K = torch.zeros(L, 1, D, dtype=torch.bfloat16)
    for t in range(L):
        K[t, 0, t] = 1.0
    V = synth.normal_bf16((L, 1, D), 71)
    q = torch.zeros(1, 1, D, dtype=torch.bfloat16)
    q[0, 0, 13] = 1024.0          # score gap 1024/8 = 128 -> weight e^-128 elsewhere
    kc, vc, bt = _dense_cache(K, V, page=16)
    out = oracle.decode_attention(q, kc, vc, bt, [L], 1 / 8)
    np.testing.assert_allclose(out[0, 0], f64(V[13, 0]), rtol=0, atol=1e-40)


def test_attention_gqa_head_mapping():
    Hq, Hkv, D, L = 8, 2, 16, 9
    K = synth.normal_bf16((L, Hkv, D), 81)
    V = torch.empty(L, Hkv, D, dtype=torch.bfloat16)
    for g in range(Hkv):
        V[:, g] = float(g + 1)
    q = synth.normal_bf16((1, Hq, D), 82)
    kc, vc, bt = _dense_cache(K, V)
    out = oracle.decode_attention(q, kc, vc, bt, [L], 0.25)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, h], h // (Hq // Hkv) + 1.0, rtol=1e-15)


def test_attention_independent_of_physical_page_order():
    kv = synth.paged_kv([37, 5, 64], 2, 32, 16, seed=91)
    q = synth.normal_bf16((3, 4, 32), 92)
    out = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.kv_lens, 0.2)
    perm = torch.randperm(kv.num_pages, generator=torch.Generator().manual_seed(5))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(kv.num_pages)
    kc2, vc2 = kv.k_cache[perm], kv.v_cache[perm]
    bt2 = inv[kv.block_table.long()].to(torch.int32)
    out2 = oracle.decode_attention(q, kc2, vc2, bt2, kv.kv_lens, 0.2)
    np.testing.assert_array_equal(out, out2)


@pytest.mark.parametrize("plan", [("size", 1), ("size", 3), ("size", 16), ("size", 64),
                                  ("size", 256), ("count", 1), ("count", 4), ("count", 7)])
def test_split_merge_equals_full_softmax(plan):
    # the log-sum-exp merge of any split plan is an exact rearrangement
    kv = synth.paged_kv([300, 1, 17, 64, 129], 2, 16, 16, seed=101)
    q = synth.normal_bf16((5, 4, 16), 102)
    full = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.kv_lens, 0.25)
    kind, val = plan
    split = oracle.attention(q, np.arange(5), kv.kv_lens, kv.k_cache, kv.v_cache, kv.block_table,
                             0.25, split_size=val if kind == "size" else 0,
                             split_count=val if kind == "count" else 0)
    np.testing.assert_allclose(split, full, rtol=1e-12, atol=1e-13)


def test_split_plans_match_pages():
    g = golden("split_plan.json")
    for c in g["fixed_size"]:
        st = oracle.split_starts_fixed_size(c["L"], c["S"])
        assert list(np.diff(st)) == c["sizes"]
    for c in g["fixed_count"]:
        st = oracle.split_starts_fixed_count(c["L"], c["count"])
        assert list(np.diff(st)) == c["sizes"]

    def chunk_start(st, k):
        return max(s for s in st[:-1] if s <= k)

    for L, start in g["key_index_300"]["fixed_size_chunk_start"].items():
        assert chunk_start(oracle.split_starts_fixed_size(int(L), 256), 300) == start
    for L, start in g["key_index_300"]["fixed_count_chunk_start"].items():
        assert chunk_start(oracle.split_starts_fixed_count(int(L), 4), 300) == start


def test_block_count_example():
    g = golden("block_count.json")
    nblk = lambda n: len(oracle.split_starts_fixed_size(n, g["block"])) - 1
    assert nblk(g["cached"]) == g["cached_blocks"]
    assert nblk(g["new"]) == g["new_blocks"]
    assert nblk(g["cached"]) + nblk(g["new"]) == g["separate_total_blocks"]
    assert nblk(g["cached"] + g["new"]) == g["together_blocks"]


def test_split_plan_boundaries_depend_only_on_absolute_index():
    # fixed size: the chunk holding key k is the same at every length > k
    for k in (0, 255, 256, 300, 1000):
        starts = {max(s for s in oracle.split_starts_fixed_size(L, 256)[:-1] if s <= k)
                  for L in range(k + 1, k + 600, 37)}
        assert starts == {k // 256 * 256}


def test_oracle_thread_count_does_not_change_results():
    A = synth.normal_bf16((33, 64), 111)
    W = synth.normal_bf16((40, 64), 112)
    np.testing.assert_array_equal(oracle.gemm(A, W, nthreads=1), oracle.gemm(A, W, nthreads=7))


# ------------------------------------------------- residual add (bf16 stream)
def _bf(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)


def _val(bits):
    return torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def test_oracle_add_bf16_zero_and_negation():
    x = synth.normal_bf16((3, 64), 9100)
    h0 = oracle.add_bf16(x, torch.zeros_like(x))              # x + 0 = x, bit for bit
    assert np.array_equal(h0, x.view(torch.int16).numpy().astype(np.uint16))
    hz = oracle.add_bf16(x, -x)                                 # x + (-x) = +0
    assert (hz == 0).all()


def test_oracle_add_bf16_exact_small_integers():
    g = torch.Generator().manual_seed(9101)
    a = torch.randint(-64, 65, (500,), generator=g)
    b = torch.randint(-64, 65, (500,), generator=g)
    h = _val(oracle.add_bf16(a.to(torch.bfloat16), b.to(torch.bfloat16)))
    assert np.array_equal(h, (a + b).to(torch.float64).numpy())  # |sum| <= 128: exact in bf16


def test_oracle_add_bf16_rounds_to_nearest_even():
    # bf16 has 8 significant bits: the spacing at 1 is 2^-7
    x = _bf([1.0, 1.0, 1.0, 1.0 + 2 ** -7, -1.0])
    r = _bf([2 ** -8, 3 * 2 ** -8, 2 ** -9, 2 ** -8, -(2 ** -8)])
    h = _val(oracle.add_bf16(x, r))
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: the even one (1) wins;
    # 1 + 3*2^-8 ties between 1 + 2^-7 and 1 + 2^-6: 1 + 2^-6 is even;
    # 1 + 2^-9 rounds down; (1 + 2^-7) + 2^-8 ties and goes up to 1 + 2^-6;
    # -1 - 2^-8 ties and keeps -1
    assert list(h) == [1.0, 1.0 + 2 ** -6, 1.0, 1.0 + 2 ** -6, -1.0]


def test_oracle_add_rmsnorm_is_rmsnorm_of_the_sum():
    x = synth.normal_bf16((5, 256), 9102)
    r = synth.normal_bf16((5, 256), 9103)
    w = synth.normal_bf16((256,), 9104, std=0.1, mean=1.0)
    h, y = oracle.add_rmsnorm(x, r, w, 1e-6)
    hv = _val(h)
    want = hv / np.sqrt((hv * hv).mean(axis=1, keepdims=True) + 1e-6) * f64(w)
    assert np.allclose(y, want, rtol=1e-12, atol=0)


# ------------------------------------------------------------ seeded sampling
U64 = (1 << 64) - 1


def _numpy_philox_words(counter, key, nwords):
    """numpy's Philox4x64-10 stream: it advances the counter before each
    block, so starting one below gives the block of `counter` first."""
    whole = sum(int(w) << (64 * i) for i, w in enumerate(counter)) - 1   # 256-bit, borrows
    whole &= (1 << 256) - 1
    c = np.array([(whole >> (64 * i)) & U64 for i in range(4)], dtype=np.uint64)
    bg = np.random.Philox(counter=c, key=np.array(key, dtype=np.uint64))
    return bg.random_raw(nwords)


@pytest.mark.parametrize("counter,key", [([0, 0, 0, 0], [0, 0]),
                                         ([5, 7, 0, 0], [0x1234567890ABCDEF, 42]),
                                         ([U64, 3, 9, 1], [0xFEDCBA9876543210, U64]),
                                         ([1 << 63, U64, 0, U64], [1, 2])])
def test_philox_matches_numpy(counter, key):
    got = oracle.philox4x64(counter, key)
    assert np.array_equal(got, _numpy_philox_words(counter, key, 4))


def test_philox_known_answer_zero_counter_and_key():
    # the published known-answer vector of Philox4x64-10 for an all-zero
    # counter and key (Random123 distribution)
    got = [int(v) for v in oracle.philox4x64([0, 0, 0, 0], [0, 0])]
    assert got == [0x16554D9ECA36314C, 0xDB20FE9D672D0FDC, 0xD7E772CEE186176B,
                   0x7E68B68AEC7BA23B]


@pytest.mark.parametrize("seed,step", [(0, 0), (2024, 17), (U64, 1 << 40)])
def test_sample_uniforms_are_the_philox_stream(seed, step):
    # entry v's uniform comes from the 32-bit word v of the little-endian
    # stream of blocks {0, step}, {1, step}, ... under key {seed, 0}
    n = 1000
    words = _numpy_philox_words([0, step, 0, 0], [seed, 0], n // 2 + 8)
    halves = words.astype("<u8").view("<u4")[:n].astype(np.float64)
    want = (np.floor(halves / 512) + 0.5) * 2.0 ** -23
    assert np.array_equal(oracle.sample_uniform(seed, step, 0, n), want)
    # an offset start reads the same stream
    assert np.array_equal(oracle.sample_uniform(seed, step, 333, 100), want[333:433])


def test_gumbel_noise_moments():
    # G = -log(-log u) is standard Gumbel: mean = Euler's constant,
    # variance = pi^2 / 6
    u = oracle.sample_uniform(99, 5, 0, 1 << 20)
    assert u.min() > 0 and u.max() < 1
    g = -np.log(-np.log(u))
    se = math.sqrt(math.pi ** 2 / 6 / u.size)
    assert abs(g.mean() - 0.5772156649015329) < 5 * se
    assert abs(g.var() - math.pi ** 2 / 6) < 0.02


def test_gumbel_max_draws_follow_softmax():
    # Gumbel-max: argmax(z / T + G) is distributed as softmax(z / T)
    z = bf([0.0, 1.0, 2.0, -1.0, 1.0])
    T, n = 0.75, 40000
    logits = z.repeat(n, 1)
    tok, _ = oracle.sample(logits, np.full(n, T, np.float32), np.full(n, 7, np.uint64),
                           np.arange(n, dtype=np.uint64))
    p = np.exp(f64(z) / T)
    p /= p.sum()
    freq = np.bincount(tok, minlength=5) / n
    assert np.all(np.abs(freq - p) < 5 * np.sqrt(p * (1 - p) / n)), (freq, p)


def test_sample_greedy_and_limits():
    z = bf([[0.5, 3.0, -1.0, 3.0, 2.0], [-2.0, -2.0, -2.0, -2.0, -2.0]])
    seed = np.array([1, 2], np.uint64)
    step = np.array([0, 0], np.uint64)
    # temperature 0 (and below): the plain argmax, lowest index on ties
    for T in (0.0, -1.0):
        tok, sc = oracle.sample(z, np.full(2, T, np.float32), seed, step)
        assert list(tok) == [1, 0]
        assert np.array_equal(sc, f64(z))
    # a tiny temperature: the logit gaps dwarf the noise
    tok, _ = oracle.sample(bf([[0.5, 3.0, -1.0, 2.0]]), np.float32([1e-3]), seed[:1], step[:1])
    assert list(tok) == [1]
    # the same (logits, seed, step) always gives the same token; the seed matters
    zz = synth.normal_bf16((64, 300), 9120)
    T = np.full(64, 1.0, np.float32)
    a, _ = oracle.sample(zz, T, np.arange(64, dtype=np.uint64), np.zeros(64, np.uint64))
    b, _ = oracle.sample(zz, T, np.arange(64, dtype=np.uint64), np.zeros(64, np.uint64))
    c, _ = oracle.sample(zz, T, np.arange(64, dtype=np.uint64) + 1000, np.zeros(64, np.uint64))
    assert np.array_equal(a, b) and not np.array_equal(a, c)


# ------------------------------------------------- element-wise decoder steps
def test_rope_position_zero_is_identity_and_pairs_keep_their_norm():
    x = synth.normal_bf16((5, 3, 64), 9130)
    pos = np.array([0, 1, 17, 4095, 100000])
    y = oracle.rope(x, pos, 500000.0)
    xv = f64(x)
    assert np.array_equal(y[0], xv[0])
    n_in = xv[..., :32] ** 2 + xv[..., 32:] ** 2
    n_out = y[..., :32] ** 2 + y[..., 32:] ** 2
    assert np.allclose(n_in, n_out, rtol=1e-12, atol=1e-12)


def test_rope_is_complex_multiplication_by_the_phase():
    # pairs (x_i, x_{i+D/2}) as complex numbers x_i + j x_{i+D/2}, multiplied
    # by exp(j pos theta^(-2i/D))
    D, theta = 16, 10000.0
    x = synth.normal_bf16((4, 2, D), 9131)
    pos = np.array([3, 10, 250, 7])
    xv = f64(x)
    z = xv[..., :D // 2] + 1j * xv[..., D // 2:]
    freq = np.array([theta ** (-2.0 * i / D) for i in range(D // 2)])
    w = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    y = oracle.rope(x, pos, theta)
    assert np.allclose(y[..., :D // 2], w.real, atol=1e-12)
    assert np.allclose(y[..., D // 2:], w.imag, atol=1e-12)


def test_rope_hand_worked_pair():
    # D = 4: pair 0 turns by pos radians, pair 1 by pos / sqrt(theta)
    x = bf([[[1.0, 2.0, 0.0, -1.0]]])
    y = oracle.rope(x, np.array([1]), 100.0)[0, 0]
    a0, a1 = 1.0, 0.1
    want = [1.0 * math.cos(a0) - 0.0 * math.sin(a0), 2.0 * math.cos(a1) + 1.0 * math.sin(a1),
            0.0 * math.cos(a0) + 1.0 * math.sin(a0), -1.0 * math.cos(a1) + 2.0 * math.sin(a1)]
    assert np.allclose(y, want, atol=1e-15)


def test_rope_scores_depend_on_relative_position_only():
    q = synth.normal_bf16((1, 1, 128), 9132)
    k = synth.normal_bf16((1, 1, 128), 9133)

    def score(m, n):
        return float((oracle.rope(q, [m], 500000.0) * oracle.rope(k, [n], 500000.0)).sum())

    for m, n, s in ((5, 2, 1000), (300, 299, 7), (0, 40, 8000)):
        assert abs(score(m, n) - score(m + s, n + s)) < 1e-9


def test_rope_qkv_splits_heads_in_order():
    Hq, Hkv, D = 4, 2, 16
    qkv = synth.normal_bf16((3, (Hq + 2 * Hkv) * D), 9134)
    pos = np.array([0, 0, 0])
    q, k, v = oracle.rope_qkv(qkv, pos, Hq, Hkv, D, 10000.0)
    flat = f64(qkv)
    assert np.array_equal(q.reshape(3, -1), flat[:, :Hq * D])
    assert np.array_equal(k.reshape(3, -1), flat[:, Hq * D:(Hq + Hkv) * D])
    assert np.array_equal(v.reshape(3, -1), flat[:, (Hq + Hkv) * D:])


def test_silu_mul_closed_forms():
    g = np.array([0.0, math.log(3.0), -math.log(3.0), 20.0, -20.0, 1.5])
    gu = bf(np.concatenate([g, np.ones(6)])[None, :])
    gb = f64(gu)[0, :6]
    y = oracle.silu_mul(gu)[0]
    assert y[0] == 0.0
    # sigmoid(ln 3) = 3/4, so silu(ln 3) = 0.75 ln 3; g holds ln 3 rounded to
    # bf16, and silu' < 1 near ln 3 bounds what that rounding moves
    assert abs(y[1] - 0.75 * math.log(3.0)) <= abs(gb[1] - math.log(3.0)) + 1e-15
    assert abs(y[2] - (y[1] - gb[1])) < 1e-15          # silu(-x) = silu(x) - x
    # silu(-x) = silu(x) - x
    xs = f64(synth.normal_bf16((1, 50), 9135))[0]
    pos = oracle.silu_mul(bf(np.concatenate([xs, np.ones(50)])[None, :]))[0]
    neg = oracle.silu_mul(bf(np.concatenate([-xs, np.ones(50)])[None, :]))[0]
    assert np.allclose(neg, pos - xs, atol=1e-14)
    assert abs(y[3] - gb[3]) < 1e-7 and abs(y[4]) < 1e-7
    # the up half multiplies
    u = f64(synth.normal_bf16((1, 6), 9136))[0]
    y2 = oracle.silu_mul(bf(np.concatenate([gb, u])[None, :]))[0]
    assert np.allclose(y2, y * u, rtol=1e-15, atol=0)


def test_gate_up_halves_reads_the_blocked_layout():
    from oracle.decoder import gate_up_halves
    # F = 256: two blocks of 128 features; columns 0-127 gate of features
    # 0-127, 128-255 their up, 256-383 gate of features 128-255, 384-511 up
    x = np.arange(512, dtype=np.float64)[None, :].repeat(2, axis=0)
    y = gate_up_halves(x)
    want = np.concatenate([np.arange(0, 128), np.arange(256, 384), np.arange(128, 256),
                           np.arange(384, 512)])
    assert np.array_equal(y[0], want) and np.array_equal(y[1], want)
    # one block: the layout is already gate-then-up
    z = np.arange(256, dtype=np.float64)[None, :]
    assert np.array_equal(gate_up_halves(z), z)


def test_gather_rows_copies_bits():
    src = synth.normal_bf16((10, 24), 9137)
    idx = np.array([3, 3, 0, 9])
    got = oracle.gather_rows(src, idx)
    bits = src.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, bits[[3, 3, 0, 9]])


# ------------------------------------------------------- decoder forward pass
def test_to_bf16_is_round_to_nearest_even():
    from oracle.decoder import to_bf16
    # float32 inputs: torch's float32 -> bfloat16 conversion rounds to nearest even
    x = torch.randn(100000, generator=torch.Generator().manual_seed(9140)) * 37.0
    want = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(to_bf16(x.double().numpy()), want)
    # from float64 it rounds once: 1 + 2^-8 + 2^-40 is above the tie
    assert to_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -40]))[0] == 0x3F81
    assert to_bf16(np.array([1 + 2.0 ** -8, 0.0, -3.0]))[0] == 0x3F80
    assert list(to_bf16(np.array([0.0, -3.0]))) == [0x0000, 0xC040]


def _tiny_weights(layers):
    from invariant_bi_rmsnorm_02_gb300.decoder import TINY, DecoderWeights
    import dataclasses
    cfg = dataclasses.replace(TINY, layers=layers)
    return cfg, DecoderWeights(cfg, 3, "cpu")


def test_decoder_without_layers_is_norm_then_lm_head():
    from oracle.decoder import forward_logits
    cfg, w = _tiny_weights(0)
    tok = [5, 0, 511, 5]
    got = forward_logits(w, cfg, tok)
    e = f64(w.embed)[tok]
    y = e / np.sqrt((e * e).mean(axis=1, keepdims=True) + cfg.eps)
    y = f64(torch.from_numpy(y).to(torch.bfloat16))
    assert np.allclose(got, y @ f64(w.lm_head).T, rtol=1e-12, atol=1e-12)
    assert np.array_equal(got[0], got[3])            # same token, no context


def test_decoder_is_causal():
    from oracle.decoder import forward_logits
    cfg, w = _tiny_weights(2)
    tok = list(np.random.default_rng(9141).integers(0, cfg.vocab, 37))
    full = forward_logits(w, cfg, tok)
    part = forward_logits(w, cfg, tok[:20])
    assert np.array_equal(full[:20], part)
    # and the last token's logits do depend on the first token
    tok2 = [(tok[0] + 1) % cfg.vocab] + tok[1:]
    assert not np.array_equal(forward_logits(w, cfg, tok2)[-1], full[-1])


# ------------------------------------------- one decoder layer, pinned by hand
# The decoder oracle's per-layer body (pre-norm attention block, then the
# SwiGLU MLP block, each added to the bf16 residual stream) is fixed below by
# cases that do not reuse its code: a pure-Python forward pass with math.fsum
# dot products and an independent bf16 rounding, and closed forms that follow
# when an output projection is zero.

def _bf16_round(v: float) -> float:
    """Nearest bf16 value of a Python float, ties to even (normal range):
    math.frexp gives v = m 2^e with 1/2 <= |m| < 1, and Python's round() of
    the exact m * 256 rounds half to even."""
    if v == 0.0 or not math.isfinite(v):
        return v
    m, e = math.frexp(v)
    return math.ldexp(round(m * 256.0), e - 8)


def _f32(v: float) -> float:
    import struct
    return struct.unpack("f", struct.pack("f", v))[0]


def _hand_forward(w, cfg, tokens):
    """Logits of a Llama-style pre-norm decoder whose activations are stored
    in bf16, with scalar Python loops (fsum dot products, math.exp/cos/sin);
    shares no code with oracle/decoder.py."""
    H, Hq, Hkv, D, F = cfg.hidden, cfg.heads, cfg.kv_heads, cfg.head_dim, cfg.ffn
    G = Hq // Hkv
    mat = lambda t: t.to(torch.float64).tolist()
    emb, lm, fn = mat(w.embed), mat(w.lm_head), mat(w.final_norm)

    def norm(x, g):
        r = math.sqrt(math.fsum(v * v for v in x) / len(x) + cfg.eps)
        return [_bf16_round(v / r * gi) for v, gi in zip(x, g)]

    def lin(x, W, rnd=True):
        out = [math.fsum(a * b for a, b in zip(x, row)) for row in W]
        return [_bf16_round(v) for v in out] if rnd else out

    def add(x, r):   # the residual add: one float32 rounding, then bf16
        return [_bf16_round(_f32(a + b)) for a, b in zip(x, r)]

    def rope(vec, p):
        half = D // 2
        out = list(vec)
        for i in range(half):
            ang = p * cfg.rope_theta ** (-2.0 * i / D)
            c, s = math.cos(ang), math.sin(ang)
            a, b = vec[i], vec[i + half]
            out[i], out[i + half] = a * c - b * s, b * c + a * s
        return [_bf16_round(v) for v in out]

    h = [list(emb[t]) for t in tokens]
    for layer in range(cfg.layers):
        wqkv, wo = mat(w.wqkv[layer]), mat(w.wo[layer])
        wgu, wd = mat(w.wgu[layer]), mat(w.wdown[layer])
        an, mn = mat(w.attn_norm[layer]), mat(w.mlp_norm[layer])
        qs, ks, vs = [], [], []
        for p, x in enumerate(h):
            qkv = lin(norm(x, an), wqkv)
            qs.append([rope(qkv[j * D:(j + 1) * D], p) for j in range(Hq)])
            ks.append([rope(qkv[(Hq + j) * D:(Hq + j + 1) * D], p) for j in range(Hkv)])
            vs.append([qkv[(Hq + Hkv + j) * D:(Hq + Hkv + j + 1) * D] for j in range(Hkv)])
        new_h = []
        for p, x in enumerate(h):
            att = []
            for j in range(Hq):
                kvh = j // G
                sc = [math.fsum(a * b for a, b in zip(qs[p][j], ks[t][kvh])) / math.sqrt(D)
                      for t in range(p + 1)]
                mx = max(sc)
                e = [math.exp(s - mx) for s in sc]
                z = math.fsum(e)
                att += [_bf16_round(math.fsum(e[t] * vs[t][kvh][d] for t in range(p + 1)) / z)
                        for d in range(D)]
            h1 = add(lin(att, wo), x)
            gu = lin(norm(h1, mn), wgu)
            act = []
            for f in range(F):
                blk, i = divmod(f, 128)
                g, u = gu[256 * blk + i], gu[256 * blk + 128 + i]
                act.append(_bf16_round(g / (1.0 + math.exp(-g)) * u))
            new_h.append(add(lin(act, wd), h1))
        h = new_h
    return np.array([lin(norm(x, fn), lm, rnd=False) for x in h])


def _small_decoder(layers, seed=5):
    import dataclasses
    from invariant_bi_rmsnorm_02_gb300.decoder import TINY, DecoderWeights
    # two gate/up blocks of 128 features, two query heads sharing one KV head
    cfg = dataclasses.replace(TINY, layers=layers, hidden=64, heads=2, kv_heads=1,
                              head_dim=32, ffn=256, vocab=40)
    w = DecoderWeights(cfg, seed, "cpu")
    # non-trivial norm weights, so that each norm's weight is read
    for k, lst in enumerate((w.attn_norm, w.mlp_norm)):
        for layer in range(layers):
            lst[layer] = synth.normal_bf16((cfg.hidden,), 9150 + 10 * layer + k, std=0.2,
                                           mean=1.0)
    w.final_norm = synth.normal_bf16((cfg.hidden,), 9149, std=0.2, mean=1.0)
    return cfg, w


@pytest.mark.parametrize("layers,tokens", [(1, [7]), (1, [3, 39, 3]), (2, [0, 17, 17, 5, 21])])
def test_decoder_layer_matches_a_hand_computed_forward_pass(layers, tokens):
    from oracle.decoder import forward_logits
    cfg, w = _small_decoder(layers)
    got = forward_logits(w, cfg, tokens)
    want = _hand_forward(w, cfg, tokens)
    # the two differ only in fp64 summation order (fsum is exactly rounded),
    # far below a bf16 step of any stored activation
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-12)


def test_decoder_hand_forward_detects_a_dropped_term():
    """The hand pass is sensitive to every branch: zeroing the O projection
    or the down projection, or one norm weight entry, moves the logits."""
    cfg, w = _small_decoder(1)
    tok = [3, 39, 3]
    base = _hand_forward(w, cfg, tok)
    for attr in ("wo", "wdown"):
        saved = getattr(w, attr)[0]
        getattr(w, attr)[0] = torch.zeros_like(saved)
        assert np.abs(_hand_forward(w, cfg, tok) - base).max() > 1e-4, attr
        getattr(w, attr)[0] = saved


def _zero_layers_closed_form(w, cfg, tok):
    e = f64(w.embed)[tok]
    y = e / np.sqrt((e * e).mean(axis=1, keepdims=True) + cfg.eps) * f64(w.final_norm)
    y = f64(torch.from_numpy(y).to(torch.bfloat16))
    return y @ f64(w.lm_head).T


def test_decoder_layers_with_zero_output_projections_are_the_identity():
    """W_o = 0 and W_down = 0: both branches add exact zeros to the residual
    stream, so every layer passes h through and the logits are those of the
    embedding's final norm and LM head alone."""
    from oracle.decoder import forward_logits
    cfg, w = _tiny_weights(2)
    for layer in range(cfg.layers):
        w.wo[layer] = torch.zeros_like(w.wo[layer])
        w.wdown[layer] = torch.zeros_like(w.wdown[layer])
    tok = list(np.random.default_rng(9143).integers(0, cfg.vocab, 21))
    got = forward_logits(w, cfg, tok)
    np.testing.assert_allclose(got, _zero_layers_closed_form(w, cfg, tok), rtol=1e-12,
                               atol=1e-12)


def test_decoder_attention_block_alone():
    """W_down = 0: one layer is h1 = bf16(h0 + bf16(bf16(attn) W_o^T)) with attn
    the causal attention of the rotated q, k (bf16) over the bf16 v; over 37
    tokens (three pages of the private cache)."""
    from oracle.decoder import forward_logits, to_bf16
    cfg, w = _tiny_weights(1)
    w.wdown[0] = torch.zeros_like(w.wdown[0])
    tok = list(np.random.default_rng(9144).integers(0, cfg.vocab, 37))
    T, Hq, Hkv, D = len(tok), cfg.heads, cfg.kv_heads, cfg.head_dim
    h0 = oracle.gather_rows(w.embed, tok)
    y = to_bf16(oracle.rmsnorm(h0, w.attn_norm[0], cfg.eps))
    q, k, v = oracle.rope_qkv(to_bf16(oracle.gemm(y, w.wqkv[0])), np.arange(T), Hq, Hkv, D,
                              cfg.rope_theta)
    # attention directly in float64 from the widened bf16 operands
    qf = f64(torch.from_numpy(to_bf16(q).view(np.int16)).view(torch.bfloat16))
    kf = f64(torch.from_numpy(to_bf16(k).view(np.int16)).view(torch.bfloat16))
    vf = f64(torch.from_numpy(to_bf16(v).view(np.int16)).view(torch.bfloat16))
    att = np.zeros((T, Hq, D))
    G = Hq // Hkv
    for hh in range(Hq):
        s = qf[:, hh] @ kf[:, hh // G].T / math.sqrt(D)
        s[np.triu_indices(T, 1)] = -np.inf
        p = np.exp(s - s.max(axis=1, keepdims=True))
        att[:, hh] = (p / p.sum(axis=1, keepdims=True)) @ vf[:, hh // G]
    o = to_bf16(oracle.gemm(to_bf16(att).reshape(T, Hq * D), w.wo[0]))
    h1 = oracle.add_bf16(o, h0)
    yf = to_bf16(oracle.rmsnorm(h1, w.final_norm, cfg.eps))
    want = oracle.gemm(yf, w.lm_head)
    np.testing.assert_allclose(forward_logits(w, cfg, tok), want, rtol=1e-9, atol=1e-12)


def test_decoder_mlp_block_alone():
    """W_o = 0: one layer is h1 = bf16(h0 + bf16(act W_down^T)) with act =
    bf16(silu(g) u), g and u the bf16 gate and up halves of the projection
    of RMSNorm(h0); attention contributes nothing."""
    from oracle.decoder import forward_logits, to_bf16
    cfg, w = _tiny_weights(1)
    w.wo[0] = torch.zeros_like(w.wo[0])
    tok = list(np.random.default_rng(9145).integers(0, cfg.vocab, 19))
    h0 = oracle.gather_rows(w.embed, tok)
    y = to_bf16(oracle.rmsnorm(h0, w.mlp_norm[0], cfg.eps))
    gu = f64(torch.from_numpy(to_bf16(oracle.gemm(y, w.wgu[0])).view(np.int16))
             .view(torch.bfloat16))
    F = cfg.ffn
    blocks = gu.reshape(len(tok), F // 128, 2, 128)
    g, u = blocks[:, :, 0].reshape(len(tok), F), blocks[:, :, 1].reshape(len(tok), F)
    act = to_bf16(g / (1.0 + np.exp(-g)) * u)
    h1 = oracle.add_bf16(to_bf16(oracle.gemm(act, w.wdown[0])), h0)
    yf = to_bf16(oracle.rmsnorm(h1, w.final_norm, cfg.eps))
    want = oracle.gemm(yf, w.lm_head)
    np.testing.assert_allclose(forward_logits(w, cfg, tok), want, rtol=1e-9, atol=1e-12)
