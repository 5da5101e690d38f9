"""Paged attention on the GPU through the C ABI: decode and chunked prefill.
Parity with the fp64 oracle (2e-3 absolute on the fp32 result; the bf16
output is that result rounded once), bitwise invariance across batch size,
batch position, neighbours, KV growth, grid size and prefill chunking, and
the fixed split-count mode as a negative control."""

import numpy as np
import pytest
import torch

import invariant_bi_rmsnorm_02_gb300 as bi
import oracle
from invariant_bi_rmsnorm_02_gb300 import synth
from gpu_util import check_close, f64, first_divergence, same_bytes

pytestmark = pytest.mark.gpu
ATOL = 2e-3


def check_attn(out, out32, ref, what):
    """fp32 result within 2e-3 of the oracle; bf16 output = fp32 result rounded."""
    check_close(f64(out32), ref, np.full(ref.shape, ATOL), what)
    assert same_bytes(out, out32.to(torch.bfloat16)), what + ": bf16 output is not RN(fp32)"


def to_dev(kv, dev):
    return synth.PagedKV(kv.k_cache.to(dev), kv.v_cache.to(dev), kv.block_table.to(dev),
                         kv.kv_lens.to(dev), kv.page_size)


def decode(q, kv, max_kv_len, S, mode=bi.INVARIANT, splits=0, kv_lens=None, bt=None):
    return bi.attn_decode(q, kv.k_cache, kv.v_cache, kv.block_table if bt is None else bt,
                          kv.kv_lens if kv_lens is None else kv_lens, max_kv_len=max_kv_len,
                          split_size=S, mode=mode, variant_splits=splits, want_f32=True)


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("mode", [bi.INVARIANT, bi.VARIANT])
def test_decode_tiny_layer_matches_oracle(cuda, mode):
    c = synth.TINY
    lens = synth.uniform_int(c["B"], 1, c["max_len"], 4000).tolist()
    kv = synth.paged_kv(lens, c["Hkv"], c["D"], c["page"], 4001)
    q = synth.normal_bf16((c["B"], c["Hq"], c["D"]), 4002)
    out, out32 = decode(q.to(cuda), to_dev(kv, cuda), c["max_len"], c["split"], mode)
    assert bi.bi_check_device_errors() == bi.OK
    ref = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.kv_lens,
                                  c["D"] ** -0.5)
    check_attn(out, out32, ref, "decode tiny mode=%d" % mode)


@pytest.mark.parametrize("mode,S", [(bi.INVARIANT, 256), (bi.INVARIANT, 64), (bi.VARIANT, 256)])
def test_decode_gqa_d128_edges_match_oracle(cuda, mode, S):
    lens = [1, 2, 63, 64, 65, 255, 256, 257, 1000, 3001]
    kv = synth.paged_kv(lens, 8, 128, 16, 4100)
    q = synth.normal_bf16((len(lens), 32, 128), 4101)
    out, out32 = decode(q.to(cuda), to_dev(kv, cuda), 4096, S, mode)
    ref = oracle.decode_attention(q, kv.k_cache, kv.v_cache, kv.block_table, kv.kv_lens,
                                  128 ** -0.5)
    check_attn(out, out32, ref, "decode d128 mode=%d S=%d" % (mode, S))


def test_decode_single_key_returns_v_exactly(cuda):
    kv = synth.paged_kv([1, 1, 1], 2, 64, 16, 4200)
    q = synth.normal_bf16((3, 4, 64), 4201)
    out, _ = decode(q.to(cuda), to_dev(kv, cuda), 16, 64)
    for b in range(3):
        page = int(kv.block_table[b, 0])
        for h in range(4):
            assert torch.equal(out[b, h].cpu(), kv.v_cache[page, h // 2, 0])


def test_decode_identical_keys_give_mean_of_v(cuda):
    L, D = 777, 128
    kv = synth.paged_kv([L], 1, D, 16, 4300)
    kv.k_cache[:] = kv.k_cache[0, 0, 0]
    q = synth.normal_bf16((1, 4, D), 4301)
    _, out32 = decode(q.to(cuda), to_dev(kv, cuda), L, 256)
    V = torch.stack([kv.v_cache[int(kv.block_table[0, t // 16]), 0, t % 16] for t in range(L)])
    mean = f64(V).mean(axis=0)
    for h in range(4):
        check_close(f64(out32[0, h]), mean, np.full(D, ATOL), "identical keys")


def test_decode_empty_sequence_gives_zeros(cuda):
    kv = synth.paged_kv([0, 5], 2, 64, 16, 4400)
    kvd = to_dev(kv, cuda)
    q = synth.normal_bf16((2, 4, 64), 4401, device=cuda)
    for mode in (bi.INVARIANT, bi.VARIANT):
        out, out32 = decode(q, kvd, 64, 64, mode)
        assert (out32[0] == 0).all() and (out[0].float() == 0).all()
        assert out32[1].abs().sum() > 0


def test_decode_batch_invariance_tiny_layer(cuda):
    # request 0 of the tiny layer: the same bytes at every batch size 1..8,
    # in every position, beside any neighbours and at any grid size
    c = synth.TINY
    lens = synth.uniform_int(c["B"], 1, c["max_len"], 4500).tolist()
    kv = to_dev(synth.paged_kv(lens, c["Hkv"], c["D"], c["page"], 4501), cuda)
    q = synth.normal_bf16((c["B"], c["Hq"], c["D"]), 4502, device=cuda)
    ref, ref32 = decode(q, kv, c["max_len"], c["split"])
    for B in range(1, c["B"] + 1):
        out, out32 = decode(q[:B].contiguous(), kv, c["max_len"], c["split"],
                            kv_lens=kv.kv_lens[:B].contiguous(),
                            bt=kv.block_table[:B].contiguous())
        assert same_bytes(out, ref[:B]) and same_bytes(out32, ref32[:B]), B
    g = torch.Generator().manual_seed(1)
    for _ in range(5):
        perm = torch.randperm(c["B"], generator=g).to(cuda)
        out, _ = decode(q[perm].contiguous(), kv, c["max_len"], c["split"],
                        kv_lens=kv.kv_lens[perm].contiguous(),
                        bt=kv.block_table[perm].contiguous())
        assert same_bytes(out, ref[perm])
    for max_len in (int(kv.kv_lens.max()), 4096):
        out, _ = decode(q, kv, max_len, c["split"])
        assert same_bytes(out, ref)


def test_decode_kv_growth_gqa_full_size(cuda):
    # 64 requests, KV lengths log-uniform, grown one token per step for 512
    # steps; at every step the batched outputs equal, byte for byte, those of
    # one request alone, of a shuffled subset, and of a larger grid
    c = synth.GQA_DECODE
    B, Hq, Hkv, D, S, steps = c["B"], c["Hq"], c["Hkv"], c["D"], c["split"], c["steps"]
    lens0 = synth.loguniform_int(B, 1, c["max_len"] - steps, 4600).tolist()
    kv = to_dev(synth.paged_kv(lens0, Hkv, D, c["page"], 4601, reserve_tokens=steps), cuda)
    lens = kv.kv_lens.clone()
    seq = torch.arange(B, dtype=torch.int32, device=cuda)
    g = torch.Generator().manual_seed(7)
    sample_steps = {0, 255, 511}
    for step in range(steps):
        k_new = synth.normal_bf16((B, Hkv, D), 5000 + 2 * step, device=cuda)
        v_new = synth.normal_bf16((B, Hkv, D), 5001 + 2 * step, device=cuda)
        bi.kv_write(k_new, v_new, seq, lens, kv.k_cache, kv.v_cache, kv.block_table)
        lens = lens + 1
        q = synth.normal_bf16((B, Hq, D), 6000 + step, device=cuda)
        out, out32 = decode(q, kv, c["max_len"], S, kv_lens=lens)
        one = step % B
        o1, _ = decode(q[one:one + 1].contiguous(), kv, c["max_len"], S,
                       kv_lens=lens[one:one + 1].contiguous(),
                       bt=kv.block_table[one:one + 1].contiguous())
        assert same_bytes(o1[0], out[one]), ("alone", step, one)
        sub = torch.randperm(B, generator=g)[:5].to(cuda)
        o5, _ = decode(q[sub].contiguous(), kv, int(lens.max()), S,
                       kv_lens=lens[sub].contiguous(), bt=kv.block_table[sub].contiguous())
        assert same_bytes(o5, out[sub]), ("subset", step)
        if step in sample_steps:
            rows = [one, int(torch.argmax(lens)), int(torch.argmin(lens))]
            ref = oracle.decode_attention(q[rows].cpu(), kv.k_cache.cpu(), kv.v_cache.cpu(),
                                          kv.block_table[rows].cpu(), lens[rows].cpu(),
                                          D ** -0.5)
            check_attn(out[rows], out32[rows], ref, "growth step %d" % step)
    assert bi.bi_check_device_errors() == bi.OK


def test_decode_large_batch_plan_matches_small_batches(cuda):
    # above 128 sequences the split plan is built by its own kernel, below it
    # inside the split kernel: both give every request the same bytes, which
    # also match the oracle on a sample
    B, Hq, Hkv, D, S = 300, 32, 8, 128, 256
    lens = synth.loguniform_int(B, 1, 2048, 5150)
    lens[7] = 0
    kv = to_dev(synth.paged_kv(lens.tolist(), Hkv, D, 16, 5151), cuda)
    q = synth.normal_bf16((B, Hq, D), 5152, device=cuda)
    for mode in (bi.INVARIANT, bi.VARIANT):
        out, out32 = decode(q, kv, 2048, S, mode, splits=3)
        for b0 in range(0, B, 100):
            sl = slice(b0, b0 + 100)
            o, o32 = decode(q[sl].contiguous(), kv, 2048, S, mode, splits=3,
                            kv_lens=kv.kv_lens[sl].contiguous(),
                            bt=kv.block_table[sl].contiguous())
            if mode == bi.INVARIANT:
                assert same_bytes(o32, out32[sl]) and same_bytes(o, out[sl]), b0
            else:
                # the variant's chunk size follows the batch: a 100-sequence
                # slice is planned differently, and only matches the oracle
                r = [0, 37, 99]
                ref = oracle.decode_attention(q[sl][r].cpu(), kv.k_cache.cpu(), kv.v_cache.cpu(),
                                              kv.block_table[sl][r].cpu(),
                                              kv.kv_lens[sl][r].cpu(), D ** -0.5)
                check_attn(o[r], o32[r], ref, "decode slice %d variant" % b0)
        assert (out32[7] == 0).all()
        rows = [0, 7, 150, 299, int(torch.argmax(kv.kv_lens))]
        ref = oracle.decode_attention(q[rows].cpu(), kv.k_cache.cpu(), kv.v_cache.cpu(),
                                      kv.block_table[rows].cpu(), kv.kv_lens[rows].cpu(),
                                      D ** -0.5)
        check_attn(out[rows], out32[rows], ref, "decode B=300 mode=%d" % mode)
    assert bi.bi_check_device_errors() == bi.OK


# ----------------------------------------------------------------- prefill
def prefill(q, cu, starts, kv, kv_lens, max_q, max_kv, S, mode=bi.INVARIANT, splits=0):
    return bi.attn_prefill_chunk(q, cu, starts, kv.k_cache, kv.v_cache, kv.block_table,
                                 kv_lens, max_q_len=max_q, max_kv_len=max_kv, split_size=S,
                                 mode=mode, variant_splits=splits, want_f32=True)


@pytest.mark.parametrize("D,Hq,Hkv,S", [(64, 8, 2, 64), (128, 8, 2, 256), (128, 32, 8, 128),
                                        (64, 6, 6, 64), (128, 6, 2, 256)])
def test_prefill_matches_oracle(cuda, D, Hq, Hkv, S):
    # (the last case: 3 q heads per kv head, so a block holds 42 tokens and
    # two padding rows)
    # two sequences: a first chunk from position 0 and a later chunk
    starts, qlens = [0, 700], [300, 77]
    kvl = [s + n for s, n in zip(starts, qlens)]
    kv = synth.paged_kv(kvl, Hkv, D, 16, 4700 + D + Hq)
    q = synth.normal_bf16((sum(qlens), Hq, D), 4701)
    cu = torch.tensor([0, qlens[0], sum(qlens)], dtype=torch.int32)
    st = torch.tensor(starts, dtype=torch.int32)
    out, out32 = prefill(q.to(cuda), cu.to(cuda), st.to(cuda), to_dev(kv, cuda),
                         kv.kv_lens.to(cuda), max(qlens), max(kvl), S)
    assert bi.bi_check_device_errors() == bi.OK
    seqs = np.repeat([0, 1], qlens)
    pos = np.concatenate([np.arange(s, s + n) for s, n in zip(starts, qlens)])
    ref = oracle.prefill_attention(q, seqs, pos, kv.k_cache, kv.v_cache, kv.block_table,
                                   D ** -0.5)
    check_attn(out, out32, ref, "prefill D=%d Hq=%d Hkv=%d S=%d" % (D, Hq, Hkv, S))


def test_prefill_equals_decode_small(cuda):
    # each prefill position p equals a decode with L = p + 1, bit for bit
    L, Hq, Hkv, D, S = 333, 8, 2, 64, 64
    kv = to_dev(synth.paged_kv([L], Hkv, D, 16, 4800), cuda)
    q = synth.normal_bf16((L, Hq, D), 4801, device=cuda)
    cu = torch.tensor([0, L], dtype=torch.int32, device=cuda)
    st = torch.zeros(1, dtype=torch.int32, device=cuda)
    pre, pre32 = prefill(q, cu, st, kv, kv.kv_lens, L, L, S)
    bt = kv.block_table.expand(L, -1).contiguous()
    lens = torch.arange(1, L + 1, dtype=torch.int32, device=cuda)
    dec, dec32 = decode(q, kv, L, S, kv_lens=lens, bt=bt)
    assert same_bytes(pre32, dec32), first_divergence(pre32, dec32)
    assert same_bytes(pre, dec)


def test_prefill_equals_decode_pairs_across_splits(cuda):
    # S over pairs of key tiles with three tiles per split (split size 192:
    # every other pair straddles a split boundary), an odd tile count (300
    # keys: the last pair holds one tile) and a second chunk that starts
    # inside a tile: every position still equals a decode with L = p + 1
    L, Hq, Hkv, D, S = 300, 8, 2, 128, 192
    kv = to_dev(synth.paged_kv([L], Hkv, D, 16, 4850), cuda)
    q = synth.normal_bf16((L, Hq, D), 4851, device=cuda)
    pre = torch.empty_like(q)
    pre32 = torch.empty(q.shape, dtype=torch.float32, device=cuda)
    for s0, n in ((0, 137), (137, L - 137)):
        cu = torch.tensor([0, n], dtype=torch.int32, device=cuda)
        st = torch.tensor([s0], dtype=torch.int32, device=cuda)
        kl = torch.tensor([s0 + n], dtype=torch.int32, device=cuda)
        o, o32 = prefill(q[s0:s0 + n].contiguous(), cu, st, kv, kl, n, s0 + n, S)
        pre[s0:s0 + n], pre32[s0:s0 + n] = o, o32
    assert bi.bi_check_device_errors() == bi.OK
    bt = kv.block_table.expand(L, -1).contiguous()
    lens = torch.arange(1, L + 1, dtype=torch.int32, device=cuda)
    dec, dec32 = decode(q, kv, L, S, kv_lens=lens, bt=bt)
    assert same_bytes(pre32, dec32), first_divergence(pre32, dec32)
    assert same_bytes(pre, dec)


def test_prefill_chunked_equivalence_full_prompt(cuda):
    # one 8192-token prompt, 32/8 heads, D=128, split 256: chunks of 512,
    # 2048 and 8192, and token-by-token decode, give the same bytes at every
    # position
    c = synth.CHUNKED_PREFILL
    T, Hq, Hkv, D, S = c["T"], c["Hq"], c["Hkv"], c["D"], c["split"]
    kv = to_dev(synth.paged_kv([T], Hkv, D, c["page"], 4900), cuda)
    q = synth.normal_bf16((T, Hq, D), 4901, device=cuda)
    results = {}
    for chunk in c["chunks"]:
        out = torch.empty(T, Hq, D, dtype=torch.bfloat16, device=cuda)
        out32 = torch.empty(T, Hq, D, dtype=torch.float32, device=cuda)
        for s0 in range(0, T, chunk):
            n = min(chunk, T - s0)
            cu = torch.tensor([0, n], dtype=torch.int32, device=cuda)
            st = torch.tensor([s0], dtype=torch.int32, device=cuda)
            kl = torch.tensor([s0 + n], dtype=torch.int32, device=cuda)
            o, o32 = prefill(q[s0:s0 + n].contiguous(), cu, st, kv, kl, n, s0 + n, S)
            out[s0:s0 + n] = o
            out32[s0:s0 + n] = o32
        results[chunk] = (out, out32)
    # token by token: one decode call per position, L = p + 1
    dec = torch.empty(T, Hq, D, dtype=torch.bfloat16, device=cuda)
    dec32 = torch.empty(T, Hq, D, dtype=torch.float32, device=cuda)
    for p in range(T):
        kl = torch.tensor([p + 1], dtype=torch.int32, device=cuda)
        o, o32 = decode(q[p:p + 1].contiguous(), kv, p + 1, S, kv_lens=kl)
        dec[p] = o[0]
        dec32[p] = o32[0]
    base, base32 = results[c["chunks"][0]]
    for chunk in c["chunks"][1:]:
        o, o32 = results[chunk]
        assert same_bytes(o32, base32), (chunk, first_divergence(o32, base32))
        assert same_bytes(o, base), chunk
    assert same_bytes(dec32, base32), ("decode", first_divergence(dec32, base32))
    assert same_bytes(dec, base)
    assert bi.bi_check_device_errors() == bi.OK
    pos = np.array([0, 1, 63, 64, 255, 256, 257, 1000, 4095, 4096, 8191])
    ref = oracle.prefill_attention(q[pos].cpu(), 0, pos, kv.k_cache.cpu(), kv.v_cache.cpu(),
                                   kv.block_table.cpu(), D ** -0.5)
    idx = torch.from_numpy(pos).to(cuda)
    check_attn(base[idx], base32[idx], ref, "8192-token prompt sample")


@pytest.mark.parametrize("Hq,Hkv,D,T,chunk", [
    (32, 8, 128, 8192, 2048), (32, 8, 128, 32768, 4096),
    (24, 8, 64, 8192, 1664),    # 3 q heads per kv head: two padding rows per block
    (16, 2, 128, 8192, 2560),   # 8 q heads per kv head: 16 tokens per block
    (8, 8, 64, 8192, 4992),     # 1 q head per kv head: 128 tokens per block
])
def test_prefill_planned_order_matches_batch_and_decode(cuda, Hq, Hkv, D, T, chunk):
    # a single sequence's blocks launch in a host-planned order (the shapes
    # here are ones it is planned for); two copies of the sequence in one
    # call launch longest first: every row's bytes agree, and sampled
    # positions equal a decode with L = p + 1
    S = 256
    kv1 = synth.paged_kv([T], Hkv, D, 16, 5300 + chunk, device=cuda)
    q = synth.normal_bf16((chunk, Hq, D), 5301 + chunk, device=cuda)
    start = T - chunk
    one, one32 = prefill(q, torch.tensor([0, chunk], dtype=torch.int32, device=cuda),
                         torch.tensor([start], dtype=torch.int32, device=cuda), kv1,
                         kv1.kv_lens, chunk, T, S)
    bt2 = kv1.block_table.expand(2, -1).contiguous()
    kv2 = synth.PagedKV(kv1.k_cache, kv1.v_cache, bt2, kv1.kv_lens.expand(2).contiguous(),
                        kv1.page_size)
    two, two32 = prefill(torch.cat([q, q]), torch.tensor([0, chunk, 2 * chunk],
                                                         dtype=torch.int32, device=cuda),
                         torch.tensor([start, start], dtype=torch.int32, device=cuda), kv2,
                         kv2.kv_lens, chunk, T, S)
    assert bi.bi_check_device_errors() == bi.OK
    for half in (two32[:chunk], two32[chunk:]):
        assert same_bytes(half, one32), first_divergence(half, one32)
    assert same_bytes(two[:chunk], one) and same_bytes(two[chunk:], one)
    rows = torch.tensor([0, 1, 31, 32, chunk // 2, chunk - 33, chunk - 1], device=cuda)
    lens = (rows + start + 1).to(torch.int32)
    dec, dec32 = decode(q[rows].contiguous(), kv1, T, S, kv_lens=lens,
                        bt=kv1.block_table.expand(len(rows), -1).contiguous())
    assert same_bytes(dec32, one32[rows]), first_divergence(dec32, one32[rows])
    assert same_bytes(dec, one[rows])


def test_prefill_independent_of_neighbour_sequences(cuda):
    Hq, Hkv, D, S = 32, 8, 128, 256
    lens = [900, 1500, 64]
    kv = to_dev(synth.paged_kv(lens, Hkv, D, 16, 5100), cuda)
    starts, qlens = [600, 1000, 0], [300, 500, 64]
    q = synth.normal_bf16((sum(qlens), Hq, D), 5101, device=cuda)
    cu = torch.tensor([0, 300, 800, 864], dtype=torch.int32, device=cuda)
    st = torch.tensor(starts, dtype=torch.int32, device=cuda)
    kl = torch.tensor(lens, dtype=torch.int32, device=cuda)
    allo, _ = prefill(q, cu, st, kv, kl, 500, 1500, S)
    cu1 = torch.tensor([0, 500], dtype=torch.int32, device=cuda)
    alone, _ = bi.attn_prefill_chunk(q[300:800].contiguous(), cu1, st[1:2].contiguous(),
                                     kv.k_cache, kv.v_cache, kv.block_table[1:2].contiguous(),
                                     kl[1:2].contiguous(), max_q_len=500, max_kv_len=1500,
                                     split_size=S, want_f32=True)
    assert same_bytes(alone, allo[300:800])


# ------------------------------------------------------- negative controls
def test_decode_variant_plan_is_not_invariant(cuda):
    # the batch-variant plan sizes its chunks from the whole batch (with at
    # most 8 chunks a sequence, the longest sequence present sets them), so
    # a request's boundaries, and its bytes, change with the other requests
    lens = synth.loguniform_int(64, 300, 32000, 5200).tolist()
    kv = to_dev(synth.paged_kv(lens, 8, 128, 16, 5201), cuda)
    q = synth.normal_bf16((64, 32, 128), 5202, device=cuda)
    ref, _ = decode(q, kv, 32768, 256, bi.VARIANT, splits=8)
    differing = 0
    for B in (1, 2, 4, 16):
        out, _ = decode(q[:B].contiguous(), kv, 32768, 256, bi.VARIANT, splits=8,
                        kv_lens=kv.kv_lens[:B].contiguous(), bt=kv.block_table[:B].contiguous())
        differing += int((out.view(torch.int16) != ref[:B].view(torch.int16)).any(-1).any(-1).sum())
        inv, _ = decode(q[:B].contiguous(), kv, 32768, 256, bi.INVARIANT,
                        kv_lens=kv.kv_lens[:B].contiguous(), bt=kv.block_table[:B].contiguous())
        assert same_bytes(inv, decode(q, kv, 32768, 256)[0][:B])
    assert differing > 0


def test_prefill_variant_depends_on_chunking(cuda):
    T, Hq, Hkv, D = 2048, 8, 2, 128
    kv = to_dev(synth.paged_kv([T], Hkv, D, 16, 5300), cuda)
    q = synth.normal_bf16((T, Hq, D), 5301, device=cuda)
    outs = []
    for chunk in (512, 2048):
        out = torch.empty(T, Hq, D, dtype=torch.bfloat16, device=cuda)
        for s0 in range(0, T, chunk):
            cu = torch.tensor([0, chunk], dtype=torch.int32, device=cuda)
            st = torch.tensor([s0], dtype=torch.int32, device=cuda)
            kl = torch.tensor([s0 + chunk], dtype=torch.int32, device=cuda)
            out[s0:s0 + chunk] = prefill(q[s0:s0 + chunk].contiguous(), cu, st, kv, kl, chunk,
                                         s0 + chunk, 256, bi.VARIANT, 4)[0]
        outs.append(out)
    assert not same_bytes(outs[0], outs[1])


# ---------------------------------------------------------------- errors
def test_bad_page_id_is_reported_not_faulted(cuda):
    kv = synth.paged_kv([100, 50], 2, 64, 16, 5400)
    kvd = to_dev(kv, cuda)
    bt = kvd.block_table.clone()
    bt[1, 2] = kv.num_pages + 5      # outside the pool
    q = synth.normal_bf16((2, 4, 64), 5401, device=cuda)
    bad, _ = decode(q, kvd, 128, 64, bt=bt)
    assert bi.bi_check_device_errors() == bi.ERR_DEVICE_BOUNDS
    assert bi.bi_check_device_errors() == bi.OK          # cleared by the read
    out, _ = decode(q, kvd, 128, 64)                      # the context still works
    assert bi.bi_check_device_errors() == bi.OK
    # the offending sequence (one split of 64: written by the split kernel)
    # comes out as zeros, the other one is untouched
    assert not bool(bad[1].float().abs().sum())
    assert same_bytes(bad[0], out[0])
    # a bad page in the second split of a two-split sequence: zeros through
    # the merge's l = -1 mark
    bt2 = kvd.block_table.clone()
    bt2[0, 5] = -3                   # keys 80..95 of the 100
    bad2, _ = decode(q, kvd, 128, 64, bt=bt2)
    assert bi.bi_check_device_errors() == bi.ERR_DEVICE_BOUNDS
    assert not bool(bad2[0].float().abs().sum())
    assert same_bytes(bad2[1], out[1])
    lens = kvd.kv_lens.clone()
    lens[0] = 10 ** 6                                      # beyond the page table
    decode(q, kvd, 128, 64, kv_lens=lens)
    assert bi.bi_check_device_errors() == bi.ERR_DEVICE_BOUNDS


def test_prefill_bad_page_id_is_reported_not_faulted(cuda):
    # two prompts in one call; a page of the second lies outside the pool:
    # the blocks that would read it refuse before any copy and report it,
    # the first prompt's rows are the bytes of a clean call
    qlens = [100, 70]
    kv = to_dev(synth.paged_kv(qlens, 2, 64, 16, 5600), cuda)
    q = synth.normal_bf16((sum(qlens), 8, 64), 5601, device=cuda)
    cu = torch.tensor([0, qlens[0], sum(qlens)], dtype=torch.int32, device=cuda)
    st = torch.zeros(2, dtype=torch.int32, device=cuda)
    good, _ = prefill(q, cu, st, kv, kv.kv_lens, 100, 100, 64)
    assert bi.bi_check_device_errors() == bi.OK
    bt = kv.block_table.clone()
    bt[1, 2] = kv.k_cache.shape[0] + 7          # keys 32..47 of the second prompt
    bad = bi.attn_prefill_chunk(q, cu, st, kv.k_cache, kv.v_cache, bt, kv.kv_lens,
                                max_q_len=100, max_kv_len=100, split_size=64)
    assert bi.bi_check_device_errors() == bi.ERR_DEVICE_BOUNDS
    assert bi.bi_check_device_errors() == bi.OK            # cleared by the read
    assert same_bytes(bad[:qlens[0]], good[:qlens[0]])
    # a chunk that ends past its sequence's KV length
    lens = kv.kv_lens.clone()
    lens[0] = 60
    bi.attn_prefill_chunk(q, cu, st, kv.k_cache, kv.v_cache, kv.block_table, lens,
                          max_q_len=100, max_kv_len=100, split_size=64)
    assert bi.bi_check_device_errors() == bi.ERR_DEVICE_BOUNDS
    again, _ = prefill(q, cu, st, kv, kv.kv_lens, 100, 100, 64)   # the context still works
    assert bi.bi_check_device_errors() == bi.OK
    assert same_bytes(again, good)


def test_kv_write_places_rows_in_pages(cuda):
    kv = to_dev(synth.paged_kv([40, 3], 2, 64, 16, 5500, reserve_tokens=20), cuda)
    kc, vc = kv.k_cache.clone(), kv.v_cache.clone()
    seq = torch.tensor([0, 1, 1, 0], dtype=torch.int32, device=cuda)
    pos = torch.tensor([40, 3, 4, 41], dtype=torch.int32, device=cuda)
    kn = synth.normal_bf16((4, 2, 64), 5501, device=cuda)
    vn = synth.normal_bf16((4, 2, 64), 5502, device=cuda)
    bi.kv_write(kn, vn, seq, pos, kv.k_cache, kv.v_cache, kv.block_table)
    for i in range(4):
        s, p = int(seq[i]), int(pos[i])
        page = int(kv.block_table[s, p // 16])
        kc[page, :, p % 16] = kn[i]
        vc[page, :, p % 16] = vn[i]
    assert same_bytes(kv.k_cache, kc) and same_bytes(kv.v_cache, vc)
    assert bi.bi_check_device_errors() == bi.OK


def test_attention_run_to_run(cuda):
    # the same call twice gives the same bytes (a race between the roles of
    # a block, or an order that depends on timing, would show up here):
    # GQA decode over log-uniform lengths and a long causal prefill chunk
    lens = synth.loguniform_int(24, 1, 9000, 5100).tolist()
    kv = to_dev(synth.paged_kv(lens, 8, 128, 16, 5101), cuda)
    q = synth.normal_bf16((24, 32, 128), 5102, device=cuda)
    d1 = decode(q, kv, 9000, 256)
    d2 = decode(q, kv, 9000, 256)
    assert same_bytes(d1[0], d2[0]) and same_bytes(d1[1], d2[1])
    T, C = 3000, 1000
    pkv = to_dev(synth.paged_kv([T], 8, 128, 16, 5103), cuda)
    pq = synth.normal_bf16((C, 32, 128), 5104, device=cuda)
    cu = torch.tensor([0, C], dtype=torch.int32, device=cuda)
    st = torch.tensor([T - C], dtype=torch.int32, device=cuda)
    p1 = prefill(pq, cu, st, pkv, pkv.kv_lens, C, T, 256)
    p2 = prefill(pq, cu, st, pkv, pkv.kv_lens, C, T, 256)
    assert same_bytes(p1[0], p2[0]) and same_bytes(p1[1], p2[1])
    assert bi.bi_check_device_errors() == bi.OK
