"""Two serving-level properties of the kernels, checked byte for byte on the GPU:

* a prompt whose prefix sits in pages shared with another request (a prefix
  cache hit) gets, for its uncached tail, exactly the attention output of a
  fresh prefill of the whole prompt in pages of its own; the next decode step
  agrees too (Defeating Nondeterminism in LLM Inference, the attention
  section: the kernel must not care which part of the KV came from a cache);
* a whole decode step of a layer (residual add + RMSNorm, QKV GEMM, KV write,
  paged decode attention) captured in a CUDA graph and replayed gives the same
  bytes as running it eagerly, step after step (the kernels take all shapes
  from host arguments fixed at capture and read lengths on the device)."""
import pytest
import torch

import invariant_bi_rmsnorm_02_gb300 as bi
from invariant_bi_rmsnorm_02_gb300 import synth
from gpu_util import first_divergence, same_bytes

pytestmark = pytest.mark.gpu
PAGE = 16


def i32(v, dev):
    return torch.tensor(v, dtype=torch.int32, device=dev)


def write_rows(k, v, seq, pos0, kc, vc, bt):
    n = k.shape[0]
    dev = k.device
    bi.kv_write(k, v, i32([seq] * n, dev), torch.arange(pos0, pos0 + n, dtype=torch.int32,
                                                        device=dev), kc, vc, bt)


def test_prefix_cache_hit_equals_fresh_prefill(cuda):
    Hq, Hkv, D, S = 32, 8, 128, 256
    P, tail_a, tail_b = 1024, 300, 517          # shared prefix: 64 whole pages
    Tb = P + tail_b
    K_pre = synth.normal_bf16((P, Hkv, D), 9900, device=cuda)
    V_pre = synth.normal_bf16((P, Hkv, D), 9901, device=cuda)
    K_a = synth.normal_bf16((tail_a, Hkv, D), 9902, device=cuda)
    V_a = synth.normal_bf16((tail_a, Hkv, D), 9903, device=cuda)
    K_b = synth.normal_bf16((tail_b + 1, Hkv, D), 9904, device=cuda)   # + one decode token
    V_b = synth.normal_bf16((tail_b + 1, Hkv, D), 9905, device=cuda)
    q_b = synth.normal_bf16((Tb, Hq, D), 9906, device=cuda)
    q_next = synth.normal_bf16((1, Hq, D), 9907, device=cuda)
    maxblk = 128
    g = torch.Generator().manual_seed(9908)

    # fresh: request B alone, every page its own, the whole prompt in one chunk
    npg = 100
    kc = torch.zeros(npg, Hkv, PAGE, D, dtype=torch.bfloat16, device=cuda)
    vc = torch.zeros_like(kc)
    bt = torch.zeros(1, maxblk, dtype=torch.int32)
    bt[0, :npg] = torch.randperm(npg, generator=g).to(torch.int32)
    bt = bt.to(cuda)
    write_rows(K_pre, V_pre, 0, 0, kc, vc, bt)
    write_rows(K_b[:tail_b], V_b[:tail_b], 0, P, kc, vc, bt)
    fresh, fresh32 = bi.attn_prefill_chunk(q_b, i32([0, Tb], cuda), i32([0], cuda), kc, vc, bt,
                                           i32([Tb], cuda), max_q_len=Tb, max_kv_len=Tb,
                                           split_size=S, want_f32=True)

    # cached: request A wrote the prefix (and its own tail); B's table points
    # its first 64 entries at A's pages and only B's tail is written and run
    npg2 = 200
    kc2 = torch.zeros(npg2, Hkv, PAGE, D, dtype=torch.bfloat16, device=cuda)
    vc2 = torch.zeros_like(kc2)
    perm = torch.randperm(npg2, generator=g).to(torch.int32)
    bt2 = torch.zeros(2, maxblk, dtype=torch.int32)
    na = -(-(P + tail_a) // PAGE)
    bt2[0, :na] = perm[:na]
    bt2[1, :P // PAGE] = perm[:P // PAGE]                      # shared prefix pages
    nb_own = -(-(Tb + 1) // PAGE) - P // PAGE
    bt2[1, P // PAGE:P // PAGE + nb_own] = perm[na:na + nb_own]
    bt2 = bt2.to(cuda)
    write_rows(K_pre, V_pre, 0, 0, kc2, vc2, bt2)
    write_rows(K_a, V_a, 0, P, kc2, vc2, bt2)
    write_rows(K_b[:tail_b], V_b[:tail_b], 1, P, kc2, vc2, bt2)
    # B's tail as the second sequence of a chunk, after a neighbour (A's last
    # 40 tail positions, recomputed)
    q_a = synth.normal_bf16((40, Hq, D), 9909, device=cuda)
    q = torch.cat([q_a, q_b[P:]]).contiguous()
    out, out32 = bi.attn_prefill_chunk(
        q, i32([0, 40, 40 + tail_b], cuda), i32([P + tail_a - 40, P], cuda), kc2, vc2, bt2,
        i32([P + tail_a, Tb], cuda), max_q_len=tail_b, max_kv_len=Tb, split_size=S,
        want_f32=True)
    assert bi.bi_check_device_errors() == bi.OK
    assert same_bytes(out[40:], fresh[P:]), first_divergence(out[40:], fresh[P:])
    assert same_bytes(out32[40:], fresh32[P:])

    # the next token of B decodes to the same bytes in both worlds
    write_rows(K_b[tail_b:], V_b[tail_b:], 0, Tb, kc, vc, bt)
    write_rows(K_b[tail_b:], V_b[tail_b:], 1, Tb, kc2, vc2, bt2)
    d1 = bi.attn_decode(q_next, kc, vc, bt, i32([Tb + 1], cuda), max_kv_len=Tb + 1,
                        split_size=S)
    d2 = bi.attn_decode(q_next, kc2, vc2, bt2[1:].contiguous(), i32([Tb + 1], cuda),
                        max_kv_len=Tb + 1, split_size=S)
    assert same_bytes(d1, d2)
    # and A's pages were only read: its prefix and tail are unchanged
    d3 = bi.attn_decode(q_next, kc2, vc2, bt2[:1].contiguous(), i32([P + tail_a], cuda),
                        max_kv_len=P + tail_a, split_size=S)
    kc3 = torch.zeros_like(kc2)
    vc3 = torch.zeros_like(vc2)
    write_rows(K_pre, V_pre, 0, 0, kc3, vc3, bt2)
    write_rows(K_a, V_a, 0, P, kc3, vc3, bt2)
    d4 = bi.attn_decode(q_next, kc3, vc3, bt2[:1].contiguous(), i32([P + tail_a], cuda),
                        max_kv_len=P + tail_a, split_size=S)
    assert same_bytes(d3, d4)


class LayerState:
    """The device state one decode step of a layer reads and writes."""

    def __init__(self, res, kc, vc, lens):
        self.res, self.kc, self.vc, self.lens = res, kc, vc, lens
        self.delta = torch.empty_like(res)

    def clone(self):
        return LayerState(self.res.clone(), self.kc.clone(), self.vc.clone(), self.lens.clone())


def test_decode_step_graph_replay_equals_eager(cuda):
    B, H, Hq, Hkv, D, S, steps = 8, 1024, 8, 2, 128, 256, 12
    max_kv = 4096
    N = (Hq + 2 * Hkv) * D
    w = synth.normal_bf16((H,), 9950, std=0.1, mean=1.0, device=cuda)
    Wqkv = synth.normal_bf16((N, H), 9951, std=0.03, device=cuda)
    lens0 = synth.loguniform_int(B, 1, 2000, 9952).tolist()
    kv = synth.paged_kv(lens0, Hkv, D, PAGE, 9953, reserve_tokens=steps, device=cuda)
    seq = torch.arange(B, dtype=torch.int32, device=cuda)
    base = LayerState(synth.normal_bf16((B, H), 9954, device=cuda), kv.k_cache, kv.v_cache,
                      kv.kv_lens)
    deltas = [synth.normal_bf16((B, H), 9960 + t, device=cuda) for t in range(steps)]

    def step(st):
        y = bi.add_rmsnorm(st.delta, st.res, w)
        qkv = bi.gemm(y, Wqkv)
        q = qkv[:, :Hq * D].reshape(B, Hq, D).contiguous()
        k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(B, Hkv, D).contiguous()
        v = qkv[:, (Hq + Hkv) * D:].reshape(B, Hkv, D).contiguous()
        bi.kv_write(k, v, seq, st.lens, st.kc, st.vc, kv.block_table)
        st.lens.add_(1)
        return bi.attn_decode(q, st.kc, st.vc, kv.block_table, st.lens, max_kv_len=max_kv,
                              split_size=S), y

    eager = base.clone()
    ref = []
    for t in range(steps):
        eager.delta.copy_(deltas[t])
        o, y = step(eager)
        ref.append((o.clone(), y.clone()))

    # warm up on a side stream with a throwaway state, then capture
    warm = base.clone()
    warm.delta.copy_(deltas[0])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(warm)
    torch.cuda.current_stream().wait_stream(side)
    graphed = base.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out_static, y_static = step(graphed)
    torch.cuda.synchronize()
    assert same_bytes(graphed.lens, base.lens)      # capture ran nothing
    for t in range(steps):
        graphed.delta.copy_(deltas[t])
        graph.replay()
        assert same_bytes(y_static, ref[t][1]), ("y", t)
        assert same_bytes(out_static, ref[t][0]), ("attention", t)
    torch.cuda.synchronize()
    assert bi.bi_check_device_errors() == bi.OK
    assert same_bytes(graphed.res, eager.res)
    assert same_bytes(graphed.kc, eager.kc) and same_bytes(graphed.vc, eager.vc)
    assert same_bytes(graphed.lens, eager.lens)
