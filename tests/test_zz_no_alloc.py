"""bi_attn_decode_noalloc: decode for callers that cannot allocate device
memory (an engine that has given all of HBM to its KV-cache pool, a plugin
whose host framework owns the allocator).  Its scratch is a fixed array inside
the library instead of a caller workspace.  This file is collected last, so a
run that stops at the first failure has run every other test before it."""
import pytest
import torch

import invariant_bi_rmsnorm_02_gb300 as bi
from invariant_bi_rmsnorm_02_gb300 import synth

pytestmark = pytest.mark.gpu
ATOL = 2e-3   # the attention tolerance used by the other GPU tests


def _case(dev, lens, Hq, Hkv, D, seed):
    kv = synth.paged_kv(lens, Hkv, D, 16, seed, device=dev)
    q = synth.normal_bf16((len(lens), Hq, D), seed + 1, device=dev)
    return q, kv


def _with_workspace(q, kv, max_kv_len, S):
    return bi.attn_decode(q, kv.k_cache, kv.v_cache, kv.block_table, kv.kv_lens,
                          max_kv_len=max_kv_len, split_size=S, want_f32=True)


def _noalloc(q, kv, max_kv_len, S):
    out = torch.empty_like(q)
    out32 = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    bi.bi_attn_decode_noalloc(q, kv.k_cache, kv.v_cache, kv.block_table, kv.kv_lens, out, out32,
                              max_kv_len=max_kv_len, split_size=S,
                              sm_scale=q.shape[-1] ** -0.5)
    return out, out32


def test_noalloc_decode_matches_workspace_decode_twice(cuda):
    # two calls in a row with different shapes: the shared scratch keeps the
    # first call's contents, which must not leak into the second
    cases = [
        (synth.uniform_int(8, 1, 512, 7000).tolist(), 4, 2, 64, 512, 64, 7001),
        (synth.loguniform_int(16, 1, 8192, 7002).tolist(), 32, 8, 128, 8192, 256, 7003),
    ]
    for lens, Hq, Hkv, D, max_len, S, seed in cases:
        q, kv = _case(cuda, lens, Hq, Hkv, D, seed)
        ref, ref32 = _with_workspace(q, kv, max_len, S)
        got, got32 = _noalloc(q, kv, max_len, S)
        torch.cuda.synchronize()
        assert bi.bi_check_device_errors() == bi.OK
        diff = (got32 - ref32).abs().max().item()
        assert diff <= ATOL, diff
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(got32.view(torch.int32), ref32.view(torch.int32))


def test_noalloc_rejects_scratch_beyond_its_limit(cuda):
    lens = [4096] * 64
    need = bi.bi_attn_decode_workspace_size(64, 32, 8, 128, 32768, 256, bi.INVARIANT)
    assert need > bi.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(64, 32, 128, dtype=torch.bfloat16, device=cuda)
    kv = synth.paged_kv([1] * 64, 8, 128, 16, 7100, device=cuda)
    out = torch.empty_like(q)
    with pytest.raises(bi.BiError) as e:
        bi.bi_attn_decode_noalloc(q, kv.k_cache, kv.v_cache, kv.block_table, kv.kv_lens, out,
                                  max_kv_len=32768, split_size=256, sm_scale=128 ** -0.5)
    assert e.value.status == bi.ERR_WORKSPACE
    assert bi.bi_check_device_errors() == bi.OK
