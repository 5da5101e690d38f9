"""Run one operation of the library on seeded inputs, a few times, with an L2
flush between runs -- the unit a profiler capture or a quick timing needs.

    python -m invariant_bi_rmsnorm_02_gb300.cases gemm --M 2048 --N 14336 --K 4096
    python -m invariant_bi_rmsnorm_02_gb300.cases rmsnorm --M 8192 --H 4096
    python -m invariant_bi_rmsnorm_02_gb300.cases decode --B 64
    python -m invariant_bi_rmsnorm_02_gb300.cases prefill --T 8192 --chunk 2048
    python -m invariant_bi_rmsnorm_02_gb300.cases add_rmsnorm --M 8192 --H 4096
    python -m invariant_bi_rmsnorm_02_gb300.cases sample --B 256 --V 128256 --temp 1.0
    python -m invariant_bi_rmsnorm_02_gb300.cases rope --M 8192
    python -m invariant_bi_rmsnorm_02_gb300.cases silu --M 8192 --F 14336
    python -m invariant_bi_rmsnorm_02_gb300.cases gather --M 8192 --H 4096
    python -m invariant_bi_rmsnorm_02_gb300.cases gemm_swiglu --M 8192 --F 14336 --K 4096
    python -m invariant_bi_rmsnorm_02_gb300.cases gemm_silu --M 8192 --F 14336 --K 4096

Prints one line per run with the CUDA-event time of the call (the device is
kept busy while the call is queued, so host launch latency is not in the
time) and, for the element-wise and sampling ops, the algorithmic bytes moved
per second; for the GEMMs, the flops per second.  gemm_swiglu is the gate/up
projection with SwiGLU in the GEMM epilogue, gemm_silu the same work as two
calls (the GEMM into [M, 2F], then the SwiGLU kernel).
"""
from __future__ import annotations

import argparse

import torch

from . import _binding as bi
from . import synth


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["rmsnorm", "gemm", "decode", "prefill", "add_rmsnorm",
                                   "sample", "rope", "silu", "gather", "gemm_swiglu",
                                   "gemm_silu"])
    ap.add_argument("--mode", type=int, default=bi.INVARIANT)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--M", type=int, default=8192)
    ap.add_argument("--H", type=int, default=4096)
    ap.add_argument("--N", type=int, default=14336)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--B", type=int, default=64)
    ap.add_argument("--max-len", type=int, default=32768)
    ap.add_argument("--split", type=int, default=256)
    ap.add_argument("--T", type=int, default=8192)
    ap.add_argument("--chunk", type=int, default=2048)
    ap.add_argument("--F", type=int, default=14336)
    ap.add_argument("--V", type=int, default=128256)
    ap.add_argument("--temp", type=float, default=0.0)
    a = ap.parse_args(argv)
    nbytes = 0  # algorithmic bytes of one call (element-wise and sampling ops)
    flops = 0   # algorithmic flops of one call (GEMMs)
    dev = torch.device("cuda", 0)
    bi.load()
    # L2 flush: write 256 MB, then read another 256 MB so that the written
    # lines have drained before the timed call starts
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    drain = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    if a.op == "rmsnorm":
        x = synth.normal_bf16((a.M, a.H), 1, device=dev)
        w = synth.normal_bf16((a.H,), 2, device=dev)
        fn = lambda: bi.rmsnorm(x, w, 1e-6, a.mode)
    elif a.op == "gemm":
        A = synth.normal_bf16((a.M, a.K), 1, device=dev)
        W = synth.normal_bf16((a.N, a.K), 2, std=0.02, device=dev)
        fn = lambda: bi.gemm(A, W, a.mode)
        flops = 2 * a.M * a.N * a.K
    elif a.op in ("gemm_swiglu", "gemm_silu"):
        A = synth.normal_bf16((a.M, a.K), 1, device=dev)
        W = synth.normal_bf16((2 * a.F, a.K), 2, std=0.02, device=dev)
        if a.op == "gemm_swiglu":
            fn = lambda: bi.gemm_swiglu(A, W, a.mode)
        else:
            fn = lambda: bi.silu_mul(bi.gemm(A, W, a.mode), block=128)
        flops = 2 * a.M * 2 * a.F * a.K
    elif a.op == "decode":
        lens = synth.loguniform_int(a.B, 1, a.max_len, 3).tolist()
        kv = synth.paged_kv(lens, 8, 128, 16, 4, device=dev)
        q = synth.normal_bf16((a.B, 32, 128), 15, device=dev)  # apart from K (5), V (6)
        fn = lambda: bi.attn_decode(q, kv.k_cache, kv.v_cache, kv.block_table, kv.kv_lens,
                                    max_kv_len=a.max_len, split_size=a.split, mode=a.mode)
    elif a.op == "add_rmsnorm":
        x = synth.normal_bf16((a.M, a.H), 1, device=dev)
        r = synth.normal_bf16((a.M, a.H), 3, device=dev)
        w = synth.normal_bf16((a.H,), 2, device=dev)
        fn = lambda: bi.add_rmsnorm(x, r, w, 1e-6, a.mode)
        nbytes = 4 * a.M * a.H * 2 + a.H * 2       # read x, r; write h, y; w once
    elif a.op == "sample":
        z = synth.normal_bf16((a.B, a.V), 1, std=2.0, device=dev)
        T = torch.full((a.B,), a.temp, device=dev)
        sd = torch.arange(a.B, dtype=torch.int64, device=dev)
        fn = lambda: bi.sample(z, T, sd, sd)
        nbytes = a.B * a.V * 2
    elif a.op == "rope":
        Hq, Hkv, D = 32, 8, 128
        qkv = synth.normal_bf16((a.M, (Hq + 2 * Hkv) * D), 1, device=dev)
        pos = synth.uniform_int(a.M, 0, 8191, 2).to(torch.int32).to(dev)
        fn = lambda: bi.rope_qkv(qkv, pos, Hq, Hkv, D)
        nbytes = 2 * a.M * (Hq + 2 * Hkv) * D * 2 + a.M * 4
    elif a.op == "silu":
        gu = synth.normal_bf16((a.M, 2 * a.F), 1, device=dev)
        fn = lambda: bi.silu_mul(gu)
        nbytes = 3 * a.M * a.F * 2
    elif a.op == "gather":
        table = synth.normal_bf16((128256, a.H), 1, device=dev)
        idx = synth.uniform_int(a.M, 0, 128255, 2).to(torch.int32).to(dev)
        fn = lambda: bi.gather_rows(table, idx)
        nbytes = 2 * a.M * a.H * 2 + a.M * 4
    else:
        kv = synth.paged_kv([a.T], 8, 128, 16, 6, device=dev)
        q = synth.normal_bf16((a.chunk, 32, 128), 17, device=dev)  # apart from K (7), V (8)
        cu = torch.tensor([0, a.chunk], dtype=torch.int32, device=dev)
        st = torch.tensor([a.T - a.chunk], dtype=torch.int32, device=dev)
        fn = lambda: bi.attn_prefill_chunk(q, cu, st, kv.k_cache, kv.v_cache, kv.block_table,
                                           kv.kv_lens, max_q_len=a.chunk, max_kv_len=a.T,
                                           split_size=a.split, mode=a.mode)
    for i in range(a.reps):
        flush.zero_()
        drain.sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(200_000)  # the device waits here while the call is queued
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        extra = "  %.1f GB/s" % (nbytes / ms / 1e6) if nbytes else ""
        if flops:
            extra = "  %.1f TFLOP/s" % (flops / ms / 1e9)
        print("%s run %d: %.3f ms%s" % (a.op, i, ms, extra))
    status = bi.bi_check_device_errors()
    if status != bi.OK:
        raise SystemExit("device error: %s" % bi.bi_status_string(status))


if __name__ == "__main__":
    main()
