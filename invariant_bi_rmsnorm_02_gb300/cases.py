"""Run one operation of the library on seeded inputs, a few times, with an L2
flush between runs -- the unit a profiler capture or a quick timing needs.

    python -m invariant_bi_rmsnorm_02_gb300.cases gemm --M 2048 --N 14336 --K 4096
    python -m invariant_bi_rmsnorm_02_gb300.cases rmsnorm --M 8192 --H 4096
    python -m invariant_bi_rmsnorm_02_gb300.cases decode --B 64
    python -m invariant_bi_rmsnorm_02_gb300.cases prefill --T 8192 --chunk 2048

Prints one line per run with the CUDA-event time of the call.
"""
from __future__ import annotations

import argparse

import torch

from . import _binding as bi
from . import synth


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["rmsnorm", "gemm", "decode", "prefill"])
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
    a = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    bi.load()
    flush = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device=dev)
    if a.op == "rmsnorm":
        x = synth.normal_bf16((a.M, a.H), 1, device=dev)
        w = synth.normal_bf16((a.H,), 2, device=dev)
        fn = lambda: bi.rmsnorm(x, w, 1e-6, a.mode)
    elif a.op == "gemm":
        A = synth.normal_bf16((a.M, a.K), 1, device=dev)
        W = synth.normal_bf16((a.N, a.K), 2, std=0.02, device=dev)
        fn = lambda: bi.gemm(A, W, a.mode)
    elif a.op == "decode":
        lens = synth.loguniform_int(a.B, 1, a.max_len, 3).tolist()
        kv = synth.paged_kv(lens, 8, 128, 16, 4, device=dev)
        q = synth.normal_bf16((a.B, 32, 128), 5, device=dev)
        fn = lambda: bi.attn_decode(q, kv.k_cache, kv.v_cache, kv.block_table, kv.kv_lens,
                                    max_kv_len=a.max_len, split_size=a.split, mode=a.mode)
    else:
        kv = synth.paged_kv([a.T], 8, 128, 16, 6, device=dev)
        q = synth.normal_bf16((a.chunk, 32, 128), 7, device=dev)
        cu = torch.tensor([0, a.chunk], dtype=torch.int32, device=dev)
        st = torch.tensor([a.T - a.chunk], dtype=torch.int32, device=dev)
        fn = lambda: bi.attn_prefill_chunk(q, cu, st, kv.k_cache, kv.v_cache, kv.block_table,
                                           kv.kv_lens, max_q_len=a.chunk, max_kv_len=a.T,
                                           split_size=a.split, mode=a.mode)
    for i in range(a.reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        print("%s run %d: %.3f ms" % (a.op, i, e0.elapsed_time(e1)))
    status = bi.bi_check_device_errors()
    if status != bi.OK:
        raise SystemExit("device error: %s" % bi.bi_status_string(status))


if __name__ == "__main__":
    main()
