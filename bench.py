#!/usr/bin/env python
"""Benchmark of the batch-invariant hot path on one GB300 (or N replicas).

One step is one pass of the whole path over one batch of synthetic input,
shaped like a Llama-3-8B layer in a serving iteration:

  1. KV write   : the 64 decode requests' newest K/V rows into the paged cache
  2. RMSNorm    : x [8192, 4096]
  3. QKV GEMM   : [8192, 4096] x [6144, 4096]^T
  4. MLP-up GEMM: [8192, 4096] x [14336, 4096]^T
  5. decode     : 64 requests, 32 q / 8 kv heads, D=128, KV lengths
                  log-uniform in 1..32768 (growing one token per step), split
                  size 256 (split kernel + merge kernel)
  6. prefill    : one 2048-token chunk (positions 6144..8191) of an 8192-token
                  prompt, same heads, split size 256

The headline is the GEMMs' TFLOP/s (flops of both GEMMs / their device time,
CUDA events on the launching stream); every other kernel is reported beside
it against its own roofline, and the whole step is also run in the
batch-variant mode to report the cost of invariance (t_invariant / t_variant
- 1 per kernel).  L2 is flushed (a 256 MB write, then a 256 MB read so the dirty
lines drain outside the timed region) before every kernel of the step, so
each kernel is timed on a cold, clean L2 and none pays for the write-back of
its predecessor's output; a short device-side sleep after the flush keeps the
host's launch latency out of the kernel's events.  The step time is the sum of
the kernels' times.
Inputs are resident in HBM when the timed region starts.  The end-to-end
line runs the same kernels back to back with host copies around them.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the fp64 CPU oracle (the only other implementation of
this path) on a bounded sample of the same workload, on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

M, H, N_QKV, N_UP = 8192, 4096, 6144, 14336
HOST_LEAD_CYCLES = 200_000  # ~0.1 ms at the SM clock
EPS = 1e-6
DEC = dict(B=64, Hq=32, Hkv=8, D=128, page=16, S=256, max_len=32768)
PRE = dict(T=8192, chunk=2048, start=6144)
METRIC = "bi_gemm TFLOP/s, RMSNorm/decode-attn HBM GB/s (% peak); invariant slowdown"
WORKLOAD = ("Llama-3-8B-shaped layer slice: RMSNorm 8192x4096 -> QKV GEMM 4096->6144 and "
            "MLP-up GEMM 4096->14336 at M=8192; GQA decode 64 requests (32/8 heads, D=128, "
            "KV log-uniform 1..32768, page 16, split 256); causal prefill chunk of 2048 at "
            "position 6144 of an 8192-token prompt; KV write of the decode tokens")


# ---------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sust=d.get("bf16_tflops_sustained", d["bf16_tflops"]), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "invariant_bi_rmsnorm_02_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "gemm_tc_kernel": ("gemm.cu", "device_common.cuh", "tcgen05.cuh"),
    "rmsnorm_row_kernel": ("rmsnorm.cu",),
    "attn_decode_split_kernel": ("attention.cu", "device_common.cuh", "tcgen05.cuh"),
    "attn_prefill_kernel": ("attention.cu", "device_common.cuh", "tcgen05.cuh"),
}


def profiled_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_sha") != source_hash(*KERNEL_SOURCES[kernel]):
        return None
    return e.get("dram_bytes_per_launch")


def fingerprint(dev, rank):
    """What a result was measured with: device, driver and toolchain, the
    library's sources, the fixed tile shapes, the seeds and the host."""
    import invariant_bi_rmsnorm_02_gb300 as bi
    driver = None
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(dev.index), "--query-gpu=driver_version",
                              "--format=csv,noheader"], capture_output=True, text=True, timeout=20)
        driver = out.stdout.strip() or None
    except (OSError, subprocess.SubprocessError):
        pass
    csrc = os.path.join(ROOT, "invariant_bi_rmsnorm_02_gb300", "csrc")
    return {
        "gpu": torch.cuda.get_device_name(dev), "sm_count":
            torch.cuda.get_device_properties(dev).multi_processor_count,
        "driver": driver, "cuda_runtime": torch.version.cuda, "torch": torch.__version__,
        "libbi": bi.bi_version(), "libbi_sources_sha": source_hash(
            *sorted(f for f in os.listdir(csrc) if os.path.isfile(os.path.join(csrc, f)))),
        "gemm_tile": "128x256 (128x64 for M<=64 where those tiles fit one wave, 128x192 where it fills the SMs better), k-block 64, tcgen05 kind::f16 M=128 K=16",
        "attention_key_tile": 64, "split_size": DEC["S"], "page_size": DEC["page"],
        "seeds": "workload seeds 100000*rank + 1..15 (rank %d)" % rank,
        "host_cores": os.cpu_count(),
    }


class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.lines = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- workload
# Input seeds of every workload, as offsets (the step's are added to
# 100000 * rank).  synth.paged_kv(seed) draws K from seed + 1 and V from
# seed + 2, so no other input of a workload may use those: queries equal to
# cached keys would be a degenerate input (their own key scores ~11 sigma
# above the rest).  "kv" entries name paged caches, the others plain tensors.
SEEDS = {
    "step": dict(x=1, w=2, wqkv=3, wup=4, lens=5, kv=6, q=13, k_new=14, v_new=9, pkv=10,
                 pq=15),
    "tiny": dict(x=1001, w=1002, W=1003, lens=1004, kv=1005, q=1016),
    "schedules": dict(kv=4001, q=4012),
}
KV_SEEDS = {"step": ("kv", "pkv"), "tiny": ("kv",), "schedules": ("kv",)}


def seed_collisions():
    """Pairs (workload, input) whose seed is the K or V stream of one of the
    workload's paged caches; empty when the inputs are independent."""
    bad = []
    for wl, seeds in SEEDS.items():
        streams = {seeds[k] + o for k in KV_SEEDS[wl] for o in (1, 2)}
        bad += [(wl, name) for name, v in seeds.items()
                if name not in KV_SEEDS[wl] and v in streams]
    return bad


class Workload:
    """Device-resident inputs of one step, seeded."""

    def __init__(self, dev, rank, reserve):
        import invariant_bi_rmsnorm_02_gb300 as bi
        from invariant_bi_rmsnorm_02_gb300 import synth
        self.bi, self.dev = bi, dev
        s = 100000 * rank
        sd = SEEDS["step"]
        self.x = synth.normal_bf16((M, H), s + sd["x"], device=dev)
        self.w = synth.normal_bf16((H,), s + sd["w"], std=0.1, mean=1.0, device=dev)
        self.Wqkv = synth.normal_bf16((N_QKV, H), s + sd["wqkv"], std=0.02, device=dev)
        self.Wup = synth.normal_bf16((N_UP, H), s + sd["wup"], std=0.02, device=dev)
        self.y = torch.empty_like(self.x)
        self.qkv = torch.empty(M, N_QKV, dtype=torch.bfloat16, device=dev)
        self.up = torch.empty(M, N_UP, dtype=torch.bfloat16, device=dev)
        d = DEC
        lens = synth.loguniform_int(d["B"], 1, d["max_len"] - reserve, s + sd["lens"]).tolist()
        self.kv = synth.paged_kv(lens, d["Hkv"], d["D"], d["page"], s + sd["kv"],
                                 reserve_tokens=reserve, device=dev)
        self.lens0 = self.kv.kv_lens.clone()
        self.lens = self.kv.kv_lens.clone()
        self.seq = torch.arange(d["B"], dtype=torch.int32, device=dev)
        self.q = synth.normal_bf16((d["B"], d["Hq"], d["D"]), s + sd["q"], device=dev)
        self.k_new = synth.normal_bf16((d["B"], d["Hkv"], d["D"]), s + sd["k_new"], device=dev)
        self.v_new = synth.normal_bf16((d["B"], d["Hkv"], d["D"]), s + sd["v_new"], device=dev)
        self.dec_out = torch.empty_like(self.q)
        self.dec_ws = {}
        for mode in (bi.INVARIANT, bi.VARIANT):
            nb = bi.bi_attn_decode_workspace_size(d["B"], d["Hq"], d["Hkv"], d["D"],
                                                  d["max_len"], d["S"], mode)
            self.dec_ws[mode] = torch.empty(nb // 4 + 4, dtype=torch.float32, device=dev)
        self.pkv = synth.paged_kv([PRE["T"]], d["Hkv"], d["D"], d["page"], s + sd["pkv"],
                                  device=dev)
        self.pq = synth.normal_bf16((PRE["chunk"], d["Hq"], d["D"]), s + sd["pq"], device=dev)
        self.pout = torch.empty_like(self.pq)
        self.cu = torch.tensor([0, PRE["chunk"]], dtype=torch.int32, device=dev)
        self.pstart = torch.tensor([PRE["start"]], dtype=torch.int32, device=dev)
        self.pkl = torch.tensor([PRE["start"] + PRE["chunk"]], dtype=torch.int32, device=dev)
        self.rms_ws = torch.empty(bi.bi_rmsnorm_workspace_size(M, H, bi.VARIANT) // 4 + 4,
                                  dtype=torch.float32, device=dev)
        gws = max(bi.bi_gemm_workspace_size(m, n, H, bi.VARIANT)
                  for n in (N_QKV, N_UP) for m in set(GEMM_M_SWEEP) | {M})
        self.gemm_ws = torch.empty(gws // 4 + 4, dtype=torch.float32, device=dev)

    def reset_lengths(self):
        self.lens.copy_(self.lens0)

    # each entry: (name, callable); launches counted per call
    def ops(self, mode):
        bi, d = self.bi, DEC
        def kv_write():
            bi.bi_kv_write(self.k_new, self.v_new, self.seq, self.lens, self.kv.k_cache,
                           self.kv.v_cache, self.kv.block_table)
            self.lens.add_(1)
        return [
            ("kv_write", kv_write, 1),
            ("rmsnorm", lambda: bi.bi_rmsnorm(self.x, self.w, self.y, EPS, mode, self.rms_ws), 1),
            ("gemm_qkv", lambda: bi.bi_gemm(self.y, self.Wqkv, self.qkv, mode, 0, self.gemm_ws), 1),
            ("gemm_up", lambda: bi.bi_gemm(self.y, self.Wup, self.up, mode, 0, self.gemm_ws), 1),
            ("decode", lambda: bi.bi_attn_decode(
                self.q, self.kv.k_cache, self.kv.v_cache, self.kv.block_table, self.lens,
                self.dec_out, None, max_kv_len=d["max_len"], split_size=d["S"],
                sm_scale=d["D"] ** -0.5, mode=mode, workspace=self.dec_ws[mode]),
             2 if d["B"] <= 128 else 3),
            ("prefill", lambda: bi.bi_attn_prefill_chunk(
                self.pq, self.cu, self.pstart, self.pkv.k_cache, self.pkv.v_cache,
                self.pkv.block_table, self.pkl, self.pout, None, max_q_len=PRE["chunk"],
                max_kv_len=PRE["T"], split_size=d["S"], sm_scale=d["D"] ** -0.5, mode=mode),
             1),
        ]

    def launches(self):
        """Our kernel launches per invariant step: KV write, RMSNorm, two GEMMs,
        decode split + merge (plus a plan kernel above 128 sequences), prefill."""
        return sum(n for _, _, n in self.ops(self.bi.INVARIANT))

    # algorithmic work per launch
    def work(self, steps):
        """Algorithmic bytes / flops of each op of one step; the decode's at the
        mean KV length of the timed steps (step s, counted from 0, attends
        over lens0 + s + 1 keys after its KV write)."""
        d = DEC
        lens = self.lens0.double() + (steps + 1) / 2.0
        kv_bytes = float(lens.sum()) * d["Hkv"] * d["D"] * 2 * 2
        qo = d["B"] * d["Hq"] * d["D"] * 2 * 2
        T0, C = PRE["start"], PRE["chunk"]
        causal_keys = sum(p + 1 for p in range(T0, T0 + C))
        return {
            "kv_write": {"bytes": d["B"] * d["Hkv"] * d["D"] * 2 * 2 * 2},
            "rmsnorm": {"bytes": 2 * M * H * 2 + H * 2},
            "gemm_qkv": {"flops": 2.0 * M * N_QKV * H, "bytes": 2.0 * (M * H + N_QKV * H + M * N_QKV)},
            "gemm_up": {"flops": 2.0 * M * N_UP * H, "bytes": 2.0 * (M * H + N_UP * H + M * N_UP)},
            "decode": {"bytes": kv_bytes + qo, "flops": 4.0 * d["Hq"] * d["D"] * float(lens.sum())},
            "prefill": {"flops": 4.0 * d["Hq"] * d["D"] * causal_keys,
                        "bytes": (T0 + C) * d["Hkv"] * d["D"] * 2 * 2 + 2 * C * d["Hq"] * d["D"] * 2},
        }


class L2Flush:
    """Evicts the step's data from L2 before a timed step: a 256 MB write (twice
    the L2), then a 256 MB read of a second buffer, so that the dirty lines the
    write leaves behind drain to HBM before the timed region, not inside it."""

    def __init__(self, dev):
        n = 256 * 1024 * 1024 // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.zeros(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def zero_(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def timed_steps(wl, mode, steps, warmup, flush, stream, dist_barrier):
    ops = wl.ops(mode)
    names = [n for n, _, _ in ops]
    per = {n: 0.0 for n in names}
    wl.reset_lengths()
    for _ in range(warmup):
        flush.zero_()
        for _, fn, _ in ops:
            fn()
    torch.cuda.synchronize()
    wl.reset_lengths()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(ops))] for _ in range(steps)]
    mean_lens = []
    dist_barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for s in range(steps):
            for i, (_, fn, _) in enumerate(ops):
                flush.zero_()
                # a short device-side wait so that the host has enqueued the
                # kernel before the start event fires: host launch latency
                # stays out of the kernel's time (the e2e line measures it)
                torch.cuda._sleep(HOST_LEAD_CYCLES)
                ev[s][2 * i].record(stream)
                fn()
                ev[s][2 * i + 1].record(stream)
    torch.cuda.synchronize()
    dist_barrier()
    step_ms = []
    for s in range(steps):
        t = 0.0
        for i, n in enumerate(names):
            d = ev[s][2 * i].elapsed_time(ev[s][2 * i + 1])
            per[n] += d
            t += d
        step_ms.append(t)
    return {n: v / steps for n, v in per.items()}, sum(step_ms) / steps


def e2e_steps(wl, steps, warmup, stream):
    """The GEMM metric end to end through the public API with host buffers:
    pinned host inputs copied in, the path run, the results copied out.  Each
    result is copied out on its own stream as soon as its kernel is done, and
    each input of the next step is copied in on another as soon as the op
    that read the current one is done, so copies overlap kernels; an op waits
    for its input to arrive and for the previous copy of its output to leave.
    Every step's inputs and results cross the link inside the timed region."""
    bi = wl.bi
    hx = wl.x.cpu().pin_memory()
    hq = wl.q.cpu().pin_memory()
    hk, hv = wl.k_new.cpu().pin_memory(), wl.v_new.cpu().pin_memory()
    hpq = wl.pq.cpu().pin_memory()
    hqkv = torch.empty(wl.qkv.shape, dtype=torch.bfloat16).pin_memory()
    hup = torch.empty(wl.up.shape, dtype=torch.bfloat16).pin_memory()
    hdec = torch.empty(wl.dec_out.shape, dtype=torch.bfloat16).pin_memory()
    hpre = torch.empty(wl.pout.shape, dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hx, hq, hk, hv, hpq))
    d2h = sum(t.numel() * t.element_size() for t in (hqkv, hup, hdec, hpre))
    ops = wl.ops(bi.INVARIANT)
    inputs = {"kv_write": ((wl.k_new, hk), (wl.v_new, hv)), "rmsnorm": ((wl.x, hx),),
              "decode": ((wl.q, hq),), "prefill": ((wl.pq, hpq),)}
    outputs = {"gemm_qkv": (wl.qkv, hqkv), "gemm_up": (wl.up, hup),
               "decode": (wl.dec_out, hdec), "prefill": (wl.pout, hpre)}
    copy_in = torch.cuda.Stream(stream.device)
    copy_out = torch.cuda.Stream(stream.device)
    loaded = {n: None for n in inputs}     # event: this step's copy of the input is in
    consumed = {n: None for n in inputs}   # event: the last op that read the input is done
    copied = {n: None for n in outputs}    # event: the last copy of the output is out

    def load_inputs():
        # each input of the next step goes in once the op that read the
        # previous one is done
        for n, pairs in inputs.items():
            if consumed[n] is not None:
                copy_in.wait_event(consumed[n])
            with torch.cuda.stream(copy_in):
                for dev_t, host_t in pairs:
                    dev_t.copy_(host_t, non_blocking=True)
            loaded[n] = torch.cuda.Event()
            loaded[n].record(copy_in)

    def one(last):
        for n, fn, _ in ops:
            if n in inputs:
                stream.wait_event(loaded[n])
            if n in outputs and copied[n] is not None:
                stream.wait_event(copied[n])   # the previous copy of this buffer is out
            fn()
            if n in inputs:
                consumed[n] = torch.cuda.Event()
                consumed[n].record(stream)
            if n in outputs:
                ready = torch.cuda.Event()
                ready.record(stream)
                copy_out.wait_event(ready)
                dev_t, host_t = outputs[n]
                with torch.cuda.stream(copy_out):
                    host_t.copy_(dev_t, non_blocking=True)
                copied[n] = torch.cuda.Event()
                copied[n].record(copy_out)
        if not last:
            load_inputs()

    wl.reset_lengths()
    with torch.cuda.stream(stream):
        load_inputs()
        for i in range(warmup):
            one(i == warmup - 1)
        torch.cuda.synchronize()
        wl.reset_lengths()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        copy_in.wait_stream(stream)            # the first step's inputs are timed too
        load_inputs()
        for i in range(steps):
            one(i == steps - 1)
        stream.wait_stream(copy_out)           # every result is on the host
        t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps, h2d, d2h


# ------------------------------------------------------------- CPU oracle leg
def oracle_gemm_sample(rows, seed=0):
    """The oracle's GEMM rows of both projections on a row sample; returns
    (flops, seconds, threads)."""
    import oracle
    from invariant_bi_rmsnorm_02_gb300 import synth
    x = synth.normal_bf16((rows, H), seed + 1)
    Wq = synth.normal_bf16((N_QKV, H), seed + 3, std=0.02)
    Wu = synth.normal_bf16((N_UP, H), seed + 4, std=0.02)
    t = time.perf_counter()
    oracle.gemm(x, Wq)
    oracle.gemm(x, Wu)
    dt = time.perf_counter() - t
    flops = 2.0 * rows * H * (N_QKV + N_UP)
    return flops, dt, oracle.default_threads()


def _repeat(fn, min_seconds, max_reps):
    """Runs fn until min_seconds have passed (at least once, at most max_reps
    times); returns (reps, total seconds)."""
    reps, tot = 0, 0.0
    while reps < max_reps and (reps == 0 or tot < min_seconds):
        t = time.perf_counter()
        fn()
        tot += time.perf_counter() - t
        reps += 1
    return reps, tot


def cpu_baseline(wl, per_op_seconds=4.0):
    """The fp64 oracle on the host cores, op by op, on the step's own inputs
    (copied to the host): RMSNorm of all 8192 rows, the two GEMMs on a row
    sample, the decode of all 64 requests and the prefill chunk on a sample of
    its query tokens.  Each op is repeated until about per_op_seconds have
    passed; the headline value is the GEMM's TFLOP/s (the bench's metric)."""
    import oracle
    oracle.build()
    th = oracle.default_threads()
    d = DEC
    x, w = wl.x.cpu(), wl.w.cpu()
    ops = {}
    reps, t = _repeat(lambda: oracle.rmsnorm(x, w, EPS), per_op_seconds, 20)
    ops["rmsnorm"] = {"s_per_call": t / reps, "gbs": (2 * M * H * 2 + H * 2) / (t / reps) / 1e9,
                      "sample": "all %d rows" % M}
    rows = 4 * th
    A, Wq, Wu = wl.x[:rows].cpu(), wl.Wqkv.cpu(), wl.Wup.cpu()
    reps, t = _repeat(lambda: (oracle.gemm(A, Wq), oracle.gemm(A, Wu)), per_op_seconds, 20)
    gf = 2.0 * rows * H * (N_QKV + N_UP)
    ops["gemm"] = {"s_per_call": t / reps, "tflops": gf / (t / reps) / 1e12,
                   "sample": "%d of %d rows, QKV + MLP-up" % (rows, M)}
    q, kc, vc = wl.q.cpu(), wl.kv.k_cache.cpu(), wl.kv.v_cache.cpu()
    bt, lens = wl.kv.block_table.cpu(), wl.lens0.cpu()
    reps, t = _repeat(lambda: oracle.decode_attention(q, kc, vc, bt, lens, d["D"] ** -0.5),
                      per_op_seconds, 20)
    kvb = float(lens.double().sum()) * d["Hkv"] * d["D"] * 4
    ops["decode"] = {"s_per_call": t / reps, "gbs": kvb / (t / reps) / 1e9,
                     "sample": "all %d requests" % d["B"]}
    T0, C = PRE["start"], PRE["chunk"]
    idx = torch.arange(0, C, C // 32)
    pq, pkc, pvc = wl.pq.cpu()[idx], wl.pkv.k_cache.cpu(), wl.pkv.v_cache.cpu()
    pbt = wl.pkv.block_table.cpu()
    pos = (idx + T0).to(torch.int32)
    reps, t = _repeat(lambda: oracle.prefill_attention(pq, 0, pos, pkc, pvc, pbt,
                                                       d["D"] ** -0.5), per_op_seconds, 20)
    pf = 4.0 * d["Hq"] * d["D"] * float((pos + 1).double().sum())
    ops["prefill"] = {"s_per_call": t / reps, "tflops": pf / (t / reps) / 1e12,
                      "sample": "%d of the %d chunk tokens" % (len(idx), C)}
    return {"value": ops["gemm"]["tflops"], "unit": "TFLOP/s", "cores": th, "kind": "oracle",
            "sample": "fp64 oracle on the step's inputs: RMSNorm %s, GEMM %s, decode %s, "
                      "prefill %s; each op repeated ~%.0f s" % (
                          ops["rmsnorm"]["sample"], ops["gemm"]["sample"],
                          ops["decode"]["sample"], ops["prefill"]["sample"], per_op_seconds),
            "per_op": {k: {kk: vv for kk, vv in v.items() if kk != "sample"}
                       for k, v in ops.items()}}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    rows = max(1, oracle.default_threads())
    for i in range(args.warmup):
        oracle_gemm_sample(rows, seed=i)
    tot_f = tot_t = 0.0
    for i in range(args.steps):
        f, dt, th = oracle_gemm_sample(rows, seed=100 + i)
        tot_f += f
        tot_t += dt
    val = tot_f / tot_t / 1e12
    cb = {"value": val, "unit": "TFLOP/s", "cores": th, "kind": "oracle",
          "sample": "per step %d rows (one per oracle thread) of the QKV and MLP-up GEMMs at "
                    "K=4096, fp64" % rows}
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * tot_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_rows_per_step": rows},
            "cpu_baseline": cb,
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


GEMM_M_SWEEP = (1, 3, 16, 64, 256, 1024, 8192)


def gemm_m_sweep(wl, flush, stream, reps=9):
    """The cost of invariance across batch sizes: the QKV and MLP-up GEMMs at
    every M of the projection workload, invariant and batch-variant (split-K),
    L2 clean before each call; returns {M: {...}} of mean times and the
    invariant slowdown t_inv / t_var - 1. The two modes alternate call by call
    so that a drift of the clock or of a neighbour's load falls on both, and
    the mean (not the median) is taken because the event times of a 20 us call
    come in steps of ~0.7 us; at the M where the variant plan takes one split
    both run the same kernel and the slowdown is timing noise."""
    bi = wl.bi
    out = {}
    modes = (bi.INVARIANT, bi.VARIANT)
    with torch.cuda.stream(stream):
        for m in GEMM_M_SWEEP:
            row = {}
            for name, W, C in (("qkv", wl.Wqkv, wl.qkv), ("up", wl.Wup, wl.up)):
                ts = {mode: [] for mode in modes}
                for r in range(reps + 1):
                    for mode in modes:
                        flush.zero_()
                        torch.cuda._sleep(HOST_LEAD_CYCLES)
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        bi.bi_gemm(wl.y[:m], W, C[:m], mode, 0, wl.gemm_ws)
                        e1.record(stream)
                        stream.synchronize()
                        if r:
                            ts[mode].append(e0.elapsed_time(e1))
                ms = {mode: statistics.fmean(ts[mode]) for mode in modes}
                row[name] = {"ms": ms[bi.INVARIANT], "ms_variant": ms[bi.VARIANT],
                             "slowdown": ms[bi.INVARIANT] / ms[bi.VARIANT] - 1.0}
            out[m] = row
    return out


def _median_ms(fn, stream, flush=None, reps=3):
    """Median CUDA-event time of fn on ``stream`` (L2 flushed before each rep
    when ``flush`` is given; one untimed rep first)."""
    ts = []
    with torch.cuda.stream(stream):
        for r in range(reps + 1):
            if flush is not None:
                flush.zero_()
            torch.cuda._sleep(HOST_LEAD_CYCLES)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            stream.synchronize()
            if r:
                ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def tiny_layer(dev, stream, reps=20):
    """The tiny-layer workload (RMSNorm over 256, GEMM 256->512, decode with
    4/2 heads of 64 over 8 requests of KV 1..512, page 16, split 64) at batch
    1 and 8: microseconds per op and for the three back to back, eager and
    replayed from a CUDA graph (launch-latency bound: no roofline fraction is
    meaningful at this size)."""
    import invariant_bi_rmsnorm_02_gb300 as bi
    from invariant_bi_rmsnorm_02_gb300 import synth
    c = synth.TINY
    sd = SEEDS["tiny"]
    x = synth.normal_bf16((c["B"], c["H"]), sd["x"], device=dev)
    w = synth.normal_bf16((c["H"],), sd["w"], std=0.1, mean=1.0, device=dev)
    W = synth.normal_bf16((c["N"], c["H"]), sd["W"], std=0.02, device=dev)
    lens = synth.uniform_int(c["B"], 1, c["max_len"], sd["lens"]).tolist()
    kv = synth.paged_kv(lens, c["Hkv"], c["D"], c["page"], sd["kv"], device=dev)
    q = synth.normal_bf16((c["B"], c["Hq"], c["D"]), sd["q"], device=dev)
    y, C, out = torch.empty_like(x), torch.empty(c["B"], c["N"], dtype=torch.bfloat16,
                                                 device=dev), torch.empty_like(q)
    ws = torch.empty(bi.bi_attn_decode_workspace_size(c["B"], c["Hq"], c["Hkv"], c["D"],
                                                      c["max_len"], c["split"]) // 4 + 4,
                     dtype=torch.float32, device=dev)
    res = {}
    for m in (1, c["B"]):
        ops = [lambda: bi.bi_rmsnorm(x[:m], w, y[:m], c["eps"]),
               lambda: bi.bi_gemm(y[:m], W, C[:m]),
               lambda: bi.bi_attn_decode(q[:m], kv.k_cache, kv.v_cache, kv.block_table[:m],
                                         kv.kv_lens[:m], out[:m], max_kv_len=c["max_len"],
                                         split_size=c["split"], sm_scale=c["D"] ** -0.5,
                                         workspace=ws)]
        per = [1000.0 * _median_ms(f, stream, reps=reps) for f in ops]
        layer = 1000.0 * _median_ms(lambda: [f() for f in ops], stream, reps=reps)
        res["b%d" % m] = {"rmsnorm_us": per[0], "gemm_us": per[1], "decode_us": per[2],
                          "layer_us": layer}
        # the same three calls captured once in a CUDA graph and replayed: what
        # is left of the launch latency
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for f in ops:
                    f()
            res["b%d" % m]["layer_us_graph"] = 1000.0 * _median_ms(g.replay, stream, reps=reps)
        except RuntimeError as e:  # capture refused: report why, keep the eager figures
            res["b%d" % m]["layer_us_graph"] = None
            res["b%d" % m]["graph_error"] = str(e).splitlines()[0][:200]
    return res


def prefill_schedules(dev, stream, flush):
    """The chunked-prefill workload: one 8192-token prompt (32/8 heads, D=128,
    split 256) as chunks of 512, 2048 and 8192 and as token-by-token decode;
    milliseconds for the whole prompt's attention under each schedule (L2
    flushed before the first call of each) and TFLOP/s of the causal work."""
    import invariant_bi_rmsnorm_02_gb300 as bi
    from invariant_bi_rmsnorm_02_gb300 import synth
    c = synth.CHUNKED_PREFILL
    T, d = c["T"], DEC
    kv = synth.paged_kv([T], c["Hkv"], c["D"], c["page"], SEEDS["schedules"]["kv"], device=dev)
    q = synth.normal_bf16((T, c["Hq"], c["D"]), SEEDS["schedules"]["q"], device=dev)
    out = torch.empty_like(q)
    scale = c["D"] ** -0.5
    flops = 4.0 * c["Hq"] * c["D"] * T * (T + 1) / 2.0
    res = {}
    for chunk in c["chunks"]:
        cus = [torch.tensor([0, chunk], dtype=torch.int32, device=dev)]
        starts = [torch.tensor([a], dtype=torch.int32, device=dev) for a in range(0, T, chunk)]
        kls = [torch.tensor([a + chunk], dtype=torch.int32, device=dev)
               for a in range(0, T, chunk)]

        def run(chunk=chunk, starts=starts, kls=kls):
            for i, a in enumerate(range(0, T, chunk)):
                bi.bi_attn_prefill_chunk(q[a:a + chunk], cus[0], starts[i], kv.k_cache,
                                         kv.v_cache, kv.block_table, kls[i],
                                         out[a:a + chunk], None, max_q_len=chunk,
                                         max_kv_len=a + chunk, split_size=c["split"],
                                         sm_scale=scale)
        ms = _median_ms(run, stream, flush, reps=2)
        res["chunk%d" % chunk] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                                  "calls": T // chunk}
    ws = torch.empty(bi.bi_attn_decode_workspace_size(1, c["Hq"], c["Hkv"], c["D"], T,
                                                      c["split"]) // 4 + 4,
                     dtype=torch.float32, device=dev)
    kl = torch.arange(1, T + 1, dtype=torch.int32, device=dev)

    def tokens():
        for p in range(T):
            bi.bi_attn_decode(q[p:p + 1], kv.k_cache, kv.v_cache, kv.block_table,
                              kl[p:p + 1], out[p:p + 1], max_kv_len=p + 1,
                              split_size=c["split"], sm_scale=scale, workspace=ws)
    ms = _median_ms(tokens, stream, flush, reps=1)
    res["token_by_token"] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12, "calls": T}
    return res


def rmsnorm_beyond_l2(dev, stream, flush, peaks, rows=32768):
    """RMSNorm at 32768 x 4096: input and output (268 MB each) both exceed
    the 129 MB L2, so the output's bytes are written to HBM inside the
    timed region, not left dirty in L2."""
    import invariant_bi_rmsnorm_02_gb300 as bi
    from invariant_bi_rmsnorm_02_gb300 import synth
    x = synth.normal_bf16((rows, H), 5001, device=dev)
    w = synth.normal_bf16((H,), 5002, std=0.1, mean=1.0, device=dev)
    y = torch.empty_like(x)
    ms = _median_ms(lambda: bi.bi_rmsnorm(x, w, y, EPS), stream, flush, reps=5)
    gbs = (2 * rows * H * 2 + H * 2) / (ms * 1e-3) / 1e9
    return {"rows": rows, "us": 1000.0 * ms, "gbs": gbs, "frac_hbm": gbs / peaks["hbm"]}


def sig(v, n=3):
    """Floats rounded to n significant digits, recursively (a short line)."""
    if isinstance(v, float):
        return v if (v == 0.0 or v != v or v in (float("inf"), float("-inf"))) else float(
            "%.*g" % (n, v))
    if isinstance(v, dict):
        return {k: sig(x, n) for k, x in v.items()}
    if isinstance(v, (list, tuple)):
        return [sig(x, n) for x in v]
    return v


# ----------------------------------------------------------------- main arm
def max_over_ranks(vals, dist=None, device="cpu"):
    """The max over ranks of each timed quantity (every rank gets the result;
    one process: the values themselves)."""
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def whole_job_tflops(world, flops_per_rank, ms_max):
    """Throughput of the whole job: every rank's work over the slowest rank's
    time (replicas process the same amount each: weak scaling)."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the tiny-layer, prefill-schedule and large-RMSNorm figures")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    def barrier():
        if dist is not None:
            dist.barrier()

    import invariant_bi_rmsnorm_02_gb300 as bi
    bi.load()
    peaks = load_peaks()
    reserve = 2 * (args.warmup + args.steps) + 8
    wl = Workload(dev, rank, reserve)
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(dev)

    # clocks over every timed region of the device-side measurement
    with ClockSampler(local) as clk:
        inv, inv_step = timed_steps(wl, bi.INVARIANT, args.steps, args.warmup, flush, stream,
                                    barrier)
        var, var_step = timed_steps(wl, bi.VARIANT, args.steps, args.warmup, flush, stream,
                                    barrier)
        sweep = gemm_m_sweep(wl, flush, stream)
        extra = {}
        if not args.no_extras:
            extra["tiny_layer"] = tiny_layer(dev, stream)
            extra["prefill_8192"] = prefill_schedules(dev, stream, flush)
            extra["rmsnorm_32768"] = rmsnorm_beyond_l2(dev, stream, flush, peaks)
    status = bi.bi_check_device_errors()
    if status != bi.OK:
        raise RuntimeError("device error during the bench: %s" % bi.bi_status_string(status))
    work = wl.work(args.steps)
    gemm_flops = work["gemm_qkv"]["flops"] + work["gemm_up"]["flops"]
    gemm_ms = inv["gemm_qkv"] + inv["gemm_up"]
    # max over ranks of the timed quantities
    gemm_ms_max, step_ms_max = max_over_ranks([gemm_ms, inv_step], dist, dev)
    value = whole_job_tflops(world, gemm_flops, gemm_ms_max)

    e2e = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = e2e_steps(wl, max(3, args.steps // 2), args.warmup, stream)
        (e2e_ms_max,) = max_over_ranks([e2e_ms], dist, dev)
        e2e = {"value": round(whole_job_tflops(world, gemm_flops, e2e_ms_max), 1),
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_ms_max, 4)}

    # kernels are timed one at a time after an L2 flush, at the clock the
    # chip runs a lone kernel at: the burst tensor peak is their ceiling
    comps = {}
    for n in inv:
        wk = work[n]
        c = {"us": 1000.0 * inv[n], "us_var": 1000.0 * var[n], "slow": inv[n] / var[n] - 1.0}
        if "flops" in wk and n in ("gemm_qkv", "gemm_up", "prefill"):
            c["tflops"] = wk["flops"] / (inv[n] * 1e-3) / 1e12
            c["frac_bf16"] = c["tflops"] / peaks["bf16"]
        elif "bytes" in wk:
            c["gbs"] = wk["bytes"] / (inv[n] * 1e-3) / 1e9
            c["frac_hbm"] = c["gbs"] / peaks["hbm"]
        comps[n] = c
    dom = max(inv, key=lambda n: inv[n])
    if dom in ("gemm_qkv", "gemm_up"):
        kname, bound, unit = "gemm_tc_kernel", "tensor", "TFLOP/s"
        achieved, peak = comps[dom]["tflops"], peaks["bf16"]
    elif dom == "prefill":
        kname, bound, unit = "attn_prefill_kernel", "tensor", "TFLOP/s"
        achieved, peak = comps[dom]["tflops"], peaks["bf16"]
    else:
        kname = {"rmsnorm": "rmsnorm_row_kernel",
                 "decode": "attn_decode_split_kernel"}.get(dom, dom)
        bound, unit, achieved, peak = "hbm", "GB/s", comps[dom]["gbs"], peaks["hbm"]
    traffic = profiled_traffic(kname) if kname in KERNEL_SOURCES else None
    roofline = {"bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kname,
                "op": dom, "peak_source": peaks["src"] + (
                    " burst bf16 (cuBLAS, kernel timed alone)" if unit == "TFLOP/s"
                    else " HBM copy")}

    launches = wl.launches() * args.steps
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms_max, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, N(0,1) K/V/Q)",
        "config": {"workload": WORKLOAD, "M": M, "hidden": H, "n_qkv": N_QKV, "n_up": N_UP,
                   "decode_requests": DEC["B"], "split_size": DEC["S"],
                   "prefill_chunk": PRE["chunk"], "mode": "invariant",
                   "l2": "flushed before every kernel (256 MB write, then 256 MB read of another "
                         "buffer); step time = sum of the kernels' times",
                   "parallelism": "replicas (dp%d, no collective on the data path)" % world},
        "fingerprint": fingerprint(dev, rank),
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "roofline": roofline,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = sig(cpu_baseline(wl))
    # the per-op figures last and short, so the end of the line carries them
    line["extra"] = sig(extra)
    line["components"] = sig(comps)
    line["invariant_slowdown"] = sig({
        "step": inv_step / var_step - 1.0,
        "gemm": gemm_ms / (var["gemm_qkv"] + var["gemm_up"]) - 1.0,
        "ms_per_step_variant": var_step,
        "gemm_by_m_us": {str(m): [1000.0 * r["qkv"]["ms"], 1000.0 * r["qkv"]["ms_variant"],
                                  1000.0 * r["up"]["ms"], 1000.0 * r["up"]["ms_variant"]]
                         for m, r in sweep.items()},
        "gemm_by_m_cols": "qkv inv, qkv var, up inv, up var (us)",
        "gemm_worst_over_m": max(r[k]["slowdown"] for r in sweep.values()
                                  for k in ("qkv", "up"))})
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
