"""Serving replay check at full scale: one random-init Llama-3-8B-shaped
decoder serves the same synthetic requests under several batch mixes and the
token sequences are compared request by request (the replay comparison of
"LLM Inference Reproducibility in Production"; the claim under test is §5.1 of
"Reproducible LLM Inference - Batch Invariance, the Cost of Determinism, and
Where Bitwise Identity Is Actually Required": with batch-invariant kernels a
request's output does not depend on the batch around it).

    python -m invariant_bi_rmsnorm_02_gb300.replay            # 256 requests
    python -m invariant_bi_rmsnorm_02_gb300.replay --requests 32 --new-tokens 64

Mixes: every request at step 0 with all slots open; Poisson arrivals into
fewer slots and a smaller token budget; and a few requests served alone.
With ``--variant`` the first two mixes are also run on the batch-variant
kernels, whose tokens are expected to part.  Prints one JSON line per mix and
a summary line; exits 1 if an invariant run differs.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import sys
import time

import torch

from . import _binding as bi
from .decoder import LLAMA3_8B, Decoder, DecoderWeights
from .serving import Scheduler, first_divergence, synthetic_requests


def run_mix(dec, reqs, **kw):
    sch = Scheduler(dec.step, page_size=dec.cfg.page_size, max_blocks=dec.max_blocks,
                    num_pages=dec.num_pages, **kw)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    out = sch.run(reqs)
    torch.cuda.synchronize()
    secs = time.perf_counter() - t0
    status = bi.bi_check_device_errors()
    if status != bi.OK:
        raise bi.BiError(status, "device error during serving")
    rec = sch.records
    gen = sum(len(t) for t in out.values())
    return out, {
        "seconds": round(secs, 3), "steps": len(rec),
        "prefill_tokens": int(sum(r.prefill_tokens for r in rec)),
        "decode_tokens": int(sum(r.decode_tokens for r in rec)),
        "generated_tokens": int(gen), "generated_tokens_per_s": round(gen / secs, 1),
        "max_sequences_in_a_step": int(max(r.sequences for r in rec)),
        "distinct_step_shapes": len({(r.decode_tokens, r.prefill_tokens) for r in rec}),
    }


def compare(base, other):
    """Requests whose tokens differ, and the earliest token where one does."""
    parted = {rid: first_divergence(base[rid], other[rid]) for rid in other}
    parted = {rid: d for rid, d in parted.items() if d is not None}
    return {"requests_compared": len(other), "requests_differing": len(parted),
            "earliest_difference": min(parted.values()) if parted else None}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--requests", type=int, default=256)
    ap.add_argument("--prompt-lo", type=int, default=16)
    ap.add_argument("--prompt-hi", type=int, default=4096)
    ap.add_argument("--new-tokens", type=int, default=256)
    ap.add_argument("--layers", type=int, default=LLAMA3_8B.layers)
    ap.add_argument("--alone", type=int, default=4, help="requests also served one at a time")
    ap.add_argument("--token-budget", type=int, default=8192)
    ap.add_argument("--seed", type=int, default=5)
    ap.add_argument("--variant", action="store_true", help="also run the batch-variant kernels")
    a = ap.parse_args(argv)

    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = dataclasses.replace(LLAMA3_8B, layers=a.layers)
    reqs = synthetic_requests(a.requests, a.prompt_lo, a.prompt_hi, a.new_tokens, cfg.vocab,
                              seed=a.seed, mean_gap=2.0)
    burst = [dataclasses.replace(r, arrival=0) for r in reqs]
    per_req = [-(-(len(r.prompt) + r.max_new_tokens) // cfg.page_size) for r in reqs]
    max_blocks = max(per_req)
    num_pages = sum(per_req) + 16
    budget = max(a.token_budget, a.requests)
    t0 = time.perf_counter()
    w = DecoderWeights(cfg, a.seed, dev)
    dec = Decoder(cfg, w, num_pages=num_pages, max_tokens=budget, max_seqs=a.requests,
                  max_blocks=max_blocks, device=dev, use_graphs=True)
    dec.use_graphs = False  # eager unless a mix asks for graphs
    setup = time.perf_counter() - t0
    half = max(1, a.requests // 2)
    mixes = [("burst, %d slots, budget %d" % (a.requests, budget), burst,
              dict(max_seqs=a.requests, token_budget=budget)),
             ("arrivals, %d slots, budget %d, chunks of 512" % (half, max(half, budget // 4)),
              reqs, dict(max_seqs=half, token_budget=max(half, budget // 4), prefill_chunk=512))]
    runs, ok = {}, True
    base_name = mixes[0][0]
    for name, rq, kw in mixes:
        out, stats = run_mix(dec, rq, **kw)
        runs[name] = out
        line = {"mode": "invariant", "mix": name, **stats}
        if name != base_name:
            line.update(compare(runs[base_name], out))
            ok &= line["requests_differing"] == 0
        print(json.dumps(line), flush=True)
    if a.alone:
        sub = [dataclasses.replace(r, arrival=0) for r in reqs[:a.alone]]
        for graphs in (False, True):
            dec.use_graphs = graphs
            out, stats = run_mix(dec, sub, max_seqs=1, token_budget=budget)
            line = {"mode": "invariant",
                    "mix": "%d requests alone%s" % (len(sub), ", decode steps from CUDA graphs"
                                                    if graphs else ""),
                    **stats, **compare(runs[base_name], out)}
            if graphs:
                line["graph_replays"] = dec.graph_replays
            ok &= line["requests_differing"] == 0
            print(json.dumps(line), flush=True)
        dec.use_graphs = False
    if a.variant:
        dec.mode = bi.VARIANT
        vruns = {}
        for name, rq, kw in mixes:
            vruns[name], stats = run_mix(dec, rq, **kw)
            line = {"mode": "variant", "mix": name, **stats}
            if name != base_name:
                line.update(compare(vruns[base_name], vruns[name]))
            line["vs_invariant_same_mix"] = compare(runs[name], vruns[name])
            print(json.dumps(line), flush=True)
        dec.mode = bi.INVARIANT
    print(json.dumps({"summary": "identical under every batch mix" if ok else "DIFFERENT",
                      "requests": a.requests, "prompt_len": [a.prompt_lo, a.prompt_hi],
                      "new_tokens": a.new_tokens, "layers": a.layers,
                      "kv_pages": num_pages, "setup_seconds": round(setup, 2)}), flush=True)
    return 0 if ok else 1


if __name__ == "__main__":
    sys.exit(main())
