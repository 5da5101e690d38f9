"""Continuous batching over a paged KV cache, and the replay check of its
output.

"Reproducible LLM Inference - Batch Invariance, the Cost of Determinism, and
Where Bitwise Identity Is Actually Required" (§6.1) places the problem in
continuous batching: the set of requests that share a forward step follows
the traffic, so without batch-invariant kernels a request's tokens depend on
who else is being served.  "LLM Inference Reproducibility in Production"
compares replays token by token and reports the first position where two runs
part.  This module provides both halves:

* ``Scheduler`` admits requests as they arrive, reserves their KV pages from a
  ``PagePool``, and each step packs one decode token for every running
  sequence plus chunks of pending prompts into a token budget (chunked
  prefill), calls the model's step function and appends the chosen tokens;
* ``first_divergence`` / ``assert_reproducible`` compare token sequences of
  several runs.

The scheduler is plain host logic; the model is any callable taking a
``StepPlan`` and returning the chosen tokens, so the logic is testable
without a GPU.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .decoder import StepPlan


@dataclass
class Request:
    rid: int
    prompt: np.ndarray
    max_new_tokens: int
    arrival: int = 0            # the step at which the request becomes visible
    temperature: float = 0.0    # 0: greedy
    seed: int = 0


class PagePool:
    """Free list of KV-cache page ids (the same ids in every layer)."""

    def __init__(self, num_pages: int):
        self.num_pages = num_pages
        self.free = list(range(num_pages - 1, -1, -1))

    @property
    def available(self) -> int:
        return len(self.free)

    def alloc(self, n: int):
        if n > len(self.free):
            return None
        pages = [self.free.pop() for _ in range(n)]
        return pages

    def release(self, pages) -> None:
        self.free.extend(reversed(pages))


@dataclass
class _Seq:
    req: Request
    pages: list
    tokens: list
    n_prompt: int
    n_cached: int = 0                      # tokens whose K/V are in the cache
    generated: list = field(default_factory=list)


@dataclass
class StepRecord:
    decode_tokens: int
    prefill_tokens: int
    sequences: int


class Scheduler:
    """Continuous-batching scheduler.

    ``max_seqs`` bounds the running sequences, ``token_budget`` the tokens of
    one step (decode tokens are served first, prompts fill the rest in
    admission order), ``prefill_chunk`` optionally caps one prompt's share of
    a step.  A request reserves the pages for its prompt and all its new
    tokens when it is admitted (no preemption); requests are admitted in
    arrival order as pages and sequence slots allow.
    """

    def __init__(self, step_fn, *, page_size: int, max_blocks: int, num_pages: int,
                 max_seqs: int, token_budget: int, prefill_chunk: int | None = None):
        if token_budget < max_seqs:
            raise ValueError("the token budget must cover one decode token per sequence")
        self.step_fn = step_fn
        self.page_size, self.max_blocks = page_size, max_blocks
        self.pool = PagePool(num_pages)
        self.max_seqs, self.token_budget = max_seqs, token_budget
        self.prefill_chunk = prefill_chunk
        self.records: list[StepRecord] = []

    def _pages_for(self, req: Request) -> int:
        need = len(req.prompt) + req.max_new_tokens
        return -(-need // self.page_size)

    def run(self, requests) -> dict:
        """Serve every request to completion; returns {rid: generated tokens}."""
        waiting = sorted(requests, key=lambda r: (r.arrival, r.rid))
        for r in waiting:
            if len(r.prompt) < 1 or r.max_new_tokens < 1:
                raise ValueError("request %d: empty prompt or no tokens to generate" % r.rid)
            if self._pages_for(r) > min(self.max_blocks, self.pool.num_pages):
                raise ValueError("request %d does not fit the page table" % r.rid)
        running: list[_Seq] = []
        done: dict = {}
        step = 0
        while waiting or running:
            while (waiting and waiting[0].arrival <= step and len(running) < self.max_seqs):
                pages = self.pool.alloc(self._pages_for(waiting[0]))
                if pages is None:
                    break
                r = waiting.pop(0)
                running.append(_Seq(r, pages, [int(t) for t in r.prompt], len(r.prompt)))
            if not running:
                step = max(step + 1, waiting[0].arrival)
                continue
            plan, served = self._plan(running)
            chosen = self.step_fn(plan)
            for (seq, n_new, samples), tok in zip(served, _split(chosen, served)):
                seq.n_cached += n_new
                for t in tok:
                    seq.tokens.append(int(t))
                    seq.generated.append(int(t))
            for seq in list(running):
                if len(seq.generated) >= seq.req.max_new_tokens:
                    done[seq.req.rid] = seq.generated[:seq.req.max_new_tokens]
                    self.pool.release(seq.pages)
                    running.remove(seq)
            step += 1
        return done

    def _plan(self, running):
        budget = self.token_budget
        dec = [s for s in running if s.n_cached == len(s.tokens) - 1 and s.n_cached >= s.n_prompt]
        pre = [s for s in running if s.n_cached < s.n_prompt]
        tokens, pos, row_seq, rows, kv_lens = [], [], [], [], []
        cu_q, q_start, sample_rows, temp, seed, counter = [0], [], [], [], [], []
        served = []
        for s in dec[:budget]:
            r = len(rows)
            tokens.append(s.tokens[-1])
            pos.append(s.n_cached)
            row_seq.append(r)
            rows.append(s)
            kv_lens.append(s.n_cached + 1)
            sample_rows.append(len(tokens) - 1)
            temp.append(s.req.temperature)
            seed.append(s.req.seed)
            counter.append(s.n_cached + 1)
            served.append((s, 1, 1))
        n_dec = len(rows)
        budget -= n_dec
        for s in pre:
            if budget <= 0:
                break
            n = min(s.n_prompt - s.n_cached, budget)
            if self.prefill_chunk:
                n = min(n, self.prefill_chunk)
            r = len(rows)
            tokens.extend(s.tokens[s.n_cached:s.n_cached + n])
            pos.extend(range(s.n_cached, s.n_cached + n))
            row_seq.extend([r] * n)
            rows.append(s)
            kv_lens.append(s.n_cached + n)
            cu_q.append(cu_q[-1] + n)
            q_start.append(s.n_cached)
            finishes = s.n_cached + n == s.n_prompt
            if finishes:
                sample_rows.append(len(tokens) - 1)
                temp.append(s.req.temperature)
                seed.append(s.req.seed)
                counter.append(s.n_prompt)
            served.append((s, n, 1 if finishes else 0))
            budget -= n
        table = np.zeros((len(rows), self.max_blocks), np.int32)
        for i, s in enumerate(rows):
            table[i, :len(s.pages)] = s.pages
        self.records.append(StepRecord(n_dec, len(tokens) - n_dec, len(rows)))
        plan = StepPlan(
            tokens=np.asarray(tokens, np.int32), pos=np.asarray(pos, np.int32),
            row_seq=np.asarray(row_seq, np.int32), table=table,
            kv_lens=np.asarray(kv_lens, np.int32), n_dec=n_dec,
            cu_q=np.asarray(cu_q, np.int32), q_start=np.asarray(q_start, np.int32),
            sample_rows=np.asarray(sample_rows, np.int32),
            temperature=np.asarray(temp, np.float32), seed=np.asarray(seed, np.uint64),
            counter=np.asarray(counter, np.uint64))
        return plan, served


def _split(chosen, served):
    out, i = [], 0
    for _, _, k in served:
        out.append(chosen[i:i + k])
        i += k
    if i != len(chosen):
        raise ValueError("the step returned %d tokens for %d samples" % (len(chosen), i))
    return out


# ------------------------------------------------------------------ replay check
def first_divergence(a, b):
    """Index of the first token where two sequences differ (a length
    difference counts at the shorter length), or None if they are equal."""
    n = min(len(a), len(b))
    for i in range(n):
        if a[i] != b[i]:
            return i
    return None if len(a) == len(b) else n


def assert_reproducible(runs: dict) -> None:
    """runs: {name: {rid: tokens}}.  Raises AssertionError naming the first
    request and position where any run departs from the first one."""
    names = list(runs)
    base = runs[names[0]]
    for name in names[1:]:
        other = runs[name]
        if set(other) != set(base):
            raise AssertionError("%s served requests %s, %s served %s"
                                 % (names[0], sorted(base), name, sorted(other)))
        for rid in sorted(base):
            d = first_divergence(base[rid], other[rid])
            if d is not None:
                raise AssertionError("request %d: %s and %s part at token %d (%r vs %r)"
                                     % (rid, names[0], name, d, base[rid][d:d + 4],
                                        other[rid][d:d + 4]))


def synthetic_requests(n: int, prompt_lo: int, prompt_hi: int, max_new_tokens: int, vocab: int,
                       seed: int, mean_gap: float = 1.0) -> list:
    """n requests with prompt lengths uniform in [prompt_lo, prompt_hi], token
    ids uniform over the vocabulary and arrival steps of a Poisson stream with
    ``mean_gap`` steps between arrivals (0: all at step 0)."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(prompt_lo, prompt_hi + 1, n)
    gaps = rng.exponential(mean_gap, n) if mean_gap > 0 else np.zeros(n)
    arrivals = np.floor(np.cumsum(gaps)).astype(int) - int(np.floor(gaps[0]))
    return [Request(rid=i, prompt=rng.integers(0, vocab, int(lens[i])).astype(np.int32),
                    max_new_tokens=max_new_tokens, arrival=int(arrivals[i]))
            for i in range(n)]
