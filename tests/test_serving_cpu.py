"""Host logic of continuous batching, without a GPU: a fake model that keeps a
paged token store and chooses each next token from the whole sequence it reads
back through the page table.  Any slip in page tables, positions, lengths,
chunk offsets or sample rows changes its output, which must equal generating
every request alone, under every batch mix."""
import numpy as np
import pytest

from invariant_bi_rmsnorm_02_gb300.serving import (PagePool, Request, Scheduler,
                                                   assert_reproducible, first_divergence,
                                                   synthetic_requests)

PAGE, VOCAB = 16, 1000


def next_token(seq):
    h = 0
    for i, t in enumerate(seq):
        h = (h * 1000003 + (i + 1) * (int(t) + 7)) % (2 ** 61 - 1)
    return h % VOCAB


class FakeModel:
    def __init__(self, num_pages):
        self.store = np.full((num_pages, PAGE), -1, np.int64)
        self.steps = 0

    def __call__(self, plan):
        self.steps += 1
        T = len(plan.tokens)
        assert T == len(plan.pos) == len(plan.row_seq)
        n_dec = plan.n_dec
        # decode rows: one token per sequence, at row r of the table
        assert list(plan.row_seq[:n_dec]) == list(range(n_dec))
        # the prefill chunks are laid out as cu_q says
        pre_rows = plan.row_seq[n_dec:]
        for j in range(len(plan.q_start)):
            a, b = plan.cu_q[j], plan.cu_q[j + 1]
            assert (pre_rows[a:b] == n_dec + j).all()
            assert list(plan.pos[n_dec + a:n_dec + b]) == list(range(plan.q_start[j],
                                                                     plan.q_start[j] + b - a))
            assert plan.kv_lens[n_dec + j] == plan.q_start[j] + b - a
        # write every token where the page table puts it
        for t, p, r in zip(plan.tokens, plan.pos, plan.row_seq):
            self.store[plan.table[r, p // PAGE], p % PAGE] = t
        out = []
        for row in plan.sample_rows:
            r, p = plan.row_seq[row], plan.pos[row]
            assert plan.kv_lens[r] == p + 1
            seq = [self.store[plan.table[r, i // PAGE], i % PAGE] for i in range(p + 1)]
            assert min(seq) >= 0
            out.append(next_token(seq))
        return np.asarray(out, np.int32)


def alone(req):
    seq = list(req.prompt)
    gen = []
    for _ in range(req.max_new_tokens):
        t = next_token(seq)
        gen.append(t)
        seq.append(t)
    return gen


def serve(reqs, num_pages=4000, **kw):
    model = FakeModel(num_pages)
    sch = Scheduler(model, page_size=PAGE, max_blocks=64, num_pages=num_pages, **kw)
    return sch.run(reqs), sch


@pytest.mark.parametrize("kw", [dict(max_seqs=1, token_budget=1),
                                dict(max_seqs=4, token_budget=64),
                                dict(max_seqs=16, token_budget=256, prefill_chunk=48),
                                dict(max_seqs=64, token_budget=4096)])
def test_scheduler_output_equals_serving_each_request_alone(kw):
    reqs = synthetic_requests(24, 16, 300, 12, VOCAB, seed=5, mean_gap=2.0)
    out, sch = serve(reqs, **kw)
    assert out == {r.rid: alone(r) for r in reqs}
    assert max(rec.sequences for rec in sch.records) <= kw["max_seqs"]
    assert all(rec.decode_tokens + rec.prefill_tokens <= kw["token_budget"]
               for rec in sch.records)
    assert sch.pool.available == 4000            # every page came back


def test_scheduler_mixes_decode_and_prefill_and_waits_for_pages():
    reqs = synthetic_requests(10, 100, 200, 20, VOCAB, seed=6, mean_gap=3.0)
    # a pool of 48 pages: fewer requests fit than the 8 sequence slots, so
    # admission waits for pages to come back
    out, sch = serve(reqs, num_pages=48, max_seqs=8, token_budget=64)
    assert out == {r.rid: alone(r) for r in reqs}
    assert any(rec.decode_tokens and rec.prefill_tokens for rec in sch.records)
    fewest = min(-(-(len(r.prompt) + 20) // PAGE) for r in reqs)
    assert max(rec.sequences for rec in sch.records) <= 48 // fewest < 8


def test_scheduler_rejects_requests_that_cannot_fit():
    big = Request(rid=0, prompt=np.zeros(2000, np.int32), max_new_tokens=10)
    with pytest.raises(ValueError):
        serve([big], num_pages=4000, max_seqs=4, token_budget=64)   # > 64 pages of 16
    with pytest.raises(ValueError):
        serve([Request(rid=1, prompt=np.zeros(0, np.int32), max_new_tokens=3)], max_seqs=1,
              token_budget=8)


def test_page_pool_hands_out_distinct_pages():
    pool = PagePool(10)
    a, b = pool.alloc(4), pool.alloc(6)
    assert sorted(a + b) == list(range(10)) and pool.alloc(1) is None
    pool.release(a)
    assert pool.available == 4 and sorted(pool.alloc(4)) == sorted(a)


def test_replay_checker():
    assert first_divergence([1, 2, 3], [1, 2, 3]) is None
    assert first_divergence([1, 2, 3], [1, 5, 3]) == 1
    assert first_divergence([1, 2], [1, 2, 3]) == 2
    assert_reproducible({"a": {0: [1, 2], 1: [3]}, "b": {0: [1, 2], 1: [3]}})
    with pytest.raises(AssertionError, match="request 1: a and b part at token 0"):
        assert_reproducible({"a": {0: [1, 2], 1: [3]}, "b": {0: [1, 2], 1: [4]}})


def test_synthetic_requests_follow_the_recipe():
    reqs = synthetic_requests(200, 16, 4096, 256, 128256, seed=7, mean_gap=1.5)
    lens = np.array([len(r.prompt) for r in reqs])
    assert lens.min() >= 16 and lens.max() <= 4096
    assert all(r.prompt.max() < 128256 for r in reqs)
    arr = np.array([r.arrival for r in reqs])
    assert arr[0] == 0 and (np.diff(arr) >= 0).all()
    assert synthetic_requests(5, 16, 32, 4, 100, seed=7)[3].prompt.tolist() == \
        synthetic_requests(5, 16, 32, 4, 100, seed=7)[3].prompt.tolist()
