"""The runtime's scheduler on the host (no GPU): batch formation against an
independent restatement of the pages' rules ("NanoFlow: Towards Optimal LLM
Serving Throughput", "The NanoFlow Runtime System": constant dense batch,
decode requests first, prompts chunked first come first served to fill the
rest; asynchronous scheduling with the end-of-sequence check one iteration
late), KV page accounting and request lifecycles."""
import numpy as np
import pytest

from nano_intra_device_gb300 import _lib, workload as wl

P = 16


class RefScheduler:
    """The batch-formation rules restated in Python from the pages, for
    comparison with the library's scheduler."""

    def __init__(self, b_dense, max_requests):
        self.b, self.max_req = b_dense, max_requests
        self.reqs = {}
        self.waiting, self.active = [], []

    def submit(self, rid, prompt_len, max_new):
        self.reqs[rid] = dict(plen=prompt_len, max_new=max_new, done=0, sched=0, out=0,
                              finished=False, kv=0)
        self.waiting.append(rid)

    def form(self):
        rows = []      # (request, position, is_prompt_row, emit)
        dec = []
        for rid in self.active:
            r = self.reqs[rid]
            if r["finished"] or r["done"] < r["plen"] or r["sched"] < 1 or r["sched"] >= r["max_new"]:
                continue
            if len(dec) == self.b:
                break
            dec.append(rid)
        cap = self.b - len(dec)
        chunks = []
        for rid in list(self.active):
            r = self.reqs[rid]
            if cap and not r["finished"] and r["done"] < r["plen"]:
                c = min(r["plen"] - r["done"], cap)
                chunks.append((rid, c))
                cap -= c
        while cap and self.waiting and len(self.active) < self.max_req:
            rid = self.waiting.pop(0)
            r = self.reqs[rid]
            c = min(r["plen"], cap)
            chunks.append((rid, c))
            cap -= c
            self.active.append(rid)
        for rid in dec:
            r = self.reqs[rid]
            rows.append((rid, r["kv"], False, 1))
            r["kv"] += 1
            r["sched"] += 1
        for rid, c in chunks:
            r = self.reqs[rid]
            last = r["done"] + c == r["plen"]
            for i in range(c):
                rows.append((rid, r["done"] + i, True, int(last and i == c - 1)))
            r["done"] += c
            r["kv"] = r["done"]
            if last:
                r["sched"] = 1
        return rows, len(dec), [c for _, c in chunks]

    def apply(self, rows, sampled, eos):
        for (rid, _, _, emit), tok in zip(rows, sampled):
            r = self.reqs[rid]
            if not emit or r["finished"]:
                continue
            r["out"] += 1
            if tok == eos or r["out"] >= r["max_new"]:
                r["finished"] = True
                self.active.remove(rid)


def _token(rid, k):
    return (7 * rid + 3 * k + 1) % 90


def _drive(b_dense, max_requests, reqs, eos_at, num_pages=4096, max_pages=64):
    """Run the library scheduler and the restatement side by side, results of
    iteration i given back after iteration i+1 is formed (the asynchronous
    order).  reqs: list of (prompt_len, max_new); eos_at[rid] = output index
    whose token is the end token (99)."""
    shape = wl.tiny_shape()
    rt = _lib.Runtime(shape, b_dense, max_requests, max_pages, num_pages, 104, eos_token=99,
                      host_only=True)
    ref = RefScheduler(b_dense, max_requests)
    rng = np.random.default_rng(0)
    for i, (pl, mn) in enumerate(reqs):
        prompt = rng.integers(0, 90, pl).tolist()
        assert rt.submit(prompt, mn) == i
        ref.submit(i, pl, mn)
    emitted = {i: 0 for i in range(len(reqs))}
    history, pending = [], []
    for it in range(10000):
        b = rt.form()
        rows, n_dec, chunks = ref.form()
        assert b["iteration"] == it
        assert b["row_request"] == [r[0] for r in rows]
        assert b["row_pos"] == [r[1] for r in rows]
        assert b["row_emit"] == [r[3] for r in rows]
        assert b["n_decode"] == n_dec and b["prefill_q_lens"] == chunks
        assert all((tok >= 0) == is_prompt for tok, (_, _, is_prompt, _) in zip(b["row_token"], rows))
        history.append(b)
        sampled = []
        for rid, emit in zip(b["row_request"], b["row_emit"]):
            if emit:
                k = emitted[rid]
                emitted[rid] += 1
                sampled.append(99 if eos_at.get(rid) == k else _token(rid, k))
            else:
                sampled.append(-1)
        pending.append((b, rows, sampled))
        if len(pending) == 2:      # iteration i's tokens arrive once i+1 is formed
            ob, orows, osamp = pending.pop(0)
            rt.apply(ob["iteration"], osamp)
            ref.apply(orows, osamp, 99)
        if b["n_tokens"] == 0 and not pending:
            break
        if b["n_tokens"] == 0:
            ob, orows, osamp = pending.pop(0)
            rt.apply(ob["iteration"], osamp)
            ref.apply(orows, osamp, 99)
    return rt, history


def test_batches_follow_the_rules_and_keep_b_dense():
    rng = np.random.default_rng(1)
    reqs = [(int(rng.integers(1, 90)), int(rng.integers(1, 12))) for _ in range(40)]
    rt, hist = _drive(64, 16, reqs, eos_at={3: 2, 7: 0, 11: 5})
    # the budget is met exactly while prompts are waiting
    total_prompt = sum(p for p, _ in reqs)
    seen_prompt = 0
    for b in hist:
        seen_prompt += sum(1 for t in b["row_token"] if t >= 0)
        if seen_prompt < total_prompt - 64:
            assert b["n_tokens"] == 64
        # decode rows first, one per request; rows of a sequence are contiguous
        nd = b["n_decode"]
        assert all(t == -1 for t in b["row_token"][:nd])
        assert len(set(b["row_request"][:nd])) == nd
    for rid, (pl, mn) in enumerate(reqs):
        fin, toks = rt.result(rid)
        assert fin
        if rid in (3, 7, 11):
            k = {3: 2, 7: 0, 11: 5}[rid]
            assert toks[-1] == 99 and len(toks) == min(k + 1, mn) if k < mn else len(toks) == mn
        else:
            assert len(toks) == mn and toks == [_token(rid, k) for k in range(mn)]
    w, a, f = rt.counts()
    assert (w, a, f) == (0, 0, 4096)   # every page back in the pool
    rt.close()


def test_end_token_costs_exactly_one_more_iteration():
    """A request whose k-th output is the end token (produced in iteration i)
    is still scheduled in i+1 (formed before the token is known) and never in
    i+2."""
    rt, hist = _drive(8, 4, [(3, 20), (3, 20)], eos_at={0: 4})
    iters = [b["iteration"] for b in hist if 0 in b["row_request"]]
    emits = [b for b in hist
             if any(e for r, e in zip(b["row_request"], b["row_emit"]) if r == 0)]
    # outputs 0..4 come from 5 emitting iterations; one more runs, then none
    fifth = emits[4]["iteration"]
    assert iters[-1] == fifth + 1
    fin, toks = rt.result(0)
    assert fin and toks[-1] == 99 and len(toks) == 5
    rt.close()


def test_block_tables_and_page_accounting():
    rng = np.random.default_rng(2)
    reqs = [(int(rng.integers(10, 70)), int(rng.integers(5, 30))) for _ in range(24)]
    shape = wl.tiny_shape()
    rt = _lib.Runtime(shape, 48, 12, 8, 96, 104, eos_token=-1, host_only=True)
    for i, (pl, mn) in enumerate(reqs):
        rt.submit(rng.integers(0, 100, pl).tolist(), mn)
    pending = []
    for it in range(2000):
        b = rt.form()
        ns = b["n_decode"] + b["n_prefill"]
        bt = np.array(b["block_table"], np.int64).reshape(ns, 8) if ns else np.zeros((0, 8))
        used = []
        seqs = []
        i = 0
        for s_ in range(ns):
            seqs.append(b["row_request"][i])
            q = 1 if s_ < b["n_decode"] else b["prefill_q_lens"][s_ - b["n_decode"]]
            L = b["seq_lens"][s_]
            pages = bt[s_][bt[s_] >= 0]
            assert (L + P - 1) // P <= len(pages) <= 8 and np.all(pages < 96)
            # positions of this step's rows lie inside the sequence's pages
            assert b["row_pos"][i + q - 1] == L - 1
            used += pages.tolist()
            i += q
        assert len(set(seqs)) == ns
        assert len(used) == len(set(used))      # no page shared between two sequences
        assert len(used) <= 96 - b["free_pages"]
        sampled = [1 if e else -1 for e in b["row_emit"]]
        pending.append((b["iteration"], sampled))
        if len(pending) == 2 or b["n_tokens"] == 0:
            itn, smp = pending.pop(0)
            rt.apply(itn, smp)
        if b["n_tokens"] == 0 and not pending:
            break
    assert rt.counts() == (0, 0, 96)
    for i, (_, mn) in enumerate(reqs):
        fin, toks = rt.result(i)
        assert fin and len(toks) == mn
    rt.close()


def test_runtime_rejects_bad_requests_and_out_of_order_results():
    rt = _lib.Runtime(wl.tiny_shape(), 16, 4, 4, 32, 104, host_only=True)
    with pytest.raises(_lib.NanoflowError):
        rt.submit([1] * 60, 10)           # 70 tokens > 4 pages of 16
    with pytest.raises(_lib.NanoflowError):
        rt.submit([200], 1)               # token outside the vocabulary
    rt.submit([1, 2, 3], 2)
    b0 = rt.form()
    rt.form()
    with pytest.raises(_lib.NanoflowError):
        rt.form()                         # iteration 0 still awaits its tokens
    rt.apply(b0["iteration"], [5 if e else -1 for e in b0["row_emit"]])
    with pytest.raises(_lib.NanoflowError):
        rt.apply(b0["iteration"], [5])    # given twice
    rt.close()


# ---------------------------------------------------------------- a real model
def _alone(shape, model, prompt, n_out, max_pages):
    """Greedy outputs of one request served alone: the whole prompt as one
    prefill chunk into fresh pools, then one decode step per output."""
    from tests.serving import OracleServer, greedy
    srv = OracleServer(shape, model, max_pages, max_pages)
    bt = list(range(max_pages))
    out, logits = [], []
    L = len(prompt)
    b = dict(n_decode=0, n_prefill=1, block_table=bt, seq_lens=[L], prefill_q_lens=[L],
             row_emit=[0] * (L - 1) + [1])
    lg = srv.step(b, prompt)
    out.append(int(greedy(lg)[0]))
    logits.append(lg[0])
    for i in range(1, n_out):
        b = dict(n_decode=1, n_prefill=0, block_table=bt, seq_lens=[L + i], prefill_q_lens=[],
                 row_emit=[1])
        lg = srv.step(b, [out[-1]])
        out.append(int(greedy(lg)[0]))
        logits.append(lg[0])
    return out, logits


def test_served_model_equals_each_request_served_alone():
    """A random-weight two-layer stack served through the scheduler (host-only
    runtime; the oracle computes every batch it forms, with its own K/V pools)
    gives every request exactly the greedy outputs, and to float64 rounding the
    logits, of the same request served alone.  Batches mix decode rows with
    prompt chunks that continue over several iterations, and decode rows read
    K/V appended in earlier iterations, so batching, chunking, page allocation
    and the one-iteration-late token arrival must all leave the arithmetic of
    each request unchanged."""
    from tests.serving import OracleServer, greedy, row_tokens, serving_model
    shape = wl.tiny_shape()
    vocab, n_layers, b_dense, max_pages, num_pages = 96, 2, 40, 8, 64
    model = serving_model(shape, n_layers, vocab, seed=0)
    rt = _lib.Runtime(shape, b_dense, 8, max_pages, num_pages, vocab, eos_token=-1, host_only=True)
    rng = np.random.default_rng(2)
    prompts, n_out = {}, {}
    for _ in range(10):
        pl = int(rng.integers(1, 60))
        prompt = rng.integers(0, vocab, pl).tolist()
        mn = int(rng.integers(1, 20))
        rid = rt.submit(prompt, mn)
        prompts[rid], n_out[rid] = prompt, mn
    srv = OracleServer(shape, model, num_pages, max_pages)
    gen = {r: [] for r in prompts}
    glog = {r: [] for r in prompts}
    pending, continued, cross_iter_decode = [], 0, 0
    for _ in range(1000):
        b = rt.form()
        if b["n_tokens"]:
            toks = row_tokens(b, prompts, gen)
            lg = srv.step(b, toks)
            emit = [t for t, e in enumerate(b["row_emit"]) if e]
            sampled = [-1] * b["n_tokens"]
            for j, t in enumerate(emit):
                rid = b["row_request"][t]
                gen[rid].append(int(greedy(lg[j:j + 1])[0]))
                glog[rid].append(lg[j])
                sampled[t] = gen[rid][-1]
            nd = b["n_decode"]
            continued += sum(1 for t in range(nd, b["n_tokens"])
                             if b["row_token"][t] >= 0 and b["row_pos"][t] > 0
                             and (t == nd or b["row_request"][t - 1] != b["row_request"][t]))
            cross_iter_decode += nd
            pending.append((b["iteration"], sampled))
        if len(pending) == 2 or (b["n_tokens"] == 0 and pending):
            itn, smp = pending.pop(0)
            rt.apply(itn, smp)
        if b["n_tokens"] == 0 and not pending:
            break
    assert continued >= 3 and cross_iter_decode >= 20     # the batches exercise both
    for rid in prompts:
        fin, toks = rt.result(rid)
        assert fin and toks == gen[rid][: n_out[rid]]
        want, wlog = _alone(shape, model, prompts[rid], n_out[rid], max_pages)
        assert toks == want, rid
        np.testing.assert_allclose(np.stack(glog[rid][: n_out[rid]]), np.stack(wlog),
                                   rtol=1e-9, atol=1e-9)
    rt.close()
