"""The runtime on the GPU, and a plan following a changing batch.

The runtime test uses a model whose greedy output is known exactly: every
layer's projection matrices are zero, so a layer passes its input through
(h = x, y = h), and the LM head is the embedding shifted by one row, so the
largest logit of token t is t + 1 (a row's product with itself dominates its
products with the other random rows).  A request's outputs must then be
last_prompt_token + 1, + 2, ... (mod vocab): any slip in the token plumbing
(prompt rows, a decode row's previous output kept on the device, sampling,
read-back, end token) changes them."""
import numpy as np
import pytest
import torch

from nano_intra_device_gb300 import _lib, workload as wl
from oracle import layer as orc
from tests.helpers import f64, parity
from tests.serving import OracleServer, greedy, row_tokens, serving_model

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_plan_follows_a_smaller_batch():
    """One plan, created for a larger batch, runs a different structure after
    nf_plan_set_batch (fewer tokens, other prefill chunks) and matches the
    oracle; then switches back."""
    shape = wl.tiny_shape()
    big = wl.make_batch(shape, [17, 33, 48, 64, 20, 9], [32, 12], None, seed_bt=3, max_pages=8)
    small = wl.make_batch(shape, [5, 40], [7], None, seed_bt=4, max_pages=8)
    small.num_pages = big.num_pages  # one pool for both
    plan = _lib.Plan(shape, big, _lib.make_opts(big.n_tokens, [0, 20, big.n_tokens],
                                                executor=_lib.NF_EXEC_STREAMS, attn_sms=24,
                                                kv_chunk=32))
    w = wl.make_weights(shape, seed=5, gain_std=0.1)
    wd = {k: v.to(DEV) for k, v in w.items()}
    for batch, opts in ((small, None),
                        (small, _lib.make_opts(small.n_tokens, [0, 4, small.n_tokens],
                                               executor=_lib.NF_EXEC_STREAMS, attn_sms=24,
                                               kv_chunk=32)),
                        (big, None)):
        kp, vp = wl.make_pools(shape, batch, DEV, seed=6)
        x = wl.make_x(shape, batch.n_tokens, seed=7)
        w64 = orc.weights_f64(w)
        ex, em = (orc.layer_step(shape, w64, x, kp, vp, batch.block_table, batch.seq_lens,
                                 batch.q_lens, store=st) for st in (None, "bf16"))
        plan.set_batch(batch, opts)
        y = torch.empty(batch.n_tokens, shape.hidden, dtype=torch.bfloat16, device=DEV)
        _lib.layer_step(plan, wd, x.to(DEV), kp, vp, torch.from_numpy(batch.block_table).to(DEV),
                        torch.from_numpy(batch.seq_lens).to(DEV), y)
        plan.poll()
        assert plan.info()[1] == batch.n_tokens
        parity(f64(y), ex["y"], em["y"], f"y after set_batch ({batch.n_tokens} tokens)")
    with pytest.raises(_lib.NanoflowError):       # more tokens than the plan holds
        plan.set_batch(wl.make_batch(shape, [4] * 60, [], None, max_pages=8))
    plan.close()


def test_set_batch_calls_queued_behind_a_long_step():
    """The host runs three nf_plan_set_batch calls ahead of the stream (a long
    busy kernel holds it): each batch's staged tables are still the ones its
    own step reads, so every step equals that batch run alone on a fresh plan,
    bit for bit."""
    shape = wl.tiny_shape()
    batches = [wl.make_batch(shape, [17, 33, 48, 64, 20, 9], [32, 12], None, seed_bt=3, max_pages=8),
               wl.make_batch(shape, [5, 40], [7], None, seed_bt=4, max_pages=8),
               wl.make_batch(shape, [9, 9, 30], [20], None, seed_bt=5, max_pages=8)]
    for b in batches[1:]:
        b.num_pages = batches[0].num_pages  # one pool for all
    T = batches[0].n_tokens
    w = wl.make_weights(shape, seed=5, gain_std=0.1)
    wd = {k: v.to(DEV) for k, v in w.items()}
    inputs = []
    for i, b in enumerate(batches):
        kp, vp = wl.make_pools(shape, b, DEV, seed=20 + i)
        x = wl.make_x(shape, b.n_tokens, seed=30 + i).to(DEV)
        inputs.append((x, kp, vp, torch.from_numpy(b.block_table).to(DEV),
                       torch.from_numpy(b.seq_lens).to(DEV)))

    def opts_for(b):
        return _lib.make_opts(b.n_tokens, [0, b.n_tokens // 2, b.n_tokens],
                              executor=_lib.NF_EXEC_STREAMS, attn_sms=24, kv_chunk=32)

    alone = []
    for b, (x, kp, vp, bt, sl) in zip(batches, inputs):
        plan = _lib.Plan(shape, b, opts_for(b))
        kq, vq = kp.clone(), vp.clone()
        y = torch.empty(b.n_tokens, shape.hidden, dtype=torch.bfloat16, device=DEV)
        _lib.layer_step(plan, wd, x, kq, vq, bt, sl, y)
        plan.poll(wait=True)
        plan.close()
        alone.append(y)
    plan = _lib.Plan(shape, batches[0], opts_for(batches[0]))
    ys, pools = [], [(kp.clone(), vp.clone()) for (_, kp, vp, _, _) in inputs]
    torch.cuda.synchronize()
    torch.cuda._sleep(200_000_000)  # ~0.1 s of spinning ahead of every step below
    for b, (x, _, _, bt, sl), (kq, vq) in zip(batches, inputs, pools):
        plan.set_batch(b, opts_for(b))
        y = torch.empty(b.n_tokens, shape.hidden, dtype=torch.bfloat16, device=DEV)
        _lib.layer_step(plan, wd, x, kq, vq, bt, sl, y)
        ys.append(y)
    plan.poll(wait=True)
    plan.close()
    assert T == max(b.n_tokens for b in batches)
    for i, (y, ya) in enumerate(zip(ys, alone)):
        assert torch.equal(y, ya), f"batch {i} read another batch's staged tables"


def _successor_model(shape, n_layers, vocab):
    g = torch.Generator().manual_seed(1)
    H = shape.hidden
    embed = torch.randn(vocab, H, generator=g).to(torch.bfloat16)
    lm_head = torch.roll(embed, shifts=1, dims=0)          # lm_head[v] = embed[v - 1]
    norm_f = torch.ones(H, dtype=torch.bfloat16)
    layers = []
    for i in range(n_layers):
        w = wl.make_weights(shape, seed=10 + i)
        layers.append({k: (torch.zeros_like(v) if k.startswith("w_") else v).to(DEV)
                       for k, v in w.items()})
    return embed.to(DEV), norm_f.to(DEV), lm_head.to(DEV), layers


@pytest.mark.parametrize("replan", [0.1, -1.0])
def test_runtime_serves_requests_end_to_end(replan):
    shape = wl.tiny_shape()
    vocab, L, b_dense, max_pages, num_pages = 96, 2, 40, 8, 64
    embed, norm_f, lm_head, layers = _successor_model(shape, L, vocab)
    pools = [(torch.zeros(num_pages, shape.n_kv, 16, shape.head_dim, dtype=torch.bfloat16, device=DEV),
              torch.zeros(num_pages, shape.n_kv, 16, shape.head_dim, dtype=torch.bfloat16, device=DEV))
             for _ in range(L)]
    sa = _lib.StackArgs(embed, norm_f, lm_head, layers, pools)
    eos = 70
    rt = _lib.Runtime(shape, b_dense, 8, max_pages, num_pages, vocab, eos_token=eos,
                      replan_threshold=replan)
    rng = np.random.default_rng(2)
    reqs = []
    for i in range(14):
        plen = int(rng.integers(1, 60))
        prompt = rng.integers(0, vocab, plen).tolist()
        if i == 3:
            prompt[-1] = 66          # outputs 67, 68, 69, 70 = end token
        mn = int(rng.integers(1, 30))
        reqs.append((rt.submit(prompt, mn), prompt, mn))
    stream = torch.cuda.current_stream()
    replanned, sizes = 0, []
    for _ in range(500):
        b = rt.step(sa, stream)
        if b["n_tokens"] == 0:
            break
        replanned += b["replanned"]
        sizes.append(b["n_tokens"])
    rt.sync()
    for rid, prompt, mn in reqs:
        fin, toks = rt.result(rid)
        expect = [(prompt[-1] + 1 + i) % vocab for i in range(mn)]
        if eos in expect:
            expect = expect[: expect.index(eos) + 1]
        assert fin, rid
        assert toks == expect, (rid, toks, expect)
    assert rt.counts() == (0, 0, num_pages)
    assert max(sizes) == b_dense
    if replan >= 0:
        assert replanned >= 2      # the mix moved from prompts to decoding
    else:
        assert replanned == 0
    rt.close()


@pytest.mark.parametrize("replan", [0.1, -1.0])
def test_runtime_serves_a_real_model_like_the_oracle(replan):
    """A random-weight two-layer stack (non-zero projections, norm gains other
    than 1, an LM head with a clear top-1 margin) served by nf_runtime on the
    GPU.  After every iteration the batch the scheduler formed is replayed
    through the oracle's stack step with the oracle's own K/V pools (updated
    from the K/V it appends), on the tokens the GPU's decode rows consumed:
    the GPU's logits of the emitting rows match both oracles at the stated
    bounds, its greedy tokens equal the oracle's, and the runtime's final
    outputs are those tokens.  Prompt chunks continue over several iterations
    and decode rows read K/V appended in earlier ones (dropping that K/V moves
    these logits by 1.5 to 4)."""
    shape = wl.tiny_shape()
    vocab, n_layers, b_dense, max_pages, num_pages = 96, 2, 40, 8, 64
    model = serving_model(shape, n_layers, vocab, seed=0)
    embed, norm_f, lm_head, layers = model
    pools = [(torch.zeros(num_pages, shape.n_kv, 16, shape.head_dim, dtype=torch.bfloat16, device=DEV),
              torch.zeros(num_pages, shape.n_kv, 16, shape.head_dim, dtype=torch.bfloat16, device=DEV))
             for _ in range(n_layers)]
    sa = _lib.StackArgs(embed.to(DEV), norm_f.to(DEV), lm_head.to(DEV),
                        [{k: v.to(DEV) for k, v in w.items()} for w in layers], pools)
    rt = _lib.Runtime(shape, b_dense, 8, max_pages, num_pages, vocab, eos_token=-1,
                      replan_threshold=replan)
    rng = np.random.default_rng(2)
    prompts, n_out = {}, {}
    for _ in range(10):
        pl = int(rng.integers(1, 60))
        prompt = rng.integers(0, vocab, pl).tolist()
        mn = int(rng.integers(1, 20))
        rid = rt.submit(prompt, mn)
        prompts[rid], n_out[rid] = prompt, mn
    exact = OracleServer(shape, model, num_pages, max_pages)
    emul = OracleServer(shape, model, num_pages, max_pages, store="bf16")
    gen = {r: [] for r in prompts}
    stream = torch.cuda.current_stream()
    iters, replanned = 0, 0
    for _ in range(500):
        b = rt.step(sa, stream)
        if b["n_tokens"] == 0:
            break
        iters += 1
        replanned += b["replanned"]
        lg = f64(rt.logits())                       # waits for this iteration
        toks = row_tokens(b, prompts, gen)
        ex, em = exact.step(b, toks), emul.step(b, toks)
        if lg.size:
            parity(lg, ex, em, f"served logits, iteration {b['iteration']}")
            assert np.array_equal(greedy(lg), greedy(ex)), b["iteration"]
        emit = [t for t, e in enumerate(b["row_emit"]) if e]
        for j, t in enumerate(emit):
            gen[b["row_request"][t]].append(int(greedy(lg[j:j + 1])[0]))
    rt.sync()
    assert iters >= 10
    for rid in prompts:
        fin, toks = rt.result(rid)
        assert fin and toks == gen[rid][: n_out[rid]], rid
    assert rt.counts() == (0, 0, num_pages)
    if replan >= 0:
        assert replanned >= 2
    else:
        assert replanned == 0
    rt.close()
