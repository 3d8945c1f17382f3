"""Pins for the CPU oracle: closed forms, invariants, brute force, special cases.

Each test checks the oracle against something other than itself, chosen so
that a plausible slip (a dropped term, a wrong sign or index, a transposed
operand, a wrong GQA grouping, a wrong page/slot mapping) fails at least one.
"""
import math

import numpy as np
import pytest
import torch

from nano_intra_device_gb300 import workload as wl
from oracle import layer as orc


# ----------------------------------------------------------------- RMSNorm

def test_rmsnorm_constant_row_closed_form():
    H, c, eps = 64, 1.7, 1e-5
    g = np.linspace(0.5, 1.5, H)
    x = np.full((1, H), c)
    y = orc.rmsnorm(x, g, eps)
    np.testing.assert_allclose(y[0], g * c / math.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_zero_row_and_scale_invariance():
    rng = np.random.default_rng(0)
    g = rng.uniform(0.5, 2, 32)
    assert np.all(orc.rmsnorm(np.zeros((1, 32)), g, 1e-5) == 0)
    x = rng.standard_normal((3, 32))
    a = orc.rmsnorm(x, g, 0.0)
    b = orc.rmsnorm(7.5 * x, g, 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-13)
    # unit mean square after dividing out the gains
    np.testing.assert_allclose(np.mean((a / g) ** 2, axis=-1), 1.0, rtol=1e-13)


# -------------------------------------------------------------------- RoPE

def test_rope_position_zero_is_identity():
    u = np.random.default_rng(1).standard_normal((4, 3, 64))
    np.testing.assert_array_equal(orc.rope(u, np.zeros(4, np.int64), 1e4), u)


def test_rope_rotate_half_closed_form():
    d, theta = 8, 1e4
    for i in range(d // 2):
        for p in (1, 5, 123):
            u = np.zeros((1, 1, d))
            u[0, 0, i] = 1.0
            r = orc.rope(u, np.array([p]), theta)[0, 0]
            ang = p * theta ** (-2.0 * i / d)
            expect = np.zeros(d)
            expect[i] = math.cos(ang)
            expect[i + d // 2] = math.sin(ang)
            np.testing.assert_allclose(r, expect, atol=1e-15)


def test_rope_keeps_pair_norms_and_is_relative():
    rng = np.random.default_rng(2)
    d = 64
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))
    rq = orc.rope(q, np.array([37]), 1e4)
    half = d // 2
    np.testing.assert_allclose(rq[..., :half] ** 2 + rq[..., half:] ** 2,
                               q[..., :half] ** 2 + q[..., half:] ** 2, rtol=1e-12)
    dots = []
    for m, n in ((37, 11), (137, 111), (1037, 1011)):
        dots.append(float(np.sum(orc.rope(q, np.array([m]), 1e4) * orc.rope(k, np.array([n]), 1e4))))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-10)


# --------------------------------------------------------------- attention

def _brute_attention(q, K, V, n_q, n_kv):
    """Pure-Python softmax attention with explicit loops (tiny inputs)."""
    L, d = K.shape[0], q.shape[1]
    out = []
    for h in range(n_q):
        g = h * n_kv // n_q
        s = [sum(q[h, c] * K[j, g, c] for c in range(d)) / math.sqrt(d) for j in range(L)]
        mx = max(s)
        e = [math.exp(v - mx) for v in s]
        z = sum(e)
        out.append([sum(e[j] * V[j, g, c] for j in range(L)) / z for c in range(d)])
    return np.asarray(out)


def test_attention_matches_brute_force():
    rng = np.random.default_rng(3)
    for n_q, n_kv, L in ((4, 2, 7), (8, 8, 3), (4, 1, 11)):
        q = rng.standard_normal((n_q, 8))
        K = rng.standard_normal((L, n_kv, 8))
        V = rng.standard_normal((L, n_kv, 8))
        np.testing.assert_allclose(orc.attention_one(q, K, V, n_q, n_kv),
                                   _brute_attention(q, K, V, n_q, n_kv), rtol=1e-12, atol=1e-13)


def test_attention_matches_torch_sdpa_with_expanded_gqa():
    rng = np.random.default_rng(4)
    n_q, n_kv, L, d = 8, 2, 40, 16
    q = rng.standard_normal((n_q, d))
    K = rng.standard_normal((L, n_kv, d))
    V = rng.standard_normal((L, n_kv, d))
    grp = n_q // n_kv
    Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(grp, 0)   # [n_q, L, d]
    Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(grp, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None, :], Kt, Vt)[:, 0, :].numpy()
    np.testing.assert_allclose(orc.attention_one(q, K, V, n_q, n_kv), ref, rtol=1e-11, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(5)
    d = 16
    # one key: output is that key's value
    V = rng.standard_normal((1, 2, d))
    o = orc.attention_one(rng.standard_normal((4, d)), rng.standard_normal((1, 2, d)), V, 4, 2)
    np.testing.assert_allclose(o[:2], np.repeat(V[:, 0], 2, 0), rtol=1e-14)
    np.testing.assert_allclose(o[2:], np.repeat(V[:, 1], 2, 0), rtol=1e-14)
    # identical keys: mean of the values
    K = np.repeat(rng.standard_normal((1, 1, d)), 9, axis=0)
    V = rng.standard_normal((9, 1, d))
    o = orc.attention_one(rng.standard_normal((2, d)), K, V, 2, 1)
    np.testing.assert_allclose(o, np.repeat(V[:, 0].mean(0, keepdims=True), 2, 0), rtol=1e-12)
    # a large one-hot query picks the key with the largest matching coordinate
    K = rng.standard_normal((12, 1, d))
    q = np.zeros((1, d)); q[0, 3] = 1e4
    V = rng.standard_normal((12, 1, d))
    o = orc.attention_one(q, K, V, 1, 1)
    np.testing.assert_allclose(o[0], V[np.argmax(K[:, 0, 3]), 0], rtol=1e-9)


def test_attention_gqa_groups_are_contiguous():
    d, L = 8, 5
    K = np.zeros((L, 2, d))
    V = np.zeros((L, 2, d)); V[:, 1, :] = 1.0
    o = orc.attention_one(np.ones((4, d)), K, V, 4, 2)
    np.testing.assert_array_equal(o[:2], 0.0)   # heads 0,1 -> KV head 0
    np.testing.assert_array_equal(o[2:], 1.0)   # heads 2,3 -> KV head 1


# ---------------------------------------------------------- metadata, paging

def test_token_map_and_slots_roundtrip_contiguous():
    shape = wl.tiny_shape()
    b = wl.tiny_batch()
    P = shape.page_size
    # every (sequence, position) maps to a distinct slot inside its own pages,
    # and reading them back through the block table returns the logical order
    seen = set()
    for s in range(b.n_seq):
        L = int(b.seq_lens[s])
        pos = np.arange(L)
        sl = orc.slot_of(np.full(L, s), pos, b.block_table, P)
        own = set()
        for j in range((L + P - 1) // P):
            own.update(range(b.block_table[s, j] * P, b.block_table[s, j] * P + P))
        assert set(sl.tolist()) <= own
        assert len(set(sl.tolist())) == L
        assert not (seen & set(sl.tolist()))
        seen |= set(sl.tolist())
        # brute-force page walk
        for p in (0, L - 1, L // 2):
            page_list = [int(x) for x in b.block_table[s] if x >= 0]
            assert sl[p] == page_list[p // P] * P + (p % P)


def test_token_map_decode_and_prefill_positions():
    q_lens = np.array([1, 1, 5, 1, 3])
    seq_lens = np.array([10, 1, 12, 7, 3])
    seq, pos = orc.token_map(q_lens, seq_lens)
    assert seq.tolist() == [0, 1, 2, 2, 2, 2, 2, 3, 4, 4, 4]
    assert pos.tolist() == [9, 0, 7, 8, 9, 10, 11, 6, 0, 1, 2]


def test_split_kv_items_cover_each_row_once():
    ctx = np.array([1, 15, 16, 17, 512, 513, 1030])
    for chunk in (16, 64, 512):
        items = orc.split_kv_items(ctx, chunk)
        for t, L in enumerate(ctx.tolist()):
            mine = [(b, n) for (r, b, n) in items if r == t]
            assert len(mine) == math.ceil(L / chunk)
            cover = np.zeros(L, int)
            for b0, n in mine:
                assert 1 <= n <= chunk and b0 % chunk == 0
                cover[b0:b0 + n] += 1
            assert np.all(cover == 1)


# ------------------------------------------------------------ whole layer

def _tiny_inputs(gain_std=0.1, seed=0):
    shape = wl.tiny_shape()
    b = wl.tiny_batch()
    w = wl.make_weights(shape, seed=seed, gain_std=gain_std)
    x = wl.make_x(shape, b.n_tokens, seed=seed)
    k, v = wl.make_pools(shape, b, "cpu")
    return shape, b, w, x, k, v


def _brute_layer(shape, w, x, k_pool, v_pool, b, store=False, inter=None):
    """Independent float64 restatement of the layer on tiny inputs: complex
    rotation for RoPE, each sequence's full contiguous K/V rebuilt position by
    position, one dense masked softmax per sequence and head.  With store=True
    the stored tensors (n1, q and k after RoPE, v, o, h, n2, a) go through
    torch's own bf16 conversion (via float32) where they are produced; inter,
    if a dict, receives them."""
    H, nq, nkv, d, F, P = (shape.hidden, shape.n_q, shape.n_kv, shape.head_dim,
                           shape.ffn, shape.page_size)
    rnd = (lambda u: u.float().to(torch.bfloat16).double()) if store else (lambda u: u)
    inter = {} if inter is None else inter
    X = x.double()
    W = {kk: vv.double() for kk, vv in w.items()}
    n1 = rnd(X * torch.rsqrt((X * X).mean(-1, keepdim=True) + shape.rms_eps) * W["norm1"])
    proj = torch.einsum("th,rh->tr", n1, W["w_qkv"])
    q = proj[:, :nq * d].reshape(-1, nq, d)
    k = proj[:, nq * d:(nq + nkv) * d].reshape(-1, nkv, d)
    v = rnd(proj[:, (nq + nkv) * d:].reshape(-1, nkv, d))
    # positions
    pos, sid = [], []
    for s in range(b.n_seq):
        for i in range(int(b.q_lens[s])):
            pos.append(int(b.seq_lens[s]) - int(b.q_lens[s]) + i)
            sid.append(s)
    pos_t = torch.tensor(pos, dtype=torch.float64)
    half = d // 2
    freq = shape.rope_theta ** (-torch.arange(half, dtype=torch.float64) * 2 / d)
    rot = torch.polar(torch.ones(len(pos), half, dtype=torch.float64), pos_t[:, None] * freq)

    def cplx(u):
        z = torch.complex(u[..., :half], u[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], -1)
    q, k = rnd(cplx(q)), rnd(cplx(k))
    o = torch.zeros(len(pos), nq, d, dtype=torch.float64)
    for s in range(b.n_seq):
        L = int(b.seq_lens[s])
        cached = L - int(b.q_lens[s])
        toks = [t for t in range(len(pos)) if sid[t] == s]
        Kc = torch.zeros(L, nkv, d, dtype=torch.float64)
        Vc = torch.zeros(L, nkv, d, dtype=torch.float64)
        for p in range(L):
            if p < cached:
                pg = int(b.block_table[s, p // P])
                Kc[p] = k_pool[pg, :, p % P, :].double()
                Vc[p] = v_pool[pg, :, p % P, :].double()
            else:
                Kc[p] = k[toks[p - cached]]
                Vc[p] = v[toks[p - cached]]
        for h in range(nq):
            g = h // (nq // nkv)
            S = torch.stack([q[t, h] for t in toks]) @ Kc[:, g, :].T / math.sqrt(d)
            mask = torch.tensor([[j <= pos[t] for j in range(L)] for t in toks])
            S = S.masked_fill(~mask, -math.inf)
            o[toks, h] = torch.softmax(S, -1) @ Vc[:, g, :]
    o = rnd(o)
    hres = rnd(X + o.reshape(len(pos), nq * d) @ W["w_o"].T)
    n2 = rnd(hres * torch.rsqrt((hres * hres).mean(-1, keepdim=True) + shape.rms_eps) * W["norm2"])
    gu = n2 @ W["w_gate_up"].T
    a = rnd(torch.nn.functional.silu(gu[:, :F]) * gu[:, F:])
    y = hres + a @ W["w_down"].T
    inter.update(n1=n1.numpy(), q=q.numpy(), o=o.numpy(), h=hres.numpy(), n2=n2.numpy(),
                 a=a.numpy())
    return y.numpy(), k.numpy(), v.numpy()


def test_layer_matches_independent_brute_force():
    shape, b, w, x, kp, vp = _tiny_inputs()
    out = orc.layer_step(shape, orc.weights_f64(w), x, kp, vp, b.block_table, b.seq_lens, b.q_lens)
    y, k, v = _brute_layer(shape, w, x, kp, vp, b)
    np.testing.assert_allclose(out["y"], y, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(out["k_new"], k, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out["v_new"], v, rtol=1e-11, atol=1e-12)
    assert np.all(np.isfinite(out["y"]))


def test_bf16_rounding_matches_torch_and_the_definition():
    """oracle.bf16 against torch's float32 -> bfloat16 conversion (random
    normal values, exact ties between two bf16 neighbours, values near powers
    of two), and on float64 inputs against the definition: the nearer of the
    two bf16 neighbours, enumerated from the float32 bit pattern, ties to the
    even one."""
    rng = np.random.default_rng(0)
    vals = [rng.standard_normal(50000).astype(np.float32) * 8,
            ((rng.integers(0x0080, 0x7F7F, 20000).astype(np.uint32) << 16) | 0x8000).view(np.float32),
            ((rng.integers(0x0080, 0x7F7F, 20000).astype(np.uint32) << 16) | 0x7FFF).view(np.float32)]
    for v in vals:
        v = v * np.where(rng.random(v.shape) < 0.5, -1, 1).astype(np.float32)
        ref = torch.from_numpy(v).to(torch.bfloat16).double().numpy()
        assert np.array_equal(orc.bf16(v.astype(np.float64)), ref)
    # float64 inputs: brute force over the two neighbours
    x = rng.standard_normal(20000) * np.exp2(rng.integers(-20, 20, 20000))
    lo_bits = (np.abs(x).astype(np.float32).view(np.uint32) & 0xFFFF0000)   # truncate to bf16
    lo = lo_bits.view(np.float32).astype(np.float64)
    lo = np.where(lo > np.abs(x), (lo_bits - 0x10000).view(np.float32).astype(np.float64), lo)
    lo_bits = np.abs(lo).astype(np.float32).view(np.uint32)
    hi = (lo_bits + 0x10000).view(np.float32).astype(np.float64)
    a = np.abs(x)
    pick_hi = (hi - a < a - lo) | ((hi - a == a - lo) & ((lo_bits >> 16) & 1 == 1))
    want = np.sign(x) * np.where(pick_hi, hi, lo)
    assert np.array_equal(orc.bf16(x), want)
    assert orc.bf16(np.array([0.0]))[0] == 0.0


def test_layer_bf16_storage_matches_the_brute_force_with_torch_rounding():
    """store="bf16" rounds exactly the stored tensors, where they are produced:
    every intermediate it returns is a bf16 value and equals the independent
    restatement's, which rounds through torch's conversion (rare one-step
    differences allowed: torch rounds float64 via float32, and a difference
    propagates), and the output moves off the exact layer by the expected
    bf16-sized amount."""
    shape, b, w, x, kp, vp = _tiny_inputs()
    w64 = orc.weights_f64(w)
    ex = orc.layer_step(shape, w64, x, kp, vp, b.block_table, b.seq_lens, b.q_lens, keep=True)
    st = orc.layer_step(shape, w64, x, kp, vp, b.block_table, b.seq_lens, b.q_lens, keep=True,
                        store="bf16")
    inter = {}
    y, k, v = _brute_layer(shape, w, x, kp, vp, b, store=True, inter=inter)
    inter.update(k_new=k, v_new=v)
    for key in ("n1", "q", "k_new", "v_new", "o", "h", "n2", "a"):
        got = st[key].reshape(inter[key].shape)
        assert np.array_equal(orc.bf16(got), got), key            # stored values are bf16
        same = np.mean(got == inter[key])
        step = 2 * np.ldexp(1.0, np.frexp(np.abs(inter[key]))[1] - 9)
        assert same > 0.99 and np.all(np.abs(got - inter[key]) <= step + 1e-300), (key, same)
        assert not np.array_equal(got, ex[key].reshape(got.shape)), key   # rounding happened
    np.testing.assert_allclose(st["y"], y, rtol=0, atol=1e-3)
    d = st["y"] - ex["y"]
    rl = np.linalg.norm(d) / np.linalg.norm(ex["y"])
    assert 1e-5 < rl < 5e-3


def test_stack_bf16_storage_rounds_between_layers_only():
    """layers_step with store="bf16": the last layer's output is returned
    unrounded, the layers before hand the next a bf16 value (equal to running
    the layers one at a time, rounding in between)."""
    shape, b, w, x, kp, vp = _tiny_inputs()
    w2 = wl.make_weights(shape, seed=5, gain_std=0.1)
    k2, v2 = wl.make_pools(shape, b, "cpu", seed=8)
    L = [orc.weights_f64(w), orc.weights_f64(w2)]
    both = orc.layers_step(shape, L, x, [(kp, vp), (k2, v2)], b.block_table, b.seq_lens,
                           b.q_lens, store="bf16")
    one = orc.layer_step(shape, L[0], x, kp, vp, b.block_table, b.seq_lens, b.q_lens, store="bf16")
    two = orc.layer_step(shape, L[1], orc.bf16(one["y"]), k2, v2, b.block_table, b.seq_lens,
                         b.q_lens, store="bf16")
    assert np.array_equal(both["y"], two["y"])
    assert not np.array_equal(orc.bf16(two["y"]), two["y"])


def test_layer_zero_weights_is_identity_and_zero_gate_gives_h():
    shape, b, w, x, kp, vp = _tiny_inputs()
    w0 = {k: (torch.zeros_like(v) if k.startswith("w_") else v) for k, v in w.items()}
    out = orc.layer_step(shape, orc.weights_f64(w0), x, kp, vp, b.block_table, b.seq_lens, b.q_lens)
    np.testing.assert_array_equal(out["y"], orc.f64(x))
    wg = dict(w)
    gu = w["w_gate_up"].clone()
    gu[: shape.ffn] = 0
    wg["w_gate_up"] = gu
    out = orc.layer_step(shape, orc.weights_f64(wg), x, kp, vp, b.block_table, b.seq_lens,
                         b.q_lens, keep=True)
    np.testing.assert_array_equal(out["a"], 0.0)
    np.testing.assert_array_equal(out["y"], out["h"])


def test_layer_projection_orientation_one_hot():
    # x = e_j with unit gains and eps=0 gives n1 = sqrt(H) e_j, so the fused
    # projection returns sqrt(H) * column j of W_qkv split into q | k | v
    shape = wl.Shape(hidden=64, n_q=2, n_kv=1, head_dim=16, ffn=32, rms_eps=0.0)
    b = wl.make_batch(shape, [1], [], seed_bt=0)
    w = wl.make_weights(shape, seed=3)
    j = 5
    x = torch.zeros(1, 64, dtype=torch.bfloat16); x[0, j] = 1
    kp, vp = wl.make_pools(shape, b)
    out = orc.layer_step(shape, orc.weights_f64(w), x, kp, vp, b.block_table, b.seq_lens,
                         b.q_lens, keep=True)
    col = orc.f64(w["w_qkv"])[:, j] * 8.0      # sqrt(64); position 0 -> RoPE identity
    np.testing.assert_allclose(out["q"].reshape(-1), col[:32], rtol=1e-14)
    np.testing.assert_allclose(out["k_new"].reshape(-1), col[32:48], rtol=1e-14)
    np.testing.assert_allclose(out["v_new"].reshape(-1), col[48:], rtol=1e-14)
    # a single position: attention returns v, so o == v_new for both q heads
    np.testing.assert_allclose(out["o"][0, 0], out["v_new"][0, 0], rtol=1e-14)
    np.testing.assert_allclose(out["o"][0, 1], out["v_new"][0, 0], rtol=1e-14)


def test_layer_shuffled_block_table_invariance():
    shape, b, w, x, kp, vp = _tiny_inputs()
    w64 = orc.weights_f64(w)
    base = orc.layer_step(shape, w64, x, kp, vp, b.block_table, b.seq_lens, b.q_lens)
    perm = np.random.default_rng(9).permutation(b.num_pages)
    bt2 = np.where(b.block_table >= 0, perm[np.maximum(b.block_table, 0)], -1).astype(np.int32)
    kp2 = torch.empty_like(kp); vp2 = torch.empty_like(vp)
    kp2[torch.as_tensor(perm)] = kp
    vp2[torch.as_tensor(perm)] = vp
    out = orc.layer_step(shape, w64, x, kp2, vp2, bt2, b.seq_lens, b.q_lens)
    np.testing.assert_array_equal(out["y"], base["y"])
    np.testing.assert_array_equal(out["k_new"], base["k_new"])


def test_layer_rows_subset_equals_full():
    shape, b, w, x, kp, vp = _tiny_inputs()
    w64 = orc.weights_f64(w)
    full = orc.layer_step(shape, w64, x, kp, vp, b.block_table, b.seq_lens, b.q_lens)
    rows = [2, 9, 20, 35]
    sub = orc.layer_step(shape, w64, x, kp, vp, b.block_table, b.seq_lens, b.q_lens, rows=rows)
    np.testing.assert_allclose(sub["y"], full["y"][rows], rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(sub["slots"], full["slots"][rows])


def test_prefill_chunk_in_two_steps_equals_one_step():
    """Splitting a prefill chunk across two steps (the first appends its K/V to
    the cache, the second continues after that prefix) gives the same rows as
    one step: the nano-batch dependency rule the pipeline relies on."""
    shape = wl.tiny_shape()
    P = shape.page_size
    w = wl.make_weights(shape, seed=1, gain_std=0.1)
    w64 = orc.weights_f64(w)
    b_one = wl.make_batch(shape, [], [32], [0], seed_bt=4)
    x = wl.make_x(shape, 32, seed=5)
    kp, vp = wl.make_pools(shape, b_one)
    kp = kp.double(); vp = vp.double()
    one = orc.layer_step(shape, w64, x, kp, vp, b_one.block_table, b_one.seq_lens, b_one.q_lens)
    first = orc.layer_step(shape, w64, x[:12], kp, vp, b_one.block_table, np.array([12]),
                           np.array([12]))
    kp2, vp2 = kp.clone(), vp.clone()
    for i, sl in enumerate(first["slots"].tolist()):
        kp2[sl // P, :, sl % P, :] = torch.from_numpy(first["k_new"][i])
        vp2[sl // P, :, sl % P, :] = torch.from_numpy(first["v_new"][i])
    second = orc.layer_step(shape, w64, x[12:], kp2, vp2, b_one.block_table, np.array([32]),
                            np.array([20]))
    np.testing.assert_allclose(first["y"], one["y"][:12], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(second["y"], one["y"][12:], rtol=1e-12, atol=1e-12)


def test_silu_values():
    z = np.array([0.0, 1.0, -1.0, 20.0])
    np.testing.assert_allclose(orc.silu(z), [0.0, 1 / (1 + math.exp(-1)), -1 / (1 + math.e), 20 / (1 + math.exp(-20))],
                               rtol=1e-15)


# ------------------------------------------------------------------ stack

def _stack_inputs(n_layers=2, vocab=97):
    shape = wl.tiny_shape()
    b = wl.tiny_batch()
    g = torch.Generator().manual_seed(11)
    embed = torch.randn(vocab, shape.hidden, generator=g).to(torch.bfloat16)
    lm_head = (torch.randn(vocab, shape.hidden, generator=g) * 0.02).to(torch.bfloat16)
    norm_f = (1 + 0.1 * torch.randn(shape.hidden, generator=g)).to(torch.bfloat16)
    tokens = torch.randint(0, vocab, (b.n_tokens,), generator=g).numpy()
    layers = [wl.make_weights(shape, seed=20 + i, gain_std=0.1) for i in range(n_layers)]
    pools = [wl.make_pools(shape, b, "cpu", seed=40 + i) for i in range(n_layers)]
    return shape, b, embed, norm_f, lm_head, tokens, layers, pools


def test_stack_one_layer_is_embed_layer_head():
    shape, b, embed, norm_f, lm_head, tokens, layers, pools = _stack_inputs(1)
    w64 = [orc.weights_f64(layers[0])]
    st = orc.stack_step(shape, embed, norm_f, lm_head, w64, tokens, pools, b.block_table,
                        b.seq_lens, b.q_lens)
    x = embed[torch.as_tensor(tokens)]
    lay = orc.layer_step(shape, w64[0], x, pools[0][0], pools[0][1], b.block_table, b.seq_lens,
                         b.q_lens)
    ref = orc.rmsnorm(lay["y"], orc.f64(norm_f), shape.rms_eps) @ orc.f64(lm_head).T
    np.testing.assert_allclose(st["logits"], ref, rtol=1e-12, atol=1e-12)


def test_stack_with_silent_layers_is_a_normed_embedding_lookup():
    shape, b, embed, norm_f, lm_head, tokens, layers, pools = _stack_inputs(3)
    zero = [{k: (torch.zeros_like(v) if k.startswith("w_") else v) for k, v in L.items()}
            for L in layers]
    st = orc.stack_step(shape, embed, norm_f, lm_head, [orc.weights_f64(z) for z in zero], tokens,
                        pools, b.block_table, b.seq_lens, b.q_lens)
    e = orc.f64(embed)[tokens]
    ref = (e / np.sqrt(np.mean(e * e, -1, keepdims=True) + shape.rms_eps)) * orc.f64(norm_f)
    np.testing.assert_allclose(st["logits"], ref @ orc.f64(lm_head).T, rtol=1e-12, atol=1e-12)


def test_stack_rows_subset_equals_full():
    shape, b, embed, norm_f, lm_head, tokens, layers, pools = _stack_inputs(2)
    w64 = [orc.weights_f64(L) for L in layers]
    full = orc.stack_step(shape, embed, norm_f, lm_head, w64, tokens, pools, b.block_table,
                          b.seq_lens, b.q_lens)
    rows = [1, 4, 20, 35]
    sub = orc.stack_step(shape, embed, norm_f, lm_head, w64, tokens, pools, b.block_table,
                         b.seq_lens, b.q_lens, rows=rows)
    np.testing.assert_allclose(sub["logits"], full["logits"][rows], rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ layers only

def test_layers_with_a_silent_layer_inside_equal_the_others_alone():
    """A layer whose projection matrices are zero passes x through (h = x,
    y = h), so inserting one changes nothing downstream."""
    shape, b, _, _, _, _, layers, pools = _stack_inputs(3)
    x = wl.make_x(shape, b.n_tokens, seed=5)
    w64 = [orc.weights_f64(L) for L in layers]
    zero = orc.weights_f64({k: (torch.zeros_like(v) if k.startswith("w_") else v)
                            for k, v in layers[1].items()})
    with_zero = orc.layers_step(shape, [w64[0], zero, w64[2]], x, pools, b.block_table,
                                b.seq_lens, b.q_lens)
    without = orc.layers_step(shape, [w64[0], w64[2]], x, [pools[0], pools[2]], b.block_table,
                              b.seq_lens, b.q_lens)
    np.testing.assert_allclose(with_zero["y"], without["y"], rtol=1e-12, atol=1e-12)


def test_layers_rows_subset_equals_full():
    """Rows of a prefill chunk need the earlier rows of the chunk in every
    layer; the subset must still equal the full computation."""
    shape, b, _, _, _, _, layers, pools = _stack_inputs(2)
    x = wl.make_x(shape, b.n_tokens, seed=6)
    w64 = [orc.weights_f64(L) for L in layers]
    full = orc.layers_step(shape, w64, x, pools, b.block_table, b.seq_lens, b.q_lens)
    rows = [0, 3, 10, 35]
    sub = orc.layers_step(shape, w64, x, pools, b.block_table, b.seq_lens, b.q_lens, rows=rows)
    np.testing.assert_allclose(sub["y"], full["y"][rows], rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------- MoE (routing)

def test_route_picks_the_largest_logits_with_ties_to_the_lower_index():
    rng = np.random.default_rng(3)
    logits = rng.integers(-3, 4, size=(64, 8)).astype(np.float64)   # many ties
    experts, weights = orc.route(logits, 2)
    for t in range(64):
        e0, e1 = experts[t]
        assert e0 != e1
        # brute force over all ordered pairs: the chosen pair is the
        # lexicographically best (higher logit first, then lower index)
        best = min(((a, b) for a in range(8) for b in range(8) if a != b),
                   key=lambda ab: (-logits[t, ab[0]], ab[0], -logits[t, ab[1]], ab[1]))
        assert (e0, e1) == best
        # softmax over two logits: w0 = 1 / (1 + exp(r1 - r0))
        w0 = 1.0 / (1.0 + np.exp(logits[t, e1] - logits[t, e0]))
        np.testing.assert_allclose(weights[t], [w0, 1.0 - w0], rtol=1e-14, atol=1e-15)


def test_expert_groups_cover_every_choice_once_in_token_order():
    rng = np.random.default_rng(4)
    experts, _ = orc.route(rng.standard_normal((50, 6)), 2)
    pairs, offs = orc.expert_groups(experts, 6)
    assert offs[0] == 0 and offs[-1] == 100 and len(pairs) == 100
    assert sorted(map(tuple, pairs.tolist())) == [(t, j) for t in range(50) for j in range(2)]
    for e in range(6):
        grp = pairs[offs[e]:offs[e + 1]]
        assert all(experts[t, j] == e for t, j in grp)
        assert list(grp[:, 0]) == sorted(grp[:, 0])          # tokens increase


def _moe_dense_pair(E=4, top_k=2):
    shape = wl.tiny_moe_shape()
    dense = wl.make_weights(wl.tiny_shape(), seed=5)
    w = {k: v for k, v in dense.items() if k not in ("w_gate_up", "w_down")}
    w["w_experts_gate_up"] = dense["w_gate_up"][None].repeat(E, 1, 1)
    w["w_experts_down"] = dense["w_down"][None].repeat(E, 1, 1)
    return shape, dense, w


def test_moe_with_identical_experts_is_the_dense_ffn():
    """The routing weights of a token sum to 1, so identical experts give the
    dense SwiGLU FFN whatever the routing."""
    shape, dense, w = _moe_dense_pair()
    d64, m64 = orc.weights_f64(dense), orc.weights_f64(w)
    rng = np.random.default_rng(6)
    n2 = rng.standard_normal((9, shape.hidden))
    logits = rng.standard_normal((9, shape.n_experts))
    F = shape.ffn
    ref = (orc.silu(n2 @ d64["w_gate_up"][:F].T) * (n2 @ d64["w_gate_up"][F:].T)) @ d64["w_down"].T
    np.testing.assert_allclose(orc.moe_ffn(n2, m64, logits, 2, F), ref, rtol=1e-12, atol=1e-12)


def test_moe_top1_is_the_argmax_experts_ffn():
    shape = wl.tiny_moe_shape()
    w = orc.weights_f64(wl.make_moe_weights(shape, seed=7))
    rng = np.random.default_rng(8)
    n2 = rng.standard_normal((5, shape.hidden))
    logits = rng.standard_normal((5, shape.n_experts))
    F = shape.ffn
    got = orc.moe_ffn(n2, w, logits, 1, F)
    for i in range(5):
        e = int(np.argmax(logits[i]))
        gu, dn = w["w_experts_gate_up"][e], w["w_experts_down"][e]
        ref = (orc.silu(n2[i] @ gu[:F].T) * (n2[i] @ gu[F:].T)) @ dn.T
        np.testing.assert_allclose(got[i], ref, rtol=1e-12, atol=1e-12)


def test_moe_layer_with_identical_experts_equals_the_dense_layer():
    shape, dense, w = _moe_dense_pair()
    b = wl.tiny_batch()
    kp, vp = wl.make_pools(wl.tiny_shape(), b, "cpu", seed=9)
    x = wl.make_x(shape, b.n_tokens, seed=10)
    logits = wl.make_router_logits(b.n_tokens, shape.n_experts, seed=11)
    moe = orc.layer_step(shape, orc.weights_f64(w), x, kp, vp, b.block_table, b.seq_lens,
                         b.q_lens, router_logits=logits.numpy())
    den = orc.layer_step(wl.tiny_shape(), orc.weights_f64(dense), x, kp, vp, b.block_table,
                         b.seq_lens, b.q_lens)
    np.testing.assert_allclose(moe["y"], den["y"], rtol=1e-12, atol=1e-12)
