"""Per-step parity on the GPU: each kernel through the C ABI against the oracle
(or, for the GEMM primitive, a float64 matmul of the same bf16 inputs)."""
import numpy as np
import pytest
import torch

from nano_intra_device_gb300 import _lib, workload as wl
from oracle import layer as orc
from tests.helpers import compare, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rand(*shape, std=1.0, seed=0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


# ------------------------------------------------------------------- GEMM
GEMM_SHAPES = [(128, 256, 64), (36, 512, 256), (300, 688, 256), (1, 8, 8), (129, 264, 200),
               (1024, 1024, 4096), (2048, 6144, 4096), (640, 4096, 14336),
               # few output tiles: split-K across CTAs
               (64, 4096, 14336), (128, 6144, 4096), (8, 1024, 4096), (256, 2048, 8192)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_store_matches_float64(M, N, K):
    A, B = _rand(M, K, seed=1), _rand(N, K, std=0.02, seed=2)
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    _lib.gemm(A.to(DEV), B.to(DEV), C)
    torch.cuda.synchronize()
    ref = f64(A) @ f64(B).T
    compare(f64(C), ref, f"gemm {M}x{N}x{K}", rel_l2=5e-3)


@pytest.mark.parametrize("M,N,K", [(300, 688, 256), (2048, 4096, 4096), (64, 4096, 14336)])
def test_gemm_residual_matches_float64(M, N, K):
    A, B, R = _rand(M, K, seed=3), _rand(N, K, std=0.02, seed=4), _rand(M, N, seed=5)
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    _lib.gemm(A.to(DEV), B.to(DEV), C, R=R.to(DEV), epilogue=_lib.NF_EPI_RESID)
    torch.cuda.synchronize()
    compare(f64(C), f64(R) + f64(A) @ f64(B).T, "gemm+residual", rel_l2=5e-3)


@pytest.mark.parametrize("M,F,K", [(36, 688, 256), (1024, 14336, 4096), (200, 320, 512),
                                   (64, 1024, 4096)])
def test_gemm_swiglu_matches_float64(M, F, K):
    A, B = _rand(M, K, seed=6), _rand(2 * F, K, std=0.02, seed=7)
    C = torch.empty(M, F, dtype=torch.bfloat16, device=DEV)
    _lib.gemm(A.to(DEV), B.to(DEV), C, epilogue=_lib.NF_EPI_SWIGLU)
    torch.cuda.synchronize()
    g = f64(A) @ f64(B[:F]).T
    u = f64(A) @ f64(B[F:]).T
    compare(f64(C), orc.silu(g) * u, "gemm+swiglu", rel_l2=5e-3)


def test_gemm_split_k_repeats_identically():
    # the per-tile arrival counters reset themselves: a second call splits the same way
    A, B = _rand(64, 14336, seed=12), _rand(4096, 14336, std=0.02, seed=13)
    Ad, Bd = A.to(DEV), B.to(DEV)
    C1 = torch.empty(64, 4096, dtype=torch.bfloat16, device=DEV)
    C2 = torch.empty_like(C1)
    _lib.gemm(Ad, Bd, C1)
    _lib.gemm(Ad, Bd, C2)
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


# weight-row kernel: (M tokens, N, K, splits); ragged N (136, 688), K not a
# multiple of 64 (200), one and two token tiles' sizes, every cluster size
WROWS_SHAPES = [(1, 136, 64, 1), (17, 256, 200, 0), (64, 4096, 4096, 0), (64, 4096, 14336, 4),
                (65, 688, 256, 4), (128, 1024, 4096, 8), (36, 512, 256, 3), (100, 6144, 4096, 6),
                (8, 1024, 512, 2), (64, 2048, 4096, 5), (64, 2048, 4096, 7),
                # two 128-token tiles
                (256, 4096, 4096, 0), (200, 1032, 512, 3)]


@pytest.mark.parametrize("M,N,K,splits", WROWS_SHAPES)
def test_gemm_wrows_store_matches_float64(M, N, K, splits):
    A, B = _rand(M, K, seed=21), _rand(N, K, std=0.02, seed=22)
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    _lib.gemm_wrows(A.to(DEV), B.to(DEV), C, splits=splits)
    torch.cuda.synchronize()
    compare(f64(C), f64(A) @ f64(B).T, f"wrows {M}x{N}x{K}/{splits}", rel_l2=5e-3)


@pytest.mark.parametrize("M,N,K,splits", [(64, 4096, 14336, 0), (33, 688, 256, 2), (128, 512, 1024, 8)])
def test_gemm_wrows_residual_matches_float64(M, N, K, splits):
    A, B, R = _rand(M, K, seed=23), _rand(N, K, std=0.02, seed=24), _rand(M, N, seed=25)
    C = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    _lib.gemm_wrows(A.to(DEV), B.to(DEV), C, R=R.to(DEV), epilogue=_lib.NF_EPI_RESID, splits=splits)
    torch.cuda.synchronize()
    compare(f64(C), f64(R) + f64(A) @ f64(B).T, "wrows+residual", rel_l2=5e-3)


@pytest.mark.parametrize("M,F,K,splits", [(36, 688, 256, 0), (64, 14336, 4096, 0), (120, 320, 512, 3),
                                          (1, 1024, 4096, 8)])
def test_gemm_wrows_swiglu_matches_float64(M, F, K, splits):
    A, B = _rand(M, K, seed=26), _rand(2 * F, K, std=0.02, seed=27)
    C = torch.empty(M, F, dtype=torch.bfloat16, device=DEV)
    _lib.gemm_wrows(A.to(DEV), B.to(DEV), C, epilogue=_lib.NF_EPI_SWIGLU, splits=splits)
    torch.cuda.synchronize()
    g = f64(A) @ f64(B[:F]).T
    u = f64(A) @ f64(B[F:]).T
    compare(f64(C), orc.silu(g) * u, "wrows+swiglu", rel_l2=5e-3)


def test_gemm_wrows_sum_is_timing_independent_and_leaves_other_rows():
    """The cluster's partial tiles are added in rank order: repeated calls give
    the same bits; rows of C past M are never written."""
    A, B = _rand(64, 14336, seed=28), _rand(4096, 14336, std=0.02, seed=29)
    Ad, Bd = A.to(DEV), B.to(DEV)
    outs = []
    for _ in range(3):
        C = torch.full((80, 4096), 7.0, dtype=torch.bfloat16, device=DEV)
        _lib.gemm_wrows(Ad, Bd, C[:64], splits=8)
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert bool((outs[0][64:] == 7.0).all())


def test_gemm_wrows_rejects_what_it_cannot_do():
    A, B = _rand(257, 256, seed=1).to(DEV), _rand(256, 256, seed=2).to(DEV)
    C = torch.empty(257, 256, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(_lib.NanoflowError):
        _lib.gemm_wrows(A, B, C)                      # more than 256 rows of A
    with pytest.raises(_lib.NanoflowError):
        _lib.gemm_wrows(A[:64], B, C[:64], splits=5)  # 4 K blocks cannot take 5 splits
    with pytest.raises(_lib.NanoflowError):
        _lib.gemm_wrows(A[:64], B, C[:64], splits=9)


def test_gemm_sm_cap_gives_identical_bits():
    # 256 output tiles: no split-K at any cap, so the bits must not depend on it
    A, B = _rand(2048, 4096, seed=8), _rand(4096, 4096, std=0.02, seed=9)
    Ad, Bd = A.to(DEV), B.to(DEV)
    outs = []
    for cap in (0, 7, 64):
        C = torch.empty(2048, 4096, dtype=torch.bfloat16, device=DEV)
        _lib.gemm(Ad, Bd, C, max_sms=cap)
        outs.append(C)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


# ---------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("rows,H", [(36, 256), (2048, 4096), (3, 8192)])
def test_rmsnorm_matches_oracle(rows, H):
    x, g = _rand(rows, H, seed=10), (1 + 0.1 * _rand(H, seed=11).float()).to(torch.bfloat16)
    out = torch.empty(rows, H, dtype=torch.bfloat16, device=DEV)
    _lib.rmsnorm(x.to(DEV), g.to(DEV), out, 1e-5)
    torch.cuda.synchronize()
    compare(f64(out), orc.rmsnorm(f64(x), f64(g), 1e-5), "rmsnorm", rel_l2=5e-3)


# --------------------------------------------------------- step metadata
def _meta_case(shape, batch, bounds, kv_chunk):
    T = batch.n_tokens
    plan = _lib.Plan(shape, batch, _lib.make_opts(T, bounds, kv_chunk=kv_chunk))
    bt = torch.from_numpy(batch.block_table).to(DEV)
    sl = torch.from_numpy(batch.seq_lens).to(DEV)
    _lib.step_metadata(plan, bt, sl)
    plan.poll()
    seq = plan.buffer(_lib.NF_BUF_TOK_SEQ, torch.int32, (T,)).numpy()
    pos = plan.buffer(_lib.NF_BUF_TOK_POS, torch.int32, (T,)).numpy()
    slot = plan.buffer(_lib.NF_BUF_TOK_SLOT, torch.int32, (T,)).numpy()
    segs = plan.buffer(_lib.NF_BUF_ITEM_SEG, torch.int32, (len(bounds),)).numpy()
    n_items = int(segs[-1])
    items = plan.buffer(_lib.NF_BUF_ITEMS, torch.int32, (2 * n_items,)).numpy().reshape(-1, 2)
    plan.close()
    rseq, rpos = orc.token_map(batch.q_lens, batch.seq_lens)
    np.testing.assert_array_equal(seq, rseq)
    np.testing.assert_array_equal(pos, rpos)
    np.testing.assert_array_equal(slot, orc.slot_of(rseq, rpos, batch.block_table, shape.page_size))
    for i in range(len(bounds) - 1):
        got = items[segs[i]:segs[i + 1]]
        ctx = rpos + 1
        want = orc.split_kv_items(ctx, kv_chunk, bounds[i], bounds[i + 1])
        got_set = sorted((int(t), int(c) * kv_chunk, int(min(kv_chunk, ctx[t] - c * kv_chunk))) for t, c in got)
        assert got_set == want, f"segment {i}"
        # longest pieces first inside a segment
        lens = [min(kv_chunk, ctx[t] - c * kv_chunk) for t, c in got]
        pages = [(n + 15) // 16 for n in lens]
        assert pages == sorted(pages, reverse=True)


def test_metadata_tiny_bit_exact():
    _meta_case(wl.tiny_shape(), wl.tiny_batch(), [0, 18, 36], 32)


def test_metadata_llama8b_bit_exact():
    b = wl.llama8b_batch()
    _meta_case(wl.llama8b_shape(), b, [0, 1024, 2048], 512)


def test_metadata_edge_lengths():
    shape = wl.tiny_shape()
    b = wl.make_batch(shape, [1, 16, 17, 2048], [1, 40], [0, 23], seed_bt=5)
    _meta_case(shape, b, [0, 2, 3, 6, b.n_tokens], 16)


def test_metadata_flags_bad_page_without_faulting():
    shape = wl.tiny_shape()
    b = wl.tiny_batch()
    bt = b.block_table.copy()
    bt[1, 2] = b.num_pages + 5          # decode token 1 (position 32) lands on page index 2
    plan = _lib.Plan(shape, b, _lib.make_opts(b.n_tokens, kv_chunk=32, validate=1))
    _lib.step_metadata(plan, torch.from_numpy(bt).to(DEV), torch.from_numpy(b.seq_lens).to(DEV))
    with pytest.raises(_lib.NanoflowError) as e:
        plan.poll()
    assert e.value.code == _lib.NF_ERR_DEVICE
    slot = plan.buffer(_lib.NF_BUF_TOK_SLOT, torch.int32, (b.n_tokens,)).numpy()
    assert slot[1] == -1
    plan.poll()   # the status word was cleared by the previous poll
    plan.close()


# -------------------------------------------------------------- attention
def _attention_case(shape, batch, rows, bounds, kv_chunk, seed=0, warps=0, impl=0):
    T = batch.n_tokens
    kp, vp = wl.make_pools(shape, batch, DEV, seed=seed + 3, appended=True)
    q = _rand(T, shape.n_q, shape.head_dim, seed=seed + 20)
    seq, pos = orc.token_map(batch.q_lens, batch.seq_lens)
    P = shape.page_size
    ref = {}
    for t in rows:   # oracle first: it reads only the generator's pool
        s, L = int(seq[t]), int(pos[t]) + 1
        j = np.arange(L)
        pages = torch.as_tensor(batch.block_table[s, j // P].astype(np.int64), device=DEV)
        offs = torch.as_tensor(j % P, device=DEV)
        K = f64(kp[pages, :, offs, :])
        V = f64(vp[pages, :, offs, :])
        ref[t] = orc.attention_one(f64(q[t]), K, V, shape.n_q, shape.n_kv)
    plan = _lib.Plan(shape, batch, _lib.make_opts(T, bounds, kv_chunk=kv_chunk, attn_warps=warps,
                                                  attn_impl=impl))
    o = torch.empty(T, shape.n_q, shape.head_dim, dtype=torch.bfloat16, device=DEV)
    _lib.attention(plan, q.to(DEV), kp, vp, torch.from_numpy(batch.block_table).to(DEV),
                   torch.from_numpy(batch.seq_lens).to(DEV), o)
    plan.poll()
    plan.close()
    got = f64(o)
    compare(np.stack([got[t] for t in rows]), np.stack([ref[t] for t in rows]), "attention",
            rel_l2=1e-2)


MMA = _lib.NF_ATTN_MMA
# warps per CTA of the tensor-core kernel: 8 (default), more with shallower
# rings, and 4 (the configuration that shares an SM with a 2-stage GEMM CTA)
ATTN_WARPS = [8, 14, 12, 10, 7, 6, 5, 4]


@pytest.mark.parametrize("kv_chunk", [16, 32, 512])
def test_attention_tiny_all_rows(kv_chunk):
    b = wl.tiny_batch()
    _attention_case(wl.tiny_shape(), b, list(range(b.n_tokens)), [0, 18, 36], kv_chunk, impl=MMA)


@pytest.mark.parametrize("grp,d", [(1, 64), (2, 128), (4, 128), (8, 128), (8, 64), (4, 64)])
@pytest.mark.parametrize("warps", ATTN_WARPS)
def test_attention_gqa_and_head_dims(grp, d, warps):
    shape = wl.Shape(hidden=512, n_q=2 * grp, n_kv=2, head_dim=d, ffn=512)
    b = wl.make_batch(shape, [1, 15, 16, 17, 700, 1100], [9], [40], seed_bt=7)
    _attention_case(shape, b, list(range(b.n_tokens)), [0, 3, b.n_tokens], 256, seed=grp,
                    warps=warps)


@pytest.mark.parametrize("grp,d", [(1, 64), (2, 128), (4, 128), (8, 64), (8, 128)])
def test_attention_prefill_tiles_cross_chunks_and_nano_batches(grp, d):
    """Prefill chunks through the tiled causal kernel: chunks longer than a
    tile (128 / grp rows), prefixes 0 to 513, a one-row chunk, and nano-batch
    boundaries that cut chunks; every row against the oracle."""
    shape = wl.Shape(hidden=512, n_q=2 * grp, n_kv=2, head_dim=d, ffn=512)
    b = wl.make_batch(shape, [5, 300], [150, 37, 1, 200], [0, 90, 7, 513], seed_bt=8)
    T = b.n_tokens
    _attention_case(shape, b, list(range(T)), [0, 70, 200, T], 128, seed=10 + grp)


def test_attention_automatic_is_the_tensor_core_kernel():
    """attn_impl 0 and 2 run the same kernel bit for bit; nf_plan_info reports it."""
    shape = wl.llama8b_shape()
    b = wl.make_batch(shape, wl.lognormal_contexts(64, 600.0, 1.0, 1, 4096, seed=5), [48], None,
                      seed_bt=6, max_pages=4096 // 16)
    T = b.n_tokens
    kp, vp = wl.make_pools(shape, b, DEV, seed=8, appended=True)
    q = _rand(T, shape.n_q, shape.head_dim, seed=9).to(DEV)
    bt = torch.from_numpy(b.block_table).to(DEV)
    sl = torch.from_numpy(b.seq_lens).to(DEV)
    outs = {}
    for impl in (0, MMA):
        plan = _lib.Plan(shape, b, _lib.make_opts(T, kv_chunk=256, attn_impl=impl))
        assert plan.info()[0].attn_impl == MMA
        o = torch.empty(T, shape.n_q, shape.head_dim, dtype=torch.bfloat16, device=DEV)
        _lib.attention(plan, q, kp, vp, bt, sl, o)
        plan.poll()
        plan.close()
        outs[impl] = o
    assert torch.equal(outs[0], outs[MMA])


def test_attention_rejects_configurations_the_kernel_lacks():
    shape, b = wl.tiny_shape(), wl.tiny_batch()
    for warps, impl in [(16, MMA), (3, 0), (9, 0), (11, 0), (8, 1), (8, 3)]:
        with pytest.raises(_lib.NanoflowError):
            _lib.Plan(shape, b, _lib.make_opts(b.n_tokens, attn_warps=warps, attn_impl=impl))


@pytest.mark.parametrize("warps", [8, 12, 14, 4])
def test_attention_llama8b_sampled_rows(warps):
    b = wl.llama8b_batch()
    T = b.n_tokens
    ctx = b.seq_lens[: b.n_decode]
    rng = np.random.default_rng(0)
    rows = sorted(set([int(np.argmax(ctx)), int(np.argmin(ctx))] +
                      rng.choice(b.n_decode, 40, replace=False).tolist() +
                      [b.n_decode, b.n_decode + 1, T - 1] +
                      (b.n_decode + rng.choice(256, 8, replace=False)).tolist()))
    _attention_case(wl.llama8b_shape(), b, rows, [0, 1024, T], 512, warps=warps)
