"""ctypes binding of libnanoflow.so: the C ABI declared in include/nanoflow.h.

Argument marshalling only.  Every step of the layer runs in the library's CUDA
kernels; if the library is missing this module raises instead of falling back
to anything else.
"""
from __future__ import annotations

import ctypes
import os
import re
from ctypes import POINTER, Structure, c_char_p, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libnanoflow.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "nanoflow.h")
NF_MAX_NANO = 8

NF_OK, NF_ERR_INVALID_ARG, NF_ERR_UNSUPPORTED, NF_ERR_OOM, NF_ERR_CUDA, NF_ERR_TIMEOUT, \
    NF_ERR_DEVICE, NF_ERR_INTERNAL = range(8)
NF_EXEC_SEQUENTIAL, NF_EXEC_STREAMS = 0, 1
NF_ATTN_AUTO, NF_ATTN_MMA = 0, 2
NF_EPI_STORE, NF_EPI_RESID, NF_EPI_SWIGLU = 0, 1, 2
(NF_BUF_TOK_SEQ, NF_BUF_TOK_POS, NF_BUF_TOK_SLOT, NF_BUF_ITEMS, NF_BUF_ITEM_SEG, NF_BUF_N1,
 NF_BUF_Q, NF_BUF_O, NF_BUF_H, NF_BUF_N2, NF_BUF_A, NF_BUF_MOE_OFF, NF_BUF_MOE_PERM,
 NF_BUF_MOE_PAIR_ROW, NF_BUF_MOE_PAIR_W) = range(15)


class nf_model_shape(Structure):
    _fields_ = [("hidden", c_int32), ("n_q_heads", c_int32), ("n_kv_heads", c_int32),
                ("head_dim", c_int32), ("ffn", c_int32), ("page_size", c_int32),
                ("rms_eps", c_float), ("rope_theta", c_float), ("n_experts", c_int32),
                ("top_k", c_int32)]


class nf_batch_desc(Structure):
    _fields_ = [("n_decode", c_int32), ("n_prefill", c_int32),
                ("prefill_q_lens", POINTER(c_int32)), ("seq_lens_hint", POINTER(c_int32)),
                ("max_pages_per_seq", c_int32), ("num_pages", c_int32)]


class nf_plan_opts(Structure):
    _fields_ = [("n_attn", c_int32), ("attn_bounds", c_int32 * (NF_MAX_NANO + 1)),
                ("n_ffn", c_int32), ("ffn_bounds", c_int32 * (NF_MAX_NANO + 1)),
                ("executor", c_int32), ("attn_sms", c_int32), ("gemm_sms", c_int32),
                ("kv_chunk", c_int32), ("attn_warps", c_int32), ("gemm_stages", c_int32),
                ("gemm_split_k", c_int32), ("attn_impl", c_int32), ("validate", c_int32),
                ("timeout_ns", c_int64)]


class nf_runtime_opts(Structure):
    _fields_ = [("b_dense", c_int32), ("max_requests", c_int32), ("max_pages_per_seq", c_int32),
                ("num_pages", c_int32), ("vocab", c_int32), ("eos_token", c_int32),
                ("replan_threshold", c_float), ("host_only", c_int32)]


class nf_runtime_batch(Structure):
    _fields_ = [("iteration", c_int32), ("n_tokens", c_int32), ("n_decode", c_int32),
                ("n_prefill", c_int32), ("row_request", POINTER(c_int32)),
                ("row_pos", POINTER(c_int32)), ("row_token", POINTER(c_int32)),
                ("row_emit", POINTER(c_int32)), ("seq_lens", POINTER(c_int32)),
                ("block_table", POINTER(c_int32)), ("prefill_q_lens", POINTER(c_int32)),
                ("replanned", c_int32), ("free_pages", c_int32)]


class nf_trace_entry(Structure):
    _fields_ = [("op", c_int32), ("nano", c_int32), ("step", c_int32), ("start_ms", c_float),
                ("ms", c_float)]


NF_OP_NAMES = {0: "meta", 1: "qkv", 2: "attn", 3: "oproj", 4: "ffn"}


class nf_layer_weights(Structure):
    _fields_ = [(n, c_void_p) for n in ("norm1", "w_qkv", "w_o", "norm2", "w_gate_up", "w_down",
                                        "w_experts_gate_up", "w_experts_down", "router_logits")]


class nf_stack_weights(Structure):
    _fields_ = [("embed", c_void_p), ("norm_f", c_void_p), ("lm_head", c_void_p),
                ("vocab", c_int32), ("n_layers", c_int32), ("layers", POINTER(nf_layer_weights))]


_SIGS = {
    "nf_plan_create": (c_int, [POINTER(nf_model_shape), POINTER(nf_batch_desc), POINTER(nf_plan_opts), POINTER(c_void_p)]),
    "nf_plan_info": (c_int, [c_void_p, POINTER(nf_plan_opts), POINTER(c_int32)]),
    "nf_plan_save": (c_int, [c_void_p, c_char_p]),
    "nf_plan_load": (c_int, [c_char_p, POINTER(c_void_p)]),
    "nf_plan_destroy": (None, [c_void_p]),
    "nf_layer_step": (c_int, [c_void_p, POINTER(nf_layer_weights), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "nf_layer_step_host": (c_int, [c_void_p, POINTER(nf_layer_weights), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "nf_layer_step_host_async": (c_int, [c_void_p, POINTER(nf_layer_weights), c_void_p, c_void_p, c_void_p, c_void_p,
                                         c_void_p, c_void_p, c_void_p]),
    "nf_plan_host_wait": (c_int, [c_void_p]),
    "nf_plan_poll": (c_int, [c_void_p, c_int]),
    "nf_plan_selftest_wait": (c_int, [c_void_p, c_int64, c_int32, c_void_p, c_void_p]),
    "nf_stack_step": (c_int, [c_void_p, POINTER(nf_stack_weights), c_void_p, POINTER(c_void_p), POINTER(c_void_p), c_void_p, c_void_p, c_void_p, c_void_p]),
    "nf_stack_step_rows": (c_int, [c_void_p, POINTER(nf_stack_weights), c_void_p, POINTER(c_void_p), POINTER(c_void_p),
                                   c_void_p, c_void_p, c_void_p, c_int32, c_void_p, c_void_p]),
    "nf_layers_step": (c_int, [c_void_p, POINTER(nf_layer_weights), c_int32, c_void_p, POINTER(c_void_p), POINTER(c_void_p), c_void_p, c_void_p, c_void_p, c_void_p]),
    "nf_plan_set_batch": (c_int, [c_void_p, POINTER(nf_batch_desc), POINTER(nf_plan_opts), c_void_p]),
    "nf_runtime_create": (c_int, [POINTER(nf_model_shape), POINTER(nf_runtime_opts), POINTER(c_void_p)]),
    "nf_runtime_destroy": (None, [c_void_p]),
    "nf_runtime_submit": (c_int, [c_void_p, POINTER(c_int32), c_int32, c_int32, POINTER(c_int32)]),
    "nf_runtime_step": (c_int, [c_void_p, POINTER(nf_stack_weights), POINTER(c_void_p), POINTER(c_void_p), c_void_p, POINTER(nf_runtime_batch)]),
    "nf_runtime_sync": (c_int, [c_void_p]),
    "nf_runtime_result": (c_int, [c_void_p, c_int32, POINTER(c_int32), POINTER(c_int32), POINTER(c_int32), c_int32]),
    "nf_runtime_counts": (c_int, [c_void_p, POINTER(c_int32), POINTER(c_int32), POINTER(c_int32)]),
    "nf_runtime_form": (c_int, [c_void_p, POINTER(nf_runtime_batch)]),
    "nf_runtime_apply": (c_int, [c_void_p, c_int32, POINTER(c_int32)]),
    "nf_runtime_logits": (c_int, [c_void_p, c_void_p, c_int32, POINTER(c_int32)]),
    "nf_last_error": (c_char_p, []),
    "nf_device_sm_count": (c_int32, []),
    "nf_step_metadata": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p]),
    "nf_attention": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "nf_attention_noalloc": (c_int, [POINTER(nf_model_shape), POINTER(nf_batch_desc), c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]),
    "nf_attention_noalloc_poll": (c_int, [c_void_p]),
    "nf_rmsnorm": (c_int, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_float, c_void_p]),
    "nf_gemm": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p]),
    "nf_gemm_wrows": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32,
                              c_int32, c_int32, c_void_p]),
    "nf_plan_buffer_size": (c_int, [c_void_p, c_int32, POINTER(c_size_t)]),
    "nf_plan_copy_buffer": (c_int, [c_void_p, c_int32, c_void_p, c_size_t]),
    "nf_plan_trace_enable": (c_int, [c_void_p, c_int32]),
    "nf_plan_trace_ops": (c_int, [c_void_p, ctypes.c_uint32]),
    "nf_plan_trace_read": (c_int, [c_void_p, POINTER(nf_trace_entry), c_int32, POINTER(c_int32)]),
    "nf_profile": (c_int, [POINTER(nf_model_shape), c_int32, c_int32, c_char_p]),
    "nf_profile_step": (c_int, [POINTER(nf_model_shape), POINTER(nf_batch_desc), c_int32, c_char_p]),
    "nf_profile_use": (c_int, [POINTER(nf_model_shape), c_char_p]),
    "nf_plan_search": (c_int, [POINTER(nf_model_shape), POINTER(nf_batch_desc), c_char_p, c_int32, POINTER(nf_plan_opts), POINTER(c_double)]),
    "nf_plan_search_layers": (c_int, [POINTER(nf_model_shape), POINTER(nf_batch_desc), c_char_p, c_int32, c_int32, POINTER(nf_plan_opts), POINTER(c_double)]),
    "nf_plan_predict": (c_int, [POINTER(nf_model_shape), POINTER(nf_batch_desc), c_char_p, c_int32, c_int32, POINTER(nf_plan_opts), POINTER(c_double)]),
    "nf_window_schedule": (c_int, [POINTER(nf_plan_opts), c_int32, POINTER(c_int32), c_int32, POINTER(c_int32)]),
}

_lib = None


class NanoflowError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"nanoflow error {code}: {msg}")
        self.code = code


def header_functions() -> list:
    """Names of the functions include/nanoflow.h declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\**\s+\**\s*(nf_\w+)\s*\(", text, re.M)))


def lib():
    """Load the library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def check(code):
    if code != NF_OK:
        raise NanoflowError(code, lib().nf_last_error().decode())


def ptr(t):
    """Device/host address of a torch tensor (None -> NULL)."""
    return None if t is None else c_void_p(t.data_ptr())


def stream_handle(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return c_void_p(s.cuda_stream)


def make_shape(shape) -> nf_model_shape:
    return nf_model_shape(shape.hidden, shape.n_q, shape.n_kv, shape.head_dim, shape.ffn,
                          shape.page_size, shape.rms_eps, shape.rope_theta,
                          getattr(shape, "n_experts", 0), getattr(shape, "top_k", 0))


def make_batch_desc(batch, hint=True):
    pq = (c_int32 * max(1, len(batch.prefill_q_lens)))(*batch.prefill_q_lens)
    sl = (c_int32 * batch.n_seq)(*[int(v) for v in batch.seq_lens]) if hint else None
    d = nf_batch_desc(batch.n_decode, len(batch.prefill_q_lens), pq, sl,
                      batch.max_pages, batch.num_pages)
    d._keep = (pq, sl)
    return d


def make_opts(T, attn_bounds=None, ffn_bounds=None, executor=NF_EXEC_SEQUENTIAL, attn_sms=0,
              gemm_sms=0, kv_chunk=1024, validate=0, timeout_ns=2_000_000_000,
              attn_warps=0, gemm_stages=0, gemm_split_k=0, attn_impl=0) -> nf_plan_opts:
    ab = list(attn_bounds) if attn_bounds is not None else [0, T]
    fb = list(ffn_bounds) if ffn_bounds is not None else list(ab)
    o = nf_plan_opts()
    o.n_attn = len(ab) - 1
    for i, v in enumerate(ab):
        o.attn_bounds[i] = v
    o.n_ffn = len(fb) - 1
    for i, v in enumerate(fb):
        o.ffn_bounds[i] = v
    o.executor, o.attn_sms, o.gemm_sms = executor, attn_sms, gemm_sms
    o.kv_chunk, o.validate, o.timeout_ns = kv_chunk, validate, timeout_ns
    o.attn_warps = attn_warps
    o.gemm_stages = gemm_stages
    o.gemm_split_k = gemm_split_k
    o.attn_impl = attn_impl
    return o


def opts_dict(o: nf_plan_opts) -> dict:
    return {"attn_bounds": list(o.attn_bounds[: o.n_attn + 1]),
            "ffn_bounds": list(o.ffn_bounds[: o.n_ffn + 1]),
            "executor": "streams" if o.executor == NF_EXEC_STREAMS else "sequential",
            "attn_sms": o.attn_sms, "gemm_sms": o.gemm_sms, "kv_chunk": o.kv_chunk,
            "attn_warps": o.attn_warps, "gemm_stages": o.gemm_stages,
            "gemm_split_k": o.gemm_split_k,
            "attn_impl": {NF_ATTN_MMA: "mma"}.get(o.attn_impl, "auto")}


def make_weights_struct(w: dict) -> nf_layer_weights:
    """Device pointers of a layer's weights (a MoE layer has w_experts_gate_up,
    w_experts_down and this step's router_logits instead of w_gate_up/w_down)."""
    return nf_layer_weights(*[(w[k].data_ptr() if k in w else None) for k in
                              ("norm1", "w_qkv", "w_o", "norm2", "w_gate_up", "w_down",
                               "w_experts_gate_up", "w_experts_down", "router_logits")])


class Plan:
    """Owns an nf_plan."""

    def __init__(self, shape, batch, opts: nf_plan_opts | None = None, hint=True):
        self.h = c_void_p()
        self._shape = make_shape(shape)
        self._batch = make_batch_desc(batch, hint)
        check(lib().nf_plan_create(ctypes.byref(self._shape), ctypes.byref(self._batch),
                                   ctypes.byref(opts) if opts is not None else None,
                                   ctypes.byref(self.h)))

    @classmethod
    def from_handle(cls, handle):
        p = cls.__new__(cls)
        p.h = handle
        return p

    def info(self):
        o = nf_plan_opts()
        n = c_int32()
        check(lib().nf_plan_info(self.h, ctypes.byref(o), ctypes.byref(n)))
        return o, n.value

    def set_batch(self, batch, opts: nf_plan_opts | None = None, stream=None, hint=True):
        """nf_plan_set_batch: the next steps run `batch` (same page geometry,
        at most the sequences and tokens the plan was created for)."""
        self._batch = make_batch_desc(batch, hint)
        check(lib().nf_plan_set_batch(self.h, ctypes.byref(self._batch),
                                      ctypes.byref(opts) if opts is not None else None,
                                      stream_handle(stream)))

    def close(self):
        if self.h:
            lib().nf_plan_destroy(self.h)
            self.h = c_void_p()

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass

    def buffer(self, which, dtype, shape):
        import torch
        out = torch.empty(shape, dtype=dtype)
        check(lib().nf_plan_copy_buffer(self.h, which, ptr(out), out.numel() * out.element_size()))
        return out

    def trace_enable(self, max_steps):
        check(lib().nf_plan_trace_enable(self.h, max_steps))

    def trace_ops(self, ops=None):
        """Record only the named operations ("meta", "qkv", "attn", "oproj",
        "ffn"); None: all."""
        mask = 0xFFFFFFFF if ops is None else sum(
            1 << k for k, v in NF_OP_NAMES.items() if v in ops)
        check(lib().nf_plan_trace_ops(self.h, mask))

    def trace_read(self):
        n = c_int32()
        check(lib().nf_plan_trace_read(self.h, None, 0, ctypes.byref(n)))
        buf = (nf_trace_entry * max(1, n.value))()
        check(lib().nf_plan_trace_read(self.h, buf, n.value, ctypes.byref(n)))
        return [{"op": NF_OP_NAMES.get(e.op, str(e.op)), "nano": e.nano, "step": e.step,
                 "start_ms": e.start_ms, "ms": e.ms} for e in buf[: n.value]]

    def poll(self, wait=True):
        check(lib().nf_plan_poll(self.h, 1 if wait else 0))

    def selftest_wait(self, timeout_ns, arrive, waited_ns=None, stream=None):
        """Enqueue the failure-detection self-test (a bounded wait on a barrier
        nothing arrives at unless `arrive`); waited_ns: optional int64 device
        tensor that receives the time waited."""
        check(lib().nf_plan_selftest_wait(self.h, int(timeout_ns), 1 if arrive else 0,
                                          ptr(waited_ns), stream_handle(stream)))


def layer_step(plan: Plan, w: dict, x, k_pool, v_pool, block_table, seq_lens, y, stream=None):
    ws = make_weights_struct(w)
    check(lib().nf_layer_step(plan.h, ctypes.byref(ws), ptr(x), ptr(k_pool), ptr(v_pool),
                              ptr(block_table), ptr(seq_lens), ptr(y), stream_handle(stream)))


class StackArgs:
    """Keeps the ctypes arrays of one stack's weights and pools alive."""

    def __init__(self, embed, norm_f, lm_head, layers: list, pools: list):
        self.layer_structs = (nf_layer_weights * len(layers))(*[make_weights_struct(w) for w in layers])
        self.w = nf_stack_weights(embed.data_ptr(), norm_f.data_ptr(), lm_head.data_ptr(),
                                  embed.shape[0], len(layers), self.layer_structs)
        self.kps = (c_void_p * len(pools))(*[k.data_ptr() for k, _ in pools])
        self.vps = (c_void_p * len(pools))(*[v.data_ptr() for _, v in pools])
        self._keep = (embed, norm_f, lm_head, layers, pools)


def stack_step(plan: Plan, args: StackArgs, tokens, block_table, seq_lens, logits, stream=None):
    check(lib().nf_stack_step(plan.h, ctypes.byref(args.w), ptr(tokens), args.kps, args.vps,
                              ptr(block_table), ptr(seq_lens), ptr(logits), stream_handle(stream)))


def stack_step_rows(plan: Plan, args: StackArgs, tokens, block_table, seq_lens, rows, logits,
                    stream=None):
    """nf_stack_step_rows: logits [len(rows), vocab] for the listed token rows only."""
    check(lib().nf_stack_step_rows(plan.h, ctypes.byref(args.w), ptr(tokens), args.kps, args.vps,
                                   ptr(block_table), ptr(seq_lens), ptr(rows), rows.numel(),
                                   ptr(logits), stream_handle(stream)))


class LayersArgs:
    """Keeps the ctypes arrays of a run of layers (weights and pools) alive."""

    def __init__(self, layers: list, pools: list):
        self.n = len(layers)
        self.layer_structs = (nf_layer_weights * self.n)(*[make_weights_struct(w) for w in layers])
        self.kps = (c_void_p * len(pools))(*[k.data_ptr() for k, _ in pools])
        self.vps = (c_void_p * len(pools))(*[v.data_ptr() for _, v in pools])
        self._keep = (layers, pools)


def layers_step(plan: Plan, args: LayersArgs, x, block_table, seq_lens, y, stream=None):
    check(lib().nf_layers_step(plan.h, args.layer_structs, args.n, ptr(x), args.kps, args.vps,
                               ptr(block_table), ptr(seq_lens), ptr(y), stream_handle(stream)))


def layer_step_host(plan: Plan, w: dict, x_host, k_pool, v_pool, bt_host, sl_host, y_host, stream=None):
    ws = make_weights_struct(w)
    check(lib().nf_layer_step_host(plan.h, ctypes.byref(ws), ptr(x_host), ptr(k_pool), ptr(v_pool),
                                   ptr(bt_host), ptr(sl_host), ptr(y_host), stream_handle(stream)))


def layer_step_host_async(plan: Plan, w: dict, x_host, k_pool, v_pool, bt_host, sl_host, y_host,
                          stream=None):
    """nf_layer_step_host_async: enqueue a host-buffer step (pipelined copies);
    host_wait(plan) waits for every enqueued y."""
    ws = make_weights_struct(w)
    check(lib().nf_layer_step_host_async(plan.h, ctypes.byref(ws), ptr(x_host), ptr(k_pool), ptr(v_pool),
                                         ptr(bt_host), ptr(sl_host), ptr(y_host), stream_handle(stream)))


def host_wait(plan: Plan):
    check(lib().nf_plan_host_wait(plan.h))


def step_metadata(plan: Plan, block_table, seq_lens, stream=None):
    check(lib().nf_step_metadata(plan.h, ptr(block_table), ptr(seq_lens), stream_handle(stream)))


def attention(plan: Plan, q, k_pool, v_pool, block_table, seq_lens, o, stream=None):
    check(lib().nf_attention(plan.h, ptr(q), ptr(k_pool), ptr(v_pool), ptr(block_table),
                             ptr(seq_lens), ptr(o), stream_handle(stream)))


def attention_noalloc(shape, batch, q, k_pool, v_pool, block_table, seq_lens, o, stream=None):
    """nf_attention_noalloc: attention without a plan and without any device
    allocation (fixed working memory inside the library)."""
    s = make_shape(shape)
    b = make_batch_desc(batch, hint=False)
    check(lib().nf_attention_noalloc(ctypes.byref(s), ctypes.byref(b), ptr(q), ptr(k_pool),
                                     ptr(v_pool), ptr(block_table), ptr(seq_lens), ptr(o),
                                     stream_handle(stream)))


def attention_noalloc_poll(stream=None):
    """nf_attention_noalloc_poll: wait for the stream, then report and clear the
    device-side status of nf_attention_noalloc calls on the current device."""
    check(lib().nf_attention_noalloc_poll(stream_handle(stream)))


def rmsnorm(x, g, out, eps, stream=None):
    check(lib().nf_rmsnorm(ptr(x), ptr(g), ptr(out), x.shape[0], x.shape[1], eps, stream_handle(stream)))


def gemm(A, B, C, R=None, epilogue=NF_EPI_STORE, max_sms=0, stream=None):
    M, K = A.shape
    N = C.shape[1]
    check(lib().nf_gemm(ptr(A), ptr(B), ptr(C), ptr(R), M, N, K, epilogue, max_sms,
                        stream_handle(stream)))


def gemm_wrows(A, B, C, R=None, epilogue=NF_EPI_STORE, splits=0, max_sms=0, stream=None):
    """nf_gemm_wrows: the weight-row kernel (M <= 128 rows of A)."""
    M, K = A.shape
    N = C.shape[1]
    check(lib().nf_gemm_wrows(ptr(A), ptr(B), ptr(C), ptr(R), M, N, K, epilogue, splits, max_sms,
                              stream_handle(stream)))


def plan_search(shape, batch, profile_json=None, num_sms=152, n_layers=1):
    """Host-only plan search; n_layers > 1 scores the cross-layer window of
    nf_layers_step / nf_stack_step (predicted time of all the layers)."""
    o = nf_plan_opts()
    t = c_double()
    s = make_shape(shape)
    b = make_batch_desc(batch, True)
    prof = None if profile_json is None else profile_json.encode()
    if n_layers == 1:
        check(lib().nf_plan_search(ctypes.byref(s), ctypes.byref(b), prof, num_sms,
                                   ctypes.byref(o), ctypes.byref(t)))
    else:
        check(lib().nf_plan_search_layers(ctypes.byref(s), ctypes.byref(b), prof, num_sms,
                                          n_layers, ctypes.byref(o), ctypes.byref(t)))
    return o, t.value


def plan_predict(shape, batch, opts, profile_json=None, num_sms=152, n_layers=1):
    """Microseconds the search's model predicts for `opts` over n_layers layers."""
    t = c_double()
    s = make_shape(shape)
    b = make_batch_desc(batch, True)
    check(lib().nf_plan_predict(ctypes.byref(s), ctypes.byref(b),
                                None if profile_json is None else profile_json.encode(), num_sms,
                                n_layers, ctypes.byref(opts), ctypes.byref(t)))
    return t.value


def profile_step(shape, batch, n_layers, out_json):
    """nf_profile_step: the R -> P table measured in traced steps of this batch
    structure; writes out_json and registers it for the shape."""
    s = make_shape(shape)
    b = make_batch_desc(batch, True)
    check(lib().nf_profile_step(ctypes.byref(s), ctypes.byref(b), n_layers, out_json.encode()))


def profile_use(shape, json_path):
    """nf_profile_use: register (or, with None, forget) a profile for the shape."""
    s = make_shape(shape)
    check(lib().nf_profile_use(ctypes.byref(s), None if json_path is None else json_path.encode()))


def window_schedule(opts, n_layers):
    """The cross-layer window's issue order: [(kind, layer, nano, full)], kind
    "qkv" (then that nano-batch's attention), "o" or "ffn"."""
    n = c_int32()
    check(lib().nf_window_schedule(ctypes.byref(opts), n_layers, None, 0, ctypes.byref(n)))
    buf = (c_int32 * (4 * max(1, n.value)))()
    check(lib().nf_window_schedule(ctypes.byref(opts), n_layers, buf, n.value, ctypes.byref(n)))
    kinds = {0: "qkv", 1: "o", 2: "ffn"}
    return [(kinds[buf[4 * k]], buf[4 * k + 1], buf[4 * k + 2], buf[4 * k + 3]) for k in range(n.value)]


def device_sm_count():
    return lib().nf_device_sm_count()


# ---------------------------------------------------------------- runtime

class Runtime:
    """nf_runtime: requests in, greedy tokens out (batch formation, async
    scheduling, KV pages, online re-planning)."""

    def __init__(self, shape, b_dense, max_requests, max_pages_per_seq, num_pages, vocab,
                 eos_token=-1, replan_threshold=0.1, host_only=False):
        self.h = c_void_p()
        self._shape = make_shape(shape)
        self.opts = nf_runtime_opts(b_dense, max_requests, max_pages_per_seq, num_pages, vocab,
                                    eos_token, replan_threshold, 1 if host_only else 0)
        self.max_pages = max_pages_per_seq
        check(lib().nf_runtime_create(ctypes.byref(self._shape), ctypes.byref(self.opts),
                                      ctypes.byref(self.h)))

    def submit(self, prompt, max_new_tokens):
        arr = (c_int32 * len(prompt))(*[int(t) for t in prompt])
        rid = c_int32()
        check(lib().nf_runtime_submit(self.h, arr, len(prompt), max_new_tokens, ctypes.byref(rid)))
        return rid.value

    @staticmethod
    def _view(b, max_pages):
        n, ns = b.n_tokens, b.n_decode + b.n_prefill
        get = lambda p, k: [p[i] for i in range(k)] if k else []  # noqa: E731
        return {"iteration": b.iteration, "n_tokens": n, "n_decode": b.n_decode,
                "n_prefill": b.n_prefill, "row_request": get(b.row_request, n),
                "row_pos": get(b.row_pos, n), "row_token": get(b.row_token, n),
                "row_emit": get(b.row_emit, n), "seq_lens": get(b.seq_lens, ns),
                "block_table": get(b.block_table, ns * max_pages),
                "prefill_q_lens": get(b.prefill_q_lens, b.n_prefill),
                "replanned": b.replanned, "free_pages": b.free_pages}

    def form(self):
        b = nf_runtime_batch()
        check(lib().nf_runtime_form(self.h, ctypes.byref(b)))
        return self._view(b, self.max_pages)

    def apply(self, iteration, sampled):
        arr = (c_int32 * max(1, len(sampled)))(*[int(t) for t in sampled])
        check(lib().nf_runtime_apply(self.h, iteration, arr))

    def step(self, stack_args, stream=None):
        b = nf_runtime_batch()
        check(lib().nf_runtime_step(self.h, ctypes.byref(stack_args.w), stack_args.kps, stack_args.vps,
                                    stream_handle(stream), ctypes.byref(b)))
        return self._view(b, self.max_pages)

    def sync(self):
        check(lib().nf_runtime_sync(self.h))

    def logits(self):
        """The last launched iteration's logits ([emitting rows, vocab] bf16, CPU)."""
        import torch
        n = c_int32()
        check(lib().nf_runtime_logits(self.h, None, 0, ctypes.byref(n)))
        out = torch.empty(max(n.value, 1), self.opts.vocab, dtype=torch.bfloat16)
        check(lib().nf_runtime_logits(self.h, ptr(out), n.value, ctypes.byref(n)))
        return out[: n.value]

    def result(self, rid, cap=4096):
        fin, n = c_int32(), c_int32()
        toks = (c_int32 * cap)()
        check(lib().nf_runtime_result(self.h, rid, ctypes.byref(fin), ctypes.byref(n), toks, cap))
        return bool(fin.value), [toks[i] for i in range(min(n.value, cap))]

    def counts(self):
        w, a, f = c_int32(), c_int32(), c_int32()
        check(lib().nf_runtime_counts(self.h, ctypes.byref(w), ctypes.byref(a), ctypes.byref(f)))
        return w.value, a.value, f.value

    def close(self):
        if self.h:
            lib().nf_runtime_destroy(self.h)
            self.h = c_void_p()

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass
