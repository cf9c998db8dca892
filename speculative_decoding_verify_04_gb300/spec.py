"""Thin Python binding of libspec.so (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks shapes, passes raw device pointers of torch
tensors and the current CUDA stream, and raises :class:`SpecError` with the
library's message on a non-zero status.  If the compiled library is missing
the loader raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_double, c_float, c_int32, c_void_p

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libspec.so")

SPEC_DTYPE_F32 = 0
SPEC_DTYPE_BF16 = 1
DEVERR_TOKEN, DEVERR_CAPACITY, DEVERR_TIMEOUT, DEVERR_POSITION, DEVERR_TREE = 1, 2, 4, 8, 16
MAX_SEQ_ROWS = 64
EXPORTS = [
    "spec_last_error", "spec_device_info", "spec_model_create", "spec_model_destroy", "spec_device_error",
    "spec_kv_create", "spec_kv_destroy", "spec_kv_set_lengths", "spec_kv_get_lengths", "spec_kv_import",
    "spec_kv_export", "spec_prefill", "spec_draft", "spec_verify", "spec_accept", "spec_accept_greedy",
    "kv_commit", "spec_row_probs", "spec_schedule_k", "spec_profile", "spec_profile_read", "spec_launch_count",
    "spec_verify_noalloc", "spec_draft_sample", "spec_probs", "spec_sample", "spec_schedule_aimd",
    "spec_schedule_decay", "spec_draft_tree", "spec_kv_create_paged", "spec_kv_free_pages", "spec_kv_page_table",
    "spec_draft_tree_dynamic", "spec_verify_trees", "spec_set_exit_layer", "spec_kv_read_page",
    "spec_test_stall_next_chain",
]


class SpecError(RuntimeError):
    pass


class ModelConfig(ctypes.Structure):
    _fields_ = [(n, c_int32) for n in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim", "d_ff",
                                       "vocab", "exit_layer", "dtype", "max_rows", "max_batch", "max_position")] + \
               [("rms_eps", c_float), ("rope_theta", c_float)]


class KSchedule(ctypes.Structure):
    _fields_ = [("min_k", c_int32), ("max_k", c_int32), ("low", c_double), ("high", c_double), ("decay", c_double),
                ("first_reject_min", c_int32)]


class AIMDSchedule(ctypes.Structure):
    _fields_ = [("window", c_int32), ("min_k", c_int32), ("max_k", c_int32), ("up_num", c_int32),
                ("up_den", c_int32), ("down_num", c_int32), ("down_den", c_int32)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libspec.so once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise SpecError(f"{path} is missing: build it with speculative_decoding_verify_04_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, I = c_void_p, c_int32
    sig = {
        "spec_last_error": ([], ctypes.c_char_p),
        "spec_device_info": ([POINTER(I), POINTER(I), POINTER(I)], I),
        "spec_model_create": ([POINTER(ModelConfig), POINTER(P), P, POINTER(P)], I),
        "spec_model_destroy": ([P], None),
        "spec_device_error": ([P, POINTER(I)], I),
        "spec_kv_create": ([P, I, I, POINTER(P)], I),
        "spec_kv_destroy": ([P], None),
        "spec_kv_set_lengths": ([P, POINTER(I), P], I),
        "spec_kv_get_lengths": ([P, POINTER(I), P], I),
        "spec_kv_import": ([P, I, I, I, I, I, P, P, P], I),
        "spec_kv_export": ([P, I, I, I, I, I, P, P, P], I),
        "spec_prefill": ([P, P, I, P, I, P, P, P], I),
        "spec_draft": ([P, P, I, P, I, P, P, P, P], I),
        "spec_verify": ([P, P, I, POINTER(I), P, I, P, I, POINTER(I), P, P, P, P, P, P], I),
        "spec_accept": ([P, P, P, I, P, I, I, I, P, P, P], I),
        "spec_draft_sample": ([P, P, I, P, I, c_float, P, P, P, P, P, P], I),
        "spec_probs": ([P, ctypes.c_int64, I, I, c_float, c_float, P, ctypes.c_int64, P], I),
        "spec_sample": ([P, ctypes.c_int64, I, I, P, P, P], I),
        "spec_schedule_aimd": ([P, P, P, I, POINTER(AIMDSchedule), P, P], I),
        "spec_schedule_decay": ([P, P, I, I, P, P], I),
        "spec_draft_tree": ([P, P, I, P, POINTER(I), I, P, P, P, P], I),
        "spec_draft_tree_dynamic": ([P, P, I, P, POINTER(I), I, c_float, P, P, P, P, P, P], I),
        "spec_set_exit_layer": ([P, I], I),
        "spec_verify_trees": ([P, P, I, POINTER(I), P, I, P, I, P, I, P, P, P, P, P, P], I),
        "spec_kv_create_paged": ([P, I, I, I, I, POINTER(P)], I),
        "spec_kv_free_pages": ([P, POINTER(I), P], I),
        "spec_kv_page_table": ([P, POINTER(I), P], I),
        "spec_kv_read_page": ([P, I, I, I, P, P], I),
        "spec_test_stall_next_chain": ([P, I, ctypes.c_int64], I),
        "spec_accept_greedy": ([P, P, POINTER(I), I, I, I, P, P, P, P], I),
        "kv_commit": ([P, I, P, P, I, P], I),
        "spec_row_probs": ([P, I, P, P], I),
        "spec_schedule_k": ([P, POINTER(I), P, P, I, POINTER(KSchedule), P, P, P], I),
        "spec_profile": ([P, I], I),
        "spec_profile_read": ([P, I, POINTER(c_double), POINTER(c_double), POINTER(I)], I),
        "spec_launch_count": ([P, POINTER(ctypes.c_int64)], I),
        "spec_verify_noalloc": ([P, P, I, POINTER(I), P, I, P, I, POINTER(I), P, P, P, P, P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(rc):
    if rc != 0:
        raise SpecError(f"libspec error {rc}: {_lib.spec_last_error().decode()}")


def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return c_void_p(s.cuda_stream)


def _i32_array(vals):
    vals = [int(v) for v in vals]
    return (c_int32 * len(vals))(*vals)


def _need(t, dtype, name, numel=None):
    if t is None:
        return
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise SpecError(f"{name}: need a contiguous CUDA {dtype} tensor")
    if numel is not None and t.numel() < numel:
        raise SpecError(f"{name}: needs at least {numel} elements, has {t.numel()}")


def device_info():
    lib = load()
    a, b, c = c_int32(), c_int32(), c_int32()
    _check(lib.spec_device_info(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


class Model:
    """A packed model on the current device (owns the library handle)."""

    def __init__(self, shape, weights, max_rows=64, max_batch=8, max_position=8192, stream=None):
        lib = load()
        self.shape = shape
        dt = SPEC_DTYPE_BF16 if shape.dtype == "bf16" else SPEC_DTYPE_F32
        self.torch_dtype = torch.bfloat16 if dt == SPEC_DTYPE_BF16 else torch.float32
        cfg = ModelConfig(shape.n_layers if weights is None else len(weights["layers"]), shape.d_model,
                          shape.n_heads, shape.n_kv_heads, shape.head_dim, shape.d_ff, shape.vocab,
                          shape.exit_layer, dt, max_rows, max_batch, max_position, shape.rms_eps, shape.rope_theta)
        self.cfg = cfg
        order = [weights["embed"], weights["lm_head"], weights["final_norm"]]
        for lw in weights["layers"]:
            order += [lw[k] for k in ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")]
        for t in order:
            _need(t, self.torch_dtype, "weight")
        arr = (c_void_p * len(order))(*[t.data_ptr() for t in order])
        h = c_void_p()
        _check(lib.spec_model_create(ctypes.byref(cfg), arr, _stream(stream), ctypes.byref(h)))
        self.handle = h
        self.n_layers = cfg.n_layers

    def test_stall_next_chain(self, cta, wait_ns):
        """Failure injection (tests): the next multi-phase GEMM chain launch has CTA
        ``cta`` withhold its first grid-barrier arrival and gives up after ``wait_ns``."""
        _check(load().spec_test_stall_next_chain(self.handle, cta, int(wait_ns)))

    def set_exit_layer(self, exit_layer):
        """Exit layer of the calls that follow (between rounds only)."""
        _check(load().spec_set_exit_layer(self.handle, int(exit_layer)))
        self.cfg.exit_layer = int(exit_layer)

    def profile(self, enable):
        _check(load().spec_profile(self.handle, 1 if enable else 0))

    def profile_read(self, kind):
        """(total ms, algorithmic bytes, launches) of kind 0 = GEMM, 1 = attention."""
        ms, by, n = c_double(), c_double(), c_int32()
        _check(load().spec_profile_read(self.handle, kind, ctypes.byref(ms), ctypes.byref(by), ctypes.byref(n)))
        return ms.value, by.value, n.value

    def launch_count(self):
        c = ctypes.c_int64()
        _check(load().spec_launch_count(self.handle, ctypes.byref(c)))
        return c.value

    def device_error(self):
        v = c_int32()
        _check(load().spec_device_error(self.handle, ctypes.byref(v)))
        return v.value

    def close(self):
        if getattr(self, "handle", None):
            load().spec_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class KVCache:
    """KV cache of ``batch`` sequences x ``max_ctx`` slots (owns the library handle).

    With ``page`` (a multiple of 64) the cache is paged: a pool of ``n_pages``
    pages of ``page`` slots shared by the sequences through their page tables.
    """

    def __init__(self, model: Model, batch, max_ctx, page=None, n_pages=None):
        self.model = model
        self.batch = batch
        self.max_ctx = max_ctx
        self.page = page
        h = c_void_p()
        if page:
            if n_pages is None:
                n_pages = batch * ((max_ctx + page - 1) // page)
            _check(load().spec_kv_create_paged(model.handle, batch, max_ctx, page, n_pages, ctypes.byref(h)))
        else:
            _check(load().spec_kv_create(model.handle, batch, max_ctx, ctypes.byref(h)))
        self.handle = h

    def free_pages(self, stream=None):
        n = c_int32()
        _check(load().spec_kv_free_pages(self.handle, ctypes.byref(n), _stream(stream)))
        return n.value

    def page_table(self, stream=None):
        cols = (self.max_ctx + self.page - 1) // self.page if self.page else 1
        arr = (c_int32 * (self.batch * cols))()
        _check(load().spec_kv_page_table(self.handle, arr, _stream(stream)))
        return [list(arr[b * cols:(b + 1) * cols]) for b in range(self.batch)]

    def read_page(self, which, layer, page, stream=None):
        """Raw physical page ``page`` of the K (which 0) or V (which 1) pool of
        ``layer``, read without the page table: host tensor [Hkv][page slots][hd]."""
        s = self.model.shape
        slots = self.page if self.page else self.max_ctx
        out = torch.empty((s.n_kv_heads, slots, s.head_dim), dtype=self.model.torch_dtype).pin_memory()
        _check(load().spec_kv_read_page(self.handle, which, layer, page, c_void_p(out.data_ptr()), _stream(stream)))
        return out

    def set_lengths(self, lens, stream=None):
        _check(load().spec_kv_set_lengths(self.handle, _i32_array(lens), _stream(stream)))

    def get_lengths(self, stream=None):
        arr = (c_int32 * self.batch)()
        _check(load().spec_kv_get_lengths(self.handle, arr, _stream(stream)))
        return list(arr)

    def import_rows(self, seq, layer0, k, v, slot0=0, stream=None):
        """k, v: CUDA tensors [n_layers][n_slots][Hkv][hd] in the model dtype."""
        _need(k, self.model.torch_dtype, "k")
        _need(v, self.model.torch_dtype, "v")
        _check(load().spec_kv_import(self.handle, seq, layer0, k.shape[0], slot0, k.shape[1], _ptr(k), _ptr(v),
                                     _stream(stream)))

    def export_rows(self, seq, layer0, n_layers, slot0, n_slots, stream=None):
        s = self.model.shape
        k = torch.empty((n_layers, n_slots, s.n_kv_heads, s.head_dim), dtype=self.model.torch_dtype, device="cuda")
        v = torch.empty_like(k)
        _check(load().spec_kv_export(self.handle, seq, layer0, n_layers, slot0, n_slots, _ptr(k), _ptr(v),
                                     _stream(stream)))
        return k, v

    def close(self):
        if getattr(self, "handle", None):
            load().spec_kv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def spec_prefill(model, kv, seq, tokens, last_logits=None, next_tok=None, stream=None):
    _need(tokens, torch.int32, "tokens")
    _need(last_logits, torch.float32, "last_logits", model.cfg.vocab)
    _need(next_tok, torch.int32, "next_tok", 1)
    _check(load().spec_prefill(model.handle, kv.handle, seq, _ptr(tokens), tokens.numel(), _ptr(last_logits),
                               _ptr(next_tok), _stream(stream)))


def spec_draft(model, kv, t0, k, cand, h_L, draft_logits=None, stream=None):
    B = t0.numel()
    _need(t0, torch.int32, "t0")
    _need(cand, torch.int32, "cand", B * (k + 1))
    _need(h_L, torch.float32, "h_L", B * (k + 1) * model.cfg.d_model)
    _need(draft_logits, torch.float32, "draft_logits", B * k * model.cfg.vocab)
    _check(load().spec_draft(model.handle, kv.handle, B, _ptr(t0), k, _ptr(cand), _ptr(h_L), _ptr(draft_logits),
                             _stream(stream)))


def spec_draft_sample(model, kv, t0, k, temperature, u_draft, cand, h_L, q, draft_logits=None, stream=None):
    """Sampling draft: d_{j+1} drawn from q_j = softmax(draft logits / temperature)
    with ``u_draft[b, j]``; ``q`` [B, k, V] receives the draft distributions."""
    B = t0.numel()
    V = model.cfg.vocab
    _need(t0, torch.int32, "t0")
    _need(u_draft, torch.float32, "u_draft", B * k)
    _need(cand, torch.int32, "cand", B * (k + 1))
    _need(h_L, torch.float32, "h_L", B * (k + 1) * model.cfg.d_model)
    _need(q, torch.float32, "q", B * k * V)
    _need(draft_logits, torch.float32, "draft_logits", B * k * V)
    _check(load().spec_draft_sample(model.handle, kv.handle, B, _ptr(t0), k, float(temperature), _ptr(u_draft),
                                    _ptr(cand), _ptr(h_L), _ptr(q), _ptr(draft_logits), _stream(stream)))


def spec_draft_tree(model, kv, t0, tree_parent, tokens, h_L, logits, stream=None):
    """Layer-skip draft of a level-order token tree (children take their parent's
    best draft tokens).  tokens [B, n], h_L [B, n, d], logits [B * n, V] scratch."""
    B = t0.numel()
    n = len(tree_parent)
    _need(t0, torch.int32, "t0")
    _need(tokens, torch.int32, "tokens", B * n)
    _need(h_L, torch.float32, "h_L", B * n * model.cfg.d_model)
    _need(logits, torch.float32, "logits", B * n * model.cfg.vocab)
    _check(load().spec_draft_tree(model.handle, kv.handle, B, _ptr(t0), _i32_array(tree_parent), n, _ptr(tokens),
                                  _ptr(h_L), _ptr(logits), _stream(stream)))


def tree_size(branching):
    """Nodes of the full tree of a branching list (root included)."""
    n, w = 1, 1
    for b in branching:
        w *= int(b)
        n += w
    return n


def spec_draft_tree_dynamic(model, kv, t0, branching, mass, tokens, parents, n_nodes, h_L, logits, stream=None):
    """Layer-skip draft of a tree whose width follows the draft's confidence:
    each node of level l gets its fewest best draft tokens whose probability
    reaches ``mass`` (1 .. branching[l]).  tokens, parents [B, n_max], n_nodes [B],
    h_L [B, n_max, d], logits [B * n_max, V] scratch; n_max = tree_size(branching)."""
    B = t0.numel()
    n = tree_size(branching)
    _need(t0, torch.int32, "t0")
    _need(tokens, torch.int32, "tokens", B * n)
    _need(parents, torch.int32, "parents", B * n)
    _need(n_nodes, torch.int32, "n_nodes", B)
    _need(h_L, torch.float32, "h_L", B * n * model.cfg.d_model)
    _need(logits, torch.float32, "logits", B * n * model.cfg.vocab)
    _check(load().spec_draft_tree_dynamic(model.handle, kv.handle, B, _ptr(t0), _i32_array(branching), len(branching),
                                          float(mass), _ptr(tokens), _ptr(parents), _ptr(n_nodes), _ptr(h_L),
                                          _ptr(logits), _stream(stream)))


def spec_verify_trees(model, kv, n_rows, tokens, tok_stride, parents, par_stride, h_in=None, h_stride=0, logits=None,
                      stats=None, acc_len=None, next_tok=None, path=None, stream=None):
    """spec_verify with one tree a sequence: ``parents`` [B, par_stride] on the device."""
    B = len(n_rows)
    T = sum(int(n) for n in n_rows)
    _need(tokens, torch.int32, "tokens", B * tok_stride)
    _need(parents, torch.int32, "parents", B * par_stride)
    _need(h_in, torch.float32, "h_in", B * h_stride * model.cfg.d_model if h_in is not None else None)
    _need(logits, torch.float32, "logits", T * model.cfg.vocab)
    _need(stats, torch.float32, "stats", T * 4)
    _need(acc_len, torch.int32, "acc_len", B)
    _need(next_tok, torch.int32, "next_tok", B)
    _need(path, torch.int32, "path", B * MAX_SEQ_ROWS)
    _check(load().spec_verify_trees(model.handle, kv.handle, B, _i32_array(n_rows), _ptr(h_in), h_stride,
                                    _ptr(tokens), tok_stride, _ptr(parents), par_stride, _ptr(logits), _ptr(stats),
                                    _ptr(acc_len), _ptr(next_tok), _ptr(path), _stream(stream)))


def _rows2d(t, name):
    """A 2-D float32 CUDA view with unit inner stride: (pointer, rows, cols, row stride)."""
    if t is None or not t.is_cuda or t.dtype != torch.float32 or t.dim() != 2 or t.stride(1) != 1:
        raise SpecError(f"{name}: need a 2-D CUDA float32 tensor with contiguous rows")
    return c_void_p(t.data_ptr()), t.shape[0], t.shape[1], t.stride(0)


def spec_probs(logits, probs, temperature, top_p=1.0, stream=None):
    """Rows of ``probs`` = softmax(logits / temperature), cut to the top-p nucleus
    when ``top_p`` < 1 (a multiple of 2^-24).  Both are 2-D [rows, V] views."""
    lp, rows, V, ls = _rows2d(logits, "logits")
    pp, prow, pV, ps = _rows2d(probs, "probs")
    if prow < rows or pV != V:
        raise SpecError("probs: shape does not match logits")
    _check(load().spec_probs(lp, ls, rows, V, float(temperature), float(top_p), pp, ps, _stream(stream)))


def spec_sample(probs, u, tokens, stream=None):
    """One integer inverse-CDF draw per row of ``probs`` [rows, V] with ``u`` [rows]."""
    pp, rows, V, ps = _rows2d(probs, "probs")
    _need(u, torch.float32, "u", rows)
    _need(tokens, torch.int32, "tokens", rows)
    _check(load().spec_sample(pp, ps, rows, V, _ptr(u), _ptr(tokens), _stream(stream)))


def spec_verify(model, kv, n_rows, tokens, tok_stride, h_in=None, h_stride=0, tree_parent=None, logits=None,
                stats=None, acc_len=None, next_tok=None, path=None, stream=None, _entry="spec_verify"):
    B = len(n_rows)
    T = sum(int(n) for n in n_rows)
    _need(tokens, torch.int32, "tokens", B * tok_stride)
    _need(h_in, torch.float32, "h_in", B * h_stride * model.cfg.d_model if h_in is not None else None)
    _need(logits, torch.float32, "logits", T * model.cfg.vocab)
    _need(stats, torch.float32, "stats", T * 4)
    _need(acc_len, torch.int32, "acc_len", B)
    _need(next_tok, torch.int32, "next_tok", B)
    _need(path, torch.int32, "path", B * MAX_SEQ_ROWS)
    tp = _i32_array(tree_parent) if tree_parent is not None else None
    _check(getattr(load(), _entry)(model.handle, kv.handle, B, _i32_array(n_rows), _ptr(h_in), h_stride,
                                   _ptr(tokens), tok_stride, tp, _ptr(logits), _ptr(stats), _ptr(acc_len),
                                   _ptr(next_tok), _ptr(path), _stream(stream)))


def spec_verify_noalloc(model, kv, n_rows, tokens, tok_stride, **kw):
    """spec_verify whose per-call scratch is the library's static device array
    (for callers that cannot allocate device memory where they verify)."""
    spec_verify(model, kv, n_rows, tokens, tok_stride, _entry="spec_verify_noalloc", **kw)


def spec_accept(p, q, draft, u, acc_len, next_tok, stream=None):
    """Rejection-sampling acceptance.  ``draft`` is [B, k] with contiguous rows;
    a column slice such as ``cand[:, 1:]`` of the draft's candidates works."""
    B, k1, V = p.shape
    k = k1 - 1
    _need(p, torch.float32, "p")
    _need(q, torch.float32, "q", B * k * V)
    if (not draft.is_cuda or draft.dtype != torch.int32 or draft.dim() != 2 or draft.shape[0] < B
            or draft.shape[1] < k or draft.stride(1) != 1):
        raise SpecError("draft: need a [B, k] CUDA int32 tensor with contiguous rows")
    _need(u, torch.float32, "u", B * (k + 1))
    _need(acc_len, torch.int32, "acc_len", B)
    _need(next_tok, torch.int32, "next_tok", B)
    _check(load().spec_accept(_ptr(p), _ptr(q), _ptr(draft), draft.stride(0), _ptr(u), B, k, V, _ptr(acc_len),
                              _ptr(next_tok), _stream(stream)))


def spec_accept_greedy(logits, tokens, acc_len, next_tok, tree_parent=None, path=None, stream=None):
    B, n, V = logits.shape
    _need(logits, torch.float32, "logits")
    _need(tokens, torch.int32, "tokens", B * n)
    _need(path, torch.int32, "path", B * MAX_SEQ_ROWS)
    tp = _i32_array(tree_parent) if tree_parent is not None else None
    _check(load().spec_accept_greedy(_ptr(logits), _ptr(tokens), tp, B, n, V, _ptr(acc_len), _ptr(next_tok),
                                     _ptr(path), _stream(stream)))


def kv_commit(kv, acc_len, path=None, path_stride=MAX_SEQ_ROWS, batch=None, stream=None):
    _need(acc_len, torch.int32, "acc_len")
    _need(path, torch.int32, "path")
    B = acc_len.numel() if batch is None else batch
    _check(load().kv_commit(kv.handle, B, _ptr(acc_len), _ptr(path), path_stride, _stream(stream)))


def spec_row_probs(stats, out, rows=None, stream=None):
    rows = stats.shape[0] if rows is None else rows
    _need(stats, torch.float32, "stats", rows * 4)
    _need(out, torch.float64, "out", rows * 2)
    _check(load().spec_row_probs(_ptr(stats), rows, _ptr(out), _stream(stream)))


def spec_schedule_k(top_probs, n_rows, acc_len, ema, k_next, conf=None, min_k=2, max_k=16, low=0.3, high=0.8,
                    decay=0.9, first_reject_min=False, stream=None):
    B = len(n_rows)
    _need(top_probs, torch.float64, "top_probs", 2 * sum(n_rows))
    _need(acc_len, torch.int32, "acc_len", B)
    _need(ema, torch.float64, "ema", B)
    _need(k_next, torch.int32, "k_next", B)
    _need(conf, torch.float64, "conf", B)
    sch = KSchedule(min_k, max_k, low, high, decay, 1 if first_reject_min else 0)
    _check(load().spec_schedule_k(_ptr(top_probs), _i32_array(n_rows), _ptr(acc_len), _ptr(ema), B,
                                  ctypes.byref(sch), _ptr(k_next), _ptr(conf), _stream(stream)))


def aimd_state(batch, window=64, device="cuda"):
    """Zeroed per-sequence window state for spec_schedule_aimd."""
    return torch.zeros((batch, 2 * window + 2), dtype=torch.int32, device=device)


def spec_schedule_aimd(acc_len, k_cur, state, k_next, window=64, min_k=2, max_k=8, up=(85, 100), down=(7, 10),
                       stream=None):
    """Additive increase / decrease of k over the last ``window`` rounds."""
    B = acc_len.numel()
    _need(acc_len, torch.int32, "acc_len", B)
    _need(k_cur, torch.int32, "k_cur", B)
    _need(state, torch.int32, "state", B * (2 * window + 2))
    _need(k_next, torch.int32, "k_next", B)
    sch = AIMDSchedule(window, min_k, max_k, up[0], up[1], down[0], down[1])
    _check(load().spec_schedule_aimd(_ptr(acc_len), _ptr(k_cur), _ptr(state), B, ctypes.byref(sch), _ptr(k_next),
                                     _stream(stream)))


def spec_schedule_decay(generated, total, k_max, k_next, stream=None):
    """k_next = max(1, round(k_max * (1 - generated / total))), ties to even."""
    B = generated.numel()
    _need(generated, torch.int32, "generated", B)
    _need(total, torch.int32, "total", B)
    _need(k_next, torch.int32, "k_next", B)
    _check(load().spec_schedule_decay(_ptr(generated), _ptr(total), B, int(k_max), _ptr(k_next), _stream(stream)))


def stats_argmax(stats):
    """argmax column of a [rows, 4] float32 stats tensor (spec_row_stats)."""
    return stats.view(torch.int32)[:, 3]
