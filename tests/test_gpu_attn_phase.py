"""Attention as a phase of the GEMM chain (bf16), against the float64 oracle
and against the stand-alone attention kernel.

The model shape has grouped KV heads (16 query / 4 KV heads x 64, d 1024, FFN
2816, vocab 32000; 2 layers), so 4 rows per sequence fill the 16 query vectors
the phase takes per (sequence, KV head).  Committed contexts are chosen around
the phase's 64-slot units: a context shorter than one unit, new rows ending
exactly on a unit boundary, one slot past it, two full units, and a long
context whose units spread over many CTAs (partial states merged across CTAs).

* chain verification of 4 tokens per sequence (causal among the new rows);
* tree verification of a root with three children (ancestor-only mask).

Both paths must match the oracle's logits within 2e-2 and each other within
2e-3; the chained path must use fewer launches (the attention joins the
layer's GEMM launch; GEMMs this small otherwise launch one by one).
"""
import os

import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, model_pair
from oracle import spec as OS
from synthetic import SHAPES, ModelShape, make_kv_context, make_tokens

pytestmark = pytest.mark.gpu

TOL = 2e-2
N_LAYERS = 2


# 2 query heads per KV head (head dim 64): 1, 2 and 3 rows give 2, 4 and 6 query
# vectors per (sequence, KV head) -- both CUDA-core variants and the MMA path
GQA2 = ModelShape(2, 256, 4, 2, 64, 512, 2048, 0, "bf16")


def _models(max_batch, max_position, seed, shape0=None):
    """(phase model, stand-alone model, oracle decoder, shape) on the same weights."""
    pair = []
    for env in ("1", "0"):
        os.environ["SPEC_ATTN_PHASE"] = env
        try:
            model, dec, shape = model_pair(shape0 or SHAPES["tree8"], seed=seed, n_layers=N_LAYERS, max_rows=64,
                                           max_batch=max_batch, max_position=max_position)
        finally:
            os.environ.pop("SPEC_ATTN_PHASE", None)
        pair.append(model)
    return pair[0], pair[1], dec, shape


def _contexts(model, dec, shape, lens, cap, seed):
    from speculative_decoding_verify_04_gb300 import spec
    kv = spec.KVCache(model, len(lens), cap)
    caches = []
    for b, n in enumerate(lens):
        kc, vc = make_kv_context(shape, 1, n, seed * 100 + b, device="cuda")
        kv.import_rows(b, 0, kc[:, 0].contiguous(), vc[:, 0].contiguous())
        c = dec.new_cache(cap)
        c.load(kc[:, 0].float().cpu().numpy(), vc[:, 0].float().cpu().numpy())
        caches.append(c)
    kv.set_lengths(list(lens))
    return kv, caches


def _run_verify(model, kv, n_rows, tokens, parents=None, vocab=None):
    from speculative_decoding_verify_04_gb300 import spec
    T = sum(n_rows)
    logits = torch.empty((T, vocab or SHAPES["tree8"].vocab), dtype=torch.float32, device="cuda")
    before = model.launch_count()
    spec.spec_verify(model, kv, n_rows, tokens, tokens.shape[1], tree_parent=parents, logits=logits)
    torch.cuda.synchronize()
    assert model.device_error() == 0
    return logits.cpu().numpy(), model.launch_count() - before


@pytest.mark.parametrize("lens", [[3, 60, 61, 124, 1000]])
def test_attention_phase_chain_gqa(lens):
    lib()
    T_b = 4
    cap = max(lens) + 16
    fused, plain, dec, shape = _models(len(lens), cap + 8, seed=61)
    toks = make_tokens(len(lens) * T_b, shape.vocab, seed=62).reshape(len(lens), T_b)
    tk = cuda_i32(toks)
    out = []
    for model in (fused, plain):
        kv, caches = _contexts(model, dec, shape, lens, cap, seed=63)
        lg, launches = _run_verify(model, kv, [T_b] * len(lens), tk)
        out.append((lg, launches))
    (lf, nf), (lp, n_p) = out
    assert nf + N_LAYERS <= n_p, (nf, n_p)
    worst = 0.0
    for b, s in enumerate(lens):
        ref = OS.verify(dec, caches[b], s, dec.embed(toks[b]), 0)
        rows = slice(b * T_b, (b + 1) * T_b)
        e_f = np.abs(lf[rows] - ref).max()
        e_p = np.abs(lp[rows] - ref).max()
        assert e_f < TOL and e_p < TOL, (b, s, e_f, e_p)
        worst = max(worst, e_f)
    d = np.abs(lf - lp).max()
    assert d < 2e-3, d
    print(f"phase vs oracle {worst:.3g}, phase vs stand-alone kernel {d:.3g}")


def test_attention_phase_tree_gqa():
    lib()
    lens = [100, 777]
    parents = [-1, 0, 0, 0]
    cap = max(lens) + 16
    fused, plain, dec, shape = _models(len(lens), cap + 8, seed=71)
    toks = make_tokens(len(lens) * 4, shape.vocab, seed=72).reshape(len(lens), 4)
    tk = cuda_i32(toks)
    out = []
    for model in (fused, plain):
        kv, caches = _contexts(model, dec, shape, lens, cap, seed=73)
        out.append(_run_verify(model, kv, [4] * len(lens), tk, parents))
    (lf, nf), (lp, n_p) = out
    assert nf + N_LAYERS <= n_p, (nf, n_p)
    for b, s in enumerate(lens):
        ref = OS.verify(dec, caches[b], s, dec.embed(toks[b]), 0, parents=parents)
        rows = slice(b * 4, (b + 1) * 4)
        assert np.abs(lf[rows] - ref).max() < TOL
        assert np.abs(lp[rows] - ref).max() < TOL
    assert np.abs(lf - lp).max() < 2e-3


@pytest.mark.parametrize("n_rows", [[1] * 5, [2] * 5, [3] * 5, [4] * 5, [1, 5, 3, 2, 6]],
                         ids=["q2", "q4", "q6", "q8", "ragged"])
def test_attention_phase_small_query_groups(n_rows):
    """2 query vectors per (sequence, KV head) take the CUDA-core path over plain
    row copies; 4 to 8 take the tensor-box layout and the MMA path; a ragged
    batch with up to 12 mixes both paths over the tensor-box layout.  Contexts
    below, at and past one unit, and over several units."""
    lib()
    lens = [5, 60, 64, 200, 700]
    cap = max(lens) + 16
    fused, plain, dec, shape = _models(len(lens), cap + 8, seed=81 + sum(n_rows), shape0=GQA2)
    W = max(n_rows)
    toks = make_tokens(len(lens) * W, shape.vocab, seed=82).reshape(len(lens), W)
    tk = cuda_i32(toks)
    out = []
    for model in (fused, plain):
        kv, caches = _contexts(model, dec, shape, lens, cap, seed=83)
        out.append(_run_verify(model, kv, n_rows, tk, vocab=shape.vocab))
    (lf, nf), (lp, n_p) = out
    assert nf + N_LAYERS <= n_p, (nf, n_p)
    r0 = 0
    for b, s in enumerate(lens):
        n = n_rows[b]
        ref = OS.verify(dec, caches[b], s, dec.embed(toks[b, :n]), 0)
        rows = slice(r0, r0 + n)
        e_f, e_p = np.abs(lf[rows] - ref).max(), np.abs(lp[rows] - ref).max()
        assert e_f < TOL and e_p < TOL, (b, s, e_f, e_p)
        r0 += n
    assert np.abs(lf - lp).max() < 2e-3
