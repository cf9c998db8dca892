"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This module only draws data: model weights, prompts, token trees, KV
contexts, uniforms and the probability rows that the stand-alone acceptance
call consumes.  It holds none of the arithmetic of the method itself (no
decoder layer, no acceptance rule, no sampler), so the oracle and the CUDA
path can both take their inputs from here without sharing any computation.

Every stream is keyed by ``(seed, name)`` so a tensor does not change when
another tensor is added or drawn in a different order.

Workloads follow the synthetic recipes of the self-speculative decoding page
(m.lqnn.cn/news/278124, §1.1 and §2.3: a 7B half-precision Llama with a 12 of
32 layer draft), the FlashSpec page (lnrk.cn/news/47842, §2.2: a level-order
token tree) and the DSpark page (0539edu.com/news/4524681, §2.2-§2.3: the
confidence-scheduled draft length).  None of them names a dataset; all values
here are random.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, asdict

import numpy as np
import torch

__all__ = [
    "ModelShape", "SHAPES", "stream_seed", "make_weights", "weights_to_numpy",
    "make_tokens", "make_uniforms", "tree_parents", "make_kv_context",
    "make_accept_inputs", "make_ragged_contexts",
]


@dataclass(frozen=True)
class ModelShape:
    """Llama-style decoder dimensions (no biases, untied LM head)."""
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    exit_layer: int        # L: the draft runs layers [0, L)
    dtype: str             # "f32" or "bf16" storage of every weight
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0
    init_std: float = 0.02

    def asdict(self):
        return asdict(self)


SHAPES = {
    # 2 layers, d 256, 4 heads x 64, FFN 1024, vocab 1024, draft = layer 0.
    "tiny": ModelShape(2, 256, 4, 4, 64, 1024, 1024, 1, "f32"),
    # 8 layers, d 1024, 16 query heads / 4 KV heads x 64, FFN 2816, vocab 32000.
    "tree8": ModelShape(8, 1024, 16, 4, 64, 2816, 32000, 0, "bf16"),
    # 7B-shaped: 32 layers, d 4096, 32 heads x 128, FFN 11008, vocab 32000, draft = 12 layers.
    "llama7b": ModelShape(32, 4096, 32, 32, 128, 11008, 32000, 12, "bf16"),
}


def stream_seed(seed: int, name: str) -> int:
    """63-bit seed for the stream ``name`` under the run seed ``seed``."""
    h = hashlib.blake2b(f"{seed}:{name}".encode(), digest_size=8).digest()
    return int.from_bytes(h, "little") & ((1 << 63) - 1)


def _rng(seed: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(stream_seed(seed, name)))


def _normal(shape, std, seed, name, device, dtype):
    g = torch.Generator(device=device)
    g.manual_seed(stream_seed(seed, name))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(dtype)


def make_weights(shape: ModelShape, seed: int, device="cpu", n_layers: int | None = None):
    """Random-init weights N(0, std^2) for matrices and embeddings; norm gains 1.

    Returns a dict of torch tensors in the plain per-matrix layout
    ``[out_features, in_features]``: ``embed [V,d]``, ``lm_head [V,d]``,
    ``final_norm [d]`` and ``layers[i]`` with ``attn_norm [d]``,
    ``wq [H*hd, d]``, ``wk [Hkv*hd, d]``, ``wv [Hkv*hd, d]``, ``wo [d, H*hd]``,
    ``ffn_norm [d]``, ``w_gate [F, d]``, ``w_up [F, d]``, ``w_down [d, F]``.
    ``n_layers`` may draw fewer layers than the shape has (same streams).
    """
    dt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    d, H, Hk, hd, F, V = (shape.d_model, shape.n_heads, shape.n_kv_heads,
                          shape.head_dim, shape.d_ff, shape.vocab)
    std = shape.init_std
    nl = shape.n_layers if n_layers is None else n_layers
    w = {
        "embed": _normal((V, d), std, seed, "embed", device, dt),
        "lm_head": _normal((V, d), std, seed, "lm_head", device, dt),
        "final_norm": torch.ones(d, device=device, dtype=dt),
        "layers": [],
    }
    for i in range(nl):
        p = f"layer{i}."
        w["layers"].append({
            "attn_norm": torch.ones(d, device=device, dtype=dt),
            "wq": _normal((H * hd, d), std, seed, p + "wq", device, dt),
            "wk": _normal((Hk * hd, d), std, seed, p + "wk", device, dt),
            "wv": _normal((Hk * hd, d), std, seed, p + "wv", device, dt),
            "wo": _normal((d, H * hd), std, seed, p + "wo", device, dt),
            "ffn_norm": torch.ones(d, device=device, dtype=dt),
            "w_gate": _normal((F, d), std, seed, p + "w_gate", device, dt),
            "w_up": _normal((F, d), std, seed, p + "w_up", device, dt),
            "w_down": _normal((d, F), std, seed, p + "w_down", device, dt),
        })
    return w


def weights_to_numpy(w):
    """Host float32 copies (bf16 widens to f32 exactly)."""
    def cv(t):
        return t.detach().to("cpu", torch.float32).numpy()
    return {
        "embed": cv(w["embed"]), "lm_head": cv(w["lm_head"]),
        "final_norm": cv(w["final_norm"]),
        "layers": [{k: cv(v) for k, v in lw.items()} for lw in w["layers"]],
    }


def make_tokens(n, vocab, seed, name="prompt"):
    """``n`` token ids uniform over ``[0, vocab)`` as int32."""
    return _rng(seed, name).integers(0, vocab, size=n, dtype=np.int64).astype(np.int32)


def make_uniforms(shape, seed, name="uniform"):
    """U[0,1) as float32 values m * 2^-24 with integer m in [0, 2^24).

    Every value is exactly representable, so ``m = u * 2^24`` recovers the
    integer on any machine.
    """
    m = _rng(seed, name).integers(0, 1 << 24, size=shape, dtype=np.int64)
    return (m.astype(np.float64) * 2.0 ** -24).astype(np.float32)


def tree_parents(branching):
    """Parent index of every node of a level-order token tree.

    Node 0 is the root.  Level l holds ``prod(branching[:l])`` nodes, each
    node of level l-1 owning ``branching[l-1]`` consecutive children.  Returns
    an int32 array with ``parents[0] = -1``.
    """
    parents = [-1]
    level = [0]
    for b in branching:
        nxt = []
        for par in level:
            for _ in range(b):
                parents.append(par)
                nxt.append(len(parents) - 1)
        level = nxt
    return np.asarray(parents, dtype=np.int32)


def make_kv_context(shape: ModelShape, batch, ctx, seed, device="cpu", std=None):
    """Synthetic committed KV context ``[layer][b][slot][kvh][hd]`` for K and V.

    Stands in for a prefilled random prompt when the context is too long for
    the CPU oracle to prefill.  Values are N(0, std^2) with std defaulting to
    ``init_std * sqrt(d_model)``, the scale of a projection of a unit-RMS
    hidden state.  Stored in the model's dtype.
    """
    dt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    if std is None:
        std = shape.init_std * float(np.sqrt(shape.d_model))
    shp = (shape.n_layers, batch, ctx, shape.n_kv_heads, shape.head_dim)
    k = _normal(shp, std, seed, "kv.k", device, dt)
    v = _normal(shp, std, seed, "kv.v", device, dt)
    return k, v


def make_ragged_contexts(batch, lo, hi, seed):
    """Per-sequence context lengths uniform over the integers [lo, hi]."""
    return _rng(seed, "ragged_ctx").integers(lo, hi + 1, size=batch).astype(np.int32)


def _softmax64(z):
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def make_accept_inputs(batch, k, vocab, seed, sigma=3.0, noise=1.0, first=0):
    """Inputs of the stand-alone acceptance call.

    Target logits are i.i.d. N(0, sigma^2) at k+1 positions; draft logits are
    the first k target rows plus N(0, noise^2).  ``p`` and ``q`` are their
    softmax at temperature 1, formed in float64 and rounded to float32 once.
    Draft tokens ``x[b, j]`` are drawn from ``q[b, j]`` (float64 CDF,
    independent stream); ``u[b, :]`` holds k+1 uniforms (integer multiples of
    2^-24).  Every sequence has streams of its own, keyed by its index in the
    whole batch, ``first + b``: the sequences ``first .. first + batch - 1`` are
    the same whether they are drawn alone or as part of a larger batch (so a
    batch split over several processes reproduces the undivided one).
    """
    p = np.empty((batch, k + 1, vocab), dtype=np.float32)
    q = np.empty((batch, k, vocab), dtype=np.float32)
    x = np.empty((batch, k), dtype=np.int32)
    u = np.empty((batch, k + 1), dtype=np.float32)
    for b in range(batch):
        g = first + b
        rng = _rng(seed, f"accept.logits.{g}")
        zp = rng.standard_normal((k + 1, vocab)) * sigma
        zq = zp[:k, :] + rng.standard_normal((k, vocab)) * noise
        p[b] = _softmax64(zp).astype(np.float32)
        qb = _softmax64(zq)
        q[b] = qb.astype(np.float32)
        draw = _rng(seed, f"accept.draft.{g}").random(k)
        cdf = np.cumsum(qb, axis=-1)
        for j in range(k):
            x[b, j] = min(int(np.searchsorted(cdf[j], draw[j] * cdf[j, -1], side="right")), vocab - 1)
        m = _rng(seed, f"accept.u.{g}").integers(0, 1 << 24, size=k + 1, dtype=np.int64)
        u[b] = (m.astype(np.float64) * 2.0 ** -24).astype(np.float32)
    return p, q, x, u
