"""Float64 Llama-style decoder (oracle).  Test infrastructure only.

The pages build speculative decoding on a Hugging Face Llama-2 causal LM
(SPORK page, pwwt.cn/news/4102842, §2; FlashSpec page, lnrk.cn/news/47842,
§2.1).  None of them prints the block, so this module uses the plain Llama
reading:

    h0 = embed[token]
    per layer:  x = RMSNorm(h) ; q,k,v = x Wq^T, x Wk^T, x Wv^T
                q,k <- rotate-half RoPE at the row's position id
                o = softmax(q k^T / sqrt(hd) over the visible slots) v   (GQA)
                h = h + o Wo^T
                x = RMSNorm(h) ; h = h + (silu(x Wg^T) * (x Wu^T)) Wd^T
    logits = RMSNorm_final(h) Wlm^T

RMSNorm(x) = x / sqrt(mean(x^2) + eps) * g.  RoPE pairs dimension i with
i + hd/2 and rotates by pos * theta^(-2i/hd).  No biases; untied LM head.

The layer-skip draft of the self-speculative decoding page
(m.lqnn.cn/news/278124, §2.1 and §4.2) is ``run_layers(0, L)`` followed by
the same final norm and LM head; the page stresses that the final norm must
not be skipped (§3.1).

Every projection of a batch of at most ``ROWWISE_MAX`` rows is evaluated one
row at a time (matrix-vector product), and attention is evaluated one row at
a time, so a row's result does not depend on which other rows share its
batch: a batched verification is bit-identical to one-row decoding inside
the oracle.  Larger batches (prefill) use a matrix product.
"""
from __future__ import annotations

import numpy as np

ROWWISE_MAX = 64


def rms_norm(x, g, eps):
    """x / sqrt(mean(x^2) + eps) * g over the last axis (float64)."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=np.float64)


def rope(x, pos, theta):
    """Rotate-half rotary embedding of ``x [..., hd]`` at integer position ``pos``."""
    hd = x.shape[-1]
    half = hd // 2
    inv = np.asarray(theta, dtype=np.float64) ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = float(pos) * inv
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


def softmax(z):
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def linear(x, w):
    """``x [T, in] @ w[out, in]^T`` in float64."""
    w64 = np.asarray(w, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    if x.shape[0] <= ROWWISE_MAX:
        return np.stack([w64 @ x[t] for t in range(x.shape[0])]) if x.shape[0] else \
            np.zeros((0, w64.shape[0]))
    return x @ w64.T


class KVCache:
    """Per-sequence KV cache: ``k[l][slot, kvh, hd]`` and ``v[l][...]``.

    ``length`` is the committed length (slots ``[0, length)`` are valid).
    Slots beyond it hold draft / verify rows of the current round or stale
    rows of rejected candidates; they are never read unless a row's
    visibility set names them.
    """

    def __init__(self, n_layers, max_ctx, n_kv_heads, head_dim, dtype=np.float64):
        self.k = [np.zeros((max_ctx, n_kv_heads, head_dim), dtype=dtype) for _ in range(n_layers)]
        self.v = [np.zeros((max_ctx, n_kv_heads, head_dim), dtype=dtype) for _ in range(n_layers)]
        self.length = 0
        self.max_ctx = max_ctx

    def load(self, k_ctx, v_ctx):
        """Take a committed context ``[layer][slot][kvh][hd]`` (any float dtype)."""
        n = k_ctx.shape[1]
        for l in range(len(self.k)):
            self.k[l][:n] = k_ctx[l]
            self.v[l][:n] = v_ctx[l]
        self.length = n


class Decoder:
    """Oracle decoder over host weights from ``synthetic.weights_to_numpy``."""

    def __init__(self, shape, w):
        self.shape = shape
        self.w = w
        self.n_layers = len(w["layers"])

    # -- pieces -----------------------------------------------------------
    def new_cache(self, max_ctx, dtype=np.float64):
        s = self.shape
        return KVCache(self.n_layers, max_ctx, s.n_kv_heads, s.head_dim, dtype)

    def embed(self, tokens):
        return np.asarray(self.w["embed"][np.asarray(tokens, dtype=np.int64)], dtype=np.float64)

    def logits(self, h):
        """Final RMSNorm then the LM head: ``[T, V]`` float64."""
        x = rms_norm(h, self.w["final_norm"], self.shape.rms_eps)
        return linear(x, self.w["lm_head"])

    def _attend(self, q, kc, vc, visible):
        """One row: ``q [H, hd]`` over cache slots ``visible``; returns ``[H*hd]``."""
        s = self.shape
        grp = s.n_heads // s.n_kv_heads
        kv = kc[visible].astype(np.float64)     # [n, Hkv, hd]
        vv = vc[visible].astype(np.float64)
        scale = 1.0 / np.sqrt(s.head_dim)
        out = np.empty((s.n_heads, s.head_dim))
        for h in range(s.n_heads):
            g = h // grp
            sc = (kv[:, g, :] @ q[h]) * scale
            p = softmax(sc)
            out[h] = p @ vv[:, g, :]
        return out.reshape(-1)

    def layer(self, l, h, pos, slots, visible, cache):
        """Decoder layer ``l`` on rows ``h [T, d]``.

        Row t sits at rotary position ``pos[t]``, writes its K/V into cache
        slot ``slots[t]`` and attends to the cache slots ``visible[t]`` (which
        include its own slot).  All rows' K/V are written before any row
        attends, so rows of one batch can see each other.
        """
        s = self.shape
        W = self.w["layers"][l]
        T = h.shape[0]
        H, Hk, hd = s.n_heads, s.n_kv_heads, s.head_dim
        x = rms_norm(h, W["attn_norm"], s.rms_eps)
        q = linear(x, W["wq"]).reshape(T, H, hd)
        k = linear(x, W["wk"]).reshape(T, Hk, hd)
        v = linear(x, W["wv"]).reshape(T, Hk, hd)
        for t in range(T):
            q[t] = rope(q[t], pos[t], s.rope_theta)
            k[t] = rope(k[t], pos[t], s.rope_theta)
            cache.k[l][slots[t]] = k[t]
            cache.v[l][slots[t]] = v[t]
        if T <= ROWWISE_MAX:
            att = np.stack([self._attend(q[t], cache.k[l], cache.v[l], visible[t]) for t in range(T)])
        else:
            att = self._attend_causal_block(q, cache.k[l], cache.v[l], pos, slots, visible)
        h = h + linear(att, W["wo"])
        x = rms_norm(h, W["ffn_norm"], s.rms_eps)
        h = h + linear(silu(linear(x, W["w_gate"])) * linear(x, W["w_up"]), W["w_down"])
        return h

    def _attend_causal_block(self, q, kc, vc, pos, slots, visible):
        """Many-row attention (prefill): same math, matrix form per head.

        Each row's visibility set must be a prefix ``[0, n_t)`` of the cache.
        """
        s = self.shape
        T = q.shape[0]
        n = np.array([len(vs) for vs in visible])
        for t in range(T):
            assert visible[t][0] == 0 and visible[t][-1] == n[t] - 1
        ctx = int(n.max())
        kk = kc[:ctx].astype(np.float64)
        vv = vc[:ctx].astype(np.float64)
        grp = s.n_heads // s.n_kv_heads
        scale = 1.0 / np.sqrt(s.head_dim)
        mask = np.arange(ctx)[None, :] >= n[:, None]
        out = np.empty((T, s.n_heads, s.head_dim))
        for h in range(s.n_heads):
            g = h // grp
            sc = (q[:, h, :] @ kk[:, g, :].T) * scale
            sc[mask] = -np.inf
            out[:, h, :] = softmax(sc) @ vv[:, g, :]
        return out.reshape(T, -1)

    def run_layers(self, h, lo, hi, pos, slots, visible, cache):
        for l in range(lo, hi):
            h = self.layer(l, h, pos, slots, visible, cache)
        return h

    # -- whole passes -----------------------------------------------------
    def prefill(self, cache, tokens):
        """Causal pass of all layers over ``tokens`` at positions ``[s, s+n)``.

        Writes KV at slots ``[s, s+n)``, commits them, and returns the logits
        of the last row (the distribution of the first generated token).
        """
        s0 = cache.length
        n = len(tokens)
        pos = np.arange(s0, s0 + n)
        vis = [np.arange(0, s0 + t + 1) for t in range(n)]
        h = self.run_layers(self.embed(tokens), 0, self.n_layers, pos, pos, vis, cache)
        cache.length = s0 + n
        return self.logits(h[-1:])[0]
