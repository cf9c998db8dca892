"""Pins of the oracle decoder against closed forms, invariants and special cases.

None of these re-types the oracle's own formulas: each checks a value the
mathematics fixes (a 2-D rotation, a one-key softmax, a single-token layer in
closed form, relative-position invariance, causality).
"""
import numpy as np
import pytest

from oracle import decoder as D
from oracle.decoder import Decoder, rms_norm, rope
from synthetic import ModelShape, make_weights, weights_to_numpy, make_tokens


def test_rms_norm_constant_vector():
    # x = c * 1: mean(x^2) = c^2, so RMSNorm(x) = c / sqrt(c^2 + eps) * g.
    for c in (-3.0, 0.5, 2.0):
        g = np.linspace(0.5, 1.5, 8)
        got = rms_norm(np.full(8, c), g, 1e-5)
        np.testing.assert_allclose(got, c / np.sqrt(c * c + 1e-5) * g, rtol=1e-14)


def test_rms_norm_unit_rms():
    x = np.random.default_rng(0).standard_normal((4, 64)) * 7
    y = rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-13)


def test_rope_two_dims_is_plane_rotation():
    # hd = 2: one pair, frequency theta^0 = 1, angle = pos.
    for pos in (0, 1, 7, 100):
        x = np.array([0.3, -1.2])
        th = float(pos)
        want = np.array([x[0] * np.cos(th) - x[1] * np.sin(th), x[1] * np.cos(th) + x[0] * np.sin(th)])
        np.testing.assert_allclose(rope(x, pos, 10000.0), want, rtol=1e-13, atol=1e-15)


def test_rope_pairs_and_frequencies():
    # hd = 8: dimension i pairs with i+4 and turns by pos * theta^(-2i/8).
    theta, pos = 500.0, 3
    x = np.arange(1.0, 9.0)
    y = rope(x, pos, theta)
    for i in range(4):
        a = pos * theta ** (-2 * i / 8)
        np.testing.assert_allclose(y[i], x[i] * np.cos(a) - x[i + 4] * np.sin(a), rtol=1e-13)
        np.testing.assert_allclose(y[i + 4], x[i + 4] * np.cos(a) + x[i] * np.sin(a), rtol=1e-13)


def test_rope_relative_position():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    a = rope(q, 10, 1e4) @ rope(k, 3, 1e4)
    b = rope(q, 1010, 1e4) @ rope(k, 1003, 1e4)
    np.testing.assert_allclose(a, b, rtol=1e-9)
    np.testing.assert_allclose(np.linalg.norm(rope(q, 77, 1e4)), np.linalg.norm(q), rtol=1e-13)
    np.testing.assert_allclose(rope(q, 0, 1e4), q, rtol=0, atol=0)


def _micro_shape(H=4, Hkv=2, hd=4, d=8, F=12, V=16, L=1, n_layers=2):
    return ModelShape(n_layers, d, H, Hkv, hd, F, V, L, "f32")


def _rand_weights(shape, seed=0):
    w = weights_to_numpy(make_weights(shape, seed=seed))
    rng = np.random.default_rng(seed)
    for lw in w["layers"]:           # non-unit gains so a dropped gain shows
        lw["attn_norm"] = rng.uniform(0.5, 1.5, shape.d_model).astype(np.float32)
        lw["ffn_norm"] = rng.uniform(0.5, 1.5, shape.d_model).astype(np.float32)
        for key in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
            lw[key] = (lw[key] * 20).astype(np.float32)
    w["final_norm"] = rng.uniform(0.5, 1.5, shape.d_model).astype(np.float32)
    return w


def test_single_token_layer_closed_form():
    """At position 0 with one visible key the softmax is 1 and RoPE is the identity,

    so one layer is  h + concat_h(v_{h // group}) Wo^T  followed by the SwiGLU
    residual; written out here with explicit matrix orientation and GQA grouping.
    """
    shape = _micro_shape()
    w = _rand_weights(shape)
    dec = Decoder(shape, w)
    cache = dec.new_cache(4)
    tok = 5
    h = dec.embed([tok])
    out = dec.layer(0, h, [0], [0], [np.array([0])], cache)

    W = w["layers"][0]
    h0 = w["embed"][tok].astype(np.float64)
    x = h0 / np.sqrt(np.mean(h0 ** 2) + shape.rms_eps) * W["attn_norm"]
    v = np.einsum("od,d->o", W["wv"].astype(np.float64), x).reshape(shape.n_kv_heads, shape.head_dim)
    grp = shape.n_heads // shape.n_kv_heads
    att = np.concatenate([v[hh // grp] for hh in range(shape.n_heads)])
    h1 = h0 + np.einsum("dj,j->d", W["wo"].astype(np.float64), att)
    x2 = h1 / np.sqrt(np.mean(h1 ** 2) + shape.rms_eps) * W["ffn_norm"]
    g = np.einsum("fd,d->f", W["w_gate"].astype(np.float64), x2)
    u = np.einsum("fd,d->f", W["w_up"].astype(np.float64), x2)
    h2 = h1 + np.einsum("df,f->d", W["w_down"].astype(np.float64), g / (1 + np.exp(-g)) * u)
    np.testing.assert_allclose(out[0], h2, rtol=1e-12, atol=1e-14)
    # the cache holds the unrotated (pos 0) K and the V row
    np.testing.assert_allclose(cache.v[0][0].reshape(-1), v.reshape(-1), rtol=1e-13)


def test_attention_two_keys_weights():
    # two visible keys: weights are the logistic of the scaled score difference
    shape = _micro_shape(H=2, Hkv=1, hd=4)
    dec = Decoder(shape, _rand_weights(shape))
    kc = np.zeros((4, 1, 4))
    vc = np.zeros((4, 1, 4))
    kc[0, 0] = [1, 0, 0, 0]
    kc[2, 0] = [0, 1, 0, 0]
    vc[0, 0] = [1, 2, 3, 4]
    vc[2, 0] = [-1, 0, 5, 1]
    q = np.array([[2.0, 0.5, 0, 0], [0.0, 0.0, 0, 0]])
    out = dec._attend(q, kc, vc, np.array([0, 2])).reshape(2, 4)
    w0 = 1.0 / (1.0 + np.exp(-(2.0 - 0.5) / 2.0))    # 1/sqrt(hd) = 1/2
    np.testing.assert_allclose(out[0], w0 * vc[0, 0] + (1 - w0) * vc[2, 0], rtol=1e-13)
    np.testing.assert_allclose(out[1], 0.5 * (vc[0, 0] + vc[2, 0]), rtol=1e-13)


def test_gqa_head_grouping():
    # H=4 over Hkv=2: heads 0,1 read KV head 0 and heads 2,3 read KV head 1.
    shape = _micro_shape(H=4, Hkv=2, hd=4)
    dec = Decoder(shape, _rand_weights(shape))
    kc = np.zeros((1, 2, 4))
    vc = np.zeros((1, 2, 4))
    vc[0, 0] = 1.0
    vc[0, 1] = -1.0
    out = dec._attend(np.ones((4, 4)), kc, vc, np.array([0])).reshape(4, 4)
    np.testing.assert_array_equal(out[:2], 1.0)
    np.testing.assert_array_equal(out[2:], -1.0)


@pytest.fixture(scope="module")
def micro():
    shape = _micro_shape(n_layers=3, L=2, V=32)
    return Decoder(shape, _rand_weights(shape, seed=3))


def test_incremental_equals_batched(micro):
    toks = make_tokens(9, micro.shape.vocab, 4)
    c1 = micro.new_cache(16)
    full = micro.prefill(c1, toks)
    c2 = micro.new_cache(16)
    micro.prefill(c2, toks[:5])
    for t in toks[5:]:
        from oracle.spec import decode_step
        last = decode_step(micro, c2, int(t))
    np.testing.assert_allclose(last, full, rtol=1e-10, atol=1e-12)
    for l in range(micro.n_layers):
        np.testing.assert_allclose(c1.k[l][:9], c2.k[l][:9], rtol=1e-10, atol=1e-12)


def test_causal(micro):
    toks = make_tokens(8, micro.shape.vocab, 5)
    c1 = micro.new_cache(8)
    c2 = micro.new_cache(8)
    a = micro.prefill(c1, toks[:5])
    micro.prefill(c2, np.concatenate([toks[:5], toks[5:] + 1]))
    # logits at row 4 do not depend on later tokens: recompute row 4 from c2's cache
    h = micro.run_layers(micro.embed(toks[:5]), 0, micro.n_layers, np.arange(5), np.arange(5),
                         [np.arange(t + 1) for t in range(5)], c2)
    np.testing.assert_allclose(micro.logits(h[-1:])[0], a, rtol=1e-12)


def test_position_shift_invariance(micro):
    """Attention sees only relative positions, so shifting every position id
    by the same amount leaves the logits unchanged."""
    toks = make_tokens(6, micro.shape.vocab, 6)
    c = micro.new_cache(6)
    vis = [np.arange(t + 1) for t in range(6)]
    h0 = micro.run_layers(micro.embed(toks), 0, micro.n_layers, np.arange(6), np.arange(6), vis, c)
    h1 = micro.run_layers(micro.embed(toks), 0, micro.n_layers, np.arange(6) + 4000, np.arange(6), vis, c)
    np.testing.assert_allclose(micro.logits(h1), micro.logits(h0), rtol=1e-8, atol=1e-10)


def test_rowwise_and_matrix_paths_agree(micro, monkeypatch):
    toks = make_tokens(12, micro.shape.vocab, 7)
    c1, c2 = micro.new_cache(12), micro.new_cache(12)
    a = micro.prefill(c1, toks)
    monkeypatch.setattr(D, "ROWWISE_MAX", 4)
    b = micro.prefill(c2, toks)
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-12)


def test_final_norm_applied(micro):
    # draft logits are the final-normed hidden state through the LM head: scaling
    # the hidden state must not change them (it would without the norm).
    h = np.random.default_rng(2).standard_normal((1, micro.shape.d_model))
    np.testing.assert_allclose(micro.logits(h * 37.0), micro.logits(h), rtol=1e-5, atol=1e-9)
