"""Pins of the oracle's draft / verify / round loop on the tiny fp32 model.

* greedy self-speculative output equals plain greedy decoding token for token
  (self-speculative decoding page, §5.2: the lossless check);
* an all-accepted round emits k+1 tokens and a first-position rejection
  emits exactly one (same page, §2.1);
* the draft's first-L KV equals a full forward's first-L KV (KV reuse, §2.1);
* the draft logits are the layer-L hidden state through the final norm and
  LM head of a full forward;
* after many rounds a fresh prefill of the committed tokens reproduces every
  committed KV row and the write pointer equals the committed count (§3.3);
* a tree with unit branching verifies exactly like a chain.
"""
import numpy as np
import pytest

from oracle import spec as S
from oracle.accept import accept_greedy_chain, accept_greedy_tree, argmax_lowest
from synthetic import SHAPES, ModelShape, make_tokens, make_weights, weights_to_numpy, tree_parents
from oracle.decoder import Decoder


PROMPT_LEN, N_NEW = 32, 64


@pytest.fixture(scope="module")
def tiny():
    shape = SHAPES["tiny"]
    return Decoder(shape, weights_to_numpy(make_weights(shape, seed=1)))


@pytest.fixture(scope="module")
def prompt():
    return make_tokens(PROMPT_LEN, SHAPES["tiny"].vocab, seed=1)


@pytest.fixture(scope="module")
def ar_tokens(tiny, prompt):
    return S.generate_greedy_ar(tiny, prompt, N_NEW)


@pytest.mark.parametrize("k", [1, 4, 7])
def test_greedy_spec_equals_greedy_ar(tiny, prompt, ar_tokens, k):
    log = []
    out = S.generate_greedy_spec(tiny, prompt, N_NEW, k, log=log)
    assert out == ar_tokens
    assert all(0 <= a <= k for _, a in log)


def test_greedy_spec_equals_ar_deeper_draft():
    shape = ModelShape(4, 64, 4, 2, 16, 128, 96, 2, "f32", init_std=0.2)
    dec = Decoder(shape, weights_to_numpy(make_weights(shape, seed=8)))
    pr = make_tokens(10, shape.vocab, seed=8)
    ar = S.generate_greedy_ar(dec, pr, 40)
    log = []
    assert S.generate_greedy_spec(dec, pr, 40, 3, log=log) == ar
    assert any(a > 0 for _, a in log)        # the 2-of-4-layer draft is kept sometimes


def _planted_round(dec, prompt, draft_tokens, k):
    cache = dec.new_cache(PROMPT_LEN + k + 4)
    t0 = argmax_lowest(dec.prefill(cache, prompt))
    s = cache.length
    L = dec.shape.exit_layer
    hs = []
    for j, tok in enumerate([t0] + list(draft_tokens)):
        h = dec.run_layers(dec.embed([tok]), 0, L, [s + j], [s + j], [np.arange(s + j + 1)], cache)
        hs.append(h[0])
    logits = S.verify(dec, cache, s, np.stack(hs), L)
    return accept_greedy_chain(draft_tokens, logits)


def test_round_bounds(tiny, prompt, ar_tokens):
    k = 4
    a, nxt = _planted_round(tiny, prompt, ar_tokens[1:k + 1], k)
    assert a == k and nxt == ar_tokens[k + 1]                # k + 1 tokens emitted
    bad = list(ar_tokens[1:k + 1])
    bad[0] = (bad[0] + 1) % tiny.shape.vocab
    a, nxt = _planted_round(tiny, prompt, bad, k)
    assert a == 0 and nxt == ar_tokens[1]                    # exactly one token emitted


def test_draft_kv_and_logits_match_full_forward(tiny, prompt):
    k = 3
    cache = tiny.new_cache(PROMPT_LEN + k + 2)
    t0 = argmax_lowest(tiny.prefill(cache, prompt))
    s = cache.length
    d, hL, dlog, _ = S.draft(tiny, cache, s, t0, k)
    seq = np.concatenate([prompt, [t0], d])
    ref = tiny.new_cache(len(seq))
    L = tiny.shape.exit_layer
    n = len(seq)
    h = tiny.run_layers(tiny.embed(seq), 0, L, np.arange(n), np.arange(n),
                        [np.arange(t + 1) for t in range(n)], ref)
    for l in range(L):
        np.testing.assert_allclose(cache.k[l][:n], ref.k[l][:n], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(cache.v[l][:n], ref.v[l][:n], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(hL, h[s:s + k + 1], rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dlog, tiny.logits(h[s:s + k]), rtol=1e-10, atol=1e-12)
    assert d == [argmax_lowest(r) for r in tiny.logits(h[s:s + k])]


def test_committed_kv_matches_fresh_prefill(tiny, prompt):
    k = 4
    cache = tiny.new_cache(PROMPT_LEN + N_NEW + k + 2)
    t0 = argmax_lowest(tiny.prefill(cache, prompt))
    committed = list(prompt)
    for _ in range(10):
        s = cache.length
        emitted, a, nxt, _ = S.spec_round_greedy(tiny, cache, t0, k)
        committed += [t0] + emitted[:-1]
        assert cache.length == s + a + 1 == len(committed)   # write pointer == committed length
        t0 = nxt
    fresh = tiny.new_cache(len(committed))
    tiny.prefill(fresh, np.array(committed))
    n = len(committed)
    for l in range(tiny.n_layers):
        np.testing.assert_allclose(cache.k[l][:n], fresh.k[l][:n], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(cache.v[l][:n], fresh.v[l][:n], rtol=1e-9, atol=1e-11)


def test_unit_branching_tree_is_chain(tiny, prompt):
    k = 4
    toks = make_tokens(k + 1, tiny.shape.vocab, seed=3)
    c1, c2 = tiny.new_cache(PROMPT_LEN + 8), tiny.new_cache(PROMPT_LEN + 8)
    tiny.prefill(c1, prompt)
    tiny.prefill(c2, prompt)
    s = c1.length
    chain = S.verify(tiny, c1, s, tiny.embed(toks), 0)
    tree = S.verify(tiny, c2, s, tiny.embed(toks), 0, tree_parents([1] * k))
    np.testing.assert_array_equal(chain, tree)


def test_tree_rows_see_only_ancestors(tiny, prompt):
    """Changing a node's token changes only the rows of its subtree."""
    par = tree_parents([2, 2])
    toks = make_tokens(7, tiny.shape.vocab, seed=4)
    c1, c2 = tiny.new_cache(PROMPT_LEN + 8), tiny.new_cache(PROMPT_LEN + 8)
    tiny.prefill(c1, prompt)
    tiny.prefill(c2, prompt)
    s = c1.length
    a = S.verify(tiny, c1, s, tiny.embed(toks), 0, par)
    t2 = toks.copy()
    t2[1] = (t2[1] + 5) % tiny.shape.vocab          # node 1 has children 3, 4
    b = S.verify(tiny, c2, s, tiny.embed(t2), 0, par)
    changed = [i for i in range(7) if not np.array_equal(a[i], b[i])]
    assert changed == [1, 3, 4]


def test_tree_round_commit(tiny, prompt):
    par = tree_parents([2, 2])
    cache = tiny.new_cache(PROMPT_LEN + 10)
    t0 = argmax_lowest(tiny.prefill(cache, prompt))
    ar = S.generate_greedy_ar(tiny, prompt, 4)
    toks = make_tokens(7, tiny.shape.vocab, seed=5)
    toks[0] = t0
    toks[2] = ar[1]        # plant: node 2 (depth 1) and its child 6 (depth 2) on the greedy path
    toks[6] = ar[2]
    s = cache.length
    depth, node, path, nxt, logits = S.tree_round_greedy(tiny, cache, toks, par)
    assert (depth, node, path, nxt) == (2, 6, [0, 2, 6], ar[3])
    assert cache.length == s + 3
    fresh = tiny.new_cache(s + 3)
    tiny.prefill(fresh, np.concatenate([prompt, [t0, ar[1], ar[2]]]))
    for l in range(tiny.n_layers):
        np.testing.assert_allclose(cache.k[l][:s + 3], fresh.k[l][:s + 3], rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("top_p", [1.0, 0.875])
def test_sampling_round_at_cold_temperature_is_greedy(tiny, prompt, top_p):
    """At a temperature far below every logit gap each softmax row is one-hot
    (other weights floor to zero), so every draw is the argmax: the sampling
    round emits exactly what the greedy round emits."""
    k = 4
    rng = np.random.default_rng(21)
    for r in range(3):
        cg, cs = tiny.new_cache(PROMPT_LEN + 40), tiny.new_cache(PROMPT_LEN + 40)
        t0 = argmax_lowest(tiny.prefill(cg, prompt))
        tiny.prefill(cs, prompt)
        for _ in range(r + 1):
            eg, ag, ng, lg = S.spec_round_greedy(tiny, cg, t0, k)
            u_d = (rng.integers(0, 1 << 24, k) * 2.0 ** -24).astype(np.float32)
            u = (rng.integers(0, 1 << 24, k + 1) * 2.0 ** -24).astype(np.float32)
            es, as_, ns, d, q, p, ls = S.spec_round_sampling(tiny, cs, t0, k, 1e-9, top_p, u_d, u)
            gaps = np.sort(ls, axis=1)[:, -1] - np.sort(ls, axis=1)[:, -2]
            assert gaps.min() > 1e-6
            assert (es, as_, ns) == (eg, ag, ng) and cs.length == cg.length
            assert ((q == 0) | (q == 1)).all() and ((p == 0) | (p == 1)).all()
            t0 = ng


def test_sampling_round_keeps_identical_rows(tiny, prompt):
    """Draft and target at the same temperature: a draft token whose q and p rows
    agree there with u * q < p is kept; the round commits s + a + 1 and emits
    the kept tokens plus the draw."""
    k = 3
    cache = tiny.new_cache(PROMPT_LEN + 16)
    t0 = argmax_lowest(tiny.prefill(cache, prompt))
    s = cache.length
    u_d = np.array([0.5, 0.25, 0.75], dtype=np.float32)
    u = np.zeros(k + 1, dtype=np.float32)              # u = 0: every q(x) > 0 is kept
    em, a, nxt, d, q, p, _ = S.spec_round_sampling(tiny, cache, t0, k, 1.0, 1.0, u_d, u)
    assert a == k and em == list(d) + [nxt] and cache.length == s + k + 1
    assert (q[np.arange(k), d] > 0).all()


# -- layer-skip token trees ----------------------------------------------------
def test_top_children_order_and_ties():
    row = np.array([0.5, 2.0, -1.0, 2.0, 0.7, 2.0])
    assert S.top_children(row, 1) == [1]
    assert S.top_children(row, 4) == [1, 3, 5, 4]


@pytest.fixture(scope="module")
def deep():
    shape = ModelShape(4, 64, 4, 2, 16, 128, 96, 2, "f32", init_std=0.2)
    return Decoder(shape, weights_to_numpy(make_weights(shape, seed=8)))


def test_unit_branching_tree_draft_is_chain_draft(deep):
    pr = make_tokens(10, deep.shape.vocab, seed=8)
    k = 4
    c1, c2 = deep.new_cache(32), deep.new_cache(32)
    t0 = argmax_lowest(deep.prefill(c1, pr))
    deep.prefill(c2, pr)
    d, hL, lg, _ = S.draft(deep, c1, c1.length, t0, k)
    toks, hs, lgs = S.draft_tree(deep, c2, c2.length, t0, tree_parents([1] * k))
    assert toks == [t0] + list(d)
    np.testing.assert_array_equal(hs, hL)
    np.testing.assert_array_equal(lgs[:k], lg)
    for l in range(deep.shape.exit_layer):
        np.testing.assert_array_equal(c1.k[l][:c1.length + k + 1], c2.k[l][:c2.length + k + 1])


def test_tree_draft_children_are_the_parents_best_tokens(deep):
    pr = make_tokens(10, deep.shape.vocab, seed=9)
    par = tree_parents([3, 2, 2])
    c = deep.new_cache(64)
    t0 = argmax_lowest(deep.prefill(c, pr))
    toks, hs, lgs = S.draft_tree(deep, c, c.length, t0, par)
    for i in range(len(par)):
        kids = [j for j in range(len(par)) if par[j] == i]
        if kids:
            got = [toks[j] for j in kids]
            assert len(set(got)) == len(got) and got[0] == argmax_lowest(lgs[i])
            assert all(lgs[i][got[m]] >= lgs[i][got[m + 1]] for m in range(len(got) - 1))


@pytest.mark.parametrize("branching", [[3, 2], [4, 2, 2], [2, 2, 2, 2]])
def test_greedy_tree_spec_equals_greedy_ar(deep, branching):
    pr = make_tokens(10, deep.shape.vocab, seed=8)
    ar = S.generate_greedy_ar(deep, pr, 40)
    log = []
    assert S.generate_greedy_tree_spec(deep, pr, 40, tree_parents(branching), log=log) == ar
    assert any(d > 0 for _, d in log)


# -- dynamic tree width --------------------------------------------------------
def test_child_count_hand_example():
    # draft probabilities 0.15, 0.5, 0.05, 0.3 (ids 0..3): best first 1, 3, 0, 2
    row = np.log(np.array([0.15, 0.5, 0.05, 0.3])) + 3.0
    assert [S.child_count(row, 4, m) for m in (0.0, 0.49, 0.79, 0.81, 0.94, 0.96, 2.0)] == [1, 1, 2, 3, 3, 4, 4]
    assert S.child_count(row, 2, 0.96) == 2 and S.child_count(row, 1, 0.96) == 1
    # five equal logits: the mass counts probabilities (0.2 each), not logits
    assert S.child_count(np.zeros(5), 5, 0.5) == 3 and S.child_count(np.zeros(5), 5, 0.39) == 2


def test_dynamic_tree_without_mass_is_the_chain_draft(deep):
    pr = make_tokens(10, deep.shape.vocab, seed=8)
    c1, c2 = deep.new_cache(64), deep.new_cache(64)
    t0 = argmax_lowest(deep.prefill(c1, pr))
    deep.prefill(c2, pr)
    d, hL, lg, _ = S.draft(deep, c1, c1.length, t0, 3)
    toks, par, hs, lgs = S.draft_tree_dynamic(deep, c2, c2.length, t0, [4, 2, 2], 0.0)
    assert par == [-1, 0, 1, 2] and toks == [t0] + list(d)
    np.testing.assert_array_equal(hs, hL)
    np.testing.assert_array_equal(lgs[:3], lg)


def test_dynamic_tree_at_full_mass_is_the_static_tree(deep):
    pr = make_tokens(10, deep.shape.vocab, seed=9)
    c1, c2 = deep.new_cache(64), deep.new_cache(64)
    t0 = argmax_lowest(deep.prefill(c1, pr))
    deep.prefill(c2, pr)
    want = tree_parents([4, 2, 2])
    toks, hs, lgs = S.draft_tree(deep, c1, c1.length, t0, want)
    toks2, par, hs2, lgs2 = S.draft_tree_dynamic(deep, c2, c2.length, t0, [4, 2, 2], 2.0)
    assert par == [int(x) for x in want] and toks2 == toks
    np.testing.assert_array_equal(hs2, hs)
    np.testing.assert_array_equal(lgs2, lgs)


def _paths(tokens, parents):
    out = set()
    for i in range(len(tokens)):
        p, x = [], i
        while x >= 0:
            p.append(tokens[x])
            x = parents[x]
        out.add(tuple(reversed(p)))
    return out


def test_dynamic_trees_nest_and_follow_the_rule(deep):
    """A larger mass never removes a node: every token path of the tree at a
    smaller mass is a path of the tree at a larger one; each node's child count
    is child_count of its own draft row and its children are that row's best
    tokens in order; children are numbered in level order."""
    pr = make_tokens(12, deep.shape.vocab, seed=10)
    trees = []
    widths = set()
    for mass in (0.0, 0.3, 0.6, 0.9, 2.0):
        c = deep.new_cache(96)
        t0 = argmax_lowest(deep.prefill(c, pr))
        toks, par, hs, lgs = S.draft_tree_dynamic(deep, c, c.length, t0, [4, 2, 2], mass)
        depth = [0] + [0] * (len(par) - 1)
        for i in range(1, len(par)):
            assert 0 <= par[i] < i and par[i] >= par[i - 1]
            depth[i] = depth[par[i]] + 1
        for i in range(len(par)):
            kids = [j for j in range(len(par)) if par[j] == i]
            if depth[i] < 3:
                w = [4, 2, 2][depth[i]]
                assert len(kids) == S.child_count(lgs[i], w, mass)
                assert [toks[j] for j in kids] == S.top_children(lgs[i], len(kids))
                widths.add(len(kids))
            else:
                assert not kids
        trees.append(_paths(toks, par))
    for a, b in zip(trees, trees[1:]):
        assert a <= b
    assert len(trees[0]) == 4 and len(trees[-1]) == 29
    assert 1 in widths and len(widths) > 2


@pytest.mark.parametrize("mass", [0.3, 0.7, 0.95])
def test_greedy_dynamic_tree_spec_equals_greedy_ar(deep, mass):
    pr = make_tokens(10, deep.shape.vocab, seed=8)
    ar = S.generate_greedy_ar(deep, pr, 40)
    log = []
    assert S.generate_greedy_dynamic_tree_spec(deep, pr, 40, [4, 2, 2], mass, log=log) == ar
    assert any(d > 0 for _, d, _ in log)


# -- exit layer that follows the context length ------------------------------------
def test_exit_layer_for_context_table():
    table = [(0, 1), (16, 2), (40, 3)]
    assert [S.exit_layer_for_context(s, table) for s in (0, 15, 16, 39, 40, 1000)] == [1, 1, 2, 2, 3, 3]


def test_context_exit_layer_generation_is_lossless(deep):
    """The exit layer moves from 1 to 2 to 3 as the context grows: the output
    equals plain greedy decoding, and every layer of every committed row equals
    a fresh prefill of the committed tokens (each round wrote all its layers)."""
    pr = make_tokens(10, deep.shape.vocab, seed=8)
    n_new, k = 40, 3
    ar = S.generate_greedy_ar(deep, pr, n_new)
    log = []
    out, cache = S.generate_greedy_spec_context_exit(deep, pr, n_new, k, [(0, 1), (20, 2), (35, 3)], log=log)
    assert out == ar
    d3 = S.with_exit_layer(deep, 3)
    assert d3.shape.exit_layer == 3 and d3.w is deep.w and deep.shape.exit_layer == 2
    assert {L for _, L, _ in log} == {1, 2, 3}
    assert all(L == (1 if s < 20 else 2 if s < 35 else 3) for s, L, _ in log)
    n = min(cache.length, len(pr) + n_new - 1)
    committed = list(pr) + out[:n - len(pr)]
    fresh = deep.new_cache(n)
    deep.prefill(fresh, np.array(committed))
    for l in range(deep.n_layers):
        np.testing.assert_allclose(cache.k[l][:n], fresh.k[l][:n], rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(cache.v[l][:n], fresh.v[l][:n], rtol=1e-9, atol=1e-11)
