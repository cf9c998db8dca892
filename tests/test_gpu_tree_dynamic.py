"""Layer-skip token trees of dynamic width on the GPU against the oracle
(FlashSpec page, lnrk.cn/news/47842, section 6.2: nodes the draft is sure
of are not widened; self-speculative decoding page, m.lqnn.cn/news/278124,
section 2.1: the first-L-layer draft).

spec_draft_tree_dynamic grows one tree a sequence on the device (a node's
child count is the fewest of its best draft tokens whose draft probability
reaches the mass, at most the level's branching); spec_verify_trees runs
layers [L, N) over each sequence's own tree and accepts the deepest matching
path; kv_commit compacts it.  Compared round by round with the oracle: the
tree's shape and tokens (exact unless the oracle's draft row holds a near-tie
at the cut or a cumulative mass within 5e-3 of the threshold), the layer-L
states and target logits (tolerance), the accepted depth, path and next token
(exact unless a near-tie on the path), the committed lengths and KV rows.
"""
import dataclasses

import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, model_pair, top_gap
from oracle import accept as A
from oracle import spec as OS
from oracle.accept import argmax_lowest
from synthetic import SHAPES, ModelShape, make_kv_context, make_tokens, tree_parents

pytestmark = pytest.mark.gpu

# f32, 4 layers, draft = first 2; draft logits sharp enough that the width varies
SHARP = ModelShape(4, 256, 4, 2, 64, 512, 512, 2, "f32", init_std=0.3)
BRANCHING = [4, 2, 2]


def _buffers(B, n, shape):
    dev = dict(dtype=torch.int32, device="cuda")
    return dict(tokens=torch.empty((B, n), **dev), parents=torch.empty((B, n), **dev),
                n_nodes=torch.empty(B, **dev),
                hL=torch.empty((B, n, shape.d_model), dtype=torch.float32, device="cuda"),
                scratch=torch.empty((B * n, shape.vocab), dtype=torch.float32, device="cuda"),
                acc=torch.empty(B, **dev), nxt=torch.empty(B, **dev), path=torch.full((B, 64), -1, **dev))


def _round_gpu(spec, model, kv, t0, mass, shape, buf, logits_out=True):
    B = t0.numel()
    n_max = spec.tree_size(BRANCHING)
    spec.spec_draft_tree_dynamic(model, kv, t0, BRANCHING, mass, buf["tokens"], buf["parents"], buf["n_nodes"],
                                 buf["hL"], buf["scratch"])
    n_host = buf["n_nodes"].tolist()
    T = sum(n_host)
    lg = torch.empty((T, shape.vocab), dtype=torch.float32, device="cuda") if logits_out else None
    spec.spec_verify_trees(model, kv, n_host, buf["tokens"], n_max, buf["parents"], n_max, h_in=buf["hL"],
                           h_stride=n_max, logits=lg, acc_len=buf["acc"], next_tok=buf["nxt"], path=buf["path"])
    spec.kv_commit(kv, buf["acc"], buf["path"])
    torch.cuda.synchronize()
    assert model.device_error() == 0
    return dict(n=n_host, tokens=buf["tokens"].cpu().numpy(), parents=buf["parents"].cpu().numpy(),
                hL=buf["hL"].cpu().numpy(), logits=lg.cpu().numpy() if lg is not None else None,
                acc=buf["acc"].cpu().numpy(), nxt=buf["nxt"].cpu().numpy(), path=buf["path"].cpu().numpy())


def _near_cut(row, width, mass, tol=5e-3):
    """True when the oracle's count or choice at this row is fragile: a
    cumulative draft probability within ``tol`` of the mass, or a near-tie
    between the logits ranked around the taken tokens."""
    z = np.asarray(row, dtype=np.float64)
    p = np.exp(z - z.max())
    p /= p.sum()
    srt = np.sort(z)[::-1]
    cum = np.cumsum(p[OS.top_children(row, width)])
    gaps = srt[:width] - srt[1:width + 1]
    return bool((np.abs(cum - mass) < tol).any() or (gaps < 1e-2).any())


def _check_round(b, dec, cache, t0, mass, got, shape, h_rel, logit_rel):
    """Oracle round for sequence b; False when a fragile decision ends the comparison."""
    s = cache.length
    toks_o, par_o, hs_o, lgs_o = OS.draft_tree_dynamic(dec, cache, s, t0, BRANCHING, mass)
    n = got["n"][b]
    row0 = sum(got["n"][:b])
    same = n == len(toks_o) and list(got["tokens"][b, :n]) == toks_o and \
        [-1] + list(got["parents"][b, 1:n]) == par_o
    if not same:
        depth = A.tree_depths(par_o)
        fragile = [i for i in range(len(par_o)) if depth[i] < len(BRANCHING)
                   and _near_cut(lgs_o[i], BRANCHING[depth[i]], mass)]
        assert fragile, (b, n, len(toks_o), list(got["tokens"][b, :n]), toks_o)
        return False
    # padding rows past the node count: token 0 under the root
    assert (got["tokens"][b, n:] == 0).all() and (got["parents"][b, n:] == 0).all()
    scale = np.abs(hs_o).max()
    assert np.abs(got["hL"][b, :n] - hs_o).max() / scale < h_rel
    vlog = OS.verify(dec, cache, s, hs_o, shape.exit_layer, parents=par_o)
    err = np.abs(got["logits"][row0:row0 + n] - vlog).max() / np.abs(vlog).max()
    assert err < logit_rel, err
    d, node, pth, n_ref = A.accept_greedy_tree(toks_o, par_o, vlog)
    if (got["acc"][b], got["nxt"][b]) != (d, n_ref) or list(got["path"][b, :d + 1]) != pth:
        assert min(top_gap(vlog[i]) for i in range(n)) < 1e-2
        return False
    moves, new_len = A.commit_tree_moves(s, pth)
    A.apply_moves(cache, moves)
    cache.length = new_len
    return True


def test_dynamic_tree_rounds_small_model():
    """Three sequences, six rounds in lockstep with the oracle at mass 0.8;
    the trees differ in shape between sequences and rounds."""
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    model, dec, shape = model_pair(SHARP, seed=8, max_rows=96, max_batch=3, max_position=512)
    B, cap, mass = 3, 256, 0.8
    n_max = spec.tree_size(BRANCHING)
    kv = spec.KVCache(model, B, cap)
    caches, t0 = [], []
    for b in range(B):
        pr = make_tokens(16, shape.vocab, seed=8 + b)
        spec.spec_prefill(model, kv, b, cuda_i32(pr))
        c = dec.new_cache(cap)
        t0.append(argmax_lowest(dec.prefill(c, pr)))
        caches.append(c)
    t0g = cuda_i32(t0)
    buf = _buffers(B, n_max, shape)
    alive = [True] * B
    sizes, compared = set(), 0
    for rnd in range(6):
        before = kv.get_lengths()
        got = _round_gpu(spec, model, kv, t0g, mass, shape, buf)
        after = kv.get_lengths()
        for b in range(B):
            n = got["n"][b]
            sizes.add(n)
            assert 1 < n <= n_max and 0 <= got["acc"][b] <= len(BRANCHING)
            assert after[b] == before[b] + got["acc"][b] + 1
            if alive[b]:
                alive[b] = _check_round(b, dec, caches[b], int(t0g[b].item()), mass, got, shape, 1e-3, 1e-3)
                if alive[b]:
                    compared += 1
                    assert caches[b].length == after[b]
                    d = int(got["acc"][b])
                    for layer in (0, shape.n_layers - 1):
                        kk, vv = kv.export_rows(b, layer, 1, before[b], d + 1)
                        np.testing.assert_allclose(kk[0].cpu().numpy(),
                                                   caches[b].k[layer][before[b]:before[b] + d + 1], atol=2e-3, rtol=0)
                        np.testing.assert_allclose(vv[0].cpu().numpy(),
                                                   caches[b].v[layer][before[b]:before[b] + d + 1], atol=2e-3, rtol=0)
        t0g = torch.from_numpy(got["nxt"]).cuda()
    assert compared >= B * 3
    assert len(sizes) > 2, sizes


@pytest.mark.parametrize("mass", [2.0, 0.0])
def test_dynamic_tree_limits_match_the_static_calls_bf16(mass, monkeypatch):
    """bf16 GQA model, three sequences on ragged contexts.  At mass 2 every
    node takes its full width: the dynamic draft and the per-sequence verify
    give the static tree calls' tokens, states, logits, path and next token
    bit for bit.  At mass 0 every tree is the chain of depth 3: the
    per-sequence verify equals spec_verify's tree mode with that chain's
    parents (the attention as its own kernel on both sides)."""
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    monkeypatch.setenv("SPEC_ATTN_PHASE", "0")
    # the GQA shape of the 8-layer tree workload, 3 layers, draft = the first one
    small = dataclasses.replace(SHAPES["tree8"], n_layers=3, exit_layer=1)
    model, dec, shape = model_pair(small, seed=41, max_rows=128, max_batch=3, max_position=1200)
    lens = [100, 700, 1000]
    B, cap = len(lens), 1100
    n_max = spec.tree_size(BRANCHING)
    kvs = []
    for _ in range(2):
        kv = spec.KVCache(model, B, cap)
        for b, n in enumerate(lens):
            kc, vc = make_kv_context(shape, 1, n, seed=500 + b, device="cuda")
            kv.import_rows(b, 0, kc[:, 0].contiguous(), vc[:, 0].contiguous())
        kv.set_lengths(lens)
        kvs.append(kv)
    t0 = cuda_i32(make_tokens(B, shape.vocab, seed=44))
    buf = _buffers(B, n_max, shape)
    dyn = _round_gpu(spec, model, kvs[0], t0, mass, shape, buf)
    par = [int(x) for x in (tree_parents(BRANCHING) if mass > 1 else [-1, 0, 1, 2])]
    n = len(par)
    assert dyn["n"] == [n] * B
    assert all(list(dyn["parents"][b, 1:n]) == par[1:] for b in range(B))
    if mass > 1:
        toks = torch.empty((B, n), dtype=torch.int32, device="cuda")
        hL = torch.empty((B, n, shape.d_model), dtype=torch.float32, device="cuda")
        spec.spec_draft_tree(model, kvs[1], t0, par, toks, hL, torch.empty((B * n, shape.vocab), dtype=torch.float32,
                                                                          device="cuda"))
        stride = n
    else:
        # the same chain tree from the dynamic call's own tokens and states
        toks = torch.from_numpy(np.ascontiguousarray(dyn["tokens"][:, :n])).cuda()
        hL = torch.from_numpy(np.ascontiguousarray(dyn["hL"][:, :n])).cuda()
        stride = n
    lg = torch.empty((B * n, shape.vocab), dtype=torch.float32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    path = torch.full((B, 64), -1, dtype=torch.int32, device="cuda")
    spec.spec_verify(model, kvs[1], [n] * B, toks, stride, h_in=hL, h_stride=stride, tree_parent=par, logits=lg,
                     acc_len=acc, next_tok=nxt, path=path)
    spec.kv_commit(kvs[1], acc, path)
    torch.cuda.synchronize()
    assert model.device_error() == 0
    if mass > 1:
        np.testing.assert_array_equal(dyn["tokens"][:, :n], toks.cpu().numpy())
        np.testing.assert_array_equal(dyn["hL"][:, :n], hL.cpu().numpy())
    np.testing.assert_array_equal(dyn["logits"], lg.cpu().numpy())
    np.testing.assert_array_equal(dyn["acc"], acc.cpu().numpy())
    np.testing.assert_array_equal(dyn["nxt"], nxt.cpu().numpy())
    for b in range(B):
        a = int(dyn["acc"][b])
        assert list(dyn["path"][b, :a + 1]) == list(path[b, :a + 1].cpu().numpy())
    assert kvs[0].get_lengths() == kvs[1].get_lengths()


def test_verify_trees_with_a_bad_parent_sets_the_error():
    """A device parent outside [0, node) is caught by the plan: the error bit
    is set, the node reads as a child of the root, and nothing faults."""
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    model, dec, shape = model_pair(SHAPES["tiny"], seed=1, max_rows=64, max_batch=2, max_position=512)
    kv = spec.KVCache(model, 2, 128)
    for b in range(2):
        spec.spec_prefill(model, kv, b, cuda_i32(make_tokens(20, shape.vocab, seed=70 + b)))
    toks = cuda_i32(make_tokens(2 * 5, shape.vocab, seed=71).reshape(2, 5))
    par = cuda_i32(np.array([[-1, 0, 0, 1, 2], [-1, 0, 1, 7, 3]], dtype=np.int32))   # 7 >= 3
    acc = torch.empty(2, dtype=torch.int32, device="cuda")
    nxt = torch.empty(2, dtype=torch.int32, device="cuda")
    path = torch.full((2, 64), -1, dtype=torch.int32, device="cuda")
    spec.spec_verify_trees(model, kv, [5, 5], toks, 5, par, 5, acc_len=acc, next_tok=nxt, path=path)
    torch.cuda.synchronize()
    assert model.device_error() & spec.DEVERR_TREE
    assert 0 <= int(acc[0]) <= 2 and 0 <= int(acc[1]) <= 3
