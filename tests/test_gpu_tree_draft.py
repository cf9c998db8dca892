"""Layer-skip token trees on the GPU against the oracle (FlashSpec page,
lnrk.cn/news/47842, sections 2.2 and 6.2; self-speculative decoding page,
m.lqnn.cn/news/278124, section 2.1).

spec_draft_tree grows the tree level by level from the first-L-layer draft
(children take their parent's best draft tokens), spec_verify runs layers
[L, N) over every node with the tree mask and picks the deepest accepted
path, kv_commit compacts that path.  Compared round by round with the
oracle: the tree's tokens (exact unless the parent's draft logits hold a
near-tie at the cut), the layer-L states and target logits (tolerance),
the accepted depth, path and next token (exact unless a near-tie on the
path), the committed lengths and the committed KV rows.
"""
import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, model_pair, top_gap
from oracle import accept as A
from oracle import spec as OS
from oracle.accept import argmax_lowest
from oracle.decoder import Decoder
from synthetic import (SHAPES, ModelShape, make_kv_context, make_tokens, make_weights, tree_parents,
                       weights_to_numpy)

pytestmark = pytest.mark.gpu

# f32, 4 layers, draft = first 2; weights large enough that the draft is often right
SMALL = ModelShape(4, 256, 4, 2, 64, 512, 512, 2, "f32", init_std=0.1)


def _cut_gap(row, c):
    """Gap between the c-th and (c+1)-th best logits of a row (ties at the cut)."""
    z = np.sort(np.asarray(row, dtype=np.float64))[::-1]
    return z[c - 1] - z[c] if c < len(z) else np.inf


def _kids(par):
    return {i: [j for j in range(len(par)) if par[j] == i] for i in range(len(par))}


def _tree_round_gpu(spec, model, kv, t0, par, shape):
    B, n = t0.numel(), len(par)
    tokens = torch.empty((B, n), dtype=torch.int32, device="cuda")
    hL = torch.empty((B, n, shape.d_model), dtype=torch.float32, device="cuda")
    scratch = torch.empty((B * n, shape.vocab), dtype=torch.float32, device="cuda")
    logits = torch.empty((B * n, shape.vocab), dtype=torch.float32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    path = torch.full((B, 64), -1, dtype=torch.int32, device="cuda")
    spec.spec_draft_tree(model, kv, t0, par, tokens, hL, scratch)
    spec.spec_verify(model, kv, [n] * B, tokens, n, h_in=hL, h_stride=n, tree_parent=par, logits=logits,
                     acc_len=acc, next_tok=nxt, path=path)
    spec.kv_commit(kv, acc, path)
    torch.cuda.synchronize()
    assert model.device_error() == 0
    return (tokens.cpu().numpy(), hL.cpu().numpy(), logits.cpu().numpy().reshape(B, n, -1), acc.cpu().numpy(),
            nxt.cpu().numpy(), path.cpu().numpy(), nxt)


def _check_round(b, dec, cache, t0, par, got, h_rel, logit_tol, shape):
    """Oracle round for sequence b; returns False when a near-tie ends the comparison."""
    tokens, hL, logits, acc, nxt, path, _ = got
    s = cache.length
    toks_o, hs_o, lgs_o = OS.draft_tree(dec, cache, s, t0, par)
    kids = _kids(par)
    for i, ks in kids.items():
        for m, c in enumerate(ks):
            if tokens[b, c] != toks_o[c]:
                assert _cut_gap(lgs_o[i], m + 1) < 1e-2, (b, i, c, tokens[b, c], toks_o[c])
                return False
    scale = np.abs(hs_o).max()
    assert np.abs(hL[b] - hs_o).max() / scale < h_rel, np.abs(hL[b] - hs_o).max() / scale
    vlog = OS.verify(dec, cache, s, hs_o, shape.exit_layer, parents=par)
    err = np.abs(logits[b] - vlog).max()
    assert err < logit_tol, err
    d, node, pth, n_ref = A.accept_greedy_tree(toks_o, par, vlog)
    if (acc[b], nxt[b]) != (d, n_ref) or list(path[b, :d + 1]) != pth:
        assert min(top_gap(vlog[i]) for i in range(len(par))) < 1e-2
        return False
    moves, new_len = A.commit_tree_moves(s, pth)
    A.apply_moves(cache, moves)
    cache.length = new_len
    return True


@pytest.mark.parametrize("branching", [[3, 2], [4, 2, 2]])
def test_tree_rounds_small_model(branching):
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    par = [int(x) for x in tree_parents(branching)]
    n = len(par)
    model, dec, shape = model_pair(SMALL, seed=8, max_rows=64, max_batch=2, max_position=512)
    B, prompt_len, cap = 2, 16, 256
    kv = spec.KVCache(model, B, cap)
    caches, t0 = [], []
    for b in range(B):
        pr = make_tokens(prompt_len, shape.vocab, seed=8 + b)
        spec.spec_prefill(model, kv, b, cuda_i32(pr))
        c = dec.new_cache(cap)
        t0.append(argmax_lowest(dec.prefill(c, pr)))
        caches.append(c)
    t0g = cuda_i32(t0)
    alive = [True] * B
    depths = []
    for rnd in range(6):
        before = kv.get_lengths()
        got = _tree_round_gpu(spec, model, kv, t0g, par, shape)
        acc, nxt = got[3], got[4]
        after = kv.get_lengths()
        for b in range(B):
            assert 0 <= acc[b] < n and 0 <= nxt[b] < shape.vocab
            assert after[b] == before[b] + acc[b] + 1
            if alive[b]:
                alive[b] = _check_round(b, dec, caches[b], int(t0g[b].item()), par, got, 2e-4, 2e-3,
                                        shape)
                if alive[b]:
                    assert caches[b].length == after[b]
                    d = int(acc[b])
                    depths.append(d)
                    # committed KV rows of the accepted path, first and last layer
                    for layer in (0, shape.n_layers - 1):
                        kk, vv = kv.export_rows(b, layer, 1, before[b], d + 1)
                        np.testing.assert_allclose(kk[0].cpu().numpy(), caches[b].k[layer][before[b]:before[b] + d + 1],
                                                   atol=2e-3, rtol=0)
                        np.testing.assert_allclose(vv[0].cpu().numpy(), caches[b].v[layer][before[b]:before[b] + d + 1],
                                                   atol=2e-3, rtol=0)
        t0g = got[6].clone()
    assert len(depths) >= B * 3
    assert any(d > 0 for d in depths), depths


def test_tree_round_7b_ctx4096():
    """The 7B bf16 shape, tree [4, 2, 2] (29 nodes) at context 4096, batch 1."""
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    shape = SHAPES["llama7b"]
    CTX = 4096
    par = [int(x) for x in tree_parents([4, 2, 2])]
    w = make_weights(shape, seed=4, device="cuda")
    dec = Decoder(shape, weights_to_numpy(w))
    model = spec.Model(shape, w, max_rows=64, max_batch=1, max_position=CTX + 64)
    del w
    torch.cuda.empty_cache()
    cap = CTX + 64
    kv = spec.KVCache(model, 1, cap)
    kc, vc = make_kv_context(shape, 1, CTX, seed=4000, device="cuda")
    kv.import_rows(0, 0, kc[:, 0].contiguous(), vc[:, 0].contiguous())
    cache = dec.new_cache(cap)
    cache.load(kc[:, 0].float().cpu().numpy(), vc[:, 0].float().cpu().numpy())
    del kc, vc
    kv.set_lengths([CTX])
    t0 = int(make_tokens(1, shape.vocab, seed=4, name="t0")[0])
    got = _tree_round_gpu(spec, model, kv, cuda_i32([t0]), par, shape)
    assert kv.get_lengths() == [CTX + int(got[3][0]) + 1]
    # this seeded round holds no near-tie: the whole round is compared
    assert _check_round(0, dec, cache, t0, par, got, 2e-2, 2e-2, shape)
