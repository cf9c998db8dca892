"""bf16 models on the tcgen05 path against the float64 oracle.

* tree verification (8 layers, d 1024, 16 query / 4 KV heads x 64, FFN 2816,
  vocab 32000): prefill of a random prompt, a [4, 2, 2] token tree (28 nodes
  plus the root, level order, ancestor-only mask, depth position ids) with a
  planted greedy path, fused greedy longest-path acceptance, KV commit of the
  path; full size at a 2048-token context, and a 2-layer / 200-token case;
* layer-skip chain rounds on the 7B layer shape (d 4096, 32 heads x 128,
  FFN 11008, vocab 32000) with 4 layers and the draft = 2 layers, batch 2
  with different context lengths.

Logits within 2e-2 absolute; acceptance, next token, path and lengths exact
unless the oracle's top-1 / top-2 gap is below 1e-2.
"""
import numpy as np
import pytest
import torch

from _gpu_util import assert_tokens_match, cuda_i32, lib, model_pair, top_gap
from oracle import accept as A
from oracle import spec as OS
from oracle.accept import argmax_lowest
from synthetic import SHAPES, ModelShape, make_tokens, tree_parents

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _tree_case(n_layers, prompt_len, seed):
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    model, dec, shape = model_pair(SHAPES["tree8"], seed=seed, n_layers=n_layers, max_rows=64, max_batch=1,
                                   max_position=prompt_len + 64)
    prompt = make_tokens(prompt_len, shape.vocab, seed=seed)
    ctx = prompt_len + 40
    kv = spec.KVCache(model, 1, ctx)
    last = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    spec.spec_prefill(model, kv, 0, cuda_i32(prompt), last, None)
    cache = dec.new_cache(ctx)
    ref = dec.prefill(cache, prompt)
    torch.cuda.synchronize()
    np.testing.assert_allclose(last.cpu().numpy(), ref, atol=TOL, rtol=0)

    par = tree_parents([4, 2, 2])
    t0 = argmax_lowest(ref)
    greedy = OS.generate_greedy_ar(dec, prompt, 4)     # t0 and the next three greedy tokens
    assert greedy[0] == t0
    toks = make_tokens(29, shape.vocab, seed=seed + 1)
    toks[0] = t0
    toks[3] = greedy[1]          # node 3 (depth 1) -> child 10 (depth 2) -> child 23 (depth 3)
    toks[10] = greedy[2]
    toks[23] = greedy[3]
    s = cache.length
    d_ref, node_ref, path_ref, nxt_ref, logits_ref = OS.tree_round_greedy(dec, cache, toks, par)

    logits = torch.empty((29, shape.vocab), dtype=torch.float32, device="cuda")
    stats = torch.empty((29, 4), dtype=torch.float32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    path = torch.full((1, 64), -1, dtype=torch.int32, device="cuda")
    tk = cuda_i32(toks)
    spec.spec_verify(model, kv, [29], tk, 29, tree_parent=list(par), logits=logits, stats=stats, acc_len=acc,
                     next_tok=nxt, path=path)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    err = np.abs(lg - logits_ref).max()
    assert err < TOL, err
    am = spec.stats_argmax(stats).cpu().numpy()
    np.testing.assert_array_equal(am, lg.argmax(-1))
    gaps = [top_gap(r) for r in logits_ref]
    if min(gaps[i] for i in path_ref) >= 1e-2:
        assert (acc.item(), nxt.item()) == (d_ref, nxt_ref)
        assert list(path.cpu().numpy()[0, :d_ref + 1]) == path_ref
        assert d_ref == 3
    # unfused acceptance on the same logits agrees with the fused one
    acc2 = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt2 = torch.empty(1, dtype=torch.int32, device="cuda")
    path2 = torch.full((1, 64), -1, dtype=torch.int32, device="cuda")
    spec.spec_accept_greedy(logits.view(1, 29, -1), tk.view(1, 29), acc2, nxt2, tree_parent=list(par), path=path2)
    torch.cuda.synchronize()
    assert (acc2.item(), nxt2.item()) == (acc.item(), nxt.item())
    assert torch.equal(path2[:, :acc.item() + 1], path[:, :acc.item() + 1])

    spec.kv_commit(kv, acc, path)
    torch.cuda.synchronize()
    a = acc.item()
    assert kv.get_lengths() == [s + a + 1]
    if a == d_ref:
        kk, vv = kv.export_rows(0, 0, shape.n_layers, 0, s + a + 1)
        for l in range(shape.n_layers):
            np.testing.assert_allclose(kk[l].float().cpu().numpy(), cache.k[l][:s + a + 1], atol=TOL)
            np.testing.assert_allclose(vv[l].float().cpu().numpy(), cache.v[l][:s + a + 1], atol=TOL)
    assert model.device_error() == 0


def test_tree_small():
    _tree_case(2, 200, seed=31)


def test_tree_full_size():
    """8 layers, 2048-token prefilled context, 29-row tree."""
    _tree_case(8, 2048, seed=3)


def _layer_skip_rounds(n_layers, exit_layer, lens, k, rounds, seed):
    """Greedy layer-skip rounds on the 7B layer shape from a synthetic committed
    context (seeded KV rows given identically to both sides), lockstep with the oracle."""
    from speculative_decoding_verify_04_gb300 import spec
    from synthetic import make_kv_context
    import dataclasses
    lib()
    shape0 = dataclasses.replace(SHAPES["llama7b"], exit_layer=exit_layer)
    B = len(lens)
    model, dec, shape = model_pair(shape0, seed=seed, n_layers=n_layers, max_rows=64, max_batch=B,
                                   max_position=max(lens) + rounds * (k + 1) + 16, device="cpu")
    ctx = max(lens) + rounds * (k + 1) + 8
    kv = spec.KVCache(model, B, ctx)
    caches = []
    for b in range(B):
        kc, vc = make_kv_context(shape, 1, lens[b], seed * 100 + b, device="cpu")
        kv.import_rows(b, 0, kc[:, 0].contiguous().cuda(), vc[:, 0].contiguous().cuda())
        c = dec.new_cache(ctx)
        c.load(kc[:, 0].float().cpu().numpy(), vc[:, 0].float().cpu().numpy())
        caches.append(c)
        del kc, vc
    kv.set_lengths(lens)
    t0 = make_tokens(B, shape.vocab, seed=seed, name="t0")
    t0g = cuda_i32(t0)
    cand = torch.empty((B, k + 1), dtype=torch.int32, device="cuda")
    hL = torch.empty((B, k + 1, shape.d_model), dtype=torch.float32, device="cuda")
    dlog = torch.empty((B, k, shape.vocab), dtype=torch.float32, device="cuda")
    logits = torch.empty((B * (k + 1), shape.vocab), dtype=torch.float32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    worst = 0.0
    for rnd in range(rounds):
        spec.spec_draft(model, kv, t0g, k, cand, hL, dlog)
        spec.spec_verify(model, kv, [k + 1] * B, cand, k + 1, h_in=hL, h_stride=k + 1, logits=logits,
                         acc_len=acc, next_tok=nxt)
        spec.kv_commit(kv, acc)
        torch.cuda.synchronize()
        cg = cand.cpu().numpy()
        for b in range(B):
            c = caches[b]
            s = c.length
            d_ref, hL_ref, dlog_ref, _ = OS.draft(dec, c, s, int(t0g[b].item()), k)
            n_ok = assert_tokens_match(list(cg[b, 1:]), d_ref, [top_gap(r) for r in dlog_ref], what="draft")
            if n_ok < k:
                return worst, rnd
            e1 = np.abs(dlog.cpu().numpy()[b] - dlog_ref).max()
            vlog_ref = OS.verify(dec, c, s, hL_ref, shape.exit_layer)
            e2 = np.abs(logits.cpu().numpy()[b * (k + 1):(b + 1) * (k + 1)] - vlog_ref).max()
            worst = max(worst, e1, e2)
            assert e1 < TOL and e2 < TOL, (e1, e2)
            a_ref, n_ref = A.accept_greedy_chain(d_ref, vlog_ref)
            if (acc[b].item(), nxt[b].item()) != (a_ref, n_ref):
                assert min(top_gap(r) for r in vlog_ref[:a_ref + 1]) < 1e-2
                return worst, rnd
            c.length = A.commit_chain(s, a_ref)
        assert kv.get_lengths() == [c.length for c in caches]
        t0g = nxt.clone()
    for b in range(B):
        n = caches[b].length
        kk, vv = kv.export_rows(b, 0, shape.n_layers, 0, n)
        for l in range(shape.n_layers):
            np.testing.assert_allclose(kk[l].float().cpu().numpy(), caches[b].k[l][:n], atol=TOL, rtol=1e-2)
            np.testing.assert_allclose(vv[l].float().cpu().numpy(), caches[b].v[l][:n], atol=TOL, rtol=1e-2)
    assert model.device_error() == 0
    return worst, rounds


def test_layer_skip_rounds_7b_layer_shape():
    """4 layers of the 7B shape, draft = 2 layers, batch 2 with contexts 150 and 301.
    Weights and contexts are drawn on the CPU; for these values the oracle's
    top-1/top-2 logit gap at every compared position of the three rounds is at
    least 0.0144, so no near-tie may end the comparison: all three rounds count."""
    worst, compared = _layer_skip_rounds(4, 2, [150, 301], k=4, rounds=3, seed=9)
    print(f"max logit error {worst:.3g}")
    assert compared == 3, f"compared {compared} of 3 rounds"


@pytest.mark.parametrize("which", ["7b_layers", "tree8_layers"])
def test_tile_major_weights_are_bit_identical(which, monkeypatch):
    """The bf16 GEMM weights are stored tile-major (each 128-row x 64-column
    block as 16 contiguous, pre-swizzled KB, fetched with one bulk copy) unless
    SPEC_TILED_W=0 keeps them row-major (fetched as 2-D tensor boxes).  Both put
    the same bytes in shared memory, so a draft and a verification give the
    same tokens and logits bit for bit: on 3 layers of the 7B layer shape (GEMM
    chains) and on 3 layers of the d-1024 model (GEMMs launched one by one)."""
    from speculative_decoding_verify_04_gb300 import spec
    from synthetic import make_kv_context, make_weights
    from _gpu_util import to_cuda
    import dataclasses
    lib()
    if which == "7b_layers":
        shape = ModelShape(3, 4096, 32, 32, 128, 11008, 512, 1, "bf16")
    else:
        shape = dataclasses.replace(SHAPES["tree8"], n_layers=3, exit_layer=1)
    w = make_weights(shape, 11, device="cpu")
    kc, vc = make_kv_context(shape, 1, 300, 1100, device="cpu")
    k = 4
    outs = []
    for tiled in ("0", "1"):
        monkeypatch.setenv("SPEC_TILED_W", tiled)
        model = spec.Model(shape, to_cuda(w), max_rows=64, max_batch=1, max_position=400)
        kv = spec.KVCache(model, 1, 320)
        kv.import_rows(0, 0, kc[:, 0].contiguous().cuda(), vc[:, 0].contiguous().cuda())
        kv.set_lengths([300])
        cand = torch.empty((1, k + 1), dtype=torch.int32, device="cuda")
        hL = torch.empty((1, k + 1, shape.d_model), dtype=torch.float32, device="cuda")
        dlog = torch.empty((1, k, shape.vocab), dtype=torch.float32, device="cuda")
        logits = torch.empty((k + 1, shape.vocab), dtype=torch.float32, device="cuda")
        spec.spec_draft(model, kv, cuda_i32([7]), k, cand, hL, dlog)
        spec.spec_verify(model, kv, [k + 1], cand, k + 1, h_in=hL, h_stride=k + 1, logits=logits)
        torch.cuda.synchronize()
        assert model.device_error() == 0
        outs.append((cand.cpu(), dlog.cpu(), logits.cpu()))
        del kv, model
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
