"""Full-size 7B-shaped rounds against the oracle (the benchmark's configuration).

32 layers, d 4096, 32 heads x 128, FFN 11008, vocab 32000, bf16 random-init
weights (13.5 GB), draft = first 12 layers + LM head, verify = layers 12..31
on the draft's KV, chain k = 4, committed context 4096 (seeded synthetic KV,
identical on both sides), batch 1, greedy; the same launch configuration as
bench.py.  Three rounds in lockstep: draft tokens, the 4 draft rows and 5
target rows of logits (within 2e-2), acceptance and next token, the committed
length, and sampled KV rows of the new slots in the first, last-draft,
first-verify and last layers.  Weights and context are drawn on the CPU (the
CPU and GPU generators differ for one seed): for these values the oracle's
top-1/top-2 logit gap at every compared position of the three rounds is at
least 0.0119, above the 1e-2 that would excuse a different greedy choice, so
all three rounds must be compared.
"""
import numpy as np
import pytest
import torch

from _gpu_util import assert_tokens_match, cuda_i32, lib, to_cuda, top_gap
from oracle import accept as A
from oracle import spec as OS
from oracle.decoder import Decoder
from synthetic import SHAPES, make_kv_context, make_tokens, make_weights, weights_to_numpy

pytestmark = pytest.mark.gpu

TOL = 2e-2
K, CTX, ROUNDS = 4, 4096, 3


def test_full_size_rounds():
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    shape = SHAPES["llama7b"]
    w = make_weights(shape, seed=4, device="cpu")
    dec = Decoder(shape, weights_to_numpy(w))
    model = spec.Model(shape, to_cuda(w), max_rows=64, max_batch=1, max_position=CTX + 64)
    del w
    torch.cuda.empty_cache()
    cap = CTX + 32
    kv = spec.KVCache(model, 1, cap)
    kc, vc = make_kv_context(shape, 1, CTX, seed=4000, device="cpu")
    kv.import_rows(0, 0, kc[:, 0].contiguous().cuda(), vc[:, 0].contiguous().cuda())
    cache = dec.new_cache(cap)
    cache.load(kc[:, 0].float().numpy(), vc[:, 0].float().numpy())
    del kc, vc
    kv.set_lengths([CTX])
    t0 = int(make_tokens(1, shape.vocab, seed=4, name="t0")[0])

    cand = torch.empty((1, K + 1), dtype=torch.int32, device="cuda")
    hL = torch.empty((1, K + 1, shape.d_model), dtype=torch.float32, device="cuda")
    dlog = torch.empty((1, K, shape.vocab), dtype=torch.float32, device="cuda")
    logits = torch.empty((K + 1, shape.vocab), dtype=torch.float32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    compared = 0
    for rnd in range(ROUNDS):
        s = cache.length
        spec.spec_draft(model, kv, cuda_i32([t0]), K, cand, hL, dlog)
        spec.spec_verify(model, kv, [K + 1], cand, K + 1, h_in=hL, h_stride=K + 1, logits=logits, acc_len=acc,
                         next_tok=nxt)
        spec.kv_commit(kv, acc)
        torch.cuda.synchronize()

        d_ref, hL_ref, dlog_ref, _ = OS.draft(dec, cache, s, t0, K)
        n_ok = assert_tokens_match(list(cand.cpu().numpy()[0, 1:]), d_ref, [top_gap(r) for r in dlog_ref],
                                   what="draft")
        e_draft = np.abs(dlog.cpu().numpy()[0, :max(n_ok, 1)] - dlog_ref[:max(n_ok, 1)]).max()
        assert e_draft < TOL, (rnd, e_draft)
        if n_ok < K:
            break       # near-tie inside the draft: the rest of the round follows different tokens
        h_err = np.abs(hL.cpu().numpy()[0] - hL_ref).max() / np.abs(hL_ref).max()
        vlog = OS.verify(dec, cache, s, hL_ref, shape.exit_layer)
        e_verify = np.abs(logits.cpu().numpy() - vlog).max()
        print(f"round {rnd}: layer-{shape.exit_layer} state relative error {h_err:.3g}, draft logit error "
              f"{e_draft:.3g}, verify logit error {e_verify:.3g}")
        assert e_verify < TOL, (rnd, e_verify)
        a_ref, n_ref = A.accept_greedy_chain(d_ref, vlog)
        if (acc.item(), nxt.item()) != (a_ref, n_ref):
            assert min(top_gap(r) for r in vlog[:a_ref + 1]) < 1e-2
            break
        cache.length = A.commit_chain(s, a_ref)
        assert kv.get_lengths() == [cache.length]
        for layer in (0, shape.exit_layer - 1, shape.exit_layer, shape.n_layers - 1):
            kk, vv = kv.export_rows(0, layer, 1, s, a_ref + 1)
            np.testing.assert_allclose(kk[0].float().cpu().numpy(), cache.k[layer][s:s + a_ref + 1],
                                       atol=TOL, rtol=1e-2)
            np.testing.assert_allclose(vv[0].float().cpu().numpy(), cache.v[layer][s:s + a_ref + 1],
                                       atol=TOL, rtol=1e-2)
        compared += 1
        t0 = n_ref
    assert model.device_error() == 0
    assert compared == ROUNDS, f"compared {compared} of {ROUNDS} rounds"
