"""Exit layer following the context length on the GPU against the oracle
(self-speculative decoding page, m.lqnn.cn/news/278124, section 5.3).

spec_set_exit_layer moves L from 1 to 2 to 3 as the committed context of a
4-layer f32 model grows (the table of the oracle's
generate_greedy_spec_context_exit); 48 greedy tokens equal the oracle's and
every layer of every committed KV row matches it, so each round wrote all
the layers of its rows whatever L the next round drafts with.
"""
import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, model_pair
from oracle import spec as OS
from oracle.accept import argmax_lowest
from synthetic import ModelShape, make_tokens

pytestmark = pytest.mark.gpu

SMALL = ModelShape(4, 256, 4, 2, 64, 512, 512, 2, "f32", init_std=0.1)
TABLE = [(0, 1), (24, 2), (36, 3)]


def test_context_exit_layer_rounds_match_the_oracle():
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    model, dec, shape = model_pair(SMALL, seed=8, max_rows=64, max_batch=1, max_position=512)
    pr = make_tokens(16, shape.vocab, seed=8)
    n_new, k = 48, 3
    want, cache_o = OS.generate_greedy_spec_context_exit(dec, pr, n_new, k, TABLE)
    kv = spec.KVCache(model, 1, 256)
    t0 = torch.empty(1, dtype=torch.int32, device="cuda")
    spec.spec_prefill(model, kv, 0, cuda_i32(pr), next_tok=t0)
    cand = torch.empty((1, k + 1), dtype=torch.int32, device="cuda")
    hL = torch.empty((1, k + 1, shape.d_model), dtype=torch.float32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    out, seen = [int(t0.item())], set()
    while len(out) < n_new:
        s = kv.get_lengths()[0]
        L = OS.exit_layer_for_context(s, TABLE)
        seen.add(L)
        model.set_exit_layer(L)
        spec.spec_draft(model, kv, t0, k, cand, hL)
        spec.spec_verify(model, kv, [k + 1], cand, k + 1, h_in=hL, h_stride=k + 1, acc_len=acc, next_tok=nxt)
        spec.kv_commit(kv, acc)
        a = int(acc.item())
        out += cand[0, 1:1 + a].tolist() + [int(nxt.item())]
        t0 = nxt.clone()
    torch.cuda.synchronize()
    assert model.device_error() == 0
    assert seen == {1, 2, 3}
    assert out[:n_new] == want
    n = min(kv.get_lengths()[0], cache_o.length)
    for layer in range(shape.n_layers):
        kk, vv = kv.export_rows(0, layer, 1, 0, n)
        np.testing.assert_allclose(kk[0].cpu().numpy(), cache_o.k[layer][:n], atol=2e-3, rtol=0)
        np.testing.assert_allclose(vv[0].cpu().numpy(), cache_o.v[layer][:n], atol=2e-3, rtol=0)
