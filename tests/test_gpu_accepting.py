"""Greedy chain rounds that accept drafts, on the GPU against the oracle.

Self-speculative decoding page (m.lqnn.cn/news/278124), §1.2 and §2.1: a
round verifies k drafted tokens at once, keeps the longest prefix the full
model agrees with and adds the full model's own next token, so an all-kept
round emits k + 1 tokens and the committed length grows by k + 1.

Random-init weights make a layer-skip draft almost never agree with the full
model, so two constructed models exercise acceptance:

* all-accept: in the layers past the exit layer L the attention output
  projection and the FFN down projection are zero, so those layers add exactly
  nothing to the residual stream.  The full model's logits are then the
  draft's, every draft token is the target's choice and every round keeps all
  k (on the GPU bit for bit: the draft's and the verifier's LM head read the
  same residual rows);
* partial-accept: the same two projections are scaled by 0.1, so the full
  model stays close to the draft and rounds keep anything from 0 to k.

Each round runs spec_draft -> spec_verify (greedy acceptance fused into the
LM head) -> kv_commit and is compared with the oracle: draft tokens, draft
and target logits, accepted count, next token, committed lengths, and at the
end every committed K/V row of every layer.  The seeds are chosen so that the
oracle's top-1/top-2 logit gap stays above 1e-3 (f32) or 2.5e-2 (bf16) at
every compared position, so no comparison is excused by a near-tie and every
round is compared.
"""
import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib
from oracle import spec as OS
from oracle.accept import accept_greedy_chain, argmax_lowest, commit_chain
from oracle.decoder import Decoder
from synthetic import ModelShape, make_tokens, make_weights, weights_to_numpy

pytestmark = pytest.mark.gpu

K, PROMPT = 4, 16
F32 = ModelShape(2, 256, 4, 4, 64, 1024, 1024, 1, "f32")
BF16 = ModelShape(3, 256, 4, 2, 64, 512, 512, 1, "bf16", init_std=0.2)
# name: (shape, seed, scale of the upper layers' O and down projections, rounds, logit tolerance)
CASES = {
    "f32_all": (F32, 2, 0.0, 10, 2e-3),
    "f32_partial": (F32, 1, 0.1, 10, 2e-3),
    "bf16_all": (BF16, 1, 0.0, 8, 2e-2),
    "bf16_partial": (BF16, 8, 0.1, 8, 2e-2),
}


def _weights(shape, seed, scale):
    w = make_weights(shape, seed, device="cuda")
    for layer in w["layers"][shape.exit_layer:]:
        for name in ("wo", "w_down"):
            layer[name] = (layer[name].float() * scale).to(layer[name].dtype)
    return w


@pytest.mark.parametrize("case", list(CASES))
def test_accepting_rounds_match_the_oracle(case):
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    shape, seed, scale, rounds, tol = CASES[case]
    w = _weights(shape, seed, scale)
    dec = Decoder(shape, weights_to_numpy(w))
    cap = PROMPT + rounds * (K + 1) + K + 8
    model = spec.Model(shape, w, max_rows=64, max_batch=1, max_position=cap + 8)
    del w
    kv = spec.KVCache(model, 1, cap)
    prompt = make_tokens(PROMPT, shape.vocab, seed=seed)
    t0 = torch.empty(1, dtype=torch.int32, device="cuda")
    spec.spec_prefill(model, kv, 0, cuda_i32(prompt), next_tok=t0)
    cache = dec.new_cache(cap)
    t_ref = argmax_lowest(dec.prefill(cache, prompt))
    assert int(t0.item()) == t_ref

    cand = torch.empty((1, K + 1), dtype=torch.int32, device="cuda")
    hL = torch.empty((1, K + 1, shape.d_model), dtype=torch.float32, device="cuda")
    dlog = torch.empty((1, K, shape.vocab), dtype=torch.float32, device="cuda")
    logits = torch.empty((K + 1, shape.vocab), dtype=torch.float32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    kept = []
    for rnd in range(rounds):
        s = cache.length
        d_ref, hL_ref, dlog_ref, _ = OS.draft(dec, cache, s, t_ref, K)
        vlog_ref = OS.verify(dec, cache, s, hL_ref, shape.exit_layer)
        a_ref, n_ref = accept_greedy_chain(d_ref, vlog_ref)
        cache.length = commit_chain(s, a_ref)

        spec.spec_draft(model, kv, t0, K, cand, hL, dlog)
        spec.spec_verify(model, kv, [K + 1], cand, K + 1, h_in=hL, h_stride=K + 1, logits=logits, acc_len=acc,
                         next_tok=nxt)
        spec.kv_commit(kv, acc)
        torch.cuda.synchronize()
        assert cand.cpu().tolist()[0] == [t_ref] + list(d_ref), f"round {rnd}: draft tokens"
        e_d = float(np.abs(dlog.cpu().numpy()[0] - dlog_ref).max())
        e_v = float(np.abs(logits.cpu().numpy() - vlog_ref).max())
        assert e_d < tol and e_v < tol, (rnd, e_d, e_v)
        assert (int(acc.item()), int(nxt.item())) == (a_ref, n_ref), f"round {rnd}: acceptance"
        assert kv.get_lengths() == [s + a_ref + 1] == [cache.length]
        if scale == 0.0:
            # the upper layers are identities: every draft is kept, k + 1 tokens a round
            assert a_ref == K and int(acc.item()) == K
            assert torch.equal(logits[:K], dlog[0]), "draft and target logits differ with identity upper layers"
        kept.append(a_ref)
        t_ref = n_ref
        t0 = nxt.clone()
    if scale > 0.0:
        assert sum(kept) > 0 and any(0 < a < K for a in kept), kept
    n = cache.length
    kk, vv = kv.export_rows(0, 0, shape.n_layers, 0, n)
    for layer in range(shape.n_layers):
        np.testing.assert_allclose(kk[layer].float().cpu().numpy(), cache.k[layer][:n], atol=tol, rtol=1e-2)
        np.testing.assert_allclose(vv[layer].float().cpu().numpy(), cache.v[layer][:n], atol=tol, rtol=1e-2)
    assert model.device_error() == 0
