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
* partial-accept: the same two projections are scaled down (by 0.1 in the
  f32 model, by 0.2 in the bf16 one), so the full model stays close to the
  draft and rounds keep anything from 0 to k.

Each round runs spec_draft -> spec_verify (greedy acceptance fused into the
LM head) -> kv_commit and is compared with the oracle: draft tokens, draft
and target logits, accepted count, next token, committed lengths, and at the
end every committed K/V row of every layer.  The bf16 model has the 7B layer
shape (d 4096, 32 heads x 128, FFN 11008) with a 512-token vocabulary, so its
logits have the benchmark's scale and the 2e-2 tolerance applies as stated.
Its rounds start from a seeded committed context of 64 slots given to both
sides (as the 7B-shaped tests do).  Weights are drawn on the CPU, and the
seeds are chosen so that the oracle's top-1/top-2 logit gap stays at or above
3e-2 at every compared position (1e-3 for the f32 model, whose logits are
exact to ~1e-6): no comparison is excused by a near-tie, so every round is
compared.
"""
import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, to_cuda
from oracle import spec as OS
from oracle.accept import accept_greedy_chain, argmax_lowest, commit_chain
from oracle.decoder import Decoder
from synthetic import ModelShape, make_kv_context, make_tokens, make_weights, weights_to_numpy

pytestmark = pytest.mark.gpu

K, PROMPT, CTX = 4, 16, 64      # f32 models: a prefilled prompt; bf16: a synthetic context of CTX slots
F32 = ModelShape(2, 256, 4, 4, 64, 1024, 1024, 1, "f32")
BF16 = ModelShape(3, 4096, 32, 32, 128, 11008, 512, 1, "bf16")
# name: (shape, seed, scale of the upper layers' O and down projections, rounds, logit tolerance)
CASES = {
    "f32_all": (F32, 2, 0.0, 10, 2e-3),
    "f32_partial": (F32, 1, 0.1, 10, 2e-3),
    "bf16_all": (BF16, 4, 0.0, 6, 2e-2),
    "bf16_partial": (BF16, 4, 0.2, 6, 2e-2),
}


def _weights(shape, seed, scale):
    # drawn on the CPU (the seeds were chosen by running the oracle on these values)
    w = make_weights(shape, seed, device="cpu")
    for layer in w["layers"][shape.exit_layer:]:
        for name in ("wo", "w_down"):
            layer[name] = (layer[name].float() * scale).to(layer[name].dtype)
    return to_cuda(w)


@pytest.mark.parametrize("case", list(CASES))
def test_accepting_rounds_match_the_oracle(case):
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    shape, seed, scale, rounds, tol = CASES[case]
    w = _weights(shape, seed, scale)
    dec = Decoder(shape, weights_to_numpy(w))
    cap = max(PROMPT, CTX) + rounds * (K + 1) + K + 8
    model = spec.Model(shape, w, max_rows=64, max_batch=1, max_position=cap + 8)
    del w
    kv = spec.KVCache(model, 1, cap)
    cache = dec.new_cache(cap)
    if shape.dtype == "bf16":
        # a seeded committed context given to both sides (bf16 values, exact in both), as in
        # the 7B-shaped tests: only the rounds' own rows carry the cache's bf16 rounding
        kc, vc = make_kv_context(shape, 1, CTX, seed * 100, device="cpu")
        kv.import_rows(0, 0, kc[:, 0].contiguous().cuda(), vc[:, 0].contiguous().cuda())
        kv.set_lengths([CTX])
        cache.load(kc[:, 0].float().numpy(), vc[:, 0].float().numpy())
        t_ref = int(make_tokens(1, shape.vocab, seed, "t0")[0])
        t0 = cuda_i32([t_ref])
    else:
        prompt = make_tokens(PROMPT, shape.vocab, seed=seed)
        t0 = torch.empty(1, dtype=torch.int32, device="cuda")
        spec.spec_prefill(model, kv, 0, cuda_i32(prompt), next_tok=t0)
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
    # committed K/V rows: bf16 storage rounds an element to 2^-9 of its own size and
    # the rotation mixes pairs of elements, so the bound scales with the row's largest
    # element (2e-2 plus 1e-2 of it), not with the element itself
    n = cache.length
    kk, vv = kv.export_rows(0, 0, shape.n_layers, 0, n)
    for layer in range(shape.n_layers):
        for got, ref in ((kk[layer], cache.k[layer][:n]), (vv[layer], cache.v[layer][:n])):
            g = got.float().cpu().numpy()
            bound = tol + 1e-2 * np.abs(ref).max(axis=-1, keepdims=True)
            assert (np.abs(g - ref) <= bound).all(), (layer, float(np.abs(g - ref).max()))
    assert model.device_error() == 0
