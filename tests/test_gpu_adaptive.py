"""Confidence-scheduled draft length over a ragged batch, against the oracle.

32 sequences with committed contexts drawn uniformly from 64..600 (seeded
synthetic KV), greedy layer-skip rounds where each sequence's draft length k
is recomputed every round on the device from its own confidence (DSpark page,
0539edu.com/news/4524681, sections 2.2 and 2.3): EMA of the acceptance rate
(decay 0.9), mean top-1 probability and top-1 / top-2 gap over the verified
rows, linear map between the 0.3 / 0.8 thresholds onto [2, 16].  Per round the
batch verifies sum(k_b + 1) rows (up to 544: several GEMM row passes).

A mid-width model (d 512, 8 heads x 64, FFN 1408, vocab 4096, 4 layers, draft
= 2 layers) keeps the float64 oracle fast; the LM head is scaled by 8 (exact
in bf16) so the target is confident and the schedule spreads k.
"""
import numpy as np
import pytest
import torch

from _gpu_util import assert_tokens_match, cuda_i32, lib, top_gap
from oracle import accept as A
from oracle import spec as OS
from oracle.decoder import Decoder
from synthetic import (ModelShape, make_kv_context, make_ragged_contexts, make_tokens, make_uniforms,
                       make_weights, weights_to_numpy)

pytestmark = pytest.mark.gpu

TOL = 2e-2
HEAD_SCALE = 8
SCH = A.KSchedule()


def test_adaptive_k_ragged_batch():
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    shape = ModelShape(4, 512, 8, 8, 64, 1408, 4096, 2, "bf16")
    w = make_weights(shape, seed=50, device="cuda")
    w["lm_head"].mul_(HEAD_SCALE)
    dec = Decoder(shape, weights_to_numpy(w))
    B, rounds = 32, 3
    lens = make_ragged_contexts(B, 64, 600, seed=50)
    cap = int(lens.max()) + rounds * (SCH.max_k + 1) + 8
    max_rows = B * (SCH.max_k + 1)
    model = spec.Model(shape, w, max_rows=max_rows, max_batch=B, max_position=cap + 8)
    kv = spec.KVCache(model, B, cap)
    caches = []
    for b in range(B):
        kc, vc = make_kv_context(shape, 1, int(lens[b]), seed=5000 + b, device="cuda")
        kv.import_rows(b, 0, kc[:, 0].contiguous(), vc[:, 0].contiguous())
        c = dec.new_cache(cap)
        c.load(kc[:, 0].float().cpu().numpy(), vc[:, 0].float().cpu().numpy())
        caches.append(c)
    kv.set_lengths([int(x) for x in lens])

    t0 = make_tokens(B, shape.vocab, seed=51, name="t0")
    ema0 = make_uniforms(B, seed=52, name="ema").astype(np.float64)
    k_cur = [SCH.k0] * B
    ema_g = torch.from_numpy(ema0.copy()).cuda()
    ema_o = list(ema0)
    alive = [True] * B            # a sequence stops being compared after an allowed divergence
    t0g = cuda_i32(t0)
    kmax_seen = 0
    for rnd in range(rounds):
        kmax = max(k_cur)
        kmax_seen = max(kmax_seen, kmax)
        n_rows = [k + 1 for k in k_cur]
        T = sum(n_rows)
        cand = torch.empty((B, kmax + 1), dtype=torch.int32, device="cuda")
        hL = torch.empty((B, kmax + 1, shape.d_model), dtype=torch.float32, device="cuda")
        logits = torch.empty((T, shape.vocab), dtype=torch.float32, device="cuda")
        stats = torch.empty((T, 4), dtype=torch.float32, device="cuda")
        probs = torch.empty((T, 2), dtype=torch.float64, device="cuda")
        acc = torch.empty(B, dtype=torch.int32, device="cuda")
        nxt = torch.empty(B, dtype=torch.int32, device="cuda")
        kn = torch.empty(B, dtype=torch.int32, device="cuda")
        conf = torch.empty(B, dtype=torch.float64, device="cuda")
        spec.spec_draft(model, kv, t0g, kmax, cand, hL)
        spec.spec_verify(model, kv, n_rows, cand, kmax + 1, h_in=hL, h_stride=kmax + 1, logits=logits, stats=stats,
                         acc_len=acc, next_tok=nxt)
        spec.spec_row_probs(stats, probs)
        spec.spec_schedule_k(probs, n_rows, acc, ema_g, kn, conf)
        spec.kv_commit(kv, acc)
        torch.cuda.synchronize()
        cg, lg = cand.cpu().numpy(), logits.cpu().numpy()
        accg, nxtg, kng = acc.cpu().numpy(), nxt.cpu().numpy(), kn.cpu().numpy()
        r0 = 0
        for b in range(B):
            kb = k_cur[b]
            if alive[b]:
                c = caches[b]
                s = c.length
                d_ref, hL_ref, dlog_ref, _ = OS.draft(dec, c, s, int(t0g[b].item()), kb)
                n_ok = assert_tokens_match(list(cg[b, 1:kb + 1]), d_ref, [top_gap(r) for r in dlog_ref],
                                           tol_gap=1e-2 * HEAD_SCALE)
                if n_ok < kb:
                    alive[b] = False
                else:
                    vlog = OS.verify(dec, c, s, hL_ref, shape.exit_layer)
                    err = np.abs(lg[r0:r0 + kb + 1] - vlog).max()
                    assert err < TOL * HEAD_SCALE, (b, err)     # logits (and their errors) scale with the head
                    a_ref, n_ref = A.accept_greedy_chain(d_ref, vlog)
                    if (accg[b], nxtg[b]) != (a_ref, n_ref):
                        assert min(top_gap(r) for r in vlog[:a_ref + 1]) < 1e-2 * HEAD_SCALE
                        alive[b] = False
                    else:
                        c.length = A.commit_chain(s, a_ref)
                        t12 = [A.top12_probs(r) for r in vlog]
                        k_ref, ema_ref, c_ref = A.schedule_update(ema_o[b], a_ref, kb, [x[0] for x in t12],
                                                                  [x[1] for x in t12], SCH)
                        # the confidence follows the logits (error up to TOL * HEAD_SCALE): near a step of
                        # the k map the two sides may pick neighbouring k, after which they part ways
                        assert abs(conf[b].item() - c_ref) < 2e-2, (b, conf[b].item(), c_ref)
                        assert kng[b] == A.next_k(conf[b].item(), SCH)      # the device applied its own conf
                        if kng[b] != k_ref:
                            assert abs(int(kng[b]) - k_ref) <= 1, (b, kng[b], k_ref)
                            alive[b] = False
                        ema_o[b] = ema_ref
                        assert abs(ema_g[b].item() - ema_ref) < 1e-12
            r0 += kb + 1
        k_cur = [int(x) for x in kng]
        t0g = nxt.clone()
    assert sum(alive) >= B // 2
    assert len(set(k_cur)) > 1 or kmax_seen > SCH.min_k      # the schedule actually moved k
    assert model.device_error() == 0
