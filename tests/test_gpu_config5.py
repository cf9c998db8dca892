"""Adaptive-k layer-skip rounds at full size: the 7B-shaped model, batch 32,
committed contexts drawn uniformly from 512..8192 (seeded synthetic KV), each
sequence's k recomputed on the device every round from its confidence
(DSpark page, 0539edu.com/news/4524681, sections 2.2 and 2.3), in the launch
configuration bench.py --workload adaptive times.

Two rounds (all k = 2, then the scheduled k in [2, 16]).  Sampled sequences
(the two shortest contexts) go through the oracle: draft tokens, verify logits
within 2e-2, acceptance, next token, committed length.  For every sequence:
the committed length is s + a + 1 with a <= k, the next token is in range, and
the schedule's k, EMA and confidence equal the oracle's schedule evaluated on
the device's own per-row top-1 / top-2 probabilities (bit-exact inputs).
"""
import numpy as np
import pytest
import torch

from _gpu_util import assert_tokens_match, cuda_i32, lib, top_gap
from oracle import accept as A
from oracle import spec as OS
from oracle.decoder import Decoder
from synthetic import SHAPES, make_kv_context, make_ragged_contexts, make_tokens, make_weights, weights_to_numpy

pytestmark = pytest.mark.gpu

TOL = 2e-2
B = 32
SCH = A.KSchedule()


def test_adaptive_full_size():
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    shape = SHAPES["llama7b"]
    lens = [int(x) for x in make_ragged_contexts(B, 512, 8192, seed=5)]
    sampled = sorted(range(B), key=lambda b: lens[b])[:2]
    rounds = 2
    cap = max(lens) + rounds * (SCH.max_k + 1) + 8
    w = make_weights(shape, seed=4, device="cuda")
    dec = Decoder(shape, weights_to_numpy(w))
    model = spec.Model(shape, w, max_rows=B * (SCH.max_k + 1), max_batch=B, max_position=cap + 8)
    del w
    torch.cuda.empty_cache()
    kv = spec.KVCache(model, B, cap)
    caches = {}
    for b in range(B):
        kc, vc = make_kv_context(shape, 1, lens[b], seed=4000 + b, device="cuda")
        kv.import_rows(b, 0, kc[:, 0].contiguous(), vc[:, 0].contiguous())
        if b in sampled:
            c = dec.new_cache(cap)
            c.load(kc[:, 0].float().cpu().numpy(), vc[:, 0].float().cpu().numpy())
            caches[b] = c
        del kc, vc
    torch.cuda.empty_cache()
    kv.set_lengths(lens)

    t0 = make_tokens(B, shape.vocab, seed=4, name="t0")
    t0g = cuda_i32(t0)
    ema0 = np.full(B, 0.5)
    ema = torch.from_numpy(ema0.copy()).cuda()
    ema_host = list(ema0)
    k_cur = [SCH.k0] * B
    alive = {b: True for b in sampled}
    for rnd in range(rounds):
        kmax = max(k_cur)
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
        before = kv.get_lengths()
        spec.spec_draft(model, kv, t0g, kmax, cand, hL)
        spec.spec_verify(model, kv, n_rows, cand, kmax + 1, h_in=hL, h_stride=kmax + 1, logits=logits, stats=stats,
                         acc_len=acc, next_tok=nxt)
        spec.spec_row_probs(stats, probs)
        spec.spec_schedule_k(probs, n_rows, acc, ema, kn, conf)
        spec.kv_commit(kv, acc)
        torch.cuda.synchronize()
        assert model.device_error() == 0
        accg, nxtg, kng = acc.cpu().numpy(), nxt.cpu().numpy(), kn.cpu().numpy()
        pr, cg = probs.cpu().numpy(), cand.cpu().numpy()
        after = kv.get_lengths()
        r0 = 0
        for b in range(B):
            kb = k_cur[b]
            # every sequence: commit and range invariants, schedule on the device's own inputs
            assert 0 <= accg[b] <= kb and 0 <= nxtg[b] < shape.vocab
            assert after[b] == before[b] + accg[b] + 1
            rows = pr[r0:r0 + kb + 1]
            k_ref, ema_ref, c_ref = A.schedule_update(ema_host[b], int(accg[b]), kb, list(rows[:, 0]),
                                                      list(rows[:, 1]), SCH)
            assert (kng[b], conf[b].item()) == (k_ref, c_ref), (b, kng[b], k_ref, conf[b].item(), c_ref)
            assert ema[b].item() == ema_ref
            ema_host[b] = ema_ref
            if b in sampled and alive[b]:
                c = caches[b]
                s = c.length
                d_ref, hL_ref, dlog_ref, _ = OS.draft(dec, c, s, int(t0g[b].item()), kb)
                n_ok = assert_tokens_match(list(cg[b, 1:kb + 1]), d_ref, [top_gap(x) for x in dlog_ref], what="draft")
                if n_ok < kb:
                    alive[b] = False
                else:
                    vlog = OS.verify(dec, c, s, hL_ref, shape.exit_layer)
                    err = np.abs(logits[r0:r0 + kb + 1].cpu().numpy() - vlog).max()
                    assert err < TOL, (b, err)
                    a_ref, n_ref = A.accept_greedy_chain(d_ref, vlog)
                    if (accg[b], nxtg[b]) != (a_ref, n_ref):
                        assert min(top_gap(x) for x in vlog[:a_ref + 1]) < 1e-2
                        alive[b] = False
                    else:
                        c.length = A.commit_chain(s, a_ref)
                        assert after[b] == c.length
            r0 += kb + 1
        k_cur = [int(x) for x in kng]
        t0g = nxt.clone()
    assert all(SCH.min_k <= k <= SCH.max_k for k in k_cur)
    assert any(alive.values())
