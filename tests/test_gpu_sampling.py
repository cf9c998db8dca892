"""Sampling mode on the GPU against the oracle.

* spec_probs: softmax(logits / T) in f32 within 1e-5 relative of the oracle's
  float64 softmax; the top-p nucleus is bit-exact (the oracle's integer rule
  applied to the very f32 row the kernel cut) and its renormalised values
  within 1e-5 relative.
* spec_sample: the integer inverse-CDF draw, bit-exact against the oracle on
  the same rows and uniforms (ends of the unit interval included).
* Sampling rounds end to end (draft sampled at temperature T, target cut to
  its top-p nucleus at the same T, rejection sampling, KV commit) on the f32
  2-layer model and on the 7B bf16 shape at context 4096: every draft draw
  and every acceptance decision bit-exact given the q and p rows the GPU
  produced, q and p within tolerance of the oracle's rows from the same
  logits, logits within tolerance of the oracle's forward, the committed
  lengths, and the oracle's own draws equal to the GPU's except where the
  uniform falls within the two distributions' difference of a CDF step
  (self-speculative decoding page, m.lqnn.cn/news/278124, sections 2.4, 3.4
  and 4.3).
"""
import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, model_pair
from oracle import accept as A
from oracle import spec as OS
from oracle.decoder import Decoder
from synthetic import SHAPES, make_kv_context, make_tokens, make_uniforms, make_weights, weights_to_numpy

pytestmark = pytest.mark.gpu

P_RTOL = 1e-5
TOP_P = 15099494 * 2.0 ** -24          # 0.9 rounded down to a multiple of 2^-24


def _spec():
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    return spec


def _logit_rows(rows, V, seed, sigma):
    rng = np.random.default_rng(seed)
    z = (rng.standard_normal((rows, V)) * sigma).astype(np.float32)
    z[1 % rows, : V // 2] = z[1 % rows, 0]                 # a long run of ties
    z[2 % rows] = np.round(z[2 % rows])                    # many small tie groups
    return z


def _gpu_probs(spec, lg, T, top_p):
    g = torch.from_numpy(lg).cuda()
    out = torch.empty_like(g)
    spec.spec_probs(g, out, T, top_p)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("V,T,sigma", [(5, 1.0, 1.0), (1000, 0.7, 3.0), (32000, 1.0, 3.0), (32000, 0.3, 1.0),
                                       (4097, 1.7, 2.0), (53248, 1.0, 2.0)])
def test_probs_and_nucleus(V, T, sigma):
    spec = _spec()
    lg = _logit_rows(6, V, seed=V + int(10 * T), sigma=sigma)
    full = _gpu_probs(spec, lg, T, 1.0)
    ref = A.probs_at(lg, T)
    np.testing.assert_allclose(full, ref, rtol=P_RTOL, atol=1e-30)
    assert (np.abs(full.astype(np.float64).sum(axis=1) - 1.0) < 1e-5).all()
    for top_p in (TOP_P, 0.5, 2.0 ** -24, 1.0 - 2.0 ** -24):
        cut = _gpu_probs(spec, lg, T, top_p)
        for r in range(lg.shape[0]):
            keep = A.top_p_keep(full[r], top_p)
            np.testing.assert_array_equal(cut[r] != 0, keep, err_msg=f"row {r} top_p {top_p}")
            np.testing.assert_allclose(cut[r], A.top_p_filter(full[r], top_p), rtol=P_RTOL, atol=0)


def test_nucleus_ties_at_the_cut():
    """Eight equal tokens on top: top_p = 3/8 keeps exactly the three lowest ids."""
    spec = _spec()
    V = 1000
    lg = np.full((1, V), -30.0, dtype=np.float32)
    lg[0, [900, 17, 400, 5, 63, 700, 301, 999]] = 0.0
    full = _gpu_probs(spec, lg, 1.0, 1.0)
    for m in (3, 5):
        cut = _gpu_probs(spec, lg, 1.0, m / 8)
        keep = A.top_p_keep(full[0], m / 8)
        np.testing.assert_array_equal(cut[0] != 0, keep)
    assert list(np.nonzero(_gpu_probs(spec, lg, 1.0, 3 / 8)[0])[0]) == [5, 17, 63]


@pytest.mark.parametrize("V", [1, 7, 32, 1000, 32000, 53248])
def test_sample_bit_exact(V):
    spec = _spec()
    rows = 40
    lg = _logit_rows(rows, V, seed=7 + V, sigma=2.0)
    p = A.probs_at(lg, 1.0)
    p[3 % rows] = 0.0
    p[3 % rows, V - 1] = 1.0                               # one-hot on the last token
    p[4 % rows, : V // 2] = 0.0                            # zeros ahead of the mass
    u = make_uniforms(rows, seed=V, name="sample")
    u[0], u[1 % rows] = 0.0, np.float32(1.0 - 2.0 ** -24)  # both ends of [0, 1)
    pg = torch.from_numpy(p).cuda()
    tok = torch.empty(rows, dtype=torch.int32, device="cuda")
    spec.spec_sample(pg, torch.from_numpy(u).cuda(), tok)
    torch.cuda.synchronize()
    want = [A.sample_index(A.int_weights(p[r]), u[r]) if A.int_weights(p[r]).sum() > 0 else -1 for r in range(rows)]
    np.testing.assert_array_equal(tok.cpu().numpy(), want)


def test_probs_rejects_bad_arguments():
    spec = _spec()
    g = torch.zeros((2, 64), device="cuda")
    with pytest.raises(spec.SpecError):
        spec.spec_probs(g, torch.empty_like(g), 0.0)
    with pytest.raises(spec.SpecError):
        spec.spec_probs(g, torch.empty_like(g), 1.0, top_p=0.1)          # not a multiple of 2^-24
    with pytest.raises(spec.SpecError):
        big = torch.zeros((1, 53249), device="cuda")
        spec.spec_probs(big, torch.empty_like(big), 1.0)


def _near_cdf_step(q_ref, q_gpu, u, tok):
    """True when ``u`` lies within the two rows' L1 distance of the oracle's CDF
    interval of ``tok`` (the draws may then differ without an error)."""
    q_ref = np.asarray(q_ref, np.float64)
    c = np.concatenate([[0.0], np.cumsum(q_ref)]) / q_ref.sum()
    delta = np.abs(q_ref - np.asarray(q_gpu, np.float64)).sum() + 2.0 ** -20
    return c[tok] - delta <= float(u) <= c[tok + 1] + delta


def _sampling_rounds(spec, model, dec, shape, kv, caches, t0, k, T, top_p, rounds, seed, tol, check_full):
    """Run ``rounds`` sampling rounds on the GPU; returns the compared-round count.

    ``caches`` maps a sequence index to its oracle cache (the sequences the
    oracle follows); every sequence gets the bit-exact decision checks."""
    B = t0.numel()
    V = shape.vocab
    alive = {b: True for b in caches}
    compared = 0
    for rnd in range(rounds):
        u_d = make_uniforms((B, k), seed=seed + rnd, name="u_draft")
        u = make_uniforms((B, k + 1), seed=seed + rnd, name="u_accept")
        cand = torch.empty((B, k + 1), dtype=torch.int32, device="cuda")
        hL = torch.empty((B, k + 1, shape.d_model), dtype=torch.float32, device="cuda")
        q = torch.empty((B, k, V), dtype=torch.float32, device="cuda")
        dlog = torch.empty((B, k, V), dtype=torch.float32, device="cuda")
        logits = torch.empty((B * (k + 1), V), dtype=torch.float32, device="cuda")
        p = torch.empty_like(logits)
        acc = torch.empty(B, dtype=torch.int32, device="cuda")
        nxt = torch.empty(B, dtype=torch.int32, device="cuda")
        before = kv.get_lengths()
        spec.spec_draft_sample(model, kv, t0, k, T, torch.from_numpy(u_d).cuda(), cand, hL, q, dlog)
        spec.spec_verify(model, kv, [k + 1] * B, cand, k + 1, h_in=hL, h_stride=k + 1, logits=logits)
        spec.spec_probs(logits, p, T, top_p)
        spec.spec_accept(p.view(B, k + 1, V), q, cand[:, 1:], torch.from_numpy(u).cuda(), acc, nxt)
        spec.kv_commit(kv, acc)
        torch.cuda.synchronize()
        assert model.device_error() == 0
        p_full = None
        if check_full:
            pf = torch.empty_like(logits)
            spec.spec_probs(logits, pf, T, 1.0)
            p_full = pf.cpu().numpy().reshape(B, k + 1, V)
        cg, qg, dg = cand.cpu().numpy(), q.cpu().numpy(), dlog.cpu().numpy()
        pg, lg = p.cpu().numpy().reshape(B, k + 1, V), logits.cpu().numpy().reshape(B, k + 1, V)
        ag, ng = acc.cpu().numpy(), nxt.cpu().numpy()
        after = kv.get_lengths()
        for b in range(B):
            # the GPU's own rows decide bit-exactly
            for j in range(k):
                assert cg[b, j + 1] == A.sample_index(A.int_weights(qg[b, j]), u_d[b, j]), (rnd, b, j)
            np.testing.assert_allclose(qg[b], A.probs_at(dg[b], T), rtol=P_RTOL, atol=1e-30)
            a_ref, n_ref = A.accept_sampling_chain(pg[b], qg[b], cg[b, 1:], u[b])
            assert (ag[b], ng[b]) == (a_ref, n_ref), (rnd, b)
            assert after[b] == before[b] + a_ref + 1
            if p_full is not None:
                for j in range(k + 1):
                    np.testing.assert_array_equal(pg[b, j] != 0, A.top_p_keep(p_full[b, j], top_p))
                    np.testing.assert_allclose(pg[b, j], A.top_p_filter(p_full[b, j], top_p), rtol=P_RTOL, atol=0)
            # the oracle's own round on the sequences it follows
            if b not in caches or not alive[b]:
                continue
            c = caches[b]
            s = c.length
            d_ref, hL_ref, dlog_ref, q_ref = OS.draft(dec, c, s, int(cg[b, 0]), k, temp=T, u_draft=u_d[b])
            n_ok = k
            for j in range(k):
                if d_ref[j] != cg[b, j + 1]:
                    assert _near_cdf_step(q_ref[j], qg[b, j], u_d[b, j], int(cg[b, j + 1])), (rnd, b, j)
                    n_ok = j
                    break
            assert np.abs(dg[b, :max(n_ok, 1)] - dlog_ref[:max(n_ok, 1)]).max() < tol
            if n_ok < k:
                alive[b] = False
                continue
            vlog = OS.verify(dec, c, s, hL_ref, shape.exit_layer)
            assert np.abs(lg[b] - vlog).max() < tol, (rnd, b)
            p_ref = np.stack([A.top_p_filter(r, top_p) for r in A.probs_at(vlog, T)])
            a_o, n_o = A.accept_sampling_chain(p_ref, q_ref, d_ref, u[b])
            if (a_o, n_o) != (a_ref, n_ref):
                alive[b] = False             # p or q moved across a decision: stop following
                continue
            c.length = A.commit_chain(s, a_o)
            assert after[b] == c.length
            compared += 1
        t0 = nxt.clone()
    return compared


def test_sampling_rounds_f32_model():
    """Config-1 shape (f32, 2 layers, exit layer 1), 3 sequences, k = 4, T = 0.8,
    top-p 0.9, 4 rounds; the oracle follows every sequence."""
    spec = _spec()
    shape = SHAPES["tiny"]
    model, dec, shape = model_pair(shape, seed=1, max_rows=64, max_batch=4, max_position=512)
    B, k, T = 3, 4, 0.8
    prompt_len = 32
    kv = spec.KVCache(model, B, 256)
    caches = {}
    t0 = []
    for b in range(B):
        pr = make_tokens(prompt_len, shape.vocab, seed=10 + b)
        last = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        spec.spec_prefill(model, kv, b, cuda_i32(pr), last_logits=last)
        c = dec.new_cache(256)
        ref_last = dec.prefill(c, pr)
        assert np.abs(last.cpu().numpy() - ref_last).max() < 2e-3
        caches[b] = c
        t0.append(int(np.argmax(ref_last)))
    n = _sampling_rounds(spec, model, dec, shape, kv, caches, cuda_i32(t0), k, T, TOP_P, rounds=4, seed=30,
                         tol=2e-3, check_full=True)
    assert n >= 2 * B


def test_sampling_round_7b_ctx4096():
    """The 7B bf16 shape at context 4096 (exit layer 12, k = 4), batch 2, T = 0.8,
    top-p 0.9, 2 rounds; the oracle follows sequence 0."""
    spec = _spec()
    shape = SHAPES["llama7b"]
    CTX, B, k, T = 4096, 2, 4, 0.8
    w = make_weights(shape, seed=4, device="cuda")
    dec = Decoder(shape, weights_to_numpy(w))
    model = spec.Model(shape, w, max_rows=64, max_batch=B, max_position=CTX + 64)
    del w
    torch.cuda.empty_cache()
    cap = CTX + 32
    kv = spec.KVCache(model, B, cap)
    caches = {}
    for b in range(B):
        kc, vc = make_kv_context(shape, 1, CTX, seed=4000 + b, device="cuda")
        kv.import_rows(b, 0, kc[:, 0].contiguous(), vc[:, 0].contiguous())
        if b == 0:
            c = dec.new_cache(cap)
            c.load(kc[:, 0].float().cpu().numpy(), vc[:, 0].float().cpu().numpy())
            caches[b] = c
        del kc, vc
    torch.cuda.empty_cache()
    kv.set_lengths([CTX] * B)
    t0 = cuda_i32(make_tokens(B, shape.vocab, seed=4, name="t0"))
    n = _sampling_rounds(spec, model, dec, shape, kv, caches, t0, k, T, TOP_P, rounds=2, seed=40,
                         tol=2e-2, check_full=True)
    assert n >= 1
