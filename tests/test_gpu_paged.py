"""Paged KV cache ("self-speculative decoding" page, m.lqnn.cn/news/278124,
sections 3.3 and 4.5: page-granular rollback and compaction).

The same rounds run on a contiguous cache and on a paged one whose pool is
smaller than the batch's full capacity, so pages move between sequences as
they are rolled back and taken again.  Every output must be bit-identical
(the arithmetic and its order do not depend on where a slot lives), and after
every commit each sequence holds exactly the pages that cover its committed
slots, no page twice, the rest free.
"""
import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, model_pair
from synthetic import SHAPES, ModelShape, make_kv_context, make_tokens, tree_parents

pytestmark = pytest.mark.gpu

PAGE = 64


def _check_pages(kv, n_pages):
    lens = kv.get_lengths()
    table = kv.page_table()
    held = []
    for b, row in enumerate(table):
        need = (lens[b] + PAGE - 1) // PAGE
        assert all(p >= 0 for p in row[:need]) and all(p < 0 for p in row[need:]), (b, lens[b], row)
        held += row[:need]
    assert len(set(held)) == len(held) and all(0 <= p < n_pages for p in held)
    assert kv.free_pages() == n_pages - len(held)


def test_paged_chain_rounds_f32():
    """Tiny f32 model, 3 sequences with prompts of 40, 70 and 130 tokens, 12
    greedy chain rounds of k = 4 plus a sampling round; pool of 9 pages of 64
    (the batch could address 3 x 5)."""
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    model, dec, shape = model_pair(SHAPES["tiny"], seed=1, max_rows=64, max_batch=4, max_position=512)
    B, k, cap, n_pages = 3, 4, 320, 9
    kv_c = spec.KVCache(model, B, cap)
    kv_p = spec.KVCache(model, B, cap, page=PAGE, n_pages=n_pages)
    for b, n in enumerate([40, 70, 130]):
        pr = cuda_i32(make_tokens(n, shape.vocab, seed=20 + b))
        spec.spec_prefill(model, kv_c, b, pr)
        spec.spec_prefill(model, kv_p, b, pr)
    _check_pages(kv_p, n_pages)
    t0 = cuda_i32(make_tokens(B, shape.vocab, seed=30))
    outs = {}
    for name, kv in (("c", kv_c), ("p", kv_p)):
        tc = t0.clone()
        log = []
        for rnd in range(12):
            cand = torch.empty((B, k + 1), dtype=torch.int32, device="cuda")
            hL = torch.empty((B, k + 1, shape.d_model), dtype=torch.float32, device="cuda")
            lg = torch.empty((B * (k + 1), shape.vocab), dtype=torch.float32, device="cuda")
            acc = torch.empty(B, dtype=torch.int32, device="cuda")
            nxt = torch.empty(B, dtype=torch.int32, device="cuda")
            spec.spec_draft(model, kv, tc, k, cand, hL)
            spec.spec_verify(model, kv, [k + 1] * B, cand, k + 1, h_in=hL, h_stride=k + 1, logits=lg, acc_len=acc,
                             next_tok=nxt)
            spec.kv_commit(kv, acc)
            torch.cuda.synchronize()
            assert model.device_error() == 0
            log.append((cand.cpu().numpy(), lg.cpu().numpy(), acc.cpu().numpy(), kv.get_lengths()))
            if name == "p":
                _check_pages(kv, n_pages)
            tc = nxt.clone()
        outs[name] = log
    for (c1, l1, a1, n1), (c2, l2, a2, n2) in zip(outs["c"], outs["p"]):
        np.testing.assert_array_equal(c1, c2)
        np.testing.assert_array_equal(l1, l2)
        np.testing.assert_array_equal(a1, a2)
        assert n1 == n2
    # committed rows read back identically
    lens = kv_c.get_lengths()
    for b in range(B):
        kc, vc = kv_c.export_rows(b, 0, shape.n_layers, 0, lens[b])
        kp, vp = kv_p.export_rows(b, 0, shape.n_layers, 0, lens[b])
        assert torch.equal(kc, kp) and torch.equal(vc, vp)
    # rolling lengths back returns pages
    kv_p.set_lengths([10, 0, 64])
    _check_pages(kv_p, n_pages)
    assert kv_p.free_pages() == n_pages - 2


@pytest.mark.parametrize("attn_phase", ["0", "1"])
def test_paged_bf16_chain_and_tree(attn_phase, monkeypatch):
    """bf16 GQA model (the tensor-core GEMM chain, the MMA attention kernel or
    the attention phase with its tensor maps over the page pool); chain
    verification of 4 rows and a 29-node tree round with its compaction, on
    committed contexts of 100, 700 and 1000 slots."""
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    monkeypatch.setenv("SPEC_ATTN_PHASE", attn_phase)
    model, dec, shape = model_pair(SHAPES["tree8"], seed=41, n_layers=3, max_rows=128, max_batch=3,
                                   max_position=1200)
    lens = [100, 700, 1000]
    B, cap = len(lens), 1100
    n_pages = sum((n + 40 + PAGE - 1) // PAGE for n in lens) + 2
    kv_c = spec.KVCache(model, B, cap)
    kv_p = spec.KVCache(model, B, cap, page=PAGE, n_pages=n_pages)
    for b, n in enumerate(lens):
        kc, vc = make_kv_context(shape, 1, n, seed=500 + b, device="cuda")
        for kv in (kv_c, kv_p):
            kv.import_rows(b, 0, kc[:, 0].contiguous(), vc[:, 0].contiguous())
    for kv in (kv_c, kv_p):
        kv.set_lengths(lens)
    _check_pages(kv_p, n_pages)
    par = [int(x) for x in tree_parents([4, 2, 2])]
    n = len(par)
    res = {}
    for name, kv in (("c", kv_c), ("p", kv_p)):
        toks = cuda_i32(make_tokens(B * 4, shape.vocab, seed=42).reshape(B, 4))
        lg = torch.empty((B * 4, shape.vocab), dtype=torch.float32, device="cuda")
        spec.spec_verify(model, kv, [4] * B, toks, 4, logits=lg)
        # tree round from the embeddings, greedy acceptance and commit
        tt = cuda_i32(make_tokens(B * n, shape.vocab, seed=43).reshape(B, n))
        lt = torch.empty((B * n, shape.vocab), dtype=torch.float32, device="cuda")
        acc = torch.empty(B, dtype=torch.int32, device="cuda")
        nxt = torch.empty(B, dtype=torch.int32, device="cuda")
        path = torch.full((B, 64), -1, dtype=torch.int32, device="cuda")
        spec.spec_verify(model, kv, [n] * B, tt, n, tree_parent=par, logits=lt, acc_len=acc, next_tok=nxt, path=path)
        spec.kv_commit(kv, acc, path)
        torch.cuda.synchronize()
        assert model.device_error() == 0
        after = kv.get_lengths()
        rows = [kv.export_rows(b, 0, shape.n_layers, lens[b], after[b] - lens[b]) for b in range(B)]
        res[name] = (lg.cpu().numpy(), lt.cpu().numpy(), acc.cpu().numpy(), nxt.cpu().numpy(), after, rows)
    c, p = res["c"], res["p"]
    np.testing.assert_array_equal(c[0], p[0])
    np.testing.assert_array_equal(c[1], p[1])
    np.testing.assert_array_equal(c[2], p[2])
    np.testing.assert_array_equal(c[3], p[3])
    assert c[4] == p[4]
    for (kc, vc), (kp, vp) in zip(c[5], p[5]):
        assert torch.equal(kc, kp) and torch.equal(vc, vp)
    _check_pages(kv_p, n_pages)


def test_paged_pool_exhaustion_sets_the_error():
    """A pool too small for the rows a call writes: the call's writes to slots
    without a page are skipped and the capacity bit is set (no fault)."""
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    model, dec, shape = model_pair(SHAPES["tiny"], seed=1, max_rows=64, max_batch=2, max_position=512)
    kv = spec.KVCache(model, 2, 256, page=PAGE, n_pages=2)
    spec.spec_prefill(model, kv, 0, cuda_i32(make_tokens(100, shape.vocab, seed=3)))     # takes both pages
    torch.cuda.synchronize()
    assert model.device_error() == 0 and kv.free_pages() == 0
    spec.spec_prefill(model, kv, 1, cuda_i32(make_tokens(10, shape.vocab, seed=4)))      # no page left
    torch.cuda.synchronize()
    assert model.device_error() & spec.DEVERR_CAPACITY


def test_paged_sampling_and_tree_drafts_match_contiguous():
    """The sampling draft and the layer-skip tree draft write the draft's KV
    through the page table too: two rounds of each on a paged cache give the
    contiguous cache's tokens, probabilities and logits bit for bit."""
    from speculative_decoding_verify_04_gb300 import spec
    from synthetic import make_uniforms
    lib()
    model, dec, shape = model_pair(SHAPES["tiny"], seed=1, max_rows=64, max_batch=2, max_position=512)
    B, k, cap, n_pages, T = 2, 4, 256, 6, 0.8
    par = [int(x) for x in tree_parents([3, 2])]
    n = len(par)
    kv_c = spec.KVCache(model, B, cap)
    kv_p = spec.KVCache(model, B, cap, page=PAGE, n_pages=n_pages)
    for b, ln in enumerate([60, 100]):
        pr = cuda_i32(make_tokens(ln, shape.vocab, seed=50 + b))
        spec.spec_prefill(model, kv_c, b, pr)
        spec.spec_prefill(model, kv_p, b, pr)
    out = {}
    for name, kv in (("c", kv_c), ("p", kv_p)):
        t0 = cuda_i32(make_tokens(B, shape.vocab, seed=60))
        log = []
        for rnd in range(2):
            ud = torch.from_numpy(make_uniforms((B, k), seed=70 + rnd, name="ud")).cuda()
            ua = torch.from_numpy(make_uniforms((B, k + 1), seed=70 + rnd, name="ua")).cuda()
            cand = torch.empty((B, k + 1), dtype=torch.int32, device="cuda")
            hL = torch.empty((B, k + 1, shape.d_model), dtype=torch.float32, device="cuda")
            q = torch.empty((B, k, shape.vocab), dtype=torch.float32, device="cuda")
            lg = torch.empty((B * (k + 1), shape.vocab), dtype=torch.float32, device="cuda")
            p = torch.empty_like(lg)
            acc = torch.empty(B, dtype=torch.int32, device="cuda")
            nxt = torch.empty(B, dtype=torch.int32, device="cuda")
            spec.spec_draft_sample(model, kv, t0, k, T, ud, cand, hL, q)
            spec.spec_verify(model, kv, [k + 1] * B, cand, k + 1, h_in=hL, h_stride=k + 1, logits=lg)
            spec.spec_probs(lg, p, T)
            spec.spec_accept(p.view(B, k + 1, shape.vocab), q, cand[:, 1:], ua, acc, nxt)
            spec.kv_commit(kv, acc)
            t0 = nxt.clone()
            # a layer-skip tree round from the emitted token
            toks = torch.empty((B, n), dtype=torch.int32, device="cuda")
            th = torch.empty((B, n, shape.d_model), dtype=torch.float32, device="cuda")
            scratch = torch.empty((B * n, shape.vocab), dtype=torch.float32, device="cuda")
            tl = torch.empty((B * n, shape.vocab), dtype=torch.float32, device="cuda")
            path = torch.full((B, 64), -1, dtype=torch.int32, device="cuda")
            spec.spec_draft_tree(model, kv, t0, par, toks, th, scratch)
            spec.spec_verify(model, kv, [n] * B, toks, n, h_in=th, h_stride=n, tree_parent=par, logits=tl,
                             acc_len=acc, next_tok=nxt, path=path)
            spec.kv_commit(kv, acc, path)
            torch.cuda.synchronize()
            assert model.device_error() == 0
            log.append([x.cpu() for x in (cand, q, lg, p, toks, tl, acc, nxt)] + [kv.get_lengths()])
            t0 = nxt.clone()
        out[name] = log
    for rc, rp in zip(out["c"], out["p"]):
        for a, b in zip(rc[:-1], rp[:-1]):
            assert torch.equal(a, b)
        assert rc[-1] == rp[-1]
    _check_pages(kv_p, n_pages)


def test_paged_tables_and_rows_match_the_oracle_allocator():
    """The paged cache against the oracle's page allocator (oracle/paged.py),
    call by call: after every prefill, draft, commit and change of lengths the
    GPU's page table and free count equal the allocator's.  The model's layers
    past the exit layer add nothing (zero O and down projections), so every
    round keeps all k drafts and sequences grow by k + 1 slots a round; a
    rollback midway hands pages from one sequence to the others.  At the end
    every committed K/V row of every layer is read from the raw pool at the
    (page, row) the allocator names -- not through the library's page table --
    and compared with the oracle decoder's cache."""
    from speculative_decoding_verify_04_gb300 import spec
    from oracle import spec as OS
    from oracle.decoder import Decoder
    from oracle.paged import PagePool
    from synthetic import make_weights, weights_to_numpy
    lib()
    shape = SHAPES["tiny"]
    w = make_weights(shape, 2, device="cuda")
    for layer in w["layers"][shape.exit_layer:]:
        layer["wo"].zero_()
        layer["w_down"].zero_()
    dec = Decoder(shape, weights_to_numpy(w))
    model = spec.Model(shape, w, max_rows=64, max_batch=4, max_position=512)
    del w
    B, k, cap, n_pages = 3, 4, 320, 9
    kv = spec.KVCache(model, B, cap, page=PAGE, n_pages=n_pages)
    pool = PagePool(B, cap, PAGE, n_pages)
    caches = [dec.new_cache(cap) for _ in range(B)]

    def same():
        assert kv.page_table() == pool.table
        assert kv.free_pages() == pool.free_count()

    prompts = [make_tokens(n, shape.vocab, seed=20 + b) for b, n in enumerate([40, 70, 130])]
    t0 = []
    for b, pr in enumerate(prompts):
        nxt = torch.empty(1, dtype=torch.int32, device="cuda")
        spec.spec_prefill(model, kv, b, cuda_i32(pr), next_tok=nxt)
        pool.ensure_relative([c.length for c in caches[:b + 1]], [0] * b + [len(pr)])
        same()
        t0.append(int(np.argmax(dec.prefill(caches[b], pr))))
    cand = torch.empty((B, k + 1), dtype=torch.int32, device="cuda")
    hL = torch.empty((B, k + 1, shape.d_model), dtype=torch.float32, device="cuda")
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    moved = False
    for rnd in range(10):
        if rnd == 5:
            # roll sequences 0 and 1 back: their pages past the new lengths return to the pool
            lens = [10, 64, caches[2].length]
            kv.set_lengths(lens)
            pool.set_lengths(lens)
            same()
            for b in range(B):
                caches[b].length = lens[b]
            t0 = [int(x) for x in make_tokens(B, shape.vocab, seed=29)]
            moved = True
        lens = [c.length for c in caches]
        spec.spec_draft(model, kv, cuda_i32(t0), k, cand, hL)
        pool.ensure_relative(lens, [k + 1] * B)
        same()
        spec.spec_verify(model, kv, [k + 1] * B, cand, k + 1, h_in=hL, h_stride=k + 1, acc_len=acc, next_tok=nxt)
        spec.kv_commit(kv, acc)
        torch.cuda.synchronize()
        outs = [OS.spec_round_greedy(dec, caches[b], t0[b], k) for b in range(B)]
        assert acc.cpu().tolist() == [o[1] for o in outs] == [k] * B
        assert nxt.cpu().tolist() == [o[2] for o in outs]
        assert kv.get_lengths() == [c.length for c in caches]
        pool.release([c.length for c in caches])
        same()
        t0 = [o[2] for o in outs]
    assert moved and model.device_error() == 0
    # committed rows, read from the raw pool at the allocator's (page, row)
    pages = {}
    for b in range(B):
        for s in range(caches[b].length):
            page, row = pool.locate(b, s)
            assert page >= 0
            for layer in range(shape.n_layers):
                for which, ref in ((0, caches[b].k[layer]), (1, caches[b].v[layer])):
                    key = (which, layer, page)
                    if key not in pages:
                        pages[key] = kv.read_page(which, layer, page).float().numpy()
                    np.testing.assert_allclose(pages[key][:, row, :], ref[s], atol=2e-3, rtol=0)
