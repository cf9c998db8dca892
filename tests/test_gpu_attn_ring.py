"""The TMA-ring attention kernel (attn_ring.cu) against the register-tile
kernel and the float64 oracle.

The ring kernel takes calls whose sequences have at most 8 query vectors per
KV head (the layer-skip draft's single row, a chain of a few rows), with the
queries on the MMA's N side; SPEC_ATTN_RING=1 runs one CTA an SM (eight
consumer warps, 12 ring slots), =2 two (four consumer warps, 6 slots each), =0
sends the same calls to the register-tile kernel.  Cases, for both shapes:

* the 7B attention shape (32 heads x 128, no grouping) at batch 1, one row
  (a draft pass) and five rows (a k = 4 chain), contexts long enough for every
  KV head's units to spread over several CTAs (partial states merged across
  CTAs) and short ones that fit in one unit;
* a grouped shape (4 query / 2 KV heads x 64; units of 64 slots), 1..4 rows
  per sequence (2..8 query vectors), ragged contexts over three sequences,
  chain and tree masks, contiguous and paged caches.

Logits must match the oracle within 2e-2 and the register-tile kernel within
2e-3 (the two sum in different orders).
"""
import os

import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, model_pair
from oracle import spec as OS
from synthetic import SHAPES, ModelShape, make_kv_context, make_tokens

pytestmark = pytest.mark.gpu

TOL = 2e-2
GQA2 = ModelShape(2, 256, 4, 2, 64, 512, 2048, 0, "bf16")
WIDE = ModelShape(2, 4096, 32, 32, 128, 11008, 512, 0, "bf16")      # the 7B attention shape, 2 layers


def _models(shape, seed, max_batch, max_position, ring="1"):
    out = []
    for env in (ring, "0"):
        os.environ["SPEC_ATTN_RING"] = env
        os.environ["SPEC_ATTN_PHASE"] = "0"
        try:
            model, dec, sh = model_pair(shape, seed=seed, max_rows=64, max_batch=max_batch,
                                        max_position=max_position)
        finally:
            os.environ.pop("SPEC_ATTN_RING", None)
            os.environ.pop("SPEC_ATTN_PHASE", None)
        out.append(model)
    return out[0], out[1], dec, sh


def _verify(model, shape, lens, n_rows, toks, parents, cap, page, seed):
    from speculative_decoding_verify_04_gb300 import spec
    kv = spec.KVCache(model, len(lens), cap, page=page)
    for b, n in enumerate(lens):
        kc, vc = make_kv_context(shape, 1, n, seed * 100 + b, device="cuda")
        kv.import_rows(b, 0, kc[:, 0].contiguous(), vc[:, 0].contiguous())
    kv.set_lengths(list(lens))
    logits = torch.empty((sum(n_rows), shape.vocab), dtype=torch.float32, device="cuda")
    spec.spec_verify(model, kv, n_rows, toks, toks.shape[1], tree_parent=parents, logits=logits)
    torch.cuda.synchronize()
    assert model.device_error() == 0
    return logits.cpu().numpy()


def _oracle(dec, shape, lens, n_rows, toks, parents, cap, seed):
    out = []
    for b, n in enumerate(lens):
        kc, vc = make_kv_context(shape, 1, n, seed * 100 + b, device="cuda")
        c = dec.new_cache(cap)
        c.load(kc[:, 0].float().cpu().numpy(), vc[:, 0].float().cpu().numpy())
        T = n_rows[b]
        h = dec.embed(toks[b, :T].cpu().numpy())
        out.append(OS.verify(dec, c, n, h, 0, parents=parents))
    return np.concatenate(out)


@pytest.mark.parametrize("variant", ["1", "2"])
@pytest.mark.parametrize("rows,lens", [(1, [4096]), (5, [4096]), (5, [20]), (1, [33])])
def test_ring_attention_7b_shape(rows, lens, variant):
    lib()
    seed = 61
    ring, ref, dec, shape = _models(WIDE, seed, 1, 4200, variant)
    toks = cuda_i32(make_tokens(rows, shape.vocab, seed=seed).reshape(1, rows))
    cap = max(lens) + 16
    got = _verify(ring, shape, lens, [rows], toks, None, cap, None, seed)
    alt = _verify(ref, shape, lens, [rows], toks, None, cap, None, seed)
    want = _oracle(dec, shape, lens, [rows], toks, None, cap, seed)
    assert np.abs(got - want).max() < TOL, np.abs(got - want).max()
    assert np.abs(got - alt).max() < 2e-3, np.abs(got - alt).max()


@pytest.mark.parametrize("variant", ["1", "2"])
@pytest.mark.parametrize("page", [None, 64])
@pytest.mark.parametrize("mode", ["chain", "tree"])
def test_ring_attention_grouped_ragged(mode, page, variant):
    lib()
    seed = 62
    lens = [5, 64, 700]
    if mode == "tree":
        parents = [-1, 0, 0, 1]                  # root, two children, a grandchild
        n_rows = [4, 4, 4]
    else:
        parents = None
        n_rows = [1, 3, 4]
    ring, ref, dec, shape = _models(GQA2, seed, 3, 800, variant)
    cap = 768
    toks = cuda_i32(make_tokens(3 * 4, shape.vocab, seed=seed).reshape(3, 4))
    got = _verify(ring, shape, lens, n_rows, toks, parents, cap, page, seed)
    alt = _verify(ref, shape, lens, n_rows, toks, parents, cap, page, seed)
    want = _oracle(dec, shape, lens, n_rows, toks, parents, cap, seed)
    assert np.abs(got - want).max() < TOL, np.abs(got - want).max()
    assert np.abs(got - alt).max() < 2e-3, np.abs(got - alt).max()
