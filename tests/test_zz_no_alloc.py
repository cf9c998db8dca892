"""spec_verify_noalloc against spec_verify.

The no-allocation entry point serves callers that cannot call cudaMalloc
where they verify (a stream being captured by someone else, a device whose
memory is all in the caller's pool).  Its scratch is a static device array;
the first call on a device looks up that array's address.  Here it runs twice
in a row -- the second call finds the first call's contents in the array --
and each time its logits, row summaries and greedy acceptance must match the
ordinary entry point on the same inputs, in chain and in tree mode.
"""
import dataclasses

import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, model_pair
from synthetic import SHAPES, make_tokens, tree_parents

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _run(entry, model, kv, n_rows, toks, stride, parents, V):
    from speculative_decoding_verify_04_gb300 import spec
    T = sum(n_rows)
    B = len(n_rows)
    logits = torch.full((T, V), float("nan"), dtype=torch.float32, device="cuda")
    stats = torch.zeros((T, 4), dtype=torch.float32, device="cuda")
    acc = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -1, dtype=torch.int32, device="cuda")
    path = torch.full((B, 64), -1, dtype=torch.int32, device="cuda")
    entry(model, kv, n_rows, toks, stride, tree_parent=parents, logits=logits, stats=stats, acc_len=acc,
          next_tok=nxt, path=path)
    torch.cuda.synchronize()
    return logits.cpu().numpy(), stats.cpu(), acc.cpu().numpy(), nxt.cpu().numpy(), path.cpu().numpy()


@pytest.mark.parametrize("mode", ["chain", "tree"])
def test_noalloc_matches_verify_twice(mode):
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    shape0 = dataclasses.replace(SHAPES["tree8"], exit_layer=0)
    model, _, shape = model_pair(shape0, seed=77, n_layers=2, max_rows=64, max_batch=2, max_position=512)
    B = 2
    kv = spec.KVCache(model, B, 256)
    for b in range(B):
        spec.spec_prefill(model, kv, b, cuda_i32(make_tokens(60 + 37 * b, shape.vocab, seed=70 + b)))
    if mode == "tree":
        parents = list(tree_parents([4, 2, 2]))
        n_rows = [len(parents)] * B
    else:
        parents = None
        n_rows = [5, 3]
    stride = max(n_rows)
    toks = cuda_i32(make_tokens(B * stride, shape.vocab, seed=71).reshape(B, stride))
    ref = _run(spec.spec_verify, model, kv, n_rows, toks, stride, parents, shape.vocab)
    for _ in range(2):
        got = _run(spec.spec_verify_noalloc, model, kv, n_rows, toks, stride, parents, shape.vocab)
        assert np.isfinite(got[0]).all()
        assert np.abs(got[0] - ref[0]).max() < TOL
        assert torch.equal(got[1].view(torch.int32)[:, 3], ref[1].view(torch.int32)[:, 3])
        np.testing.assert_array_equal(got[2], ref[2])
        np.testing.assert_array_equal(got[3], ref[3])
        if parents is not None:
            for b in range(B):
                a = int(ref[2][b])
                np.testing.assert_array_equal(got[4][b, :a + 1], ref[4][b, :a + 1])
    assert kv.get_lengths() == [60, 97]
    assert model.device_error() == 0


def test_noalloc_rejects_oversized_call():
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    shape0 = dataclasses.replace(SHAPES["llama7b"], exit_layer=0)
    model, _, shape = model_pair(shape0, seed=78, n_layers=1, max_rows=1024, max_batch=64, max_position=256)
    B = 64
    kv = spec.KVCache(model, B, 128)
    toks = cuda_i32(np.zeros((B, 16), dtype=np.int32))
    with pytest.raises(spec.SpecError, match="scratch"):
        spec.spec_verify_noalloc(model, kv, [16] * B, toks, 16)
