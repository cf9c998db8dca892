"""spec_verify_noalloc against spec_verify.

The no-allocation entry point serves callers that cannot call cudaMalloc
where they verify: a runtime whose device memory all belongs to its own pool,
or a loop that cannot take the synchronisation an allocation may imply.  Its
scratch is a static device array; the first call on a device looks up that
array's address.  Here it runs twice in a row -- the second call finds the
first call's contents in the array -- and each time its logits, row summaries
and greedy acceptance must equal the ordinary entry point's bit for bit on the
same inputs (the same kernels run with the same work split and the same fixed
reduction order; only the scratch lives elsewhere), in chain and in tree mode,
on a bf16 model (tensor-core GEMMs) and on an f32 one (CUDA-core GEMMs).
"""
import dataclasses

import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, model_pair
from synthetic import SHAPES, make_tokens, tree_parents

pytestmark = pytest.mark.gpu



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


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mode", ["chain", "tree"])
def test_noalloc_matches_verify_twice(mode, dtype):
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    base = SHAPES["tree8"] if dtype == "bf16" else SHAPES["tiny"]
    shape0 = dataclasses.replace(base, exit_layer=0)
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
        np.testing.assert_array_equal(got[0], ref[0])
        assert torch.equal(got[1].view(torch.int32), ref[1].view(torch.int32))
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


def test_noalloc_checks_arguments_before_enqueueing():
    """A cache of another model, a null token pointer or more rows than the
    model holds are refused with the argument error, not a scratch error."""
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    shape0 = dataclasses.replace(SHAPES["tiny"], exit_layer=0)
    m1, _, shape = model_pair(shape0, seed=79, n_layers=1, max_rows=16, max_batch=2, max_position=128)
    m2, _, _ = model_pair(shape0, seed=80, n_layers=1, max_rows=16, max_batch=2, max_position=128)
    kv2 = spec.KVCache(m2, 2, 64)
    kv1 = spec.KVCache(m1, 2, 64)
    toks = cuda_i32(np.zeros((2, 12), dtype=np.int32))
    with pytest.raises(spec.SpecError, match="another model"):
        spec.spec_verify_noalloc(m1, kv2, [4, 4], toks, 12)
    with pytest.raises(spec.SpecError, match="max_rows"):
        spec.spec_verify_noalloc(m1, kv1, [12, 12], toks, 12)
    assert kv1.get_lengths() == [0, 0] and m1.device_error() == 0
