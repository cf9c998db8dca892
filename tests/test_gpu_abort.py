"""The bounded-wait abort path of the GEMM chain kernel, exercised on the GPU
without a fault or a hang.

Every wait inside the chain kernel is bounded: when one runs out, the CTA
raises its abort flag and SPEC_DEVERR_TIMEOUT, lets its copies in flight land,
drains its MMAs, frees its tensor memory and leaves; the last CTA out resets
the grid-barrier counters.  The test hook spec_test_stall_next_chain makes one
CTA of the next multi-phase chain withhold its arrival at the first grid
barrier and gives that launch's grid waits a 50 ms limit, so every other CTA's
wait runs out.  The call must come back within a fraction of a second with the
timeout bit set, and the next call on the same model and cache must give the
same logits as a call made before the stall (bit for bit) and match the oracle.
"""
import time

import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, to_cuda
from oracle import spec as OS
from oracle.decoder import Decoder
from synthetic import ModelShape, make_kv_context, make_tokens, make_weights, weights_to_numpy

pytestmark = pytest.mark.gpu

SHAPE = ModelShape(3, 4096, 32, 32, 128, 11008, 512, 1, "bf16")   # the 7B layer shape, 3 layers
K, CTX, TIMEOUT_BIT = 4, 64, 4


def test_stalled_barrier_times_out_and_the_next_call_is_clean():
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    w = make_weights(SHAPE, 4, device="cpu")
    dec = Decoder(SHAPE, weights_to_numpy(w))
    model = spec.Model(SHAPE, to_cuda(w), max_rows=64, max_batch=1, max_position=CTX + 32)
    del w
    kv = spec.KVCache(model, 1, CTX + 16)
    kc, vc = make_kv_context(SHAPE, 1, CTX, 400, device="cpu")
    kv.import_rows(0, 0, kc[:, 0].contiguous().cuda(), vc[:, 0].contiguous().cuda())
    kv.set_lengths([CTX])
    cache = dec.new_cache(CTX + 16)
    cache.load(kc[:, 0].float().numpy(), vc[:, 0].float().numpy())
    t0 = int(make_tokens(1, SHAPE.vocab, 4, "t0")[0])

    cand = torch.empty((1, K + 1), dtype=torch.int32, device="cuda")
    hL = torch.empty((1, K + 1, SHAPE.d_model), dtype=torch.float32, device="cuda")
    spec.spec_draft(model, kv, cuda_i32([t0]), K, cand, hL)
    torch.cuda.synchronize()
    assert model.device_error() == 0

    def verify():
        logits = torch.full((K + 1, SHAPE.vocab), float("nan"), dtype=torch.float32, device="cuda")
        spec.spec_verify(model, kv, [K + 1], cand, K + 1, h_in=hL, h_stride=K + 1, logits=logits)
        return logits

    before = verify()
    torch.cuda.synchronize()
    assert model.device_error() == 0

    # the verify's [O, gate/up, down, QKV] chain of layer 1: CTA 3 withholds its arrival
    model.test_stall_next_chain(3, 50_000_000)
    t = time.perf_counter()
    verify()
    torch.cuda.synchronize()
    waited = time.perf_counter() - t
    assert model.device_error() & TIMEOUT_BIT, "the withheld arrival did not end in a timeout"
    assert waited < 1.5, f"the aborted launch took {waited:.2f} s to leave"

    after = verify()
    torch.cuda.synchronize()
    assert model.device_error() == 0
    assert torch.equal(before, after), "the call after the abort differs from the call before it"
    d_ref, hL_ref, _, _ = OS.draft(dec, cache, CTX, t0, K)
    assert cand.cpu().tolist()[0] == [t0] + list(d_ref)
    vlog = OS.verify(dec, cache, CTX, hL_ref, SHAPE.exit_layer)
    err = float(np.abs(after.cpu().numpy() - vlog).max())
    assert err < 2e-2, err
