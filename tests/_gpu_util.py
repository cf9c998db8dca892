"""Helpers shared by the GPU parity tests (test infrastructure)."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from synthetic import make_weights, weights_to_numpy


def lib():
    from speculative_decoding_verify_04_gb300 import build, spec
    build.build()
    return spec.load()


def to_cuda(w):
    """The weight dict of ``make_weights`` moved to the GPU."""
    return {"embed": w["embed"].cuda(), "lm_head": w["lm_head"].cuda(), "final_norm": w["final_norm"].cuda(),
            "layers": [{k: v.cuda() for k, v in lw.items()} for lw in w["layers"]]}


def model_pair(shape, seed, n_layers=None, max_rows=64, max_batch=8, max_position=4096, device="cuda"):
    """(library Model, oracle Decoder, shape) over the same seeded weights.

    ``device`` is where the weights are drawn: the CPU and the GPU generators
    give different values for one seed, so a test whose seed was chosen by
    running the oracle on the CPU (to keep its top-1/top-2 gaps away from
    near-ties) draws them with ``device="cpu"``; they are then copied to the GPU.
    """
    from speculative_decoding_verify_04_gb300 import spec
    from oracle.decoder import Decoder
    if n_layers is not None:
        shape = dataclasses.replace(shape, n_layers=n_layers)
    w = make_weights(shape, seed, device=device)
    if device != "cuda":
        w = to_cuda(w)
    wn = weights_to_numpy(w)
    model = spec.Model(shape, w, max_rows=max_rows, max_batch=max_batch, max_position=max_position)
    del w
    torch.cuda.synchronize()
    return model, Decoder(shape, wn), shape


def stats_cols(stats):
    s = stats.detach().cpu()
    return s[:, 0].numpy(), s[:, 1].numpy(), s[:, 2].numpy(), s.view(torch.int32)[:, 3].numpy()


def top_gap(row):
    r = np.sort(np.asarray(row, dtype=np.float64))
    return r[-1] - r[-2]


def assert_tokens_match(gpu, ref, ref_gaps, tol_gap=1e-2, what="tokens"):
    """Equal token for token, except that from the first position where the oracle's
    top-1 / top-2 logit gap is below ``tol_gap`` the two may diverge.  Returns the
    number of positions compared."""
    for i, (g, r) in enumerate(zip(gpu, ref)):
        if g != r:
            assert ref_gaps[i] < tol_gap, f"{what}[{i}]: gpu {g} != oracle {r} with oracle gap {ref_gaps[i]:.3g}"
            return i
    return min(len(gpu), len(ref))


def cuda_i32(x):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).cuda()
