"""The LM head's fused row summaries against the logits the same call writes.

For every verified row the head reports a summary (largest logit, its index,
the largest value besides that element, sum of exp(l - largest)) merged from
per-tile summaries, and the fused greedy acceptance decides from the
summaries' argmax.  These must agree with the logits row the same launch
writes: the largest value, its lowest index and the second value exactly
(under a tie the second value equals the first), the sum within 1e-5
relative.  The head weights repeat scaled rows so that exact ties sit at the
top of the rows: neighbouring lanes of one 128-logit tile (rows 3 and 4), one
lane's two registers (rows 3 and 35) and, when the split arithmetic allows,
another tile (row 131).  Both heads: the tensor-core one (bf16 model) and the
CUDA-core one (f32 model); calls of 1 row, of a 5-row chain whose drafts are
planted to be accepted in full, and of a 29-node tree.
"""
import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib, stats_cols, to_cuda
from synthetic import ModelShape, make_tokens, make_weights, tree_parents

pytestmark = pytest.mark.gpu

SETS = (((3, 4, 35, 131), 900, 8.0), ((7, 8, 39, 135), 900, -8.0),
        ((11, 12, 43, 139), 901, 8.0), ((15, 16, 47, 143), 901, -8.0))


def _model(dtype, seed):
    from speculative_decoding_verify_04_gb300 import spec
    shape = ModelShape(2, 256, 4, 4, 64, 512, 1024, 1, dtype)
    w = make_weights(shape, seed, device="cpu")
    head = w["lm_head"]
    for rows, src, scale in SETS:          # scale by a power of two: exact in bf16 too
        v = (head[src].float() * scale).to(head.dtype)
        for r in rows:
            head[r] = v
    model = spec.Model(shape, to_cuda(w), max_rows=64, max_batch=1, max_position=256)
    return model, shape


def _check_rows(stats, logits):
    top1, top2, sum_exp, am = stats_cols(stats)
    lg = logits.cpu().numpy().astype(np.float64)
    ties = 0
    for i, row in enumerate(lg):
        srt = np.sort(row)
        assert top1[i] == srt[-1], (i, top1[i], srt[-1])
        assert am[i] == int(np.argmax(row)), (i, am[i], int(np.argmax(row)))   # numpy: first index of the max
        assert top2[i] == srt[-2], (i, top2[i], srt[-2])
        want = np.exp(row - srt[-1]).sum()
        assert abs(sum_exp[i] - want) <= 1e-5 * want, (i, sum_exp[i], want)
        ties += int(srt[-1] == srt[-2])
    return am, ties


def _verify(spec, model, kv, shape, toks, parents=None):
    T = toks.shape[1]
    logits = torch.empty((T, shape.vocab), dtype=torch.float32, device="cuda")
    stats = torch.empty((T, 4), dtype=torch.float32, device="cuda")
    acc = torch.empty(1, dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    path = torch.full((1, 64), -1, dtype=torch.int32, device="cuda")
    spec.spec_verify(model, kv, [T], toks, T, tree_parent=parents, logits=logits, stats=stats, acc_len=acc,
                     next_tok=nxt, path=path)
    torch.cuda.synchronize()
    assert model.device_error() == 0
    return logits, stats, acc.item(), nxt.item(), path.cpu().numpy()[0]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_head_summaries_match_the_logits(dtype):
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    model, shape = _model(dtype, seed=71)
    kv = spec.KVCache(model, 1, 128)
    spec.spec_prefill(model, kv, 0, cuda_i32(make_tokens(20, shape.vocab, seed=71)))
    torch.cuda.synchronize()
    total_ties = 0

    # one row
    toks = cuda_i32(make_tokens(1, shape.vocab, seed=72).reshape(1, 1))
    logits, stats, a, n, _ = _verify(spec, model, kv, shape, toks)
    am, t = _check_rows(stats, logits)
    total_ties += t
    assert (a, n) == (0, am[0])

    # a 5-row chain: each draft planted as the previous row's argmax, so all four are accepted
    k = 4
    toks = cuda_i32(make_tokens(k + 1, shape.vocab, seed=73).reshape(1, k + 1))
    for j in range(k):
        _, stats, _, _, _ = _verify(spec, model, kv, shape, toks)
        toks[0, j + 1] = int(stats_cols(stats)[3][j])
    logits, stats, a, n, _ = _verify(spec, model, kv, shape, toks)
    am, t = _check_rows(stats, logits)
    total_ties += t
    assert list(toks.cpu().numpy()[0, 1:]) == list(am[:k])
    assert (a, n) == (k, am[k])

    # a 29-node tree: the accepted path follows the summaries' argmax
    par = [int(p) for p in tree_parents([4, 2, 2])]
    toks = cuda_i32(make_tokens(29, shape.vocab, seed=74).reshape(1, 29))
    _, stats, _, _, _ = _verify(spec, model, kv, shape, toks, par)
    am0 = stats_cols(stats)[3]
    toks[0, 2] = int(am0[0])                 # node 2 (depth 1) continues the root
    logits, stats, a, n, path = _verify(spec, model, kv, shape, toks, par)
    am, t = _check_rows(stats, logits)
    total_ties += t
    tk = toks.cpu().numpy()[0]
    depth = [0] * 29
    ok = [True] + [False] * 28
    best = 0
    for i in range(1, 29):
        depth[i] = depth[par[i]] + 1
        ok[i] = ok[par[i]] and tk[i] == am[par[i]]
        if ok[i] and depth[i] > depth[best]:
            best = i
    assert a == depth[best] >= 1
    assert n == am[best]
    assert path[a] == best and path[0] == 0

    # the repeated head rows put exact ties at the top of the rows
    assert total_ties >= 1
