"""Acceptance kernels against the oracle: bit-exact on identical inputs.

Rejection sampling takes the pages' rule (keep x with probability
min(1, p/q), else draw from max(0, p-q), bonus from p_k) with the integer
inverse-CDF draw; greedy acceptance the prefix / tree-path rule.
"""
import numpy as np
import pytest
import torch

from _gpu_util import lib, cuda_i32
from oracle import accept as A
from synthetic import make_accept_inputs, make_uniforms, tree_parents

pytestmark = pytest.mark.gpu


def _run_accept(p, q, x, u):
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    B = p.shape[0]
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    spec.spec_accept(torch.from_numpy(p).cuda(), torch.from_numpy(q).cuda(), cuda_i32(x),
                     torch.from_numpy(u).cuda(), acc, nxt)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), nxt.cpu().numpy()


def _oracle(p, q, x, u):
    out = [A.accept_sampling_chain(p[b], q[b], x[b], u[b]) for b in range(p.shape[0])]
    return np.array([o[0] for o in out]), np.array([o[1] for o in out])


@pytest.mark.parametrize("B,k,V,sigma", [(64, 1, 5, 1.0), (64, 3, 130, 2.0), (32, 5, 1000, 3.0),
                                         (16, 8, 4097, 0.5), (8, 16, 32000, 3.0), (40, 2, 7, 0.2)])
def test_rejection_sampling_bit_exact(B, k, V, sigma):
    p, q, x, u = make_accept_inputs(B, k, V, seed=100 + V, sigma=sigma)
    ga, gn = _run_accept(p, q, x, u)
    oa, on = _oracle(p, q, x, u)
    np.testing.assert_array_equal(ga, oa)
    np.testing.assert_array_equal(gn, on)


def test_rejection_sampling_full_size():
    """256 sequences, k = 5, V = 32000, logits N(0, 3^2), draft = target + N(0, 1)."""
    p, q, x, u = make_accept_inputs(256, 5, 32000, seed=2)
    ga, gn = _run_accept(p, q, x, u)
    oa, on = _oracle(p, q, x, u)
    np.testing.assert_array_equal(ga, oa)
    np.testing.assert_array_equal(gn, on)
    assert 0 < ga.mean() < 5          # both outcomes occur


def test_rejection_sampling_edge_cases():
    V, k, B = 300, 3, 6
    p, q, x, u = make_accept_inputs(B, k, V, seed=5)
    q[0, 0, x[0, 0]] = 0.0                    # q(x) = 0 rejects
    p[1, 0] = q[1, 0]                         # p == q: always kept at position 0 ...
    p[2, 1] = q[2, 1]
    x[2, 1] = int(np.argmax(q[2, 1] == 0)) if (q[2, 1] == 0).any() else x[2, 1]
    u[3, :] = 0.0                             # smallest uniform
    u[4, :] = np.float32(1 - 2.0 ** -24)      # largest uniform
    x[5, :] = 0
    ga, gn = _run_accept(p, q, x, u)
    oa, on = _oracle(p, q, x, u)
    np.testing.assert_array_equal(ga, oa)
    np.testing.assert_array_equal(gn, on)
    assert ga[0] == 0


def test_residual_all_zero_falls_back_to_p():
    V, k = 64, 1
    rng = np.random.default_rng(0)
    z = rng.standard_normal((1, 2, V))
    p = (np.exp(z) / np.exp(z).sum(-1, keepdims=True)).astype(np.float32)
    q = p[:, :1].copy()
    zero = int(np.argmin(q[0, 0]))
    q[0, 0, zero] = 0.0
    p[0, 0, zero] = 0.0                       # residual max(0, p - q) is all zero
    x = np.array([[zero]], dtype=np.int32)    # q(x) = 0 -> rejected
    for m in (0, 1 << 20, (1 << 24) - 1):
        u = np.array([[0.5, m * 2.0 ** -24]], dtype=np.float32)
        ga, gn = _run_accept(p, q, x, u)
        oa, on = _oracle(p, q, x, u)
        assert (ga[0], gn[0]) == (oa[0], on[0]) and ga[0] == 0


def _greedy_gpu(logits, toks, parents=None):
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    B = logits.shape[0]
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    path = torch.full((B, 64), -1, dtype=torch.int32, device="cuda")
    spec.spec_accept_greedy(torch.from_numpy(logits).cuda(), cuda_i32(toks), acc, nxt,
                            tree_parent=None if parents is None else list(parents), path=path)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), nxt.cpu().numpy(), path.cpu().numpy()


def test_greedy_chain_matches_oracle():
    rng = np.random.default_rng(1)
    B, k, V = 64, 6, 500
    logits = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    am = logits.argmax(-1)
    toks = rng.integers(0, V, (B, k + 1)).astype(np.int32)
    for b in range(B):                        # plant a matched prefix of length b % (k + 1)
        for j in range(b % (k + 1)):
            toks[b, j + 1] = am[b, j]
    logits[0, 0, :] = 1.0                     # an all-tie row: argmax is index 0
    toks[0, 1] = 0
    ga, gn, _ = _greedy_gpu(logits, toks)
    for b in range(B):
        assert (ga[b], gn[b]) == A.accept_greedy_chain(toks[b, 1:], logits[b])


def test_greedy_tree_matches_oracle():
    rng = np.random.default_rng(2)
    par = tree_parents([4, 2, 2])
    B, V = 32, 50
    logits = rng.integers(-3, 3, (B, 29, V)).astype(np.float32)   # many exact ties
    toks = rng.integers(0, V, (B, 29)).astype(np.int32)
    for b in range(B):
        for i in range(1, 29):
            if rng.random() < 0.6:
                toks[b, i] = int(np.argmax(logits[b, par[i]]))
    ga, gn, gp = _greedy_gpu(logits, toks, par)
    for b in range(B):
        d, node, path, nxt = A.accept_greedy_tree(toks[b], par, logits[b])
        assert (ga[b], gn[b]) == (d, nxt)
        assert list(gp[b, :d + 1]) == path


def test_schedule_bit_exact():
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    rng = np.random.default_rng(3)
    B = 200
    ks = rng.integers(2, 17, B)
    n_rows = [int(k) + 1 for k in ks]
    T = sum(n_rows)
    p1 = rng.uniform(0, 1, T)
    p2 = p1 * rng.uniform(0, 1, T)
    probs = np.stack([p1, p2], 1)
    a = np.array([rng.integers(0, k + 1) for k in ks], dtype=np.int32)
    ema0 = rng.uniform(0, 1, B)
    ema = torch.from_numpy(ema0.copy()).cuda()
    kn = torch.empty(B, dtype=torch.int32, device="cuda")
    conf = torch.empty(B, dtype=torch.float64, device="cuda")
    spec.spec_schedule_k(torch.from_numpy(probs).cuda(), n_rows, cuda_i32(a), ema, kn, conf)
    torch.cuda.synchronize()
    r = 0
    for b in range(B):
        n = n_rows[b]
        kk, e, c = A.schedule_update(ema0[b], int(a[b]), n - 1, p1[r:r + n], p2[r:r + n])
        r += n
        assert kn[b].item() == kk and ema[b].item() == e and conf[b].item() == c
