"""Alternative draft-length schedules on the GPU, bit-exact against the oracle.

* the DSpark confidence schedule with its first-token-rejection reset
  (DSpark page, 0539edu.com/news/4524681, section 2.3);
* additive increase / decrease over a 64-round window (self-speculative
  decoding page, m.lqnn.cn/news/278124, section 3.2), followed round by round
  over 160 rounds so that the window fills, slides and both thresholds fire;
* the linearly shrinking K_t (speculative decoding principles and practice
  page, intelliparadigm.com/article/weixin_33702545/2059090, section 3.3),
  including exact half-way values.
"""
import numpy as np
import pytest
import torch

from _gpu_util import cuda_i32, lib
from oracle import accept as A

pytestmark = pytest.mark.gpu


def _spec():
    from speculative_decoding_verify_04_gb300 import spec
    lib()
    return spec


def test_first_reject_reset_bit_exact():
    spec = _spec()
    rng = np.random.default_rng(11)
    B = 160
    ks = rng.integers(2, 17, B)
    n_rows = [int(k) + 1 for k in ks]
    T = sum(n_rows)
    p1 = rng.uniform(0.5, 1, T)
    p2 = p1 * rng.uniform(0, 0.2, T)
    probs = np.stack([p1, p2], 1)
    a = np.array([0 if b % 3 == 0 else rng.integers(0, k + 1) for b, k in enumerate(ks)], dtype=np.int32)
    ema0 = rng.uniform(0.5, 1, B)
    ema = torch.from_numpy(ema0.copy()).cuda()
    kn = torch.empty(B, dtype=torch.int32, device="cuda")
    conf = torch.empty(B, dtype=torch.float64, device="cuda")
    spec.spec_schedule_k(torch.from_numpy(probs).cuda(), n_rows, cuda_i32(a), ema, kn, conf, first_reject_min=True)
    torch.cuda.synchronize()
    sch = A.KSchedule(first_reject_min=True)
    r, resets = 0, 0
    for b in range(B):
        n = n_rows[b]
        kk, e, c = A.schedule_update(ema0[b], int(a[b]), n - 1, p1[r:r + n], p2[r:r + n], sch)
        plain = A.schedule_update(ema0[b], int(a[b]), n - 1, p1[r:r + n], p2[r:r + n])[0]
        resets += plain != kk
        r += n
        assert kn[b].item() == kk and ema[b].item() == e and conf[b].item() == c
    assert resets > 0


def test_aimd_rounds_bit_exact():
    spec = _spec()
    rng = np.random.default_rng(12)
    B, W, rounds = 48, 64, 160
    sch = A.AIMDSchedule()
    state = spec.aimd_state(B, W)
    hist = [[] for _ in range(B)]
    k_host = [2] * B
    # acceptance propensity per sequence: mostly kept, mixed, mostly rejected
    prop = np.concatenate([np.full(B // 3, 0.97), np.full(B // 3, 0.78), np.full(B - 2 * (B // 3), 0.3)])
    seen_up = seen_down = False
    k_cur = cuda_i32(k_host)
    k_next = torch.empty(B, dtype=torch.int32, device="cuda")
    for rnd in range(rounds):
        phase = prop if rnd < 100 else prop[::-1]        # flip the regimes to make k come back down
        a = np.array([rng.binomial(k_host[b], phase[b]) for b in range(B)], dtype=np.int32)
        spec.spec_schedule_aimd(cuda_i32(a), k_cur, state, k_next, window=W)
        torch.cuda.synchronize()
        got = k_next.cpu().numpy()
        for b in range(B):
            want, hist[b] = A.aimd_update(hist[b], int(a[b]), k_host[b], sch)
            assert got[b] == want, (rnd, b, got[b], want)
            seen_up |= want > k_host[b]
            seen_down |= want < k_host[b]
            k_host[b] = want
        k_cur = k_next.clone()
    assert seen_up and seen_down
    assert min(k_host) >= sch.min_k and max(k_host) <= sch.max_k


def test_decay_bit_exact():
    spec = _spec()
    rng = np.random.default_rng(13)
    B = 4096
    T = rng.integers(1, 400, B)
    t = rng.integers(0, 500, B)
    k_max = 7
    # exact halves: k_max (1 - t/T) = j + 1/2 for T = 2 k_max and odd t
    T[:64] = 2 * k_max
    t[:64] = np.arange(64) % (2 * k_max)
    kn = torch.empty(B, dtype=torch.int32, device="cuda")
    spec.spec_schedule_decay(cuda_i32(t), cuda_i32(T), k_max, kn)
    torch.cuda.synchronize()
    got = kn.cpu().numpy()
    want = [A.decay_k(int(t[b]), int(T[b]), k_max) for b in range(B)]
    np.testing.assert_array_equal(got, want)
