"""Closed-form speedup models printed on the pages (oracle).  Test infrastructure only.

* Self-speculative decoding page (m.lqnn.cn/news/278124, §3.2): with
  independent per-position acceptance alpha and draft length k a round emits
  E(k) = (1 - alpha^(k+1)) / (1 - alpha) tokens on average and costs
  c*k + 1 full forwards (c = draft cost relative to a full forward), so the
  speedup is E(k) / (c*k + 1).
* DSpark page (0539edu.com/news/4524681, §2.4): a round of one target
  forward (time T) and K draft forwards (time t each) yielding a tokens gives
  a*T / (T + K*t).
"""
from __future__ import annotations


def expected_tokens(alpha, k):
    """E(k) = (1 - alpha^(k+1)) / (1 - alpha); k + 1 at alpha = 1."""
    if alpha == 1.0:
        return float(k + 1)
    return (1.0 - alpha ** (k + 1)) / (1.0 - alpha)


def expected_tokens_positional(betas):
    """Mean emitted tokens with per-position acceptance probabilities ``betas``.

    1 + sum_j prod_{i<=j} beta_i: the j-th draft token is kept only if all
    before it are; a round always emits at least one token.
    """
    tot, run = 1.0, 1.0
    for b in betas:
        run *= b
        tot += run
    return tot


def layer_skip_speedup(alpha, k, c):
    """E(k) / (c*k + 1)."""
    return expected_tokens(alpha, k) / (c * k + 1.0)


def best_k(alpha, c, k_max=16):
    """Draft length maximising :func:`layer_skip_speedup` over 1..k_max."""
    return max(range(1, k_max + 1), key=lambda k: layer_skip_speedup(alpha, k, c))


def dspark_speedup(a, K, t_over_T):
    """a*T / (T + K*t) with t expressed as a fraction of T."""
    return a / (1.0 + K * t_over_T)
