"""Acceptance, sampling, KV commit and draft-length scheduling (oracle).

Test infrastructure only.  Sources:

* Greedy chain acceptance: the draft token at position j is kept while it
  equals the target's argmax at the previous row; the first mismatch is
  replaced by the target's argmax and the rest is dropped.  With every draft
  token kept, the target's argmax after the last one is emitted as a bonus
  token (self-speculative decoding page, m.lqnn.cn/news/278124, §1.2, §2.1,
  §2.4; DSpark page, 0539edu.com/news/4524681, §2.1).
* Rejection sampling: keep draft token x with probability min(1, p(x)/q(x))
  (ratio 0 when q(x) = 0); on rejection resample from max(0, p - q)
  normalised, falling back to p when that residual is all zero; after k
  kept tokens draw one bonus token from the last target row
  (self-speculative decoding page, §2.4 and §4.3; §5.2 insists on the clip).
* Tree acceptance: the longest root-to-node path whose every token equals the
  argmax of its parent's row (FlashSpec page, lnrk.cn/news/47842, §1.2, §4.1).
* Commit / rollback: the cache keeps the accepted prefix only and its write
  pointer equals the committed length (self-speculative decoding page, §3.3).
* Draft-length schedule: DSpark page §2.2 (confidence score) and §2.3 (linear
  map with thresholds, clamped); optionally its §2.3 refinement: after a round
  whose first draft token was rejected, k drops to its minimum at once.
* Alternative schedules: the additive increase / decrease of the
  self-speculative decoding page (§3.2: window of the last 64 rounds, k + 1
  above 0.85 acceptance, k - 1 below 0.7, k in [2, 8]) and the linearly
  shrinking K_t of the speculative decoding principles and practice page
  (intelliparadigm.com/article/weixin_33702545/2059090, §3.3).

Readings where the pages are silent
-----------------------------------
* argmax ties break to the lowest token id, over the logits.
* "sample" (not specified) is an integer inverse CDF: weights
  w_x = floor(r_x * 2^32) of a float32 row r, S = sum w, a float32 uniform
  u = m * 2^-24 with integer m selects t = floor(m * S / 2^24) and the token
  is the smallest x whose inclusive prefix sum of w exceeds t.
* The ratio test is ``u * q(x) < p(x)`` evaluated exactly in float64 (the
  product of two float32 values is exact there), which equals u < p/q.
* The residual max(0, p - q) is formed with one float32 subtraction.
* u[k] (the last uniform of a sequence) drives whichever of the residual or
  bonus draw happens; u[0..k-1] drive the ratio tests.
* Additive schedule: the window's acceptance is kept / drafted over the last
  64 rounds (fewer at the start); crossing a threshold is read as being
  beyond it after the round (every round while beyond, as congestion control
  adds every round), strictly: exactly 0.85 or 0.7 leaves k unchanged.
  The comparison is exact (integers against the thresholds as fractions).
* Committed length after a round is s + a + 1 (the round's first row t0
  plus a accepted draft tokens); the emitted next token is not yet in the
  cache.  The page's own ``seq_len + i`` counts from a different origin.
* Temperature: both distributions are softmax(logits / T) with one T on both
  sides (self-speculative decoding page, §2.4 warns that unequal
  temperatures bias the output without any visible error), computed in
  float64 and rounded to float32.
* Top-p: of the page's two options (§3.4) the second is taken -- the draft
  distribution q stays whole, only the target p is truncated to its nucleus
  and renormalised there, so the ratio test runs against the full q.  The
  nucleus is the shortest run of tokens, in order of decreasing probability
  with ties to the lower token id, whose mass reaches top_p.  Mass is counted
  in the sampler's integer weights, so the cut is exact: with S = sum w and
  top_p = m * 2^-24, the run stops at the first cumulative weight
  >= ceil(m * S / 2^24).  top_p >= 1 keeps the whole row.
"""
from __future__ import annotations

from dataclasses import dataclass
from fractions import Fraction

import numpy as np

TWO24 = 1 << 24


def argmax_lowest(row):
    """Index of the largest entry; ties go to the lowest index."""
    return int(np.argmax(np.asarray(row)))


# -- greedy -----------------------------------------------------------------
def accept_greedy_chain(draft, logits):
    """Greedy chain acceptance.

    ``draft[k]`` are the draft tokens d_1..d_k; ``logits[k+1, V]`` the target
    rows of t0, d_1, ..., d_k.  Returns ``(a, next_token)``: a = number of
    leading draft tokens equal to the argmax of the preceding row, next =
    argmax of row a (the correction on a mismatch, the bonus if a == k).
    """
    k = len(draft)
    a = 0
    while a < k and int(draft[a]) == argmax_lowest(logits[a]):
        a += 1
    return a, argmax_lowest(logits[a])


def tree_depths(parents):
    d = np.zeros(len(parents), dtype=np.int64)
    for i in range(1, len(parents)):
        d[i] = d[parents[i]] + 1
    return d


def tree_path(parents, node):
    """Rows from the root to ``node`` (inclusive), root first."""
    path = [int(node)]
    while parents[path[-1]] >= 0:
        path.append(int(parents[path[-1]]))
    return path[::-1]


def accept_greedy_tree(tokens, parents, logits):
    """Greedy longest accepted root-to-node path of a level-order tree.

    ``tokens[n]`` (tokens[0] is the root), ``parents[n]`` (parents[0] = -1,
    parents[i] < i), ``logits[n, V]`` the target row of every node.  Node i
    is accepted when its parent is accepted and ``tokens[i]`` equals the
    argmax of the parent's row.  The deepest accepted node wins; equal depth
    goes to the lowest node index.  Returns ``(depth, node, path, next)``.
    """
    n = len(tokens)
    ok = np.zeros(n, dtype=bool)
    ok[0] = True
    depth = tree_depths(parents)
    best = 0
    am = [argmax_lowest(logits[i]) for i in range(n)]
    for i in range(1, n):
        par = parents[i]
        ok[i] = ok[par] and int(tokens[i]) == am[par]
        if ok[i] and depth[i] > depth[best]:
            best = i
    return int(depth[best]), best, tree_path(parents, best), am[best]


# -- sampling -----------------------------------------------------------------
def int_weights(r):
    """floor(r * 2^32) of a float32 row as uint64 (exact: a power-of-two scaling)."""
    r = np.asarray(r, dtype=np.float32).astype(np.float64)
    return np.floor(r * 4294967296.0).astype(np.uint64)


def uniform_to_int(u):
    """The integer m of a float32 uniform u = m * 2^-24."""
    m = float(np.float32(u)) * TWO24
    if not (m == int(m) and 0 <= m < TWO24):
        raise ValueError(f"uniform {u!r} is not a multiple of 2^-24 in [0,1)")
    return int(m)


def sample_threshold(S, m):
    """floor(m * S / 2^24) for S < 2^48 and m < 2^24, in 64-bit pieces."""
    return m * (S >> 24) + ((m * (S & 0xFFFFFF)) >> 24)


def sample_index(w, u):
    """Integer inverse-CDF draw from weights ``w`` (uint64, sum > 0) with uniform ``u``."""
    w = np.asarray(w, dtype=np.uint64)
    S = int(w.sum(dtype=np.uint64))
    if S <= 0:
        raise ValueError("all-zero weights")
    t = sample_threshold(S, uniform_to_int(u))
    c = np.cumsum(w, dtype=np.uint64)
    return int(np.searchsorted(c, np.uint64(t), side="right"))


def probs_at(logits, temp):
    """softmax(logits / temp) along the last axis: float64, rounded to float32."""
    if not (np.isfinite(temp) and temp > 0.0):
        raise ValueError(f"temperature must be positive, got {temp!r}")
    z = np.asarray(logits, dtype=np.float64) / float(temp)
    e = np.exp(z - z.max(axis=-1, keepdims=True))
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def top_p_keep(p_row, top_p):
    """Nucleus of one float32 probability row as a boolean mask."""
    p = np.asarray(p_row, dtype=np.float32)
    V = p.shape[0]
    if top_p >= 1.0:
        return np.ones(V, dtype=bool)
    m = uniform_to_int(top_p)
    if m == 0:
        raise ValueError("top_p must be positive")
    w = int_weights(p)
    S = int(w.sum(dtype=np.uint64))
    t = (m * S + TWO24 - 1) >> 24                       # ceil(m * S / 2^24)
    order = np.lexsort((np.arange(V), -p.astype(np.float64)))   # p descending, then id
    keep = np.zeros(V, dtype=bool)
    mass = 0
    for x in order:
        keep[x] = True
        mass += int(w[x])
        if mass >= t:
            break
    return keep


def top_p_filter(p_row, top_p):
    """The row restricted to its nucleus and renormalised (float64, rounded to float32)."""
    keep = top_p_keep(p_row, top_p)
    p = np.where(keep, np.asarray(p_row, dtype=np.float32).astype(np.float64), 0.0)
    return (p / p.sum()).astype(np.float32)


def ratio_accept(u, qx, px):
    """Keep x iff q(x) > 0 and u < p(x)/q(x), evaluated as exact u*q(x) < p(x)."""
    qx = float(np.float32(qx))
    return qx > 0.0 and float(np.float32(u)) * qx < float(np.float32(px))


def residual(p_row, q_row):
    """max(0, p - q) with one float32 subtraction per entry."""
    d = np.asarray(p_row, dtype=np.float32) - np.asarray(q_row, dtype=np.float32)
    return np.maximum(d, np.float32(0.0))


def accept_sampling_chain(p, q, draft, u):
    """Rejection-sampling chain acceptance for one sequence.

    ``p[k+1, V]`` target probabilities (float32), ``q[k, V]`` draft
    probabilities, ``draft[k]`` draft tokens, ``u[k+1]`` uniforms.  Returns
    ``(a, next_token)``: a = number of kept draft tokens; next is the residual
    draw at the first rejection or the bonus draw from p[k] when all are kept.
    """
    k = len(draft)
    for j in range(k):
        x = int(draft[j])
        if ratio_accept(u[j], q[j, x], p[j, x]):
            continue
        w = int_weights(residual(p[j], q[j]))
        if int(w.sum(dtype=np.uint64)) == 0:
            w = int_weights(p[j])
        return j, sample_index(w, u[k])
    return k, sample_index(int_weights(p[k]), u[k])


# -- commit -----------------------------------------------------------------
def commit_chain(s, a):
    """New committed length after a chain round: t0 plus a kept tokens."""
    return s + a + 1


def commit_tree_moves(s, path):
    """Slot moves that compact a tree path into consecutive slots.

    Node ``path[d]`` (depth d) was verified in slot ``s + path[d]`` and must
    end in slot ``s + d``.  Moves run in increasing depth; a destination is
    never a later source because path rows grow at least as fast as depth.
    Returns ``(moves, new_length)``.
    """
    moves = [(s + int(path[d]), s + d) for d in range(1, len(path))]
    return moves, s + len(path)


def apply_moves(cache, moves, layers=None):
    layers = range(len(cache.k)) if layers is None else layers
    for l in layers:
        for src, dst in moves:
            cache.k[l][dst] = cache.k[l][src]
            cache.v[l][dst] = cache.v[l][src]


# -- confidence-scheduled draft length ---------------------------------------
@dataclass
class KSchedule:
    """DSpark schedule constants (min/max k, thresholds, EMA decay)."""
    min_k: int = 2
    max_k: int = 16
    low: float = 0.3
    high: float = 0.8
    decay: float = 0.9
    k0: int = 2
    ema0: float = 0.5
    first_reject_min: bool = False   # a round whose first draft token is rejected resets k to min_k


def top12_probs(logits_row):
    """Softmax probabilities of the largest and second-largest logits (float64)."""
    z = np.asarray(logits_row, dtype=np.float64)
    m = z.max()
    S = np.exp(z - m).sum()
    i1 = int(np.argmax(z))
    z2 = np.delete(z, i1).max()
    return 1.0 / S, float(np.exp(z2 - m) / S)


def confidence(avg_top1, avg_gap, ema):
    """conf = 0.4 avg_top1 + 0.3 min(5 avg_gap, 1) + 0.3 ema (DSpark §2.2)."""
    return 0.4 * avg_top1 + 0.3 * min(avg_gap * 5.0, 1.0) + 0.3 * ema


def next_k(conf, sch: KSchedule = KSchedule()):
    """Linear map of conf onto [min_k, max_k] between the thresholds, truncated and clamped."""
    k = int(sch.min_k + (sch.max_k - sch.min_k) * (conf - sch.low) / (sch.high - sch.low))
    return max(sch.min_k, min(sch.max_k, k))


def schedule_update(ema, a, k, top1, top2, sch: KSchedule = KSchedule()):
    """One round of the schedule for one sequence.

    ``a`` kept of ``k`` drafted; ``top1``/``top2`` are the target's two largest
    probabilities at each of the k+1 verified rows.  acceptance = a / k, the
    EMA is updated before the score.  Means are left-to-right float64 sums
    divided by the count.  Returns ``(k_next, ema_next, conf)``.
    """
    acc = a / k
    ema = sch.decay * ema + (1.0 - sch.decay) * acc
    n = len(top1)
    s1 = 0.0
    sg = 0.0
    for i in range(n):
        s1 = s1 + float(top1[i])
        sg = sg + (float(top1[i]) - float(top2[i]))
    c = confidence(s1 / n, sg / n, ema)
    k_next = next_k(c, sch)
    if sch.first_reject_min and a == 0:
        k_next = sch.min_k
    return k_next, ema, c


# -- alternative draft-length schedules ---------------------------------------
@dataclass
class AIMDSchedule:
    """Additive increase / decrease of k from a sliding acceptance window
    (self-speculative decoding page, §3.2, last paragraph)."""
    window: int = 64
    up: float = 0.85          # alpha above this: k + 1
    down: float = 0.7         # alpha below this: k - 1
    min_k: int = 2
    max_k: int = 8


def aimd_update(history, a, k, sch: AIMDSchedule = AIMDSchedule()):
    """One round of the additive schedule for one sequence.

    ``history`` is the list of ``(a_i, k_i)`` of earlier rounds (oldest
    first); this round's ``(a, k)`` is appended and only the last
    ``sch.window`` rounds are kept.  alpha = kept / drafted over the window.
    Returns ``(k_next, history)``.
    """
    history = (list(history) + [(int(a), int(k))])[-sch.window:]
    kept = sum(x for x, _ in history)
    drafted = sum(y for _, y in history)
    alpha = Fraction(kept, drafted)
    k_next = k
    if alpha > Fraction(sch.up).limit_denominator(1000):
        k_next = k + 1
    elif alpha < Fraction(sch.down).limit_denominator(1000):
        k_next = k - 1
    return max(sch.min_k, min(sch.max_k, k_next)), history


def decay_k(t, T, k_max):
    """K_t = max(1, round(K_max * (1 - t / T))) (speculative decoding principles
    and practice page, intelliparadigm.com/article/weixin_33702545/2059090, §3.3): the
    draft length shrinks as the generated count t nears the predicted total T.
    float64 arithmetic; round is to the nearest integer, ties to even."""
    return max(1, int(round(float(k_max) * (1.0 - float(t) / float(T)))))
