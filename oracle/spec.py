"""Layer-skip self-drafting, chain / tree verification and the round loop (oracle).

Test infrastructure only.

A round at committed length s with last emitted token t0 (not yet in the
cache), following the self-speculative decoding page (m.lqnn.cn/news/278124,
§2.1, §3.3, §4.2, §4.3):

1. draft: k passes of layers [0, L) with one row each, t0 at position s
   then d_1 .. d_{k-1} at s+1 .., each through the final norm and the shared
   LM head; d_{j+1} = argmax (greedy) or a draw from q_j = softmax(logits/T).
   Each pass writes layers [0, L) of the cache at its slot.
2. one more first-L pass on d_k at position s+k, without the LM head.  The
   page sends k+1 rows through the upper layers but drafts only k tokens;
   this pass is the plainest way to give the verifier the layer-L hidden
   state of every row while the first-L KV of all k+1 rows comes from the
   draft (KV reuse, §2.1).
3. verify: layers [L, N) on the k+1 hidden rows at positions s .. s+k, each
   row seeing the committed context plus the rows before it (causal), then
   final norm and LM head: k+1 target rows.
4. accept (accept.py), 5. commit: length s + a + 1.

Tree verification (FlashSpec page, lnrk.cn/news/47842, §2.2, §3.2, §4.1,
§5.2): the nodes go in level order, node i at position s + depth(i) in slot
s + i, each seeing the committed context, its ancestors and itself (padding
and siblings masked).  The page's "parent offset + 1" rule is the depth; its
remark that depth ids broke its outputs concerns a target trained with
injected position ids, which a plain target does not have.

Layer-skip trees (same page, §6.2, with the first-L-layer draft): the draft
grows the tree level by level, children taking their parent's best draft
tokens, either in a fixed branching or with a width that follows the
draft's confidence (child_count).
"""
from __future__ import annotations

import dataclasses

import numpy as np

from .accept import (accept_greedy_chain, accept_greedy_tree, accept_sampling_chain,
                     argmax_lowest, commit_chain, commit_tree_moves, apply_moves,
                     int_weights, probs_at, sample_index, top_p_filter, tree_depths)


def draft(dec, cache, s, t0, k, temp=0.0, u_draft=None):
    """Layer-skip draft at committed length ``s`` from token ``t0``.

    Returns ``(draft_tokens[k], h_L[k+1, d], draft_logits[k, V], q[k, V] or None)``.
    ``q`` (float32 softmax at ``temp``) is returned in sampling mode only,
    where ``u_draft[j]`` drives the draw of d_{j+1}.
    """
    L = dec.shape.exit_layer
    toks, hs, lgs, qs = [], [], [], []
    cur = int(t0)
    for j in range(k + 1):
        h = dec.embed([cur])
        vis = [np.arange(0, s + j + 1)]
        h = dec.run_layers(h, 0, L, [s + j], [s + j], vis, cache)
        hs.append(h[0])
        if j == k:
            break
        lg = dec.logits(h)[0]
        lgs.append(lg)
        if temp == 0.0:
            cur = argmax_lowest(lg)
        else:
            q = probs_at(lg, temp)
            qs.append(q)
            cur = sample_index(int_weights(q), u_draft[j])
        toks.append(cur)
    lgs = np.stack(lgs) if lgs else np.zeros((0, dec.shape.vocab))
    return toks, np.stack(hs), lgs, (np.stack(qs) if qs else None)


def top_children(row, c):
    """The ``c`` highest-logit token ids of a row, best first, ties to the lower id."""
    z = np.asarray(row, dtype=np.float64)
    order = np.lexsort((np.arange(z.shape[0]), -z))
    return [int(x) for x in order[:c]]


def draft_tree(dec, cache, s, t0, parents):
    """Layer-skip draft of a level-order token tree at committed length ``s``.

    The root is ``t0``; level by level, the nodes of the current level run
    layers [0, L) (node i in slot s + i at position s + depth(i), seeing the
    committed context, its ancestors and itself) and the shared LM head, and
    the children of node i take the best draft tokens of i's row in order:
    the k-th child (by node index) gets the k-th highest logit (FlashSpec page,
    lnrk.cn/news/47842, §2.2 and §6.2: a tree of candidates from the draft's
    top choices; self-speculative decoding page §2.1: the first L layers and
    the LM head are the draft).  A last pass runs layers [0, L) on the deepest
    level without the head so that every node has its layer-L state.
    Returns ``(tokens[n], h_L[n, d], draft_logits[n, V] (rows of the nodes
    that have children, else zero))``.
    """
    L = dec.shape.exit_layer
    n = len(parents)
    depth = tree_depths(parents)
    vis_all = tree_visibility(s, parents)
    tokens = [0] * n
    tokens[0] = int(t0)
    hs = np.zeros((n, dec.shape.d_model))
    lgs = np.zeros((n, dec.shape.vocab))
    for lev in range(int(depth.max()) + 1):
        nodes = [i for i in range(n) if depth[i] == lev]
        h = dec.embed([tokens[i] for i in nodes])
        h = dec.run_layers(h, 0, L, [s + lev] * len(nodes), [s + i for i in nodes], [vis_all[i] for i in nodes],
                           cache)
        for r, i in enumerate(nodes):
            hs[i] = h[r]
        kids = {i: [c for c in range(n) if parents[c] == i] for i in nodes}
        if not any(kids.values()):
            break
        lg = dec.logits(h)
        for r, i in enumerate(nodes):
            if kids[i]:
                lgs[i] = lg[r]
                for c, tok in zip(kids[i], top_children(lg[r], len(kids[i]))):
                    tokens[c] = tok
    return tokens, hs, lgs


def tree_round_layerskip(dec, cache, t0, parents):
    """One greedy round of the layer-skip tree: draft_tree, layers [L, N) over
    every node (tree mask), greedy tree acceptance, commit of the path.
    Returns ``(emitted, depth, path, next, tokens, target_logits)``."""
    s = cache.length
    L = dec.shape.exit_layer
    tokens, hL, _ = draft_tree(dec, cache, s, t0, parents)
    logits = verify(dec, cache, s, hL, L, parents=parents)
    depth, node, path, nxt = accept_greedy_tree(tokens, parents, logits)
    moves, new_len = commit_tree_moves(s, path)
    apply_moves(cache, moves)
    cache.length = new_len
    return [tokens[i] for i in path[1:]] + [nxt], depth, path, nxt, tokens, logits


def generate_greedy_tree_spec(dec, prompt, n_new, parents, max_ctx=None, log=None):
    """Greedy decoding by layer-skip tree rounds; equals :func:`generate_greedy_ar`."""
    n = len(parents)
    cache = dec.new_cache(max_ctx or (len(prompt) + n_new + n + 2))
    t0 = argmax_lowest(dec.prefill(cache, prompt))
    out = [t0]
    while len(out) < n_new:
        s = cache.length
        emitted, depth, _, t0, _, _ = tree_round_layerskip(dec, cache, t0, parents)
        out += emitted
        if log is not None:
            log.append((s, depth))
    return out[:n_new]


def child_count(row, width, mass):
    """Children of a node under the dynamic tree width (FlashSpec page,
    lnrk.cn/news/47842, §6.2: the draft judges its own confidence; a node it
    is sure of is not widened, an unsure one gets more branches).

    Reading: the children are the node's best draft tokens, best first, and
    their number is the fewest whose draft probabilities (softmax of the
    draft logits at temperature 1, float64) add up to at least ``mass``, at
    least one and at most ``width``.  ``mass`` <= 0 gives one child (a
    chain), ``mass`` > 1 always ``width`` (the static tree).
    """
    z = np.asarray(row, dtype=np.float64)
    e = np.exp(z - z.max())
    p = e / e.sum()
    cum = 0.0
    for c, x in enumerate(top_children(row, width), start=1):
        cum += p[x]
        if cum >= mass:
            return c
    return width


def draft_tree_dynamic(dec, cache, s, t0, branching, mass):
    """Layer-skip draft of a tree whose width follows the draft's confidence.

    As :func:`draft_tree`, level by level, but node i of level l gets
    ``child_count(draft logits of i, branching[l], mass)`` children, the
    best draft tokens of its row in order; children are numbered in level
    order (the children of earlier nodes first).  ``branching`` bounds the
    tree: at most branching[l] children a node of level l, depth
    len(branching).  Returns ``(tokens[n], parents[n], h_L[n, d],
    draft_logits[n, V] (rows of the nodes with children, else zero))``.
    """
    L = dec.shape.exit_layer
    tokens, parents = [int(t0)], [-1]
    hs, lgs = {}, {}
    level = [0]
    for lev in range(len(branching) + 1):
        vis_all = tree_visibility(s, parents)
        h = dec.embed([tokens[i] for i in level])
        h = dec.run_layers(h, 0, L, [s + lev] * len(level), [s + i for i in level], [vis_all[i] for i in level],
                           cache)
        for r, i in enumerate(level):
            hs[i] = h[r]
        if lev == len(branching):
            break
        lg = dec.logits(h)
        nxt = []
        for r, i in enumerate(level):
            lgs[i] = lg[r]
            for tok in top_children(lg[r], child_count(lg[r], branching[lev], mass)):
                tokens.append(tok)
                parents.append(i)
                nxt.append(len(tokens) - 1)
        level = nxt
    n = len(tokens)
    h_l = np.stack([hs[i] for i in range(n)])
    logit_rows = np.zeros((n, dec.shape.vocab))
    for i, row in lgs.items():
        logit_rows[i] = row
    return tokens, parents, h_l, logit_rows


def tree_round_dynamic(dec, cache, t0, branching, mass):
    """One greedy round of the layer-skip tree of dynamic width: the draft
    tree, layers [L, N) over its nodes (tree mask), greedy tree acceptance,
    commit of the path.  Returns ``(emitted, depth, path, next, tokens,
    parents, target_logits)``."""
    s = cache.length
    L = dec.shape.exit_layer
    tokens, parents, hL, _ = draft_tree_dynamic(dec, cache, s, t0, branching, mass)
    logits = verify(dec, cache, s, hL, L, parents=parents)
    depth, node, path, nxt = accept_greedy_tree(tokens, parents, logits)
    moves, new_len = commit_tree_moves(s, path)
    apply_moves(cache, moves)
    cache.length = new_len
    return [tokens[i] for i in path[1:]] + [nxt], depth, path, nxt, tokens, parents, logits


def generate_greedy_dynamic_tree_spec(dec, prompt, n_new, branching, mass, max_ctx=None, log=None):
    """Greedy decoding by dynamic-width tree rounds; equals :func:`generate_greedy_ar`."""
    n_max = sum(int(np.prod(branching[:l])) for l in range(len(branching) + 1))
    cache = dec.new_cache(max_ctx or (len(prompt) + n_new + n_max + 2))
    t0 = argmax_lowest(dec.prefill(cache, prompt))
    out = [t0]
    while len(out) < n_new:
        s = cache.length
        emitted, depth, _, t0, tokens, _, _ = tree_round_dynamic(dec, cache, t0, branching, mass)
        out += emitted
        if log is not None:
            log.append((s, depth, len(tokens)))
    return out[:n_new]


def chain_visibility(s, T):
    return [np.arange(0, s + t + 1) for t in range(T)]


def tree_visibility(s, parents):
    vis = []
    for i in range(len(parents)):
        anc = [i]
        while parents[anc[-1]] >= 0:
            anc.append(int(parents[anc[-1]]))
        vis.append(np.concatenate([np.arange(0, s), s + np.array(sorted(anc))]))
    return vis


def verify(dec, cache, s, h_in, lo, parents=None):
    """Layers ``[lo, N)`` over rows ``h_in [T, d]`` in slots ``s .. s+T-1``.

    Chain when ``parents`` is None (positions s+t, causal), else a
    level-order tree (positions s + depth, ancestor-only visibility).
    Returns the target logits ``[T, V]``.
    """
    T = h_in.shape[0]
    slots = s + np.arange(T)
    if parents is None:
        pos, vis = slots, chain_visibility(s, T)
    else:
        pos, vis = s + tree_depths(parents), tree_visibility(s, parents)
    h = dec.run_layers(np.asarray(h_in, dtype=np.float64), lo, dec.n_layers, pos, slots, vis, cache)
    return dec.logits(h)


def decode_step(dec, cache, token):
    """One plain autoregressive step: all layers on ``token`` at the committed end."""
    s = cache.length
    h = dec.run_layers(dec.embed([token]), 0, dec.n_layers, [s], [s], [np.arange(0, s + 1)], cache)
    cache.length = s + 1
    return dec.logits(h)[0]


def generate_greedy_ar(dec, prompt, n_new, max_ctx=None):
    """Plain greedy decoding: the first ``n_new`` tokens after ``prompt``."""
    cache = dec.new_cache(max_ctx or (len(prompt) + n_new + 1))
    out = [argmax_lowest(dec.prefill(cache, prompt))]
    while len(out) < n_new:
        out.append(argmax_lowest(decode_step(dec, cache, out[-1])))
    return out


def spec_round_greedy(dec, cache, t0, k):
    """One greedy chain round; returns ``(emitted, a, next, target_logits)``."""
    s = cache.length
    L = dec.shape.exit_layer
    d, hL, _, _ = draft(dec, cache, s, t0, k)
    logits = verify(dec, cache, s, hL, L)
    a, nxt = accept_greedy_chain(d, logits)
    cache.length = commit_chain(s, a)
    return list(d[:a]) + [nxt], a, nxt, logits


def exit_layer_for_context(s, table):
    """Exit layer for a committed context of ``s`` slots under a caller's table.

    The self-speculative decoding page (m.lqnn.cn/news/278124, §5.3) asks for
    a shallower exit on short contexts and a deeper one on long contexts, to
    hold the acceptance rate as the draft's attention grows; it gives the
    direction, not the numbers.  ``table`` holds (min_context, exit_layer)
    pairs in increasing min_context, the first at 0: the pair with the
    largest min_context <= s applies.
    """
    L = None
    for lo, layer in table:
        if s >= lo:
            L = int(layer)
    return L


def with_exit_layer(dec, L):
    """The same decoder and weights with draft exit layer ``L``."""
    return type(dec)(dataclasses.replace(dec.shape, exit_layer=int(L)), dec.w)


def generate_greedy_spec_context_exit(dec, prompt, n_new, k, table, max_ctx=None, log=None):
    """Greedy self-speculative decoding whose exit layer follows the committed
    context length: before each round's draft, L = exit_layer_for_context(s,
    table).  A round writes every layer of its rows (layers [0, L) in the
    draft, [L, N) in the verify), so the next round at another L finds its
    whole context; equals :func:`generate_greedy_ar` for any table.  ``log``
    receives ``(s, L, a)`` per round; returns ``(tokens, cache)``.
    """
    cache = dec.new_cache(max_ctx or (len(prompt) + n_new + k + 2))
    t0 = argmax_lowest(dec.prefill(cache, prompt))
    out = [t0]
    while len(out) < n_new:
        s = cache.length
        L = exit_layer_for_context(s, table)
        emitted, a, t0, _ = spec_round_greedy(with_exit_layer(dec, L), cache, t0, k)
        out += emitted
        if log is not None:
            log.append((s, L, a))
    return out[:n_new], cache


def spec_round_sampling(dec, cache, t0, k, temp, top_p, u_draft, u):
    """One sampling chain round at temperature ``temp``.

    The draft samples d_{j+1} from q_j = softmax(draft logits / temp) with
    ``u_draft[j]``; the target rows become p_j = softmax(target logits / temp),
    truncated to their top-p nucleus; rejection sampling with ``u[0..k]``
    decides (self-speculative decoding page, §2.4, §3.4, §4.3).  Returns
    ``(emitted, a, next, draft_tokens, q, p, target_logits)`` and commits.
    """
    s = cache.length
    L = dec.shape.exit_layer
    d, hL, _, q = draft(dec, cache, s, t0, k, temp=temp, u_draft=u_draft)
    logits = verify(dec, cache, s, hL, L)
    p = np.stack([top_p_filter(r, top_p) for r in probs_at(logits, temp)])
    a, nxt = accept_sampling_chain(p, q, d, u)
    cache.length = commit_chain(s, a)
    return list(d[:a]) + [nxt], a, nxt, d, q, p, logits


def generate_greedy_spec(dec, prompt, n_new, k, max_ctx=None, log=None):
    """Greedy self-speculative decoding; equals :func:`generate_greedy_ar`.

    ``log`` (a list) receives ``(s, a)`` per round.
    """
    cache = dec.new_cache(max_ctx or (len(prompt) + n_new + k + 2))
    t0 = argmax_lowest(dec.prefill(cache, prompt))
    out = [t0]
    while len(out) < n_new:
        s = cache.length
        emitted, a, t0, _ = spec_round_greedy(dec, cache, t0, k)
        out += emitted
        if log is not None:
            log.append((s, a))
    return out[:n_new]


def tree_round_greedy(dec, cache, tokens, parents):
    """Greedy tree round over level-order ``tokens`` (all layers from the embedding).

    Returns ``(depth, node, path, next, logits)`` and commits the path.
    """
    s = cache.length
    logits = verify(dec, cache, s, dec.embed(tokens), 0, parents)
    depth, node, path, nxt = accept_greedy_tree(tokens, parents, logits)
    moves, new_len = commit_tree_moves(s, path)
    apply_moves(cache, moves)
    cache.length = new_len
    return depth, node, path, nxt, logits
