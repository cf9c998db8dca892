// Row statistics of logits rows and the greedy acceptance rules applied to them.
//
// A row summary holds the largest logit (ties to the lowest index), the second
// largest value and sum(exp(l - top1)).  Summaries of disjoint index ranges merge
// exactly for top1/argmax/top2 and with one rescale for the sum, so per-tile
// summaries of the LM-head epilogue combine into the row's summary in any fixed
// order.
#pragma once

#include <cmath>
#include "model.cuh"

namespace spec {

SPEC_DEV spec_row_stats stat_empty() {
    spec_row_stats s;
    s.top1 = -INFINITY;
    s.top2 = -INFINITY;
    s.sum_exp = 0.f;
    s.argmax = 0x7fffffff;
    return s;
}

SPEC_DEV bool stat_wins(const spec_row_stats& a, const spec_row_stats& b) {
    return a.top1 > b.top1 || (a.top1 == b.top1 && a.argmax < b.argmax);
}

// a <- merge(a, b); commutative (ties broken by index).
SPEC_DEV void stat_merge(spec_row_stats& a, const spec_row_stats& b) {
    if (b.sum_exp == 0.f) return;
    if (a.sum_exp == 0.f) { a = b; return; }
    if (stat_wins(a, b)) {
        a.top2 = fmaxf(a.top2, b.top1);
        a.sum_exp = a.sum_exp + b.sum_exp * expf(b.top1 - a.top1);
    } else {
        const float t2 = fmaxf(b.top2, a.top1);
        a.sum_exp = b.sum_exp + a.sum_exp * expf(a.top1 - b.top1);
        a.top1 = b.top1;
        a.argmax = b.argmax;
        a.top2 = t2;
    }
}

SPEC_DEV spec_row_stats stat_shfl_xor(const spec_row_stats& s, int o) {
    spec_row_stats r;
    r.top1 = __shfl_xor_sync(0xffffffffu, s.top1, o);
    r.top2 = __shfl_xor_sync(0xffffffffu, s.top2, o);
    r.sum_exp = __shfl_xor_sync(0xffffffffu, s.sum_exp, o);
    r.argmax = __shfl_xor_sync(0xffffffffu, s.argmax, o);
    return r;
}

// Butterfly merge across the warp: every lane ends with the same summary.
SPEC_DEV spec_row_stats stat_warp_merge(spec_row_stats s) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        spec_row_stats t = stat_shfl_xor(s, o);
        // merge in a lane-independent order so all lanes compute the same bits
        spec_row_stats lo = (threadIdx.x & o) ? t : s;
        spec_row_stats hi = (threadIdx.x & o) ? s : t;
        stat_merge(lo, hi);
        s = lo;
    }
    return s;
}

// Greedy chain acceptance of one sequence: rows r0 .. r0+n-1 with tokens
// tok[0..n-1] (tok[0] = t0, tok[j] = d_j).  a = leading draft tokens equal to
// the previous row's argmax; next = argmax of row a.
SPEC_DEV void accept_chain_one(const spec_row_stats* rs, int r0, int n, const int* tok,
                               int* acc_len, int* next_tok, int* path) {
    int a = 0;
    while (a < n - 1 && tok[a + 1] == rs[r0 + a].argmax) ++a;
    *acc_len = a;
    *next_tok = rs[r0 + a].argmax;
    if (path)
        for (int d = 0; d <= a; ++d) path[d] = d;
}

// Greedy tree acceptance: node i (level order, parent[i] < i) is accepted when
// its parent is and its token equals the parent's argmax; the deepest accepted
// node wins, ties to the lowest index.  path = root .. node.
SPEC_DEV void accept_tree_one(const spec_row_stats* rs, int r0, int n, const int* tok,
                              const int* parent, const int* depth,
                              int* acc_len, int* next_tok, int* path) {
    unsigned long long ok = 1ull;     // bit i: node i accepted (n <= 64)
    int best = 0;
    for (int i = 1; i < n; ++i) {
        const int par = parent[i];
        if (((ok >> par) & 1ull) && tok[i] == rs[r0 + par].argmax) {
            ok |= 1ull << i;
            if (depth[i] > depth[best]) best = i;
        }
    }
    const int a = depth[best];
    *acc_len = a;
    *next_tok = rs[r0 + best].argmax;
    if (path) {
        int node = best;
        for (int d = a; d >= 0; --d) { path[d] = node; node = parent[node]; }
    }
}

}  // namespace spec
