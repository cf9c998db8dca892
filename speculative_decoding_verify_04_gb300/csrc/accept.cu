// Greedy acceptance (unfused form), KV commit and draft-length scheduling
// kernels.  Rejection-sampling acceptance shares the row machinery of the
// sampling kernels and lives beside them.
#include <algorithm>

#include "model.cuh"
#include "stats.cuh"

namespace spec {

// Unfused greedy acceptance: per sequence, row summaries from the logits then
// the chain or tree rule.  The tree (parent and depth of each node) travels in
// the kernel parameters.
struct TreeArrays { int parent[kMaxSeqRows]; int depth[kMaxSeqRows]; };

__global__ void __launch_bounds__(256)
accept_greedy_kernel(const float* __restrict__ logits, const int* __restrict__ tokens, int n_rows, int V,
                     int tree, TreeArrays ta, int* acc_len, int* next_tok, int* path) {
    __shared__ spec_row_stats rs[kMaxSeqRows];
    __shared__ int par[kMaxSeqRows], dep[kMaxSeqRows];
    const int b = blockIdx.x, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x < kMaxSeqRows) { par[threadIdx.x] = ta.parent[threadIdx.x]; dep[threadIdx.x] = ta.depth[threadIdx.x]; }
    for (int j = w; j < n_rows; j += 8) {
        const float* row = logits + ((size_t)b * n_rows + j) * V;
        spec_row_stats s = stat_empty();
        for (int x = lane; x < V; x += 32) {
            spec_row_stats one;
            one.top1 = row[x]; one.top2 = -INFINITY; one.sum_exp = 1.f; one.argmax = x;
            stat_merge(s, one);
        }
        s = stat_warp_merge(s);
        if (lane == 0) rs[j] = s;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int* tok = tokens + (size_t)b * n_rows;
        int* pth = path ? path + (size_t)b * kMaxSeqRows : nullptr;
        if (tree) accept_tree_one(rs, 0, n_rows, tok, par, dep, acc_len + b, next_tok + b, pth);
        else accept_chain_one(rs, 0, n_rows, tok, acc_len + b, next_tok + b, pth);
    }
}

// Tree commit: rows of depth 1..a move from slot s+path[d] to slot s+d, in
// increasing depth (a move never overwrites a later move's source).  One CTA
// per (layer, kv head, sequence); lengths are updated by a second launch.
template <typename KT>
__global__ void commit_tree_kernel(KT* kc, KT* vc, const int* len, const int* acc_len, const int* path,
                                   int path_stride, int n_kv_heads, KVPages kvp, int kv_ctx, int hd, int* err) {
    pdl_wait();
    pdl_trigger();
    const int lh = blockIdx.x, b = blockIdx.y;
    const int layer = lh / n_kv_heads, kvh = lh % n_kv_heads;
    const int s = len[b], a = acc_len[b];
    for (int d = 1; d <= a; ++d) {
        const int src = s + path[(size_t)b * path_stride + d], dst = s + d;
        if (src >= kv_ctx || dst >= kv_ctx) { if (threadIdx.x == 0) dev_error(err, SPEC_DEVERR_CAPACITY); return; }
        const long long rs = kv_row(kvp, n_kv_heads, layer, b, kvh, src), rd = kv_row(kvp, n_kv_heads, layer, b, kvh, dst);
        if (rs < 0 || rd < 0) { if (threadIdx.x == 0) dev_error(err, SPEC_DEVERR_CAPACITY); return; }
        KT kv0 = KT(), vv0 = KT();
        const int i = threadIdx.x;
        if (i < hd) { kv0 = kc[(size_t)rs * hd + i]; vv0 = vc[(size_t)rs * hd + i]; }
        __syncthreads();
        if (i < hd) { kc[(size_t)rd * hd + i] = kv0; vc[(size_t)rd * hd + i] = vv0; }
        __syncthreads();
    }
}

// Paged caches.  One thread walks every sequence in order, so which page a
// block of slots gets is deterministic.
//   ensure: before a call writes slots, every block of slots below end[b]
//   (len[b] + n[b] when relative, else n[b]) holds a page, popped from the free
//   stack; an empty stack sets the capacity error.
//   release (page-granular rollback, "self-speculative decoding" page section
//   3.3): the blocks past the committed length give their pages back.
struct PageNeed { int batch; int relative; int n[kMaxPlanBatch]; };

__global__ void ensure_pages_kernel(const int* __restrict__ len, PageNeed need, int* table, int page, int max_pages,
                                    const int* free_pages, int* free_top, int* err) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int top = *free_top;
    for (int b = 0; b < need.batch; ++b) {
        const int end = need.relative ? len[b] + need.n[b] : need.n[b];
        const int blocks = min(max_pages, (end + page - 1) / page);
        if ((end + page - 1) / page > max_pages) dev_error(err, SPEC_DEVERR_CAPACITY);
        for (int p = 0; p < blocks; ++p) {
            int* e = table + (size_t)b * max_pages + p;
            if (*e >= 0) continue;
            if (top == 0) { dev_error(err, SPEC_DEVERR_CAPACITY); break; }
            *e = free_pages[--top];
        }
    }
    *free_top = top;
}

__global__ void release_pages_kernel(const int* __restrict__ len, int batch, int* table, int page, int max_pages,
                                     int* free_pages, int* free_top, int n_pages) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int top = *free_top;
    for (int b = 0; b < batch; ++b) {
        const int keep = (len[b] + page - 1) / page;
        for (int p = max_pages - 1; p >= keep; --p) {
            int* e = table + (size_t)b * max_pages + p;
            if (*e < 0) continue;
            if (top < n_pages) free_pages[top++] = *e;
            *e = -1;
        }
    }
    *free_top = top;
}

__global__ void commit_len_kernel(int* len, const int* acc_len, int batch, int kv_ctx, int* err) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int n = len[b] + acc_len[b] + 1;
    if (n > kv_ctx) dev_error(err, SPEC_DEVERR_CAPACITY);
    len[b] = min(n, kv_ctx);
}

// Draft-length schedule: float64, explicit rounding (no contraction), in the
// order written in the header.
struct SchedParams {
    int batch;
    int row0[kMaxPlanBatch];
    int n_rows[kMaxPlanBatch];
    int min_k, max_k;
    double low, high, decay;
    int first_reject_min;
};

__global__ void schedule_kernel(const double* __restrict__ probs, const int* __restrict__ acc_len, double* ema,
                                SchedParams sp, int* k_next, double* conf_out) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= sp.batch) return;
    const int n = sp.n_rows[b], k = n - 1, r0 = sp.row0[b];
    const double acc = __ddiv_rn((double)acc_len[b], (double)k);
    const double e = __dadd_rn(__dmul_rn(sp.decay, ema[b]), __dmul_rn(__dsub_rn(1.0, sp.decay), acc));
    double s1 = 0.0, sg = 0.0;
    for (int i = 0; i < n; ++i) {
        const double p1 = probs[2 * (size_t)(r0 + i)], p2 = probs[2 * (size_t)(r0 + i) + 1];
        s1 = __dadd_rn(s1, p1);
        sg = __dadd_rn(sg, __dsub_rn(p1, p2));
    }
    const double avg1 = __ddiv_rn(s1, (double)n), avgg = __ddiv_rn(sg, (double)n);
    const double gap = fmin(__dmul_rn(avgg, 5.0), 1.0);
    const double c = __dadd_rn(__dadd_rn(__dmul_rn(0.4, avg1), __dmul_rn(0.3, gap)), __dmul_rn(0.3, e));
    const double lin = __dadd_rn((double)sp.min_k,
                                 __ddiv_rn(__dmul_rn((double)(sp.max_k - sp.min_k), __dsub_rn(c, sp.low)),
                                           __dsub_rn(sp.high, sp.low)));
    long long kk = (long long)lin;            // truncation toward zero
    kk = kk < sp.min_k ? sp.min_k : (kk > sp.max_k ? sp.max_k : kk);
    if (sp.first_reject_min && acc_len[b] == 0) kk = sp.min_k;
    ema[b] = e;
    k_next[b] = (int)kk;
    if (conf_out) conf_out[b] = c;
}

// Additive schedule: one thread per sequence; its window lives in `state` as
// [count, next slot, kept[W], drafted[W]].
__global__ void aimd_kernel(const int* __restrict__ acc_len, const int* __restrict__ k_cur, int* state, int batch,
                            spec_aimd_schedule sch, int* k_next) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int W = sch.window;
    int* st = state + (size_t)b * (2 * W + 2);
    int count = st[0], slot = st[1];
    const int k = k_cur[b];
    st[2 + slot] = acc_len[b];
    st[2 + W + slot] = k;
    slot = slot + 1 == W ? 0 : slot + 1;
    count = count < W ? count + 1 : W;
    st[0] = count;
    st[1] = slot;
    long long kept = 0, drafted = 0;
    for (int i = 0; i < count; ++i) {
        kept += st[2 + i];
        drafted += st[2 + W + i];
    }
    int kn = k;
    if (kept * sch.up_den > (long long)sch.up_num * drafted) kn = k + 1;
    else if (kept * sch.down_den < (long long)sch.down_num * drafted) kn = k - 1;
    k_next[b] = kn < sch.min_k ? sch.min_k : (kn > sch.max_k ? sch.max_k : kn);
}

__global__ void decay_kernel(const int* __restrict__ generated, const int* __restrict__ total, int batch, int k_max,
                             int* k_next) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    const int T = total[b];
    if (T < 1) { k_next[b] = 1; return; }
    const double x = __dmul_rn((double)k_max, __dsub_rn(1.0, __ddiv_rn((double)generated[b], (double)T)));
    const double r = rint(x);                       // nearest, ties to even
    k_next[b] = r < 1.0 ? 1 : (int)r;
}

__global__ void row_probs_kernel(const spec_row_stats* __restrict__ st, int rows, double* out) {
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= rows) return;
    const spec_row_stats s = st[r];
    const double S = (double)s.sum_exp;
    out[2 * (size_t)r] = __ddiv_rn(1.0, S);
    out[2 * (size_t)r + 1] = __ddiv_rn(exp((double)s.top2 - (double)s.top1), S);
}

int kv_ensure_pages(spec_kv* kv, int batch, const int* n, bool relative, cudaStream_t st) {
    if (!kv->paged) return SPEC_OK;
    if (batch > kMaxPlanBatch) return set_error(SPEC_ERR_CAPACITY, "paged cache: too many sequences in one call");
    PageNeed need{};
    need.batch = batch;
    need.relative = relative ? 1 : 0;
    for (int b = 0; b < batch; ++b) need.n[b] = n[b];
    spec_model* m = kv->m;
    launch_k(m->pdl, ensure_pages_kernel, dim3(1), dim3(32), 0, st, (const int*)kv->len, need, kv->table, kv->page,
             kv->max_pages, (const int*)kv->free_pages, kv->free_top, m->err);
    ++m->launches;
    return check_cuda(cudaGetLastError(), "page allocation launch");
}

int kv_release_pages(spec_kv* kv, int batch, cudaStream_t st) {
    if (!kv->paged) return SPEC_OK;
    spec_model* m = kv->m;
    launch_k(m->pdl, release_pages_kernel, dim3(1), dim3(32), 0, st, (const int*)kv->len, batch, kv->table, kv->page,
             kv->max_pages, kv->free_pages, kv->free_top, kv->n_pages);
    ++m->launches;
    return check_cuda(cudaGetLastError(), "page release launch");
}

}  // namespace spec

using namespace spec;

extern "C" int spec_accept_greedy(const float* logits, const int32_t* tokens, const int32_t* tree_parent,
                                  int32_t batch, int32_t n_rows, int32_t vocab, int32_t* acc_len,
                                  int32_t* next_tok, int32_t* path, void* stream) {
    if (!logits || !tokens || !acc_len || !next_tok) return set_error(SPEC_ERR_ARG, "spec_accept_greedy: null pointer");
    if (batch <= 0 || n_rows < 1 || n_rows > kMaxSeqRows || vocab <= 0)
        return set_error(SPEC_ERR_ARG, "spec_accept_greedy: bad sizes");
    if (tree_parent && !path) return set_error(SPEC_ERR_ARG, "spec_accept_greedy: tree mode needs path");
    TreeArrays ta{};
    if (tree_parent) {
        if (tree_parent[0] != -1) return set_error(SPEC_ERR_ARG, "tree_parent[0] must be -1");
        ta.parent[0] = -1;
        for (int i = 1; i < n_rows; ++i) {
            if (tree_parent[i] < 0 || tree_parent[i] >= i) return set_error(SPEC_ERR_ARG, "tree_parent[i] must be in [0, i)");
            ta.parent[i] = tree_parent[i];
            ta.depth[i] = ta.depth[tree_parent[i]] + 1;
        }
    }
    accept_greedy_kernel<<<batch, 256, 0, (cudaStream_t)stream>>>(logits, tokens, n_rows, vocab, tree_parent ? 1 : 0,
                                                                  ta, acc_len, next_tok, path);
    return check_cuda(cudaGetLastError(), "spec_accept_greedy launch");
}

extern "C" int kv_commit(spec_kv* kv, int32_t batch, const int32_t* acc_len, const int32_t* path,
                         int32_t path_stride, void* stream) {
    if (!kv || !acc_len) return set_error(SPEC_ERR_ARG, "kv_commit: null pointer");
    if (batch <= 0 || batch > kv->batch) return set_error(SPEC_ERR_ARG, "kv_commit: bad batch");
    spec_model* m = kv->m;
    cudaStream_t st = (cudaStream_t)stream;
    if (path) {
        if (path_stride < 1) return set_error(SPEC_ERR_ARG, "kv_commit: bad path stride");
        dim3 grid(m->cfg.n_layers * m->cfg.n_kv_heads, batch);
        const int threads = m->cfg.head_dim;
        if (m->bf16)
            launch_k(m->pdl, commit_tree_kernel<__nv_bfloat16>, grid, dim3(threads), 0, st,
                (__nv_bfloat16*)kv->k, (__nv_bfloat16*)kv->v, kv->len, acc_len, path, path_stride,
                m->cfg.n_kv_heads, kv->pages(), kv->max_ctx, m->cfg.head_dim, m->err);
        else
            launch_k(m->pdl, commit_tree_kernel<float>, grid, dim3(threads), 0, st, (float*)kv->k, (float*)kv->v,
                     kv->len, acc_len, path, path_stride, m->cfg.n_kv_heads, kv->pages(), kv->max_ctx,
                     m->cfg.head_dim, m->err);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return check_cuda(e, "kv_commit tree launch");
    }
    launch_k(m->pdl, commit_len_kernel, dim3((batch + 127) / 128), dim3(128), 0, st, kv->len, acc_len, batch, kv->max_ctx,
             m->err);
    m->launches += path ? 2 : 1;
    const int rc = check_cuda(cudaGetLastError(), "kv_commit launch");
    if (rc) return rc;
    return kv->paged ? kv_release_pages(kv, batch, st) : SPEC_OK;
}

extern "C" int spec_row_probs(const spec_row_stats* stats, int32_t rows, double* out, void* stream) {
    if (!stats || !out || rows <= 0) return set_error(SPEC_ERR_ARG, "spec_row_probs: bad arguments");
    row_probs_kernel<<<(rows + 127) / 128, 128, 0, (cudaStream_t)stream>>>(stats, rows, out);
    return check_cuda(cudaGetLastError(), "spec_row_probs launch");
}

extern "C" int spec_schedule_k(const double* top_probs, const int32_t* n_rows, const int32_t* acc_len, double* ema,
                               int32_t batch, const spec_k_schedule* sch, int32_t* k_next, double* conf,
                               void* stream) {
    if (!top_probs || !n_rows || !acc_len || !ema || !sch || !k_next)
        return set_error(SPEC_ERR_ARG, "spec_schedule_k: null pointer");
    if (batch <= 0 || batch > kMaxPlanBatch) return set_error(SPEC_ERR_ARG, "spec_schedule_k: bad batch");
    if (sch->min_k < 1 || sch->max_k < sch->min_k || !(sch->high > sch->low))
        return set_error(SPEC_ERR_ARG, "spec_schedule_k: bad schedule");
    SchedParams sp{};
    sp.batch = batch;
    int r = 0;
    for (int b = 0; b < batch; ++b) {
        if (n_rows[b] < 2) return set_error(SPEC_ERR_ARG, "spec_schedule_k: n_rows must be >= 2 (k >= 1)");
        sp.row0[b] = r;
        sp.n_rows[b] = n_rows[b];
        r += n_rows[b];
    }
    sp.min_k = sch->min_k; sp.max_k = sch->max_k;
    sp.low = sch->low; sp.high = sch->high; sp.decay = sch->decay;
    sp.first_reject_min = sch->first_reject_min;
    schedule_kernel<<<(batch + 127) / 128, 128, 0, (cudaStream_t)stream>>>(top_probs, acc_len, ema, sp, k_next, conf);
    return check_cuda(cudaGetLastError(), "spec_schedule_k launch");
}

extern "C" int spec_schedule_aimd(const int32_t* acc_len, const int32_t* k_cur, int32_t* state, int32_t batch,
                                  const spec_aimd_schedule* sch, int32_t* k_next, void* stream) {
    if (!acc_len || !k_cur || !state || !sch || !k_next) return set_error(SPEC_ERR_ARG, "spec_schedule_aimd: null pointer");
    if (batch <= 0) return set_error(SPEC_ERR_ARG, "spec_schedule_aimd: bad batch");
    if (sch->window < 1 || sch->window > 256 || sch->min_k < 1 || sch->max_k < sch->min_k || sch->up_den <= 0 ||
        sch->down_den <= 0)
        return set_error(SPEC_ERR_ARG, "spec_schedule_aimd: bad schedule");
    aimd_kernel<<<(batch + 127) / 128, 128, 0, (cudaStream_t)stream>>>(acc_len, k_cur, state, batch, *sch, k_next);
    return check_cuda(cudaGetLastError(), "spec_schedule_aimd launch");
}

extern "C" int spec_schedule_decay(const int32_t* generated, const int32_t* total, int32_t batch, int32_t k_max,
                                   int32_t* k_next, void* stream) {
    if (!generated || !total || !k_next) return set_error(SPEC_ERR_ARG, "spec_schedule_decay: null pointer");
    if (batch <= 0 || k_max < 1) return set_error(SPEC_ERR_ARG, "spec_schedule_decay: bad sizes");
    decay_kernel<<<(batch + 127) / 128, 128, 0, (cudaStream_t)stream>>>(generated, total, batch, k_max, k_next);
    return check_cuda(cudaGetLastError(), "spec_schedule_decay launch");
}
