// C ABI entry points: model and KV lifecycle, row plans, the forward passes
// behind spec_prefill / spec_draft / spec_verify.
//
// Layer-skip self-drafting ("self-speculative decoding" page,
// m.lqnn.cn/news/278124, sections 2.1, 3.3, 4.2, 4.3): one KV cache serves the
// draft (layers [0, L)) and the verifier (layers [L, N)); the draft's pass over
// a row writes that row's first-L KV and leaves its layer-L residual state,
// which the verifier continues from.  Position ids are the committed length
// plus the row's offset (chain) or depth (tree).
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "model.cuh"
#include "stats.cuh"

namespace spec {

static thread_local std::string g_err;

int set_error(int code, const std::string& msg) {
    g_err = msg;
    return code;
}

int check_cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return SPEC_OK;
    g_err = std::string(what) + ": " + cudaGetErrorString(e);
    return SPEC_ERR_CUDA;
}

int prof_start(spec_model* m, cudaStream_t st) {
    if (!m->prof_on) return -1;
    const size_t i = m->prof_n;
    if (2 * i + 2 > m->prof_ev.size()) {
        cudaEvent_t a, b;
        if (cudaEventCreate(&a) != cudaSuccess) return -1;
        if (cudaEventCreate(&b) != cudaSuccess) { cudaEventDestroy(a); return -1; }
        m->prof_ev.push_back(a);
        m->prof_ev.push_back(b);
        m->prof_kind.push_back(0);
        m->prof_bytes.push_back(0.0);
    }
    cudaEventRecord(m->prof_ev[2 * i], st);
    m->prof_n = i + 1;
    return (int)i;
}

void prof_stop(spec_model* m, int slot, cudaStream_t st, int kind, double bytes) {
    if (slot < 0) return;
    cudaEventRecord(m->prof_ev[2 * slot + 1], st);
    m->prof_kind[slot] = kind;
    m->prof_bytes[slot] = bytes;
}

#define SPEC_CUDA(x, what) SPEC_TRY(check_cuda((x), what))

// ---------------------------------------------------------------------------
// small kernels
template <typename T>
__global__ void to_f32_kernel(const T* __restrict__ src, float* __restrict__ dst, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) dst[i] = to_f32<T>(src[i]);
}

// Tile-major copy of a bf16 GEMM weight [N][K] (N a multiple of 128, K of 64).
// Block (tile, k-block) -- 128 rows x 64 columns -- becomes 16 contiguous KB in
// the order the tensor-core operand takes in shared memory: row r at r * 128
// bytes, its 16-byte chunk c at chunk c ^ (r % 8) (the 128-byte swizzle).  One
// 16 KB bulk copy then fills a ring stage exactly as a swizzled 2-D tensor copy
// of the row-major matrix does, and a CTA's run of k-blocks is one sequential
// stream of HBM.  Indices in 16-byte chunks.
__global__ void tile_weights_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int N, int K) {
    const int cpr = K / 8;                       // chunks a row
    const int kbs = K / 64;                      // k-blocks a row
    const long long n_chunks = (long long)N * cpr;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_chunks;
         i += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(i / cpr), cc = (int)(i % cpr);
        const int tile = n >> 7, r = n & 127, kb = cc >> 3, c = cc & 7;
        dst[((long long)tile * kbs + kb) * 1024 + r * 8 + (c ^ (r & 7))] = src[i];
    }
}

// cos/sin of pos * theta^(-2i/hd), evaluated in float64 and rounded once
__global__ void rope_table_kernel(float* cs, float* sn, int max_pos, int half, double theta) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)max_pos * half) return;
    const int pos = (int)(idx / half), i = (int)(idx % half);
    const double inv = pow(theta, -2.0 * (double)i / (double)(2 * half));
    const double ang = (double)pos * inv;
    cs[idx] = (float)cos(ang);
    sn[idx] = (float)sin(ang);
}

struct PlanArgs {
    PlanParams p;
    int row0[kMaxPlanBatch];
    const int* dev_parent;   // tree mode: nullable device [batch][dev_stride] parents, one tree a sequence
    int dev_stride;
};

// Row plan.  mode 0 chain: row j of sequence b at slot / position s_b + j.
// mode 1 tree: slot s_b + j, position s_b + depth(j); one tree for the batch
// (the host's parents, written to the first kMaxSeqRows entries of the tree
// arrays) or, with dev_parent, one tree a sequence (parents read on the
// device; row j of sequence b writes entry b * kMaxSeqRows + j).  mode 2
// draft pass j: one row per sequence at slot / position s_b + j, seeing slots
// [0, s_b + j] (the earlier passes' rows count as context: base s_b + j,
// local row 0).
__global__ void plan_kernel(PlanArgs a, RowPlan plan, const int* __restrict__ len, int T, int* err) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    const PlanParams& p = a.p;
    // a draft pass sees the rows of the earlier passes as context: its base is s + j
    const int extra = (p.mode == 2) ? p.pass : 0;
    if (t < p.batch) {
        plan.seq_row0[t] = (p.mode == 2) ? t : a.row0[t];
        plan.seq_nrows[t] = (p.mode == 2) ? 1 : p.n_rows[t];
        plan.seq_base[t] = len[t] + extra;
    }
    if (t < kMaxSeqRows && !a.dev_parent) {
        plan.tree_parent[t] = p.parent[t];
        plan.tree_depth[t] = p.depth[t];
    }
    if (t >= T) return;
    int b, j;
    if (p.mode == 2) {
        b = t;
        j = 0;
    } else {
        int lo = 0, hi = p.batch - 1;      // last sequence with row0 <= t
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.row0[mid] <= t) lo = mid; else hi = mid - 1;
        }
        b = lo;
        j = t - a.row0[b];
    }
    const int s = len[b] + extra;
    plan.row_seq[t] = b;
    plan.row_local[t] = j;
    plan.row_slot[t] = s + j;
    int dep = j;
    if (p.mode == 1 && a.dev_parent) {
        // depth by walking to the root; a parent outside [0, x) is an error and reads as the root
        const int* par = a.dev_parent + (size_t)b * a.dev_stride;
        int pj = -1;
        dep = 0;
        for (int x = j; x > 0; ++dep) {
            int q = par[x];
            if (q < 0 || q >= x) { dev_error(err, SPEC_DEVERR_TREE); q = 0; }
            if (x == j) pj = q;
            x = q;
        }
        plan.tree_parent[(size_t)b * kMaxSeqRows + j] = pj;
        plan.tree_depth[(size_t)b * kMaxSeqRows + j] = dep;
    } else if (p.mode == 1) {
        dep = p.depth[j];
    }
    plan.row_pos[t] = s + dep;
}

// First residual rows of a forward: from the layer-L state (h_in) or the token
// embedding.  Writes h, the gained GEMM input and per-128-feature sums of h^2.
// One CTA per (row, 128-feature tile).
template <typename WT>
__global__ void __launch_bounds__(128)
prologue_kernel(const float* __restrict__ h_in, int h_stride, const int* __restrict__ tok, int tok_stride,
                int tok_col, const WT* __restrict__ embed, RowPlan plan, int d, int vocab,
                const float* __restrict__ gain, float* h, WT* x, size_t x_lo, float* ss, int ss_stride, int* err) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[4];
    const int r = blockIdx.x, tile = blockIdx.y, t = threadIdx.x;
    const int b = plan.row_seq[r], j = plan.row_local[r];
    const int n = tile * 128 + t;
    float v = 0.f;
    if (n < d) {
        if (h_in) {
            v = h_in[((size_t)b * h_stride + j) * d + n];
        } else {
            int token = tok[(size_t)b * tok_stride + tok_col + j];
            if (token < 0 || token >= vocab) {
                if (t == 0 && tile == 0) dev_error(err, SPEC_DEVERR_TOKEN);
                token = 0;
            }
            v = to_f32<WT>(embed[(size_t)token * d + n]);
        }
        h[(size_t)r * d + n] = v;
        store_act(x, (size_t)r * d + n, x_lo, v * gain[n]);
    }
    const float s = warp_sum(v * v);
    if ((t & 31) == 0) red[t >> 5] = s;
    __syncthreads();
    if (t == 0) ss[(size_t)tile * ss_stride + r] = (red[0] + red[1]) + (red[2] + red[3]);
}

__global__ void copy_rows_kernel(const float* __restrict__ h, float* __restrict__ dst, int rows, int d,
                                 int dst_row_stride, int dst_col) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x;
    for (int n = threadIdx.x; n < d; n += blockDim.x)
        dst[((size_t)r * dst_row_stride + dst_col) * d + n] = h[(size_t)r * d + n];
}

__global__ void set_col0_kernel(const int* __restrict__ t0, int* cand, int stride, int batch) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < batch) cand[(size_t)b * stride] = t0[b];
}

// Children of the nodes of one tree level take their parent's best draft
// tokens: the k-th child (by node index) the k-th highest logit, ties to the
// lower token id.  One CTA per (sequence, parent node); rounds of block-wide
// argmax that skip the ids already taken.
struct TreeKids {
    int start[kMaxSeqRows + 1];   // children of node i: kid[start[i] .. start[i+1])
    int kid[kMaxSeqRows];
};
constexpr int kMaxTreeKids = 16;

__global__ void __launch_bounds__(256)
tree_expand_kernel(const float* __restrict__ logits, int V, int rows_per_seq, int node0, TreeKids tk, int* tokens,
                   int n_nodes) {
    pdl_wait();
    pdl_trigger();
    __shared__ float s_v[8];
    __shared__ int s_i[8];
    __shared__ int taken[kMaxTreeKids];
    const int b = blockIdx.x, i = node0 + blockIdx.y, t = threadIdx.x, lane = t & 31, w = t >> 5;
    const int c0 = tk.start[i], nc = min(tk.start[i + 1] - c0, kMaxTreeKids);
    const float* row = logits + ((size_t)b * rows_per_seq + i) * V;
    for (int k = 0; k < nc; ++k) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        for (int x = t; x < V; x += 256) {
            bool skip = false;
            for (int q = 0; q < k; ++q) skip |= taken[q] == x;
            const float v = row[x];
            if (!skip && (v > bv || (v == bv && x < bi))) { bv = v; bi = x; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { s_v[w] = bv; s_i[w] = bi; }
        __syncthreads();
        if (t == 0) {
            float v = s_v[0];
            int id = s_i[0];
            for (int q = 1; q < 8; ++q)
                if (s_v[q] > v || (s_v[q] == v && s_i[q] < id)) { v = s_v[q]; id = s_i[q]; }
            taken[k] = id;
            tokens[(size_t)b * n_nodes + tk.kid[c0 + k]] = id;
        }
        __syncthreads();
    }
}

// Tree of dynamic width (FlashSpec page, lnrk.cn/news/47842, section 6.2: the
// draft widens the nodes it is unsure of).  Node i of level l gets the fewest
// of its best draft tokens whose draft probabilities (softmax of its draft
// logits, float32) reach `mass`, at least one and at most branching[l]; the
// children of a level are numbered in level order after the nodes so far.
// The tree lives in the caller's tokens / parents arrays ([batch][n_max]) and
// its node count in n_nodes[batch]; rows past the count are padding (token 0
// under the root) that the draft passes compute and nothing reads.  Per
// sequence the staging block holds the level being expanded (first node,
// node count), each node's child count and its best tokens.
constexpr int kTreeStage = 2 + kMaxSeqRows + kMaxSeqRows * kMaxTreeKids;

__global__ void tree_init_kernel(const int* __restrict__ t0, int* tokens, int* parents, int* n_nodes, int* stage,
                                 int batch, int n_max) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= batch * n_max) return;
    const int b = i / n_max, j = i % n_max;
    tokens[i] = j == 0 ? t0[b] : 0;
    parents[i] = j == 0 ? -1 : 0;
    if (j == 0) {
        n_nodes[b] = 1;
        stage[(size_t)b * kTreeStage + 0] = 0;
        stage[(size_t)b * kTreeStage + 1] = 1;
    }
}

// One CTA per (sequence, node of the level), one pass over the row: each
// thread keeps a running max and sum of exp and its own `width` best
// (logit, id) pairs, ties to the lower id; a block tournament of the threads'
// list heads then ranks the row's best tokens (the owner of id x is thread
// x % kWidthThreads), and the count stops at the first rank where their
// probability reaches `mass` (at most `width`).
constexpr int kWidthThreads = 256;

__global__ void __launch_bounds__(kWidthThreads)
tree_width_kernel(const float* __restrict__ logits, int V, int rows_per_seq, int width, float mass, int* stage) {
    pdl_wait();
    pdl_trigger();
    constexpr int NW = kWidthThreads / 32;
    __shared__ float s_v[NW], s_m[NW], s_s[NW];
    __shared__ int s_i[NW];
    const int b = blockIdx.x, y = blockIdx.y, t = threadIdx.x, lane = t & 31, w = t >> 5;
    int* st = stage + (size_t)b * kTreeStage;
    const int start = st[0], count = st[1];
    if (y >= count) return;
    const int i = start + y;
    const float* row = logits + ((size_t)b * rows_per_seq + i) * V;
    float tv[kMaxTreeKids];
    int ti[kMaxTreeKids];
    for (int q = 0; q < kMaxTreeKids; ++q) { tv[q] = -INFINITY; ti[q] = INT_MAX; }
    float m = -INFINITY, sum = 0.f;
#pragma unroll 4
    for (int x = t; x < V; x += kWidthThreads) {
        const float v = __ldg(row + x);
        if (v > m) { sum = sum * expf(m - v) + 1.f; m = v; } else { sum += expf(v - m); }
        if (v > tv[width - 1]) {            // x grows: an equal value ranks after the kept ones
            int q = width - 1;
            while (q > 0 && v > tv[q - 1]) { tv[q] = tv[q - 1]; ti[q] = ti[q - 1]; --q; }
            tv[q] = v;
            ti[q] = x;
        }
    }
    // the row's max and sum of exp
    float mx = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_m[w] = mx;
    __syncthreads();
    mx = s_m[0];
    for (int q = 1; q < NW; ++q) mx = fmaxf(mx, s_m[q]);
    float part = sum * expf(m - mx);        // a thread without elements adds 0 * 0
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if (lane == 0) s_s[w] = part;
    __syncthreads();
    float total = 0.f;
    for (int q = 0; q < NW; ++q) total += s_s[q];
    // tournament: `width` rounds of block argmax over the list heads
    int head = 0, c = 0;
    float cum = 0.f;
    for (int k = 0; k < width; ++k) {
        float bv = head < width ? tv[head] : -INFINITY;
        int bi = head < width ? ti[head] : INT_MAX;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) { s_v[w] = bv; s_i[w] = bi; }
        __syncthreads();
        float v = s_v[0];
        int id = s_i[0];
        for (int q = 1; q < NW; ++q)
            if (s_v[q] > v || (s_v[q] == v && s_i[q] < id)) { v = s_v[q]; id = s_i[q]; }
        if (head < width && ti[head] == id) ++head;
        if (t == 0) {
            st[2 + kMaxSeqRows + y * kMaxTreeKids + k] = id;
            cum += expf(v - mx) / total;
            if (c == 0 && cum >= mass) c = k + 1;
        }
        __syncthreads();
    }
    if (t == 0) st[2 + y] = c > 0 ? c : width;
}

// One thread per sequence: the children of the level's nodes in order.
__global__ void tree_assign_kernel(int* tokens, int* parents, int* n_nodes, int* stage, int batch, int n_max,
                                   int* err) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    int* st = stage + (size_t)b * kTreeStage;
    const int start = st[0], count = st[1], n = n_nodes[b];
    int at = n;
    for (int y = 0; y < count; ++y) {
        const int c = st[2 + y];
        for (int k = 0; k < c; ++k) {
            if (at >= n_max) { dev_error(err, SPEC_DEVERR_TREE); break; }
            tokens[(size_t)b * n_max + at] = st[2 + kMaxSeqRows + y * kMaxTreeKids + k];
            parents[(size_t)b * n_max + at] = start + y;
            ++at;
        }
    }
    st[0] = n;
    st[1] = at - n;
    n_nodes[b] = at;
}

// Greedy tree acceptance for one tree a sequence, from the row summaries of
// the verify forward and the plan's per-sequence tree arrays.
__global__ void accept_trees_kernel(const spec_row_stats* __restrict__ rs, RowPlan plan, const int* tokens,
                                    int tok_stride, int batch, int* acc_len, int* next_tok, int* path) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= batch) return;
    accept_tree_one(rs, plan.seq_row0[b], plan.seq_nrows[b], tokens + (size_t)b * tok_stride,
                    plan.tree_parent + (size_t)b * kMaxSeqRows, plan.tree_depth + (size_t)b * kMaxSeqRows,
                    acc_len + b, next_tok + b, path ? path + (size_t)b * kMaxSeqRows : nullptr);
}

__global__ void add_len_kernel(int* len, int seq, int n, int cap, int* err) {
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        const int v = len[seq] + n;
        if (v > cap) dev_error(err, SPEC_DEVERR_CAPACITY);
        len[seq] = min(v, cap);
    }
}

template <typename T>
__global__ void kv_copy_kernel(T* cache, T* buf, int to_cache, int seq, int layer0, int n_layers, int slot0,
                               int n_slots, KVPages kvp, int Hkv, int hd, int* err) {
    pdl_wait();
    pdl_trigger();
    const size_t total = (size_t)n_layers * n_slots * Hkv * hd;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int e = (int)(i % hd);
        size_t rest = i / hd;
        const int h = (int)(rest % Hkv); rest /= Hkv;
        const int s = (int)(rest % n_slots);
        const int l = (int)(rest / n_slots);
        const long long row = kv_row(kvp, Hkv, layer0 + l, seq, h, slot0 + s);
        if (row < 0) { dev_error(err, SPEC_DEVERR_CAPACITY); continue; }
        const size_t c = (size_t)row * hd + e;
        if (to_cache) cache[c] = buf[i]; else buf[i] = cache[c];
    }
}

// ---------------------------------------------------------------------------
// forward orchestration
struct HeadSpec {
    int mode;                      // HeadMode
    int T, r0;                     // rows of the head launch
    float* logits; int logits_stride; int logits_row0;
    spec_row_stats* user_stats;
    int* cand; int cand_stride; int cand_col;
    const int* tokens; int tok_stride;
    int* acc_len; int* next_tok; int* path;
    int batch;
};

static EpiParams base_epi(spec_model* m, spec_kv* kv, int T) {
    const spec_model_config& c = m->cfg;
    EpiParams e{};
    e.T = T;
    e.r0 = 0;
    e.ss_in = m->ss_part;
    e.ss_tiles = (c.d_model + kTileN - 1) / kTileN;
    e.ss_stride = c.max_rows;
    e.inv_d = 1.0f / (float)c.d_model;
    e.eps = c.rms_eps;
    e.plan = m->plan;
    e.err = m->err;
    e.q = m->q;
    e.kc = kv->k;
    e.vc = kv->v;
    e.kv_ctx = kv->max_ctx;
    e.kvp = kv->pages();
    e.n_heads = c.n_heads;
    e.n_kv_heads = c.n_kv_heads;
    e.head_dim = c.head_dim;
    e.rope_cos = m->rope_cos;
    e.rope_sin = m->rope_sin;
    e.max_position = c.max_position;
    e.q_scale = 1.0f / sqrtf((float)c.head_dim);
    e.h = m->h;
    e.d_model = c.d_model;
    e.ss_out = m->ss_part;
    e.act = m->x_act;
    e.act_lo = (size_t)m->max_rows_pad * c.d_ff;
    e.x_next_lo = (size_t)m->max_rows_pad * c.d_model;
    e.d_ff = c.d_ff;
    e.vocab = c.vocab;
    e.stat_part = m->stat_part;
    e.row_stats = m->row_stats;
    e.done_counter = m->counters + m->n_counters - 1;
    return e;
}

static GemmStep head_step(spec_model* m, spec_kv* kv, const HeadSpec& hs) {
    const spec_model_config& c = m->cfg;
    EpiParams e = base_epi(m, kv, hs.T);
    e.kind = EPI_HEAD;
    e.r0 = hs.r0;
    e.N = c.vocab;
    e.logits = hs.logits;
    e.logits_stride = hs.logits_stride;
    e.logits_row0 = hs.logits_row0;
    e.user_stats = hs.user_stats;
    e.head_mode = hs.mode;
    e.cand = hs.cand;
    e.cand_stride = hs.cand_stride;
    e.cand_col = hs.cand_col;
    e.tokens = hs.tokens;
    e.tok_stride = hs.tok_stride;
    e.acc_len = hs.acc_len;
    e.next_tok = hs.next_tok;
    e.path = hs.path;
    e.batch = hs.batch;
    return GemmStep{GemmLaunch{&m->tm_head, nullptr, m->head, m->x_in, c.d_model, c.vocab, c.d_model}, e, 0};
}

// Layers [lo, hi) on the T rows of the current plan, then (head != nullptr) the
// LM head.  GEMMs between two attentions go out as one chain:
//   [QKV lo]  attn  [O, gate|up, down, QKV lo+1]  attn  ...  [O, gate|up, down, head]
// head_follows picks the gain of the last down projection's next-input
// (the final norm when the LM head reads it).
static int run_layers(spec_model* m, spec_kv* kv, int T, int batch, int max_rows_per_seq, int lo, int hi,
                      int tree, bool head_follows, const HeadSpec* head, cudaStream_t st) {
    const spec_model_config& c = m->cfg;
    const int qdim = c.n_heads * c.head_dim;
    // attention as the first phase of the chain that follows it (one launch per layer)
    // (the phase reads one tree for the batch: a tree a sequence takes the separate kernel)
    const bool fused = tree != 2 && T <= kMaxTPad && attn_phase_ok(m, kv, batch, max_rows_per_seq);
    // otherwise, for a few query vectors per (sequence, KV head), the TMA-ring kernel
    const bool ring = !fused && tree != 2 && m->attn_ring && attn_ring_fits(m, kv, batch, max_rows_per_seq);
    GemmStep pend[5];
    int np = 0;
    for (int l = lo; l < hi; ++l) {
        LayerWeights& L = m->layers[l];
        EpiParams e = base_epi(m, kv, T);
        e.layer = l;
        {   // Q|K|V (closes the chain of the previous layer's MLP)
            EpiParams q = e;
            q.kind = EPI_QKV;
            q.N = m->qkv_n;
            pend[np++] = GemmStep{GemmLaunch{&L.tm_qkv, nullptr, L.qkv, m->x_in, c.d_model, m->qkv_n, c.d_model}, q, 0};
            SPEC_TRY(launch_gemm_chain(m, pend, np, st));
            np = 0;
        }
        if (fused) {   // attention phase of the chain that follows
            GemmStep at{};
            at.kind = PH_ATTN;
            at.g.tmW = &kv->tm_k;
            at.g.tmX = &kv->tm_v;
            at.e = e;
            at.at.q = m->q;
            at.at.out = m->x_attn;
            at.at.out_lo = (size_t)m->max_rows_pad * qdim;
            at.at.plan = m->plan;
            at.at.batch = batch;
            at.at.kv_ctx = kv->max_ctx;
            at.at.layer = l;
            at.at.n_heads = c.n_heads;
            at.at.n_kv_heads = c.n_kv_heads;
            at.at.head_dim = c.head_dim;
            at.at.tree = tree;
            at.at.linear = max_rows_per_seq * (c.n_heads / c.n_kv_heads) <= kAttnSimtQ;
            at.at.kc = kv->k;
            at.at.vc = kv->v;
            pend[np++] = at;
        } else {   // attention
            AttnParams a{};
            a.q = m->q;
            a.kc = kv->k;
            a.vc = kv->v;
            a.out = m->x_attn;
            a.out_lo = (size_t)m->max_rows_pad * qdim;
            a.plan = m->plan;
            a.batch = batch;
            a.kv_ctx = kv->max_ctx;
            a.layer = l;
            a.n_heads = c.n_heads;
            a.n_kv_heads = c.n_kv_heads;
            a.head_dim = c.head_dim;
            a.tree = tree;
            a.kvp = kv->pages();
            a.err = m->err;
            if (ring) SPEC_TRY(launch_attention_ring(m, kv, a, st));
            else SPEC_TRY(launch_attention(m, a, max_rows_per_seq, st));
        }
        {   // O projection + residual
            EpiParams o = e;
            o.kind = EPI_RESID;
            o.N = c.d_model;
            o.gain_next = L.ffn_g;
            o.x_next = m->x_in;
            pend[np++] = GemmStep{GemmLaunch{&L.tm_o, nullptr, L.o, m->x_attn, qdim, c.d_model, qdim}, o, 1};
        }
        {   // gate | up -> SwiGLU
            EpiParams sg = e;
            sg.kind = EPI_SWIGLU;
            sg.N = m->gu_n;
            pend[np++] = GemmStep{GemmLaunch{&L.tm_gu, nullptr, L.gu, m->x_in, c.d_model, m->gu_n, c.d_model}, sg, 0};
        }
        {   // down projection + residual
            EpiParams dn = e;
            dn.kind = EPI_RESID;
            dn.N = c.d_model;
            dn.gain_next = (l + 1 < hi || !head_follows) ? (l + 1 < c.n_layers ? m->layers[l + 1].attn_g : m->final_g)
                                                         : m->final_g;
            dn.x_next = m->x_in;
            pend[np++] = GemmStep{GemmLaunch{&L.tm_down, nullptr, L.down, m->x_act, c.d_ff, c.d_model, c.d_ff}, dn, 2};
        }
    }
    if (head && np > 0 && head->T == T && head->r0 == 0) {
        pend[np++] = head_step(m, kv, *head);
        return launch_gemm_chain(m, pend, np, st);
    }
    SPEC_TRY(launch_gemm_chain(m, pend, np, st));
    if (head) {
        const GemmStep h = head_step(m, kv, *head);
        return launch_gemm(m, h.g, h.e, h.xbuf, st);
    }
    return SPEC_OK;
}

static int launch_plan(spec_model* m, const PlanParams& p, int T, const int* len, cudaStream_t st,
                       const int* dev_parent = nullptr, int dev_stride = 0) {
    PlanArgs a{};
    a.p = p;
    a.dev_parent = dev_parent;
    a.dev_stride = dev_stride;
    int r = 0;
    for (int b = 0; b < p.batch; ++b) {
        a.row0[b] = r;
        r += (p.mode == 2) ? 1 : p.n_rows[b];
    }
    const int n = std::max(std::max(T, p.batch), kMaxSeqRows);
    cudaError_t le = launch_k(m->pdl, plan_kernel, dim3((n + 127) / 128), dim3(128), 0, st, a, m->plan, len, T,
                              m->err);
    if (le != cudaSuccess) return check_cuda(le, "plan launch");
    ++m->launches;
    return check_cuda(cudaGetLastError(), "plan launch");
}

static int launch_prologue(spec_model* m, int T, const float* h_in, int h_stride, const int* tok, int tok_stride,
                           int tok_col, int layer_lo, cudaStream_t st) {
    const spec_model_config& c = m->cfg;
    const float* gain = layer_lo < c.n_layers ? m->layers[layer_lo].attn_g : m->final_g;
    if (m->bf16)
        launch_k(m->pdl, prologue_kernel<__nv_bfloat16>, dim3(T, (c.d_model + 127) / 128), dim3(128), 0, st, h_in, h_stride, tok, tok_stride, tok_col,
                                                         (const __nv_bfloat16*)m->embed, m->plan, c.d_model, c.vocab,
                                                         gain, m->h, (__nv_bfloat16*)m->x_in,
                                                         (size_t)m->max_rows_pad * c.d_model, m->ss_part, c.max_rows,
                                                         m->err);
    else
        launch_k(m->pdl, prologue_kernel<float>, dim3(T, (c.d_model + 127) / 128), dim3(128), 0, st, h_in, h_stride, tok, tok_stride, tok_col, (const float*)m->embed,
                                                 m->plan, c.d_model, c.vocab, gain, m->h, (float*)m->x_in, 0,
                                                 m->ss_part, c.max_rows, m->err);
    ++m->launches;
    return check_cuda(cudaGetLastError(), "prologue launch");
}

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace spec

using namespace spec;

// ---------------------------------------------------------------------------
extern "C" const char* spec_last_error(void) { return g_err.c_str(); }

extern "C" int spec_device_info(int32_t* num_sms, int32_t* cc_major, int32_t* cc_minor) {
    int dev = 0;
    SPEC_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
    int v = 0;
    if (num_sms) { SPEC_CUDA(cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev), "attr"); *num_sms = v; }
    if (cc_major) { SPEC_CUDA(cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev), "attr"); *cc_major = v; }
    if (cc_minor) { SPEC_CUDA(cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMinor, dev), "attr"); *cc_minor = v; }
    return SPEC_OK;
}

extern "C" void spec_model_destroy(spec_model* m) {
    if (!m) return;
    for (cudaEvent_t e : m->prof_ev) cudaEventDestroy(e);
    cudaFree(m->wmem);
    cudaFree(m->ws);
    delete m;
}

extern "C" int spec_model_create(const spec_model_config* cfg, const void* const* weights, void* stream,
                                 spec_model** out) {
    if (!cfg || !weights || !out) return set_error(SPEC_ERR_ARG, "spec_model_create: null pointer");
    *out = nullptr;
    const spec_model_config c = *cfg;
    if (c.n_layers < 1 || c.d_model < 1 || c.n_heads < 1 || c.n_kv_heads < 1 || c.head_dim < 1 || c.d_ff < 1 ||
        c.vocab < 2 || c.max_rows < 1 || c.max_batch < 1 || c.max_position < 1 || !(c.rms_eps >= 0.f) ||
        !(c.rope_theta > 0.f))
        return set_error(SPEC_ERR_ARG, "spec_model_create: non-positive size");
    if (c.exit_layer < 0 || c.exit_layer >= c.n_layers) return set_error(SPEC_ERR_ARG, "exit_layer must be in [0, N)");
    if (c.dtype != SPEC_DTYPE_F32 && c.dtype != SPEC_DTYPE_BF16) return set_error(SPEC_ERR_ARG, "unknown dtype");
    if (c.head_dim != 64 && c.head_dim != 128) return set_error(SPEC_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (c.n_heads % c.n_kv_heads) return set_error(SPEC_ERR_UNSUPPORTED, "n_heads must be a multiple of n_kv_heads");
    if (c.d_model % 64 || (c.n_heads * c.head_dim) % 64 || c.d_ff % 64)
        return set_error(SPEC_ERR_UNSUPPORTED, "d_model, n_heads*head_dim and d_ff must be multiples of 64");
    if (c.max_rows > 4096 || c.max_batch > kMaxPlanBatch)
        return set_error(SPEC_ERR_CAPACITY, "max_rows <= 4096 and max_batch <= 256");
    for (int i = 0; i < SPEC_W_COUNT(c.n_layers); ++i)
        if (!weights[i]) return set_error(SPEC_ERR_ARG, "spec_model_create: null weight pointer");

    spec_model* m = new spec_model();
    m->cfg = c;
    cudaStream_t st = (cudaStream_t)stream;
    auto fail = [&](int rc) { spec_model_destroy(m); return rc; };
    int rc;
    if ((rc = check_cuda(cudaGetDevice(&m->device), "cudaGetDevice"))) return fail(rc);
    if ((rc = check_cuda(cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device), "attr")))
        return fail(rc);
    m->bf16 = c.dtype == SPEC_DTYPE_BF16;
    {   // SPEC_PDL=0 turns programmatic dependent launch off (kernels then run back to back)
        const char* e = getenv("SPEC_PDL");
        m->pdl = !(e && e[0] == '0');
        // SPEC_CHAIN=0 launches every GEMM on its own
        const char* ce = getenv("SPEC_CHAIN");
        m->chain = !(ce && ce[0] == '0');
        // attention as the first phase of each layer's GEMM chain (one launch per layer) or as
        // its own kernel: SPEC_ATTN_PHASE=1 / 0 forces either; by default the phase runs for calls
        // of two or more sequences (measured faster there; the separate kernel is faster for one)
        const char* ae = getenv("SPEC_ATTN_PHASE");
        m->attn_phase = (ae && ae[0] == '1') ? 1 : ((ae && ae[0] == '0') ? 0 : -1);
        // SPEC_ATTN_RING=1 (one CTA an SM) or 2 (two): attention outside a chain with few query
        // vectors takes the TMA-ring kernel; otherwise the register-tile kernel
        const char* re = getenv("SPEC_ATTN_RING");
        m->attn_ring = re && (re[0] == '1' || re[0] == '2');
        m->attn_ring_pairs = (re && re[0] == '2') ? 1 : 0;
    }
    m->elem = m->bf16 ? 2 : 4;
    if (m->bf16) {
        int major = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, m->device);
        if (major < 10) return fail(set_error(SPEC_ERR_UNSUPPORTED, "bf16 path needs a Blackwell (sm_10x) GPU"));
    }
    const size_t E = m->elem;
    const int d = c.d_model, qdim = c.n_heads * c.head_dim, F = c.d_ff, V = c.vocab;
    const int gu_blocks = (F + 63) / 64;
    m->qkv_n = (c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
    m->gu_n = gu_blocks * 128;
    m->max_rows_pad = (c.max_rows + 15) / 16 * 16;
    const int half = c.head_dim / 2;

    // ---- packed weights
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const size_t o_embed = take((size_t)V * d * E), o_head = take((size_t)V * d * E), o_fg = take((size_t)d * 4);
    std::vector<size_t> o_l(c.n_layers * 6);
    for (int l = 0; l < c.n_layers; ++l) {
        o_l[l * 6 + 0] = take((size_t)m->qkv_n * d * E);
        o_l[l * 6 + 1] = take((size_t)d * qdim * E);
        o_l[l * 6 + 2] = take((size_t)m->gu_n * d * E);
        o_l[l * 6 + 3] = take((size_t)d * F * E);
        o_l[l * 6 + 4] = take((size_t)d * 4);
        o_l[l * 6 + 5] = take((size_t)d * 4);
    }
    const size_t o_cos = take((size_t)c.max_position * half * 4), o_sin = take((size_t)c.max_position * half * 4);
    if ((rc = check_cuda(cudaMalloc(&m->wmem, off), "cudaMalloc(weights)"))) return fail(rc);
    char* W = m->wmem;
    m->embed = W + o_embed;
    m->head = W + o_head;
    m->final_g = (float*)(W + o_fg);
    m->rope_cos = (float*)(W + o_cos);
    m->rope_sin = (float*)(W + o_sin);
    auto cp = [&](void* dst, const void* src, size_t bytes) {
        return check_cuda(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st), "weight copy");
    };
    auto gain = [&](float* dst, const void* src) {
        if (m->bf16) to_f32_kernel<__nv_bfloat16><<<(d + 255) / 256, 256, 0, st>>>((const __nv_bfloat16*)src, dst, d);
        else to_f32_kernel<float><<<(d + 255) / 256, 256, 0, st>>>((const float*)src, dst, d);
        return check_cuda(cudaGetLastError(), "gain copy");
    };
    if ((rc = cp(m->embed, weights[SPEC_W_EMBED], (size_t)V * d * E))) return fail(rc);
    if ((rc = cp(m->head, weights[SPEC_W_LM_HEAD], (size_t)V * d * E))) return fail(rc);
    if ((rc = gain(m->final_g, weights[SPEC_W_FINAL_NORM]))) return fail(rc);
    m->layers.resize(c.n_layers);
    const size_t row = (size_t)d * E;
    for (int l = 0; l < c.n_layers; ++l) {
        const void* const* wl = weights + SPEC_W_LAYER0 + 9 * l;
        LayerWeights& L = m->layers[l];
        L.qkv = W + o_l[l * 6 + 0];
        L.o = W + o_l[l * 6 + 1];
        L.gu = W + o_l[l * 6 + 2];
        L.down = W + o_l[l * 6 + 3];
        L.attn_g = (float*)(W + o_l[l * 6 + 4]);
        L.ffn_g = (float*)(W + o_l[l * 6 + 5]);
        char* qkv = (char*)L.qkv;
        if ((rc = cp(qkv, wl[SPEC_WL_Q], (size_t)qdim * row))) return fail(rc);
        if ((rc = cp(qkv + (size_t)qdim * row, wl[SPEC_WL_K], (size_t)c.n_kv_heads * c.head_dim * row))) return fail(rc);
        if ((rc = cp(qkv + (size_t)(qdim + c.n_kv_heads * c.head_dim) * row, wl[SPEC_WL_V],
                     (size_t)c.n_kv_heads * c.head_dim * row))) return fail(rc);
        if ((rc = cp(L.o, wl[SPEC_WL_O], (size_t)d * qdim * E))) return fail(rc);
        // gate/up: per block of 64 features, 64 gate rows then 64 up rows
        if ((rc = check_cuda(cudaMemcpy2DAsync(L.gu, 128 * row, wl[SPEC_WL_GATE], 64 * row, 64 * row, F / 64,
                                               cudaMemcpyDeviceToDevice, st), "gate pack"))) return fail(rc);
        if ((rc = check_cuda(cudaMemcpy2DAsync((char*)L.gu + 64 * row, 128 * row, wl[SPEC_WL_UP], 64 * row, 64 * row,
                                               F / 64, cudaMemcpyDeviceToDevice, st), "up pack"))) return fail(rc);
        if ((rc = cp(L.down, wl[SPEC_WL_DOWN], (size_t)d * F * E))) return fail(rc);
        if ((rc = gain(L.attn_g, wl[SPEC_WL_ATTN_NORM]))) return fail(rc);
        if ((rc = gain(L.ffn_g, wl[SPEC_WL_FFN_NORM]))) return fail(rc);
    }
    {
        const long long n = (long long)c.max_position * half;
        rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(m->rope_cos, m->rope_sin, c.max_position, half,
                                                                       (double)c.rope_theta);
        if ((rc = check_cuda(cudaGetLastError(), "rope table"))) return fail(rc);
    }

    // ---- workspace
    const int R = c.max_rows, Rp = m->max_rows_pad;
    const int t_pad_max = m->bf16 ? std::min(kMaxTPad, Rp) : 32;
    size_t part = 0;
    const int shapes[5][2] = {{m->qkv_n, d}, {d, qdim}, {m->gu_n, d}, {d, F}, {V, d}};
    int max_tiles = 0;
    for (auto& s : shapes) {
        part = std::max(part, gemm_partial_floats_needed(m, s[0], s[1], t_pad_max));
        max_tiles = std::max(max_tiles, (s[0] + kTileN - 1) / kTileN);
    }
    m->gemm_part_floats = part;
    m->n_counters = max_tiles + 3;
    const int rows_per_seq = std::min(kMaxSeqRows, R);
    m->attn_part_floats = attn_partial_floats_needed(m, c.max_batch, rows_per_seq);
    const int G = c.n_heads / c.n_kv_heads;
    m->n_attn_counters = c.max_batch * c.n_kv_heads * ((rows_per_seq * G + 15) / 16);
    off = 0;
    const size_t w_h = take((size_t)R * d * 4);
    const int xr = m->bf16 ? 2 * Rp : Rp;    // bf16: hi rows then lo rows
    const size_t w_xin = take((size_t)xr * d * E), w_xat = take((size_t)xr * qdim * E), w_xac = take((size_t)xr * F * E);
    const size_t w_q = take((size_t)R * qdim * 4);
    const size_t w_ss = take((size_t)((d + 127) / 128) * R * 4);
    const size_t w_sp = take((size_t)((V + 127) / 128) * R * sizeof(spec_row_stats));
    const size_t w_rs = take((size_t)R * sizeof(spec_row_stats));
    const size_t w_gp = take(part * 4);
    const size_t w_cnt = take((size_t)m->n_counters * 4);
    const size_t w_ap = take(m->attn_part_floats * 4);
    const size_t w_ac = take((size_t)m->n_attn_counters * 4);
    const size_t w_err = take(64);
    const size_t w_pkv = take(64);
    const size_t w_plan = take((size_t)(4 * R + 3 * c.max_batch + (2 * kMaxSeqRows + kTreeStage) * c.max_batch + 64) * 4);
    const size_t w_dl = take((size_t)c.max_batch * V * 4);
    m->ws_bytes = off;
    if ((rc = check_cuda(cudaMalloc(&m->ws, off), "cudaMalloc(workspace)"))) return fail(rc);
    if ((rc = check_cuda(cudaMemsetAsync(m->ws, 0, off, st), "workspace clear"))) return fail(rc);
    char* S = m->ws;
    m->h = (float*)(S + w_h);
    m->x_in = S + w_xin;
    m->x_attn = S + w_xat;
    m->x_act = S + w_xac;
    m->q = (float*)(S + w_q);
    m->ss_part = (float*)(S + w_ss);
    m->stat_part = (spec_row_stats*)(S + w_sp);
    m->row_stats = (spec_row_stats*)(S + w_rs);
    m->gemm_part = (float*)(S + w_gp);
    m->counters = (int*)(S + w_cnt);
    m->attn_part = (float*)(S + w_ap);
    m->attn_counters = (int*)(S + w_ac);
    m->err = (int*)(S + w_err);
    m->prof_kv = (unsigned long long*)(S + w_pkv);
    m->draft_lg = (float*)(S + w_dl);
    int* pl = (int*)(S + w_plan);
    m->plan.row_seq = pl; pl += R;
    m->plan.row_slot = pl; pl += R;
    m->plan.row_pos = pl; pl += R;
    m->plan.row_local = pl; pl += R;
    m->plan.seq_row0 = pl; pl += c.max_batch;
    m->plan.seq_nrows = pl; pl += c.max_batch;
    m->plan.seq_base = pl; pl += c.max_batch;
    m->plan.tree_parent = pl; pl += (size_t)c.max_batch * kMaxSeqRows;
    m->plan.tree_depth = pl; pl += (size_t)c.max_batch * kMaxSeqRows;
    // tree_stage(m) follows: kTreeStage ints a sequence

    // ---- tile-major GEMM weights (bf16 path; SPEC_TILED_W=0 keeps them row-major)
    if (m->bf16) {
        const char* te = getenv("SPEC_TILED_W");
        struct Mat { void* w; int N, K; };
        std::vector<Mat> mats;
        for (int l = 0; l < c.n_layers; ++l) {
            LayerWeights& L = m->layers[l];
            mats.push_back({L.qkv, m->qkv_n, d});
            mats.push_back({L.o, d, qdim});
            mats.push_back({L.gu, m->gu_n, d});
            mats.push_back({L.down, d, F});
        }
        mats.push_back({m->head, V, d});
        bool fits = !(te && te[0] == '0');
        size_t most = 0;
        for (const Mat& x : mats) {
            fits &= x.N % kTileN == 0 && x.K % kTileK == 0;
            most = std::max(most, (size_t)x.N * x.K * 2);
        }
        if (fits) {
            void* tmp = nullptr;
            if ((rc = check_cuda(cudaMalloc(&tmp, most), "cudaMalloc(weight tiling)"))) return fail(rc);
            for (const Mat& x : mats) {
                const size_t bytes = (size_t)x.N * x.K * 2;
                tile_weights_kernel<<<4 * m->num_sms, 256, 0, st>>>((const uint4*)x.w, (uint4*)tmp, x.N, x.K);
                rc = check_cuda(cudaGetLastError(), "weight tiling");
                if (!rc) rc = check_cuda(cudaMemcpyAsync(x.w, tmp, bytes, cudaMemcpyDeviceToDevice, st), "weight tiling copy");
                if (rc) { cudaFree(tmp); return fail(rc); }
            }
            rc = check_cuda(cudaStreamSynchronize(st), "weight tiling sync");
            cudaFree(tmp);
            if (rc) return fail(rc);
            m->w_tiled = true;
        }
    }

    // ---- tensor maps (bf16 path)
    if (m->bf16) {
        bool ok = true;
        for (int l = 0; l < c.n_layers; ++l) {
            LayerWeights& L = m->layers[l];
            ok &= make_tmap_2d(&L.tm_qkv, L.qkv, d, m->qkv_n, (uint64_t)d * 2, kTileK, kTileN);
            ok &= make_tmap_2d(&L.tm_o, L.o, qdim, d, (uint64_t)qdim * 2, kTileK, kTileN);
            ok &= make_tmap_2d(&L.tm_gu, L.gu, d, m->gu_n, (uint64_t)d * 2, kTileK, kTileN);
            ok &= make_tmap_2d(&L.tm_down, L.down, F, d, (uint64_t)F * 2, kTileK, kTileN);
        }
        ok &= make_tmap_2d(&m->tm_head, m->head, d, V, (uint64_t)d * 2, kTileK, kTileN);
        const void* xb[3] = {m->x_in, m->x_attn, m->x_act};
        const int xk[3] = {d, qdim, F};
        for (int i = 0; i < 3; ++i)
            for (int tp = 16; tp <= t_pad_max; tp += 16)
                ok &= make_tmap_x(&m->tm_x[i][tp / 16 - 1], xb[i], xk[i], Rp, tp);
        if (!ok) return fail(set_error(SPEC_ERR_CUDA, "cuTensorMapEncodeTiled failed"));
    }
    if ((rc = check_cuda(cudaStreamSynchronize(st), "spec_model_create sync"))) return fail(rc);
    *out = m;
    return SPEC_OK;
}

extern "C" int spec_device_error(spec_model* m, int32_t* host_bits) {
    if (!m || !host_bits) return set_error(SPEC_ERR_ARG, "spec_device_error: null pointer");
    int v = 0;
    SPEC_CUDA(cudaMemcpy(&v, m->err, 4, cudaMemcpyDeviceToHost), "read device error");
    SPEC_CUDA(cudaMemset(m->err, 0, 4), "clear device error");
    *host_bits = v;
    return SPEC_OK;
}

extern "C" int spec_test_stall_next_chain(spec_model* m, int32_t cta, int64_t wait_ns) {
    if (!m) return set_error(SPEC_ERR_ARG, "spec_test_stall_next_chain: null model");
    if (cta < 0 || cta >= m->num_sms || wait_ns < 1000000 || wait_ns > 2000000000)
        return set_error(SPEC_ERR_ARG, "spec_test_stall_next_chain: cta in [0, SMs), wait_ns in [1 ms, 2 s]");
    m->test_stall_cta = cta;
    m->test_wait_ns = (unsigned long long)wait_ns;
    return SPEC_OK;
}

extern "C" int spec_set_exit_layer(spec_model* m, int32_t exit_layer) {
    if (!m) return set_error(SPEC_ERR_ARG, "spec_set_exit_layer: null model");
    if (exit_layer < 0 || exit_layer >= m->cfg.n_layers)
        return set_error(SPEC_ERR_ARG, "spec_set_exit_layer: exit_layer must be in [0, n_layers)");
    // read by every later call when it is enqueued: nothing on the device depends on it
    m->cfg.exit_layer = exit_layer;
    return SPEC_OK;
}

// page = 0: contiguous cache (one page of max_ctx slots per sequence)
static int kv_create(spec_model* m, int32_t batch, int32_t max_ctx, int32_t page, int32_t n_pages, spec_kv** out) {
    *out = nullptr;
    if (batch < 1 || max_ctx < 1) return set_error(SPEC_ERR_ARG, "spec_kv_create: bad sizes");
    if (batch > m->cfg.max_batch) return set_error(SPEC_ERR_CAPACITY, "spec_kv_create: batch > max_batch");
    spec_kv* kv = new spec_kv();
    kv->m = m;
    kv->batch = batch;
    kv->max_ctx = max_ctx;
    kv->paged = page > 0;
    kv->page = kv->paged ? page : max_ctx;
    kv->max_pages = kv->paged ? (max_ctx + page - 1) / page : 1;
    kv->n_pages = kv->paged ? n_pages : batch;
    const size_t bytes = (size_t)m->cfg.n_layers * kv->n_pages * m->cfg.n_kv_heads * kv->page * m->cfg.head_dim * m->elem;
    const size_t tab = (size_t)batch * kv->max_pages;
    int rc = check_cuda(cudaMalloc(&kv->k, bytes), "cudaMalloc(K cache)");
    if (!rc) rc = check_cuda(cudaMalloc(&kv->v, bytes), "cudaMalloc(V cache)");
    if (!rc) rc = check_cuda(cudaMalloc(&kv->len, (size_t)batch * 4), "cudaMalloc(lengths)");
    if (!rc) rc = check_cuda(cudaMalloc(&kv->table, tab * 4), "cudaMalloc(page table)");
    if (!rc) rc = check_cuda(cudaMemset(kv->k, 0, bytes), "clear K");
    if (!rc) rc = check_cuda(cudaMemset(kv->v, 0, bytes), "clear V");
    if (!rc) rc = check_cuda(cudaMemset(kv->len, 0, (size_t)batch * 4), "clear lengths");
    if (!rc) {
        // contiguous: sequence b is page b; paged: no page held, every page free
        std::vector<int> t(tab, -1);
        if (!kv->paged) for (int b = 0; b < batch; ++b) t[b] = b;
        rc = check_cuda(cudaMemcpy(kv->table, t.data(), tab * 4, cudaMemcpyHostToDevice), "page table");
    }
    if (!rc && kv->paged) {
        rc = check_cuda(cudaMalloc(&kv->free_pages, (size_t)(n_pages + 1) * 4), "cudaMalloc(free pages)");
        if (!rc) {
            std::vector<int> f(n_pages + 1);
            for (int i = 0; i < n_pages; ++i) f[i] = n_pages - 1 - i;      // popped from the top: page 0 first
            f[n_pages] = n_pages;
            rc = check_cuda(cudaMemcpy(kv->free_pages, f.data(), f.size() * 4, cudaMemcpyHostToDevice), "free pages");
            kv->free_top = kv->free_pages + n_pages;
        }
    }
    if (!rc && !make_kv_tmaps(kv)) rc = set_error(SPEC_ERR_CUDA, "spec_kv_create: K/V tensor maps");
    if (rc) {
        spec_kv_destroy(kv);
        return rc;
    }
    *out = kv;
    return SPEC_OK;
}

extern "C" int spec_kv_create(spec_model* m, int32_t batch, int32_t max_ctx, spec_kv** out) {
    if (!m || !out) return set_error(SPEC_ERR_ARG, "spec_kv_create: null pointer");
    return kv_create(m, batch, max_ctx, 0, 0, out);
}

extern "C" int spec_kv_create_paged(spec_model* m, int32_t batch, int32_t max_ctx, int32_t page, int32_t n_pages,
                                    spec_kv** out) {
    if (!m || !out) return set_error(SPEC_ERR_ARG, "spec_kv_create_paged: null pointer");
    *out = nullptr;
    if (page < 64 || (page & (page - 1)) != 0)
        return set_error(SPEC_ERR_ARG, "spec_kv_create_paged: page must be a power of two, at least 64");
    if (n_pages < 1) return set_error(SPEC_ERR_ARG, "spec_kv_create_paged: n_pages must be positive");
    return kv_create(m, batch, max_ctx, page, n_pages, out);
}

extern "C" int spec_kv_free_pages(spec_kv* kv, int32_t* host_free, void* stream) {
    if (!kv || !host_free) return set_error(SPEC_ERR_ARG, "spec_kv_free_pages: null pointer");
    if (!kv->paged) { *host_free = 0; return SPEC_OK; }
    SPEC_CUDA(cudaMemcpyAsync(host_free, kv->free_top, 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream), "free pages");
    SPEC_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "free pages sync");
    return SPEC_OK;
}

extern "C" int spec_kv_page_table(spec_kv* kv, int32_t* host_table, void* stream) {
    if (!kv || !host_table) return set_error(SPEC_ERR_ARG, "spec_kv_page_table: null pointer");
    SPEC_CUDA(cudaMemcpyAsync(host_table, kv->table, (size_t)kv->batch * kv->max_pages * 4, cudaMemcpyDeviceToHost,
                              (cudaStream_t)stream), "page table");
    SPEC_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "page table sync");
    return SPEC_OK;
}

extern "C" int spec_kv_read_page(spec_kv* kv, int32_t which, int32_t layer, int32_t page, void* host_dst,
                                 void* stream) {
    if (!kv || !host_dst) return set_error(SPEC_ERR_ARG, "spec_kv_read_page: null pointer");
    const spec_model_config& c = kv->m->cfg;
    if (which < 0 || which > 1 || layer < 0 || layer >= c.n_layers || page < 0 || page >= kv->n_pages)
        return set_error(SPEC_ERR_ARG, "spec_kv_read_page: which, layer or page out of range");
    const size_t page_bytes = (size_t)c.n_kv_heads * kv->page * c.head_dim * kv->m->elem;
    const char* src = static_cast<const char*>(which ? kv->v : kv->k) +
                      ((size_t)layer * kv->n_pages + page) * page_bytes;
    SPEC_CUDA(cudaMemcpyAsync(host_dst, src, page_bytes, cudaMemcpyDeviceToHost, (cudaStream_t)stream), "read page");
    SPEC_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "read page sync");
    return SPEC_OK;
}

extern "C" void spec_kv_destroy(spec_kv* kv) {
    if (!kv) return;
    cudaFree(kv->k);
    cudaFree(kv->v);
    cudaFree(kv->len);
    cudaFree(kv->table);
    cudaFree(kv->free_pages);
    delete kv;
}

extern "C" int spec_kv_set_lengths(spec_kv* kv, const int32_t* host_len, void* stream) {
    if (!kv || !host_len) return set_error(SPEC_ERR_ARG, "spec_kv_set_lengths: null pointer");
    for (int b = 0; b < kv->batch; ++b)
        if (host_len[b] < 0 || host_len[b] > kv->max_ctx) return set_error(SPEC_ERR_CAPACITY, "length beyond max_ctx");
    SPEC_CUDA(cudaMemcpyAsync(kv->len, host_len, (size_t)kv->batch * 4, cudaMemcpyHostToDevice, (cudaStream_t)stream),
              "set lengths");
    if (kv->paged) {          // pages for the slots below the new lengths, the rest back
        SPEC_TRY(kv_release_pages(kv, kv->batch, (cudaStream_t)stream));
        SPEC_TRY(kv_ensure_pages(kv, kv->batch, host_len, false, (cudaStream_t)stream));
    }
    SPEC_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "set lengths sync");
    return SPEC_OK;
}

extern "C" int spec_kv_get_lengths(spec_kv* kv, int32_t* host_len, void* stream) {
    if (!kv || !host_len) return set_error(SPEC_ERR_ARG, "spec_kv_get_lengths: null pointer");
    SPEC_CUDA(cudaMemcpyAsync(host_len, kv->len, (size_t)kv->batch * 4, cudaMemcpyDeviceToHost, (cudaStream_t)stream),
              "get lengths");
    SPEC_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "get lengths sync");
    return SPEC_OK;
}

static int kv_copy(spec_kv* kv, int32_t seq, int32_t layer0, int32_t n_layers, int32_t slot0, int32_t n_slots,
                   void* k, void* v, int to_cache, void* stream) {
    if (!kv || !k || !v) return set_error(SPEC_ERR_ARG, "spec_kv_import/export: null pointer");
    spec_model* m = kv->m;
    const spec_model_config& c = m->cfg;
    if (seq < 0 || seq >= kv->batch || layer0 < 0 || n_layers < 1 || layer0 + n_layers > c.n_layers || slot0 < 0 ||
        n_slots < 1 || slot0 + n_slots > kv->max_ctx)
        return set_error(SPEC_ERR_ARG, "spec_kv_import/export: range outside the cache");
    cudaStream_t st = (cudaStream_t)stream;
    if (kv->paged && to_cache) {          // pages for the imported slots
        int need[kMaxPlanBatch] = {0};
        need[seq] = slot0 + n_slots;
        SPEC_TRY(kv_ensure_pages(kv, seq + 1, need, false, st));
    }
    for (int which = 0; which < 2; ++which) {
        void* cache = which ? kv->v : kv->k;
        void* buf = which ? v : k;
        if (m->bf16)
            kv_copy_kernel<__nv_bfloat16><<<1024, 256, 0, st>>>((__nv_bfloat16*)cache, (__nv_bfloat16*)buf, to_cache,
                                                               seq, layer0, n_layers, slot0, n_slots, kv->pages(),
                                                               c.n_kv_heads, c.head_dim, m->err);
        else
            kv_copy_kernel<float><<<1024, 256, 0, st>>>((float*)cache, (float*)buf, to_cache, seq, layer0, n_layers,
                                                       slot0, n_slots, kv->pages(), c.n_kv_heads, c.head_dim, m->err);
    }
    return check_cuda(cudaGetLastError(), "kv copy launch");
}

extern "C" int spec_kv_import(spec_kv* kv, int32_t seq, int32_t layer0, int32_t n_layers, int32_t slot0,
                              int32_t n_slots, const void* k, const void* v, void* stream) {
    return kv_copy(kv, seq, layer0, n_layers, slot0, n_slots, const_cast<void*>(k), const_cast<void*>(v), 1, stream);
}

extern "C" int spec_kv_export(spec_kv* kv, int32_t seq, int32_t layer0, int32_t n_layers, int32_t slot0,
                              int32_t n_slots, void* k, void* v, void* stream) {
    return kv_copy(kv, seq, layer0, n_layers, slot0, n_slots, k, v, 0, stream);
}

extern "C" int spec_prefill(spec_model* m, spec_kv* kv, int32_t seq, const int32_t* tokens, int32_t n,
                            float* last_logits, int32_t* next_tok, void* stream) {
    if (!m || !kv || !tokens) return set_error(SPEC_ERR_ARG, "spec_prefill: null pointer");
    if (kv->m != m) return set_error(SPEC_ERR_ARG, "spec_prefill: cache of another model");
    if (seq < 0 || seq >= kv->batch || n < 1) return set_error(SPEC_ERR_ARG, "spec_prefill: bad seq or n");
    const spec_model_config& c = m->cfg;
    cudaStream_t st = (cudaStream_t)stream;
    const int chunk = std::min(kMaxSeqRows, c.max_rows);
    for (int done = 0; done < n; done += chunk) {
        const int T = std::min(chunk, n - done);
        PlanParams p{};
        p.batch = seq + 1;
        p.mode = 0;
        p.n_rows[seq] = T;
        SPEC_TRY(kv_ensure_pages(kv, seq + 1, p.n_rows, true, st));
        SPEC_TRY(launch_plan(m, p, T, kv->len, st));
        SPEC_TRY(launch_prologue(m, T, nullptr, 0, tokens + done, 0, 0, 0, st));
        const bool last = done + T >= n;
        const bool head = last && (last_logits || next_tok);
        HeadSpec hs{};
        hs.mode = next_tok ? HEAD_DRAFT : HEAD_STATS;
        hs.T = 1;
        hs.r0 = T - 1;
        hs.logits = last_logits;
        hs.logits_stride = c.vocab;
        hs.logits_row0 = T - 1;
        hs.cand = next_tok;
        hs.cand_stride = 0;
        hs.cand_col = 0;
        hs.batch = seq + 1;
        SPEC_TRY(run_layers(m, kv, T, seq + 1, T, 0, c.n_layers, 0, head, head ? &hs : nullptr, st));
        launch_k(m->pdl, add_len_kernel, dim3(1), dim3(32), 0, st, kv->len, seq, T, kv->max_ctx, m->err);
        ++m->launches;
        SPEC_CUDA(cudaGetLastError(), "length update");
    }
    return SPEC_OK;
}

// Draft passes; greedy (temp == 0: the LM head epilogue picks the argmax) or
// sampling (the head writes logits, then one CTA per sequence forms
// q = softmax(logits / temp) and draws the next token with u_draft).
static int draft_impl(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* t0, int32_t k, int32_t* cand,
                      float* h_L, float* draft_logits, float temp, const float* u_draft, float* q, cudaStream_t st) {
    const spec_model_config& c = m->cfg;
    if (c.exit_layer < 1) return set_error(SPEC_ERR_ARG, "spec_draft: exit_layer must be >= 1");
    if (batch < 1 || batch > kv->batch || batch > c.max_rows) return set_error(SPEC_ERR_ARG, "spec_draft: bad batch");
    if (k < 1 || k + 1 > kMaxSeqRows) return set_error(SPEC_ERR_ARG, "spec_draft: k must be in [1, 63]");
    const bool sampling = temp > 0.f;
    if (sampling && batch > c.max_batch) return set_error(SPEC_ERR_ARG, "spec_draft_sample: batch > max_batch");
    if (kv->paged) {
        int need[kMaxPlanBatch];
        for (int b = 0; b < batch; ++b) need[b] = k + 1;
        SPEC_TRY(kv_ensure_pages(kv, batch, need, true, st));
    }
    launch_k(m->pdl, set_col0_kernel, dim3((batch + 127) / 128), dim3(128), 0, st, t0, cand, k + 1, batch);
    ++m->launches;
    SPEC_CUDA(cudaGetLastError(), "draft init");
    for (int j = 0; j <= k; ++j) {
        PlanParams p{};
        p.batch = batch;
        p.mode = 2;
        p.pass = j;
        SPEC_TRY(launch_plan(m, p, batch, kv->len, st));
        SPEC_TRY(launch_prologue(m, batch, nullptr, 0, cand, k + 1, j, 0, st));
        HeadSpec hs{};
        hs.mode = sampling ? HEAD_STATS : HEAD_DRAFT;
        hs.T = batch;
        hs.r0 = 0;
        if (draft_logits) {
            hs.logits = draft_logits + (size_t)j * c.vocab;
            hs.logits_stride = k * c.vocab;
        } else if (sampling) {
            hs.logits = m->draft_lg;
            hs.logits_stride = c.vocab;
        }
        hs.logits_row0 = 0;
        hs.cand = cand;
        hs.cand_stride = k + 1;
        hs.cand_col = j + 1;
        hs.batch = batch;
        // the LM head leaves the residual stream alone, so the layer-L state is copied after it
        SPEC_TRY(run_layers(m, kv, batch, batch, 1, 0, c.exit_layer, 0, j < k, j < k ? &hs : nullptr, st));
        if (sampling && j < k) {
            SampleArgs a{};
            a.in = hs.logits;
            a.in_stride = hs.logits_stride;
            a.out = q + (size_t)j * c.vocab;
            a.out_stride = (long long)k * c.vocab;
            a.u = u_draft + j;
            a.u_stride = k;
            a.tok = cand + j + 1;
            a.tok_stride = k + 1;
            a.rows = batch;
            a.V = c.vocab;
            a.temp = temp;
            a.err = m->err;
            SPEC_TRY(launch_sample_rows(a, m->pdl, st));
            ++m->launches;
        }
        launch_k(m->pdl, copy_rows_kernel, dim3(batch), dim3(256), 0, st, (const float*)m->h, h_L, batch, c.d_model, k + 1, j);
        ++m->launches;
        SPEC_CUDA(cudaGetLastError(), "draft state copy");
    }
    return SPEC_OK;
}

extern "C" int spec_draft(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* t0, int32_t k, int32_t* cand,
                          float* h_L, float* draft_logits, void* stream) {
    if (!m || !kv || !t0 || !cand || !h_L) return set_error(SPEC_ERR_ARG, "spec_draft: null pointer");
    if (kv->m != m) return set_error(SPEC_ERR_ARG, "spec_draft: cache of another model");
    return draft_impl(m, kv, batch, t0, k, cand, h_L, draft_logits, 0.f, nullptr, nullptr, (cudaStream_t)stream);
}

extern "C" int spec_draft_sample(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* t0, int32_t k,
                                 float temperature, const float* u_draft, int32_t* cand, float* h_L, float* q,
                                 float* draft_logits, void* stream) {
    if (!m || !kv || !t0 || !cand || !h_L || !u_draft || !q) return set_error(SPEC_ERR_ARG, "spec_draft_sample: null pointer");
    if (kv->m != m) return set_error(SPEC_ERR_ARG, "spec_draft_sample: cache of another model");
    if (!(temperature > 0.f) || !(temperature <= 3.402823466e38f))
        return set_error(SPEC_ERR_ARG, "spec_draft_sample: temperature must be positive and finite");
    return draft_impl(m, kv, batch, t0, k, cand, h_L, draft_logits, temperature, u_draft, q, (cudaStream_t)stream);
}

extern "C" int spec_draft_tree(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* t0, const int32_t* tree_parent,
                               int32_t n_nodes, int32_t* tokens, float* h_L, float* logits, void* stream) {
    if (!m || !kv || !t0 || !tree_parent || !tokens || !h_L || !logits)
        return set_error(SPEC_ERR_ARG, "spec_draft_tree: null pointer");
    if (kv->m != m) return set_error(SPEC_ERR_ARG, "spec_draft_tree: cache of another model");
    const spec_model_config& c = m->cfg;
    if (c.exit_layer < 1) return set_error(SPEC_ERR_ARG, "spec_draft_tree: exit_layer must be >= 1");
    if (batch < 1 || batch > kv->batch) return set_error(SPEC_ERR_ARG, "spec_draft_tree: bad batch");
    if (n_nodes < 2 || n_nodes > kMaxSeqRows) return set_error(SPEC_ERR_ARG, "spec_draft_tree: n_nodes must be in [2, 64]");
    if ((long long)batch * n_nodes > c.max_rows) return set_error(SPEC_ERR_CAPACITY, "spec_draft_tree: batch * n_nodes > max_rows");
    if (tree_parent[0] != -1) return set_error(SPEC_ERR_ARG, "tree_parent[0] must be -1");
    PlanParams p{};
    p.batch = batch;
    p.mode = 1;
    p.parent[0] = -1;
    p.depth[0] = 0;
    for (int i = 1; i < n_nodes; ++i) {
        if (tree_parent[i] < 0 || tree_parent[i] >= i) return set_error(SPEC_ERR_ARG, "tree_parent[i] must be in [0, i)");
        p.parent[i] = tree_parent[i];
        p.depth[i] = p.depth[tree_parent[i]] + 1;
        if (p.depth[i] < p.depth[i - 1]) return set_error(SPEC_ERR_ARG, "spec_draft_tree: nodes must be in level order");
    }
    TreeKids tk{};
    {
        int at = 0;
        for (int i = 0; i < n_nodes; ++i) {
            tk.start[i] = at;
            int nk = 0;
            for (int j = i + 1; j < n_nodes; ++j)
                if (tree_parent[j] == i) { tk.kid[at++] = j; ++nk; }
            if (nk > kMaxTreeKids) return set_error(SPEC_ERR_ARG, "spec_draft_tree: at most 16 children a node");
        }
        tk.start[n_nodes] = at;
    }
    cudaStream_t st = (cudaStream_t)stream;
    if (kv->paged) {
        int need[kMaxPlanBatch];
        for (int b = 0; b < batch; ++b) need[b] = n_nodes;
        SPEC_TRY(kv_ensure_pages(kv, batch, need, true, st));
    }
    launch_k(m->pdl, set_col0_kernel, dim3((batch + 127) / 128), dim3(128), 0, st, t0, tokens, n_nodes, batch);
    ++m->launches;
    SPEC_CUDA(cudaGetLastError(), "tree draft init");
    const int D = p.depth[n_nodes - 1];
    int l0 = 0;
    for (int lev = 0; lev <= D; ++lev) {
        int l1 = l0;
        while (l1 < n_nodes && p.depth[l1] == lev) ++l1;
        // layers [0, L) over every node up to this level (earlier levels again: the
        // cost is the weight stream, the same for these few rows)
        for (int b = 0; b < batch; ++b) p.n_rows[b] = l1;
        const int T = batch * l1;
        SPEC_TRY(launch_plan(m, p, T, kv->len, st));
        SPEC_TRY(launch_prologue(m, T, nullptr, 0, tokens, n_nodes, 0, 0, st));
        const bool expand = lev < D;
        HeadSpec hs{};
        hs.mode = HEAD_STATS;
        hs.T = T;
        hs.r0 = 0;
        hs.logits = logits;
        hs.logits_stride = c.vocab;
        hs.logits_row0 = 0;
        hs.batch = batch;
        SPEC_TRY(run_layers(m, kv, T, batch, l1, 0, c.exit_layer, 1, expand, expand ? &hs : nullptr, st));
        if (expand) {
            launch_k(m->pdl, tree_expand_kernel, dim3(batch, l1 - l0), dim3(256), 0, st, (const float*)logits,
                     c.vocab, l1, l0, tk, tokens, n_nodes);
            ++m->launches;
            SPEC_CUDA(cudaGetLastError(), "tree expansion");
        } else {
            launch_k(m->pdl, copy_rows_kernel, dim3(T), dim3(256), 0, st, (const float*)m->h, h_L, T, c.d_model, 1, 0);
            ++m->launches;
            SPEC_CUDA(cudaGetLastError(), "tree draft state copy");
        }
        l0 = l1;
    }
    return SPEC_OK;
}

// The dynamic tree's staging block sits after the plan's tree arrays.
static int* tree_stage(spec_model* m) { return m->plan.tree_depth + (size_t)m->cfg.max_batch * kMaxSeqRows; }

extern "C" int spec_draft_tree_dynamic(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* t0,
                                       const int32_t* branching, int32_t depth, float mass, int32_t* tokens,
                                       int32_t* parents, int32_t* n_nodes, float* h_L, float* logits, void* stream) {
    if (!m || !kv || !t0 || !branching || !tokens || !parents || !n_nodes || !h_L || !logits)
        return set_error(SPEC_ERR_ARG, "spec_draft_tree_dynamic: null pointer");
    if (kv->m != m) return set_error(SPEC_ERR_ARG, "spec_draft_tree_dynamic: cache of another model");
    const spec_model_config& c = m->cfg;
    if (c.exit_layer < 1) return set_error(SPEC_ERR_ARG, "spec_draft_tree_dynamic: exit_layer must be >= 1");
    if (batch < 1 || batch > kv->batch) return set_error(SPEC_ERR_ARG, "spec_draft_tree_dynamic: bad batch");
    if (depth < 1) return set_error(SPEC_ERR_ARG, "spec_draft_tree_dynamic: depth must be >= 1");
    if (mass != mass) return set_error(SPEC_ERR_ARG, "spec_draft_tree_dynamic: mass is NaN");
    // the widest tree: level l holds at most lw[l] nodes, levels up to l at most cum[l]
    int lw[kMaxSeqRows + 1], cum[kMaxSeqRows + 1];
    lw[0] = 1;
    cum[0] = 1;
    for (int l = 0; l < depth; ++l) {
        if (branching[l] < 1 || branching[l] > kMaxTreeKids || branching[l] > c.vocab)
            return set_error(SPEC_ERR_ARG, "spec_draft_tree_dynamic: branching must be in [1, min(16, vocab)]");
        if ((long long)lw[l] * branching[l] + cum[l] > kMaxSeqRows)
            return set_error(SPEC_ERR_ARG, "spec_draft_tree_dynamic: the widest tree has more than 64 nodes");
        lw[l + 1] = lw[l] * branching[l];
        cum[l + 1] = cum[l] + lw[l + 1];
    }
    const int n_max = cum[depth];
    if ((long long)batch * n_max > c.max_rows)
        return set_error(SPEC_ERR_CAPACITY, "spec_draft_tree_dynamic: batch * nodes of the widest tree > max_rows");
    cudaStream_t st = (cudaStream_t)stream;
    if (kv->paged) {
        int need[kMaxPlanBatch];
        for (int b = 0; b < batch; ++b) need[b] = n_max;
        SPEC_TRY(kv_ensure_pages(kv, batch, need, true, st));
    }
    int* stage = tree_stage(m);
    launch_k(m->pdl, tree_init_kernel, dim3((batch * n_max + 255) / 256), dim3(256), 0, st, t0, tokens, parents,
             n_nodes, stage, batch, n_max);
    ++m->launches;
    SPEC_CUDA(cudaGetLastError(), "dynamic tree init");
    PlanParams p{};
    p.batch = batch;
    p.mode = 1;
    for (int lev = 0; lev <= depth; ++lev) {
        // layers [0, L) over every row the tree can hold up to this level
        const int rows = cum[lev];
        for (int b = 0; b < batch; ++b) p.n_rows[b] = rows;
        const int T = batch * rows;
        SPEC_TRY(launch_plan(m, p, T, kv->len, st, parents, n_max));
        SPEC_TRY(launch_prologue(m, T, nullptr, 0, tokens, n_max, 0, 0, st));
        const bool expand = lev < depth;
        HeadSpec hs{};
        hs.mode = HEAD_STATS;
        hs.T = T;
        hs.r0 = 0;
        hs.logits = logits;
        hs.logits_stride = c.vocab;
        hs.logits_row0 = 0;
        hs.batch = batch;
        SPEC_TRY(run_layers(m, kv, T, batch, rows, 0, c.exit_layer, 2, expand, expand ? &hs : nullptr, st));
        if (expand) {
            launch_k(m->pdl, tree_width_kernel, dim3(batch, lw[lev]), dim3(kWidthThreads), 0, st, (const float*)logits, c.vocab,
                     rows, (int)branching[lev], mass, stage);
            launch_k(m->pdl, tree_assign_kernel, dim3((batch + 127) / 128), dim3(128), 0, st, tokens, parents, n_nodes,
                     stage, batch, n_max, m->err);
            m->launches += 2;
            SPEC_CUDA(cudaGetLastError(), "dynamic tree expansion");
        } else {
            launch_k(m->pdl, copy_rows_kernel, dim3(T), dim3(256), 0, st, (const float*)m->h, h_L, T, c.d_model, 1, 0);
            ++m->launches;
            SPEC_CUDA(cudaGetLastError(), "dynamic tree state copy");
        }
    }
    return SPEC_OK;
}

// Verification forward: one tree for the batch (tree_parent, host), one tree a
// sequence (dev_parent, device [batch][par_stride]) or a chain (neither).
static int verify_impl(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* n_rows, const float* h_in,
                       int32_t h_stride, const int32_t* tokens, int32_t tok_stride, const int32_t* tree_parent,
                       const int32_t* dev_parent, int32_t par_stride, float* logits, spec_row_stats* stats,
                       int32_t* acc_len, int32_t* next_tok, int32_t* path, cudaStream_t st) {
    if (!m || !kv || !n_rows || !tokens) return set_error(SPEC_ERR_ARG, "spec_verify: null pointer");
    if (kv->m != m) return set_error(SPEC_ERR_ARG, "spec_verify: cache of another model");
    const spec_model_config& c = m->cfg;
    if (batch < 1 || batch > kv->batch) return set_error(SPEC_ERR_ARG, "spec_verify: bad batch");
    if ((acc_len == nullptr) != (next_tok == nullptr)) return set_error(SPEC_ERR_ARG, "acc_len and next_tok go together");
    const bool trees = dev_parent != nullptr;
    if ((tree_parent || trees) && acc_len && !path) return set_error(SPEC_ERR_ARG, "tree acceptance needs path");
    if (h_in && c.exit_layer < 1) return set_error(SPEC_ERR_ARG, "h_in needs exit_layer >= 1");
    int T = 0, max_r = 0;
    PlanParams p{};
    p.batch = batch;
    p.mode = (tree_parent || trees) ? 1 : 0;
    for (int b = 0; b < batch; ++b) {
        if (n_rows[b] < 1 || n_rows[b] > kMaxSeqRows) return set_error(SPEC_ERR_ARG, "n_rows[b] must be in [1, 64]");
        if (h_in && n_rows[b] > h_stride) return set_error(SPEC_ERR_ARG, "n_rows[b] > h_stride");
        if (n_rows[b] > tok_stride) return set_error(SPEC_ERR_ARG, "n_rows[b] > tok_stride");
        if (trees && n_rows[b] > par_stride) return set_error(SPEC_ERR_ARG, "n_rows[b] > par_stride");
        p.n_rows[b] = n_rows[b];
        T += n_rows[b];
        max_r = std::max(max_r, (int)n_rows[b]);
    }
    if (T > c.max_rows) return set_error(SPEC_ERR_CAPACITY, "sum of n_rows > max_rows");
    if (tree_parent) {
        const int n = n_rows[0];
        if (tree_parent[0] != -1) return set_error(SPEC_ERR_ARG, "tree_parent[0] must be -1");
        p.parent[0] = -1;
        p.depth[0] = 0;
        for (int i = 1; i < n; ++i) {
            if (tree_parent[i] < 0 || tree_parent[i] >= i) return set_error(SPEC_ERR_ARG, "tree_parent[i] must be in [0, i)");
            p.parent[i] = tree_parent[i];
            p.depth[i] = p.depth[tree_parent[i]] + 1;
        }
        for (int b = 0; b < batch; ++b)
            if (n_rows[b] != n) return set_error(SPEC_ERR_ARG, "tree mode: every sequence has the tree's node count");
    }
    const int lo = h_in ? c.exit_layer : 0;
    SPEC_TRY(kv_ensure_pages(kv, batch, p.n_rows, true, st));
    SPEC_TRY(launch_plan(m, p, T, kv->len, st, dev_parent, par_stride));
    SPEC_TRY(launch_prologue(m, T, h_in, h_stride, tokens, tok_stride, 0, lo, st));
    HeadSpec hs{};
    // one tree a sequence: summaries in the head, acceptance in its own kernel
    hs.mode = (acc_len && !trees) ? (tree_parent ? HEAD_ACCEPT_TREE : HEAD_ACCEPT_CHAIN) : HEAD_STATS;
    hs.T = T;
    hs.r0 = 0;
    hs.logits = logits;
    hs.logits_stride = c.vocab;
    hs.logits_row0 = 0;
    hs.user_stats = stats;
    hs.tokens = tokens;
    hs.tok_stride = tok_stride;
    hs.acc_len = acc_len;
    hs.next_tok = next_tok;
    hs.path = path;
    hs.batch = batch;
    SPEC_TRY(run_layers(m, kv, T, batch, max_r, lo, c.n_layers, trees ? 2 : (tree_parent ? 1 : 0), true, &hs, st));
    if (trees && acc_len) {
        launch_k(m->pdl, accept_trees_kernel, dim3((batch + 127) / 128), dim3(128), 0, st,
                 (const spec_row_stats*)m->row_stats, m->plan, tokens, tok_stride, batch, acc_len, next_tok, path);
        ++m->launches;
        SPEC_CUDA(cudaGetLastError(), "tree acceptance");
    }
    return SPEC_OK;
}

extern "C" int spec_verify(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* n_rows, const float* h_in,
                           int32_t h_stride, const int32_t* tokens, int32_t tok_stride, const int32_t* tree_parent,
                           float* logits, spec_row_stats* stats, int32_t* acc_len, int32_t* next_tok, int32_t* path,
                           void* stream) {
    return verify_impl(m, kv, batch, n_rows, h_in, h_stride, tokens, tok_stride, tree_parent, nullptr, 0, logits,
                       stats, acc_len, next_tok, path, (cudaStream_t)stream);
}

extern "C" int spec_verify_trees(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* n_rows, const float* h_in,
                                 int32_t h_stride, const int32_t* tokens, int32_t tok_stride, const int32_t* parents,
                                 int32_t par_stride, float* logits, spec_row_stats* stats, int32_t* acc_len,
                                 int32_t* next_tok, int32_t* path, void* stream) {
    if (!parents) return set_error(SPEC_ERR_ARG, "spec_verify_trees: null parents");
    return verify_impl(m, kv, batch, n_rows, h_in, h_stride, tokens, tok_stride, nullptr, parents, par_stride, logits,
                       stats, acc_len, next_tok, path, (cudaStream_t)stream);
}

extern "C" int spec_profile(spec_model* m, int32_t enable) {
    if (!m) return set_error(SPEC_ERR_ARG, "spec_profile: null model");
    m->prof_on = enable != 0;
    if (m->prof_on) {
        m->prof_n = 0;
        SPEC_CUDA(cudaMemset(m->prof_kv, 0, sizeof(unsigned long long)), "profile reset");
    }
    return SPEC_OK;
}

extern "C" int spec_profile_read(spec_model* m, int32_t kind, double* total_ms, double* bytes, int32_t* launches) {
    if (!m || !total_ms || !bytes || !launches) return set_error(SPEC_ERR_ARG, "spec_profile_read: null pointer");
    double ms = 0.0, by = 0.0;
    int n = 0;
    for (size_t i = 0; i < m->prof_n; ++i) {
        if (m->prof_kind[i] != kind) continue;
        SPEC_CUDA(cudaEventSynchronize(m->prof_ev[2 * i + 1]), "profile sync");
        float t = 0.f;
        SPEC_CUDA(cudaEventElapsedTime(&t, m->prof_ev[2 * i], m->prof_ev[2 * i + 1]), "profile elapsed");
        ms += t;
        by += m->prof_bytes[i];
        ++n;
    }
    if (kind == PROF_GEMM && n > 0) {
        // K/V bytes read by attention phases of the chains (counted on the device)
        unsigned long long kvb = 0;
        SPEC_CUDA(cudaMemcpy(&kvb, m->prof_kv, sizeof(kvb), cudaMemcpyDeviceToHost), "profile read");
        by += (double)kvb;
    }
    *total_ms = ms;
    *bytes = by;
    *launches = n;
    return SPEC_OK;
}

extern "C" int spec_launch_count(spec_model* m, int64_t* count) {
    if (!m || !count) return set_error(SPEC_ERR_ARG, "spec_launch_count: null pointer");
    *count = m->launches;
    return SPEC_OK;
}
