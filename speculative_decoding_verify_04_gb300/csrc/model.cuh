// Library-internal structures shared by the translation units of libspec.so.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "common.cuh"

namespace spec {

constexpr int kMaxSeqRows = 64;       // rows of one sequence in one call
constexpr int kMaxPlanBatch = 256;    // sequences described in one plan
constexpr int kTileN = 128;           // W rows (output features) per GEMM tile
constexpr int kTileK = 64;            // K per pipeline stage: 64 bf16 = 128 B rows
constexpr int kMaxTPad = 256;         // activation rows per tcgen05 pass (MMA N)
constexpr int kRowChunk = 16;         // epilogue granularity (tcgen05.ld .x16)

enum EpiKind : int { EPI_QKV = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_HEAD = 3 };
enum HeadMode : int { HEAD_STATS = 0, HEAD_DRAFT = 1, HEAD_ACCEPT_CHAIN = 2, HEAD_ACCEPT_TREE = 3 };

// Row plan of one forward call: rows of all sequences back to back.
struct RowPlan {
    int* row_seq;      // [max_rows] sequence of the row
    int* row_slot;     // [max_rows] KV slot written by the row
    int* row_pos;      // [max_rows] rotary position id
    int* row_local;    // [max_rows] index of the row within its sequence
    int* seq_row0;     // [max_batch] first row of the sequence
    int* seq_nrows;    // [max_batch] rows of the sequence
    int* seq_base;     // [max_batch] committed length when the plan was made
    int* tree_parent;  // [kMaxSeqRows] parent of each local row (-1 root); tree mode only
    int* tree_depth;   // [kMaxSeqRows]
};

// Parameters of the plan kernel, passed by value.
// Where slot s of sequence b lives in the cache: page table[b * max_pages +
// s / page], row s % page of that page; a page holds `page` slots of every KV
// head of one layer ([layer][page][kv head][slot in page][hd]).  A contiguous
// cache is the special case of one page per sequence (page = capacity,
// table = 0, 1, ..., batch - 1).
struct KVPages {
    const int* table;     // [kv batch][max_pages], -1 where no page is held
    int page;             // slots a page (a power of two for paged caches)
    int max_pages;        // pages a sequence can address
    int n_pages;          // pages a layer holds
    int shift;            // log2(page) for paged caches; -1: contiguous (sequence b is page b)
};

// Row of slot `slot` (sequence seq, KV head kvh) counted inside one layer's
// block of the cache; -1 when the slot's page is not held.  A contiguous
// cache needs no table read.
SPEC_DEV long long kv_row_in_layer(const KVPages& p, int n_kv_heads, int seq, int kvh, int slot) {
    if (p.shift < 0) return ((long long)seq * n_kv_heads + kvh) * p.page + slot;
    const int blk = slot >> p.shift;
    const int pg = p.table[(size_t)seq * p.max_pages + blk];
    if (pg < 0) return -1;
    return ((long long)pg * n_kv_heads + kvh) * p.page + (slot & (p.page - 1));
}
// The same row counted from the start of the cache (layer blocks of n_pages pages).
SPEC_DEV long long kv_row(const KVPages& p, int n_kv_heads, int layer, int seq, int kvh, int slot) {
    const long long r = kv_row_in_layer(p, n_kv_heads, seq, kvh, slot);
    return r < 0 ? -1 : (long long)layer * p.n_pages * n_kv_heads * p.page + r;
}

struct PlanParams {
    int batch;
    int mode;                        // 0 chain, 1 tree, 2 one-row-per-sequence draft pass
    int pass;                        // draft pass index j (mode 2)
    int n_rows[kMaxPlanBatch];
    int parent[kMaxSeqRows];
    int depth[kMaxSeqRows];
};

struct LayerWeights {
    void* qkv;       // [(H + 2 Hkv) hd][d]
    void* o;         // [d][H hd]
    void* gu;        // [2 * ceil(F/64) * 64][d]: per 64-block: 64 gate rows then 64 up rows
    void* down;      // [d][F]
    float* attn_g;   // [d]
    float* ffn_g;    // [d]
    CUtensorMap tm_qkv, tm_o, tm_gu, tm_down;
};

struct GemmShape {
    int N;           // output features (rows of W, packed)
    int K;           // input features
};


// One CTA per row: softmax at a temperature (or rows given as probabilities),
// optional top-p nucleus, optional integer inverse-CDF draw (sample.cu).
constexpr int kSampMaxVocab = 53248;        // the row lives in shared memory (208 KB)
struct SampleArgs {
    const float* in; long long in_stride;   // logits (softmax) or probabilities (draw only)
    float* out; long long out_stride;       // nullable: the row's probabilities
    const float* u; int u_stride;           // nullable: uniform of row r at u[r * u_stride]
    int* tok; int tok_stride;               // drawn token of row r at tok[r * tok_stride]
    int rows, V;
    float temp;                             // softmax at this temperature; <= 0: rows are probabilities
    unsigned top_p_m;                       // 0: whole row; else the nucleus of top_p = m * 2^-24
    int* err;                               // nullable device error word
};

int launch_sample_rows(const SampleArgs& a, bool pdl, cudaStream_t st);

}  // namespace spec

struct spec_model {
    spec_model_config cfg;
    int device = 0;
    int num_sms = 0;
    bool bf16 = true;
    size_t elem = 2;                 // bytes per weight / KV element
    int qkv_n = 0, gu_n = 0;         // packed output widths
    int max_rows_pad = 0;            // max_rows rounded up to 16
    int x_cols = 0;                  // widest activation row (d, H hd, F)

    char* wmem = nullptr;            // packed weights (one allocation)
    void* embed = nullptr;           // [V][d]
    void* head = nullptr;            // [V][d]
    float* final_g = nullptr;        // [d]
    CUtensorMap tm_head;
    std::vector<spec::LayerWeights> layers;
    float* rope_cos = nullptr;       // [max_position][hd/2]
    float* rope_sin = nullptr;

    char* ws = nullptr;              // workspace (one allocation)
    size_t ws_bytes = 0;
    float* h = nullptr;              // [max_rows][d] f32 residual stream
    // GEMM inputs, model dtype; bf16 models keep [2][max_rows_pad][K]: hi rows then lo rows
    void* x_in = nullptr;            // [max_rows_pad][d]   gained residual
    void* x_attn = nullptr;          // [max_rows_pad][H hd] attention output
    void* x_act = nullptr;           // [max_rows_pad][F]   SwiGLU output
    float* q = nullptr;              // [max_rows][H hd] rotated, pre-scaled queries
    float* ss_part = nullptr;        // [d/128][max_rows] per-tile sums of squares of h
    spec_row_stats* stat_part = nullptr;  // [ceil(V/128)][max_rows]
    spec_row_stats* row_stats = nullptr;  // [max_rows]
    float* draft_lg = nullptr;       // [max_batch][V] draft logits of a sampling pass
    float* gemm_part = nullptr;      // split-K partial tiles
    size_t gemm_part_floats = 0;
    int* counters = nullptr;         // tile arrival counters, then chain barrier, chain exits, head tiles
                                     // (all zero between launches)
    int n_counters = 0;
    float* attn_part = nullptr;      // attention split partials
    size_t attn_part_floats = 0;
    int* attn_counters = nullptr;
    int n_attn_counters = 0;
    int* err = nullptr;              // device error word
    int* scratch_i32 = nullptr;      // small device scratch (path, acc staging)
    spec::RowPlan plan;

    // X tensor maps by buffer (0 x_in, 1 x_attn, 2 x_act) and T_pad/16 - 1
    CUtensorMap tm_x[3][spec::kMaxTPad / 16];

    bool w_tiled = false;            // bf16: GEMM weights stored tile-major (16 KB blocks, pre-swizzled)
    bool pdl = true;                 // launch forward kernels with programmatic dependent launch
    bool chain = true;               // bf16: consecutive GEMMs of a layer share one launch
    int attn_phase = -1;             // bf16: attention as the first phase of each layer's chain:
                                     // 1 always, 0 never, -1 for calls of two or more sequences
    int test_stall_cta = -1;         // failure injection for tests (spec_test_stall_next_chain)
    unsigned long long test_wait_ns = 0;
    bool attn_ring = false;          // bf16: attention outside a chain with <= 8 query vectors per
                                     // (sequence, KV head) takes the TMA-ring kernel (measured slower
                                     // than the register-tile kernel at batch 1: off unless asked for)
    int attn_ring_pairs = 0;         // ring kernel shape: 0 one CTA an SM (8 warps), 1 two (4 warps each)

    // tracing: kernel launches issued, and (when enabled) CUDA events around
    // every GEMM / attention launch with the launch's algorithmic bytes
    long long launches = 0;
    bool prof_on = false;
    std::vector<cudaEvent_t> prof_ev;      // start/stop pairs
    std::vector<int> prof_kind;
    std::vector<double> prof_bytes;
    size_t prof_n = 0;
    unsigned long long* prof_kv = nullptr;   // device: K/V bytes read by attention phases while profiling
};

struct spec_kv {
    spec_model* m = nullptr;
    int batch = 0;
    int max_ctx = 0;
    void* k = nullptr;               // [layer][seq][kvh][slot][hd]
    void* v = nullptr;
    int* len = nullptr;              // [batch] committed lengths (device)
    // pages: a contiguous cache is one page per sequence; a paged cache shares a
    // pool of n_pages pages of `page` slots between its sequences
    bool paged = false;
    int page = 0, max_pages = 0, n_pages = 0;
    int* table = nullptr;            // [batch][max_pages] page of each block of slots, -1 if none
    int* free_pages = nullptr;       // paged: stack of free pages [n_pages], top at free_top[0]
    int* free_top = nullptr;
    spec::KVPages pages() const {
        int sh = -1;
        if (paged) { sh = 0; while ((1 << sh) < page) ++sh; }
        return spec::KVPages{table, page, max_pages, n_pages, sh};
    }
    // bf16 caches: 3-D TMA maps {head dim, seq * kvh * slot, layer} with boxes
    // of 64 dims x (8 KB / 128 B) slots, 128-byte swizzle (attention phase of the
    // GEMM chain); tmaps is false where the cache is too large to address
    alignas(64) CUtensorMap tm_k;
    alignas(64) CUtensorMap tm_v;
    bool tmaps = false;
};

namespace spec {

// error reporting (capi.cu)
int set_error(int code, const std::string& msg);
int check_cuda(cudaError_t e, const char* what);
// returns the first non-OK status of x from the enclosing function
#define SPEC_TRY(x)                          \
    do {                                     \
        int rc_ = (x);                       \
        if (rc_ != SPEC_OK) return rc_;      \
    } while (0)

// tracing (capi.cu): bracket one kernel launch with events when enabled
enum ProfKind : int { PROF_GEMM = 0, PROF_ATTN = 1 };
int prof_start(spec_model* m, cudaStream_t st);
void prof_stop(spec_model* m, int slot, cudaStream_t st, int kind, double bytes);

// tensor maps (gemm.cu)
bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer);
bool make_tmap_x(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows_pad, uint32_t tp);

// Epilogue parameters of one GEMM launch (passed by value).
struct EpiParams {
    int kind;               // EpiKind
    int T;                  // rows of this launch
    int r0;                 // first row (of the plan) of this launch
    int N;                  // real output features of the GEMM
    int layer;
    // RMSNorm row scale: rs[r] = rsqrt(sum_t ss_part[t][r] / d + eps)
    const float* ss_in;
    int ss_tiles;
    int ss_stride;
    float inv_d, eps;
    RowPlan plan;
    int* err;
    // QKV
    float* q;
    void* kc; void* vc;     // cache bases
    KVPages kvp;
    int n_heads, n_kv_heads, head_dim;
    int kv_ctx;             // slots a sequence can address
    const float* rope_cos; const float* rope_sin;
    int max_position;
    float q_scale;
    // residual
    float* h;
    const float* gain_next;
    void* x_next;
    size_t x_next_lo;       // element offset of the lo half (bf16 models)
    float* ss_out;
    // SwiGLU
    void* act;
    size_t act_lo;
    int d_model, d_ff;
    // LM head
    float* logits;          // nullable; row r goes to logits[(r - logits_row0) * logits_stride]
    int logits_stride, logits_row0;
    spec_row_stats* stat_part;
    spec_row_stats* row_stats;
    spec_row_stats* user_stats;   // nullable
    int vocab;
    int head_mode;
    int* done_counter;
    // draft / acceptance outputs
    int* cand; int cand_stride; int cand_col;   // draft: cand[seq*stride + col] = argmax
    const int* tokens;                           // acceptance: row tokens (tok_stride a sequence)
    int* acc_len; int* next_tok; int* path;
    int tok_stride;
    int batch;
};

struct GemmLaunch {
    const CUtensorMap* tmW;
    const CUtensorMap* tmX;     // unused: X maps come from the model by buffer index
    const void* W;          // f32 path
    const void* X;          // f32 path
    int x_stride;           // f32 path: elements per X row
    int N, K;
};

// gemm.cu
int launch_gemm(spec_model* m, const GemmLaunch& g, EpiParams e, int xbuf, cudaStream_t st);
// Attention over the KV cache as a phase of the GEMM chain (bf16 caches, at
// most 16 query vectors per sequence and KV head).  The key range of every
// (sequence, KV head) is cut into units of 8 KB of K (4096 / hd slots); the
// units of all pairs are split evenly over the CTAs.
struct AttnPhase {
    const float* q;          // [rows][H hd] queries, pre-scaled by 1/sqrt(hd)
    void* out;               // [rows][H hd] bf16 hi rows, then lo rows at out_lo
    size_t out_lo;
    RowPlan plan;
    int batch, kv_ctx, layer;
    int n_heads, n_kv_heads, head_dim;
    int tree;
    int linear;              // every segment has <= kAttnSimtQ query vectors: K/V arrive by plain bulk copies
                             // (rows in order) instead of swizzled tensor boxes
    const void* kc;          // cache bases (bulk copies); the page table is the phase's EpiParams kvp
    const void* vc;
    float* part;             // [CTAs][2][16][hd + 2] partial softmax states
    int* counters;           // [batch * n_kv_heads] arrivals (zero between launches)
    int* err;
    unsigned long long* kv_bytes;   // nullable: K/V bytes read are added here (profiling)
};

enum PhaseKind { PH_GEMM = 0, PH_ATTN = 1 };
constexpr int kAttnMaxQ = 16;    // attention phase: query vectors per (sequence, KV head)
constexpr int kAttnSimtQ = 2;    // up to this many: CUDA-core path, else tensor-core MMAs

// One step of a chain: a GEMM (operands, epilogue, activation buffer index)
// or an attention phase.
struct GemmStep {
    GemmLaunch g;
    EpiParams e;
    int xbuf;
    int kind = PH_GEMM;
    AttnPhase at{};
};
// Runs the GEMMs in order.  bf16 models with every step on the same rows
// (T <= kMaxTPad) run them in one launch separated by grid barriers.
int launch_gemm_chain(spec_model* m, const GemmStep* steps, int n, cudaStream_t st);
// Attention phase usable for this launch (bf16, cache maps, <= 16 queries per
// sequence and KV head, workspace large enough)?
bool attn_phase_ok(const spec_model* m, const spec_kv* kv, int batch, int max_rows_per_seq);
size_t attn_phase_part_floats(const spec_model* m);
bool make_kv_tmaps(spec_kv* kv);
size_t gemm_partial_floats_needed(const spec_model* m, int N, int K, int T_pad);
int gemm_grid(const spec_model* m, int N, int K);

// attention.cu
struct AttnParams {
    const float* q;         // [rows][H hd]
    const void* kc; const void* vc;
    void* out;              // [rows][H hd] model dtype (O-projection input)
    size_t out_lo;          // element offset of the lo half (bf16 models)
    RowPlan plan;
    int batch, kv_ctx, layer;
    int n_heads, n_kv_heads, head_dim;
    int tree;               // 0 chain, 1 tree
    KVPages kvp;
    int splits;
    float* part;
    int* counters;
    int* err;
};
int launch_attention(spec_model* m, const AttnParams& a, int max_rows_per_seq, cudaStream_t st);
// attn_ring.cu: the TMA-ring attention kernel for calls of <= 8 query vectors per
// (sequence, KV head) (bf16 caches with tensor maps, hd 64 or 128)
bool attn_ring_fits(const spec_model* m, const spec_kv* kv, int batch, int max_rows_per_seq);
int launch_attention_ring(spec_model* m, const spec_kv* kv, const AttnParams& a, cudaStream_t st);
// paged caches (no-ops for contiguous ones): pages for slots below len[b] + n[b]
// (relative) or n[b] (absolute) of sequences [0, batch); pages past the lengths back
int kv_ensure_pages(spec_kv* kv, int batch, const int* n, bool relative, cudaStream_t st);
int kv_release_pages(spec_kv* kv, int batch, cudaStream_t st);
int attn_splits(const spec_model* m, int blocks, int kv_ctx);
size_t attn_scratch_floats(const spec_model* m, int batch, int max_rows_per_seq, int kv_ctx, int* n_counters);
size_t attn_partial_floats_needed(const spec_model* m, int batch, int max_rows_per_seq);

// accept.cu
SPEC_DEV void stat_merge(spec_row_stats& a, const spec_row_stats& b);

}  // namespace spec
