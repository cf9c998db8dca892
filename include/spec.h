/*
 * spec.h -- C ABI of libspec.so, the GB300 (sm_103a) verification path of
 * speculative decoding with layer-skip self-drafting.
 *
 * What the calls compute (one round at committed length s, last emitted
 * token t0 not yet in the cache):
 *   spec_draft   k+1 passes of layers [0, L) (one row per sequence each):
 *                t0, d_1, ..., d_k at positions s .. s+k; the first k passes
 *                go through the final RMSNorm and the shared LM head and
 *                pick d_{j+1} = argmax.  Writes layers [0, L) of the KV cache
 *                and returns the layer-L hidden state of all k+1 rows
 *                ("self-speculative decoding" page, m.lqnn.cn/news/278124,
 *                section 2.1 layer skip and KV reuse, section 4.2 draft stage).
 *   spec_verify  layers [L, N) over the candidate rows -- a chain (row j sees
 *                the context and rows 0..j) or a level-order token tree (a
 *                node sees the context, its ancestors and itself; position id
 *                s + depth) -- then final norm and LM head; optionally fused
 *                greedy acceptance (same page, sections 2.1, 4.3; FlashSpec
 *                page, lnrk.cn/news/47842, sections 2.2, 3.2, 4.1, 5.2).
 *   spec_accept  rejection sampling: keep x with probability min(1, p/q),
 *                else draw from max(0, p - q) normalised (p when that is all
 *                zero); all kept -> bonus draw from the last target row
 *                (self-speculative decoding page, sections 2.4 and 4.3).
 *   kv_commit    keep the accepted rows, drop the rest: length s + a + 1,
 *                tree paths compacted into consecutive slots (same page,
 *                sections 3.3 and 4.5; FlashSpec page, section 4.1).
 *   spec_schedule_k  confidence-scheduled draft length (DSpark page,
 *                0539edu.com/news/4524681, sections 2.2 and 2.3).
 *
 * Conventions
 *   - Every pointer argument documented "device" is a CUDA device pointer
 *     on the current device; "host" is ordinary host memory.  The caller owns
 *     every buffer it passes; the library only borrows it for the call (or,
 *     for asynchronous calls, until the work on `stream` completes).
 *   - The library owns the packed weights (spec_model), the KV cache and
 *     lengths (spec_kv) and its internal workspaces.  Calls on one model
 *     must be ordered on one stream: the workspaces are shared.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls
 *     marked "async" only enqueue work; calls marked "sync" return after the
 *     stream has drained.
 *   - Return value: SPEC_OK (0) or a negative SPEC_ERR_* code; the message
 *     of the last error on the calling thread is spec_last_error().  No C++
 *     exception crosses the ABI.  Errors found on the device (token id out of
 *     range, KV capacity exceeded, a bounded wait that ran out) set the
 *     model's device error word, read and cleared by spec_device_error().
 *   - Layouts are row-major; "[a][b]" means b is contiguous.
 */
#ifndef SPEC_H
#define SPEC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_OK               0
#define SPEC_ERR_ARG         -1   /* bad argument (null, size, range)           */
#define SPEC_ERR_CAPACITY    -2   /* rows, batch or context beyond the limits   */
#define SPEC_ERR_CUDA        -3   /* a CUDA runtime call failed                 */
#define SPEC_ERR_DEVICE      -4   /* device error word was set                  */
#define SPEC_ERR_UNSUPPORTED -5   /* shape or mode the library does not handle  */

#define SPEC_DTYPE_F32  0
#define SPEC_DTYPE_BF16 1

/* device error word bits (spec_device_error) */
#define SPEC_DEVERR_TOKEN     1   /* a token id outside [0, vocab)              */
#define SPEC_DEVERR_CAPACITY  2   /* a row slot at or beyond the KV capacity    */
#define SPEC_DEVERR_TIMEOUT   4   /* a bounded pipeline wait ran out            */
#define SPEC_DEVERR_POSITION  8   /* a position id beyond the rotary table      */
#define SPEC_DEVERR_TREE     16   /* a device tree parent outside [0, node)     */

typedef struct spec_model spec_model;
typedef struct spec_kv spec_kv;

/* Llama-style decoder: RMSNorm, rotate-half RoPE, GQA attention, SwiGLU FFN,
 * untied LM head, no biases.  Limits of the library: head_dim in {64, 128};
 * n_heads a multiple of n_kv_heads; d_model, n_heads*head_dim and d_ff
 * multiples of 64; bf16 weights run on the tcgen05 tensor-core GEMM, f32
 * weights on a CUDA-core GEMM. */
typedef struct spec_model_config {
    int32_t n_layers;      /* N                                                  */
    int32_t d_model;       /* d                                                  */
    int32_t n_heads;       /* H query heads                                      */
    int32_t n_kv_heads;    /* Hkv                                                */
    int32_t head_dim;      /* hd                                                 */
    int32_t d_ff;          /* F                                                  */
    int32_t vocab;         /* V                                                  */
    int32_t exit_layer;    /* L: the draft runs layers [0, L), 0 <= L < N        */
    int32_t dtype;         /* SPEC_DTYPE_F32 or SPEC_DTYPE_BF16 (all weights)    */
    int32_t max_rows;      /* most candidate rows of all sequences in one call   */
    int32_t max_batch;     /* most sequences in one call                         */
    int32_t max_position;  /* every position id must be < max_position           */
    float   rms_eps;       /* RMSNorm epsilon                                    */
    float   rope_theta;    /* RoPE base                                          */
} spec_model_config;

/* Per-row summary of a target logits row. */
typedef struct spec_row_stats {
    float   top1;          /* largest logit                                      */
    float   top2;          /* second largest logit (another index)               */
    float   sum_exp;       /* sum over the vocabulary of exp(logit - top1)       */
    int32_t argmax;        /* lowest index holding top1                          */
} spec_row_stats;

/* Order of the weight pointers given to spec_model_create. */
#define SPEC_W_EMBED       0   /* [V][d]                                   */
#define SPEC_W_LM_HEAD     1   /* [V][d]                                   */
#define SPEC_W_FINAL_NORM  2   /* [d]                                      */
#define SPEC_W_LAYER0      3   /* then 9 per layer l at 3 + 9*l + j:       */
#define SPEC_WL_ATTN_NORM  0   /* [d]                                      */
#define SPEC_WL_Q          1   /* [H*hd][d]                                */
#define SPEC_WL_K          2   /* [Hkv*hd][d]                              */
#define SPEC_WL_V          3   /* [Hkv*hd][d]                              */
#define SPEC_WL_O          4   /* [d][H*hd]                                */
#define SPEC_WL_FFN_NORM   5   /* [d]                                      */
#define SPEC_WL_GATE       6   /* [F][d]                                   */
#define SPEC_WL_UP         7   /* [F][d]                                   */
#define SPEC_WL_DOWN       8   /* [d][F]                                   */
#define SPEC_W_COUNT(n_layers) (3 + 9 * (n_layers))

/* Bounds of the confidence-scheduled draft length (DSpark page, 2.2-2.3). */
typedef struct spec_k_schedule {
    int32_t min_k, max_k;  /* clamp range of k                                   */
    double  low, high;     /* confidence thresholds mapped to min_k and max_k    */
    double  decay;         /* EMA decay of the acceptance rate                   */
    int32_t first_reject_min;  /* nonzero: a round whose first draft token was
                              rejected (acc_len 0) sets k to min_k (DSpark 2.3) */
} spec_k_schedule;

/* Additive increase / decrease of k over a sliding window ("self-speculative
 * decoding" page, m.lqnn.cn/news/278124, section 3.2): alpha = kept / drafted
 * draft tokens over the last `window` rounds; alpha > up -> k + 1, alpha <
 * down -> k - 1 (strict, every round), clamped to [min_k, max_k].  The
 * thresholds are exact fractions. */
typedef struct spec_aimd_schedule {
    int32_t window;              /* rounds in the window, 1..256                  */
    int32_t min_k, max_k;
    int32_t up_num, up_den;      /* e.g. 85 / 100                                 */
    int32_t down_num, down_den;  /* e.g. 7 / 10                                   */
} spec_aimd_schedule;

/* Last error message of the calling thread ("" if none).  The string stays
 * valid until the next failing call on the same thread. */
const char* spec_last_error(void);

/* Number of SMs and compute capability of the current device (sync). */
int spec_device_info(int32_t* num_sms, int32_t* cc_major, int32_t* cc_minor);

/* Create a model on the current device from weights in the order of
 * SPEC_W_* (`weights`: host array of SPEC_W_COUNT(n_layers) device
 * pointers, each tensor of cfg->dtype, row-major [out][in]).  The library
 * packs them into its own memory (fused Q|K|V rows, gate/up rows
 * interleaved in blocks of 64), builds the rotary tables and workspaces, and
 * synchronises `stream` before returning: the caller may free its copies
 * afterwards.  sync.  Errors: ARG (null / non-positive sizes), UNSUPPORTED
 * (outside the limits above), CUDA (allocation or copy failed).
 * The decoder is a Llama-style target: a 7B-class model in the self-speculative
 * decoding page, section 4.1; a 7B LLaMA architecture in the FlashSpec page,
 * section 2.1.
 */
int spec_model_create(const spec_model_config* cfg, const void* const* weights,
                      void* stream, spec_model** out);
void spec_model_destroy(spec_model* m);

/* Read and clear the model's device error word (SPEC_DEVERR_* bits). sync. */
int spec_device_error(spec_model* m, int32_t* host_bits);

/* Failure injection for tests of the bounded-wait abort path (no counterpart
 * in the pages' method).  The next GEMM chain launch of this model that has
 * two or more phases runs with CTA `cta` withholding its arrival at the grid
 * barrier after the first phase, and every grid-barrier wait of that launch
 * gives up after `wait_ns` nanoseconds instead of 2 s.  The launch then ends
 * through its abort path: the waiting CTAs raise SPEC_DEVERR_TIMEOUT, let
 * their copies in flight land, drain their MMAs, free their tensor memory and
 * exit; the last one out resets the barrier counters, so the next call runs
 * normally.  That call's results are invalid.  Nothing faults or hangs: the
 * kernel returns within about `wait_ns`.  cta in [0, SMs), wait_ns in
 * [1e6, 2e9].  One-shot; host only. */
int spec_test_stall_next_chain(spec_model* m, int32_t cta, int64_t wait_ns);

/* Exit layer L of the calls that follow: the drafts run layers [0, L), a
 * verify from h_in runs layers [L, N).  Lets L follow the committed context
 * length, shallower on short contexts and deeper on long ones.  The value is
 * read when a call is enqueued: change it between rounds, never between a
 * round's draft and its verify (h_in must come from a draft at the same L).
 * A round writes every layer of its rows (layers [0, L) in the draft,
 * [L, N) in the verify), so a later round at another L finds its whole
 * context.  0 <= exit_layer < n_layers (0: verify from embeddings only).
 * Host only.  Self-speculative decoding page, m.lqnn.cn/news/278124,
 * section 5.3.
 */
int spec_set_exit_layer(spec_model* m, int32_t exit_layer);

/* KV cache for `batch` sequences of up to `max_ctx` slots each, every layer,
 * K and V, in the model dtype: layout [layer][seq][kv_head][slot][hd]
 * (one allocation, never grown).  Lengths start at 0.  sync.
 * One static allocation, as the FlashSpec page, lnrk.cn/news/47842, section
 * 4.3 advises.
 */
int spec_kv_create(spec_model* m, int32_t batch, int32_t max_ctx, spec_kv** out);

/* Paged KV cache ("self-speculative decoding" page, m.lqnn.cn/news/278124,
 * sections 3.3 and 4.5: rollback by page, compaction): a pool of n_pages
 * pages of `page` slots (a power of two, at least 64) per layer, shared by the batch
 * sequences, each addressing up to max_ctx slots through its page table.
 * Calls that write slots take the pages they need from the pool first (in
 * sequence order, deterministic); kv_commit and spec_kv_set_lengths return
 * the pages past the committed lengths (page-granular rollback); a tree
 * commit compacts the accepted path through the table.  An empty pool sets
 * SPEC_DEVERR_CAPACITY.  Every other call behaves as with spec_kv_create and
 * gives the same results bit for bit.  sync. */
int spec_kv_create_paged(spec_model* m, int32_t batch, int32_t max_ctx, int32_t page, int32_t n_pages,
                         spec_kv** out);

/* Pages left in the pool of a paged cache (0 for a contiguous one).  sync. */
int spec_kv_free_pages(spec_kv* kv, int32_t* host_free, void* stream);

/* Page table, host int32 [batch][ceil(max_ctx / page)] (-1: no page; a
 * contiguous cache reports page b for sequence b).  sync. */
int spec_kv_page_table(spec_kv* kv, int32_t* host_table, void* stream);

/* Raw contents of one physical page of the pool, read without the page
 * table: host buffer [n_kv_heads][page][head_dim] of the model dtype (bf16
 * or f32) for K (which = 0) or V (which = 1) of `layer`.  A contiguous cache
 * is read as pages of max_ctx slots, page b holding sequence b.  For
 * inspection (tests, debugging): lets a caller check where the page table
 * put each slot.  SPEC_ERR_ARG for a page, layer or `which` out of range.
 * sync.  Self-speculative decoding page, m.lqnn.cn/news/278124, section 3.3
 * (the pages a rollback keeps). */
int spec_kv_read_page(spec_kv* kv, int32_t which, int32_t layer, int32_t page, void* host_dst, void* stream);
void spec_kv_destroy(spec_kv* kv);

/* Committed lengths: set from / copy to host int32 [batch].  sync. */
int spec_kv_set_lengths(spec_kv* kv, const int32_t* host_len, void* stream);
int spec_kv_get_lengths(spec_kv* kv, int32_t* host_len, void* stream);

/* Copy KV rows between the cache and a device buffer laid out
 * [n_layers][n_slots][Hkv][hd] in the model dtype, for sequence `seq`,
 * layers [layer0, layer0+n_layers), slots [slot0, slot0+n_slots).  Used to
 * load a synthetic committed context and to inspect the cache.  Lengths
 * are not changed.  async. */
int spec_kv_import(spec_kv* kv, int32_t seq, int32_t layer0, int32_t n_layers,
                   int32_t slot0, int32_t n_slots, const void* k, const void* v,
                   void* stream);
int spec_kv_export(spec_kv* kv, int32_t seq, int32_t layer0, int32_t n_layers,
                   int32_t slot0, int32_t n_slots, void* k, void* v, void* stream);

/* Causal pass of all layers over `n` prompt tokens (device int32 [n]) of
 * sequence `seq`, appended at its committed length, which then grows by n.
 * Optional outputs for the last row: `last_logits` (device f32 [V]) and
 * `next_tok` (device int32 [1], its argmax).  async. */
int spec_prefill(spec_model* m, spec_kv* kv, int32_t seq, const int32_t* tokens,
                 int32_t n, float* last_logits, int32_t* next_tok, void* stream);

/* Greedy layer-skip draft for sequences [0, batch) with draft length k.
 *   t0       device int32 [batch]    last emitted token of each sequence
 *   cand     device int32 [batch][k+1]  out: cand[b][0] = t0[b], cand[b][j] = d_j
 *   h_L      device f32 [batch][k+1][d] out: layer-L residual state of each row
 *   draft_logits device f32 [batch][k][V] out, nullable: the k draft rows
 * Writes KV layers [0, L) at slots s_b .. s_b+k; lengths unchanged.  async.
 * Requires exit_layer >= 1.
 * Self-speculative decoding page, m.lqnn.cn/news/278124, sections 2.1 and 4.2.
 */
int spec_draft(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* t0, int32_t k,
               int32_t* cand, float* h_L, float* draft_logits, void* stream);

/* Sampling layer-skip draft ("self-speculative decoding" page, sections 2.4
 * and 4.2): as spec_draft, but d_{j+1} is drawn from q_j = softmax(draft
 * logits / temperature) with the integer inverse-CDF sampler of spec_sample
 * driven by u_draft[b][j].
 *   temperature  > 0, finite; the verifier's p must use the same value
 *   u_draft  device f32 [batch][k], each m * 2^-24 with integer m in [0, 2^24)
 *   q        device f32 [batch][k][V] out: the draft distributions (whole,
 *            never top-p cut), the q of spec_accept
 *   cand, h_L, draft_logits as for spec_draft (draft_logits nullable).
 * batch <= max_batch; vocab <= 53248.  async. */
int spec_draft_sample(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* t0, int32_t k,
                      float temperature, const float* u_draft, int32_t* cand, float* h_L,
                      float* q, float* draft_logits, void* stream);

/* Layer-skip draft of a level-order token tree per sequence (FlashSpec page,
 * lnrk.cn/news/47842, sections 2.2 and 6.2, with the self-speculative
 * decoding page's first-L-layer draft): level by level, layers [0, L) run on
 * the tree's nodes (node i in slot s_b + i at position s_b + depth(i), seeing
 * the committed context, its ancestors and itself) and the shared LM head
 * gives each node of the level its children: the k-th child (by node index)
 * takes the k-th highest draft logit, ties to the lower token id.  A last
 * pass gives every node its layer-L state.  Writes KV layers [0, L) at slots
 * s_b .. s_b + n_nodes - 1; lengths unchanged.
 *   t0           device int32 [batch]: each tree's root token
 *   tree_parent  host int32 [n_nodes]: parent[0] = -1, parent[i] in [0, i),
 *                depths non-decreasing (level order), at most 16 children a node
 *   tokens       device int32 [batch][n_nodes] out (tokens[b][0] = t0[b])
 *   h_L          device f32 [batch][n_nodes][d] out: layer-L state of every node
 *   logits       device f32 [batch * n_nodes][V]: scratch for the draft rows
 * Follow with spec_verify(h_in = h_L, tree_parent, tokens) and kv_commit with
 * the accepted path.  batch * n_nodes <= max_rows; 2 <= n_nodes <= 64.  async. */
int spec_draft_tree(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* t0,
                    const int32_t* tree_parent, int32_t n_nodes, int32_t* tokens,
                    float* h_L, float* logits, void* stream);

/* Verification forward of the candidate rows of sequences [0, batch).
 *   n_rows   host int32 [batch]: rows of sequence b (chain: k_b+1; tree:
 *            node count).  Sum <= max_rows, each <= 64.
 *   h_in     device f32 [batch][h_stride][d]: layer-L state of each row (from
 *            spec_draft); the forward runs layers [L, N).  NULL: rows are
 *            embedded from `tokens` and the forward runs layers [0, N).
 *   tokens   device int32 [batch][tok_stride]: row tokens (row 0 = t0, then
 *            the draft tokens or tree nodes in level order).
 *   tree_parent  host int32 [n_rows[0]] parent of each node (parent[0] = -1,
 *            parent[i] < i), shared by all sequences; NULL = chain.
 *   logits   device f32 [sum n_rows][V], nullable: target logits.
 *   stats    device spec_row_stats [sum n_rows], nullable.
 *   acc_len, next_tok  device int32 [batch], nullable (both or neither):
 *            fused greedy acceptance -- chain: leading draft tokens equal to
 *            the previous row's argmax; tree: deepest node whose whole path
 *            matches (ties to the lowest node index); next_tok = argmax of
 *            the last accepted row.
 *   path     device int32 [batch][64]: accepted rows root first (tree mode
 *            with fused acceptance; nullable in chain mode).
 * Writes KV of the forward's layers at slots s_b .. s_b+n_rows[b]-1; lengths
 * unchanged.  async.
 * Self-speculative decoding page, sections 2.1 and 4.3; FlashSpec page,
 * sections 2.2, 3.2, 4.1 and 5.2.
 */
int spec_verify(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* n_rows,
                const float* h_in, int32_t h_stride, const int32_t* tokens,
                int32_t tok_stride, const int32_t* tree_parent, float* logits,
                spec_row_stats* stats, int32_t* acc_len, int32_t* next_tok,
                int32_t* path, void* stream);

/* Layer-skip draft of a token tree whose width follows the draft's
 * confidence, one tree a sequence (FlashSpec page, lnrk.cn/news/47842,
 * section 6.2: nodes the draft is sure of are not widened, unsure ones get
 * more branches).  As spec_draft_tree, level by level, but node i of level l
 * gets c children: its c best draft tokens (ties to the lower id), c the
 * fewest whose draft probabilities (softmax of the draft logits, float32)
 * add up to at least `mass`, 1 <= c <= branching[l].  Children are numbered
 * in level order after the nodes so far.  mass <= 0 gives a chain of depth
 * `depth`; mass > 1 the full tree of `branching`.
 *   t0         device int32 [batch]: each tree's root token
 *   branching  host int32 [depth]: at most this many children a node of
 *              level l, each in [1, min(16, V)]; the full tree has n_max <= 64
 *              nodes
 *   tokens, parents  device int32 [batch][n_max] out: node tokens (tokens[b][0]
 *              = t0[b]) and parents (parents[b][0] = -1); entries at and past
 *              n_nodes[b] are padding (token 0, parent 0)
 *   n_nodes    device int32 [batch] out: nodes of each tree
 *   h_L        device f32 [batch][n_max][d] out: layer-L state of every node
 *   logits     device f32 [batch * n_max][V]: scratch for the draft rows
 * Every draft pass runs over the full tree's n_max rows a sequence (the node
 * counts stay on the device); KV layers [0, L) are written at slots s_b ..
 * s_b + n_max - 1, lengths unchanged.  Follow with spec_verify_trees
 * (n_rows = n_nodes read back, h_in = h_L, strides n_max) and kv_commit with
 * the accepted path.  batch * n_max <= max_rows.  async. */
int spec_draft_tree_dynamic(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* t0,
                            const int32_t* branching, int32_t depth, float mass,
                            int32_t* tokens, int32_t* parents, int32_t* n_nodes, float* h_L,
                            float* logits, void* stream);

/* spec_verify with one tree a sequence: the parents of sequence b's nodes
 * are parents[b * par_stride + i] on the device (parent[0] ignored, the
 * others in [0, i); a parent outside that range sets SPEC_DEVERR_TREE and
 * reads as the root).  n_rows[b] is the node count of sequence b's tree
 * (<= par_stride).  Acceptance (acc_len, next_tok and path, all three or
 * none) runs as its own kernel after the forward, with the tree rule of
 * spec_verify.  The attention always runs as its own kernel.  async.
 * FlashSpec page, lnrk.cn/news/47842, sections 2.2 and 6.2.
 */
int spec_verify_trees(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* n_rows,
                      const float* h_in, int32_t h_stride, const int32_t* tokens,
                      int32_t tok_stride, const int32_t* parents, int32_t par_stride,
                      float* logits, spec_row_stats* stats, int32_t* acc_len,
                      int32_t* next_tok, int32_t* path, void* stream);

/* Rejection-sampling acceptance of a chain (no model needed).
 *   p      device f32 [batch][k+1][vocab]  target probabilities
 *   q      device f32 [batch][k][vocab]    draft probabilities
 *   draft  device int32 [batch][draft_stride]  draft tokens in columns 0..k-1
 *          (draft_stride 0 means k; cand + 1 with stride k+1 reads the
 *          draft tokens of spec_draft's candidate rows)
 *   u      device f32 [batch][k+1]         uniforms, each m * 2^-24, m in [0, 2^24)
 *   acc_len, next_tok  device int32 [batch] out
 * Ratio test u_j * q_j(x) < p_j(x) exactly (q_j(x) = 0 rejects); the draw
 * (residual max(0, p - q) in f32, or p when that is all zero, or the bonus
 * row p_k) is an integer inverse CDF over w = floor(r * 2^32) driven by
 * u[k].  Bit-exact and deterministic.  1 <= k <= 32, vocab <= 65536; a
 * target row of all zeros (invalid input) gives next_tok -1.  async.
 * Self-speculative decoding page, m.lqnn.cn/news/278124, sections 2.4 and 4.3.
 */
int spec_accept(const float* p, const float* q, const int32_t* draft, int32_t draft_stride,
                const float* u, int32_t batch, int32_t k, int32_t vocab, int32_t* acc_len,
                int32_t* next_tok, void* stream);

/* Probability rows at a temperature, optionally cut to the top-p nucleus
 * (self-speculative decoding page, sections 2.4 and 3.4: the target row is
 * cut, the draft row stays whole).
 *   logits   device f32, row r at logits + r * lg_stride (lg_stride >= vocab)
 *   probs    device f32 out, row r at probs + r * p_stride
 *   temperature > 0: probs = softmax(logits / temperature) in f32
 *   top_p    >= 1: whole rows; else a multiple of 2^-24 in (0, 1): the row is
 *            restricted to the shortest run of tokens, by decreasing
 *            probability (ties to the lower id), whose integer weights
 *            w = floor(p * 2^32) reach ceil(m * S / 2^24) (S = sum w,
 *            top_p = m * 2^-24), then renormalised (zeros elsewhere).
 * One CTA per row, the row in shared memory: vocab <= 53248.  Rows must be
 * finite.  async. */
int spec_probs(const float* logits, int64_t lg_stride, int32_t rows, int32_t vocab,
               float temperature, float top_p, float* probs, int64_t p_stride, void* stream);

/* One integer inverse-CDF draw per probability row: w = floor(r * 2^32),
 * S = sum w, t = floor(m * S / 2^24) for u = m * 2^-24, token = smallest x
 * whose inclusive prefix sum of w exceeds t (-1 for a row of zero weights).
 *   probs device f32, row r at probs + r * p_stride; u device f32 [rows];
 *   tokens device int32 [rows] out.  vocab <= 53248.  async.
 * The draws of the self-speculative decoding page, sections 2.4 and 4.3, in an
 * exact integer form.
 */
int spec_sample(const float* probs, int64_t p_stride, int32_t rows, int32_t vocab,
                const float* u, int32_t* tokens, void* stream);

/* Greedy acceptance from target logits (the unfused form of spec_verify's
 * fused acceptance).  logits device f32 [batch][n_rows][vocab]; tokens device
 * int32 [batch][n_rows]; tree_parent host int32 [n_rows] or NULL (chain);
 * path device int32 [batch][64], nullable in chain mode.  async.
 * Self-speculative decoding page, section 4.3; FlashSpec page, section 4.1.
 */
int spec_accept_greedy(const float* logits, const int32_t* tokens,
                       const int32_t* tree_parent, int32_t batch, int32_t n_rows,
                       int32_t vocab, int32_t* acc_len, int32_t* next_tok,
                       int32_t* path, void* stream);

/* Commit the accepted rows of sequences [0, batch): acc_len device int32
 * [batch].  Chain (path NULL): length s_b + acc_len[b] + 1.  Tree: path
 * device int32 [batch][path_stride] (root first) -- the rows of depth
 * 1..acc_len[b] move from slot s_b + path[b][d] to slot s_b + d in every
 * layer, then the length becomes s_b + acc_len[b] + 1.  async.
 * Self-speculative decoding page, sections 3.3 and 4.5; FlashSpec page,
 * section 4.1.
 */
int kv_commit(spec_kv* kv, int32_t batch, const int32_t* acc_len, const int32_t* path,
              int32_t path_stride, void* stream);

/* Probabilities of the two largest logits of each row, from row summaries:
 * out[2r] = 1 / sum_exp, out[2r+1] = exp(top2 - top1) / sum_exp (float64).
 * stats device [rows]; out device f64 [rows][2].  async.
 * The confidence inputs of the DSpark page, 0539edu.com/news/4524681, section 2.2.
 */
int spec_row_probs(const spec_row_stats* stats, int32_t rows, double* out, void* stream);

/* Confidence-scheduled draft length, one round, sequences [0, batch):
 *   top_probs device f64 [sum n_rows][2]: top-1 and top-2 target probabilities
 *            of every verified row (spec_row_probs)
 *   n_rows   host int32 [batch]: k_b + 1 rows of sequence b (k_b >= 1)
 *   acc_len  device int32 [batch]; ema device f64 [batch] (updated in place)
 *   k_next   device int32 [batch] out; conf device f64 [batch] out, nullable
 * acceptance = a/k_b; ema = decay*ema + (1-decay)*acceptance;
 * conf = 0.4*mean(top1) + 0.3*min(5*mean(top1 - top2), 1) + 0.3*ema;
 * k_next = clamp(trunc(min_k + (max_k-min_k)*(conf-low)/(high-low)), min_k, max_k).
 * Float64 with one rounding per written operation, left to right, no
 * contraction; means are left-to-right sums divided by the count.  async.
 * DSpark page, 0539edu.com/news/4524681, sections 2.2 and 2.3.
 */
int spec_schedule_k(const double* top_probs, const int32_t* n_rows, const int32_t* acc_len,
                    double* ema, int32_t batch, const spec_k_schedule* sch, int32_t* k_next,
                    double* conf, void* stream);

/* One round of the additive schedule, sequences [0, batch):
 *   acc_len  device int32 [batch]: draft tokens kept this round
 *   k_cur    device int32 [batch]: draft length of this round
 *   state    device int32 [batch][2 * window + 2]: each sequence's window
 *            (count, next slot, kept[window], drafted[window]); zero it
 *            before the first round
 *   k_next   device int32 [batch] out.  async.
 * Self-speculative decoding page, m.lqnn.cn/news/278124, section 3.2.
 */
int spec_schedule_aimd(const int32_t* acc_len, const int32_t* k_cur, int32_t* state, int32_t batch,
                       const spec_aimd_schedule* sch, int32_t* k_next, void* stream);

/* Draft length shrinking with the generated count (speculative decoding
 * principles and practice page, intelliparadigm.com/article/weixin_33702545/
 * 2059090, section 3.3): k_next = max(1, round(k_max * (1 - t / T))) in
 * float64, rounded to nearest with ties to even.
 *   generated device int32 [batch]: t, tokens generated so far
 *   total     device int32 [batch]: T, the predicted total (>= 1; smaller
 *             values give 1)
 *   k_next    device int32 [batch] out.  async. */
int spec_schedule_decay(const int32_t* generated, const int32_t* total, int32_t batch, int32_t k_max,
                        int32_t* k_next, void* stream);

/* spec_verify without any device memory of its own per call: same arguments,
 * results and stream semantics as spec_verify.  This entry point has no
 * counterpart in the method the pages describe.  It is for callers that
 * cannot call cudaMalloc where they verify: a serving runtime that hands all
 * of the device's memory to its own pool at start-up (an allocation at verify
 * time would fail or take memory the pool owns), or a latency-critical loop
 * that cannot afford the device-wide synchronisation that cudaMalloc and
 * cudaFree may imply.  The call's scratch -- the GEMM split-K partial tiles
 * and arrival counters and the attention split partials and counters -- comes
 * from a 32 MiB static __device__ array that every GPU loading the library
 * keeps until the process exits.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) and caches it; make that
 * first call before any stream capture.  The array is shared by every call
 * and keeps the last call's contents, so each call clears the counters it
 * needs on `stream`; calls that overlap on the GPU (other streams, other
 * threads) race on the array and must not be issued.  Returns
 * SPEC_ERR_CAPACITY with a message when a call needs more scratch than the
 * array holds, and checks its other arguments as spec_verify does before it
 * enqueues anything.  Makes no cudaMalloc / cudaFree or other allocating
 * call.  async. */
int spec_verify_noalloc(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* n_rows,
                        const float* h_in, int32_t h_stride, const int32_t* tokens,
                        int32_t tok_stride, const int32_t* tree_parent, float* logits,
                        spec_row_stats* stats, int32_t* acc_len, int32_t* next_tok,
                        int32_t* path, void* stream);

/* Tracing.  spec_profile(m, 1) starts a fresh record: from then on every GEMM
 * and attention launch of this model is bracketed by CUDA events on its
 * stream, with the launch's algorithmic bytes (weights once, activation rows
 * in and out).  spec_profile(m, 0) stops recording.  spec_profile_read sums
 * the recorded launches of one kind (0 GEMM, 1 attention): total device
 * milliseconds, bytes and launch count; sync.  spec_launch_count returns the
 * number of kernels this model has launched since it was created. */
int spec_profile(spec_model* m, int32_t enable);
int spec_profile_read(spec_model* m, int32_t kind, double* total_ms, double* bytes, int32_t* launches);
int spec_launch_count(spec_model* m, int64_t* count);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_H */
