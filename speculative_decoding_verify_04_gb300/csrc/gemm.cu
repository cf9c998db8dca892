// Skinny weight-streaming GEMM  Y[T, N] = X[T, K] * W[N, K]^T  with fused epilogues.
//
// Decode-time verification multiplies a handful of rows (T = k+1 .. a few
// hundred) by every weight matrix, so the kernel is a weight stream: each
// weight byte is read once from HBM and used T times ("self-speculative
// decoding" page, section 1.1: decoding is bandwidth bound at ~2 flop/byte;
// section 1.2: verifying k positions costs one weight pass instead of k).
//
// bf16 path (tcgen05): swap-AB -- a 128-row W tile is the MMA's M side and the
// activation rows are its N side (padded to a multiple of 16), so one
// tcgen05.mma.kind::f16 of M=128, N=T_pad, K=16 consumes 32 B of every W row.
// W and X tiles arrive by TMA (128-byte swizzle) into a ring of stages; one
// thread issues the MMAs, accumulators live in tensor memory.  Activations are
// kept as bf16 hi/lo pairs (x = hi + lo to ~16 bits): each k-step issues one MMA
// with the hi rows and one with the lo rows into the same f32 accumulator, so
// weights stream once and the product keeps near-f32 activation precision.  The work is
// split stream-K: the (tile, k-block) units are cut into one contiguous range
// per CTA (one CTA per SM), so every SM streams the same number of bytes.  A
// tile cut between CTAs is reduced deterministically (fixed order of the
// partial slots) by the last CTA to finish it, which then runs the epilogue.
//
// f32 path (CUDA cores): the same decomposition and epilogues; used by f32
// models (small correctness configurations).
//
// Epilogues (applied once per finished tile, on 16-row chunks in shared memory):
//   QKV    RMSNorm row scale, rotate-half RoPE on Q and K, Q pre-scaled by
//          1/sqrt(hd) to f32, K and V appended to the KV cache.
//   RESID  residual add into the f32 stream, the next GEMM input
//          x = (h * g_next) in the model dtype, per-tile sums of h^2 for the
//          next RMSNorm.
//   SWIGLU RMSNorm row scale, silu(gate) * up.
//   HEAD   RMSNorm row scale, optional logits, per-tile row summaries
//          (top1, argmax, top2, sum exp); the last tile of the launch merges
//          them per row and applies the draft pick or greedy acceptance.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <cudaTypedefs.h>

#include "attn_phase.cuh"
#include "model.cuh"
#include "stats.cuh"

namespace spec {

// ---------------------------------------------------------------------------
// host: tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

static bool load_encoder() {
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return false;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return true;
}

bool make_tmap_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
    if (!load_encoder()) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Activation buffer of bf16 hi rows then lo rows ([2][rows_pad][K]) as a 3-D
// map {K, rows_pad, 2}: one box {64, tp, 2} is a k-block of tp rows, hi tile
// then lo tile, as the MMA's B operand wants them (one copy instead of two).
bool make_tmap_x(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows_pad, uint32_t tp) {
    if (!load_encoder()) return false;
    cuuint64_t dims[3] = {K, rows_pad, 2};
    cuuint64_t strides[2] = {K * 2, rows_pad * K * 2};
    cuuint32_t box[3] = {(cuuint32_t)kTileK, tp, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// K and V cache maps of a bf16 cache: {hd, seq * kvh * slot, layer}, boxes of
// 64 dims x (4096 / hd) slots x 1 layer, 128-byte swizzle (the attention phase
// reads a unit of 8 KB of K and 8 KB of V per ring slot).
bool make_kv_tmaps(spec_kv* kv) {
    const spec_model* m = kv->m;
    const spec_model_config& c = m->cfg;
    kv->tmaps = false;
    if (!m->bf16 || (c.head_dim != 64 && c.head_dim != 128)) return true;
    const uint64_t rows = (uint64_t)kv->n_pages * c.n_kv_heads * kv->page;
    if (rows >= (1ull << 31)) return true;            // slot coordinates are 32-bit
    if (!load_encoder()) return false;
    for (int w = 0; w < 2; ++w) {
        cuuint64_t dims[3] = {(cuuint64_t)c.head_dim, rows, (cuuint64_t)c.n_layers};
        cuuint64_t strides[2] = {(cuuint64_t)c.head_dim * 2, rows * c.head_dim * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)(4096 / c.head_dim), 1};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = g_encode(w ? &kv->tm_v : &kv->tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w ? kv->v : kv->k, dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return false;
    }
    kv->tmaps = true;
    return true;
}

size_t attn_phase_part_floats(const spec_model* m) {
    return (size_t)m->num_sms * 2 * kAttnMaxQ * (m->cfg.head_dim + 2);
}

static bool attn_phase_fits(const spec_model* m, const spec_kv* kv, int batch, int max_rows_per_seq) {
    const int G = m->cfg.n_heads / m->cfg.n_kv_heads;
    return kv->tmaps && max_rows_per_seq * G <= kAttnMaxQ && batch <= kMaxPlanBatch &&
           m->attn_part_floats >= attn_phase_part_floats(m) && m->n_attn_counters >= batch * m->cfg.n_kv_heads;
}

bool attn_phase_ok(const spec_model* m, const spec_kv* kv, int batch, int max_rows_per_seq) {
    const bool wanted = m->attn_phase == 1 || (m->attn_phase == -1 && batch >= 2);
    return wanted && attn_phase_fits(m, kv, batch, max_rows_per_seq);
}

// ---------------------------------------------------------------------------
// split bookkeeping shared by host and device
struct Split {
    int n_tiles, kb;      // tiles of 128 features, k-blocks of 64
    long long units;      // n_tiles * kb
    int G;                // CTAs
    int T_pad;            // row stride of the partial tiles
    int max_slots;
    float* part;          // [n_tiles][max_slots][T_pad][128]
    int* counters;        // [n_tiles]
};

__host__ __device__ inline long long unit_begin(const Split& s, int c) { return (long long)c * s.units / s.G; }
// CTA whose range holds unit u
__host__ __device__ inline int cta_of(const Split& s, long long u) {
    return (int)(((u + 1) * s.G - 1) / s.units);
}
// units of CTA c; a chain launches as many CTAs as its widest phase, so a
// narrower phase leaves the CTAs past its own count without work
__host__ __device__ inline void cta_units(const Split& s, int c, long long& ub, long long& ue) {
    if (c < s.G) {
        ub = unit_begin(s, c);
        ue = unit_begin(s, c + 1);
    } else {
        ub = ue = 0;
    }
}

// ---------------------------------------------------------------------------
// epilogue shared memory
struct EpiSmem {
    float tile[kRowChunk][kTileN + 1];
    float rs_all[kMaxTPad];     // RMSNorm row scale of every row of the launch
    long long row_kv[kRowChunk]; // QKV: cache row of KV head 0 for each row of the chunk, -1 none
    int row_pos[kRowChunk];     // QKV: rotary position of each row of the chunk, -1 out of range
    int flag;
    int wait_ok;
};

SPEC_DEV int etid() { return threadIdx.x & 127; }

// RMSNorm row scales of all rows of the launch, computed once per CTA by the
// epilogue threads before the first accumulator is ready (so off the critical
// path): warp per row, lanes over the per-tile sums of squares.
SPEC_DEV void load_row_scales(const EpiParams& e, EpiSmem& sm) {
    if (e.kind != EPI_RESID) {
        const int w = etid() >> 5, lane = etid() & 31;
        for (int j = w; j < e.T; j += 4) {
            float s = 0.f;
            for (int i = lane; i < e.ss_tiles; i += 32) s += __ldcg(e.ss_in + (size_t)i * e.ss_stride + e.r0 + j);
            s = warp_sum(s);
            if (lane == 0) sm.rs_all[j] = 1.0f / sqrtf(s * e.inv_d + e.eps);
        }
    }
    named_bar(1, 128);
}

// Q|K|V epilogue of one chunk of rows: rotary embedding on Q and K, Q to its
// buffer, K and V to the cache.  This form walks the chunk element by element
// (each row reads its position, rotary values and cache slot as it goes); it
// is the faster one for chunks of a few rows.
template <typename KT>
SPEC_DEV void apply_qkv_rows(const EpiParams& e, int tile, int j0, int nr, EpiSmem& sm) {
    const int hd = e.head_dim, half = hd >> 1;
    const int qd = e.n_heads * hd, kvd = e.n_kv_heads * hd;
    for (int idx = etid(); idx < nr * kTileN; idx += 128) {
        const int j = idx >> 7, mm = idx & 127;
        const int n = tile * kTileN + mm;
        if (n >= e.N) continue;
        const int r = e.r0 + j0 + j;
        const float v = sm.tile[j][mm] * sm.rs_all[j0 + j];
        if (n < qd + kvd) {
            const int i = n & (hd - 1);
            const int pm = (i < half) ? mm + half : mm - half;
            const float pv = sm.tile[j][pm] * sm.rs_all[j0 + j];
            const int pos = e.plan.row_pos[r];
            if (pos < 0 || pos >= e.max_position) { dev_error(e.err, SPEC_DEVERR_POSITION); continue; }
            const int fi = i & (half - 1);
            const float c = e.rope_cos[(size_t)pos * half + fi], s = e.rope_sin[(size_t)pos * half + fi];
            const float o = (i < half) ? (v * c - pv * s) : (v * c + pv * s);
            if (n < qd) {
                e.q[(size_t)r * qd + n] = o * e.q_scale;
            } else {
                const int kvh = (n - qd) / hd;
                const int seq = e.plan.row_seq[r], slot = e.plan.row_slot[r];
                if (slot < 0 || slot >= e.kv_ctx) { dev_error(e.err, SPEC_DEVERR_CAPACITY); continue; }
                const long long row = kv_row(e.kvp, e.n_kv_heads, e.layer, seq, kvh, slot);
                if (row < 0) { dev_error(e.err, SPEC_DEVERR_CAPACITY); continue; }
                static_cast<KT*>(e.kc)[(size_t)row * hd + i] = from_f32<KT>(o);
            }
        } else {
            const int i = n & (hd - 1);
            const int kvh = (n - qd - kvd) / hd;
            const int seq = e.plan.row_seq[r], slot = e.plan.row_slot[r];
            if (slot < 0 || slot >= e.kv_ctx) { dev_error(e.err, SPEC_DEVERR_CAPACITY); continue; }
            const long long row = kv_row(e.kvp, e.n_kv_heads, e.layer, seq, kvh, slot);
            if (row < 0) { dev_error(e.err, SPEC_DEVERR_CAPACITY); continue; }
            static_cast<KT*>(e.vc)[(size_t)row * hd + i] = from_f32<KT>(v);
        }
    }
}

// The same for chunks of more rows: the rows' positions and cache rows are
// looked up once per chunk, and every rotary value a thread needs is loaded
// before its first store, so the chunk waits for one round of dependent loads
// instead of one a row (measured: the 29-row tree verification's QKV epilogue
// 20 -> 13 us; chunks of up to 8 rows keep the element walk, which measured
// faster there).
template <typename KT>
SPEC_DEV void apply_qkv(const EpiParams& e, int tile, int j0, int nr, EpiSmem& sm) {
    const int hd = e.head_dim, half = hd >> 1;
    const int qd = e.n_heads * hd, kvd = e.n_kv_heads * hd;
    if (nr <= 8) { apply_qkv_rows<KT>(e, tile, j0, nr, sm); return; }
    if (etid() < nr) {
        const int r = e.r0 + j0 + etid();
        int pos = e.plan.row_pos[r];
        if (pos < 0 || pos >= e.max_position) { dev_error(e.err, SPEC_DEVERR_POSITION); pos = -1; }
        const int seq = e.plan.row_seq[r], slot = e.plan.row_slot[r];
        long long row = -1;
        if (slot < 0 || slot >= e.kv_ctx) dev_error(e.err, SPEC_DEVERR_CAPACITY);
        else if ((row = kv_row(e.kvp, e.n_kv_heads, e.layer, seq, 0, slot)) < 0) dev_error(e.err, SPEC_DEVERR_CAPACITY);
        sm.row_pos[etid()] = pos;
        sm.row_kv[etid()] = row;
    }
    named_bar(1, 128);
    const int mm = etid();
    const int n = tile * kTileN + mm;
    if (n >= e.N) return;
    const int i = n & (hd - 1);
    if (n < qd + kvd) {
        const int pm = (i < half) ? mm + half : mm - half;
        const int fi = i & (half - 1);
        float cs[kRowChunk], sn[kRowChunk];
#pragma unroll
        for (int j = 0; j < kRowChunk; ++j) {
            const int pos = j < nr ? sm.row_pos[j] : -1;
            cs[j] = pos >= 0 ? __ldg(e.rope_cos + (size_t)pos * half + fi) : 0.f;
            sn[j] = pos >= 0 ? __ldg(e.rope_sin + (size_t)pos * half + fi) : 0.f;
        }
        const int kvh = (n - qd) / hd;       // K features only
#pragma unroll
        for (int j = 0; j < kRowChunk; ++j) {
            if (j >= nr || sm.row_pos[j] < 0) continue;
            const float v = sm.tile[j][mm] * sm.rs_all[j0 + j];
            const float pv = sm.tile[j][pm] * sm.rs_all[j0 + j];
            const float o = (i < half) ? (v * cs[j] - pv * sn[j]) : (v * cs[j] + pv * sn[j]);
            if (n < qd) {
                e.q[(size_t)(e.r0 + j0 + j) * qd + n] = o * e.q_scale;
            } else {
                const long long row = sm.row_kv[j];
                if (row >= 0) static_cast<KT*>(e.kc)[(size_t)(row + (long long)kvh * e.kvp.page) * hd + i] = from_f32<KT>(o);
            }
        }
    } else {
        const int kvh = (n - qd - kvd) / hd;
#pragma unroll
        for (int j = 0; j < kRowChunk; ++j) {
            if (j >= nr) continue;
            const long long row = sm.row_kv[j];
            if (row >= 0)
                static_cast<KT*>(e.vc)[(size_t)(row + (long long)kvh * e.kvp.page) * hd + i] =
                    from_f32<KT>(sm.tile[j][mm] * sm.rs_all[j0 + j]);
        }
    }
}

// Residual rows of a chunk for this thread's feature (etid()): loaded ahead of
// the accumulator so that the load is off the epilogue's critical path.
SPEC_DEV void load_resid(const EpiParams& e, int tile, int j0, int nr, float (&hv)[kRowChunk]) {
    const int n = tile * kTileN + etid();
#pragma unroll
    for (int j = 0; j < kRowChunk; ++j)
        hv[j] = (j < nr && n < e.N) ? __ldcg(e.h + (size_t)(e.r0 + j0 + j) * e.d_model + n) : 0.f;
}

template <typename XT>
SPEC_DEV void apply_resid(const EpiParams& e, int tile, int j0, int nr, EpiSmem& sm, const float (&hv)[kRowChunk]) {
    const int mm = etid();
    const int n = tile * kTileN + mm;
    // the feature's gain, read once: loaded inside the row loop it would be
    // re-read after every store (the compiler cannot rule out aliasing)
    const float gain = n < e.N ? e.gain_next[n] : 0.f;
#pragma unroll
    for (int j = 0; j < kRowChunk; ++j) {
        if (j >= nr) break;
        float sq = 0.f;
        if (n < e.N) {
            const int r = e.r0 + j0 + j;
            const size_t o = (size_t)r * e.d_model + n;
            const float hn = hv[j] + sm.tile[j][mm];
            e.h[o] = hn;
            store_act(static_cast<XT*>(e.x_next), o, e.x_next_lo, hn * gain);
            sq = hn * hn;
        }
        sm.tile[j][mm] = sq;
    }
    named_bar(1, 128);
    const int w = etid() >> 5, lane = etid() & 31;
    for (int j = w; j < nr; j += 4) {
        float s = sm.tile[j][lane] + sm.tile[j][lane + 32] + sm.tile[j][lane + 64] + sm.tile[j][lane + 96];
        s = warp_sum(s);
        if (lane == 0) e.ss_out[(size_t)tile * e.ss_stride + e.r0 + j0 + j] = s;
    }
}

template <typename XT>
SPEC_DEV void apply_swiglu(const EpiParams& e, int tile, int j0, int nr, EpiSmem& sm) {
    for (int idx = etid(); idx < nr * 64; idx += 128) {
        const int j = idx >> 6, mm = idx & 63;
        const int f = tile * 64 + mm;
        if (f >= e.d_ff) continue;
        const int r = e.r0 + j0 + j;
        const float g = sm.tile[j][mm] * sm.rs_all[j0 + j];
        const float u = sm.tile[j][mm + 64] * sm.rs_all[j0 + j];
        store_act(static_cast<XT*>(e.act), (size_t)r * e.d_ff + f, e.act_lo, g / (1.0f + expf(-g)) * u);
    }
}

SPEC_DEV void apply_head(const EpiParams& e, int tile, int j0, int nr, EpiSmem& sm) {
    for (int idx = etid(); idx < nr * kTileN; idx += 128) {
        const int j = idx >> 7, mm = idx & 127;
        const int v = tile * kTileN + mm;
        float l = -INFINITY;
        if (v < e.vocab) {
            l = sm.tile[j][mm] * sm.rs_all[j0 + j];
            if (e.logits) e.logits[(size_t)(e.r0 + j0 + j - e.logits_row0) * e.logits_stride + v] = l;
        }
        sm.tile[j][mm] = l;
    }
    named_bar(1, 128);
    // The tile's summary of a row: the largest logit with its lowest index, the
    // largest value besides that element, and sum exp(l - top1).  A warp takes
    // four rows at once (independent chains), reduces (top1, index, top2) across
    // its lanes, then sums one exponential a logit.
    const int w = etid() >> 5, lane = etid() & 31;
    for (int jb = w; jb < nr; jb += 16) {
        float t1[4], t2[4], x[4][4];
        int ix[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int j = jb + 4 * q;
            t1[q] = -INFINITY;
            t2[q] = -INFINITY;
            ix[q] = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int v = tile * kTileN + lane + 32 * i;
                const float l = (j < nr && v < e.vocab) ? sm.tile[j][lane + 32 * i] : -INFINITY;
                x[q][i] = l;
                if (l > t1[q]) {          // indices rise with i: a tie keeps the lower one
                    t2[q] = t1[q];
                    t1[q] = l;
                    ix[q] = v;
                } else {
                    t2[q] = fmaxf(t2[q], l);
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float u1 = __shfl_xor_sync(0xffffffffu, t1[q], o);
                const float u2 = __shfl_xor_sync(0xffffffffu, t2[q], o);
                const int ui = __shfl_xor_sync(0xffffffffu, ix[q], o);
                const bool other = u1 > t1[q] || (u1 == t1[q] && ui < ix[q]);
                t2[q] = fmaxf(fmaxf(t2[q], u2), other ? t1[q] : u1);
                if (other) {
                    t1[q] = u1;
                    ix[q] = ui;
                }
            }
        }
        float se[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            se[q] = 0.f;
            if (t1[q] != -INFINITY) {
#pragma unroll
                for (int i = 0; i < 4; ++i) se[q] += expf(x[q][i] - t1[q]);      // exp(-inf) = 0
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int q = 0; q < 4; ++q) se[q] += __shfl_xor_sync(0xffffffffu, se[q], o);
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = jb + 4 * q;
                if (j >= nr) break;
                spec_row_stats st = stat_empty();
                if (t1[q] != -INFINITY) {
                    st.top1 = t1[q];
                    st.top2 = t2[q];
                    st.sum_exp = se[q];
                    st.argmax = ix[q];
                }
                e.stat_part[(size_t)tile * e.ss_stride + e.r0 + j0 + j] = st;
            }
        }
    }
}

template <typename XT>
SPEC_DEV void apply_chunk(const EpiParams& e, int tile, int j0, int nr, EpiSmem& sm, const float (&hv)[kRowChunk]) {
    switch (e.kind) {
        case EPI_QKV: apply_qkv<XT>(e, tile, j0, nr, sm); break;
        case EPI_RESID: apply_resid<XT>(e, tile, j0, nr, sm, hv); break;
        case EPI_SWIGLU: apply_swiglu<XT>(e, tile, j0, nr, sm); break;
        default: apply_head(e, tile, j0, nr, sm); break;
    }
    named_bar(1, 128);
}

// Data written by other CTAs of the same launch is read past L1 (L2 is coherent).
SPEC_DEV spec_row_stats ldcg_stats(const spec_row_stats* p) {
    const float4 f = __ldcg(reinterpret_cast<const float4*>(p));
    spec_row_stats s;
    s.top1 = f.x;
    s.top2 = f.y;
    s.sum_exp = f.z;
    s.argmax = __float_as_int(f.w);
    return s;
}

// Last tile of an LM-head launch: merge the per-tile summaries of every row of
// the launch (warp per row, fixed order), then the draft pick or acceptance.
SPEC_DEV void head_finalize(const EpiParams& e, int n_tiles) {
    const int w = etid() >> 5, lane = etid() & 31;
    for (int j = w; j < e.T; j += 4) {
        const int r = e.r0 + j;
        spec_row_stats s = stat_empty();
        for (int t0 = lane; t0 < n_tiles; t0 += 32 * 8) {
            spec_row_stats v[8];             // independent loads first, then the merges
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int t = t0 + 32 * i;
                v[i] = t < n_tiles ? ldcg_stats(e.stat_part + (size_t)t * e.ss_stride + r) : stat_empty();
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) stat_merge(s, v[i]);
        }
        s = stat_warp_merge(s);
        if (lane == 0) {
            e.row_stats[r] = s;
            if (e.user_stats) e.user_stats[r] = s;
            if (e.head_mode == HEAD_DRAFT) {
                const int seq = e.plan.row_seq[r];
                e.cand[(size_t)seq * e.cand_stride + e.cand_col] = s.argmax;
            }
        }
    }
    if (e.head_mode == HEAD_ACCEPT_CHAIN || e.head_mode == HEAD_ACCEPT_TREE) {
        named_bar(1, 128);
        for (int b = etid(); b < e.batch; b += 128) {
            const int r0 = e.plan.seq_row0[b], n = e.plan.seq_nrows[b];
            const int* tok = e.tokens + (size_t)b * e.tok_stride;
            int* path = e.path ? e.path + (size_t)b * kMaxSeqRows : nullptr;
            if (e.head_mode == HEAD_ACCEPT_CHAIN)
                accept_chain_one(e.row_stats, r0, n, tok, e.acc_len + b, e.next_tok + b, path);
            else
                accept_tree_one(e.row_stats, r0, n, tok, e.plan.tree_parent, e.plan.tree_depth,
                                e.acc_len + b, e.next_tok + b, path);
        }
    }
}

// Called by all 128 epilogue threads after a tile's epilogue has run.
SPEC_DEV void head_tile_done(const EpiParams& e, int n_tiles, EpiSmem& sm) {
    if (e.kind != EPI_HEAD) return;
    named_bar(1, 128);
    if (etid() == 0) sm.flag = (atomic_add_acq_rel(e.done_counter, 1) == n_tiles - 1);
    named_bar(1, 128);
    if (sm.flag) {
        head_finalize(e, n_tiles);
        if (etid() == 0) *e.done_counter = 0;
    }
    named_bar(1, 128);
}

// One finished segment of a tile.  `load(ch, v)` gives this thread's 16 values
// (feature mm = etid(), rows ch*16 .. ch*16+15) of the segment's accumulator;
// `release()` is called once every value has been read.
template <typename XT, typename Loader>
SPEC_DEV void finish_segment(const EpiParams& e, const Split& sp, int tile, int slot, int nc,
                             EpiSmem& sm, Loader& ld, float (&hv)[kRowChunk], bool hv_ready) {
    const int mm = etid();
    const int nchunks = (e.T + kRowChunk - 1) / kRowChunk;
    const bool resid = e.kind == EPI_RESID;
    float v[16];
    if (nc == 1 && nchunks == 1) {
        // one chunk: read the accumulator out and release it to the next
        // segment's MMAs before the epilogue runs
        if (resid && !hv_ready) load_resid(e, tile, 0, e.T, hv);
        ld.load(0, v);
        ld.release();
#pragma unroll
        for (int i = 0; i < 16; ++i) sm.tile[i][mm] = v[i];
        named_bar(1, 128);
        apply_chunk<XT>(e, tile, 0, e.T, sm, hv);
        head_tile_done(e, sp.n_tiles, sm);
        return;
    }
    if (nc == 1) {
        for (int ch = 0; ch < nchunks; ++ch) {
            if (resid && (ch > 0 || !hv_ready)) load_resid(e, tile, ch * kRowChunk, min(kRowChunk, e.T - ch * kRowChunk), hv);
            ld.load(ch, v);
            const int nr = min(kRowChunk, e.T - ch * kRowChunk);
#pragma unroll
            for (int i = 0; i < 16; ++i) sm.tile[i][mm] = v[i];
            named_bar(1, 128);
            apply_chunk<XT>(e, tile, ch * kRowChunk, nr, sm, hv);
        }
        ld.release();
        head_tile_done(e, sp.n_tiles, sm);
        return;
    }
    float* my = sp.part + ((size_t)tile * sp.max_slots + slot) * sp.T_pad * kTileN;
    for (int ch = 0; ch < nchunks; ++ch) {
        ld.load(ch, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int j = ch * kRowChunk + i;
            if (j < e.T) my[(size_t)j * kTileN + mm] = v[i];
        }
    }
    ld.release();
    named_bar(1, 128);
    if (mm == 0) sm.flag = (atomic_add_acq_rel(sp.counters + tile, 1) == nc - 1);
    named_bar(1, 128);
    if (!sm.flag) return;
    const float* base = sp.part + (size_t)tile * sp.max_slots * sp.T_pad * kTileN;
    for (int ch = 0; ch < nchunks; ++ch) {
        const int nr = min(kRowChunk, e.T - ch * kRowChunk);
        // residual rows load alongside the partial slots (independent)
        if (resid && (ch > 0 || !hv_ready)) load_resid(e, tile, ch * kRowChunk, nr, hv);
        float acc[kRowChunk];
#pragma unroll
        for (int i = 0; i < kRowChunk; ++i) acc[i] = 0.f;
        for (int q = 0; q < nc; ++q) {           // slots in a fixed order: deterministic sums
            const float* src = base + ((size_t)q * sp.T_pad + ch * kRowChunk) * kTileN + mm;
            float v2[kRowChunk];
#pragma unroll
            for (int i = 0; i < kRowChunk; ++i) v2[i] = (i < nr) ? __ldcg(src + (size_t)i * kTileN) : 0.f;
#pragma unroll
            for (int i = 0; i < kRowChunk; ++i) acc[i] += v2[i];
        }
#pragma unroll
        for (int i = 0; i < kRowChunk; ++i) sm.tile[i][mm] = acc[i];
        named_bar(1, 128);
        apply_chunk<XT>(e, tile, ch * kRowChunk, nr, sm, hv);
    }
    if (mm == 0) sp.counters[tile] = 0;
    head_tile_done(e, sp.n_tiles, sm);
}

// ---------------------------------------------------------------------------
// tcgen05 kernel
constexpr int kTcThreads = 192;           // warps 0-3 epilogue, 4 TMA, 5 MMA
constexpr uint32_t kATileBytes = kTileN * kTileK * 2;

struct TcLayout {
    int stages;
    uint32_t b_bytes;     // hi + lo activation tiles of one stage
    uint32_t tmem_cols;
    int rows_pad;         // first row of the lo half in the X buffers
    uint32_t attn_bytes;  // AttnSmem when the chain has an attention phase, else 0
    int attn_slots;       // attention ring: all 16 KB slots (weight slots, activation region, spare)
    int attn_nb;          // of which in the activation-tile region
};

constexpr size_t kEpiSmemBytes = (sizeof(EpiSmem) + 15) & ~size_t(15);

constexpr size_t kBarBytes = 512;     // ring, accumulator and attention-ring barriers, TMEM slot, abort flag

// everything but the attention ring's spare slots
__host__ __device__ inline size_t tc_smem_core(const TcLayout& L) {
    return 1024 + (size_t)L.stages * (kATileBytes + L.b_bytes) + kBarBytes + kEpiSmemBytes + L.attn_bytes;
}
// spare attention slots start at the next 1 KB boundary after the core
__host__ __device__ inline size_t tc_smem_bytes(const TcLayout& L) {
    const int spare = L.attn_slots > 0 ? L.attn_slots - L.stages - L.attn_nb : 0;
    return ((tc_smem_core(L) + 1023) & ~size_t(1023)) + (size_t)spare * kAttnUnitBytes + 64;
}

struct TmemLoader {
    uint32_t taddr;
    uint64_t* acc_empty;
    SPEC_DEV void load(int ch, float (&v)[16]) { tmem_ld16(taddr + ch * 16, v); }
    SPEC_DEV void release() {
        tc_fence_before();
        mbar_arrive(acc_empty);
    }
};

// One launch runs a chain of up to kMaxPhases GEMMs (for example O projection ->
// gate/up -> down -> next QKV) separated by grid barriers.  The TMA producer
// streams the next phase's weight tiles into the ring while the previous phase
// finishes; only the activation tiles wait for the barrier.  One phase is a
// plain GEMM launch.
constexpr int kMaxPhases = 5;
constexpr int kMaxStages = 8;

// A GEMM phase uses tmW, tmX, sp and e; an attention phase uses tmW / tmX as
// the K / V cache maps and `at`.
struct GemmPhase {
    CUtensorMap tmW;
    CUtensorMap tmX;
    const uint8_t* wt;  // tile-major weights (16 KB per (tile, k-block)), or null: 2-D tensor copies via tmW
    Split sp;
    EpiParams e;
    AttnPhase at;
    int kind;      // PhaseKind
};

struct GemmChain {
    GemmPhase ph[kMaxPhases];
    int n;
    int attn;      // index of the attention phase, -1 if none (at most one)
    int* bar;      // per launch: CTAs that finished a phase, summed over phases
    int* done;     // CTAs that finished the chain; the last one resets both counters
    unsigned long long wait_ns;   // limit of the grid-barrier waits
    int stall_cta; // failure injection (tests): this CTA withholds its arrival after phase 0; -1 none
};

SPEC_DEV int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
SPEC_DEV void red_release_gpu_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
// orders this thread's generic-proxy global accesses with later async-proxy (TMA) ones
SPEC_DEV void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// bounded wait until every CTA has finished `phases` phases (at most limit_ns)
SPEC_DEV bool grid_wait(const int* bar, int target, volatile int* abort_flag, int* err, uint64_t limit_ns) {
    if (ld_acquire_gpu(bar) >= target) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        // two pollers a CTA share one counter with every arrival: back off a
        // little between plain reads, acquire once the count is reached
        __nanosleep(40);
        if (*reinterpret_cast<const volatile int*>(bar) >= target) {
            (void)ld_acquire_gpu(bar);
            return true;
        }
        if ((it & 63u) == 0u) {
            if (abort_flag && *abort_flag) return false;
            if (global_timer_ns() - t0 > limit_ns) {
                if (abort_flag) *abort_flag = 1;
                dev_error(err, SPEC_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// ATTN: the chain may hold an attention phase (instantiated only then, so the
// plain GEMM chains carry none of its code or registers).
template <bool ATTN, bool PAGED = false>
__global__ void __launch_bounds__(kTcThreads, 1)
gemm_tc_kernel(const __grid_constant__ GemmChain ch, TcLayout L) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = base;
    uint8_t* sB = sA + (size_t)L.stages * kATileBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + (size_t)L.stages * L.b_bytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + L.stages;
    uint64_t* acc_full = bars + 2 * L.stages;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* drain = acc_full + 2;
    uint64_t* attn_done = acc_full + 3;      // the epilogue warps finished the attention phase
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint64_t* attn_full = acc_full + 6;
    uint64_t* attn_empty = attn_full + kAttnMaxSlots;
    EpiSmem& sm = *reinterpret_cast<EpiSmem*>(reinterpret_cast<uint8_t*>(bars) + kBarBytes);
    AttnSmem& as = *reinterpret_cast<AttnSmem*>(reinterpret_cast<uint8_t*>(bars) + kBarBytes + kEpiSmemBytes);
    // the attention ring: the weight slots, the activation-tile region, then spare memory
    AttnRing R;
    R.a = sA;
    R.na = L.stages;
    R.b = sB;
    R.nb = L.attn_nb;
    R.x = reinterpret_cast<uint8_t*>(((reinterpret_cast<uintptr_t>(&as) + L.attn_bytes) + 1023) & ~uintptr_t(1023));
    R.n = L.attn_slots;
    R.full = attn_full;
    R.empty = attn_empty;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, G = gridDim.x;
    int* err = ch.ph[0].e.err;

    if (threadIdx.x == 0) {
        for (int s = 0; s < L.stages; ++s) { mbar_init(full + s, 1); mbar_init(empty + s, 1); }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 128);
        mbar_init(drain, 1);
        mbar_init(attn_done, 1);
        for (int s = 0; s < L.attn_slots; ++s) { mbar_init(attn_full + s, 1); mbar_init(attn_empty + s, 1); }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        tmem_alloc(tmem_slot, L.tmem_cols);
        tmem_relinquish();
    }
    // the attention phase's unit table reads the row plan, which a kernel at
    // least two launches back wrote (every kernel of the stream triggers its
    // dependants only after its own wait, so that one has completed)
    if constexpr (ATTN)
        if (ch.attn >= 0 && warp == 4) attn_unit_table(ch.ph[ch.attn].at, as);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        if (lane == 0) {
            for (int p = 0; p < ch.n; ++p) {
                tma_prefetch_desc(&ch.ph[p].tmW);
                tma_prefetch_desc(&ch.ph[p].tmX);
            }
            const uint64_t pw = l2_policy_evict_first(), px = l2_policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            int a_slot = 0;           // attention ring position
            uint32_t a_phase = 0;
            long long a_issued = 0;
            int def_stage[kMaxStages];
            int def_kb[kMaxStages];
            int n_def = 0;
            bool ok = true;
            const GemmPhase* P = &ch.ph[0];
            auto load_x = [&](const GemmPhase& Q, int st, int kbi) {     // hi and lo tiles in one box
                tma_load_3d(sB + (size_t)st * L.b_bytes, &Q.tmX, kbi * kTileK, Q.e.r0, 0, full + st, px);
            };
            // what a phase reads from the previous phase (the previous kernel for
            // phase 0) waits for it; weight tiles and committed KV slots do not
            auto dep_wait = [&](int p) -> bool {
                if (p == 0) { pdl_wait(); return true; }
                if (!grid_wait(ch.bar, G * p, abort_flag, err, ch.wait_ns)) return false;
                fence_proxy_async_global();     // the rows were written by other CTAs' epilogues
                return true;
            };
            for (int p = 0; ok && p < ch.n; ++p) {
                P = &ch.ph[p];
                n_def = 0;
                if (ATTN && P->kind == PH_ATTN) {
                    const AttnPhase& A = P->at;
                    long long ub, ue;
                    attn_range(as.prefix[A.batch], G, c, ub, ue);
                    const int ku = attn_keys_per_unit(A.head_dim), nbox = A.head_dim / 64;
                    const uint32_t box = (uint32_t)ku * 128u;
                    bool dep = false;
                    // (sequence, head, slot tile) of the current unit, stepped without divisions
                    const int n_units = (int)(ue - ub);
                    AttnUnit au = n_units > 0 ? attn_locate(as, A.batch, A.n_kv_heads, ub) : AttnUnit{0, 0, 0, 1};
                    int seq_base = as.base[au.b];
                    int seq_keys = min(seq_base + as.nrows[au.b], A.kv_ctx);
                    // a unit's first row: (page * Hkv + head) * page size + slot in page; a
                    // contiguous cache has page = sequence (the paged variant keeps the last
                    // page-table entry it read)
                    const KVPages& kvp = P->e.kvp;
                    const size_t layer_bytes =
                        (size_t)A.layer * kvp.n_pages * A.n_kv_heads * kvp.page * A.head_dim * 2;
                    [[maybe_unused]] int pg_b = -1, pg_blk = -1, pg_page = -1;
                    for (int i = 0; i < n_units; ++i) {
                        if (i > 0 && ++au.tile == au.tiles) {
                            au.tile = 0;
                            if (++au.g == A.n_kv_heads) {
                                au.g = 0;
                                ++au.b;
                                au.tiles = (as.prefix[au.b + 1] - as.prefix[au.b]) / A.n_kv_heads;
                                seq_base = as.base[au.b];
                                seq_keys = min(seq_base + as.nrows[au.b], A.kv_ctx);
                            }
                        }
                        const int key0 = au.tile * ku;
                        // units holding new (or unused) slots wait for the rows' writer
                        if (!dep && key0 + ku > seq_base) {
                            if (!dep_wait(p)) { ok = false; break; }
                            dep = true;
                        }
                        if (!mbar_wait(R.empty + a_slot, a_phase ^ 1u, abort_flag, err)) { ok = false; break; }
                        uint8_t* dst = R.slot(a_slot);
                        uint64_t* fb = R.full + a_slot;
                        // the unit's first cache row (a unit never crosses a page; the last page
                        // looked up is kept); a page not held reads row 0 and flags the error
                        int krow;
                        if constexpr (PAGED) {
                            const int blk = key0 >> kvp.shift;
                            if (au.b != pg_b || blk != pg_blk) {
                                pg_b = au.b;
                                pg_blk = blk;
                                pg_page = kvp.table[(size_t)au.b * kvp.max_pages + blk];
                            }
                            krow = pg_page < 0 ? -1
                                               : (pg_page * A.n_kv_heads + au.g) * kvp.page + (key0 & (kvp.page - 1));
                        } else {
                            krow = (au.b * A.n_kv_heads + au.g) * A.kv_ctx + key0;
                        }
                        if (krow < 0) { dev_error(err, SPEC_DEVERR_CAPACITY); krow = 0; }
                        if (A.linear) {
                            // the unit's valid K rows and V rows: two contiguous copies
                            const uint32_t bytes = (uint32_t)min(ku, seq_keys - key0) * A.head_dim * 2;
                            const size_t off = layer_bytes + (size_t)krow * A.head_dim * 2;
                            mbar_arrive_expect_tx(fb, 2 * bytes);
                            bulk_load(dst, static_cast<const char*>(A.kc) + off, bytes, fb, pw);
                            bulk_load(dst + kAttnUnitBytes / 2, static_cast<const char*>(A.vc) + off, bytes, fb, pw);
                        } else {
                            mbar_arrive_expect_tx(fb, kAttnUnitBytes);
                            const int row = krow;
                            for (int db = 0; db < nbox; ++db) {
                                tma_load_3d(dst + db * box, &P->tmW, 64 * db, row, A.layer, fb, pw);
                                tma_load_3d(dst + (nbox + db) * box, &P->tmX, 64 * db, row, A.layer, fb, pw);
                            }
                        }
                        ++a_issued;
                        if (++a_slot == R.n) { a_slot = 0; a_phase ^= 1u; }
                    }
                    // wait for the dependency even without a dependent unit: the grid
                    // barrier of the next phase is only meaningful once the previous
                    // kernel (which resets it) has completed
                    if (ok && !dep && !dep_wait(p)) ok = false;
                    // the attention slots overlap the GEMM ring: reuse them once the
                    // epilogue warps have finished the phase
                    if (ok && !mbar_wait(attn_done, 0, abort_flag, err)) ok = false;
                    continue;
                }
                const Split& sp = P->sp;
                long long ub, ue;
                cta_units(sp, c, ub, ue);
                bool dep = false;
                // (tile, k-block) of the current unit, stepped without divisions
                int tile = (int)(ub / sp.kb), kbi = (int)(ub % sp.kb);
                const int n_units = (int)(ue - ub);
                for (int i = 0; i < n_units; ++i) {
                    if (!dep && n_def == L.stages) {
                        if (!dep_wait(p)) { ok = false; break; }
                        dep = true;
                        for (int i = 0; i < n_def; ++i) load_x(*P, def_stage[i], def_kb[i]);
                        n_def = 0;
                    }
                    if (!mbar_wait(empty + stage, phase ^ 1u, abort_flag, err)) { ok = false; break; }
                    mbar_arrive_expect_tx(full + stage, kATileBytes + L.b_bytes);
                    if (P->wt)
                        bulk_load(sA + (size_t)stage * kATileBytes,
                                  P->wt + ((size_t)tile * sp.kb + kbi) * kATileBytes, kATileBytes, full + stage, pw);
                    else
                        tma_load_2d(sA + (size_t)stage * kATileBytes, &P->tmW, kbi * kTileK, tile * kTileN,
                                    full + stage, pw);
                    if (dep) {
                        load_x(*P, stage, kbi);
                    } else {
                        def_stage[n_def] = stage;
                        def_kb[n_def] = kbi;
                        ++n_def;
                    }
                    ++issued;
                    if (++stage == L.stages) { stage = 0; phase ^= 1u; }
                    if (++kbi == sp.kb) { kbi = 0; ++tile; }
                }
                if (ok && !dep) {
                    if (!dep_wait(p)) { ok = false; }
                    else {
                        for (int i = 0; i < n_def; ++i) load_x(*P, def_stage[i], def_kb[i]);
                        n_def = 0;
                    }
                }
            }
            if (*abort_flag) {
                // complete the deferred stages (their barriers expect the activation bytes), then
                // let every copy still in flight land before the CTA exits
                for (int i = 0; i < n_def; ++i) load_x(*P, def_stage[i], def_kb[i]);
                const long long n = issued < L.stages ? issued : L.stages;
                for (long long i = 0; i < n; ++i) {
                    if (--stage < 0) { stage = L.stages - 1; phase ^= 1u; }
                    mbar_wait(full + stage, phase, nullptr, err);
                }
                const long long na = a_issued < R.n ? a_issued : R.n;
                for (long long i = 0; i < na; ++i) {
                    if (--a_slot < 0) { a_slot = R.n - 1; a_phase ^= 1u; }
                    mbar_wait(R.full + a_slot, a_phase, nullptr, err);
                }
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int p = 0; ok && p < ch.n; ++p) {
                if (ch.ph[p].kind == PH_ATTN) continue;    // the epilogue warps run it on the attention ring
                const Split& sp = ch.ph[p].sp;
                const uint32_t idesc = idesc_bf16_f32(128, sp.T_pad);
                long long ub, ue;
                cta_units(sp, c, ub, ue);
                for (long long u = ub; ok && u < ue;) {
                    const int tile = (int)(u / sp.kb);
                    const long long seg_end = min(ue, (long long)(tile + 1) * sp.kb);
                    if (!mbar_wait(acc_empty, acc_phase ^ 1u, abort_flag, err)) { ok = false; break; }
                    acc_phase ^= 1u;
                    tc_fence_after();
                    const long long seg_begin = u;
                    for (; u < seg_end; ++u) {
                        if (!mbar_wait(full + stage, phase, abort_flag, err)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t ad = smem_desc_sw128(smem_u32(sA + (size_t)stage * kATileBytes));
                        const uint64_t bh = smem_desc_sw128(smem_u32(sB + (size_t)stage * L.b_bytes));
                        const uint64_t bl = smem_desc_sw128(smem_u32(sB + (size_t)stage * L.b_bytes + L.b_bytes / 2));
#pragma unroll
                        for (int k = 0; k < kTileK / 16; ++k) {
                            tc_mma_f16(tmem, ad + 2u * k, bh + 2u * k, idesc, (u > seg_begin || k > 0) ? 1u : 0u);
                            tc_mma_f16(tmem, ad + 2u * k, bl + 2u * k, idesc, 1u);
                        }
                        tc_commit(empty + stage);
                        if (++stage == L.stages) { stage = 0; phase ^= 1u; }
                    }
                    if (ok) tc_commit(acc_full);
                }
            }
            tc_commit(drain);
            mbar_wait(drain, 0, nullptr, err);
        }
    } else {
        TmemLoader ld;
        ld.taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        ld.acc_empty = acc_empty;
        uint32_t acc_phase = 0;
        bool ok = true;
        pdl_wait();
        // only now may the next kernel launch (see the unit table above)
        if (etid() == 0) pdl_trigger();
        for (int p = 0; ok && p < ch.n; ++p) {
            const GemmPhase& P = ch.ph[p];
            if (p > 0) {
                if (etid() == 0) sm.wait_ok = grid_wait(ch.bar, G * p, abort_flag, err, ch.wait_ns) ? 1 : 0;
                named_bar(1, 128);
                const int w_ok = sm.wait_ok;
                named_bar(1, 128);
                if (!w_ok) break;
            }
            if (ATTN && P.kind == PH_ATTN) {
                const AttnPhase& A = P.at;
                bool a_ok = false;
                if constexpr (ATTN)
                    a_ok = A.head_dim == 128 ? consume_attn<128>(A, as, R, c, G, abort_flag, err)
                                             : consume_attn<64>(A, as, R, c, G, abort_flag, err);
                if (etid() == 0) mbar_arrive(attn_done);     // all 128 threads are past their last unit
                if (!a_ok) { ok = false; break; }
            } else {
                const Split& sp = P.sp;
                load_row_scales(P.e, sm);
                long long ub, ue;
                cta_units(sp, c, ub, ue);
                for (long long u = ub; u < ue;) {
                    const int tile = (int)(u / sp.kb);
                    const long long seg_end = min(ue, (long long)(tile + 1) * sp.kb);
                    const int first = cta_of(sp, (long long)tile * sp.kb);
                    const int last = cta_of(sp, (long long)(tile + 1) * sp.kb - 1);
                    // the residual rows of the tile load while its accumulator is computed
                    float hv[kRowChunk];
                    const bool hv_ready = P.e.kind == EPI_RESID;
                    if (hv_ready) load_resid(P.e, tile, 0, min(kRowChunk, P.e.T), hv);
                    // one thread waits (bounded) and broadcasts, so all 128 leave together
                    if (etid() == 0) sm.wait_ok = mbar_wait(acc_full, acc_phase, abort_flag, err) ? 1 : 0;
                    named_bar(1, 128);
                    const int w_ok = sm.wait_ok;
                    named_bar(1, 128);
                    if (!w_ok) { ok = false; break; }
                    acc_phase ^= 1u;
                    tc_fence_after();
                    finish_segment<__nv_bfloat16>(P.e, sp, tile, c - first, last - first + 1, sm, ld, hv, hv_ready);
                    u = seg_end;
                }
            }
            if (ok && ch.n > 1) {
                // this CTA's share of phase p is written: count it (release)
                named_bar(1, 128);
                // the release reduction orders the CTA's writes (they reach thread 0
                // through the barrier above); the proxy fence lets the next phase's
                // tensor copies see them
                if (etid() == 0 && !(c == ch.stall_cta && p == 0)) {
                    fence_proxy_async_global();
                    red_release_gpu_add(ch.bar, 1);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, L.tmem_cols);
    }
    if (threadIdx.x == 0 && ch.n > 1) {
        if (atomic_add_acq_rel(ch.done, 1) == G - 1) {
            *ch.bar = 0;
            *ch.done = 0;
        }
    }
}

// ---------------------------------------------------------------------------
// f32 CUDA-core kernel (f32 models)
constexpr int kSimtMaxT = 32;
constexpr int kSimtK = 32;

struct SmemTileLoader {
    const float* acc;   // [kSimtMaxT][129]
    SPEC_DEV void load(int ch, float (&v)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = acc[(ch * 16 + i) * (kTileN + 1) + etid()];
    }
    SPEC_DEV void release() {}
};

__global__ void __launch_bounds__(128)
gemm_f32_kernel(const float* __restrict__ W, const float* __restrict__ X, int x_stride, int N, int K,
                Split sp, EpiParams e) {
    union WorkSmem {
        float w[kTileN][kSimtK + 1];               // weight sub-tile
        float acc[kSimtMaxT * (kTileN + 1)];       // finished segment, rows x features
    };
    __shared__ WorkSmem ws;
    __shared__ float sX[kSimtMaxT][kSimtK + 1];
    __shared__ EpiSmem sm;
    const int c = blockIdx.x, t = threadIdx.x;
    const long long u_begin = unit_begin(sp, c), u_end = unit_begin(sp, c + 1);
    pdl_wait();
    pdl_trigger();
    load_row_scales(e, sm);
    for (long long u = u_begin; u < u_end;) {
        const int tile = (int)(u / sp.kb);
        const long long seg_end = min(u_end, (long long)(tile + 1) * sp.kb);
        float acc[kSimtMaxT];
#pragma unroll
        for (int j = 0; j < kSimtMaxT; ++j) acc[j] = 0.f;
        for (; u < seg_end; ++u) {
            const int kb = (int)(u % sp.kb);
            for (int k0 = 0; k0 < kTileK; k0 += kSimtK) {
                __syncthreads();
                for (int i = t; i < kTileN * kSimtK; i += 128) {
                    const int rr = i / kSimtK, kk = i % kSimtK;
                    const int n = tile * kTileN + rr, k = kb * kTileK + k0 + kk;
                    ws.w[rr][kk] = (n < N && k < K) ? W[(size_t)n * K + k] : 0.f;
                }
                for (int i = t; i < kSimtMaxT * kSimtK; i += 128) {
                    const int j = i / kSimtK, kk = i % kSimtK;
                    const int k = kb * kTileK + k0 + kk;
                    sX[j][kk] = (j < e.T && k < K) ? X[(size_t)(e.r0 + j) * x_stride + k] : 0.f;
                }
                __syncthreads();
                for (int kk = 0; kk < kSimtK; ++kk) {
                    const float w = ws.w[t][kk];
#pragma unroll
                    for (int j = 0; j < kSimtMaxT; ++j) acc[j] = fmaf(w, sX[j][kk], acc[j]);
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kSimtMaxT; ++j) ws.acc[j * (kTileN + 1) + t] = acc[j];
        __syncthreads();
        const int first = cta_of(sp, (long long)tile * sp.kb);
        const int last = cta_of(sp, (long long)(tile + 1) * sp.kb - 1);
        SmemTileLoader ld{ws.acc};
        float hv[kRowChunk];
        finish_segment<float>(e, sp, tile, c - first, last - first + 1, sm, ld, hv, false);
        __syncthreads();
        u = seg_end;
    }
}

// ---------------------------------------------------------------------------
// host launch
constexpr int kMaxSlices = 8;
constexpr double kChainMinPhaseBytes = 16.0 * 1024 * 1024;

static int max_slots_of(const Split& s) {
    int mx = 1;
    for (int t = 0; t < s.n_tiles; ++t) {
        const int a = cta_of(s, (long long)t * s.kb), b = cta_of(s, (long long)(t + 1) * s.kb - 1);
        mx = std::max(mx, b - a + 1);
    }
    return mx;
}

static Split make_split(const spec_model* m, int N, int K, int T_pad) {
    Split s{};
    s.n_tiles = (N + kTileN - 1) / kTileN;
    s.kb = (K + kTileK - 1) / kTileK;
    s.units = (long long)s.n_tiles * s.kb;
    // CTAs a tile: the last one to finish adds the others' partial tiles, one
    // slot after another (about 1 us each), while each k-block a CTA streams costs
    // about 0.36 us (16 KB at an SM's share of the bandwidth); about sqrt(0.36 kb)
    // slices balance the two, at most kMaxSlices.  The large GEMMs still fill
    // every SM; small ones (few k-blocks a tile) take fewer CTAs.
    const int slices = std::min(kMaxSlices, std::max(2, (int)std::ceil(std::sqrt(0.36 * s.kb))));
    s.G = (int)std::min<long long>(std::min<long long>(m->num_sms, s.units), (long long)slices * s.n_tiles);
    s.T_pad = T_pad;
    s.max_slots = max_slots_of(s);
    return s;
}

size_t gemm_partial_floats_needed(const spec_model* m, int N, int K, int T_pad) {
    Split s = make_split(m, N, K, T_pad);
    return (size_t)s.n_tiles * s.max_slots * T_pad * kTileN;
}

int gemm_grid(const spec_model* m, int N, int K) { return make_split(m, N, K, 16).G; }

static TcLayout tc_layout(int T_pad, int rows_pad, bool attn) {
    TcLayout L;
    L.rows_pad = rows_pad;
    L.b_bytes = 2u * (uint32_t)T_pad * kTileK * 2;
    L.attn_bytes = attn ? (uint32_t)((sizeof(AttnSmem) + 15) & ~size_t(15)) : 0u;
    const size_t budget = 225 * 1024 - 1024 - kBarBytes - kEpiSmemBytes - L.attn_bytes - 64;
    L.stages = (int)std::min<size_t>(kMaxStages, budget / (kATileBytes + L.b_bytes));
    uint32_t cols = 32;
    while (cols < (uint32_t)T_pad) cols <<= 1;
    L.tmem_cols = cols;
    L.attn_slots = 0;
    L.attn_nb = 0;
    if (attn) {
        // attention ring: the weight slots, whole 16 KB slots of the activation region,
        // then as many spare slots as the 227 KB limit leaves
        L.attn_nb = (int)((size_t)L.stages * L.b_bytes / kAttnUnitBytes);
        const size_t core = (tc_smem_core(L) + 1023) & ~size_t(1023);
        const int spare = (int)((227 * 1024 - 64 - core) / kAttnUnitBytes);
        L.attn_slots = std::min(kAttnMaxSlots, L.stages + L.attn_nb + std::max(0, spare));
        L.attn_nb = std::min(L.attn_nb, L.attn_slots - L.stages);
    }
    return L;
}

// kernel parameters beyond 4 KB need CUDA 12.1+ (all of this code needs 13)
static_assert(sizeof(GemmChain) + sizeof(TcLayout) <= 32764, "chain parameters exceed the kernel parameter space");
static_assert(kAttnUnitBytes == kATileBytes, "an attention unit fills one weight slot of the ring");

// counters past the per-tile ones: chain barrier, chain exit count, LM-head tile count
static int* chain_bar(spec_model* m) { return m->counters + m->n_counters - 3; }
static int* chain_done(spec_model* m) { return m->counters + m->n_counters - 2; }

static int check_split(spec_model* m, const Split& s) {
    if ((size_t)s.n_tiles * s.max_slots * s.T_pad * kTileN > m->gemm_part_floats || s.n_tiles > m->n_counters - 3)
        return set_error(SPEC_ERR_CAPACITY, "GEMM workspace too small for this launch");
    return SPEC_OK;
}

static double algorithmic_bytes(const spec_model* m, const GemmLaunch& g, int T) {
    // weights once, activation rows in, output rows out
    return (double)g.N * g.K * m->elem + (double)T * g.K * m->elem + (double)T * g.N * m->elem;
}

// bf16: one launch of the chain kernel over steps[0..n) (rows T <= kMaxTPad, all
// phases on the same rows)
static int launch_tc_chain(spec_model* m, const GemmStep* steps, int n, cudaStream_t st) {
    GemmChain ch{};
    ch.attn = -1;
    const int T = steps[0].e.T;
    const int T_pad = ((T + 15) / 16) * 16;
    int G = 1;
    double bytes = 0.0;
    for (int p = 0; p < n; ++p) {
        GemmPhase& P = ch.ph[p];
        P.kind = steps[p].kind;
        P.e = steps[p].e;
        P.e.err = m->err;
        if (P.kind == PH_ATTN) {
            if (ch.attn >= 0) return set_error(SPEC_ERR_ARG, "GEMM chain: one attention phase at most");
            ch.attn = p;
            P.tmW = *steps[p].g.tmW;        // K cache map
            P.tmX = *steps[p].g.tmX;        // V cache map
            P.at = steps[p].at;
            P.at.err = m->err;
            P.at.part = m->attn_part;
            P.at.counters = m->attn_counters;
            P.at.kv_bytes = m->prof_on ? m->prof_kv : nullptr;
            G = std::max(G, m->num_sms);
            // output rows (K/V bytes are counted on the device)
            bytes += (double)T * P.at.n_heads * P.at.head_dim * m->elem;
            continue;
        }
        P.tmW = *steps[p].g.tmW;
        P.wt = m->w_tiled ? static_cast<const uint8_t*>(steps[p].g.W) : nullptr;
        P.tmX = m->tm_x[steps[p].xbuf][T_pad / 16 - 1];
        P.sp = make_split(m, steps[p].g.N, steps[p].g.K, T_pad);
        P.sp.part = m->gemm_part;
        P.sp.counters = m->counters;
        SPEC_TRY(check_split(m, P.sp));
        G = std::max(G, P.sp.G);
        bytes += algorithmic_bytes(m, steps[p].g, T);
    }
    ch.n = n;
    ch.bar = chain_bar(m);
    ch.done = chain_done(m);
    ch.wait_ns = kWaitLimitNs;
    ch.stall_cta = -1;
    if (n > 1 && m->test_stall_cta >= 0) {      // one-shot failure injection (tests)
        ch.stall_cta = m->test_stall_cta;
        ch.wait_ns = m->test_wait_ns;
        m->test_stall_cta = -1;
    }
    TcLayout L = tc_layout(T_pad, m->max_rows_pad, ch.attn >= 0);
    const size_t smem = tc_smem_bytes(L);
    if (smem > 227 * 1024) return set_error(SPEC_ERR_CAPACITY, "GEMM chain: shared memory layout too large");
    // the attention phase's four warps take ring positions in turn: the ring must be longer
    if (ch.attn >= 0 && L.attn_slots <= 4) return set_error(SPEC_ERR_CAPACITY, "GEMM chain: attention ring too short");
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(gemm_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        cudaFuncSetAttribute(gemm_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        cudaFuncSetAttribute(gemm_tc_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        attr_set = true;
    }
    const int slot = prof_start(m, st);
    if (ch.attn >= 0 && ch.ph[ch.attn].e.kvp.shift >= 0)
        launch_k(m->pdl, gemm_tc_kernel<true, true>, dim3(G), dim3(kTcThreads), smem, st, ch, L);
    else if (ch.attn >= 0)
        launch_k(m->pdl, gemm_tc_kernel<true>, dim3(G), dim3(kTcThreads), smem, st, ch, L);
    else
        launch_k(m->pdl, gemm_tc_kernel<false>, dim3(G), dim3(kTcThreads), smem, st, ch, L);
    ++m->launches;
    prof_stop(m, slot, st, PROF_GEMM, bytes);
    return check_cuda(cudaGetLastError(), "GEMM launch");
}

int launch_gemm(spec_model* m, const GemmLaunch& g, EpiParams e, int xbuf, cudaStream_t st) {
    const int T_total = e.T, r_base = e.r0;
    const int max_t = m->bf16 ? kMaxTPad : kSimtMaxT;
    for (int done = 0; done < T_total; done += max_t) {
        EpiParams ec = e;
        ec.T = std::min(max_t, T_total - done);
        ec.r0 = r_base + done;
        if (ec.kind == EPI_HEAD && (e.head_mode == HEAD_ACCEPT_CHAIN || e.head_mode == HEAD_ACCEPT_TREE) &&
            done + max_t < T_total)
            ec.head_mode = HEAD_STATS;   // acceptance once every row has its summary
        if (m->bf16) {
            GemmStep one{g, ec, xbuf};
            SPEC_TRY(launch_tc_chain(m, &one, 1, st));
            continue;
        }
        Split s = make_split(m, g.N, g.K, kSimtMaxT);
        s.part = m->gemm_part;
        s.counters = m->counters;
        SPEC_TRY(check_split(m, s));
        const int slot = prof_start(m, st);
        launch_k(m->pdl, gemm_f32_kernel, dim3(s.G), dim3(128), 0, st, static_cast<const float*>(g.W),
                 static_cast<const float*>(g.X), g.x_stride, g.N, g.K, s, ec);
        ++m->launches;
        prof_stop(m, slot, st, PROF_GEMM, algorithmic_bytes(m, g, ec.T));
        cudaError_t err = cudaGetLastError();
        if (err != cudaSuccess) return check_cuda(err, "GEMM launch");
    }
    return SPEC_OK;
}

int launch_gemm_chain(spec_model* m, const GemmStep* steps, int n, cudaStream_t st) {
    if (n <= 0) return SPEC_OK;
    if (n > kMaxPhases) return set_error(SPEC_ERR_ARG, "GEMM chain longer than kMaxPhases");
    bool has_attn = false;
    for (int p = 0; p < n; ++p) has_attn |= steps[p].kind == PH_ATTN;
    // chain only GEMMs large enough for the grid barriers to pay: below about 16 MB of
    // weights a phase, separate launches overlapped by programmatic dependent launch
    // are faster (measured: 8-layer d-1024 tree verification 0.92 -> 0.86 ms)
    double w_bytes = 0.0;
    for (int p = 0; p < n; ++p)
        if (steps[p].kind != PH_ATTN) w_bytes += (double)steps[p].g.N * steps[p].g.K * m->elem;
    const bool big = w_bytes >= (double)n * kChainMinPhaseBytes;
    bool one_launch = m->bf16 && ((m->chain && big) || has_attn) && (n > 1 || has_attn) && steps[0].e.T <= kMaxTPad;
    for (int p = 1; p < n && one_launch; ++p)
        one_launch = steps[p].e.T == steps[0].e.T && steps[p].e.r0 == steps[0].e.r0;
    if (one_launch) return launch_tc_chain(m, steps, n, st);
    if (has_attn) return set_error(SPEC_ERR_ARG, "attention phase outside a single-launch chain");
    for (int p = 0; p < n; ++p) SPEC_TRY(launch_gemm(m, steps[p].g, steps[p].e, steps[p].xbuf, st));
    return SPEC_OK;
}

}  // namespace spec
