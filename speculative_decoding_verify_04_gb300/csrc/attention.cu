// Tree / causal masked decode attention over the KV cache, with GQA.
//
// Query row j of sequence b (committed length s_b, T_b new rows in slots
// s_b .. s_b+T_b-1) sees every committed slot and the new slots of its
// ancestors and itself: a chain row sees new rows 0..j (causal), a tree node
// sees its root-to-node path ("FlashSpec" page, lnrk.cn/news/47842, sections
// 2.2 and 5.2: level-order tree batch under an ancestor mask, padding never
// visible).  Both cases are one 64-bit mask per row over the new slots.
//
// Work split (flash-decoding): CTA (split, kv head, sequence x query block)
// owns up to 16 query vectors -- the (row, head) pairs of one KV head's group,
// so K/V are read once per group (GQA) -- and one contiguous key range.  It
// streams 64-key tiles of K and V through shared memory (16-byte loads),
// keeps a running max / sum / weighted value per query (online softmax), and
// writes that partial state.  The last split of a (sequence, head, block) to
// finish merges the partials in split order and writes the output rows.
#include <algorithm>

#include "model.cuh"

namespace spec {

constexpr int kQPerCta = 16;
constexpr int kKeyTile = 64;
constexpr int kAttnThreads = 128;

struct AttnSmemLayout {
    static size_t bytes(int hd) {
        return sizeof(float) * ((size_t)kKeyTile * (hd + 1) + (size_t)kKeyTile * hd + (size_t)kQPerCta * hd +
                                kQPerCta * (kKeyTile + 1) + 4 * kQPerCta) + sizeof(unsigned long long) * kQPerCta + 16;
    }
};

template <typename KT, int HD>
__global__ void __launch_bounds__(kAttnThreads)
attention_kernel(AttnParams a, int n_rb) {
    constexpr int QPT = kQPerCta * HD / kAttnThreads;   // queries per thread in the PV step
    extern __shared__ float smf[];
    float* sK = smf;                                     // [64][HD+1]
    float* sV = sK + kKeyTile * (HD + 1);                // [64][HD]
    float* sQ = sV + kKeyTile * HD;                      // [16][HD]
    float* sP = sQ + kQPerCta * HD;                      // [16][65]
    float* sM = sP + kQPerCta * (kKeyTile + 1);          // running max
    float* sL = sM + kQPerCta;                           // running sum
    float* sA = sL + kQPerCta;                           // rescale of this tile
    int* sFlag = reinterpret_cast<int*>(sA + kQPerCta);
    unsigned long long* sMask = reinterpret_cast<unsigned long long*>(
        reinterpret_cast<uintptr_t>(sFlag + 4) + 7 & ~uintptr_t(7));

    const int split = blockIdx.x, g = blockIdx.y;
    const int b = blockIdx.z / n_rb, rb = blockIdx.z % n_rb;
    const int t = threadIdx.x;
    const int G = a.n_heads / a.n_kv_heads;
    const int T_b = a.plan.seq_nrows[b];
    const int nq_total = T_b * G;
    const int q0 = rb * kQPerCta;
    if (q0 >= nq_total) return;
    const int nq = min(kQPerCta, nq_total - q0);
    const int base = a.plan.seq_base[b];
    const int n_keys = base + T_b;
    int chunk = (n_keys + a.splits - 1) / a.splits;
    chunk = ((chunk + kKeyTile - 1) / kKeyTile) * kKeyTile;
    const int n_split = (n_keys + chunk - 1) / chunk;
    if (split >= n_split) return;
    const int k_begin = split * chunk, k_end = min(n_keys, k_begin + chunk);
    if (n_keys > a.kv_ctx) { if (t == 0) dev_error(a.err, SPEC_DEVERR_CAPACITY); return; }

    const int row0 = a.plan.seq_row0[b];
    const int qdim = a.n_heads * HD;
    // queries and their visibility masks over the new slots
    for (int i = t; i < nq * HD; i += kAttnThreads) {
        const int qi = i / HD, d = i % HD;
        const int qg = q0 + qi;
        const int j = qg / G, h = g * G + qg % G;
        sQ[qi * HD + d] = a.q[(size_t)(row0 + j) * qdim + h * HD + d];
    }
    if (t < nq) {
        const int j = (q0 + t) / G;
        unsigned long long mk;
        if (a.tree) {
            mk = 0ull;
            for (int x = j; x >= 0; x = a.plan.tree_parent[x]) mk |= 1ull << x;
        } else {
            mk = (j >= 63) ? ~0ull : ((2ull << j) - 1ull);
        }
        sMask[t] = mk;
        sM[t] = -INFINITY;
        sL[t] = 0.f;
    }

    const size_t head_off = (((size_t)a.layer * a.kv_batch + b) * a.n_kv_heads + g) * a.kv_ctx;
    const KT* Kg = static_cast<const KT*>(a.kc) + head_off * HD;
    const KT* Vg = static_cast<const KT*>(a.vc) + head_off * HD;

    const int d_own = t % HD;
    const int i_own = (t / HD) * QPT;
    float acc[QPT];
#pragma unroll
    for (int i = 0; i < QPT; ++i) acc[i] = 0.f;

    for (int kt = k_begin; kt < k_end; kt += kKeyTile) {
        const int nk = min(kKeyTile, k_end - kt);
        __syncthreads();
        // K, V tile -> shared (f32)
        constexpr int VEC = 16 / sizeof(KT);
        for (int i = t; i < kKeyTile * HD / VEC; i += kAttnThreads) {
            const int kk = (i * VEC) / HD, d0 = (i * VEC) % HD;
            if (kk < nk) {
                const uint4 kr = *reinterpret_cast<const uint4*>(Kg + (size_t)(kt + kk) * HD + d0);
                const uint4 vr = *reinterpret_cast<const uint4*>(Vg + (size_t)(kt + kk) * HD + d0);
                const KT* kp = reinterpret_cast<const KT*>(&kr);
                const KT* vp = reinterpret_cast<const KT*>(&vr);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    sK[kk * (HD + 1) + d0 + e] = to_f32<KT>(kp[e]);
                    sV[kk * HD + d0 + e] = to_f32<KT>(vp[e]);
                }
            }
        }
        __syncthreads();
        // scores
        {
            const int kk = t % kKeyTile;
            const int slot = kt + kk;
            for (int qi = t / kKeyTile; qi < nq; qi += kAttnThreads / kKeyTile) {
                float s = -INFINITY;
                const bool vis = kk < nk && (slot < base || ((sMask[qi] >> (slot - base)) & 1ull));
                if (vis) {
                    float dot = 0.f;
#pragma unroll 16
                    for (int d = 0; d < HD; ++d) dot = fmaf(sQ[qi * HD + d], sK[kk * (HD + 1) + d], dot);
                    s = dot;
                }
                sP[qi * (kKeyTile + 1) + kk] = s;
            }
        }
        __syncthreads();
        // online softmax, one warp per query
        {
            const int w = t >> 5, lane = t & 31;
            for (int qi = w; qi < nq; qi += kAttnThreads / 32) {
                const float s0 = sP[qi * (kKeyTile + 1) + lane];
                const float s1 = sP[qi * (kKeyTile + 1) + lane + 32];
                const float mt = warp_max(fmaxf(s0, s1));
                const float mo = sM[qi];
                const float mn = fmaxf(mo, mt);
                float p0 = 0.f, p1 = 0.f, alpha = 1.f;
                if (mn != -INFINITY) {
                    p0 = expf(s0 - mn);
                    p1 = expf(s1 - mn);
                    alpha = (mo == -INFINITY) ? 0.f : expf(mo - mn);
                }
                sP[qi * (kKeyTile + 1) + lane] = p0;
                sP[qi * (kKeyTile + 1) + lane + 32] = p1;
                const float ps = warp_sum(p0 + p1);
                if (lane == 0) {
                    sL[qi] = sL[qi] * alpha + ps;
                    sM[qi] = mn;
                    sA[qi] = alpha;
                }
            }
        }
        __syncthreads();
        // weighted values
#pragma unroll
        for (int i = 0; i < QPT; ++i) {
            const int qi = i_own + i;
            if (qi < nq) {
                float s = acc[i] * sA[qi];
                for (int kk = 0; kk < nk; ++kk) s = fmaf(sP[qi * (kKeyTile + 1) + kk], sV[kk * HD + d_own], s);
                acc[i] = s;
            }
        }
    }

    // partial state
    const int blk = (b * a.n_kv_heads + g) * n_rb + rb;
    float* part = a.part + ((size_t)blk * a.splits + split) * kQPerCta * (HD + 2);
#pragma unroll
    for (int i = 0; i < QPT; ++i) {
        const int qi = i_own + i;
        if (qi < nq) part[qi * (HD + 2) + 2 + d_own] = acc[i];
    }
    if (t < nq) {
        part[t * (HD + 2)] = sM[t];
        part[t * (HD + 2) + 1] = sL[t];
    }
    __threadfence();
    __syncthreads();
    if (t == 0) sFlag[0] = (atomicAdd(a.counters + blk, 1) == n_split - 1);
    __syncthreads();
    if (!sFlag[0]) return;
    __threadfence();
    // merge the splits in order
    const float* pb = a.part + (size_t)blk * a.splits * kQPerCta * (HD + 2);
    for (int i = t; i < nq * HD; i += kAttnThreads) {
        const int qi = i / HD, d = i % HD;
        float M = -INFINITY;
        for (int s = 0; s < n_split; ++s) M = fmaxf(M, __ldcg(pb + ((size_t)s * kQPerCta + qi) * (HD + 2)));
        float L = 0.f, O = 0.f;
        for (int s = 0; s < n_split; ++s) {
            const float* ps = pb + ((size_t)s * kQPerCta + qi) * (HD + 2);
            const float ms = __ldcg(ps);
            if (ms == -INFINITY) continue;
            const float w = expf(ms - M);
            L += __ldcg(ps + 1) * w;
            O += __ldcg(ps + 2 + d) * w;
        }
        const int qg = q0 + qi;
        const int j = qg / G, h = g * G + qg % G;
        store_act(static_cast<KT*>(a.out), (size_t)(row0 + j) * qdim + h * HD + d, a.out_lo, O / L);
    }
    if (t == 0) a.counters[blk] = 0;
}

static int rows_blocks(int max_rows_per_seq, int G) {
    return (max_rows_per_seq * G + kQPerCta - 1) / kQPerCta;
}

// key-range splits per (sequence, kv head, query block): about two CTAs per SM
int attn_splits(const spec_model* m, int blocks, int kv_ctx) {
    int s = std::max(1, std::min(32, (2 * m->num_sms + blocks - 1) / blocks));
    return std::min(s, std::max(1, (kv_ctx + kKeyTile - 1) / kKeyTile));
}

size_t attn_scratch_floats(const spec_model* m, int batch, int max_rows_per_seq, int kv_ctx, int* n_counters) {
    const spec_model_config& c = m->cfg;
    const int n_rb = rows_blocks(max_rows_per_seq, c.n_heads / c.n_kv_heads);
    const int blocks = batch * c.n_kv_heads * n_rb;
    *n_counters = blocks;
    return (size_t)blocks * attn_splits(m, blocks, kv_ctx) * kQPerCta * (c.head_dim + 2);
}

size_t attn_partial_floats_needed(const spec_model* m, int batch, int max_rows_per_seq) {
    const spec_model_config& c = m->cfg;
    const int G = c.n_heads / c.n_kv_heads;
    const int n_rb = rows_blocks(max_rows_per_seq, G);
    return (size_t)batch * c.n_kv_heads * n_rb * 32 * kQPerCta * (c.head_dim + 2);
}

int launch_attention(spec_model* m, const AttnParams& a0, int max_rows_per_seq, cudaStream_t st) {
    AttnParams a = a0;
    const int G = a.n_heads / a.n_kv_heads;
    const int n_rb = rows_blocks(max_rows_per_seq, G);
    const int blocks = a.batch * a.n_kv_heads * n_rb;
    a.splits = attn_splits(m, blocks, a.kv_ctx);
    if ((size_t)blocks * a.splits * kQPerCta * (a.head_dim + 2) > m->attn_part_floats || blocks > m->n_attn_counters)
        return set_error(SPEC_ERR_CAPACITY, "attention workspace too small");
    a.part = m->attn_part;
    a.counters = m->attn_counters;
    dim3 grid(a.splits, a.n_kv_heads, a.batch * n_rb);
    const size_t smem = AttnSmemLayout::bytes(a.head_dim);
    const int slot = prof_start(m, st);
    if (a.head_dim == 128) {
        if (m->bf16) {
            cudaFuncSetAttribute(attention_kernel<__nv_bfloat16, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            attention_kernel<__nv_bfloat16, 128><<<grid, kAttnThreads, smem, st>>>(a, n_rb);
        } else {
            cudaFuncSetAttribute(attention_kernel<float, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            attention_kernel<float, 128><<<grid, kAttnThreads, smem, st>>>(a, n_rb);
        }
    } else {
        if (m->bf16) {
            cudaFuncSetAttribute(attention_kernel<__nv_bfloat16, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            attention_kernel<__nv_bfloat16, 64><<<grid, kAttnThreads, smem, st>>>(a, n_rb);
        } else {
            cudaFuncSetAttribute(attention_kernel<float, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            attention_kernel<float, 64><<<grid, kAttnThreads, smem, st>>>(a, n_rb);
        }
    }
    ++m->launches;
    prof_stop(m, slot, st, PROF_ATTN, 0.0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return check_cuda(e, "attention launch");
    return SPEC_OK;
}

}  // namespace spec
