// Tree / causal masked decode attention over the KV cache, with GQA.
//
// Query row j of sequence b (committed length s_b, T_b new rows in slots
// s_b .. s_b+T_b-1) sees every committed slot and the new slots of its
// ancestors and itself: a chain row sees new rows 0..j (causal), a tree node
// sees its root-to-node path ("FlashSpec" page, lnrk.cn/news/47842, sections
// 2.2 and 5.2: level-order tree batch under an ancestor mask, padding never
// visible).  Both cases are one 64-bit mask per row over the new slots.  A
// tree is one for the batch (tree 1: the plan's first kMaxSeqRows entries) or
// one a sequence (tree 2: entries b * kMaxSeqRows + j).
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

// Merge the split partials of one (sequence, kv head, query block) in split
// order and write the output rows.  Loads go out in parallel: the splits'
// (max, sum) pairs into shared memory first, then the normalised split weights,
// then the weighted values (independent loads, fixed summation order).
template <typename KT, int HD>
__device__ void merge_splits(const AttnParams& a, const float* pb, int n_split, int nq, int q0, int G, int g,
                             int row0, float* sbuf) {
    const int t = threadIdx.x;
    float* sw = sbuf;                            // [n_split][kQPerCta] weights
    float* sm = sbuf + 64 * kQPerCta;            // [n_split][kQPerCta] maxima
    float* sl = sm + 64 * kQPerCta;              // [n_split][kQPerCta] sums
    for (int i = t; i < n_split * nq; i += kAttnThreads) {
        const int s2 = i / nq, qi = i % nq;
        const float* ps = pb + ((size_t)s2 * kQPerCta + qi) * (HD + 2);
        sm[s2 * kQPerCta + qi] = __ldcg(ps);
        sl[s2 * kQPerCta + qi] = __ldcg(ps + 1);
    }
    __syncthreads();
    if (t < nq) {
        float M = -INFINITY;
        for (int s2 = 0; s2 < n_split; ++s2) M = fmaxf(M, sm[s2 * kQPerCta + t]);
        float L = 0.f;
        for (int s2 = 0; s2 < n_split; ++s2) {
            const float ms = sm[s2 * kQPerCta + t];
            const float w = (ms == -INFINITY) ? 0.f : expf(ms - M);
            sw[s2 * kQPerCta + t] = w;
            L += sl[s2 * kQPerCta + t] * w;
        }
        for (int s2 = 0; s2 < n_split; ++s2) sw[s2 * kQPerCta + t] /= L;
    }
    __syncthreads();
    const int qdim = a.n_heads * HD;
    // four consecutive dims per thread; the splits' loads go out in batches of 16
    for (int i = t; i < nq * (HD / 4); i += kAttnThreads) {
        const int qi = i / (HD / 4), d = 4 * (i % (HD / 4));
        float O[4] = {0.f, 0.f, 0.f, 0.f};
        for (int s0 = 0; s0 < n_split; s0 += 16) {
            float v[16][4];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int s2 = s0 + u;
                if (s2 < n_split) {
                    const float* src = pb + ((size_t)s2 * kQPerCta + qi) * (HD + 2) + 2 + d;
                    // rows of HD + 2 floats: 8-byte aligned, so two 8-byte loads
                    const float2 x0 = __ldcg(reinterpret_cast<const float2*>(src));
                    const float2 x1 = __ldcg(reinterpret_cast<const float2*>(src + 2));
                    v[u][0] = x0.x; v[u][1] = x0.y; v[u][2] = x1.x; v[u][3] = x1.y;
                } else {
                    v[u][0] = v[u][1] = v[u][2] = v[u][3] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const float w = (s0 + u < n_split) ? sw[(s0 + u) * kQPerCta + qi] : 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) O[e] += w * v[u][e];
            }
        }
        const int qg = q0 + qi;
        const int j = qg / G, h = g * G + qg % G;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            store_act(static_cast<KT*>(a.out), (size_t)(row0 + j) * qdim + h * HD + d + e, a.out_lo, O[e]);
    }
}

template <typename KT, int HD>
__global__ void __launch_bounds__(kAttnThreads)
attention_kernel(AttnParams a, int n_rb) {
    pdl_wait();
    pdl_trigger();
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
            const int* tp = a.plan.tree_parent + (a.tree == 2 ? (size_t)b * kMaxSeqRows : 0);
            for (int x = j; x >= 0; x = tp[x]) mk |= 1ull << x;
        } else {
            mk = (j >= 63) ? ~0ull : ((2ull << j) - 1ull);
        }
        sMask[t] = mk;
        sM[t] = -INFINITY;
        sL[t] = 0.f;
    }

    const int d_own = t % HD;
    const int i_own = (t / HD) * QPT;
    float acc[QPT];
#pragma unroll
    for (int i = 0; i < QPT; ++i) acc[i] = 0.f;

    for (int kt = k_begin; kt < k_end; kt += kKeyTile) {
        const int nk = min(kKeyTile, k_end - kt);
        long long row = kv_row(a.kvp, a.n_kv_heads, a.layer, b, g, kt);      // a tile never crosses a page
        if (row < 0) { if (t == 0) dev_error(a.err, SPEC_DEVERR_CAPACITY); row = 0; }
        const KT* Kt = static_cast<const KT*>(a.kc) + (size_t)row * HD;
        const KT* Vt = static_cast<const KT*>(a.vc) + (size_t)row * HD;
        __syncthreads();
        // K, V tile -> shared (f32)
        constexpr int VEC = 16 / sizeof(KT);
        for (int i = t; i < kKeyTile * HD / VEC; i += kAttnThreads) {
            const int kk = (i * VEC) / HD, d0 = (i * VEC) % HD;
            if (kk < nk) {
                const uint4 kr = *reinterpret_cast<const uint4*>(Kt + (size_t)kk * HD + d0);
                const uint4 vr = *reinterpret_cast<const uint4*>(Vt + (size_t)kk * HD + d0);
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
    __syncthreads();
    if (t == 0) sFlag[0] = (atomic_add_acq_rel(a.counters + blk, 1) == n_split - 1);
    __syncthreads();
    if (!sFlag[0]) return;
    // merge the splits in order
    const float* pb = a.part + (size_t)blk * a.splits * kQPerCta * (HD + 2);
    merge_splits<KT, HD>(a, pb, n_split, nq, q0, G, g, row0, sK);
    if (t == 0) a.counters[blk] = 0;
}

// Register-resident decode attention for up to RB query vectors per (sequence,
// kv head): the draft passes (one row) and chain verification (k+1 rows).
// A group of LPK lanes holds one K/V row (16 bytes per lane, read once from
// global memory with non-coherent 16-byte loads, U row groups in flight per
// warp); scores are reduced across the group with shuffles and the online
// softmax state (max, sum, weighted values) of each group lives in registers,
// updated once per U keys.  Group states merge through shared memory in a
// fixed order, then splits merge as in the tiled kernel.
template <typename KT, int HD, int RB>
__global__ void __launch_bounds__(kAttnThreads)
attention_decode_kernel(AttnParams a) {
    pdl_wait();
    pdl_trigger();
    constexpr int EPL = 16 / (int)sizeof(KT);        // elements per lane
    constexpr int LPK = HD / EPL;                    // lanes per key row
    constexpr int KPW = 32 / LPK;                    // key rows per warp step
    constexpr int U = (RB <= 2) ? 4 : 2;             // warp steps in flight
    constexpr int NGRP = (kAttnThreads / 32) * KPW;  // lane groups per CTA
    extern __shared__ float smf[];
    float* sState = smf;                             // [NGRP][RB][HD + 2]
    float* sQ = sState + NGRP * RB * (HD + 2);       // [RB][HD]
    int* sFlag = reinterpret_cast<int*>(sQ + RB * HD);

    const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int grp = lane / LPK, lk = lane % LPK;
    const int G = a.n_heads / a.n_kv_heads;
    const int T_b = a.plan.seq_nrows[b];
    const int nq = T_b * G;
    if (nq == 0) return;
    const int base = a.plan.seq_base[b];
    const int n_keys = base + T_b;
    int chunk = (n_keys + a.splits - 1) / a.splits;
    chunk = ((chunk + 31) / 32) * 32;
    const int n_split = (n_keys + chunk - 1) / chunk;
    if (split >= n_split) return;
    if (n_keys > a.kv_ctx) { if (t == 0) dev_error(a.err, SPEC_DEVERR_CAPACITY); return; }
    const int k_begin = split * chunk, k_end = min(n_keys, k_begin + chunk);
    // contiguous quarter of the chunk per warp
    const int per_w = (k_end - k_begin + 3) / 4;
    const int w_begin = k_begin + warp * per_w, w_end = min(k_end, w_begin + per_w);

    const int row0 = a.plan.seq_row0[b];
    const int qdim = a.n_heads * HD;
    for (int i = t; i < RB * HD; i += kAttnThreads) {
        const int r = i / HD, d = i % HD;
        sQ[i] = (r < nq) ? a.q[(size_t)(row0 + r / G) * qdim + (g * G + r % G) * HD + d] : 0.f;
    }
    __syncthreads();
    unsigned long long mk[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        mk[r] = 0ull;
        if (r < nq) {
            const int j = r / G;
            if (a.tree) {
                const int* tp = a.plan.tree_parent + (a.tree == 2 ? (size_t)b * kMaxSeqRows : 0);
                for (int x = j; x >= 0; x = tp[x]) mk[r] |= 1ull << x;
            } else {
                mk[r] = (j >= 63) ? ~0ull : ((2ull << j) - 1ull);
            }
        }
    }
    float m[RB], l[RB], acc[RB][EPL];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[r][e] = 0.f;
    }

    const KT* Kc = static_cast<const KT*>(a.kc) + lk * EPL;
    const KT* Vc = static_cast<const KT*>(a.vc) + lk * EPL;

    for (int kb = w_begin; kb < w_end; kb += KPW * U) {
        uint4 kr[U], vr[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int key = kb + u * KPW + grp;
            const long long row = key < w_end ? kv_row(a.kvp, a.n_kv_heads, a.layer, b, g, key) : -1;
            if (row >= 0) {
                kr[u] = __ldg(reinterpret_cast<const uint4*>(Kc + (size_t)row * HD));
                vr[u] = __ldg(reinterpret_cast<const uint4*>(Vc + (size_t)row * HD));
            } else {
                if (key < w_end) dev_error(a.err, SPEC_DEVERR_CAPACITY);
                kr[u] = make_uint4(0, 0, 0, 0);
                vr[u] = make_uint4(0, 0, 0, 0);
            }
        }
        float sc[U][RB];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const KT* kp = reinterpret_cast<const KT*>(&kr[u]);
            float kf[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) kf[e] = to_f32<KT>(kp[e]);
            const int key = kb + u * KPW + grp;
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float* qr = sQ + r * HD + lk * EPL;
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < EPL; ++e) d = fmaf(qr[e], kf[e], d);
#pragma unroll
                for (int o = LPK / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                const bool vis = r < nq && key < w_end && (key < base || ((mk[r] >> (key - base)) & 1ull));
                sc[u][r] = vis ? d : -INFINITY;
            }
        }
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            float mb = sc[0][r];
#pragma unroll
            for (int u = 1; u < U; ++u) mb = fmaxf(mb, sc[u][r]);
            const float mn = fmaxf(m[r], mb);
            if (mn == -INFINITY) continue;
            const float scale = (m[r] == -INFINITY) ? 0.f : expf(m[r] - mn);
            float p[U], ps = 0.f;
#pragma unroll
            for (int u = 0; u < U; ++u) { p[u] = expf(sc[u][r] - mn); ps += p[u]; }
            l[r] = l[r] * scale + ps;
            m[r] = mn;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                float x = acc[r][e] * scale;
#pragma unroll
                for (int u = 0; u < U; ++u) x = fmaf(p[u], to_f32<KT>(reinterpret_cast<const KT*>(&vr[u])[e]), x);
                acc[r][e] = x;
            }
        }
    }
    // group states -> shared, merged in a fixed order
    const int gi = warp * KPW + grp;
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        float* st = sState + ((size_t)gi * RB + r) * (HD + 2);
        if (lk == 0) { st[0] = m[r]; st[1] = l[r]; }
#pragma unroll
        for (int e = 0; e < EPL; ++e) st[2 + lk * EPL + e] = acc[r][e];
    }
    __syncthreads();
    const int blk = b * a.n_kv_heads + g;
    float* part = a.part + ((size_t)blk * a.splits + split) * kQPerCta * (HD + 2);
    for (int i = t; i < nq * HD; i += kAttnThreads) {
        const int r = i / HD, d = i % HD;
        float M = -INFINITY;
        for (int q2 = 0; q2 < NGRP; ++q2) M = fmaxf(M, sState[((size_t)q2 * RB + r) * (HD + 2)]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int q2 = 0; q2 < NGRP; ++q2) {
                const float* st = sState + ((size_t)q2 * RB + r) * (HD + 2);
                if (st[0] == -INFINITY) continue;
                const float w = expf(st[0] - M);
                L += st[1] * w;
                O += st[2 + d] * w;
            }
        }
        part[r * (HD + 2) + 2 + d] = O;
        if (d == 0) { part[r * (HD + 2)] = M; part[r * (HD + 2) + 1] = L; }
    }
    __syncthreads();
    if (t == 0) sFlag[0] = (atomic_add_acq_rel(a.counters + blk, 1) == n_split - 1);
    __syncthreads();
    if (!sFlag[0]) return;
    const float* pb = a.part + (size_t)blk * a.splits * kQPerCta * (HD + 2);
    __syncthreads();
    merge_splits<KT, HD>(a, pb, n_split, nq, 0, G, g, row0, sState);
    if (t == 0) a.counters[blk] = 0;
}

template <typename KT, int HD, int RB>
static void launch_decode(bool pdl, const AttnParams& a, dim3 grid, cudaStream_t st) {
    constexpr int EPL = 16 / (int)sizeof(KT);
    constexpr int NGRP = (kAttnThreads / 32) * (32 / (HD / EPL));
    const size_t smem = sizeof(float) * (std::max((size_t)NGRP * RB * (HD + 2), (size_t)3 * 64 * kQPerCta) +
                                         RB * HD) + 16;
    static bool set = false;
    if (!set) {
        cudaFuncSetAttribute(attention_decode_kernel<KT, HD, RB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        set = true;
    }
    launch_k(pdl, attention_decode_kernel<KT, HD, RB>, grid, dim3(kAttnThreads), smem, st, a);
}

template <typename KT, int HD>
static void launch_decode_rb(bool pdl, const AttnParams& a, int nq, dim3 grid, cudaStream_t st) {
    if (nq <= 1) launch_decode<KT, HD, 1>(pdl, a, grid, st);
    else if (nq <= 2) launch_decode<KT, HD, 2>(pdl, a, grid, st);
    else if (nq <= 4) launch_decode<KT, HD, 4>(pdl, a, grid, st);
    else launch_decode<KT, HD, 8>(pdl, a, grid, st);
}

// ---------------------------------------------------------------------------
// Tensor-core decode attention (bf16 K/V, mma.sync m16n8k16, f32 accumulate).
//
// A CTA handles 16 query vectors of one (sequence, kv head) -- the M side of
// the MMAs -- over one key range; its 4 warps take 16-key tiles in turn.
// Per tile:  S[16 q x 16 keys] = Q K^T  (Q split into bf16 hi + lo, two MMAs
// per k-step),  online softmax on S,  O += P V  (P split the same way).
// The order of the head dimensions inside a k-step and of the keys inside a
// tile is free (both sides of each product use the same order), so it is
// chosen to make every global load a contiguous 16-byte piece of a K or V row
// and to make the S accumulator fragment the A fragment of P V directly:
//   QK^T, k-step ks = 2*kp + s: lane (g, c) holds logical k {2c, 2c+1, 2c+8,
//     2c+9} = head dims 32*kp + 8*c + 4*s + {0, 1, 2, 3};
//   QK^T, key half h: column n = g is tile key 4*(g/2) + 2*h + g%2, so the S
//     accumulator of lane (g, c) holds tile keys 4c, 4c+1 (half 0) and 4c+2,
//     4c+3 (half 1) -- the A fragment of P V for keys {4c .. 4c+3};
//   P V, n-tile nt: column n = g is head dim (HD/8)*g + nt, so lane (g, c)
//     reads V rows 4c .. 4c+3 at dims (HD/8)*g .. (HD/8)*g + HD/8 - 1.


template <int HD>
__global__ void __launch_bounds__(kAttnThreads)
attention_mma_kernel(AttnParams a, int n_qb) {
    pdl_wait();
    pdl_trigger();
    constexpr int KP = HD / 32;          // 16-byte pieces of a K row per lane
    constexpr int KS = HD / 16;          // QK^T k-steps
    constexpr int VD = HD / 8;           // P V n-tiles = V dims per lane
    constexpr int VP = VD / 8;           // 16-byte pieces of a V row per lane
    extern __shared__ float smf[];
    uint4* sQ = reinterpret_cast<uint4*>(smf);                    // [2][KS][32] fragments (hi, lo)
    float* sState = smf + 2 * KS * 32 * 4;                        // [4 warps][16][HD + 2]
    int* sFlag = reinterpret_cast<int*>(sState + 4 * 16 * (HD + 2));
    unsigned long long* sMask = reinterpret_cast<unsigned long long*>(sFlag + 4);   // [16]

    const int split = blockIdx.x / n_qb, qb = blockIdx.x % n_qb, g = blockIdx.y, b = blockIdx.z;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int gq = lane >> 2, cq = lane & 3;
    const int G = a.n_heads / a.n_kv_heads;
    const int T_b = a.plan.seq_nrows[b];
    const int nq_total = T_b * G;
    const int q0 = qb * 16;
    if (q0 >= nq_total) return;
    const int nq = min(16, nq_total - q0);
    const int base = a.plan.seq_base[b];
    const int n_keys = base + T_b;
    int chunk = (n_keys + a.splits - 1) / a.splits;
    chunk = ((chunk + 63) / 64) * 64;
    const int n_split = (n_keys + chunk - 1) / chunk;
    if (split >= n_split) return;
    if (n_keys > a.kv_ctx) { if (t == 0) dev_error(a.err, SPEC_DEVERR_CAPACITY); return; }
    const int k_begin = split * chunk, k_end = min(n_keys, k_begin + chunk);
    const int row0 = a.plan.seq_row0[b];
    const int qdim = a.n_heads * HD;

    // Q fragments (pre-scaled f32 -> bf16 hi + lo) in shared memory, in lane order
    for (int i = t; i < KS * 32; i += kAttnThreads) {
        const int ks = i / 32, ln = i % 32, fg = ln >> 2, fc = ln & 3;
        const int kp = ks >> 1, s = ks & 1;
        const int d0 = 32 * kp + 8 * fc + 4 * s;
        float x[2][4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int qi = fg + 8 * rr;
#pragma unroll
            for (int e = 0; e < 4; ++e) x[rr][e] = 0.f;
            if (qi < nq) {
                const int qg = q0 + qi;
                const float* qp = a.q + (size_t)(row0 + qg / G) * qdim + (g * G + qg % G) * HD + d0;
#pragma unroll
                for (int e = 0; e < 4; ++e) x[rr][e] = qp[e];
            }
        }
        // A fragment: {row g: k 2c,2c+1} {row g+8: k 2c,2c+1} {row g: k 2c+8,+9} {row g+8: k 2c+8,+9}
        sQ[i] = make_uint4(pack_bf16(x[0][0], x[0][1]), pack_bf16(x[1][0], x[1][1]), pack_bf16(x[0][2], x[0][3]),
                           pack_bf16(x[1][2], x[1][3]));
        sQ[KS * 32 + i] = make_uint4(pack_bf16_lo(x[0][0], x[0][1]), pack_bf16_lo(x[1][0], x[1][1]),
                                     pack_bf16_lo(x[0][2], x[0][3]), pack_bf16_lo(x[1][2], x[1][3]));
    }
    if (t < 16) {
        unsigned long long mk = 0ull;
        if (t < nq) {
            const int j = (q0 + t) / G;
            if (a.tree) {
                const int* tp = a.plan.tree_parent + (a.tree == 2 ? (size_t)b * kMaxSeqRows : 0);
            for (int x = j; x >= 0; x = tp[x]) mk |= 1ull << x;
            } else {
                mk = (j >= 63) ? ~0ull : ((2ull << j) - 1ull);
            }
        }
        sMask[t] = mk;
    }
    __syncthreads();

    const unsigned long long mk0 = sMask[gq], mk1 = sMask[gq + 8];

    float o[VD][4];
#pragma unroll
    for (int nt = 0; nt < VD; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};

    for (int kt = k_begin + 16 * warp; kt < k_end; kt += 64) {
        // the tile's rows: a 16-key tile never crosses a page (keys past the
        // capacity read the last slot's row and are masked)
        long long trow = kv_row(a.kvp, a.n_kv_heads, a.layer, b, g, kt);
        if (trow < 0) { dev_error(a.err, SPEC_DEVERR_CAPACITY); trow = 0; }
        const __nv_bfloat16* Kg = static_cast<const __nv_bfloat16*>(a.kc) + (size_t)trow * HD;
        const __nv_bfloat16* Vg = static_cast<const __nv_bfloat16*>(a.vc) + (size_t)trow * HD;
        uint4 kr[2][KP], vr[4][VP];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int key = min(kt + 4 * (gq >> 1) + 2 * h + (gq & 1), a.kv_ctx - 1);
            const uint4* row = reinterpret_cast<const uint4*>(Kg + (size_t)(key - kt) * HD);
#pragma unroll
            for (int p = 0; p < KP; ++p) kr[h][p] = __ldg(row + 4 * p + cq);
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int key = kt + 4 * cq + r;
            const uint4* row = reinterpret_cast<const uint4*>(Vg + (size_t)(min(key, a.kv_ctx - 1) - kt) * HD);
#pragma unroll
            for (int p = 0; p < VP; ++p) vr[r][p] = __ldg(row + VP * gq + p);
        }
        // S = Q K^T for the two key halves
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const uint4 qh = sQ[ks * 32 + lane], ql = sQ[KS * 32 + ks * 32 + lane];
            const int kp = ks >> 1, s = ks & 1;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t w[4] = {kr[h][kp].x, kr[h][kp].y, kr[h][kp].z, kr[h][kp].w};
                const uint32_t b0 = w[2 * s], b1 = w[2 * s + 1];
                mma16816(sc[h], qh.x, qh.y, qh.z, qh.w, b0, b1);
                mma16816(sc[h], ql.x, ql.y, ql.z, ql.w, b0, b1);
            }
        }
        // mask: lane holds rows g (sc[h][0..1]) and g+8 (sc[h][2..3]) at tile keys 4c + 2h + {0, 1}
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int key = kt + 4 * cq + 2 * h + e;
                const bool in = key < k_end;
                const bool v0 = in && (key < base || ((mk0 >> (key - base)) & 1ull));
                const bool v1 = in && (key < base || ((mk1 >> (key - base)) & 1ull));
                if (!v0) sc[h][e] = -INFINITY;
                if (!v1) sc[h][2 + e] = -INFINITY;
            }
        }
        // online softmax per row (the 16 keys of a row sit in the 4 lanes of a quad)
        float alpha[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            float mt = fmaxf(fmaxf(sc[0][2 * rr], sc[0][2 * rr + 1]), fmaxf(sc[1][2 * rr], sc[1][2 * rr + 1]));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
            mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
            const float mn = fmaxf(m_r[rr], mt);
            float ps = 0.f;
            if (mn == -INFINITY) {
                alpha[rr] = 1.f;
#pragma unroll
                for (int h = 0; h < 2; ++h) sc[h][2 * rr] = sc[h][2 * rr + 1] = 0.f;
            } else {
                alpha[rr] = (m_r[rr] == -INFINITY) ? 0.f : expf(m_r[rr] - mn);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    sc[h][2 * rr] = expf(sc[h][2 * rr] - mn);
                    sc[h][2 * rr + 1] = expf(sc[h][2 * rr + 1] - mn);
                    ps += sc[h][2 * rr] + sc[h][2 * rr + 1];
                }
            }
            ps += __shfl_xor_sync(0xffffffffu, ps, 1);
            ps += __shfl_xor_sync(0xffffffffu, ps, 2);
            l_r[rr] = l_r[rr] * alpha[rr] + ps;
            m_r[rr] = mn;
        }
        // P (A fragment of P V, bf16 hi + lo): keys 4c..4c+1 from half 0, 4c+2..4c+3 from half 1
        const uint32_t pa0 = pack_bf16(sc[0][0], sc[0][1]), pa1 = pack_bf16(sc[0][2], sc[0][3]);
        const uint32_t pa2 = pack_bf16(sc[1][0], sc[1][1]), pa3 = pack_bf16(sc[1][2], sc[1][3]);
        const uint32_t pl0 = pack_bf16_lo(sc[0][0], sc[0][1]), pl1 = pack_bf16_lo(sc[0][2], sc[0][3]);
        const uint32_t pl2 = pack_bf16_lo(sc[1][0], sc[1][1]), pl3 = pack_bf16_lo(sc[1][2], sc[1][3]);
        // keys past the range contribute p = 0; clear their V rows so stale values cannot reach O
#pragma unroll
        for (int r = 0; r < 4; ++r)
            if (kt + 4 * cq + r >= k_end)
#pragma unroll
                for (int p = 0; p < VP; ++p) vr[r][p] = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int nt = 0; nt < VD; ++nt) {
            const int p = nt >> 3, e = nt & 7, wi = e >> 1;
            const uint32_t w0 = (&vr[0][p].x)[wi], w1 = (&vr[1][p].x)[wi];
            const uint32_t w2 = (&vr[2][p].x)[wi], w3 = (&vr[3][p].x)[wi];
            const uint32_t b0 = (e & 1) ? pair_hi(w0, w1) : pair_lo(w0, w1);
            const uint32_t b1 = (e & 1) ? pair_hi(w2, w3) : pair_lo(w2, w3);
            o[nt][0] *= alpha[0];
            o[nt][1] *= alpha[0];
            o[nt][2] *= alpha[1];
            o[nt][3] *= alpha[1];
            mma16816(o[nt], pa0, pa1, pa2, pa3, b0, b1);
            mma16816(o[nt], pl0, pl1, pl2, pl3, b0, b1);
        }
    }
    // warp states -> shared: rows g and g+8, dims VD*2c + nt and VD*(2c+1) + nt
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        float* st = sState + ((size_t)warp * 16 + gq + 8 * rr) * (HD + 2);
        if (cq == 0) { st[0] = m_r[rr]; st[1] = l_r[rr]; }
#pragma unroll
        for (int nt = 0; nt < VD; ++nt) {
            st[2 + VD * (2 * cq) + nt] = o[nt][2 * rr];
            st[2 + VD * (2 * cq + 1) + nt] = o[nt][2 * rr + 1];
        }
    }
    __syncthreads();
    const int blk = ((b * a.n_kv_heads + g) * n_qb) + qb;
    float* part = a.part + ((size_t)blk * a.splits + split) * kQPerCta * (HD + 2);
    for (int i = t; i < nq * HD; i += kAttnThreads) {
        const int r = i / HD, d = i % HD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, sState[((size_t)w * 16 + r) * (HD + 2)]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float* st = sState + ((size_t)w * 16 + r) * (HD + 2);
                if (st[0] == -INFINITY) continue;
                const float wt = expf(st[0] - M);
                L += st[1] * wt;
                O += st[2 + d] * wt;
            }
        }
        part[r * (HD + 2) + 2 + d] = O;
        if (d == 0) { part[r * (HD + 2)] = M; part[r * (HD + 2) + 1] = L; }
    }
    __syncthreads();
    if (t == 0) sFlag[0] = (atomic_add_acq_rel(a.counters + blk, 1) == n_split - 1);
    __syncthreads();
    if (!sFlag[0]) return;
    const float* pb = a.part + (size_t)blk * a.splits * kQPerCta * (HD + 2);
    merge_splits<__nv_bfloat16, HD>(a, pb, n_split, nq, q0, G, g, row0, sState);
    if (t == 0) a.counters[blk] = 0;
}

static size_t mma_smem_bytes(int hd) {
    return sizeof(float) * (2 * (hd / 16) * 32 * 4 + 4 * 16 * (hd + 2)) + 16 + 16 * 8 + 16 * 4 + 64;
}

static int rows_blocks(int max_rows_per_seq, int G) {
    return (max_rows_per_seq * G + kQPerCta - 1) / kQPerCta;
}

// key-range splits of the register-resident kernel: about four CTAs per SM
int decode_splits(const spec_model* m, int blocks, int kv_ctx) {
    int s = std::max(1, std::min(64, (4 * m->num_sms + blocks - 1) / blocks));
    return std::min(s, std::max(1, (kv_ctx + 255) / 256));
}

// key-range splits per (sequence, kv head, query block): about two CTAs per SM
int attn_splits(const spec_model* m, int blocks, int kv_ctx) {
    int s = std::max(1, std::min(32, (2 * m->num_sms + blocks - 1) / blocks));
    return std::min(s, std::max(1, (kv_ctx + kKeyTile - 1) / kKeyTile));
}

// Launch shape of one attention call: bf16 models use the tensor-core kernel
// (query blocks of 16), f32 models the CUDA-core kernels.
struct AttnShape { int kind; int n_qb; int blocks; int splits; };   // kind 0 mma, 1 decode, 2 tiled

static AttnShape attn_shape(const spec_model* m, int batch, int max_rows_per_seq, int kv_ctx) {
    const spec_model_config& c = m->cfg;
    const int G = c.n_heads / c.n_kv_heads;
    const int nq_max = max_rows_per_seq * G;
    AttnShape s{};
    if (m->bf16) {
        // one wave: as many key splits as resident CTAs allow
        static int occ[2] = {0, 0};
        const int hi = c.head_dim == 128;
        if (!occ[hi]) {
            int n = 0;
            if (hi) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attention_mma_kernel<128>, kAttnThreads,
                                                                  mma_smem_bytes(128));
            else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attention_mma_kernel<64>, kAttnThreads,
                                                               mma_smem_bytes(64));
            occ[hi] = std::max(1, n);
        }
        s.kind = 0;
        s.n_qb = (nq_max + 15) / 16;
        s.blocks = batch * c.n_kv_heads * s.n_qb;
        s.splits = std::max(1, std::min(64, (occ[hi] * m->num_sms) / s.blocks));
        // at least 320 keys a split (five 16-key tiles a warp): below that the
        // cross-split merge costs more than the extra CTAs give (measured: the
        // 29-node tree over 2048 keys, 19 -> 8 splits, 22.5 -> 19.3 us a launch)
        s.splits = std::min(s.splits, std::max(1, (kv_ctx + 319) / 320));
    } else if (nq_max <= 8) {
        s.kind = 1;
        s.n_qb = 1;
        s.blocks = batch * c.n_kv_heads;
        s.splits = decode_splits(m, s.blocks, kv_ctx);
    } else {
        s.kind = 2;
        s.n_qb = rows_blocks(max_rows_per_seq, G);
        s.blocks = batch * c.n_kv_heads * s.n_qb;
        s.splits = attn_splits(m, s.blocks, kv_ctx);
    }
    return s;
}

size_t attn_scratch_floats(const spec_model* m, int batch, int max_rows_per_seq, int kv_ctx, int* n_counters) {
    const spec_model_config& c = m->cfg;
    if (m->bf16) {
        const AttnShape sh = attn_shape(m, batch, max_rows_per_seq, kv_ctx);
        // also room for the attention phase of the GEMM chain
        *n_counters = std::max(sh.blocks, batch * c.n_kv_heads);
        return std::max((size_t)sh.blocks * sh.splits * kQPerCta * (c.head_dim + 2), attn_phase_part_floats(m));
    }
    if (max_rows_per_seq * (c.n_heads / c.n_kv_heads) <= 8) {
        const int blocks = batch * c.n_kv_heads;
        *n_counters = blocks;
        return (size_t)blocks * decode_splits(m, blocks, kv_ctx) * kQPerCta * (c.head_dim + 2);
    }
    const int n_rb = rows_blocks(max_rows_per_seq, c.n_heads / c.n_kv_heads);
    const int blocks = batch * c.n_kv_heads * n_rb;
    *n_counters = blocks;
    return (size_t)blocks * attn_splits(m, blocks, kv_ctx) * kQPerCta * (c.head_dim + 2);
}

size_t attn_partial_floats_needed(const spec_model* m, int batch, int max_rows_per_seq) {
    const spec_model_config& c = m->cfg;
    const int G = c.n_heads / c.n_kv_heads;
    const int n_rb = rows_blocks(max_rows_per_seq, G);
    const size_t own = std::max((size_t)batch * c.n_kv_heads * n_rb * 32, (size_t)batch * c.n_kv_heads * 64) *
                       kQPerCta * (c.head_dim + 2);
    return m->bf16 ? std::max(own, attn_phase_part_floats(m)) : own;
}

int launch_attention(spec_model* m, const AttnParams& a0, int max_rows_per_seq, cudaStream_t st) {
    AttnParams a = a0;
    const int G = a.n_heads / a.n_kv_heads;
    const int nq_max = max_rows_per_seq * G;
    if (m->bf16) {
        const AttnShape sh = attn_shape(m, a.batch, max_rows_per_seq, a.kv_ctx);
        a.splits = sh.splits;
        if ((size_t)sh.blocks * a.splits * kQPerCta * (a.head_dim + 2) > m->attn_part_floats ||
            sh.blocks > m->n_attn_counters)
            return set_error(SPEC_ERR_CAPACITY, "attention workspace too small");
        a.part = m->attn_part;
        a.counters = m->attn_counters;
        dim3 grid(a.splits * sh.n_qb, a.n_kv_heads, a.batch);
        const size_t smem = mma_smem_bytes(a.head_dim);
        const int slot = prof_start(m, st);
        cudaError_t e;
        if (a.head_dim == 128)
            e = launch_k(m->pdl, attention_mma_kernel<128>, grid, dim3(kAttnThreads), smem, st, a, sh.n_qb);
        else
            e = launch_k(m->pdl, attention_mma_kernel<64>, grid, dim3(kAttnThreads), smem, st, a, sh.n_qb);
        ++m->launches;
        prof_stop(m, slot, st, PROF_ATTN, 0.0);
        if (e != cudaSuccess) return check_cuda(e, "attention launch");
        return check_cuda(cudaGetLastError(), "attention launch");
    }
    if (nq_max <= 8) {
        // every query vector of a (sequence, kv head) in one register-resident block
        const int blocks = a.batch * a.n_kv_heads;
        a.splits = decode_splits(m, blocks, a.kv_ctx);
        if ((size_t)blocks * a.splits * kQPerCta * (a.head_dim + 2) > m->attn_part_floats ||
            blocks > m->n_attn_counters)
            return set_error(SPEC_ERR_CAPACITY, "attention workspace too small");
        a.part = m->attn_part;
        a.counters = m->attn_counters;
        dim3 grid(a.splits, a.n_kv_heads, a.batch);
        const int slot = prof_start(m, st);
        if (a.head_dim == 128) {
            if (m->bf16) launch_decode_rb<__nv_bfloat16, 128>(m->pdl, a, nq_max, grid, st);
            else launch_decode_rb<float, 128>(m->pdl, a, nq_max, grid, st);
        } else {
            if (m->bf16) launch_decode_rb<__nv_bfloat16, 64>(m->pdl, a, nq_max, grid, st);
            else launch_decode_rb<float, 64>(m->pdl, a, nq_max, grid, st);
        }
        ++m->launches;
        prof_stop(m, slot, st, PROF_ATTN, 0.0);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return check_cuda(e, "attention launch");
        return SPEC_OK;
    }
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
            launch_k(m->pdl, attention_kernel<__nv_bfloat16, 128>, grid, dim3(kAttnThreads), smem, st, a, n_rb);
        } else {
            cudaFuncSetAttribute(attention_kernel<float, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            launch_k(m->pdl, attention_kernel<float, 128>, grid, dim3(kAttnThreads), smem, st, a, n_rb);
        }
    } else {
        if (m->bf16) {
            cudaFuncSetAttribute(attention_kernel<__nv_bfloat16, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            launch_k(m->pdl, attention_kernel<__nv_bfloat16, 64>, grid, dim3(kAttnThreads), smem, st, a, n_rb);
        } else {
            cudaFuncSetAttribute(attention_kernel<float, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            launch_k(m->pdl, attention_kernel<float, 64>, grid, dim3(kAttnThreads), smem, st, a, n_rb);
        }
    }
    ++m->launches;
    prof_stop(m, slot, st, PROF_ATTN, 0.0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return check_cuda(e, "attention launch");
    return SPEC_OK;
}

}  // namespace spec
