// Attention as a phase of the GEMM chain kernel (gemm.cu), bf16 caches.
//
// The phase computes the same masked decode attention as attention.cu (query
// row j of sequence b sees the committed slots and the new slots of its
// ancestors and itself; "FlashSpec" page, lnrk.cn/news/47842, sections 2.2 and
// 5.2), with the key loop fed by the chain kernel's TMA ring instead of
// per-thread loads:
//
//  * work: the key range of every (sequence, KV head) pair is cut into units
//    of 8 KB of K (4096 / hd slots); the units of all pairs, in (sequence,
//    head, slot) order, are split evenly over the CTAs.  A unit's K and V
//    arrive as 3-D TMA boxes of 64 dims x (4096 / hd) slots, 128-byte swizzle,
//    into one 16 KB ring slot.  Units made only of committed slots do not
//    depend on the previous kernel (only its new rows do), so the producer
//    issues them before waiting for it.
//  * math: the 4 epilogue warps take a CTA's units in turn.  Per unit:
//    S = Q K^T (m16n8k16 bf16 MMAs, Q as bf16 hi + lo, K fragments by
//    ldmatrix from the swizzled tile), mask, online softmax, O += P V (P as
//    hi + lo, V fragments by ldmatrix.trans).  At the end of a (sequence,
//    head) segment the 4 warp states merge in shared memory; a segment cut
//    between CTAs leaves one partial state per CTA, merged in CTA order by
//    the last to finish, which writes the output rows (bf16 hi + lo, the O
//    projection's input).
#pragma once

#include "model.cuh"

namespace spec {

constexpr uint32_t kAttnUnitBytes = 16384;   // K (8 KB) + V (8 KB) of one unit: one ring A slot

struct AttnSmem {
    int prefix[kMaxPlanBatch + 1];           // units of the sequences before b
    int base[kMaxPlanBatch];                 // committed length of sequence b
    int nrows[kMaxPlanBatch];                // new rows of sequence b
    uint4 q[2 * 8 * 32];                     // Q A-fragments (hi, then lo), hd <= 128; or f32 rows [8][128]
    float o[kAttnMaxQ][128];                 // merged O of the segment
    float ml[4][kAttnMaxQ][2];               // per-warp running (max, sum)
    float M[kAttnMaxQ], L[kAttnMaxQ];
    unsigned long long mask[kAttnMaxQ];      // visible new slots per query
    int flag;
};

__host__ __device__ constexpr int attn_keys_per_unit(int hd) { return 4096 / hd; }

// The attention phase's own ring of 16 KB slots over the chain kernel's shared
// memory: the GEMM ring's weight slots, then its activation-tile region, then
// spare memory.  Its barriers are separate from the GEMM ring's.
constexpr int kAttnMaxSlots = 16;
struct AttnRing {
    uint8_t* a;
    int na;              // slots in the weight region
    uint8_t* b;
    int nb;              // slots in the activation region
    uint8_t* x;          // spare region
    int n;               // all slots
    uint64_t* full;
    uint64_t* empty;
    SPEC_DEV uint8_t* slot(int s) const {
        return s < na ? a + (size_t)s * kAttnUnitBytes
                      : (s < na + nb ? b + (size_t)(s - na) * kAttnUnitBytes : x + (size_t)(s - na - nb) * kAttnUnitBytes);
    }
};

// Unit table of the phase (one warp): prefix[b] = units of sequences < b,
// prefix[batch] = all units; base/nrows copied from the row plan, which an
// earlier kernel wrote (so it may be read before waiting for the previous one).
SPEC_DEV void attn_unit_table(const AttnPhase& A, AttnSmem& S) {
    const int lane = threadIdx.x & 31;
    const int ku = attn_keys_per_unit(A.head_dim);
    int run = 0;
    for (int b0 = 0; b0 < A.batch; b0 += 32) {
        const int b = b0 + lane;
        int u = 0;
        if (b < A.batch) {
            const int base = __ldcg(A.plan.seq_base + b), nr = __ldcg(A.plan.seq_nrows + b);
            int nk = base + nr;
            if (nk > A.kv_ctx) {
                dev_error(A.err, SPEC_DEVERR_CAPACITY);
                nk = A.kv_ctx;
            }
            S.base[b] = base;
            S.nrows[b] = nr;
            u = A.n_kv_heads * ((nk + ku - 1) / ku);
        }
        int x = u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (b < A.batch) S.prefix[b] = run + x - u;
        run += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) S.prefix[A.batch] = run;
    __syncwarp();
}

struct AttnUnit {
    int b, g, tile, tiles;
};

// (sequence, KV head, slot tile) of unit u; every sequence has >= 1 unit per head
SPEC_DEV AttnUnit attn_locate(const AttnSmem& S, int batch, int n_kvh, long long u) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (S.prefix[mid] <= u) lo = mid; else hi = mid - 1;
    }
    AttnUnit r;
    r.b = lo;
    r.tiles = (S.prefix[lo + 1] - S.prefix[lo]) / n_kvh;
    const int rem = (int)(u - S.prefix[lo]);
    r.g = rem / r.tiles;
    r.tile = rem - r.g * r.tiles;
    return r;
}

// The U units go to the first Ga = min(G, U) CTAs, so every CTA of Ga holds at
// least one unit and the CTAs covering a segment are consecutive non-empty ones.
SPEC_DEV int attn_ctas(long long U, int G) { return (int)(U < G ? U : G); }
SPEC_DEV long long attn_unit_begin(long long U, int Ga, int c) { return U * c / Ga; }
SPEC_DEV int attn_cta_of(long long U, int Ga, long long u) { return (int)(((u + 1) * Ga - 1) / U); }
SPEC_DEV void attn_range(long long U, int G, int c, long long& ub, long long& ue) {
    const int Ga = attn_ctas(U, G);
    if (c < Ga) {
        ub = attn_unit_begin(U, Ga, c);
        ue = attn_unit_begin(U, Ga, c + 1);
    } else {
        ub = ue = 0;
    }
}

// One unit (4096 / HD slots) of one warp: S = Q K^T, mask, online softmax, O += P V.
// `tile` holds K boxes then V boxes (64 dims x KU slots each, 128 B rows,
// 128-byte swizzle: 16-byte chunk ch of row r sits at chunk ch ^ (r & 7)).
template <int HD>
SPEC_DEV void attn_unit_mma(const uint8_t* tile, const uint4* sQ, int key0, int base, int n_keys,
                            unsigned long long mk0, unsigned long long mk1, float (&o)[HD / 8][4],
                            float (&m_r)[2], float (&l_r)[2], int lane) {
    constexpr int KU = 4096 / HD, NT = KU / 8, KS = HD / 16, VD = HD / 8, BOX = KU * 128, NB = HD / 64;
    const uint32_t kb = smem_u32(tile), vb = kb + NB * BOX;
    const int cq = lane & 3, mi = lane >> 3, r8 = lane & 7;
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    // S = Q K^T: ldmatrix matrices (slots 8nt.., chunk 2(ks%4)), (same, +1 chunk),
    // (slots 8(nt+1).., chunk), (same, +1): the B fragments of n-tiles nt, nt+1
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const uint4 qh = sQ[ks * 32 + lane], ql = sQ[(KS + ks) * 32 + lane];
        const int db = ks >> 2, ch = ((ks & 3) << 1) + (mi & 1);
        uint32_t bk[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
            const int key = 8 * (nt + (mi >> 1)) + r8;
            ldmatrix_x4(kb + db * BOX + key * 128 + ((ch ^ (key & 7)) << 4), bk[nt][0], bk[nt][1], bk[nt + 1][0],
                        bk[nt + 1][1]);
        }
        // independent accumulators back to back (hi products, then lo)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(sc[nt], qh.x, qh.y, qh.z, qh.w, bk[nt][0], bk[nt][1]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(sc[nt], ql.x, ql.y, ql.z, ql.w, bk[nt][0], bk[nt][1]);
    }
    // lane (g, c) holds rows g (sc[.][0..1]) and g+8 (sc[.][2..3]) at slots key0 + 8nt + 2c + {0, 1}
    const bool tail = key0 + KU > base;
    if (tail) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int key = key0 + 8 * nt + 2 * cq + e;
                const bool in = key < n_keys;
                const bool v0 = in && (key < base || ((mk0 >> (key - base)) & 1ull));
                const bool v1 = in && (key < base || ((mk1 >> (key - base)) & 1ull));
                if (!v0) sc[nt][e] = -INFINITY;
                if (!v1) sc[nt][2 + e] = -INFINITY;
            }
        }
    }
    float alpha[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        float mt = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mt = fmaxf(mt, fmaxf(sc[nt][2 * rr], sc[nt][2 * rr + 1]));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
        const float mn = fmaxf(m_r[rr], mt);
        float ps = 0.f;
        if (mn == -INFINITY) {
            alpha[rr] = 1.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) sc[nt][2 * rr] = sc[nt][2 * rr + 1] = 0.f;
        } else {
            alpha[rr] = (m_r[rr] == -INFINITY) ? 0.f : expf(m_r[rr] - mn);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                sc[nt][2 * rr] = expf(sc[nt][2 * rr] - mn);
                sc[nt][2 * rr + 1] = expf(sc[nt][2 * rr + 1] - mn);
                ps += sc[nt][2 * rr] + sc[nt][2 * rr + 1];
            }
        }
        ps += __shfl_xor_sync(0xffffffffu, ps, 1);
        ps += __shfl_xor_sync(0xffffffffu, ps, 2);
        l_r[rr] = l_r[rr] * alpha[rr] + ps;
        m_r[rr] = mn;
    }
#pragma unroll
    for (int dn = 0; dn < VD; ++dn) {
        o[dn][0] *= alpha[0];
        o[dn][1] *= alpha[0];
        o[dn][2] *= alpha[1];
        o[dn][3] *= alpha[1];
    }
    // O += P V per 16-slot step kk: P A-fragment from S n-tiles 2kk, 2kk+1; V
    // B-fragments by ldmatrix.trans of (slots 16kk.., dim chunk dn), (slots
    // 16kk+8.., dn), (16kk.., dn+1), (16kk+8.., dn+1)
#pragma unroll
    for (int kk = 0; kk < KU / 16; ++kk) {
        const uint32_t ph0 = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]), ph1 = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
        const uint32_t ph2 = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        const uint32_t ph3 = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
        const uint32_t pl0 = pack_bf16_lo(sc[2 * kk][0], sc[2 * kk][1]);
        const uint32_t pl1 = pack_bf16_lo(sc[2 * kk][2], sc[2 * kk][3]);
        const uint32_t pl2 = pack_bf16_lo(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        const uint32_t pl3 = pack_bf16_lo(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
        // slots past the range hold anything (p is 0 there, but 0 * inf is not): clear them
        uint32_t zm0 = 0xffffffffu, zm1 = 0xffffffffu;
        if (tail) {
            const int ka = key0 + 16 * kk + 2 * cq;
            zm0 = (ka < n_keys ? 0x0000ffffu : 0u) | (ka + 1 < n_keys ? 0xffff0000u : 0u);
            zm1 = (ka + 8 < n_keys ? 0x0000ffffu : 0u) | (ka + 9 < n_keys ? 0xffff0000u : 0u);
        }
        uint32_t bv[VD][2];
#pragma unroll
        for (int dn = 0; dn < VD; dn += 2) {
            const int key = 16 * kk + 8 * (mi & 1) + r8;
            const int dch = dn + (mi >> 1);
            ldmatrix_x4_trans(vb + (dch >> 3) * BOX + key * 128 + (((dch & 7) ^ (key & 7)) << 4), bv[dn][0], bv[dn][1],
                              bv[dn + 1][0], bv[dn + 1][1]);
        }
#pragma unroll
        for (int dn = 0; dn < VD; ++dn) {
            bv[dn][0] &= zm0;
            bv[dn][1] &= zm1;
        }
#pragma unroll
        for (int dn = 0; dn < VD; ++dn) mma16816(o[dn], ph0, ph1, ph2, ph3, bv[dn][0], bv[dn][1]);
#pragma unroll
        for (int dn = 0; dn < VD; ++dn) mma16816(o[dn], pl0, pl1, pl2, pl3, bv[dn][0], bv[dn][1]);
    }
}

SPEC_DEV float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
SPEC_DEV float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Reduce-scatter over the warp: lane l holds v[0..31] (partial sums for 32
// slots); afterwards v[0] of lane l is the sum over lanes of v[l].  Each step
// halves the values a lane keeps (31 shuffles in all).
SPEC_DEV float warp_reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < off; ++i) {
            const float send = upper ? v[i] : v[i + off];
            const float keep = upper ? v[i + off] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    return v[0];
}

// One unit of one warp on the CUDA cores, f32 arithmetic, for segments of at
// most NQ query vectors (the draft's single row, short chains).  Lane l owns
// head dims [DPL l, DPL l + DPL): it forms its share of every slot's dot
// product, the warp reduce-scatters so lane l holds slot l's score, and for
// O += P V the lane reads its dims of every V row (contiguous 8-byte pieces).
// LIN: the unit's K rows then V rows in order (bulk copies); else the
// swizzled tensor-box layout of attn_unit_mma.
template <int HD, int NQ, bool LIN>
SPEC_DEV void attn_unit_simt(const uint8_t* tile, const float* qs, int nq, int key0, int base, int n_keys,
                             const unsigned long long* mk, float (&o)[NQ][HD / 32], float (&m_r)[NQ],
                             float (&l_r)[NQ], int lane) {
    constexpr int KU = 4096 / HD, NP = KU / 32, DPL = HD / 32, BOX = KU * 128;
    const int d0 = DPL * lane;
    const int cc = (d0 & 63) >> 3;
    // byte offset of this lane's dims in slot `key` of a K (or V) block
    auto at = [&](int key) -> int {
        if constexpr (LIN) return key * (HD * 2) + d0 * 2;
        else return (d0 >> 6) * BOX + (d0 & 7) * 2 + key * 128 + ((cc ^ (key & 7)) << 4);
    };
    const uint8_t* kt = tile;
    const uint8_t* vt = tile + 8192;
    const int nvalid = min(KU, n_keys - key0);
    float sc[NQ][NP];
#pragma unroll
    for (int ps = 0; ps < NP; ++ps) {
        const int ka = key0 + 32 * ps + lane;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            if (q >= nq) { sc[q][ps] = -INFINITY; continue; }
            // this lane's share of the 32 slots' dot products (K re-read per query: few registers)
            float qr[DPL];
            if constexpr (DPL == 4) {
                const float4 x = *reinterpret_cast<const float4*>(qs + q * 128 + d0);
                qr[0] = x.x; qr[1] = x.y; qr[2] = x.z; qr[3] = x.w;
            } else {
                const float2 x = *reinterpret_cast<const float2*>(qs + q * 128 + d0);
                qr[0] = x.x; qr[1] = x.y;
            }
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int key = 32 * ps + j;
                const uint8_t* src = kt + at(key);
                if constexpr (DPL == 4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(src);
                    float a = qr[0] * bf16_lo_f(w.x);
                    a = fmaf(qr[1], bf16_hi_f(w.x), a);
                    a = fmaf(qr[2], bf16_lo_f(w.y), a);
                    v[j] = fmaf(qr[3], bf16_hi_f(w.y), a);
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
                    v[j] = fmaf(qr[1], bf16_hi_f(w), qr[0] * bf16_lo_f(w));
                }
            }
            const float s = warp_reduce_scatter32(v, lane);
            const bool vis = ka < n_keys && (ka < base || ((mk[q] >> (ka - base)) & 1ull));
            sc[q][ps] = vis ? s : -INFINITY;
        }
    }
    // online softmax per query (each lane holds NP of the unit's slots)
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        float mt = sc[q][0];
#pragma unroll
        for (int ps = 1; ps < NP; ++ps) mt = fmaxf(mt, sc[q][ps]);
        mt = warp_max(mt);
        const float mn = fmaxf(m_r[q], mt);
        float alpha = 1.f, ps_sum = 0.f;
        if (mn == -INFINITY) {
#pragma unroll
            for (int ps = 0; ps < NP; ++ps) sc[q][ps] = 0.f;
        } else {
            alpha = (m_r[q] == -INFINITY) ? 0.f : expf(m_r[q] - mn);
#pragma unroll
            for (int ps = 0; ps < NP; ++ps) {
                sc[q][ps] = expf(sc[q][ps] - mn);
                ps_sum += sc[q][ps];
            }
        }
        ps_sum = warp_sum(ps_sum);
        l_r[q] = l_r[q] * alpha + ps_sum;
        m_r[q] = mn;
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[q][d] *= alpha;
    }
    // O += P V; slots past the range may hold anything, so they read slot 0 (p is 0 there)
#pragma unroll
    for (int ps = 0; ps < NP; ++ps) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            int key = 32 * ps + j;
            key = key < nvalid ? key : 0;
            const uint8_t* src = vt + at(key);
            float vf[DPL];
            if constexpr (DPL == 4) {
                const uint2 w = *reinterpret_cast<const uint2*>(src);
                vf[0] = bf16_lo_f(w.x); vf[1] = bf16_hi_f(w.x); vf[2] = bf16_lo_f(w.y); vf[3] = bf16_hi_f(w.y);
            } else {
                const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
                vf[0] = bf16_lo_f(w); vf[1] = bf16_hi_f(w);
            }
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float pj = __shfl_sync(0xffffffffu, sc[q][ps], j);
#pragma unroll
                for (int d = 0; d < DPL; ++d) o[q][d] = fmaf(pj, vf[d], o[q][d]);
            }
        }
    }
}

// Q fragments of segment (b, g) in fragment order (k-step ks, lane):
// {row r: dims 16ks+2c, +1} {row r+8: same} {row r: 16ks+8+2c, +1} {row r+8: same},
// r = lane / 4, c = lane % 4; then the masks of the segment's queries.
template <int HD>
SPEC_DEV void attn_load_queries(const AttnPhase& A, AttnSmem& S, int b, int g, int row0, int nq, int Gq) {
    constexpr int KS = HD / 16;
    const int t = threadIdx.x & 127;
    const int qdim = A.n_heads * HD;
    for (int i = t; nq > kAttnSimtQ && i < KS * 32; i += 128) {     // MMA path only
        const int ks = i >> 5, ln = i & 31, fg = ln >> 2, fc = ln & 3;
        float x[2][4];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int qi = fg + 8 * rr;
#pragma unroll
            for (int e = 0; e < 4; ++e) x[rr][e] = 0.f;
            if (qi < nq) {
                const float* qp = A.q + (size_t)(row0 + qi / Gq) * qdim + (g * Gq + qi % Gq) * HD + 16 * ks + 2 * fc;
                x[rr][0] = __ldcg(qp);
                x[rr][1] = __ldcg(qp + 1);
                x[rr][2] = __ldcg(qp + 8);
                x[rr][3] = __ldcg(qp + 9);
            }
        }
        S.q[i] = make_uint4(pack_bf16(x[0][0], x[0][1]), pack_bf16(x[1][0], x[1][1]), pack_bf16(x[0][2], x[0][3]),
                            pack_bf16(x[1][2], x[1][3]));
        S.q[KS * 32 + i] = make_uint4(pack_bf16_lo(x[0][0], x[0][1]), pack_bf16_lo(x[1][0], x[1][1]),
                                      pack_bf16_lo(x[0][2], x[0][3]), pack_bf16_lo(x[1][2], x[1][3]));
    }
    if (nq <= kAttnSimtQ) {     // CUDA-core path: the rows in f32, [kAttnSimtQ][128], zero past nq
        float* qs = reinterpret_cast<float*>(S.q);
        for (int i = t; i < kAttnSimtQ * HD; i += 128) {
            const int qi = i / HD, d = i % HD;
            qs[qi * 128 + d] =
                qi < nq ? __ldcg(A.q + (size_t)(row0 + qi / Gq) * qdim + (g * Gq + qi % Gq) * HD + d) : 0.f;
        }
    }
    if (t < kAttnMaxQ) {
        unsigned long long mk = 0ull;
        if (t < nq) {
            const int j = t / Gq;
            if (A.tree) {
                for (int x = j; x >= 0; x = __ldcg(A.plan.tree_parent + x)) mk |= 1ull << x;
            } else {
                mk = (j >= 63) ? ~0ull : ((2ull << j) - 1ull);
            }
        }
        S.mask[t] = mk;
    }
}

// One unit of one warp for a single query vector, plain row layout: the lane's
// K and V pieces of all the unit's slots go to registers first and the ring
// slot is released before any arithmetic, so the slot turns over at copy
// speed.  Then as attn_unit_simt: lane l owns head dims [DPL l, DPL l + DPL).
template <int HD>
SPEC_DEV void attn_unit_q1_early(const uint8_t* tile, uint64_t* release, const float* qs, int key0, int base,
                                 int n_keys, unsigned long long mk, float (&o)[HD / 32], float& m_r, float& l_r,
                                 int lane) {
    constexpr int KU = 4096 / HD, NP = KU / 32, DPL = HD / 32, W = DPL / 2;   // 32-bit words per piece
    const int d0 = DPL * lane;
    const int nvalid = min(KU, n_keys - key0);
    uint32_t kw[KU][W], vw[KU][W];
#pragma unroll
    for (int j = 0; j < KU; ++j) {
        const int key = j < nvalid ? j : 0;            // past the range: slot 0 (masked, p = 0)
        const uint8_t* src = tile + key * (HD * 2) + d0 * 2;
        if constexpr (W == 2) {
            const uint2 a = *reinterpret_cast<const uint2*>(src);
            const uint2 b = *reinterpret_cast<const uint2*>(src + 8192);
            kw[j][0] = a.x; kw[j][1] = a.y; vw[j][0] = b.x; vw[j][1] = b.y;
        } else {
            kw[j][0] = *reinterpret_cast<const uint32_t*>(src);
            vw[j][0] = *reinterpret_cast<const uint32_t*>(src + 8192);
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(release);
    float qr[DPL];
#pragma unroll
    for (int d = 0; d < DPL; ++d) qr[d] = qs[d0 + d];
    float sc[NP];
#pragma unroll
    for (int ps = 0; ps < NP; ++ps) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const uint32_t* k = kw[32 * ps + j];
            float a = qr[0] * bf16_lo_f(k[0]);
            a = fmaf(qr[1], bf16_hi_f(k[0]), a);
            if constexpr (W == 2) {
                a = fmaf(qr[2], bf16_lo_f(k[1]), a);
                a = fmaf(qr[3], bf16_hi_f(k[1]), a);
            }
            v[j] = a;
        }
        const float s = warp_reduce_scatter32(v, lane);
        const int ka = key0 + 32 * ps + lane;
        const bool vis = ka < n_keys && (ka < base || ((mk >> (ka - base)) & 1ull));
        sc[ps] = vis ? s : -INFINITY;
    }
    float mt = sc[0];
#pragma unroll
    for (int ps = 1; ps < NP; ++ps) mt = fmaxf(mt, sc[ps]);
    mt = warp_max(mt);
    const float mn = fmaxf(m_r, mt);
    float alpha = 1.f, psum = 0.f;
    if (mn == -INFINITY) {
#pragma unroll
        for (int ps = 0; ps < NP; ++ps) sc[ps] = 0.f;
    } else {
        alpha = (m_r == -INFINITY) ? 0.f : expf(m_r - mn);
#pragma unroll
        for (int ps = 0; ps < NP; ++ps) {
            sc[ps] = expf(sc[ps] - mn);
            psum += sc[ps];
        }
    }
    psum = warp_sum(psum);
    l_r = l_r * alpha + psum;
    m_r = mn;
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[d] *= alpha;
#pragma unroll
    for (int j = 0; j < KU; ++j) {
        const float pj = __shfl_sync(0xffffffffu, sc[j / 32], j & 31);
        o[0] = fmaf(pj, bf16_lo_f(vw[j][0]), o[0]);
        o[1] = fmaf(pj, bf16_hi_f(vw[j][0]), o[1]);
        if constexpr (W == 2) {
            o[2] = fmaf(pj, bf16_lo_f(vw[j][1]), o[2]);
            o[3] = fmaf(pj, bf16_hi_f(vw[j][1]), o[3]);
        }
    }
}

// Wait for ring position `pos` (slot pos % n, k = pos / n-th use of the slot) to
// be full.  The warps take the positions in turn, so a warp may reach a slot
// before the slot's previous position -- another warp's -- has landed; a parity
// wait on the full barrier alone would then see that earlier phase and return
// at once.  So the warp first waits for the previous position's release (the
// empty barrier's phase k - 1): only this warp can release position pos, so the
// empty barrier is either in phase k - 1 or k and its parity decides.  After
// that release the full barrier is in phase k or k + 1, and the parity of phase
// k decides too.  Bounded; the result is the same on every lane.
SPEC_DEV bool ring_wait_full(uint64_t* full, uint64_t* empty, long long pos, int n, volatile int* abort_flag,
                             int* err) {
    const int slot = (int)(pos % n);
    const uint32_t par = (uint32_t)((pos / n) & 1);
    bool ok = true;
    if (pos >= n) ok = mbar_wait(empty + slot, par ^ 1u, abort_flag, err);
    if (ok) ok = mbar_wait(full + slot, par, abort_flag, err);
    return __all_sync(0xffffffffu, ok);
}

// Running (max, sum) of the segment per query from the four warps' (fixed order).

SPEC_DEV void attn_merge_ml(AttnSmem& S, int t) {
    if (t < kAttnMaxQ) {
        float M = -INFINITY, L = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, S.ml[w][t][0]);
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < 4; ++w)
                if (S.ml[w][t][0] != -INFINITY) L += S.ml[w][t][1] * expf(S.ml[w][t][0] - M);
        }
        S.M[t] = M;
        S.L[t] = L;
    }
}

// The units of one segment that fall to this warp on the CUDA-core path (at
// most NQ query vectors), then the merge of the four warps' states into S.
template <int HD, int NQ, bool LIN>
SPEC_DEV void attn_segment_simt(const AttnPhase& A, AttnSmem& S, const AttnRing& R, long long ring, long long ub,
                                long long su, long long seg_end, long long seg_first, int base, int n_keys, int row0,
                                int g, int nq, int Gq, volatile int* abort_flag, int* err,
                                unsigned long long& kv_bytes) {
    constexpr int KU = 4096 / HD, DPL = HD / 32;
    const int t = threadIdx.x & 127, warp = t >> 5, lane = t & 31;
    const int qdim = A.n_heads * HD;
    float o[NQ][DPL], m_r[NQ], l_r[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
        m_r[q] = -INFINITY;
        l_r[q] = 0.f;
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[q][d] = 0.f;
    }
    const float* qs = reinterpret_cast<const float*>(S.q);     // [kAttnSimtQ][128] query rows (f32)
    const long long u0 = su + ((warp - (int)((su - ub) & 3)) & 3);
    int slot = (int)((ring + (u0 - ub)) % R.n);                  // stepped by 4 below
    for (long long u = u0; u < seg_end; u += 4) {
        const bool w_ok = ring_wait_full(R.full, R.empty, ring + (u - ub), R.n, abort_flag, err);
        if (!w_ok) break;
        const int key0 = (int)(u - seg_first) * KU;
        kv_bytes += (unsigned long long)(min(key0 + KU, n_keys) - key0) * HD * 4;
        if constexpr (LIN && NQ == 1) {
            attn_unit_q1_early<HD>(R.slot(slot), R.empty + slot, qs, key0, base, n_keys, S.mask[0], o[0], m_r[0],
                                   l_r[0], lane);
        } else {
            attn_unit_simt<HD, NQ, LIN>(R.slot(slot), qs, nq, key0, base, n_keys, S.mask, o, m_r, l_r, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(R.empty + slot);
        }
        for (slot += 4; slot >= R.n; slot -= R.n) {}
    }
    if (lane == 0) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            S.ml[warp][q][0] = m_r[q];
            S.ml[warp][q][1] = l_r[q];
        }
    }
    if (lane >= NQ && lane < kAttnMaxQ) {
        S.ml[warp][lane][0] = -INFINITY;
        S.ml[warp][lane][1] = 0.f;
    }
    named_bar(1, 128);
    attn_merge_ml(S, t);
    if (t == 0) S.flag = *abort_flag;
    named_bar(1, 128);
    float sc[NQ];
#pragma unroll
    for (int q = 0; q < NQ; ++q) sc[q] = (m_r[q] == -INFINITY) ? 0.f : expf(m_r[q] - S.M[q]);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        if (warp == w) {
#pragma unroll
            for (int q = 0; q < NQ; ++q)
#pragma unroll
                for (int d = 0; d < DPL; ++d) {
                    float* dst = &S.o[q][DPL * lane + d];
                    *dst = (w == 0 ? 0.f : *dst) + o[q][d] * sc[q];
                }
        }
        named_bar(1, 128);
    }
}

// Output rows of segment (b, g): O / L as bf16 hi + lo.
template <int HD>
SPEC_DEV void attn_store_rows(const AttnPhase& A, int row0, int nq, int Gq, int g, const float* O, int o_stride,
                              const float* L) {
    const int t = threadIdx.x & 127;
    const int qdim = A.n_heads * HD;
    for (int i = t; i < nq * HD; i += 128) {
        const int qi = i / HD, d = i % HD;
        const float v = O[qi * o_stride + d] / L[qi];
        store_act(static_cast<__nv_bfloat16*>(A.out), (size_t)(row0 + qi / Gq) * qdim + (g * Gq + qi % Gq) * HD + d,
                  A.out_lo, v);
    }
}

// The attention phase on the 128 epilogue threads.  `ring` is the ring
// position of the phase's first unit.  Every thread returns the same value
// (false once the CTA has given up on a wait).
template <int HD>
SPEC_DEV bool consume_attn(const AttnPhase& A, AttnSmem& S, const AttnRing& R, int c, int G, volatile int* abort_flag,
                           int* err) {
    const long long ring = 0;     // the phase's units start the attention ring
    constexpr int KU = 4096 / HD, VD = HD / 8;
    const int t = threadIdx.x & 127, warp = t >> 5, lane = t & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int Hkv = A.n_kv_heads, Gq = A.n_heads / A.n_kv_heads;
    const long long U = S.prefix[A.batch];
    const int Ga = attn_ctas(U, G);
    long long ub, ue;
    attn_range(U, G, c, ub, ue);
    unsigned long long kv_bytes = 0;     // K and V bytes of the valid slots this warp used
    for (long long su = ub; su < ue;) {
        const AttnUnit au = attn_locate(S, A.batch, Hkv, su);
        const int b = au.b, g = au.g;
        const long long seg_first = S.prefix[b] + (long long)g * au.tiles;
        const long long seg_end = min(ue, seg_first + au.tiles);
        const int base = S.base[b], T_b = S.nrows[b];
        const int n_keys = min(base + T_b, A.kv_ctx);
        const int row0 = __ldcg(A.plan.seq_row0 + b);
        const int nq = min(T_b * Gq, kAttnMaxQ);
        attn_load_queries<HD>(A, S, b, g, row0, nq, Gq);
        named_bar(1, 128);

        if (nq <= kAttnSimtQ) {
            // few query vectors: CUDA-core path, f32 throughout
            if (A.linear) {
                if (nq == 1)
                    attn_segment_simt<HD, 1, true>(A, S, R, ring, ub, su, seg_end, seg_first, base, n_keys, row0,
                                                   g, nq, Gq, abort_flag, err, kv_bytes);
                else
                    attn_segment_simt<HD, 2, true>(A, S, R, ring, ub, su, seg_end, seg_first, base, n_keys, row0,
                                                   g, nq, Gq, abort_flag, err, kv_bytes);
            } else {
                if (nq == 1)
                    attn_segment_simt<HD, 1, false>(A, S, R, ring, ub, su, seg_end, seg_first, base, n_keys, row0,
                                                    g, nq, Gq, abort_flag, err, kv_bytes);
                else
                    attn_segment_simt<HD, 2, false>(A, S, R, ring, ub, su, seg_end, seg_first, base, n_keys, row0,
                                                    g, nq, Gq, abort_flag, err, kv_bytes);
            }
        } else {
            float o[VD][4];
    #pragma unroll
            for (int dn = 0; dn < VD; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
            float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
            const unsigned long long mk0 = S.mask[gq], mk1 = S.mask[gq + 8];
            // this warp's units: those whose index in the CTA's range is warp (mod 4)
            const long long u0 = su + ((warp - (int)((su - ub) & 3)) & 3);
            int slot = (int)((ring + (u0 - ub)) % R.n);              // stepped by 4 below
                    for (long long u = u0; u < seg_end; u += 4) {
                const bool w_ok = ring_wait_full(R.full, R.empty, ring + (u - ub), R.n, abort_flag, err);
                if (!w_ok) break;
                const int key0 = (int)(u - seg_first) * KU;
                attn_unit_mma<HD>(R.slot(slot), S.q, key0, base, n_keys, mk0, mk1, o, m_r, l_r, lane);
                kv_bytes += (unsigned long long)(min(key0 + KU, n_keys) - key0) * HD * 4;
                __syncwarp();
                if (lane == 0) mbar_arrive(R.empty + slot);
                for (slot += 4; slot >= R.n; slot -= R.n) {}
            }
            // merge the four warps' states (fixed order)
            if (cq == 0) {
                S.ml[warp][gq][0] = m_r[0];
                S.ml[warp][gq][1] = l_r[0];
                S.ml[warp][gq + 8][0] = m_r[1];
                S.ml[warp][gq + 8][1] = l_r[1];
            }
            named_bar(1, 128);
            attn_merge_ml(S, t);
            if (t == 0) S.flag = *abort_flag;
            named_bar(1, 128);
            const float s0 = (m_r[0] == -INFINITY) ? 0.f : expf(m_r[0] - S.M[gq]);
            const float s1 = (m_r[1] == -INFINITY) ? 0.f : expf(m_r[1] - S.M[gq + 8]);
    #pragma unroll
            for (int w = 0; w < 4; ++w) {
                if (warp == w) {
    #pragma unroll
                    for (int dn = 0; dn < VD; ++dn) {
                        float* r0p = &S.o[gq][8 * dn + 2 * cq];
                        float* r1p = &S.o[gq + 8][8 * dn + 2 * cq];
                        if (w == 0) {
                            r0p[0] = o[dn][0] * s0; r0p[1] = o[dn][1] * s0;
                            r1p[0] = o[dn][2] * s1; r1p[1] = o[dn][3] * s1;
                        } else {
                            r0p[0] += o[dn][0] * s0; r0p[1] += o[dn][1] * s0;
                            r1p[0] += o[dn][2] * s1; r1p[1] += o[dn][3] * s1;
                        }
                    }
                }
                named_bar(1, 128);
            }
        }
        if (S.flag) return false;
        const int first_c = attn_cta_of(U, Ga, seg_first), last_c = attn_cta_of(U, Ga, seg_first + au.tiles - 1);
        if (first_c == last_c) {
            attn_store_rows<HD>(A, row0, nq, Gq, g, &S.o[0][0], 128, S.L);
        } else {
            // partial state of this CTA: slot 1 when the segment is not the CTA's first
            const int slot = (c == first_c && ub < seg_first) ? 1 : 0;
            float* pp = A.part + (size_t)(c * 2 + slot) * kAttnMaxQ * (HD + 2);
            for (int i = t; i < nq * (HD + 2); i += 128) {
                const int qi = i / (HD + 2), d = i % (HD + 2);
                pp[i] = d == 0 ? S.M[qi] : (d == 1 ? S.L[qi] : S.o[qi][d - 2]);
            }
            named_bar(1, 128);
            if (t == 0) S.flag = (atomic_add_acq_rel(A.counters + b * Hkv + g, 1) == last_c - first_c);
            named_bar(1, 128);
            if (S.flag) {
                // last CTA of the segment: merge the partials in CTA order
                auto part_of = [&](int cp) {
                    const int sl = (cp == first_c && attn_unit_begin(U, Ga, cp) < seg_first) ? 1 : 0;
                    return A.part + (size_t)(cp * 2 + sl) * kAttnMaxQ * (HD + 2);
                };
                // chunks of up to 64 parts: their (max, sum) pairs load in parallel, the
                // values in batches of 8 independent loads; running merge across chunks
                const int n_parts = last_c - first_c + 1;
                float* pm = reinterpret_cast<float*>(S.q);          // [64][16] part maxima, then weights
                float* pl = pm + 64 * kAttnMaxQ;                    // [64][16] part sums
                constexpr int E = kAttnMaxQ * HD / 128;             // values per thread
                float acc[E];
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = 0.f;
                if (t < nq) {
                    S.M[t] = -INFINITY;
                    S.L[t] = 0.f;
                }
                for (int p0 = 0; p0 < n_parts; p0 += 64) {
                    const int np = min(64, n_parts - p0);
                    named_bar(1, 128);
                    for (int i = t; i < np * nq; i += 128) {
                        const int pp = i / nq, q = i % nq;
                        const float* src = part_of(first_c + p0 + pp) + q * (HD + 2);
                        pm[pp * kAttnMaxQ + q] = __ldcg(src);
                        pl[pp * kAttnMaxQ + q] = __ldcg(src + 1);
                    }
                    named_bar(1, 128);
                    if (t < nq) {
                        const float m_old = S.M[t];
                        float mn = m_old;
                        for (int pp = 0; pp < np; ++pp) mn = fmaxf(mn, pm[pp * kAttnMaxQ + t]);
                        const float sc_old = (m_old == -INFINITY) ? 0.f : expf(m_old - mn);
                        float L = S.L[t] * sc_old;
                        for (int pp = 0; pp < np; ++pp) {
                            const float m = pm[pp * kAttnMaxQ + t];
                            const float w = (m == -INFINITY) ? 0.f : expf(m - mn);
                            pm[pp * kAttnMaxQ + t] = w;
                            L += pl[pp * kAttnMaxQ + t] * w;
                        }
                        S.M[t] = mn;
                        S.L[t] = L;
                        S.ml[0][t][0] = sc_old;
                    }
                    named_bar(1, 128);
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const int i = t + 128 * e;
                        if (i >= nq * HD) break;
                        const int qi = i / HD, d = i % HD;
                        float a = acc[e] * S.ml[0][qi][0];
                        for (int pp0 = 0; pp0 < np; pp0 += 8) {
                            float v[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                v[j] = pp0 + j < np ? __ldcg(part_of(first_c + p0 + pp0 + j) + qi * (HD + 2) + 2 + d)
                                                    : 0.f;
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (pp0 + j < np) a = fmaf(pm[(pp0 + j) * kAttnMaxQ + qi], v[j], a);
                        }
                        acc[e] = a;
                    }
                }
                const int qdim = A.n_heads * HD;
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int i = t + 128 * e;
                    if (i >= nq * HD) break;
                    const int qi = i / HD, d = i % HD;
                    store_act(static_cast<__nv_bfloat16*>(A.out),
                              (size_t)(row0 + qi / Gq) * qdim + (g * Gq + qi % Gq) * HD + d, A.out_lo, acc[e] / S.L[qi]);
                }
                if (t == 0) A.counters[b * Hkv + g] = 0;
            }
        }
        named_bar(1, 128);     // S.q, S.o and S.M are rewritten by the next segment
        su = seg_end;
    }
    if (A.kv_bytes && lane == 0 && kv_bytes) atomicAdd(A.kv_bytes, kv_bytes);
    return true;
}

}  // namespace spec
