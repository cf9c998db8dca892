// Masked GQA decode attention for calls with few query vectors per (sequence,
// KV head) -- the layer-skip draft's single row, a short chain -- as its own
// launch fed by a TMA ring (bf16 caches).
//
// It computes the attention of attention.cu (query row j of sequence b sees
// the committed slots and the new slots of its ancestors and itself; "FlashSpec"
// page, lnrk.cn/news/47842, sections 2.2 and 5.2).  Decoding reads the whole
// KV context once per step and does little arithmetic on it, so the kernel is
// built around the stream:
//
//  * work: the key range of every (sequence, KV head) segment is cut into
//    16 KB units (4096 / hd slots of K and of V); the units of all segments, in
//    (sequence, head, slot) order, are split evenly over one CTA per SM.
//  * one producer warp: each unit's K and V arrive as 3-D TMA boxes (64 dims x
//    4096 / hd slots, 128-byte swizzle) in a ring of 16 KB slots.  Units made
//    only of committed slots do not depend on the previous kernel, so they go
//    out before the wait for it: the stream starts while that kernel finishes.
//  * eight consumer warps take the CTA's units in turn.  Per unit, with the
//    queries on the MMA's N side (m16n8k16, up to 8 query vectors, bf16 hi + lo
//    splits of Q and P): S^T = K Q^T, the mask, an online softmax per query,
//    O^T += V^T P^T (P^T reaches its operand layout by shuffles).  At the end of
//    a segment the eight warp states merge in shared memory; a segment cut
//    between CTAs leaves one partial state per CTA, merged in CTA order by the
//    last to finish, which writes the output rows (bf16 hi + lo, the O
//    projection's input).
#include "attn_phase.cuh"

namespace spec {

constexpr int kRingQ = 8;                           // query vectors a segment (MMA N)
constexpr int kRingMaxWarps = 8;                    // consumer warps (at most)

struct RingSmem {
    int prefix[kMaxPlanBatch + 1];       // units of the sequences before b
    int base[kMaxPlanBatch];             // committed length of sequence b
    int nrows[kMaxPlanBatch];            // new rows of sequence b
    uint2 qf[2][8][32];                  // Q^T B-fragments (hi, lo) by 16-dim k-step and lane; hd <= 128
    unsigned long long mask[kRingQ];     // visible new slots per query
    float ml[kRingMaxWarps][kRingQ][2];  // per-warp running (max, sum)
    float M[kRingQ], L[kRingQ];
    float o[kRingQ][128];                // merged O of the segment
    float pm[64][kRingQ];                // cross-CTA merge: part maxima, then weights
    float pl[64][kRingQ];                // part sums
    float sc[kRingQ];                    // rescale of the running merge
    int flag;
    int abort;
};

// Shapes of the kernel: consumer warps, ring slots, CTAs an SM (the ring's share of
// shared memory): one CTA of 8 warps and 12 slots, or two of 4 warps and 6 slots.
template <int NW, int NS>
constexpr size_t ring_smem_bytes() { return 1024 + (size_t)NS * kAttnUnitBytes + 2 * NS * 8 + sizeof(RingSmem); }
static_assert(ring_smem_bytes<8, 12>() <= 227 * 1024, "attention ring does not fit in shared memory");
static_assert(2 * ring_smem_bytes<4, 6>() <= 228 * 1024, "two attention rings do not fit in an SM");

static_assert(8 < 12 && 4 < 6, "the consumer warps take ring positions in turn: the ring must be longer");

template <int NW>
SPEC_DEV void ring_bar() { named_bar(1, 32 * NW); }

// (sequence, KV head, slot tile) of unit u; every sequence has >= 1 unit per head
SPEC_DEV AttnUnit ring_locate(const RingSmem& S, int batch, int n_kvh, long long u) {
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

// One unit of one consumer warp: S^T = K Q^T over the unit's KU slots (queries on
// N), mask, online softmax per query, O^T += V^T P^T.  The unit holds K boxes then
// V boxes (64 dims x KU slots each, 128 B rows, 128-byte swizzle: 16-byte chunk ch
// of row r sits at chunk ch ^ (r & 7)).  Lane (g, c) owns queries 2c, 2c+1.
template <int HD>
SPEC_DEV void ring_unit(const uint8_t* tile, const uint2 (&qh)[HD / 16], const uint2 (&ql)[HD / 16], int key0,
                        int base, int n_keys, int nq, unsigned long long mk0, unsigned long long mk1,
                        float (&o)[HD / 16][4], float (&m_r)[2], float (&l_r)[2], int lane) {
    constexpr int KU = 4096 / HD, MT = KU / 16, KS = HD / 16, DT = HD / 16, BOX = KU * 128, NB = HD / 64;
    const uint32_t kb = smem_u32(tile), vb = kb + NB * BOX;
    const int g = lane >> 2, c = lane & 3, mi = lane >> 3, r8 = lane & 7;
    // S^T: A fragments of K by ldmatrix (keys mt*16 + (mi & 1)*8 + r8, dim chunk 2 ks + (mi >> 1))
    float s[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
        const int cd = 2 * ks + (mi >> 1);
        uint32_t a[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int key = mt * 16 + ((mi & 1) << 3) + r8;
            ldmatrix_x4(kb + (cd >> 3) * BOX + key * 128 + (((cd & 7) ^ (key & 7)) << 4), a[mt][0], a[mt][1],
                        a[mt][2], a[mt][3]);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma16816(s[mt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], qh[ks].x, qh[ks].y);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mma16816(s[mt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], ql[ks].x, ql[ks].y);
    }
    // lane (g, c): s[mt] = (key mt*16+g: q 2c, 2c+1), (key mt*16+g+8: q 2c, 2c+1)
    const bool tail = key0 + KU > base;
    const bool q0ok = 2 * c < nq, q1ok = 2 * c + 1 < nq;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int key = key0 + mt * 16 + g + 8 * h;
            bool v0 = q0ok, v1 = q1ok;
            if (tail) {
                const bool in = key < n_keys;
                const bool old = key < base;
                v0 = v0 && in && (old || ((mk0 >> (key - base)) & 1ull));
                v1 = v1 && in && (old || ((mk1 >> (key - base)) & 1ull));
            }
            if (!v0) s[mt][2 * h] = -INFINITY;
            if (!v1) s[mt][2 * h + 1] = -INFINITY;
        }
    }
    // online softmax per query: max and sum over the unit's keys (the 8 lanes of a c)
    float alpha[2];
#pragma unroll
    for (int qq = 0; qq < 2; ++qq) {
        float mt_ = -INFINITY;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) mt_ = fmaxf(mt_, fmaxf(s[mt][qq], s[mt][2 + qq]));
        mt_ = fmaxf(mt_, __shfl_xor_sync(0xffffffffu, mt_, 4));
        mt_ = fmaxf(mt_, __shfl_xor_sync(0xffffffffu, mt_, 8));
        mt_ = fmaxf(mt_, __shfl_xor_sync(0xffffffffu, mt_, 16));
        const float mn = fmaxf(m_r[qq], mt_);
        float ps = 0.f;
        if (mn == -INFINITY) {
            alpha[qq] = 1.f;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) s[mt][qq] = s[mt][2 + qq] = 0.f;
        } else {
            alpha[qq] = (m_r[qq] == -INFINITY) ? 0.f : expf(m_r[qq] - mn);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                s[mt][qq] = expf(s[mt][qq] - mn);
                s[mt][2 + qq] = expf(s[mt][2 + qq] - mn);
                ps += s[mt][qq] + s[mt][2 + qq];
            }
        }
        ps += __shfl_xor_sync(0xffffffffu, ps, 4);
        ps += __shfl_xor_sync(0xffffffffu, ps, 8);
        ps += __shfl_xor_sync(0xffffffffu, ps, 16);
        l_r[qq] = l_r[qq] * alpha[qq] + ps;
        m_r[qq] = mn;
    }
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
        o[dt][0] *= alpha[0];
        o[dt][2] *= alpha[0];
        o[dt][1] *= alpha[1];
        o[dt][3] *= alpha[1];
    }
    // O^T += V^T P^T per 16-slot step kt.  P^T B-fragment of lane (g, c): slots
    // 2c, 2c+1 (b0) and 2c+8, 2c+9 (b1) of query g, gathered by shuffles from the
    // lanes holding them in the S^T layout (slot row r of query n: lane r*4 + n/2).
    const int srcA = (2 * c) * 4 + (g >> 1), srcB = (2 * c + 1) * 4 + (g >> 1);
    const bool odd = g & 1;
#pragma unroll
    for (int kt = 0; kt < MT; ++kt) {
        const float a0 = __shfl_sync(0xffffffffu, s[kt][0], srcA), a1 = __shfl_sync(0xffffffffu, s[kt][1], srcA);
        const float b0 = __shfl_sync(0xffffffffu, s[kt][0], srcB), b1 = __shfl_sync(0xffffffffu, s[kt][1], srcB);
        const float c0 = __shfl_sync(0xffffffffu, s[kt][2], srcA), c1 = __shfl_sync(0xffffffffu, s[kt][3], srcA);
        const float d0 = __shfl_sync(0xffffffffu, s[kt][2], srcB), d1 = __shfl_sync(0xffffffffu, s[kt][3], srcB);
        const float p0 = odd ? a1 : a0, p1 = odd ? b1 : b0;     // slots 2c, 2c+1
        const float p8 = odd ? c1 : c0, p9 = odd ? d1 : d0;     // slots 2c+8, 2c+9
        const uint32_t ph0 = pack_bf16(p0, p1), ph1 = pack_bf16(p8, p9);
        const uint32_t pl0 = pack_bf16_lo(p0, p1), pl1 = pack_bf16_lo(p8, p9);
        // slots past the range hold anything (p is 0 there, but 0 * inf is not): clear them
        uint32_t zm0 = 0xffffffffu, zm1 = 0xffffffffu;
        if (tail) {
            const int ka = key0 + kt * 16 + 2 * c;
            zm0 = (ka < n_keys ? 0x0000ffffu : 0u) | (ka + 1 < n_keys ? 0xffff0000u : 0u);
            zm1 = (ka + 8 < n_keys ? 0x0000ffffu : 0u) | (ka + 9 < n_keys ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
            // A = V^T (dims x slots) by ldmatrix.trans of V rows: matrix mi holds
            // slots kt*16 + (mi >> 1)*8 + r8 at dim chunk 2 dt + (mi & 1)
            const int key = kt * 16 + ((mi >> 1) << 3) + r8;
            const int cd = 2 * dt + (mi & 1);
            uint32_t v0, v1, v2, v3;
            ldmatrix_x4_trans(vb + (cd >> 3) * BOX + key * 128 + (((cd & 7) ^ (key & 7)) << 4), v0, v1, v2, v3);
            v0 &= zm0;
            v1 &= zm0;
            v2 &= zm1;
            v3 &= zm1;
            mma16816(o[dt], v0, v1, v2, v3, ph0, ph1);
            mma16816(o[dt], v0, v1, v2, v3, pl0, pl1);
        }
    }
}

// Output rows of a segment: O / L as bf16 hi + lo (the O projection's input).
template <int HD>
SPEC_DEV void ring_store_rows(const AttnParams& a, int row0, int nq, int Gq, int g, const float* O, const float* L,
                              int t, int nt) {
    const int qdim = a.n_heads * HD;
    for (int i = t; i < nq * HD; i += nt) {
        const int qi = i / HD, d = i % HD;
        store_act(static_cast<__nv_bfloat16*>(a.out), (size_t)(row0 + qi / Gq) * qdim + (g * Gq + qi % Gq) * HD + d,
                  a.out_lo, O[qi * 128 + d] / L[qi]);
    }
}

template <int HD, int kRingWarps, int kRingSlots>
__global__ void __launch_bounds__(32 * (kRingWarps + 1), kRingWarps == 8 ? 1 : 2)
attn_ring_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, AttnParams a) {
    constexpr int KU = 4096 / HD, KS = HD / 16, DT = HD / 16, NB = HD / 64;
    constexpr uint32_t BOXB = KU * 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)kRingSlots * kAttnUnitBytes);
    uint64_t* empty = full + kRingSlots;
    RingSmem& S = *reinterpret_cast<RingSmem*>(empty + kRingSlots);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, G = gridDim.x;
    const int Hkv = a.n_kv_heads, Gq = a.n_heads / a.n_kv_heads;
    volatile int* abort_flag = &S.abort;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kRingSlots; ++i) { mbar_init(full + i, 1); mbar_init(empty + i, 1); }
        S.abort = 0;
        fence_mbar_init();
    }
    // unit table: the row plan was written at least two launches back (every kernel
    // of the stream triggers its dependants only after its own wait)
    if (warp == kRingWarps) {
        int run = 0;
        for (int b0 = 0; b0 < a.batch; b0 += 32) {
            const int b = b0 + lane;
            int u = 0;
            if (b < a.batch) {
                const int base = __ldcg(a.plan.seq_base + b), nr = __ldcg(a.plan.seq_nrows + b);
                int nk = base + nr;
                if (nk > a.kv_ctx) {
                    dev_error(a.err, SPEC_DEVERR_CAPACITY);
                    nk = a.kv_ctx;
                }
                S.base[b] = base;
                S.nrows[b] = nr;
                u = Hkv * ((nk + KU - 1) / KU);
            }
            int x = u;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            if (b < a.batch) S.prefix[b] = run + x - u;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) S.prefix[a.batch] = run;
    }
    __syncthreads();
    const long long U = S.prefix[a.batch];
    const int Ga = attn_ctas(U, G);
    long long ub, ue;
    attn_range(U, G, c, ub, ue);

    if (warp == kRingWarps) {
        // ---- producer: the CTA's units in order into the ring
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            const uint64_t pol = l2_policy_evict_first();
            bool dep = false, ok = true;
            int slot = 0;
            uint32_t par = 0;
            long long issued = 0;
            for (long long u = ub; u < ue; ++u) {
                const AttnUnit au = ring_locate(S, a.batch, Hkv, u);
                const int key0 = au.tile * KU;
                // units holding new (or unused) slots wait for the kernel that writes them
                if (!dep && key0 + KU > S.base[au.b]) {
                    pdl_wait();
                    dep = true;
                }
                if (!mbar_wait(empty + slot, par ^ 1u, abort_flag, a.err)) { ok = false; break; }
                long long row = kv_row_in_layer(a.kvp, Hkv, au.b, au.g, key0);   // a unit never crosses a page
                if (row < 0) { dev_error(a.err, SPEC_DEVERR_CAPACITY); row = 0; }
                uint8_t* dst = ring + (size_t)slot * kAttnUnitBytes;
                mbar_arrive_expect_tx(full + slot, kAttnUnitBytes);
#pragma unroll
                for (int db = 0; db < NB; ++db) {
                    tma_load_3d(dst + db * BOXB, &tmK, 64 * db, (int)row, a.layer, full + slot, pol);
                    tma_load_3d(dst + (NB + db) * BOXB, &tmV, 64 * db, (int)row, a.layer, full + slot, pol);
                }
                ++issued;
                if (++slot == kRingSlots) { slot = 0; par ^= 1u; }
            }
            if (!dep) pdl_wait();
            if (!ok || *abort_flag) {
                // let every copy still in flight land before the CTA leaves
                const long long n = issued < kRingSlots ? issued : kRingSlots;
                for (long long i = 0; i < n; ++i) {
                    if (--slot < 0) { slot = kRingSlots - 1; par ^= 1u; }
                    mbar_wait(full + slot, par, nullptr, a.err);
                }
            }
        }
    } else {
        // ---- consumers
        const int t = threadIdx.x;                       // 0 .. 255
        const int g8 = lane >> 2, cq = lane & 3;
        pdl_wait();                                      // the queries come from the previous kernel
        if (t == 0) pdl_trigger();
        const int qdim = a.n_heads * HD;
        for (long long su = ub; su < ue;) {
            const AttnUnit au = ring_locate(S, a.batch, Hkv, su);
            const int b = au.b, g = au.g;
            const long long seg_first = S.prefix[b] + (long long)g * au.tiles;
            const long long seg_end = min(ue, seg_first + au.tiles);
            const int base = S.base[b], T_b = S.nrows[b];
            const int n_keys = min(base + T_b, a.kv_ctx);
            const int row0 = __ldcg(a.plan.seq_row0 + b);
            const int nq = min(T_b * Gq, kRingQ);
            // Q^T fragments of the segment: lane (g8, cq) of k-step ks holds query g8 at dims
            // 16 ks + 2 cq, +1 (x) and 16 ks + 2 cq + 8, +9 (y), bf16 hi and lo
            for (int i = t; i < KS * 32; i += 32 * kRingWarps) {
                const int ks = i >> 5, ln = i & 31, qi = ln >> 2, fc = ln & 3;
                float x[4] = {0.f, 0.f, 0.f, 0.f};
                if (qi < nq) {
                    const float* qp = a.q + (size_t)(row0 + qi / Gq) * qdim + (g * Gq + qi % Gq) * HD + 16 * ks + 2 * fc;
                    x[0] = __ldcg(qp);
                    x[1] = __ldcg(qp + 1);
                    x[2] = __ldcg(qp + 8);
                    x[3] = __ldcg(qp + 9);
                }
                S.qf[0][ks][ln] = make_uint2(pack_bf16(x[0], x[1]), pack_bf16(x[2], x[3]));
                S.qf[1][ks][ln] = make_uint2(pack_bf16_lo(x[0], x[1]), pack_bf16_lo(x[2], x[3]));
            }
            if (t < kRingQ) {
                unsigned long long mk = 0ull;
                if (t < nq) {
                    const int j = t / Gq;
                    if (a.tree) {
                        for (int x = j; x >= 0; x = __ldcg(a.plan.tree_parent + x)) mk |= 1ull << x;
                    } else {
                        mk = (j >= 63) ? ~0ull : ((2ull << j) - 1ull);
                    }
                }
                S.mask[t] = mk;
            }
            ring_bar<kRingWarps>();
            uint2 qh[KS], ql[KS];
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                qh[ks] = S.qf[0][ks][lane];
                ql[ks] = S.qf[1][ks][lane];
            }
            const unsigned long long mk0 = S.mask[2 * cq], mk1 = S.mask[2 * cq + 1];
            float o[DT][4];
#pragma unroll
            for (int dt = 0; dt < DT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
            float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
            // this warp's units: those whose index in the CTA's range is warp (mod 8)
            const long long u0 = su + ((warp - (int)((su - ub) % kRingWarps) + kRingWarps) % kRingWarps);
            int slot = (int)((u0 - ub) % kRingSlots);
            for (long long u = u0; u < seg_end; u += kRingWarps) {
                const bool w_ok = ring_wait_full(full, empty, u - ub, kRingSlots, abort_flag, a.err);
                if (!w_ok) break;
                const int key0 = (int)(u - seg_first) * KU;
                ring_unit<HD>(ring + (size_t)slot * kAttnUnitBytes, qh, ql, key0, base, n_keys, nq, mk0, mk1, o, m_r,
                              l_r, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(empty + slot);
                for (slot += kRingWarps; slot >= kRingSlots; slot -= kRingSlots) {}
            }
            // merge the eight warps' states (fixed order)
            if (g8 == 0) {
                S.ml[warp][2 * cq][0] = m_r[0];
                S.ml[warp][2 * cq][1] = l_r[0];
                S.ml[warp][2 * cq + 1][0] = m_r[1];
                S.ml[warp][2 * cq + 1][1] = l_r[1];
            }
            ring_bar<kRingWarps>();
            if (t < kRingQ) {
                float M = -INFINITY, L = 0.f;
#pragma unroll
                for (int w = 0; w < kRingWarps; ++w) M = fmaxf(M, S.ml[w][t][0]);
                if (M != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kRingWarps; ++w)
                        if (S.ml[w][t][0] != -INFINITY) L += S.ml[w][t][1] * expf(S.ml[w][t][0] - M);
                }
                S.M[t] = M;
                S.L[t] = L;
            }
            if (t == 0) S.flag = *abort_flag;
            ring_bar<kRingWarps>();
            const float s0 = (m_r[0] == -INFINITY) ? 0.f : expf(m_r[0] - S.M[2 * cq]);
            const float s1 = (m_r[1] == -INFINITY) ? 0.f : expf(m_r[1] - S.M[2 * cq + 1]);
            // o[dt]: (dim dt*16 + g8, q 2cq), (same, 2cq+1), (dim + 8, 2cq), (dim + 8, 2cq+1)
#pragma unroll
            for (int w = 0; w < kRingWarps; ++w) {
                if (warp == w) {
#pragma unroll
                    for (int dt = 0; dt < DT; ++dt) {
                        float* r0p = &S.o[2 * cq][dt * 16 + g8];
                        float* r1p = &S.o[2 * cq + 1][dt * 16 + g8];
                        if (w == 0) {
                            r0p[0] = o[dt][0] * s0; r1p[0] = o[dt][1] * s1;
                            r0p[8] = o[dt][2] * s0; r1p[8] = o[dt][3] * s1;
                        } else {
                            r0p[0] += o[dt][0] * s0; r1p[0] += o[dt][1] * s1;
                            r0p[8] += o[dt][2] * s0; r1p[8] += o[dt][3] * s1;
                        }
                    }
                }
                ring_bar<kRingWarps>();
            }
            if (S.flag) break;
            const int first_c = attn_cta_of(U, Ga, seg_first), last_c = attn_cta_of(U, Ga, seg_first + au.tiles - 1);
            if (first_c == last_c) {
                ring_store_rows<HD>(a, row0, nq, Gq, g, &S.o[0][0], S.L, t, 32 * kRingWarps);
            } else {
                // partial state of this CTA: slot 1 when the segment is not the CTA's first
                const int pslot = (c == first_c && ub < seg_first) ? 1 : 0;
                float* pp = a.part + (size_t)(c * 2 + pslot) * kAttnMaxQ * (HD + 2);
                for (int i = t; i < nq * (HD + 2); i += 32 * kRingWarps) {
                    const int qi = i / (HD + 2), d = i % (HD + 2);
                    pp[i] = d == 0 ? S.M[qi] : (d == 1 ? S.L[qi] : S.o[qi][d - 2]);
                }
                ring_bar<kRingWarps>();
                if (t == 0) S.flag = (atomic_add_acq_rel(a.counters + b * Hkv + g, 1) == last_c - first_c);
                ring_bar<kRingWarps>();
                if (S.flag) {
                    // last CTA of the segment: merge the parts in CTA order, 64 at a time
                    auto part_of = [&](int cp) {
                        const int sl = (cp == first_c && attn_unit_begin(U, Ga, cp) < seg_first) ? 1 : 0;
                        return a.part + (size_t)(cp * 2 + sl) * kAttnMaxQ * (HD + 2);
                    };
                    const int n_parts = last_c - first_c + 1;
                    constexpr int E = (kRingQ * HD + 32 * kRingWarps - 1) / (32 * kRingWarps);
                    float acc[E];
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[e] = 0.f;
                    if (t < nq) {
                        S.M[t] = -INFINITY;
                        S.L[t] = 0.f;
                    }
                    for (int p0 = 0; p0 < n_parts; p0 += 64) {
                        const int np = min(64, n_parts - p0);
                        ring_bar<kRingWarps>();
                        for (int i = t; i < np * nq; i += 32 * kRingWarps) {
                            const int pp2 = i / nq, q = i % nq;
                            const float* src = part_of(first_c + p0 + pp2) + q * (HD + 2);
                            S.pm[pp2][q] = __ldcg(src);
                            S.pl[pp2][q] = __ldcg(src + 1);
                        }
                        ring_bar<kRingWarps>();
                        if (t < nq) {
                            const float m_old = S.M[t];
                            float mn = m_old;
                            for (int pp2 = 0; pp2 < np; ++pp2) mn = fmaxf(mn, S.pm[pp2][t]);
                            const float sc_old = (m_old == -INFINITY) ? 0.f : expf(m_old - mn);
                            float L = S.L[t] * sc_old;
                            for (int pp2 = 0; pp2 < np; ++pp2) {
                                const float m = S.pm[pp2][t];
                                const float wgt = (m == -INFINITY) ? 0.f : expf(m - mn);
                                S.pm[pp2][t] = wgt;
                                L += S.pl[pp2][t] * wgt;
                            }
                            S.M[t] = mn;
                            S.L[t] = L;
                            S.sc[t] = sc_old;
                        }
                        ring_bar<kRingWarps>();
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            const int i = t + 32 * kRingWarps * e;
                            if (i >= nq * HD) break;
                            const int qi = i / HD, d = i % HD;
                            float acc2 = acc[e] * S.sc[qi];
                            for (int pp0 = 0; pp0 < np; pp0 += 8) {
                                float v[8];
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    v[j] = pp0 + j < np ? __ldcg(part_of(first_c + p0 + pp0 + j) + qi * (HD + 2) + 2 + d)
                                                        : 0.f;
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    if (pp0 + j < np) acc2 = fmaf(S.pm[pp0 + j][qi], v[j], acc2);
                            }
                            acc[e] = acc2;
                        }
                    }
#pragma unroll
                    for (int e = 0; e < E; ++e) {
                        const int i = t + 32 * kRingWarps * e;
                        if (i >= nq * HD) break;
                        const int qi = i / HD, d = i % HD;
                        store_act(static_cast<__nv_bfloat16*>(a.out),
                                  (size_t)(row0 + qi / Gq) * qdim + (g * Gq + qi % Gq) * HD + d, a.out_lo,
                                  acc[e] / S.L[qi]);
                    }
                    if (t == 0) a.counters[b * Hkv + g] = 0;
                }
            }
            ring_bar<kRingWarps>();      // S.qf, S.o and S.M are rewritten by the next segment
            su = seg_end;
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------------------
// host
bool attn_ring_fits(const spec_model* m, const spec_kv* kv, int batch, int max_rows_per_seq) {
    const spec_model_config& c = m->cfg;
    return m->bf16 && kv->tmaps && (c.head_dim == 64 || c.head_dim == 128) &&
           max_rows_per_seq * (c.n_heads / c.n_kv_heads) <= kRingQ && batch <= kMaxPlanBatch &&
           m->attn_part_floats >= attn_phase_part_floats(m) && m->n_attn_counters >= batch * c.n_kv_heads;
}

int launch_attention_ring(spec_model* m, const spec_kv* kv, const AttnParams& a0, cudaStream_t st) {
    AttnParams a = a0;
    a.part = m->attn_part;
    a.counters = m->attn_counters;
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(attn_ring_kernel<128, 8, 12>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ring_smem_bytes<8, 12>());
        cudaFuncSetAttribute(attn_ring_kernel<64, 8, 12>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ring_smem_bytes<8, 12>());
        cudaFuncSetAttribute(attn_ring_kernel<128, 4, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ring_smem_bytes<4, 6>());
        cudaFuncSetAttribute(attn_ring_kernel<64, 4, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ring_smem_bytes<4, 6>());
        attr_set = true;
    }
    const int slot = prof_start(m, st);
    cudaError_t e;
    // the CTA count bounds the partial-state slots (2 a CTA) and the units' split
    const int pairs = m->attn_ring_pairs;
    if (pairs) {
        const dim3 grid(std::min(2 * m->num_sms, (int)(m->attn_part_floats / (2 * kAttnMaxQ * (a.head_dim + 2)))));
        if (a.head_dim == 128)
            e = launch_k(m->pdl, attn_ring_kernel<128, 4, 6>, grid, dim3(160), ring_smem_bytes<4, 6>(), st, kv->tm_k,
                         kv->tm_v, a);
        else
            e = launch_k(m->pdl, attn_ring_kernel<64, 4, 6>, grid, dim3(160), ring_smem_bytes<4, 6>(), st, kv->tm_k,
                         kv->tm_v, a);
    } else {
        if (a.head_dim == 128)
            e = launch_k(m->pdl, attn_ring_kernel<128, 8, 12>, dim3(m->num_sms), dim3(288), ring_smem_bytes<8, 12>(),
                         st, kv->tm_k, kv->tm_v, a);
        else
            e = launch_k(m->pdl, attn_ring_kernel<64, 8, 12>, dim3(m->num_sms), dim3(288), ring_smem_bytes<8, 12>(),
                         st, kv->tm_k, kv->tm_v, a);
    }
    ++m->launches;
    prof_stop(m, slot, st, PROF_ATTN, 0.0);
    if (e != cudaSuccess) return check_cuda(e, "attention ring launch");
    return check_cuda(cudaGetLastError(), "attention ring launch");
}

}  // namespace spec
