// Sampling-mode rows: temperature softmax, top-p nucleus and the integer
// inverse-CDF draw, one CTA per row with the row held in shared memory.
//
// Both sides of a sampling round use one temperature T: q = softmax(draft
// logits / T), p = softmax(target logits / T) ("self-speculative decoding"
// page, m.lqnn.cn/news/278124, section 2.4 on matching temperatures).  Top-p
// follows the page's section 3.4 second option: the draft row stays whole and
// only the target row is cut to its nucleus and renormalised.  The nucleus is
// the shortest run of tokens, by decreasing probability with ties to the lower
// id, whose mass reaches top_p = m * 2^-24; mass is counted in the sampler's
// integer weights w = floor(r * 2^32), so the cut is exact: the run ends at
// the first cumulative weight >= ceil(m * S / 2^24), S = sum w.  The draw is
// the sampler of the acceptance kernel: t = floor(m_u * S / 2^24) for the
// uniform u = m_u * 2^-24, token = smallest x whose inclusive prefix of w
// exceeds t.
//
// Layout: warp w of the 24 owns the contiguous segment [w * seg, (w+1) * seg)
// of the row (seg a multiple of 32), so global loads are coalesced and the
// draw and the tie ranks walk the row in index order.
#include <cfloat>
#include <climits>

#include "model.cuh"

namespace spec {

constexpr int kSampThreads = 768;           // 24 warps: 80 registers a thread, no spills
constexpr int kSampWarps = kSampThreads / 32;

struct SampSmem {
    float f[kSampWarps];
    unsigned long long u[kSampWarps];
    int n[kSampWarps];
    unsigned hist_lo[256], hist_hi[256];   // a bin's weight sum = hi * 2^16 + lo (32-bit atomics)
    unsigned long long above;
    int digit, tok;
};

// floor(r * 2^32) for r in [0, 1] from the bit fields: r = m * 2^(e - 150)
// with the hidden bit in m, so r * 2^32 = m * 2^(e - 118) (denormals give 0).
SPEC_DEV unsigned long long samp_weight(float r) {
    const unsigned b = __float_as_uint(r);
    const int sh = (int)(b >> 23) - 118;
    const unsigned long long m = (b & 0x7FFFFFu) | 0x800000u;
    return sh >= 0 ? (m << sh) : (sh > -24 ? (m >> -sh) : 0ull);
}

// Fixed-order block reductions: lanes by a xor tree, warps in index order.
SPEC_DEV float block_max(float v, SampSmem& sm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) sm.f[threadIdx.x >> 5] = v;
    __syncthreads();
    float m = sm.f[0];
    for (int i = 1; i < kSampWarps; ++i) m = fmaxf(m, sm.f[i]);
    __syncthreads();
    return m;
}

SPEC_DEV float block_sum(float v, SampSmem& sm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) sm.f[threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.f;
    for (int i = 0; i < kSampWarps; ++i) s = __fadd_rn(s, sm.f[i]);
    __syncthreads();
    return s;
}

// Per-warp totals land in sm.u (left there for the caller); returns the block total.
SPEC_DEV unsigned long long block_sum_u64(unsigned long long v, SampSmem& sm) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) sm.u[threadIdx.x >> 5] = v;
    __syncthreads();
    unsigned long long s = 0;
    for (int i = 0; i < kSampWarps; ++i) s += sm.u[i];
    return s;                                   // caller syncs before sm.u is reused
}

// Copy a row segment into shared memory, kLoadBatch independent loads in
// flight per lane; returns the lane's maximum (-FLT_MAX when it has none).
constexpr int kLoadBatch = 8;
template <typename F>
SPEC_DEV float load_segment(float* row, int s0, int s1, F value_at) {
    const int lane = threadIdx.x & 31;
    float mx = -FLT_MAX;
    for (int base = s0; base < s1; base += 32 * kLoadBatch) {
        float v[kLoadBatch];
#pragma unroll
        for (int i = 0; i < kLoadBatch; ++i) {
            const int x = base + i * 32 + lane;
            v[i] = x < s1 ? value_at(x) : -FLT_MAX;
        }
#pragma unroll
        for (int i = 0; i < kLoadBatch; ++i) {
            const int x = base + i * 32 + lane;
            if (x < s1) row[x] = v[i];
            mx = fmaxf(mx, v[i]);
        }
    }
    return mx;
}

// Cut the probability row to its nucleus and renormalise it in place.
//
// The threshold is the bit pattern th of the probability where the mass,
// accumulated from the largest probability down, first reaches need
// (probabilities are >= 0, so their bit patterns order like their values).
// It is found by radix selection, most significant digit first (bits 30..23,
// 22..15, 14..7, 6..0): each pass sums, per digit value, the integer weights of
// the tokens that share the digits fixed so far, and fixes the digit where the
// running mass from the top reaches need.  Tokens equal to th are then kept
// in index order while the mass is short of need.
SPEC_DEV void nucleus(float* row, int s0, int s1, unsigned mp, SampSmem& sm) {
    const int lane = threadIdx.x & 31;
    unsigned long long part = 0;
    for (int x = s0 + lane; x < s1; x += 32) part += samp_weight(row[x]);
    const unsigned long long S = block_sum_u64(part, sm);
    __syncthreads();
    const unsigned long long need = (unsigned long long)mp * (S >> 24) +
                                    (((unsigned long long)mp * (S & 0xFFFFFFull) + 0xFFFFFFull) >> 24);
    unsigned mask = 0u, val = 0u;
    unsigned long long above = 0;                  // mass of the tokens above the fixed prefix
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = pass == 3 ? 0 : 23 - 8 * pass;
        const unsigned dmask = pass == 3 ? 0x7Fu : 0xFFu;
        if (threadIdx.x < 256) { sm.hist_lo[threadIdx.x] = 0u; sm.hist_hi[threadIdx.x] = 0u; }
        __syncthreads();
        for (int x = s0 + lane; x < s1; x += 32) {
            const float r = row[x];
            const unsigned b = __float_as_uint(r);
            if ((b & mask) == val) {
                const unsigned long long w = samp_weight(r);        // <= 2^32
                if (w) {
                    const unsigned d = (b >> shift) & dmask;
                    atomicAdd(&sm.hist_lo[d], (unsigned)(w & 0xFFFFu));
                    atomicAdd(&sm.hist_hi[d], (unsigned)(w >> 16));
                }
            }
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            // lane L holds digits 8L .. 8L+7; suffix sums over the lanes above
            unsigned long long h[8], ls = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                h[i] = ((unsigned long long)sm.hist_hi[8 * lane + i] << 16) + sm.hist_lo[8 * lane + i];
                ls += h[i];
            }
            unsigned long long suf = ls;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long v = __shfl_down_sync(0xffffffffu, suf, o);
                if (lane + o < 32) suf += v;
            }
            const unsigned long long top = above + suf - ls;   // mass of the digits above this lane's
            if (top < need && need <= top + ls) {
                unsigned long long c = top, at = 0;
                int dig = -1;
#pragma unroll
                for (int i = 7; i >= 0; --i) {
                    if (dig < 0) {
                        if (c + h[i] >= need) { dig = 8 * lane + i; at = c; }
                        else c += h[i];
                    }
                }
                sm.digit = dig;
                sm.above = at;
            }
        }
        __syncthreads();
        mask |= dmask << shift;
        val |= (unsigned)sm.digit << shift;
        above = sm.above;
        __syncthreads();
    }
    const float th = __uint_as_float(val);
    const unsigned long long w_th = samp_weight(th);          // > 0: th holds mass
    const unsigned long long n_keep = (need - above + w_th - 1) / w_th;
    int n_eq = 0;
    for (int x = s0 + lane; x < s1; x += 32) n_eq += (row[x] == th);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n_eq += __shfl_xor_sync(0xffffffffu, n_eq, o);
    if (lane == 0) sm.n[threadIdx.x >> 5] = n_eq;
    __syncthreads();
    long long rank = 0;                                       // equal tokens in earlier segments
    for (int i = 0; i < (int)(threadIdx.x >> 5); ++i) rank += sm.n[i];
    float z = 0.f;
    for (int base = s0; base < s1; base += 32) {
        const int x = base + lane;
        const float r = x < s1 ? row[x] : 0.f;
        const bool eq = x < s1 && r == th;
        const unsigned b = __ballot_sync(0xffffffffu, eq);
        const long long my = rank + __popc(b & ((1u << lane) - 1u));
        const bool keep = x < s1 && (r > th || (eq && my < (long long)n_keep));
        if (x < s1 && !keep) row[x] = 0.f;
        z = __fadd_rn(z, keep ? r : 0.f);
        rank += __popc(b);
    }
    __syncthreads();
    const float iz = 1.0f / block_sum(z, sm);
    for (int x = s0 + lane; x < s1; x += 32) row[x] *= iz;
    __syncthreads();
}

// Integer inverse-CDF draw from the row in shared memory; -1 when every weight
// is zero.  The warp segment holding the threshold comes from the segment
// totals, then the whole block scans that segment, one token per thread per step.
SPEC_DEV int draw(const float* row, int V, int seg, float u, SampSmem& sm) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int s0 = min(V, w * seg), s1 = min(V, s0 + seg);
    unsigned long long part = 0;
    for (int x = s0 + lane; x < s1; x += 32) part += samp_weight(row[x]);
    const unsigned long long S = block_sum_u64(part, sm);   // sm.u holds the segment totals
    if (threadIdx.x == 0) sm.tok = INT_MAX;
    unsigned long long m = (unsigned long long)(u * 16777216.0f);
    m = m > 0xFFFFFFull ? 0xFFFFFFull : m;
    const unsigned long long thr = m * (S >> 24) + ((m * (S & 0xFFFFFFull)) >> 24);   // < S when S > 0
    unsigned long long before = 0;
    int ww = 0;
    for (; ww < kSampWarps - 1; ++ww) {
        if (before + sm.u[ww] > thr) break;
        before += sm.u[ww];
    }
    __syncthreads();
    if (S == 0) return -1;
    const int g0 = min(V, ww * seg), g1 = min(V, g0 + seg);
    for (int c0 = g0; c0 < g1; c0 += kSampThreads) {
        const int x = c0 + threadIdx.x;
        unsigned long long inc = x < g1 ? samp_weight(row[x]) : 0ull;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long nb = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += nb;
        }
        if (lane == 31) sm.u[w] = inc;
        __syncthreads();
        unsigned long long off = 0, tot = 0;
        for (int i = 0; i < kSampWarps; ++i) {
            const unsigned long long t = sm.u[i];
            if (i < w) off += t;
            tot += t;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, x < g1 && before + off + inc > thr);
        if (lane == 0 && hit) atomicMin(&sm.tok, c0 + 32 * w + __ffs(hit) - 1);
        __syncthreads();
        if (sm.tok != INT_MAX) break;
        before += tot;
    }
    const int t = sm.tok;
    __syncthreads();
    return t == INT_MAX ? -1 : t;
}

__global__ void __launch_bounds__(kSampThreads, 1)
sample_rows_kernel(SampleArgs a) {
    extern __shared__ float row[];
    __shared__ SampSmem sm;
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int seg = ((a.V + kSampThreads - 1) / kSampThreads) * 32;
    const int s0 = min(a.V, w * seg), s1 = min(a.V, s0 + seg);
    for (int r = blockIdx.x; r < a.rows; r += gridDim.x) {
        const float* __restrict__ in = a.in + (size_t)r * a.in_stride;
        const float mx = block_max(load_segment(row, s0, s1, [&](int x) { return __ldg(in + x); }), sm);
        if (a.temp > 0.f) {
            const float it = 1.0f / a.temp;
            float s = 0.f;
            for (int x = s0 + lane; x < s1; x += 32) {
                const float e = expf((row[x] - mx) * it);
                row[x] = e;
                s += e;
            }
            const float is = 1.0f / block_sum(s, sm);
            for (int x = s0 + lane; x < s1; x += 32) row[x] *= is;
        }
        __syncthreads();
        if (a.top_p_m) nucleus(row, s0, s1, a.top_p_m, sm);
        if (a.out) {
            float* out = a.out + (size_t)r * a.out_stride;
            for (int x = s0 + lane; x < s1; x += 32) out[x] = row[x];
        }
        if (a.u) {
            const int t = draw(row, a.V, seg, a.u[(size_t)r * a.u_stride], sm);
            if (threadIdx.x == 0) {
                a.tok[(size_t)r * a.tok_stride] = t;
                if (t < 0) dev_error(a.err, SPEC_DEVERR_TOKEN);
            }
        }
        __syncthreads();
    }
}

// Rejection-sampling acceptance of one chain per CTA ("self-speculative
// decoding" page, sections 2.4 and 4.3).  Draft token x at position j is kept
// with probability min(1, p_j(x)/q_j(x)) -- zero when q_j(x) = 0 -- tested as
// u_j * q_j(x) < p_j(x), exact in float64 (the product of two float32 values
// has at most 48 significant bits).  At the first rejection the correction is
// drawn from max(0, p_j - q_j) (one float32 subtraction, clipped; section 5.2),
// or from p_j when that residual is all zero; when all k are kept a bonus token
// is drawn from p_k.  u[k] drives the draw.
struct AcceptArgs {
    const float* p; const float* q;
    const int* draft; int draft_stride;
    const float* u;
    int k, V;
    int* acc_len; int* next_tok;
};

// The acceptance streams its one or two rows from memory once: 32 warps each
// own a contiguous segment, walked in steps of 256 tokens (8 loads a lane in
// flight); every step's integer weight sum is kept, so the draw finds its
// segment and step from the sums and re-reads only that step.  Two such CTAs
// fit an SM, so a batch of up to twice the SM count runs in one wave.
constexpr int kAccThreads = 1024;
constexpr int kAccWarps = kAccThreads / 32;
constexpr int kAccStep = 256;
constexpr int kAccMaxSteps = 8;             // vocab <= 32 warps x 8 steps x 256 = 65536
constexpr int kAccMaxVocab = kAccWarps * kAccMaxSteps * kAccStep;

struct AccSmem {
    unsigned long long step[kAccWarps][kAccMaxSteps];
    unsigned long long tot[kAccWarps];
    unsigned long long before;
    int a, wf, sf, tok;
};

__global__ void __launch_bounds__(kAccThreads, 2)
accept_rows_kernel(AcceptArgs a) {
    __shared__ AccSmem sm;
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int k = a.k, V = a.V;
    if (w == 0) {
        bool rej = false;
        if (lane < k) {
            const int x = a.draft[(size_t)b * a.draft_stride + lane];
            if (x < 0 || x >= V) {
                rej = true;
            } else {
                const float qx = a.q[((size_t)b * k + lane) * V + x];
                const float px = a.p[((size_t)b * (k + 1) + lane) * V + x];
                const float uj = a.u[(size_t)b * (k + 1) + lane];
                rej = !(qx > 0.f && (double)uj * (double)qx < (double)px);
            }
        }
        const unsigned mask = __ballot_sync(0xffffffffu, rej);
        if (lane == 0) sm.a = mask ? (__ffs(mask) - 1) : k;
    }
    __syncthreads();
    const int acc = sm.a;
    const int seg = ((V + kAccWarps * kAccStep - 1) / (kAccWarps * kAccStep)) * kAccStep;
    const int s0 = min(V, w * seg), s1 = min(V, s0 + seg);
    const float* __restrict__ pr = a.p + ((size_t)b * (k + 1) + acc) * V;
    const float* __restrict__ qr = a.q + ((size_t)b * k + (acc < k ? acc : 0)) * V;
    // r_x: the residual max(0, p - q) after a rejection (one f32 subtraction), else p
    bool resid = acc < k;
    unsigned long long S = 0;
    for (int pass = 0; pass < 2; ++pass) {
        unsigned long long tot = 0;
        int st = 0;
        for (int base = s0; base < s1; base += kAccStep, ++st) {
            float pv[8], qv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int x = base + i * 32 + lane;
                pv[i] = x < s1 ? __ldg(pr + x) : 0.f;
                qv[i] = (resid && x < s1) ? __ldg(qr + x) : 0.f;
            }
            unsigned long long ws = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) ws += samp_weight(resid ? fmaxf(__fsub_rn(pv[i], qv[i]), 0.f) : pv[i]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
            if (lane == 0) sm.step[w][st] = ws;
            tot += ws;
        }
        if (lane == 0) sm.tot[w] = tot;
        __syncthreads();
        S = 0;
        for (int i = 0; i < kAccWarps; ++i) S += sm.tot[i];
        if (S != 0 || !resid) break;
        resid = false;                         // an all-zero residual: draw from p
        __syncthreads();
    }
    const float uk = a.u[(size_t)b * (k + 1) + k];
    unsigned long long m = (unsigned long long)(uk * 16777216.0f);
    m = m > 0xFFFFFFull ? 0xFFFFFFull : m;
    const unsigned long long thr = m * (S >> 24) + ((m * (S & 0xFFFFFFull)) >> 24);   // < S when S > 0
    if (w == 0) {
        // segment: inclusive prefix of the segment totals over lanes 0..15
        unsigned long long t = lane < kAccWarps ? sm.tot[lane] : 0ull, inc = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long nb = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += nb;
        }
        const unsigned hw = __ballot_sync(0xffffffffu, lane < kAccWarps && inc > thr);
        const int wf = hw ? __ffs(hw) - 1 : 0;
        unsigned long long before = __shfl_sync(0xffffffffu, inc - t, wf);
        // step inside that segment
        const int n_st = (min(V, wf * seg + seg) - min(V, wf * seg) + kAccStep - 1) / kAccStep;
        unsigned long long u2 = lane < n_st ? sm.step[wf][lane] : 0ull, inc2 = u2;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long nb = __shfl_up_sync(0xffffffffu, inc2, o);
            if (lane >= o) inc2 += nb;
        }
        const unsigned hs = __ballot_sync(0xffffffffu, lane < n_st && before + inc2 > thr);
        const int sf = hs ? __ffs(hs) - 1 : 0;
        before += __shfl_sync(0xffffffffu, inc2 - u2, sf);
        // the token inside that step, in index order
        const int g0 = min(V, wf * seg), g1 = min(V, g0 + seg);
        const int base = g0 + sf * kAccStep;
        int found = -1;
        for (int i = 0; i < 8 && found < 0; ++i) {
            const int x = base + i * 32 + lane;
            float r = 0.f;
            if (x < g1) r = resid ? fmaxf(__fsub_rn(__ldg(pr + x), __ldg(qr + x)), 0.f) : __ldg(pr + x);
            unsigned long long incx = samp_weight(r);
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long nb = __shfl_up_sync(0xffffffffu, incx, o);
                if (lane >= o) incx += nb;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, x < g1 && before + incx > thr);
            if (hit) found = base + i * 32 + __ffs(hit) - 1;
            before += __shfl_sync(0xffffffffu, incx, 31);
        }
        if (lane == 0) {
            a.acc_len[b] = acc;
            a.next_tok[b] = S != 0 ? found : -1;
        }
    }
}

// Host side ------------------------------------------------------------------
int launch_sample_rows(const SampleArgs& a, bool pdl, cudaStream_t st) {
    if (a.V < 1 || a.V > kSampMaxVocab)
        return set_error(SPEC_ERR_UNSUPPORTED, "sampling: vocab must be in [1, 53248]");
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(sample_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSampMaxVocab * 4);
        if (e != cudaSuccess) return check_cuda(e, "sampling kernel attribute");
        attr_set = true;
    }
    if (a.rows <= 0) return SPEC_OK;
    cudaError_t e = launch_k(pdl, sample_rows_kernel, dim3(a.rows), dim3(kSampThreads), (size_t)a.V * 4, st, a);
    return check_cuda(e, "sampling kernel launch");
}

static int launch_accept_rows(const AcceptArgs& a, int batch, cudaStream_t st) {
    if (a.V < 1 || a.V > kAccMaxVocab)
        return set_error(SPEC_ERR_UNSUPPORTED, "spec_accept: vocab must be in [1, 65536]");
    cudaError_t e = launch_k(false, accept_rows_kernel, dim3(batch), dim3(kAccThreads), 0, st, a);
    return check_cuda(e, "spec_accept launch");
}

// top_p as the integer m of m * 2^-24 (0 = whole row); an error unless top_p is
// a positive multiple of 2^-24 below 1, or >= 1.
int top_p_to_int(float top_p, unsigned* m) {
    if (!(top_p > 0.f)) return set_error(SPEC_ERR_ARG, "top_p must be positive");
    if (top_p >= 1.f) { *m = 0; return SPEC_OK; }
    const double x = (double)top_p * 16777216.0;
    if (x != (double)(unsigned)x) return set_error(SPEC_ERR_ARG, "top_p must be a multiple of 2^-24");
    *m = (unsigned)x;
    return SPEC_OK;
}

}  // namespace spec

using namespace spec;

extern "C" int spec_probs(const float* logits, int64_t lg_stride, int32_t rows, int32_t vocab, float temperature,
                          float top_p, float* probs, int64_t p_stride, void* stream) {
    if (!logits || !probs) return set_error(SPEC_ERR_ARG, "spec_probs: null pointer");
    if (rows < 0 || vocab < 1 || lg_stride < vocab || p_stride < vocab) return set_error(SPEC_ERR_ARG, "spec_probs: bad sizes");
    if (!(temperature > 0.f) || !(temperature <= FLT_MAX)) return set_error(SPEC_ERR_ARG, "spec_probs: temperature must be positive");
    SampleArgs a{};
    SPEC_TRY(top_p_to_int(top_p, &a.top_p_m));
    a.in = logits; a.in_stride = lg_stride;
    a.out = probs; a.out_stride = p_stride;
    a.rows = rows; a.V = vocab; a.temp = temperature;
    return launch_sample_rows(a, false, (cudaStream_t)stream);
}

extern "C" int spec_sample(const float* probs, int64_t p_stride, int32_t rows, int32_t vocab, const float* u,
                           int32_t* tokens, void* stream) {
    if (!probs || !u || !tokens) return set_error(SPEC_ERR_ARG, "spec_sample: null pointer");
    if (rows < 0 || vocab < 1 || p_stride < vocab) return set_error(SPEC_ERR_ARG, "spec_sample: bad sizes");
    SampleArgs a{};
    a.in = probs; a.in_stride = p_stride;
    a.u = u; a.u_stride = 1;
    a.tok = tokens; a.tok_stride = 1;
    a.rows = rows; a.V = vocab; a.temp = 0.f;
    return launch_sample_rows(a, false, (cudaStream_t)stream);
}

extern "C" int spec_accept(const float* p, const float* q, const int32_t* draft, int32_t draft_stride, const float* u,
                           int32_t batch, int32_t k, int32_t vocab, int32_t* acc_len, int32_t* next_tok, void* stream) {
    if (!p || !q || !draft || !u || !acc_len || !next_tok) return set_error(SPEC_ERR_ARG, "spec_accept: null pointer");
    if (batch <= 0 || k < 1 || k > 32 || vocab <= 0) return set_error(SPEC_ERR_ARG, "spec_accept: bad sizes");
    if (draft_stride == 0) draft_stride = k;
    if (draft_stride < k) return set_error(SPEC_ERR_ARG, "spec_accept: draft_stride < k");
    AcceptArgs a{p, q, draft, draft_stride, u, k, vocab, acc_len, next_tok};
    return launch_accept_rows(a, batch, (cudaStream_t)stream);
}
