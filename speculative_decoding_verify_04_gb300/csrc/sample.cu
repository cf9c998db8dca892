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
// Layout: warp w of the 32 owns the contiguous segment [w * seg, (w+1) * seg)
// of the row (seg a multiple of 32), so global loads are coalesced and the
// draw and the tie ranks walk the row in index order.
#include <cfloat>

#include "model.cuh"

namespace spec {

constexpr int kSampThreads = 1024;
constexpr int kSampWarps = kSampThreads / 32;

struct SampSmem {
    float f[kSampWarps];
    unsigned long long u[kSampWarps];
    int n[kSampWarps];
};

SPEC_DEV unsigned long long samp_weight(float r) {
    return __float2ull_rz(r * 4294967296.0f);    // r in [0, 1]: exact scaling, then floor
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

// Cut the probability row to its nucleus and renormalise it in place.
SPEC_DEV void nucleus(float* row, int V, int s0, int s1, unsigned mp, SampSmem& sm) {
    const int lane = threadIdx.x & 31;
    unsigned long long part = 0;
    for (int x = s0 + lane; x < s1; x += 32) part += samp_weight(row[x]);
    const unsigned long long S = block_sum_u64(part, sm);
    __syncthreads();
    const unsigned long long need = (unsigned long long)mp * (S >> 24) +
                                    (((unsigned long long)mp * (S & 0xFFFFFFull) + 0xFFFFFFull) >> 24);
    // largest bit pattern th (probabilities are >= 0, so bits order like values)
    // with W(q >= th) >= need; W(q > th) is w_hi
    unsigned lo = 0u, hi = 0x3F800001u;
    unsigned long long w_hi = 0;
    while (hi - lo > 1u) {
        const unsigned mid = lo + ((hi - lo) >> 1);
        unsigned long long c = 0;
        for (int x = s0 + lane; x < s1; x += 32) {
            const float r = row[x];
            if (__float_as_uint(r) >= mid) c += samp_weight(r);
        }
        const unsigned long long W = block_sum_u64(c, sm);
        __syncthreads();
        if (W >= need) lo = mid;
        else { hi = mid; w_hi = W; }
    }
    const float th = __uint_as_float(lo);
    const unsigned long long w_th = samp_weight(th);
    // tokens equal to th are kept in index order while the mass is short of need
    const unsigned long long short_by = need - w_hi;          // > 0, and w_th > 0
    const unsigned long long n_keep = (short_by + w_th - 1) / w_th;
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
    const float Z = block_sum(z, sm);
    for (int x = s0 + lane; x < s1; x += 32) row[x] = __fdiv_rn(row[x], Z);
    __syncthreads();
}

// Integer inverse-CDF draw from the row; -1 when every weight is zero.
SPEC_DEV int draw(const float* row, int s0, int s1, float u, SampSmem& sm) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    unsigned long long part = 0;
    for (int x = s0 + lane; x < s1; x += 32) part += samp_weight(row[x]);
    const unsigned long long S = block_sum_u64(part, sm);   // sm.u holds the warp totals
    __shared__ int s_tok;
    if (threadIdx.x == 0) s_tok = -1;
    __syncthreads();
    if (S != 0) {
        unsigned long long m = (unsigned long long)(u * 16777216.0f);
        m = m > 0xFFFFFFull ? 0xFFFFFFull : m;
        const unsigned long long thr = m * (S >> 24) + ((m * (S & 0xFFFFFFull)) >> 24);   // < S
        unsigned long long before = 0;
        int ww = 0;
        for (; ww < kSampWarps - 1; ++ww) {
            if (before + sm.u[ww] > thr) break;
            before += sm.u[ww];
        }
        if (w == ww) {
            int found = -1;
            for (int base = s0; base < s1 && found < 0; base += 32) {
                const int x = base + lane;
                unsigned long long inc = x < s1 ? samp_weight(row[x]) : 0ull;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long nb = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += nb;
                }
                const unsigned hit = __ballot_sync(0xffffffffu, before + inc > thr);
                if (hit) found = base + __ffs(hit) - 1;
                before += __shfl_sync(0xffffffffu, inc, 31);
            }
            if (lane == 0) s_tok = found;
        }
    }
    __syncthreads();
    return s_tok;
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
        const float* in = a.in + (size_t)r * a.in_stride;
        if (a.temp > 0.f) {
            float mx = -FLT_MAX;
            for (int x = s0 + lane; x < s1; x += 32) {
                const float v = in[x];
                row[x] = v;
                mx = fmaxf(mx, v);
            }
            mx = block_max(mx, sm);
            float s = 0.f;
            for (int x = s0 + lane; x < s1; x += 32) {
                const float e = expf(__fdiv_rn(__fsub_rn(row[x], mx), a.temp));
                row[x] = e;
                s = __fadd_rn(s, e);
            }
            const float S = block_sum(s, sm);
            for (int x = s0 + lane; x < s1; x += 32) row[x] = __fdiv_rn(row[x], S);
        } else {
            for (int x = s0 + lane; x < s1; x += 32) row[x] = in[x];
        }
        __syncthreads();
        if (a.top_p_m) nucleus(row, a.V, s0, s1, a.top_p_m, sm);
        if (a.out) {
            float* out = a.out + (size_t)r * a.out_stride;
            for (int x = s0 + lane; x < s1; x += 32) out[x] = row[x];
        }
        if (a.u) {
            const int t = draw(row, s0, s1, a.u[(size_t)r * a.u_stride], sm);
            if (threadIdx.x == 0) {
                a.tok[(size_t)r * a.tok_stride] = t;
                if (t < 0) dev_error(a.err, SPEC_DEVERR_TOKEN);
            }
        }
        __syncthreads();
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
