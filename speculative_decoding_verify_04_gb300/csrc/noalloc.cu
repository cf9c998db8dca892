// spec_verify_noalloc: the verification forward with its per-call scratch in a
// static device array instead of the model's workspace.
//
// Some callers cannot call cudaMalloc at the point where they verify: a
// serving runtime that hands all of the device's memory to its own pool at
// start-up, or a latency-critical loop that cannot afford the device-wide
// synchronisation cudaMalloc and cudaFree may imply.  For them this entry
// point takes the GEMM split-K partial tiles and arrival counters, and the
// attention split partials and counters, from `g_verify_scratch` below.  Every
// GPU that loads the library holds this array (kScratchBytes) until the
// process exits.
#include <mutex>

#include "model.cuh"

namespace spec {

constexpr size_t kScratchBytes = 32ull << 20;     // 32 MiB
static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
static void* g_scratch_addr[kMaxDevices];
static std::mutex g_scratch_mu;

// Device address of the array on the current device; set up on the first call
// per device (host code cannot use the symbol itself as a device address).
static int scratch_address(void** out) {
    int dev = 0;
    int rc = check_cuda(cudaGetDevice(&dev), "spec_verify_noalloc: cudaGetDevice");
    if (rc) return rc;
    if (dev < 0 || dev >= kMaxDevices) return set_error(SPEC_ERR_UNSUPPORTED, "spec_verify_noalloc: device index");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        rc = check_cuda(cudaGetSymbolAddress(&p, g_verify_scratch), "spec_verify_noalloc: cudaGetSymbolAddress");
        if (rc) return rc;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return SPEC_OK;
}

static size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Points the model's scratch fields at the static array for one call and puts
// the model's own workspace back when the call returns.
struct ScratchSwap {
    spec_model* m;
    float* gp; size_t gpf; int* cnt; int ncnt; float* ap; size_t apf; int* ac; int nac;
    explicit ScratchSwap(spec_model* mm)
        : m(mm), gp(mm->gemm_part), gpf(mm->gemm_part_floats), cnt(mm->counters), ncnt(mm->n_counters),
          ap(mm->attn_part), apf(mm->attn_part_floats), ac(mm->attn_counters), nac(mm->n_attn_counters) {}
    ~ScratchSwap() {
        m->gemm_part = gp; m->gemm_part_floats = gpf; m->counters = cnt; m->n_counters = ncnt;
        m->attn_part = ap; m->attn_part_floats = apf; m->attn_counters = ac; m->n_attn_counters = nac;
    }
};

}  // namespace spec

using namespace spec;

extern "C" int spec_verify_noalloc(spec_model* m, spec_kv* kv, int32_t batch, const int32_t* n_rows,
                                   const float* h_in, int32_t h_stride, const int32_t* tokens, int32_t tok_stride,
                                   const int32_t* tree_parent, float* logits, spec_row_stats* stats,
                                   int32_t* acc_len, int32_t* next_tok, int32_t* path, void* stream) {
    // the cheap checks spec_verify makes, before anything is sized or enqueued
    if (!m || !kv || !n_rows || !tokens) return set_error(SPEC_ERR_ARG, "spec_verify_noalloc: null pointer");
    if (kv->m != m) return set_error(SPEC_ERR_ARG, "spec_verify_noalloc: cache of another model");
    if (batch < 1 || batch > kv->batch) return set_error(SPEC_ERR_ARG, "spec_verify_noalloc: bad batch");
    const spec_model_config& c = m->cfg;
    int T = 0, max_r = 1;
    for (int b = 0; b < batch; ++b) {
        if (n_rows[b] < 1 || n_rows[b] > kMaxSeqRows) return set_error(SPEC_ERR_ARG, "n_rows[b] must be in [1, 64]");
        T += n_rows[b];
        max_r = n_rows[b] > max_r ? n_rows[b] : max_r;
    }
    if (T > c.max_rows) return set_error(SPEC_ERR_CAPACITY, "spec_verify_noalloc: sum of n_rows > max_rows");
    // scratch this call needs: counters (zeroed), GEMM partial tiles, attention partials
    const int tp = m->bf16 ? ((std::min(T, kMaxTPad) + 15) / 16) * 16 : 32;
    const int qdim = c.n_heads * c.head_dim;
    const int shapes[5][2] = {{m->qkv_n, c.d_model}, {c.d_model, qdim}, {m->gu_n, c.d_model}, {c.d_model, c.d_ff},
                              {c.vocab, c.d_model}};
    size_t gemm_floats = 0;
    int tiles = 0;
    for (auto& s : shapes) {
        gemm_floats = std::max(gemm_floats, gemm_partial_floats_needed(m, s[0], s[1], tp));
        tiles = std::max(tiles, (s[0] + kTileN - 1) / kTileN);
    }
    int attn_blocks = 0;
    const size_t attn_floats = attn_scratch_floats(m, batch, max_r, kv->max_ctx, &attn_blocks);
    const int n_counters = tiles + 3;     // + chain barrier, chain exits, head tiles
    const size_t cnt_bytes = round256((size_t)(n_counters + attn_blocks) * 4);
    const size_t need = cnt_bytes + round256(gemm_floats * 4) + round256(attn_floats * 4);
    if (need > kScratchBytes)
        return set_error(SPEC_ERR_CAPACITY, "spec_verify_noalloc: this call needs " + std::to_string(need) +
                                                " bytes of scratch; the static array holds " +
                                                std::to_string(kScratchBytes));
    void* base = nullptr;
    int rc = scratch_address(&base);
    if (rc) return rc;
    char* p = static_cast<char*>(base);
    // the array keeps the previous call's contents: the counters must start at zero
    rc = check_cuda(cudaMemsetAsync(p, 0, cnt_bytes, (cudaStream_t)stream), "spec_verify_noalloc: clear counters");
    if (rc) return rc;
    ScratchSwap keep(m);
    m->counters = reinterpret_cast<int*>(p);
    m->n_counters = n_counters;
    m->attn_counters = reinterpret_cast<int*>(p) + n_counters;
    m->n_attn_counters = attn_blocks;
    m->gemm_part = reinterpret_cast<float*>(p + cnt_bytes);
    m->gemm_part_floats = gemm_floats;
    m->attn_part = reinterpret_cast<float*>(p + cnt_bytes + round256(gemm_floats * 4));
    m->attn_part_floats = attn_floats;
    return spec_verify(m, kv, batch, n_rows, h_in, h_stride, tokens, tok_stride, tree_parent, logits, stats,
                       acc_len, next_tok, path, stream);
}
