// Shared device helpers: error word, bounded mbarrier waits, TMA and tcgen05
// inline-PTX wrappers for sm_103a.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "spec.h"

#define SPEC_DEV __device__ __forceinline__

// Launch `kernel` on `st`, with the programmatic-stream-serialization attribute
// when `pdl` is set (the kernel then overlaps the tail of the previous one).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// device error word
SPEC_DEV void dev_error(int* err, int bits) {
    if (err) atomicOr(err, bits);
}

// ---------------------------------------------------------------------------
// numeric helpers
SPEC_DEV float bf16_to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
SPEC_DEV __nv_bfloat16 f32_to_bf16(float x) { return __float2bfloat16_rn(x); }

template <typename T> SPEC_DEV float to_f32(T x);
template <> SPEC_DEV float to_f32<float>(float x) { return x; }
template <> SPEC_DEV float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> SPEC_DEV T from_f32(float x);
template <> SPEC_DEV float from_f32<float>(float x) { return x; }
template <> SPEC_DEV __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Store a GEMM input value.  f32 models store it as is.  bf16 models store a
// pair: hi = bf16(v) at base[o] and lo = bf16(v - hi) at base[o + lo_off]; the
// tensor-core GEMM multiplies both by the same weights into one f32
// accumulator, so the activation keeps ~16 significant bits instead of 8.
SPEC_DEV void store_act(float* base, size_t o, size_t, float v) { base[o] = v; }
SPEC_DEV void store_act(__nv_bfloat16* base, size_t o, size_t lo_off, float v) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    base[o] = hi;
    base[o + lo_off] = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// ---------------------------------------------------------------------------
// shared-memory address of a generic pointer
SPEC_DEV uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SPEC_DEV uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// mbarrier
SPEC_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
SPEC_DEV void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
SPEC_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
                 :: "r"(smem_u32(bar)) : "memory");
}
SPEC_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
SPEC_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Bounded wait: returns false (and raises the CTA abort flag and the device
// error word) if the phase did not complete within `limit_ns`, or if another
// role of the CTA already aborted.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
SPEC_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 255u) == 0u) {
            if (abort_flag && *abort_flag) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                if (abort_flag) *abort_flag = 1;
                dev_error(err, SPEC_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// TMA (tensor copies global -> shared, completion on an mbarrier)
SPEC_DEV void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
SPEC_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, uint64_t* bar,
                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
           "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
SPEC_DEV void tma_load_3d(void* dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z, uint64_t* bar,
                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
           "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// contiguous global -> shared copy (both 16-byte aligned, bytes a multiple of 16)
SPEC_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
SPEC_DEV uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
SPEC_DEV uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------------------
// warp-level bf16 MMA (m16n8k16, f32 accumulate) and its shared-memory loads
SPEC_DEV void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                       uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

SPEC_DEV uint32_t pack_bf16(float lo, float hi) {
    const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
    return l | (h << 16);
}
// residuals of pack_bf16: x - bf16(x) for both halves
SPEC_DEV uint32_t pack_bf16_lo(float lo, float hi) {
    return pack_bf16(lo - __bfloat162float(__float2bfloat16_rn(lo)), hi - __bfloat162float(__float2bfloat16_rn(hi)));
}
// two bf16 from 16-bit halves of two 32-bit words: (low half of x, low half of y) etc.
SPEC_DEV uint32_t pair_lo(uint32_t x, uint32_t y) { return __byte_perm(x, y, 0x5410); }
SPEC_DEV uint32_t pair_hi(uint32_t x, uint32_t y) { return __byte_perm(x, y, 0x7632); }
// four 8x8 b16 matrices from shared memory; lanes 8i..8i+7 give the row
// addresses of matrix i, register i gets matrix i (row lane/4, columns
// 2(lane%4), +1; with .trans: rows 2(lane%4), +1 of column lane/4)
SPEC_DEV void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}
SPEC_DEV void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
SPEC_DEV void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(smem_slot)), "r"(ncols) : "memory");
}
SPEC_DEV void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
SPEC_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
SPEC_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SPEC_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, f32 accumulate)
SPEC_DEV void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// arrive on `bar` once every tcgen05 op issued so far by this thread has completed
SPEC_DEV void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns: thread i of the warp gets lane (base + i)
SPEC_DEV void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, K-major operand written by TMA with the
// 128-byte swizzle: rows of 64 bf16 (128 B), 8-row atoms of 1024 B.
//   bits  0-13  start address >> 4      bits 16-29  leading byte offset >> 4
//   bits 32-45  stride byte offset >> 4 bits 46-47  descriptor version (1)
//   bits 49-51  base offset (0: 1024-B aligned atoms)  bits 61-63 swizzle (2 = 128B)
SPEC_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;            // LBO unused by swizzled K-major layouts
    d |= static_cast<uint64_t>(1024u >> 4) << 32;    // 8 rows x 128 B between row groups
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: D f32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                                  // D format: f32
         | (1u << 7)                                  // A format: bf16
         | (1u << 10)                                 // B format: bf16
         | (static_cast<uint32_t>(N >> 3) << 17)
         | (static_cast<uint32_t>(M >> 4) << 24);
}

// Programmatic dependent launch: a kernel launched with the PDL attribute may
// start while the previous kernel on the stream is still running.  It must call
// pdl_wait() before touching memory the previous kernel reads or writes;
// pdl_trigger() lets the next kernel launch early.  Both are no-ops when the
// kernel was launched without the attribute.
SPEC_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
SPEC_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Arrival counter of a "last CTA finishes the job" pattern: the caller's CTA
// has synchronised (bar.sync) after its writes; one thread adds with
// acquire-release semantics at GPU scope, publishing the CTA's writes and, for
// the last arrival, making every other CTA's published writes visible (the
// following bar.sync extends that to the whole CTA).
SPEC_DEV int atomic_add_acq_rel(int* p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// named barrier among `count` threads (id 0 is __syncthreads)
SPEC_DEV void named_bar(int id, int count) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}

SPEC_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
SPEC_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
