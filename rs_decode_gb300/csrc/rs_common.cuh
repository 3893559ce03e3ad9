// Device-side building blocks shared by the librs kernels: bf16 <-> fp32
// conversion, streaming 128-bit memory access, the per-thread tile geometry
// of a (N x P) checkpoint slab, and a CTA reduction over threads that own the
// same value columns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rs.h"

namespace rs {

constexpr int kMaxCap = 32;  // circular buffer slots per sequence (one warp lane per record)
constexpr int kMaxT = 8;     // drafts per verify launch

enum Mode { MODE_DECODE = 0, MODE_VERIFY = 1, MODE_FLUSH = 2, MODE_MATERIALIZE = 3 };

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ float bf2f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }
__device__ __forceinline__ uint32_t f2bf(float f) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) { return f2bf(lo) | (f2bf(hi) << 16); }

// ---------------------------------------------------------------- memory
// The checkpoint is touched once per launch: stream it past the caches
// (evict-first) so the small, re-read buffer records stay resident in L2.
__device__ __forceinline__ uint4 ld_stream(const void *p) { return __ldcs(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ void st_stream(void *p, uint4 v) { __stcs(reinterpret_cast<uint4 *>(p), v); }
__device__ __forceinline__ void st_stream2(void *p, uint2 v) { __stcs(reinterpret_cast<uint2 *>(p), v); }
__device__ __forceinline__ uint4 ld_u4(const void *p) { return *reinterpret_cast<const uint4 *>(p); }

// Paired fp32 arithmetic (fma.rn.f32x2, mul.rn.f32x2; sm_100 and later): one
// instruction computes two lanes held in a 64-bit register pair, with the
// rounding of two separate fp32 operations.
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
    return (unsigned long long)__float_as_uint(hi) << 32 | __float_as_uint(lo);
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float &lo, float &hi) {
    lo = __uint_as_float((unsigned)v);
    hi = __uint_as_float((unsigned)(v >> 32));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Asynchronous global -> shared copies (cp.async): a CTA issues all of its
// small staging loads back to back and waits once.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async8(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

// Brings the 128-byte line holding p into L2 (no register, no wait).
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// An always-zero value that the compiler cannot see through; adding it to an
// address makes a later memory operation wait for the loads that produced x.
__device__ __forceinline__ unsigned zero_dependent_on(unsigned x) {
    unsigned z;
    asm volatile("and.b32 %0, %1, 0;" : "=r"(z) : "r"(x));
    return z;
}

// ---------------------------------------------------------------- mbarriers and bulk copies
// Shared-memory transaction barriers and the bulk (TMA) copy engine, used by
// the streaming pipeline.  Every wait is bounded: after kWaitLimitNs of
// global time it gives up and returns false, so no launch can hang.  A build
// may shorten the limit (-DRS_WAIT_LIMIT_NS=...), as the time-out test does.
#ifndef RS_WAIT_LIMIT_NS
#define RS_WAIT_LIMIT_NS 2000000000ull  // 2 s
#endif
constexpr unsigned long long kWaitLimitNs = RS_WAIT_LIMIT_NS;

__device__ __forceinline__ unsigned smem_u32(const void *p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, unsigned bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// As mbar_try_wait, but a thread whose phase is not complete yet sleeps until
// it completes or kSleepHintNs pass, instead of returning at once: waiting
// warps then take no issue slots from the working ones.
constexpr unsigned kSleepHintNs = 100000;  // 100 us
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSleepHintNs)
        : "memory");
    return ok != 0;
}
// Waits for the phase of the given parity to complete; false on time-out.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, unsigned parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_sleep(bar, parity)) {
        if (global_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// Bulk copy of `bytes` contiguous bytes global -> shared, completing on `bar`,
// with an evict-first L2 policy (the checkpoint is read once per launch).
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], pol;\n\t}" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Tiled tensor copy (TMA) of one box global -> shared, completing on `bar`,
// evict-first in L2.  `tmap` is the address of a CUtensorMap kernel parameter;
// c0..c3 are the box's start coordinates, innermost first.
__device__ __forceinline__ void tma_load_4d(void *dst, const void *tmap, int c0, int c1, int c2, int c3,
                                            uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .b64 pol;\n\t"
        "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], pol;\n\t}" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
        : "memory");
}

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// ---------------------------------------------------------------- tensor cores (tcgen05)
// Fifth-generation tensor core operations: the accumulator lives in tensor
// memory (TMEM, 128 lanes x 512 32-bit columns per SM), operands are read from
// shared memory through 64-bit matrix descriptors, one thread issues the MMA,
// and its completion is signalled on an mbarrier.

// TMEM columns of a CTA (allocated by one whole warp; the address lands in
// shared memory).  The permit is given up at once so that the other CTA of the
// SM can allocate too.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, int ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, int ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads of them (tensor core operands, bulk copies).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (16-byte units), descriptor version 1, layout (0 = no swizzle,
// 2 = 128-byte swizzle).  Swizzled operands start on 1024-byte boundaries.
__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}
// Instruction descriptor of kind::f16 with bf16 A and B, fp32 accumulation;
// a_mn / b_mn select MN-major operands.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
// D[tmem] (+)= A * B, issued by a single thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((uint32_t)accumulate)
        : "memory");
}
// The mbarrier receives one arrival once every MMA this thread issued so far
// has completed (its operands read, its results in TMEM).
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// A warp reads NV consecutive 32-bit columns of its 32 TMEM lanes (lane
// quarter = warp % 4): lane l gets row 32 (warp % 4) + l.
template <int NV> __device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[NV]);
template <> __device__ __forceinline__ void tmem_ld<2>(uint32_t taddr, float (&v)[2]) {
    uint32_t r[2];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    v[0] = __uint_as_float(r[0]); v[1] = __uint_as_float(r[1]);
}
template <> __device__ __forceinline__ void tmem_ld<4>(uint32_t taddr, float (&v)[4]) {
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
template <> __device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
template <> __device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Named barrier over the first `count` threads of the CTA (the consumer
// warps) that also ORs a flag over them: every participant gets the same
// answer, so an abort decided on it is uniform and no thread is left waiting.
__device__ __forceinline__ bool named_sync_or(int id, int count, bool flag) {
    unsigned r;
    asm volatile(
        "{\n\t.reg .pred q, o;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred o, %2, %3, q;\n\tselp.u32 %0, 1, 0, o;\n\t}"
        : "=r"(r)
        : "r"((unsigned)flag), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------- tile geometry
// A (N x P) checkpoint slab is row-major with P contiguous.  A thread owns VEC
// consecutive value columns (one 16-byte vector) of R consecutive key rows:
// TPR threads cover one row, the CTA's NT threads cover RG = NT/TPR row
// groups.  Every row is a contiguous P*sizeof(TE)-byte segment, so each warp
// load instruction reads 32/TPR whole rows.
template <typename TE> struct Vec;
template <> struct Vec<float> { static constexpr int n = 4; };
template <> struct Vec<uint16_t> { static constexpr int n = 8; };

template <int P, int N, int NT, typename TE> struct Geo {
    static constexpr int VEC = Vec<TE>::n;
    static constexpr int TPR = P / VEC;
    static constexpr int RG = NT / TPR;
    static constexpr int R = N / RG;
    static_assert(P % VEC == 0 && TPR <= 32 && 32 % TPR == 0, "row must map onto a warp fraction");
    static_assert(NT % TPR == 0 && N % RG == 0 && R >= 1, "rows must split evenly over row groups");
};

template <typename TE, int VEC>
__device__ __forceinline__ void unpack(const uint4 &u, float (&f)[VEC]);
template <> __device__ __forceinline__ void unpack<float, 4>(const uint4 &u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
template <> __device__ __forceinline__ void unpack<uint16_t, 8>(const uint4 &u, float (&f)[8]) {
    f[0] = bf2f(u.x & 0xffffu); f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = bf2f(u.y & 0xffffu); f[3] = __uint_as_float(u.y & 0xffff0000u);
    f[4] = bf2f(u.z & 0xffffu); f[5] = __uint_as_float(u.z & 0xffff0000u);
    f[6] = bf2f(u.w & 0xffffu); f[7] = __uint_as_float(u.w & 0xffff0000u);
}

// Store VEC fp32 values to an fp32 array (16 or 32 bytes).
template <int VEC>
__device__ __forceinline__ void store_f32(float *dst, const float (&f)[VEC]) {
#pragma unroll
    for (int c = 0; c < VEC / 4; ++c)
        st_stream(dst + 4 * c, make_uint4(__float_as_uint(f[4 * c]), __float_as_uint(f[4 * c + 1]),
                                          __float_as_uint(f[4 * c + 2]), __float_as_uint(f[4 * c + 3])));
}
// Store VEC values rounded to bf16 (8 or 16 bytes).
template <int VEC>
__device__ __forceinline__ void store_bf16(uint16_t *dst, const float (&f)[VEC]) {
    if constexpr (VEC == 4) {
        st_stream2(dst, make_uint2(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3])));
    } else {
        st_stream(dst, make_uint4(pack_bf2(f[0], f[1]), pack_bf2(f[2], f[3]), pack_bf2(f[4], f[5]),
                                  pack_bf2(f[6], f[7])));
    }
}

// Copy `count` bf16 values (count % 8 == 0, 16-byte aligned) into fp32 shared memory.
__device__ __forceinline__ void bf16_row_to_smem(float *dst, const uint16_t *src, int count, int lane0,
                                                 int stride) {
    for (int c = lane0; c < count / 8; c += stride) {
        uint4 u = ld_u4(src + 8 * c);
        float f[8];
        unpack<uint16_t, 8>(u, f);
        float4 *d = reinterpret_cast<float4 *>(dst + 8 * c);
        d[0] = make_float4(f[0], f[1], f[2], f[3]);
        d[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
}

// ---------------------------------------------------------------- CTA reduction
// Each thread holds acc[NV][VEC] partial sums for value columns pv*VEC..+VEC of
// NV vectors.  Sums over all threads with the same pv and leaves the totals
// in red[v*P + p] (v < nv), using red[NW][NV*P] as scratch.  Call from all
// threads; contains two __syncthreads.
template <int NT, int TPR, int VEC, int P, int NV>
__device__ __forceinline__ void cta_reduce(float (&acc)[NV][VEC], int nv, float *red) {
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int off = TPR; off < 32; off <<= 1)
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[v][e] += __shfl_xor_sync(0xffffffffu, acc[v][e], off);
    if (lane < TPR) {
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            if (v < nv) {
                float *d = red + ((size_t)warp * nv + v) * P + lane * VEC;
#pragma unroll
                for (int c = 0; c < VEC / 4; ++c)
                    reinterpret_cast<float4 *>(d)[c] =
                        make_float4(acc[v][4 * c], acc[v][4 * c + 1], acc[v][4 * c + 2], acc[v][4 * c + 3]);
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < nv * P; i += NT) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) s += red[(size_t)w * nv * P + i];
        red[i] = s;
    }
    __syncthreads();
}

}  // namespace rs
