// Small-batch standard decode for Mamba-2 with the fp32 checkpoint: the same
// output-only replay as the streaming pipeline ("ReplaySSM: Cache SSM Inputs,
// Not State", section "How it works": y = gamma S_c q + sum_r w_r dt_r x_r
// (B_r . q) + D x, a fold S_c <- gamma S_c + sum_r w_r dt_r x_r B_r^T on the
// step that fills the window), shaped for batches too small to fill the GPU
// with pipelined units.
//
// One CTA per HPC heads of one sequence and no pipeline: every thread issues
// its checkpoint loads (HPC slabs, R rows x VEC columns each) into registers
// before anything waits; thread 0 plans the sequence from its pointers, and
// the small operands (records, keys, this step's inputs) land in shared memory
// with one batch of cp.async copies while the slabs arrive.  So the
// launch's critical path is one load latency plus the arithmetic, where the
// pipeline's is a chain of plan, stage and hand-over waits per unit, which a
// small batch cannot hide behind other units.  A CTA that folds rewrites its
// own slabs from the registers it read them into.
#include <cuda_runtime.h>

#include "rs.h"
#include "rs_common.cuh"
#include "rs_internal.h"
#include "rs_plan.cuh"

// Batches up to this size take this kernel, larger ones the pipeline.  GPU
// time per step of the 128-head Mamba-2 layer (CUDA-graph replay of whole
// windows): B = 8, 8.97 against 10.31 us; B = 16, 15.85 against 13.13 us.
#ifndef RS_DIRECT_MAX_B
#define RS_DIRECT_MAX_B 8
#endif

namespace rs {
namespace direct {

template <int P, int N, int HPC, int NT>
__global__ void __launch_bounds__(NT) decode_kernel(const ReplayParams p) {
    using Gm = Geo<P, N, NT, float>;
    constexpr int VEC = Gm::VEC, TPR = Gm::TPR, R = Gm::R, NW = NT / 32;
    constexpr int KROW_Q = kMaxCap;  // key row of the query C
    static_assert(R == 8 && VEC == 4, "a thread's rows are one 16-byte run of bf16 keys");
    __shared__ __align__(16) uint16_t kraw[(kMaxCap + 1) * N];  // records' keys B_r; row KROW_Q: C
    __shared__ __align__(16) uint16_t xb[HPC * kMaxCap * P];    // records' x, per head
    __shared__ float sr[HPC * kMaxCap], ar[HPC * kMaxCap];       // dt_r, alpha_r
    __shared__ float dq[kMaxCap];                                // B_r . C
    __shared__ float cy[HPC * kMaxCap], fw[HPC * kMaxCap];       // output / fold coefficients
    __shared__ float cst[2 * HPC], gy[HPC];                      // A_h, D_h; gamma
    __shared__ __align__(16) float rec[HPC * P];                 // record parts of the outputs
    __shared__ __align__(16) float red[NW * HPC * P];
    __shared__ SeqPlan sp;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.y, h0 = blockIdx.x * HPC;
    const int H = p.H, G = p.G, cap = p.cap;
    const int g = h0 / (H / G);
    // ---- 1. the checkpoint slabs, into registers (their addresses do not
    // depend on the sequence's pointers, so the loads go out first)
    const int n0 = (tid / TPR) * R, p0 = (tid % TPR) * VEC;
    const size_t slab = (size_t)N * P;
    uint4 tile[HPC][R];
#pragma unroll
    for (int hd = 0; hd < HPC; ++hd) {
        const float *src = p.ckpt_hp + ((size_t)b * H + h0 + hd) * slab + (size_t)n0 * P + p0;
#pragma unroll
        for (int k = 0; k < R; ++k) tile[hd][k] = __ldg(reinterpret_cast<const uint4 *>(src + (size_t)k * P));
    }
    if (tid == 0) sp = plan_sequence(p, b);
    __syncthreads();
    const SeqPlan s = sp;
    const int base = s.base, hc = s.hc, nrec = hc + 1;
    auto slot = [&](int r) {  // base < cap and r < cap (plan_sequence)
        const int v = base + r;
        return v >= cap ? v - cap : v;
    };
    if (!s.work) {
        if (tid == 0) arrive_and_update(p, s, b, (unsigned)(H / HPC), h0 == 0);
        return;
    }

    // ---- 2. the small operands: one batch of cp.async copies
    {
        constexpr int KC = N / 8, XC = P / 8;
        for (int i2 = tid; i2 < (nrec + 1) * KC; i2 += NT) {
            const int rr = i2 / KC, c = i2 % KC;
            const uint16_t *src = rr < hc    ? p.buf_k + (((size_t)b * cap + slot(rr)) * G + g) * N
                                  : rr == hc ? p.Bm + ((size_t)b * G + g) * N
                                             : p.Cm + ((size_t)b * G + g) * N;
            cp_async16(kraw + (size_t)(rr <= hc ? rr : KROW_Q) * N + 8 * c, src + 8 * c);
        }
        for (int i2 = tid; i2 < HPC * nrec * XC; i2 += NT) {
            const int c = i2 % XC, r = (i2 / XC) % nrec, hd = i2 / (XC * nrec), hh = h0 + hd;
            const uint16_t *src = r < hc
                ? static_cast<const uint16_t *>(p.buf_v) + (((size_t)b * cap + slot(r)) * H + hh) * P
                : p.x + ((size_t)b * H + hh) * P;
            cp_async16(xb + ((size_t)hd * kMaxCap + r) * P + 8 * c, src + 8 * c);
        }
        for (int i2 = tid; i2 < HPC * nrec; i2 += NT) {
            const int r = i2 % nrec, hd = i2 / nrec, hh = h0 + hd;
            if (r < hc) {
                const size_t ri = ((size_t)b * cap + slot(r)) * H + hh;
                cp_async4(ar + hd * kMaxCap + r, p.buf_a + ri);
                cp_async4(sr + hd * kMaxCap + r, p.buf_s + ri);
            } else {
                cp_async4(sr + hd * kMaxCap + r, p.dt + (size_t)b * H + hh);
            }
        }
        if (tid < HPC) {
            cp_async4(cst + tid, p.A + h0 + tid);
            if (p.D) cp_async4(cst + HPC + tid, p.D + h0 + tid);
            else cst[HPC + tid] = 0.f;
        }
        // the arrival follows this CTA's pointer reads (the last arriver writes
        // the new pointers); its atomic overlaps the copies in flight
        if (tid == 0) arrive_and_update(p, s, b, (unsigned)(H / HPC), h0 == 0);
        cp_async_wait_all();
    }
    __syncthreads();

    // ---- 3. this step's record: its decay alpha = exp(dt A); the append
    if (tid < HPC) {
        const float a = expf(sr[tid * kMaxCap + hc] * cst[tid]);
        ar[tid * kMaxCap + hc] = a;
        if (s.append) {
            const size_t ri = ((size_t)b * cap + slot(hc)) * H + h0 + tid;
            p.buf_a[ri] = a;
            p.buf_s[ri] = sr[tid * kMaxCap + hc];
        }
    }
    if (s.append) {
        if (h0 % (H / G) == 0) {  // the group's first CTA appends the key
            uint16_t *dst = p.buf_k + (((size_t)b * cap + slot(hc)) * G + g) * N;
            for (int c = tid; c < N / 8; c += NT)
                reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(kraw + (size_t)hc * N)[c];
        }
        for (int i2 = tid; i2 < HPC * (P / 8); i2 += NT) {
            const int c = i2 % (P / 8), hd = i2 / (P / 8);
            uint16_t *dst = static_cast<uint16_t *>(p.buf_v) + (((size_t)b * cap + slot(hc)) * H + h0 + hd) * P;
            reinterpret_cast<uint4 *>(dst)[c] = reinterpret_cast<const uint4 *>(xb + ((size_t)hd * kMaxCap + hc) * P)[c];
        }
    }

    // ---- 4. key / query dots B_r . C, 8 lanes per record (nrec <= 32 <= NT / 8)
    {
        const int d = tid / 8, sub = tid % 8;
        float acc = 0.f;
        if (d < nrec) {
            for (int n = sub * 8; n < N; n += 64) {
                float fa[8], fb[8];
                unpack<uint16_t, 8>(ld_u4(kraw + (size_t)d * N + n), fa);
                unpack<uint16_t, 8>(ld_u4(kraw + (size_t)KROW_Q * N + n), fb);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(fa[e], fb[e], acc);
            }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
        if (d < nrec && sub == 0) dq[d] = acc;
    }
    __syncthreads();

    // ---- 5. decay coefficients, one warp per head and one lane per record:
    // with E(r) = prod_{s = r+1 .. hc} alpha_s and gamma = prod_{s <= hc} alpha_s,
    // the output takes E(r) dt_r (B_r . C) x_r and the fold E(r) dt_r x_r B_r^T
    for (int hd = warp; hd < HPC; hd += NW) {
        const float al = lane < nrec ? ar[hd * kMaxCap + lane] : 1.f;
        float inc = al;  // prod_{s >= lane} alpha_s
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_down_sync(0xffffffffu, inc, off);
            if (lane + off < 32) inc *= o;
        }
        float E = __shfl_down_sync(0xffffffffu, inc, 1);
        if (lane == 31) E = 1.f;
        const float gam = __shfl_sync(0xffffffffu, inc, 0);
        if (lane < nrec) {
            const float w = E * sr[hd * kMaxCap + lane];
            cy[hd * kMaxCap + lane] = w * dq[lane];
            fw[hd * kMaxCap + lane] = w;
        }
        if (lane == 0) gy[hd] = gam;
    }
    __syncthreads();

    // ---- 6. record parts of the outputs, rec[p] = sum_r cy_r x_r[p] + D x[p]
    for (int i2 = tid; i2 < HPC * P; i2 += NT) {
        const int pp = i2 % P, hd = i2 / P;
        const uint16_t *xr = xb + (size_t)hd * kMaxCap * P + pp;
        float a = cst[HPC + hd] * bf2f(xr[(size_t)hc * P]);
        for (int r = 0; r < nrec; ++r) a = fmaf(cy[hd * kMaxCap + r], bf2f(xr[(size_t)r * P]), a);
        rec[i2] = a;
    }

    // ---- 7. the checkpoint dotted with C; y = gamma (S_c C) + rec
    float cq[R];
    unpack<uint16_t, 8>(ld_u4(kraw + (size_t)KROW_Q * N + n0), cq);
    float acc[HPC][VEC];
#pragma unroll
    for (int hd = 0; hd < HPC; ++hd) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[hd][e] = 0.f;
#pragma unroll
        for (int k = 0; k < R; ++k) {
            float sv[VEC];
            unpack<float, VEC>(tile[hd][k], sv);
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[hd][e] = fmaf(sv[e], cq[k], acc[hd][e]);
        }
    }
    cta_reduce<NT, TPR, VEC, P, HPC>(acc, HPC, red);  // (rec is complete after its barriers)
    for (int i2 = tid; i2 < HPC * P; i2 += NT) {
        const int pp = i2 % P, hd = i2 / P;
        p.y[((size_t)b * H + h0 + hd) * P + pp] = fmaf(gy[hd], red[i2], rec[i2]);
    }

    // ---- 8. the fold on the step that fills the window (F = hc + 1 records)
    if (s.fold) {
#pragma unroll
        for (int hd = 0; hd < HPC; ++hd) {
            const float gf = gy[hd];
            float o[R][VEC];
#pragma unroll
            for (int k = 0; k < R; ++k) {
                unpack<float, VEC>(tile[hd][k], o[k]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[k][e] *= gf;
            }
            const uint16_t *xr = xb + (size_t)hd * kMaxCap * P + p0;
            for (int r = 0; r < nrec; ++r) {
                float xv[VEC], kv[R];
                const uint2 xu = *reinterpret_cast<const uint2 *>(xr + (size_t)r * P);
                xv[0] = bf2f(xu.x & 0xffffu); xv[1] = __uint_as_float(xu.x & 0xffff0000u);
                xv[2] = bf2f(xu.y & 0xffffu); xv[3] = __uint_as_float(xu.y & 0xffff0000u);
                unpack<uint16_t, 8>(ld_u4(kraw + (size_t)r * N + n0), kv);
                const float w = fw[hd * kMaxCap + r];
#pragma unroll
                for (int e = 0; e < VEC; ++e) xv[e] *= w;
#pragma unroll
                for (int k = 0; k < R; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) o[k][e] = fmaf(xv[e], kv[k], o[k][e]);
            }
            const size_t off = ((size_t)b * H + h0 + hd) * slab + (size_t)n0 * P + p0;
#pragma unroll
            for (int k = 0; k < R; ++k) {
                store_f32<VEC>(p.ckpt_hp + off + (size_t)k * P, o[k]);
                if (p.ckpt_lp) store_bf16<VEC>(p.ckpt_lp + off + (size_t)k * P, o[k]);
            }
        }
    }
}

}  // namespace direct

// Whether a replay launch takes the small-batch decode kernel.
bool replay_direct_applies(const ReplayParams &p, int kind, int P, int N) {
    return kind == RS_MAMBA2 && P == 64 && N == 128 && p.mode == MODE_DECODE && p.prec == RS_PREC_FP32 &&
           p.B <= RS_DIRECT_MAX_B && p.cap <= kMaxCap && (p.H / p.G) % 2 == 0;
}

cudaError_t replay_direct_launch(const ReplayParams &p, cudaStream_t s) {
    constexpr int HPC = 2, NT = 256;
    direct::decode_kernel<64, 128, HPC, NT><<<dim3(p.H / HPC, p.B), NT, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace rs
